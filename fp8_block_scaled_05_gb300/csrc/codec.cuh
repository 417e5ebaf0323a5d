// Device-side pieces of the block quantisers: bf16 unpacking, block amax,
// the two scale rules, the per-element cast and the E4M3 conversion.
//
// Method (page "NVIDIA NeMo RL достигает ускорения на 48% благодаря
// сквозному обучению с точностью FP8", greentreeone.com, §Технический
// прорыв; power-of-two option: upppp.jp NeMo RL FP8 article, §設定方法):
//   s = RN_fp32(amax / 448)   or   s = 2^ceil(log2(amax / 448)) (clamped to
//   [2^-127, 2^127]); s = 1 for an all-zero block;
//   q = e4m3_RNE_satfinite( RN_fp32(x * r) ),  r = RN_fp32(448 / amax)
//   (r = 2^-e for the power-of-two scale; the division x / s where r
//   overflows fp32).
#pragma once
#include <cstdint>

namespace fp8bs {

// Two bf16 values packed in a 32-bit word (element 2i in the low half) to fp32.
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Element-wise max of the magnitudes of two bf16 pairs, as bf16 bit patterns.
// For non-NaN bf16, |x| ordered as floats equals its bits ordered as
// unsigned integers, so a packed unsigned 16-bit max gives the amax.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) {
    uint32_t r;
    const uint32_t a = w & 0x7FFF7FFFu;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(a));
    return r;
}

// Larger of the two halves, as the fp32 value of that bf16.
__device__ __forceinline__ float absmax_pair_to_f32(uint32_t m) {
    const uint32_t lo = m & 0xFFFFu, hi = m >> 16;
    return __uint_as_float((lo > hi ? lo : hi) << 16);
}

// Power-of-two exponent e = ceil(log2(amax / 448)), clamped to [-127, 127];
// 0 for amax == 0.  448 = 1.75 * 2^8: with amax = F * 2^E, F in [1, 2),
// e = E - 8 when F <= 1.75 and E - 7 when F > 1.75.
__device__ __forceinline__ int pow2_exponent(float amax) {
    const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
    if (b == 0) return 0;
    int E;
    uint32_t mant;                       // 23-bit fraction of F
    const uint32_t ef = b >> 23;
    if (ef != 0) {
        E = (int)ef - 127;
        mant = b & 0x7FFFFFu;
    } else {                             // fp32 subnormal: normalise
        const int lz = __clz(b) - 8;     // leading zeros inside the 23-bit field (+1 for the hidden bit)
        E = -126 - lz;
        mant = (b << lz) & 0x7FFFFFu;
    }
    int e = E - 8 + (mant > 0x600000u ? 1 : 0);   // F > 1.75  <=>  fraction > 0.75
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
    return e;
}

// 2^e as fp32 for e in [-127, 127] (2^-127 is subnormal, exact).
__device__ __forceinline__ float exp2_int(int e) {
    return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// Per-block constants of the cast.  The pages give the scale as amax/448 and
// leave open whether the cast divides by it or multiplies by its
// reciprocal; the cast here multiplies by the reciprocal factor r (the usual
// form of an FP8 cast): code = e4m3(RN(x r)) with r = RN(448/amax) for an
// fp32 scale, r = 2^-e (exact, so x r = x/s) for a power-of-two scale, and
// r = RN(1/s) for a cast with a given scale.  Where r overflows fp32 (amax
// below 448 * 2^-128, or s below 2^-128) the cast divides by s instead.
struct BlockScale {
    float s;         // the stored scale
    float r;         // the cast's factor (see above)
    int mode;        // 1: product x * r, 2: IEEE division x / s (r not finite)
};

__device__ __forceinline__ int cast_mode(float r) {
    return (__float_as_uint(r) & 0x7FFFFFFFu) < 0x7F800000u ? 1 : 2;
}

__device__ __forceinline__ BlockScale make_scale(float amax, bool pow2) {
    BlockScale bs;
    if (pow2) {
        const int e = pow2_exponent(amax);
        bs.s = exp2_int(e);
        bs.r = exp2_int(-e);             // exact; x * 2^-e == x / 2^e for every bf16 x in the block
        bs.mode = 1;
        return bs;
    }
    if (!(amax > 0.0f)) {
        bs.s = 1.0f;
        bs.r = 1.0f;
        bs.mode = 1;
        return bs;
    }
    bs.s = __fdiv_rn(amax, 448.0f);
    bs.r = __fdiv_rn(448.0f, amax);
    bs.mode = cast_mode(bs.r);
    return bs;
}

// The per-block constants from a stored scale s and the cast's factor r (as
// make_scale produced them); lets one lane compute a block's scale and others
// rebuild it from two shuffled values.
__device__ __forceinline__ BlockScale scale_from_sr(float s, float r, bool pow2) {
    BlockScale bs;
    bs.s = s;
    bs.r = r;
    bs.mode = pow2 ? 1 : cast_mode(r);
    return bs;
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Two fp32 values to two E4M3 codes (round to nearest even, saturating to
// +-448); `lo` goes to bits 0..7, `hi` to bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

// Both elements of a pair times one factor, as one packed multiply (each
// lane an IEEE mul.rn.f32, so the products equal two scalar multiplies).
__device__ __forceinline__ void mul2(float a, float b, float f, float &pa, float &pb) {
    uint64_t x, k;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
    asm("mov.b64 %0, {%1, %1};" : "=l"(k) : "f"(f));
    asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(x) : "l"(k));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(pa), "=f"(pb) : "l"(x));
}

// Codes of two elements: one packed multiply and one conversion per pair
// (mode 2, a block whose reciprocal factor overflows, divides).  The test of
// the mode per pair is costly in a hot loop (in the GEMM's fused epilogue it
// made the cast 3.5x slower): where the mode can be decided once, for a warp
// (a vote) or a whole tile, callers take quant8_mul when it is 1.
__device__ __forceinline__ uint32_t quant_pair(float xa, float xb, const BlockScale &bs) {
    if (bs.mode == 1) {
        float qa, qb;
        mul2(xa, xb, bs.r, qa, qb);
        return e4m3x2(qa, qb);
    }
    return e4m3x2(__fdiv_rn(xa, bs.s), __fdiv_rn(xb, bs.s));
}

// Quantises eight bf16 values (one 16-byte load) to eight codes (8 bytes).
__device__ __forceinline__ uint2 quant8(const uint4 &v, const BlockScale &bs) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = quant_pair(bf16lo_to_f32(w[i]), bf16hi_to_f32(w[i]), bs);
    return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

// quant8 for a block in mode 1 (every power-of-two scale, and every fp32
// scale whose factor r is finite): both elements of a pair in one packed
// multiply, then one conversion.
__device__ __forceinline__ uint2 quant8_mul(const uint4 &v, float r) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float qa, qb;
        mul2(bf16lo_to_f32(w[i]), bf16hi_to_f32(w[i]), r, qa, qb);
        p[i] = e4m3x2(qa, qb);
    }
    return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

// The cast of eight values with the choice fixed at compile time: MUL, the
// product path (mode 1); otherwise the per-pair test.  with_cast(all_mul, f)
// calls f with CastTag<true> or CastTag<false> once, so that a caller branches
// on its warp-uniform choice outside its loops (a test inside them, even a
// uniform one, cost 10-17% in the quantisers).
template <bool MUL>
struct CastTag {
    static constexpr bool mul = MUL;
};

template <bool MUL>
__device__ __forceinline__ uint2 quant8_as(const uint4 &v, const BlockScale &bs) {
    if constexpr (MUL)
        return quant8_mul(v, bs.r);
    else
        return quant8(v, bs);
}

template <typename F>
__device__ __forceinline__ void with_cast(bool all_mul, F &&f) {
    if (all_mul)
        f(CastTag<true>{});
    else
        f(CastTag<false>{});
}

__device__ __forceinline__ uint32_t absmax8(uint32_t acc, const uint4 &v) {
    acc = absmax_bf16x2(acc, v.x);
    acc = absmax_bf16x2(acc, v.y);
    acc = absmax_bf16x2(acc, v.z);
    return absmax_bf16x2(acc, v.w);
}

}  // namespace fp8bs
