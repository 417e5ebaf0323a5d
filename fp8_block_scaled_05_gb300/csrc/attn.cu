// FP8 KV cache and decode attention.
//
// Page "NVIDIA NeMo RL FP8" (upppp.jp), §KVキャッシュとAttentionにも拡張: the
// KV cache and the attention run in FP8 during rollout; the Q, K and V scales
// are recomputed after every training step (the policy changes) and used for
// the next rollout.  Here: one fp32 scale per tensor for each of Q, K and V;
// the cache holds E4M3 codes cast with the calibrated scales; one decode step
// computes, per sequence b and query head h (KV head g = h / G),
//
//   o[b, h] = softmax_t( q[b, h] . k[b, g, t] / sqrt(D) ) v[b, g, t],   t < len[b]
//
// on the dequantised values, in fp32.
//
// k_decode_attn: one CTA per (key split, KV head, sequence), 4 warps.  The G
// query heads of the group share every K/V byte the CTA reads.
//   scores  Q K^T on the tensor cores straight from the E4M3 codes
//           (mma.sync m16n8k32 e4m3, fp32 accumulation): the G <= 8 heads
//           are the MMA's rows (the rest zero), 8 keys per MMA column tile,
//           4 tiles = the warp's block of 32 keys, 4 k-steps = D.  The dot
//           product sums over all dims, so the k positions can take the dims
//           in any order that A and B share: lane (group r, j = lane % 4)
//           loads the 32-byte segment j of its key's row, and k-step s uses
//           bytes 8s .. 8s+7 of it (the query segment likewise);
//   softmax online per warp, on the C fragments (head r's scores sit in
//           lanes 4r .. 4r+3: two shuffles per reduction), exp2 with the
//           scale product and log2(e)/sqrt(D) folded in;
//   P V     on the CUDA cores, lanes over dims: lane l adds p_t v[t, 4l .. 4l+3]
//           for the block's 32 keys, packed fma.rn.f32x2;
//   loads   each warp streams its key blocks through two shared-memory
//           stages with cp.async (16 bytes per lane, zero-filled past the
//           sequence), the next block's K and V landing while the current one
//           is computed;
//   merge   the 4 warps' (m, l, o) in shared memory; with several splits the
//           CTA writes (m, l, o) and k_attn_combine merges the splits.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "codec.cuh"
#include "internal.h"

namespace fp8bs {

constexpr int kAttnD = 128;
constexpr int kAttnWarps = 4;
constexpr int kAttnSplit = 512;   // keys per CTA (4 warps x 4 blocks of 32)

// Four E4M3 codes (bytes of w, byte 0 first) -> fp32.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float (&f)[4]) {
    uint32_t h01, h23;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"((uint16_t)(w & 0xFFFFu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"((uint16_t)(w >> 16)));
    const __half2 a = *reinterpret_cast<const __half2*>(&h01);
    const __half2 b = *reinterpret_cast<const __half2*>(&h23);
    f[0] = __low2float(a);
    f[1] = __high2float(a);
    f[2] = __low2float(b);
    f[3] = __high2float(b);
}

// fp32 -> bf16 bits, round to nearest even.
__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// 16-byte global -> shared copy, zero-filled when !valid (nothing is read).
__device__ __forceinline__ void cp16(void* dst, const void* src, bool valid) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Per warp, per stage: 32 key rows (16-byte chunk c of row r at chunk
// c ^ (r % 8), so the fragment reads below spread over all banks) and 32
// value rows, 4 KB each.
constexpr int kAttnStages = 2;
constexpr int kAttnStageBytes = 2 * 32 * kAttnD;
constexpr int kAttnSmemBytes = kAttnWarps * kAttnStages * kAttnStageBytes;

// D = A B + C for one m16n8k32 tile, A (16 x 32) and B (32 x 8) E4M3, fp32 C/D.
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// acc[0..1] += p * (v0, v1) as one packed FMA.
__device__ __forceinline__ void fma2(float& a0, float& a1, float p, float v0, float v1) {
    uint64_t a, v, pp;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(v0), "f"(v1));
    asm("mov.b64 %0, {%1, %1};" : "=l"(pp) : "f"(p));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(v), "l"(pp));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
}

// part: [B][Hq][n_split][2 + D] floats (m in log2 units, l, o unnormalised)
// when n_split > 1; otherwise the output is written directly.
template <int G>
__global__ void __launch_bounds__(32 * kAttnWarps) k_decode_attn(
    const uint8_t* __restrict__ q, const float* __restrict__ sq, const uint8_t* __restrict__ kc,
    const float* __restrict__ sk, const uint8_t* __restrict__ vc, const float* __restrict__ sv,
    const int32_t* __restrict__ seq_lens, int Hkv, int T, int n_split, float* __restrict__ part,
    uint16_t* __restrict__ out) {
    constexpr int D = kAttnD;
    static_assert(G >= 1 && G <= 8, "query heads per KV head");
    __shared__ float ps[kAttnWarps][G][32];
    __shared__ float cs[kAttnWarps][G];
    __shared__ float wm[kAttnWarps][G], wl[kAttnWarps][G];
    __shared__ __align__(16) float wo[kAttnWarps][G][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane >> 2, j = lane & 3;   // MMA row (head) and 32-byte segment
    const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int Hq = Hkv * G;
    const int L = min(max(seq_lens[b], 0), T);
    const int t0 = sp * kAttnSplit, t1 = min(t0 + kAttnSplit, L);

    // A fragments: head grp's query segment j (zero rows past the group)
    uint32_t qa[8];
    {
        uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
        if (grp < G) {
            const uint4* qrow = reinterpret_cast<const uint4*>(q + ((size_t)b * Hq + g * G + grp) * D + 32 * j);
            q0 = __ldg(qrow);
            q1 = __ldg(qrow + 1);
        }
        qa[0] = q0.x; qa[1] = q0.y; qa[2] = q0.z; qa[3] = q0.w;
        qa[4] = q1.x; qa[5] = q1.y; qa[6] = q1.z; qa[7] = q1.w;
    }
    // scores in log2 units: raw code products times sq sk log2(e) / sqrt(D)
    const float c = sq[0] * sk[0] * (1.4426950408889634f * 0.08838834764831845f);
    const float vscale = sv[0];
    const size_t head_base = ((size_t)b * Hkv + g) * (size_t)T * D;
    float m = -INFINITY, l = 0.0f;             // head grp's state (lanes 4 grp .. 4 grp + 3)
    float o[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[h][e] = 0.0f;

    // the warp's key blocks: tb = t0 + 32 warp + 128 i
    extern __shared__ __align__(128) uint8_t attn_smem[];
    uint8_t* wbuf = attn_smem + (size_t)warp * kAttnStages * kAttnStageBytes;
    auto issue = [&](int tb, int stage) {   // cp.async of block tb into `stage`
        uint8_t* ks = wbuf + stage * kAttnStageBytes;
        uint8_t* vs = ks + 32 * D;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int qi = lane + 32 * u, r = qi >> 3, c = qi & 7;
            const bool valid = tb + r < t1;
            const size_t off = head_base + (size_t)(valid ? tb + r : 0) * D + 16 * c;
            cp16(ks + r * D + 16 * (c ^ (r & 7)), kc + off, valid);
            cp16(vs + r * D + 16 * c, vc + off, valid);
        }
    };
    int tb = t0 + 32 * warp;
    if (tb < t1) issue(tb, 0);
    cp_commit();
    for (int it = 0; tb < t1; tb += 32 * kAttnWarps, ++it) {
        const int stage = it & 1;
        if (tb + 32 * kAttnWarps < t1) issue(tb + 32 * kAttnWarps, stage ^ 1);
        cp_commit();
        cp_wait<1>();   // this block's copies (all but the newest group) have landed
        __syncwarp();
        const uint8_t* ks = wbuf + stage * kAttnStageBytes;
        const uint8_t* vs = ks + 32 * D;
        const int nk = min(32, t1 - tb);   // warp-uniform
        float sc[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            // B fragments: key row 8 nt + grp, 32-byte segment j (chunks 2j, 2j+1)
            const int r = 8 * nt + grp;
            const uint4 k0 = *reinterpret_cast<const uint4*>(ks + r * D + 16 * ((2 * j) ^ (r & 7)));
            const uint4 k1 = *reinterpret_cast<const uint4*>(ks + r * D + 16 * ((2 * j + 1) ^ (r & 7)));
            const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[nt][e] = 0.0f;
#pragma unroll
            for (int ksx = 0; ksx < 4; ++ksx) mma_e4m3_16832(sc[nt], qa[2 * ksx], qa[2 * ksx + 1], kw[2 * ksx], kw[2 * ksx + 1]);
        }
        // this lane: head grp, keys tb + 8 nt + 2 j + e (e = 0, 1)
        float s8[8];
        float bm = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const bool valid = 8 * nt + 2 * j + e < nk;
                s8[2 * nt + e] = valid ? sc[nt][e] * c : -INFINITY;
                bm = fmaxf(bm, s8[2 * nt + e]);
            }
        bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, 1));
        bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, 2));   // key tb is valid: bm is finite
        const float mn = fmaxf(m, bm);
        const float corr = exp2f(m - mn);                        // 0 while m is -inf
        float psum = 0.0f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float pv = exp2f(s8[2 * nt + e] - mn);     // 0 for the invalid keys
                psum += pv;
                if (grp < G) ps[warp][grp][8 * nt + 2 * j + e] = pv;
            }
        psum += __shfl_xor_sync(0xFFFFFFFFu, psum, 1);
        psum += __shfl_xor_sync(0xFFFFFFFFu, psum, 2);
        l = l * corr + psum;
        m = mn;
        if (grp < G && j == 0) cs[warp][grp] = corr;
        __syncwarp();
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float cf = cs[warp][h];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[h][e] *= cf;
        }
#pragma unroll 8
        for (int u = 0; u < nk; ++u) {
            float vf[4];
            e4m3x4_to_f32(*reinterpret_cast<const uint32_t*>(vs + u * D + 4 * lane), vf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float pw = ps[warp][h][u];
                fma2(o[h][0], o[h][1], pw, vf[0], vf[1]);
                fma2(o[h][2], o[h][3], pw, vf[2], vf[3]);
            }
        }
        __syncwarp();   // the stage is read before the next issue overwrites it
    }
    cp_wait<0>();

    // merge the warps
    if (grp < G && j == 0) {
        wm[warp][grp] = m;
        wl[warp][grp] = l;
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
        *reinterpret_cast<float4*>(&wo[warp][h][4 * lane]) = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
    __syncthreads();
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
        const int h = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, wm[w][h]);
        float lsum = 0.0f, osum = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) {
                const float f = exp2f(wm[w][h] - M);
                lsum += wl[w][h] * f;
                osum += wo[w][h][d] * f;
            }
        }
        osum *= vscale;
        const int hq = g * G + h;
        if (n_split == 1) {
            const float r = lsum > 0.0f ? osum / lsum : 0.0f;
            out[((size_t)b * Hq + hq) * D + d] = f32_to_bf16(r);
        } else {
            float* pp = part + (((size_t)b * Hq + hq) * n_split + sp) * (2 + D);
            if (d == 0) {
                pp[0] = M;
                pp[1] = lsum;
            }
            pp[2 + d] = osum;
        }
    }
}

// One CTA of D threads per (b, h): merges the n_split partial states.
__global__ void __launch_bounds__(kAttnD) k_attn_combine(const float* __restrict__ part, int n_split,
                                                         uint16_t* __restrict__ out) {
    constexpr int D = kAttnD;
    const size_t bh = blockIdx.x;
    const float* pp = part + bh * n_split * (2 + D);
    float M = -INFINITY;
    for (int i = 0; i < n_split; ++i) M = fmaxf(M, pp[(size_t)i * (2 + D)]);
    float lsum = 0.0f, osum = 0.0f;
    if (M != -INFINITY) {
        for (int i = 0; i < n_split; ++i) {
            const float* pi = pp + (size_t)i * (2 + D);
            const float f = exp2f(pi[0] - M);
            lsum += pi[1] * f;
            osum += pi[2 + threadIdx.x] * f;
        }
    }
    const float r = lsum > 0.0f ? osum / lsum : 0.0f;
    out[bh * D + threadIdx.x] = f32_to_bf16(r);
}

// Cache append for one decode step: the new token's K and V rows of every
// (sequence b, KV head g), cast with the calibrated scales, go to slot
// seq_lens[b] of the cache (skipped when that is outside [0, T)).  One warp
// per (b, g): lanes 0..15 cast K (8 values each), lanes 16..31 V.
__global__ void __launch_bounds__(32) k_kv_append(const uint16_t* __restrict__ k_new,
                                                  const uint16_t* __restrict__ v_new, const float* __restrict__ sk,
                                                  const float* __restrict__ sv, const int32_t* __restrict__ seq_lens,
                                                  uint8_t* __restrict__ kc, uint8_t* __restrict__ vc, int Hkv, int T) {
    constexpr int D = kAttnD;
    const int bg = blockIdx.x, b = bg / Hkv, lane = threadIdx.x;
    const int pos = seq_lens[b];
    if (pos < 0 || pos >= T) return;
    const bool is_v = lane >= 16;
    const int c = lane & 15;
    const float s = __ldg(is_v ? sv : sk);
    const BlockScale bs = scale_from_sr(s, __frcp_rn(s), false);
    const uint16_t* src = (is_v ? v_new : k_new) + (size_t)bg * D + 8 * c;
    uint8_t* dst = (is_v ? vc : kc) + ((size_t)bg * T + pos) * D + 8 * c;
    *reinterpret_cast<uint2*>(dst) = quant8(*reinterpret_cast<const uint4*>(src), bs);
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, const float* sk, const float* sv,
                             const int32_t* seq_lens, uint8_t* kc, uint8_t* vc, int B, int Hkv, int T,
                             cudaStream_t st) {
    if (B == 0) return cudaSuccess;
    k_kv_append<<<(unsigned)(B * Hkv), 32, 0, st>>>(static_cast<const uint16_t*>(k_new),
                                                      static_cast<const uint16_t*>(v_new), sk, sv, seq_lens, kc, vc,
                                                      Hkv, T);
    return cudaGetLastError();
}

int attn_splits(int T) { return (T + kAttnSplit - 1) / kAttnSplit; }

size_t attn_workspace_bytes(int B, int Hq, int T) {
    const int ns = attn_splits(T);
    return ns > 1 ? (size_t)B * Hq * ns * (2 + kAttnD) * sizeof(float) : 0;
}

cudaError_t launch_decode_attention(const uint8_t* q, const float* sq, const uint8_t* kc, const float* sk,
                                    const uint8_t* vc, const float* sv, const int32_t* seq_lens, int B, int Hq,
                                    int Hkv, int T, void* workspace, uint16_t* out, cudaStream_t st) {
    const int ns = attn_splits(T);
    const dim3 grid((unsigned)ns, (unsigned)Hkv, (unsigned)B);
    float* part = static_cast<float*>(workspace);
    const int G = Hq / Hkv;
    static DeviceOnce attr_done;   // dynamic shared memory above 48 KB, per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_done.test(dev)) {
        for (auto kern : {k_decode_attn<1>, k_decode_attn<2>, k_decode_attn<4>, k_decode_attn<8>}) {
            const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmemBytes);
            if (e != cudaSuccess) return e;
        }
        attr_done.set(dev);
    }
    switch (G) {
        case 1: k_decode_attn<1><<<grid, 32 * kAttnWarps, kAttnSmemBytes, st>>>(q, sq, kc, sk, vc, sv, seq_lens, Hkv, T, ns, part, out); break;
        case 2: k_decode_attn<2><<<grid, 32 * kAttnWarps, kAttnSmemBytes, st>>>(q, sq, kc, sk, vc, sv, seq_lens, Hkv, T, ns, part, out); break;
        case 4: k_decode_attn<4><<<grid, 32 * kAttnWarps, kAttnSmemBytes, st>>>(q, sq, kc, sk, vc, sv, seq_lens, Hkv, T, ns, part, out); break;
        case 8: k_decode_attn<8><<<grid, 32 * kAttnWarps, kAttnSmemBytes, st>>>(q, sq, kc, sk, vc, sv, seq_lens, Hkv, T, ns, part, out); break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || ns == 1) return e;
    k_attn_combine<<<(unsigned)(B * Hq), kAttnD, 0, st>>>(part, ns, out);
    return cudaGetLastError();
}

}  // namespace fp8bs
