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
//   scores  lanes over keys (32 keys per warp block), each lane the full
//           128-dim dot products of its key with the G dequantised queries
//           (shared memory, the scale product and log2(e)/sqrt(D) folded in);
//   softmax online per warp (max and sum by shuffles, exp2);
//   P V     lanes over dims: lane l adds p_t v[t, 4l .. 4l+3] for the
//           block's 32 keys (a 128-byte coalesced row per key);
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

// part: [B][Hq][n_split][2 + D] floats (m in log2 units, l, o unnormalised)
// when n_split > 1; otherwise the output is written directly.
template <int G>
__global__ void __launch_bounds__(32 * kAttnWarps) k_decode_attn(
    const uint8_t* __restrict__ q, const float* __restrict__ sq, const uint8_t* __restrict__ kc,
    const float* __restrict__ sk, const uint8_t* __restrict__ vc, const float* __restrict__ sv,
    const int32_t* __restrict__ seq_lens, int Hkv, int T, int n_split, float* __restrict__ part,
    uint16_t* __restrict__ out) {
    constexpr int D = kAttnD;
    __shared__ __align__(16) float qs[G][D];
    __shared__ float ps[kAttnWarps][G][32];
    __shared__ float wm[kAttnWarps][G], wl[kAttnWarps][G];
    __shared__ __align__(16) float wo[kAttnWarps][G][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int Hq = Hkv * G;
    const int L = min(max(seq_lens[b], 0), T);
    const int t0 = sp * kAttnSplit, t1 = min(t0 + kAttnSplit, L);

    // queries of the group, dequantised, with sq * sk * log2(e) / sqrt(D)
    const float c = sq[0] * sk[0] * (1.4426950408889634f * 0.08838834764831845f);
    for (int i = threadIdx.x; i < G * D / 4; i += blockDim.x) {
        const int h = i / (D / 4), d4 = i % (D / 4);
        const uint32_t w = *reinterpret_cast<const uint32_t*>(q + ((size_t)b * Hq + g * G + h) * D + 4 * d4);
        float f[4];
        e4m3x4_to_f32(w, f);
        *reinterpret_cast<float4*>(&qs[h][4 * d4]) = make_float4(f[0] * c, f[1] * c, f[2] * c, f[3] * c);
    }
    __syncthreads();

    const float vscale = sv[0];
    const size_t head_base = ((size_t)b * Hkv + g) * (size_t)T * D;
    float m[G], l[G], o[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) o[h][j] = 0.0f;
    }
    for (int tb = t0 + 32 * warp; tb < t1; tb += 32 * kAttnWarps) {
        const int t = tb + lane;
        const bool valid = t < t1;
        float s[G];
#pragma unroll
        for (int h = 0; h < G; ++h) s[h] = 0.0f;
        if (valid) {
            // the key's whole 128-byte row first, then the arithmetic
            const uint4* krow = reinterpret_cast<const uint4*>(kc + head_base + (size_t)t * D);
            uint4 kr[D / 16];
#pragma unroll
            for (int ch = 0; ch < D / 16; ++ch) kr[ch] = __ldg(krow + ch);
#pragma unroll
            for (int ch = 0; ch < D / 16; ++ch) {
                const uint32_t w[4] = {kr[ch].x, kr[ch].y, kr[ch].z, kr[ch].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float kf[4];
                    e4m3x4_to_f32(w[e], kf);
                    const int d = 16 * ch + 4 * e;
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float4 qv = *reinterpret_cast<const float4*>(&qs[h][d]);
                        s[h] = fmaf(qv.x, kf[0], s[h]);
                        s[h] = fmaf(qv.y, kf[1], s[h]);
                        s[h] = fmaf(qv.z, kf[2], s[h]);
                        s[h] = fmaf(qv.w, kf[3], s[h]);
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float bm = warp_max(valid ? s[h] : -INFINITY);   // lane 0's key is valid: bm is finite
            const float mn = fmaxf(m[h], bm);
            const float corr = exp2f(m[h] - mn);                  // 0 while m[h] is -inf
            const float p = valid ? exp2f(s[h] - mn) : 0.0f;
            l[h] = l[h] * corr + warp_sum(p);
            m[h] = mn;
#pragma unroll
            for (int j = 0; j < 4; ++j) o[h][j] *= corr;
            ps[warp][h][lane] = p;
        }
        __syncwarp();
        const int nk = min(32, t1 - tb);   // warp-uniform
        const uint32_t* vrow = reinterpret_cast<const uint32_t*>(vc + head_base + (size_t)tb * D) + lane;
        for (int j0 = 0; j0 < nk; j0 += 8) {
            uint32_t vw[8];   // 8 value rows in flight
#pragma unroll
            for (int u = 0; u < 8; ++u) vw[u] = j0 + u < nk ? __ldg(vrow + (size_t)(j0 + u) * (D / 4)) : 0u;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (j0 + u < nk) {
                    float vf[4];
                    e4m3x4_to_f32(vw[u], vf);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float p = ps[warp][h][j0 + u];
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[h][e] = fmaf(p, vf[e], o[h][e]);
                    }
                }
            }
        }
        __syncwarp();
    }

    // merge the warps
#pragma unroll
    for (int h = 0; h < G; ++h) {
        if (lane == 0) {
            wm[warp][h] = m[h];
            wl[warp][h] = l[h];
        }
        *reinterpret_cast<float4*>(&wo[warp][h][4 * lane]) = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
    }
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
    switch (G) {
        case 1: k_decode_attn<1><<<grid, 32 * kAttnWarps, 0, st>>>(q, sq, kc, sk, vc, sv, seq_lens, Hkv, T, ns, part, out); break;
        case 2: k_decode_attn<2><<<grid, 32 * kAttnWarps, 0, st>>>(q, sq, kc, sk, vc, sv, seq_lens, Hkv, T, ns, part, out); break;
        case 4: k_decode_attn<4><<<grid, 32 * kAttnWarps, 0, st>>>(q, sq, kc, sk, vc, sv, seq_lens, Hkv, T, ns, part, out); break;
        case 8: k_decode_attn<8><<<grid, 32 * kAttnWarps, 0, st>>>(q, sq, kc, sk, vc, sv, seq_lens, Hkv, T, ns, part, out); break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || ns == 1) return e;
    k_attn_combine<<<(unsigned)(B * Hq), kAttnD, 0, st>>>(part, ns, out);
    return cudaGetLastError();
}

}  // namespace fp8bs
