// Per-tensor dynamic scaling: one scale for the whole tensor, recomputed from
// its current amax so that every value fits the FP8 range (page
// "エンドツーエンドFP8精度で実現する高スループット強化学習トレーニング",
// ai.warp-studio.com, §FP8強化学習における精度と安定性の確保).  The scale rule
// and the cast are the block quantisers' (codec.cuh) applied to one block
// that is the whole tensor.
//
// Two passes: k_amax_bf16 reduces max |x| into a device word (the bits of a
// non-negative float order like unsigned integers, so atomicMax on the bits
// is the float max), then k_quant_tensor reads it, derives the scale and
// casts.  The first pass uses ordinary loads so that a tensor smaller than
// the L2 is still there for the second.
#include <cstdint>
#include <cuda_runtime.h>

#include "codec.cuh"
#include "internal.h"

namespace fp8bs {

constexpr int kPtThreads = 256;
constexpr int kPtUnroll = 8;   // 16-byte loads in flight per thread

// The tensor as 16-byte chunks: contiguous (ldx == K: one flat range, no
// per-row work) or pitched (rows over CTAs, a row's chunks over threads).
struct ChunkWalk {
    int64_t M, cpr, ld;   // rows, chunks per row, row pitch in elements
    bool flat;
};

// Element offset of chunk c of row r (pitched walk).
__device__ __forceinline__ int64_t chunk_offset(const ChunkWalk& w, int64_t r, int64_t c) { return r * w.ld + c * 8; }

// Block-wide max of packed |bf16| pairs, one atomicMax per CTA.
__device__ __forceinline__ void cta_amax_commit(uint32_t m2, uint32_t* __restrict__ amax_bits) {
    __shared__ uint32_t red[kPtThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m2 = max_u16x2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m2;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t m = red[0];
#pragma unroll
        for (int i = 1; i < kPtThreads / 32; ++i) m = max_u16x2(m, red[i]);
        atomicMax(amax_bits, __float_as_uint(absmax_pair_to_f32(m)));
    }
}

__global__ void __launch_bounds__(kPtThreads) k_amax_bf16(const uint16_t* __restrict__ x, ChunkWalk w,
                                                          uint32_t* __restrict__ amax_bits) {
    uint32_t m2 = 0u;
    if (w.flat) {
        const int64_t total = w.M * w.cpr, step = (int64_t)gridDim.x * kPtThreads;
        for (int64_t c0 = (int64_t)blockIdx.x * kPtThreads + threadIdx.x; c0 < total; c0 += step * kPtUnroll) {
            uint4 v[kPtUnroll];
#pragma unroll
            for (int u = 0; u < kPtUnroll; ++u) {
                const int64_t c = c0 + u * step;
                v[u] = c < total ? *reinterpret_cast<const uint4*>(x + c * 8) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kPtUnroll; ++u) m2 = absmax8(m2, v[u]);
        }
    } else {
        for (int64_t r = blockIdx.x; r < w.M; r += gridDim.x) {
            for (int64_t c0 = threadIdx.x; c0 < w.cpr; c0 += kPtThreads * kPtUnroll) {
                uint4 v[kPtUnroll];
#pragma unroll
                for (int u = 0; u < kPtUnroll; ++u) {
                    const int64_t c = c0 + (int64_t)u * kPtThreads;
                    v[u] = c < w.cpr ? *reinterpret_cast<const uint4*>(x + chunk_offset(w, r, c))
                                     : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < kPtUnroll; ++u) m2 = absmax8(m2, v[u]);
            }
        }
    }
    cta_amax_commit(m2, amax_bits);
}

// The cast walk shared by both kernels: every 16-byte chunk of x through
// one cast (MUL: the product by bs.r; otherwise the per-pair test), chosen
// once by the caller.
template <bool MUL>
__device__ __forceinline__ void cast_walk(const uint16_t* __restrict__ x, const ChunkWalk& w, uint8_t* __restrict__ q,
                                          int64_t ldq, const BlockScale& bs) {
    if (w.flat) {
        const int64_t total = w.M * w.cpr, step = (int64_t)gridDim.x * kPtThreads;
        for (int64_t c0 = (int64_t)blockIdx.x * kPtThreads + threadIdx.x; c0 < total; c0 += step * kPtUnroll) {
            uint4 v[kPtUnroll];
#pragma unroll
            for (int u = 0; u < kPtUnroll; ++u) {
                const int64_t c = c0 + u * step;
                v[u] = c < total ? __ldcs(reinterpret_cast<const uint4*>(x + c * 8)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kPtUnroll; ++u) {
                const int64_t c = c0 + u * step;
                if (c < total) __stcs(reinterpret_cast<uint2*>(q + c * 8), quant8_as<MUL>(v[u], bs));
            }
        }
    } else {
        for (int64_t r = blockIdx.x; r < w.M; r += gridDim.x) {
            for (int64_t c0 = threadIdx.x; c0 < w.cpr; c0 += kPtThreads * kPtUnroll) {
                uint4 v[kPtUnroll];
#pragma unroll
                for (int u = 0; u < kPtUnroll; ++u) {
                    const int64_t c = c0 + (int64_t)u * kPtThreads;
                    v[u] = c < w.cpr ? __ldcs(reinterpret_cast<const uint4*>(x + chunk_offset(w, r, c)))
                                     : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < kPtUnroll; ++u) {
                    const int64_t c = c0 + (int64_t)u * kPtThreads;
                    if (c < w.cpr) __stcs(reinterpret_cast<uint2*>(q + r * ldq + c * 8), quant8_as<MUL>(v[u], bs));
                }
            }
        }
    }
}

// scale_amax[1] holds the amax (as written by k_amax_bf16); CTA 0 writes the
// scale to scale_amax[0].  POW2: power-of-two scale, exact multiply.  The
// flat walk needs ldq == ldx == K.
template <bool POW2>
__global__ void __launch_bounds__(kPtThreads, 4) k_quant_tensor(const uint16_t* __restrict__ x, ChunkWalk w,
                                                             uint8_t* __restrict__ q, int64_t ldq,
                                                             float* __restrict__ scale_amax) {
    const float amax = __ldcg(scale_amax + 1);
    const BlockScale bs = make_scale(amax, POW2);
    if (blockIdx.x == 0 && threadIdx.x == 0) scale_amax[0] = bs.s;
    // one scale for the tensor: the warp-uniform choice of cast made once
    const bool all_mul = POW2 || __all_sync(0xFFFFFFFFu, bs.mode == 1);
    with_cast(all_mul, [&](auto cast) { cast_walk<decltype(cast)::mul>(x, w, q, ldq, bs); });
}

// Cast under a given scale (scale[0], a positive normal fp32 in device
// memory: a calibrated KV-cache or query scale): q = e4m3(RN(x * RN(1/s))),
// values beyond +-448 s saturating.
__global__ void __launch_bounds__(kPtThreads, 4) k_cast_scale(const uint16_t* __restrict__ x, ChunkWalk w,
                                                             uint8_t* __restrict__ q, int64_t ldq,
                                                             const float* __restrict__ scale) {
    const float sc = __ldg(scale);
    const BlockScale bs = scale_from_sr(sc, __frcp_rn(sc), false);
    const bool all_mul = __all_sync(0xFFFFFFFFu, bs.mode == 1);   // one scale for the tensor
    with_cast(all_mul, [&](auto cast) { cast_walk<decltype(cast)::mul>(x, w, q, ldq, bs); });
}

cudaError_t launch_cast_with_scale(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                                   const float* scale, int sm_count, cudaStream_t st) {
    if (M == 0) return cudaSuccess;
    ChunkWalk w{M, K / 8, ldx, ldx == K && ldq == K};
    const int64_t chunks = M * w.cpr;
    int64_t grid = (int64_t)sm_count * 4;
    const int64_t need = w.flat ? (chunks + (int64_t)kPtThreads * kPtUnroll - 1) / ((int64_t)kPtThreads * kPtUnroll) : M;
    if (need < grid) grid = need < 1 ? 1 : need;
    k_cast_scale<<<(unsigned)grid, kPtThreads, 0, st>>>(static_cast<const uint16_t*>(x), w, q, ldq, scale);
    return cudaGetLastError();
}

cudaError_t launch_quant_per_tensor(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                                    float* scale_amax, bool pow2, int sm_count, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(scale_amax + 1, 0, sizeof(float), st);
    if (e != cudaSuccess) return e;
    if (M == 0) return cudaSuccess;
    ChunkWalk w{M, K / 8, ldx, ldx == K && ldq == K};
    const int64_t chunks = M * w.cpr;
    // 4 CTAs per SM, fewer if the tensor is small (each thread keeps
    // kPtUnroll loads in flight); the pitched walk takes a CTA per row.
    int64_t grid = (int64_t)sm_count * 4;
    const int64_t need = w.flat ? (chunks + (int64_t)kPtThreads * kPtUnroll - 1) / ((int64_t)kPtThreads * kPtUnroll) : M;
    if (need < grid) grid = need < 1 ? 1 : need;
    const uint16_t* xp = static_cast<const uint16_t*>(x);
    k_amax_bf16<<<(unsigned)grid, kPtThreads, 0, st>>>(xp, w, reinterpret_cast<uint32_t*>(scale_amax + 1));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (pow2)
        k_quant_tensor<true><<<(unsigned)grid, kPtThreads, 0, st>>>(xp, w, q, ldq, scale_amax);
    else
        k_quant_tensor<false><<<(unsigned)grid, kPtThreads, 0, st>>>(xp, w, q, ldq, scale_amax);
    return cudaGetLastError();
}

}  // namespace fp8bs
