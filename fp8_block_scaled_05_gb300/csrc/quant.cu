// Block quantisers: bf16 -> FP8 E4M3 codes + fp32 scales.
//
// 1x128 activation blocks and 128x128 weight blocks, scale from the block's
// own amax (page "NVIDIA NeMo RL достигает ускорения на 48% благодаря
// сквозному обучению с точностью FP8", greentreeone.com, §Технический
// прорыв); the weight quantiser runs after every optimizer step because the
// policy's weights change each step (same page, §Реальные прирост
// производительности).
//
// Both kernels are HBM streams (2 bytes read + 1 byte written per element):
// every thread issues all of its 16-byte loads before using any of them, the
// amax is reduced with shuffles, and the cast is fused into the same pass over
// registers, so each input byte is read once.
#include <cstdint>
#include <cuda_runtime.h>

#include "codec.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {

// ---------------------------------------------------------------------------
// 1x128 activations.  CTA tile: 16 rows x 8 K-blocks.  Warp w owns rows
// 2w, 2w+1; a warp-wide 512-byte load covers two adjacent K-blocks of one
// row, half-warp h handling K-block 2p+h.  A warp therefore holds 16 blocks
// (8 "items" i = 4r+p per half).  Their amax values are reduced over each
// half with one plain exchange and a butterfly reduce-scatter (15 shuffles
// instead of 32), after which lane 16h+(i mod 8) holds the amax of item i of
// half h and computes that one block's scale; the other lanes fetch (s, 1/s)
// with two shuffles per item.  Scales are gathered in shared memory and
// written K-block-major (16 consecutive rows per store).
// ---------------------------------------------------------------------------
constexpr int kActRowsPerWarp = 2;
constexpr int kActRows = 8 * kActRowsPerWarp;
constexpr int kActKB = 8;
constexpr int kActPairs = kActKB / 2;
constexpr int kActItems = kActRowsPerWarp * kActPairs;   // blocks per half-warp
static_assert(kActItems <= 16 && (kActItems & (kActItems - 1)) == 0, "items per half-warp");

// POW2: power-of-two scales (the exponent instead of the two divisions).
// One CTA tile (bx, by) of 16 rows x 8 K-blocks; 256 threads.
template <bool POW2>
__device__ __forceinline__ void act_tile_1x128(const uint16_t* __restrict__ x, int64_t M, int64_t KB, int64_t ldx,
                                               uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ s,
                                               int64_t lds, uint8_t* __restrict__ s8, int64_t bx, int64_t by) {
    __shared__ float s_tile[kActKB][kActRows];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, half = lane >> 4, l16 = lane & 15;
    const int64_t m0 = bx * kActRows;
    const int64_t kb0 = by * kActKB;

    uint4 v[kActItems];
#pragma unroll
    for (int i = 0; i < kActItems; ++i) {
        const int r = i / kActPairs, p = i % kActPairs;
        const int64_t m = m0 + warp * kActRowsPerWarp + r;
        const int64_t kb = kb0 + 2 * p + half;
        if (m < M && kb < KB)
            v[i] = __ldcs(reinterpret_cast<const uint4*>(x + m * ldx + kb * 128 + l16 * 8));
        else
            v[i] = make_uint4(0, 0, 0, 0);
    }

    uint32_t a[kActItems];
#pragma unroll
    for (int i = 0; i < kActItems; ++i) a[i] = absmax8(0u, v[i]);
    // Plain exchange over the lane bits above the item count...
#pragma unroll
    for (int o = 8; o >= kActItems; o >>= 1)
#pragma unroll
        for (int j = 0; j < kActItems; ++j) a[j] = max_u16x2(a[j], __shfl_xor_sync(0xFFFFFFFFu, a[j], o));
    // ...then a butterfly reduce-scatter: after the step with offset o, a lane
    // keeps the items whose index bit o matches its own lane bit o.
#pragma unroll
    for (int o = kActItems / 2; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < o; ++j) {
            const uint32_t send = upper ? a[j] : a[j + o];
            const uint32_t keep = upper ? a[j + o] : a[j];
            a[j] = max_u16x2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, o));
        }
    }
    // this lane's block: item (l16 mod kActItems) of half `half`
    const BlockScale own = make_scale(absmax_pair_to_f32(a[0]), POW2);
    // every block of the warp is some lane's own: one vote picks the cast
    const bool all_mul = POW2 || __all_sync(0xFFFFFFFFu, own.mode == 1);
    if (l16 < kActItems) {
        const int r = l16 / kActPairs, p = l16 % kActPairs;
        const int rl = warp * kActRowsPerWarp + r;
        if (m0 + rl < M && kb0 + 2 * p + half < KB) s_tile[2 * p + half][rl] = own.s;
    }
    with_cast(all_mul, [&](auto cast) {
#pragma unroll
        for (int i = 0; i < kActItems; ++i) {
            const int r = i / kActPairs, p = i % kActPairs;
            const int src = (lane & 16) | i;
            const float si = __shfl_sync(0xFFFFFFFFu, own.s, src);
            const float ri = __shfl_sync(0xFFFFFFFFu, own.r, src);
            const int64_t m = m0 + warp * kActRowsPerWarp + r;
            const int64_t kb = kb0 + 2 * p + half;
            if (m < M && kb < KB)
                __stcs(reinterpret_cast<uint2*>(q + m * ldq + kb * 128 + l16 * 8),
                       quant8_as<decltype(cast)::mul>(v[i], scale_from_sr(si, ri, false)));
        }
    });
    __syncthreads();
    if (threadIdx.x < kActKB * kActRows) {
        const int kbl = threadIdx.x / kActRows, rl = threadIdx.x % kActRows;
        const int64_t kb = kb0 + kbl, m = m0 + rl;
        if (kb < KB && m < M) {
            // s8: UE8M0 bytes (power-of-two scales): the fp32 exponent field,
            // which is also right for 2^-127 (stored as a subnormal)
            if (s8 != nullptr)
                s8[kb * lds + m] = (uint8_t)(__float_as_uint(s_tile[kbl][rl]) >> 23);
            else
                s[kb * lds + m] = s_tile[kbl][rl];
        }
    }
}

template <bool POW2>
__global__ void __launch_bounds__(256, 4) k_quant_act_1x128(const uint16_t* __restrict__ x, int64_t M, int64_t KB,
                                                            int64_t ldx, uint8_t* __restrict__ q, int64_t ldq,
                                                            float* __restrict__ s, int64_t lds,
                                                            uint8_t* __restrict__ s8) {
    griddep_wait();                  // x may come from the previous kernel in the stream
    griddep_launch_dependents();     // the GEMM that follows may start its prologue
    act_tile_1x128<POW2>(x, M, KB, ldx, q, ldq, s, lds, s8, blockIdx.x, blockIdx.y);
}

cudaError_t launch_quant_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                                   float* s, int64_t lds, bool pow2, cudaStream_t st, uint8_t* s8) {
    if (M == 0) return cudaSuccess;
    const int64_t KB = K / 128;
    dim3 grid((unsigned)((M + kActRows - 1) / kActRows), (unsigned)((KB + kActKB - 1) / kActKB));
    auto kern = pow2 ? k_quant_act_1x128<true> : k_quant_act_1x128<false>;
    if (pdl_for_tokens(M))   // a decode step: overlap with the kernels around it
        return launch_pdl(kern, grid, dim3(256), 0, st, static_cast<const uint16_t*>(x), M, KB, ldx, q, ldq, s, lds,
                          s8);
    kern<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(x), M, KB, ldx, q, ldq, s, lds, s8);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// 128x128 weights.  One CTA per tile, 256 threads; warp w owns rows
// 16w..16w+15, one warp-wide load covering two rows (half-warp each).  Each
// lane keeps its 64 values in registers across the CTA-wide amax reduction.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void weight_tile_128x128(const uint16_t* __restrict__ w, int64_t KB, int64_t ldw,
                                                    uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ s,
                                                    bool pow2, uint8_t* __restrict__ s8, int64_t kb, int64_t nb) {
    __shared__ float s_red[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, half = lane >> 4, l16 = lane & 15;
    const int64_t row0 = nb * 128 + warp * 16 + half;
    const int64_t col = kb * 128 + l16 * 8;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = __ldcs(reinterpret_cast<const uint4*>(w + (row0 + 2 * i) * ldw + col));
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) m2 = absmax8(m2, v[i]);
    float amax = absmax_pair_to_f32(m2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (lane == 0) s_red[warp] = amax;
    __syncthreads();
    amax = s_red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, s_red[i]);
    const BlockScale bs = make_scale(amax, pow2);
    if (bs.mode == 1) {   // one scale for the tile: a uniform choice of cast
#pragma unroll
        for (int i = 0; i < 8; ++i)
            __stcs(reinterpret_cast<uint2*>(q + (row0 + 2 * i) * ldq + col), quant8_mul(v[i], bs.r));
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            __stcs(reinterpret_cast<uint2*>(q + (row0 + 2 * i) * ldq + col), quant8(v[i], bs));
    }
    if (threadIdx.x == 0) {
        if (s8 != nullptr)
            s8[nb * KB + kb] = (uint8_t)(__float_as_uint(bs.s) >> 23);   // UE8M0 byte of a power of two
        else
            s[nb * KB + kb] = bs.s;
    }
}

__global__ void __launch_bounds__(256) k_quant_w_128x128(const uint16_t* __restrict__ w, int64_t KB, int64_t ldw,
                                                         uint8_t* __restrict__ q, int64_t ldq,
                                                         float* __restrict__ s, int pow2, uint8_t* __restrict__ s8) {
    weight_tile_128x128(w, KB, ldw, q, ldq, s, pow2 != 0, s8, blockIdx.x, blockIdx.y);
}

// ---------------------------------------------------------------------------
// A layer's activations (1x128) and weights (128x128) in one launch: CTAs
// 0 .. NB*KB-1 take the weight tiles (kb fastest), the rest the activation
// tiles (row tiles fastest), so neither quantiser's ramp and tail is paid
// on its own.  Same tiles, same code as the two kernels above.
// ---------------------------------------------------------------------------
template <bool POW2>
__global__ void __launch_bounds__(256, 4) k_quant_act_weight(const uint16_t* __restrict__ x, int64_t M, int64_t ldx,
                                                             uint8_t* __restrict__ qa, int64_t ldqa,
                                                             float* __restrict__ sa, int64_t ldsa,
                                                             const uint16_t* __restrict__ w, int64_t NB, int64_t ldw,
                                                             uint8_t* __restrict__ qw, int64_t ldqw,
                                                             float* __restrict__ sw, int64_t KB, int64_t act_rows) {
    const int64_t b = blockIdx.x, wt = NB * KB;
    if (b < wt) {
        weight_tile_128x128(w, KB, ldw, qw, ldqw, sw, POW2, nullptr, b % KB, b / KB);
    } else {
        const int64_t a = b - wt;
        act_tile_1x128<POW2>(x, M, KB, ldx, qa, ldqa, sa, ldsa, nullptr, a % act_rows, a / act_rows);
    }
}

cudaError_t launch_quant_act_weight(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* qa, int64_t ldqa,
                                    float* sa, int64_t ldsa, const void* w, int64_t N, int64_t ldw, uint8_t* qw,
                                    int64_t ldqw, float* sw, bool pow2, cudaStream_t st) {
    const int64_t KB = K / 128, NB = N / 128;
    const int64_t act_rows = (M + kActRows - 1) / kActRows, act_kbs = (KB + kActKB - 1) / kActKB;
    const int64_t blocks = NB * KB + act_rows * act_kbs;
    auto kern = pow2 ? k_quant_act_weight<true> : k_quant_act_weight<false>;
    kern<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint16_t*>(x), M, ldx, qa, ldqa, sa, ldsa,
                                          static_cast<const uint16_t*>(w), NB, ldw, qw, ldqw, sw, KB, act_rows);
    return cudaGetLastError();
}

cudaError_t launch_quant_weight_128x128(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                                        int64_t ldq, float* s, bool pow2, cudaStream_t st, uint8_t* s8) {
    const int64_t KB = K / 128, NB = N / 128;
    dim3 grid((unsigned)KB, (unsigned)NB);
    k_quant_w_128x128<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(w), KB, ldw, q, ldq, s, pow2 ? 1 : 0, s8);
    return cudaGetLastError();
}

}  // namespace fp8bs
