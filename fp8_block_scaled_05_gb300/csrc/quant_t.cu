// Transposing block quantisers: the operands of the training-side GEMMs of a
// linear layer y = x W^T.
//
// The pages run FP8 through training as well as generation (page "NVIDIA
// NeMo RL достигает ускорения на 48% благодаря сквозному обучению с
// точностью FP8", greentreeone.com, §Технический прорыв; ai.warp-studio.com
// end-to-end FP8 RL article, opening section: activations and gradients
// too).  With every operand blocked along the dimension its GEMM reduces:
//   dgrad  dX = dY W     needs W^T with W's own 128x128 blocks
//                        (k_quant_w_128x128_t: W^T codes, optionally W's too);
//   wgrad  dW = dY^T X   needs dY and X in 128x1 blocks (128 tokens of one
//                        column), stored transposed so that the tokens are
//                        contiguous (k_quant_act_128x1; optionally also the
//                        1x128 codes that the forward GEMM or dgrad takes).
// One pass over the bf16 input writes both layouts, so an operand that two
// GEMMs need is read from HBM once.
//
// A CTA takes a 128 x 128 tile with 256 threads.  Thread t holds tile rows
// 8 rg .. 8 rg + 7 (rg = t / 16) and columns 8 cg .. 8 cg + 7 (cg = t % 16),
// one 16-byte load per row (a half-warp reads 256 contiguous bytes of one
// row).  Codes of a tile column are formed from the thread's 8 rows and
// written as one 8-byte piece into a 16 KB shared-memory tile: row 8 cg + j
// (the tile column), 16-byte chunk (rg / 2) ^ (cg % 8) -- the XOR keeps the
// 16 threads of a half-warp on 8 distinct chunks -- then each warp stores 16
// of its rows with 16-byte stores, 128 contiguous bytes per output row.
#include <cstdint>
#include <cuda_runtime.h>

#include "codec.cuh"
#include "internal.h"
#include "sched.cuh"

namespace fp8bs {

constexpr int kTT = 128;   // tile edge (one block edge)

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Element (row i, column j) of the thread's 8 x 8 sub-tile as fp32.
__device__ __forceinline__ float elem(const uint4 (&v)[8], int i, int j) {
    const uint32_t w = word_of(v[i], j >> 1);
    return (j & 1) ? bf16hi_to_f32(w) : bf16lo_to_f32(w);
}

// The column codes with one cast throughout: MUL, the product by each
// column's factor r; otherwise the per-pair choice of quant_pair.
template <bool MUL, typename ScaleOf>
__device__ __forceinline__ void col_codes_to_smem_as(const uint4 (&v)[8], int rg, int cg, uint8_t *tcodes,
                                                     ScaleOf scale_of) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const BlockScale bs = scale_of(j);
        uint32_t part[2] = {0u, 0u};
#pragma unroll
        for (int p = 0; p < 4; ++p) {   // rows 2p (low byte) and 2p + 1
            uint32_t pair;
            if constexpr (MUL) {
                float qa, qb;
                mul2(elem(v, 2 * p, j), elem(v, 2 * p + 1, j), bs.r, qa, qb);
                pair = e4m3x2(qa, qb);
            } else {
                pair = quant_pair(elem(v, 2 * p, j), elem(v, 2 * p + 1, j), bs);
            }
            part[p >> 1] |= pair << (16 * (p & 1));
        }
        const int R = 8 * cg + j;
        *reinterpret_cast<uint2 *>(tcodes + R * kTT + ((((rg >> 1) ^ (cg & 7))) << 4) + ((rg & 1) << 3)) =
            make_uint2(part[0], part[1]);
    }
}

// Codes of the thread's 8 columns (8 rows each) into the shared tile;
// scale_of(j) gives column j's BlockScale.  The product cast for the whole
// warp unless one of its columns divides (POW2: power-of-two scales, always
// an exact multiply); the choice is made once, outside the loops.
template <bool POW2, typename ScaleOf>
__device__ __forceinline__ void col_codes_to_smem(const uint4 (&v)[8], int rg, int cg, uint8_t *tcodes,
                                                  ScaleOf scale_of) {
    bool all_mul = POW2;
    if constexpr (!POW2) {
        bool mine = true;
#pragma unroll
        for (int j = 0; j < 8; ++j) mine = mine && scale_of(j).mode == 1;
        all_mul = __all_sync(0xFFFFFFFFu, mine);
    }
    if (all_mul)
        col_codes_to_smem_as<true>(v, rg, cg, tcodes, scale_of);
    else
        col_codes_to_smem_as<false>(v, rg, cg, tcodes, scale_of);
}

// 4 x 4 byte transpose: words a, b, c, d are rows (byte 0 = column 0); word
// j of the result holds column j (byte 0 from a).
__device__ __forceinline__ void transpose4x4_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                                   uint32_t (&o)[4]) {
    const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(a, b, 0x7362);
    const uint32_t t2 = __byte_perm(c, d, 0x5140), t3 = __byte_perm(c, d, 0x7362);
    o[0] = __byte_perm(t0, t2, 0x5410);
    o[1] = __byte_perm(t0, t2, 0x7632);
    o[2] = __byte_perm(t1, t3, 0x5410);
    o[3] = __byte_perm(t1, t3, 0x7632);
}

// The thread's 8 x 8 codes, given as rows (rc[i]: row i, 8 columns), into
// the shared tile column by column -- the same placement as
// col_codes_to_smem, with the codes transposed in registers instead of
// computed again.
__device__ __forceinline__ void row_codes_to_smem_transposed(const uint2 (&rc)[8], int rg, int cg,
                                                             uint8_t *tcodes) {
    uint32_t lo03[4], hi03[4], lo47[4], hi47[4];
    transpose4x4_bytes(rc[0].x, rc[1].x, rc[2].x, rc[3].x, lo03);   // columns 0..3, rows 0..3
    transpose4x4_bytes(rc[4].x, rc[5].x, rc[6].x, rc[7].x, hi03);   // columns 0..3, rows 4..7
    transpose4x4_bytes(rc[0].y, rc[1].y, rc[2].y, rc[3].y, lo47);   // columns 4..7, rows 0..3
    transpose4x4_bytes(rc[4].y, rc[5].y, rc[6].y, rc[7].y, hi47);   // columns 4..7, rows 4..7
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int R = 8 * cg + j;
        const uint2 val = j < 4 ? make_uint2(lo03[j], hi03[j]) : make_uint2(lo47[j - 4], hi47[j - 4]);
        *reinterpret_cast<uint2 *>(tcodes + R * kTT + ((((rg >> 1) ^ (cg & 7))) << 4) + ((rg & 1) << 3)) = val;
    }
}

// The shared tile (after a barrier) to out[(row0 + R) * ldo + col0 + ...]:
// warp w stores tile rows 16 w .. 16 w + 15, four rows per instruction.
__device__ __forceinline__ void store_transposed(const uint8_t *tcodes, uint8_t *out, int64_t ldo, int64_t row0,
                                                 int64_t col0, int warp, int lane) {
    const int lc = lane & 7;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int R = 16 * warp + 4 * u + (lane >> 3);
        const uint4 val = *reinterpret_cast<const uint4 *>(tcodes + R * kTT + ((lc ^ ((R >> 3) & 7)) << 4));
        __stcs(reinterpret_cast<uint4 *>(out + (row0 + R) * ldo + col0 + 16 * lc), val);
    }
}

// ---------------------------------------------------------------------------
// 128x1 activation blocks (tile (kb, mb) = blockIdx (x, y)), transposed
// codes qt[k][m] and scales st[mb * ldst + k]; with ROWWISE also the 1x128
// codes q[m][k] and scales s[kb * lds + m] of the same tile.
// ---------------------------------------------------------------------------
//
// GROUPED (mixture-of-experts weight gradients): x holds the tokens of G
// experts sorted by expert, expert g on rows offsets[g] .. offsets[g+1]-1
// (device array).  Each expert's tokens are blocked on their own, the last
// block of an expert padded with zero rows, and the blocks are written to
// consecutive token slots: blockIdx.y = b is the b-th padded block overall,
// expert g's blocks are b = P_g .. P_{g+1}-1 with P_g = sum_{g' < g}
// ceil(M_g' / 128), and its codes go to qt columns 128 b .. 128 b + 127 and
// its scales to st[b * ldst + k].  Blocks past P_G do nothing.
template <bool ROWWISE, bool POW2, bool GROUPED = false>
__global__ void __launch_bounds__(256, ROWWISE ? 3 : 4) k_quant_act_128x1(const uint16_t *__restrict__ x, int64_t ldx,
                                                         uint8_t *__restrict__ qt, int64_t ldqt,
                                                         float *__restrict__ st, int64_t ldst,
                                                         uint8_t *__restrict__ q, int64_t ldq,
                                                         float *__restrict__ s, int64_t lds, int64_t M,
                                                         const int32_t *__restrict__ offsets = nullptr,
                                                         int G = 0) {
    __shared__ __align__(16) uint8_t tcodes[kTT * kTT];
    __shared__ __align__(16) uint32_t colpart[8][16][4];   // per warp: packed |bf16| maxima of column pairs
    __shared__ float2 colscale[kTT];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cg = lane & 15, rg = 2 * warp + (lane >> 4);
    const int64_t k0 = (int64_t)blockIdx.x * kTT;
    // m0: first input row of the block; rows at or past M are zeros; the
    // transposed codes go to qt columns mo .. mo + 127
    int64_t m0 = (int64_t)blockIdx.y * kTT, mo = m0;
    if constexpr (GROUPED) {
        __shared__ int32_t cum[kMaxGroupedQuantExperts + 1];
        __shared__ int32_t total;
        if (warp == 0) {
            const int t = build_group_table<kTT>(offsets, G, (int)M, 1, cum);
            if (lane == 0) total = t;
        }
        __syncthreads();
        const int b = (int)blockIdx.y;
        if (b >= total) return;   // past the last expert's blocks (the grid is an upper bound)
        int lo = 0, hi = G;       // largest g with cum[g] <= b
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cum[mid] <= b) lo = mid; else hi = mid;
        }
        int rlo, rhi;
        group_rows(offsets, lo, (int)M, rlo, rhi);
        m0 = rlo + (int64_t)(b - cum[lo]) * kTT;
        M = rhi;                  // the expert's rows end here
        mo = (int64_t)b * kTT;
    }

    // rows past M (a ragged last token block) are zeros: they change no
    // block's amax and their transposed codes are zero
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t m = m0 + 8 * rg + i;
        v[i] = m < M ? __ldcs(reinterpret_cast<const uint4 *>(x + m * ldx + k0 + 8 * cg)) : make_uint4(0, 0, 0, 0);
    }

    // column maxima over the thread's rows, then over the warp's two halves
    uint32_t cm[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        cm[0] = absmax_bf16x2(cm[0], v[i].x);
        cm[1] = absmax_bf16x2(cm[1], v[i].y);
        cm[2] = absmax_bf16x2(cm[2], v[i].z);
        cm[3] = absmax_bf16x2(cm[3], v[i].w);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) cm[j] = max_u16x2(cm[j], __shfl_xor_sync(0xFFFFFFFFu, cm[j], 16));
    if (lane < 16) *reinterpret_cast<uint4 *>(&colpart[warp][cg][0]) = make_uint4(cm[0], cm[1], cm[2], cm[3]);

    if constexpr (ROWWISE) {
        // 1x128 blocks: row 8 rg + i spans the 16 lanes of this half-warp.  A
        // plain exchange over lane bit 3, then a butterfly reduce-scatter over
        // bits 2..0 leaves the amax of row item (lane % 8) in a[0].
        uint32_t a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = absmax8(0u, v[i]);
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = max_u16x2(a[j], __shfl_xor_sync(0xFFFFFFFFu, a[j], 8));
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int j = 0; j < o; ++j) {
                const uint32_t send = upper ? a[j] : a[j + o];
                const uint32_t keep = upper ? a[j + o] : a[j];
                a[j] = max_u16x2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, o));
            }
        }
        const BlockScale own = make_scale(absmax_pair_to_f32(a[0]), POW2);
        if (cg < 8 && m0 + 8 * rg + cg < M) s[(size_t)blockIdx.x * lds + m0 + 8 * rg + cg] = own.s;
        const bool all_mul = POW2 || __all_sync(0xFFFFFFFFu, own.mode == 1);
        with_cast(all_mul, [&](auto cast) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int src = (lane & 16) | i;
                const float si = __shfl_sync(0xFFFFFFFFu, own.s, src);
                const float ri = __shfl_sync(0xFFFFFFFFu, own.r, src);
                if (m0 + 8 * rg + i < M)
                    __stcs(reinterpret_cast<uint2 *>(q + (m0 + 8 * rg + i) * ldq + k0 + 8 * cg),
                           quant8_as<decltype(cast)::mul>(v[i], scale_from_sr(si, ri, false)));
            }
        });
    }
    __syncthreads();
    if (threadIdx.x < kTT) {
        const int c = threadIdx.x;
        uint32_t m2 = 0u;
#pragma unroll
        for (int w = 0; w < 8; ++w) m2 = max_u16x2(m2, colpart[w][c >> 3][(c & 7) >> 1]);
        const uint32_t bits = (c & 1) ? (m2 >> 16) : (m2 & 0xFFFFu);
        const BlockScale bs = make_scale(__uint_as_float(bits << 16), POW2);
        colscale[c] = make_float2(bs.s, bs.r);
        st[(size_t)blockIdx.y * ldst + k0 + c] = bs.s;
    }
    __syncthreads();
    col_codes_to_smem<POW2>(v, rg, cg, tcodes, [&](int j) {
        const float2 sr = colscale[8 * cg + j];
        return scale_from_sr(sr.x, sr.y, POW2);
    });
    __syncthreads();
    store_transposed(tcodes, qt, ldqt, k0, mo, warp, lane);
}

// ---------------------------------------------------------------------------
// 128x128 weight blocks (tile (kb, nb) = blockIdx (x, y)): W^T codes
// qt[k][n] and scales st[kb * NB + nb]; with q != nullptr also W's codes
// q[n][k] and scales s[nb * KB + kb].
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_quant_w_128x128_t(const uint16_t *__restrict__ w, int64_t ldw, int64_t KB,
                                                           int64_t NB, uint8_t *__restrict__ q, int64_t ldq,
                                                           float *__restrict__ s, uint8_t *__restrict__ qt,
                                                           int64_t ldqt, float *__restrict__ st, int pow2) {
    __shared__ __align__(16) uint8_t tcodes[kTT * kTT];
    __shared__ float red[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cg = lane & 15, rg = 2 * warp + (lane >> 4);
    const int64_t k0 = (int64_t)blockIdx.x * kTT, n0 = (int64_t)blockIdx.y * kTT;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = __ldcs(reinterpret_cast<const uint4 *>(w + (n0 + 8 * rg + i) * ldw + k0 + 8 * cg));
    uint32_t m2 = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) m2 = absmax8(m2, v[i]);
    float amax = absmax_pair_to_f32(m2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const BlockScale bs = make_scale(amax, pow2 != 0);

    // One scale for the whole tile: W's codes and W^T's are the same bytes,
    // computed once and transposed in registers.
    uint2 rc[8];
    if (bs.mode == 1) {   // one scale for the tile: a uniform choice of cast
#pragma unroll
        for (int i = 0; i < 8; ++i) rc[i] = quant8_mul(v[i], bs.r);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) rc[i] = quant8(v[i], bs);
    }
    if (q != nullptr) {
#pragma unroll
        for (int i = 0; i < 8; ++i) __stcs(reinterpret_cast<uint2 *>(q + (n0 + 8 * rg + i) * ldq + k0 + 8 * cg), rc[i]);
    }
    row_codes_to_smem_transposed(rc, rg, cg, tcodes);
    __syncthreads();
    store_transposed(tcodes, qt, ldqt, k0, n0, warp, lane);
    if (threadIdx.x == 0) {
        st[(size_t)blockIdx.x * NB + blockIdx.y] = bs.s;
        if (q != nullptr) s[(size_t)blockIdx.y * KB + blockIdx.x] = bs.s;
    }
}

cudaError_t launch_quant_act_128x1(const void *x, int64_t M, int64_t K, int64_t ldx, uint8_t *qt, int64_t ldqt,
                                   float *st, int64_t ldst, uint8_t *q, int64_t ldq, float *s, int64_t lds,
                                   bool pow2, cudaStream_t stream) {
    if (M == 0) return cudaSuccess;
    const dim3 grid((unsigned)(K / kTT), (unsigned)((M + kTT - 1) / kTT));   // last token block padded with zeros
    const uint16_t *xp = static_cast<const uint16_t *>(x);
    auto kern = q != nullptr ? (pow2 ? k_quant_act_128x1<true, true> : k_quant_act_128x1<true, false>)
                             : (pow2 ? k_quant_act_128x1<false, true> : k_quant_act_128x1<false, false>);
    kern<<<grid, 256, 0, stream>>>(xp, ldx, qt, ldqt, st, ldst, q, ldq, s, lds, M, nullptr, 0);
    return cudaGetLastError();
}

cudaError_t launch_quant_act_128x1_grouped(const void *x, int64_t T, int64_t K, int64_t ldx, const int32_t *offsets,
                                           int32_t G, uint8_t *qt, int64_t ldqt, float *st, int64_t ldst, bool pow2,
                                           cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const dim3 grid((unsigned)(K / kTT), (unsigned)grouped_token_blocks(T, G));
    const uint16_t *xp = static_cast<const uint16_t *>(x);
    auto kern = pow2 ? k_quant_act_128x1<false, true, true> : k_quant_act_128x1<false, false, true>;
    kern<<<grid, 256, 0, stream>>>(xp, ldx, qt, ldqt, st, ldst, nullptr, 0, nullptr, 0, T, offsets, G);
    return cudaGetLastError();
}

cudaError_t launch_quant_weight_128x128_t(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq,
                                          float *s, uint8_t *qt, int64_t ldqt, float *st, bool pow2,
                                          cudaStream_t stream) {
    const int64_t KB = K / kTT, NB = N / kTT;
    const dim3 grid((unsigned)KB, (unsigned)NB);
    k_quant_w_128x128_t<<<grid, 256, 0, stream>>>(static_cast<const uint16_t *>(w), ldw, KB, NB, q, ldq, s, qt, ldqt,
                                                  st, pow2 ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace fp8bs
