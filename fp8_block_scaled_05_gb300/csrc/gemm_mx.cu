// Block-scaled FP8 GEMM for power-of-two scales, dense and grouped (MoE),
// with the scales applied by the tensor core itself.
//
//   C[m, n] = bf16( sum_kb sA[kb, m] * sB[n/128, kb] * P[m, n, kb] ),
//   P[m, n, kb] = sum_{k in kb} dec(qa[m, k]) dec(qb[n, k])
//
// The same layer as the promote kernel; it applies when every scale is a
// power of two, the option that restricts FP8 scale factors to powers of two
// (upppp.jp NeMo RL FP8 article, §設定方法; greentreeone.com page, §Почему
// это важно).  A power of two is exactly a UE8M0 scale factor, so
// tcgen05.mma kind::mxf8f6f4.block_scale multiplies each 32-wide K slice by
// 2^(ea + eb - 254) inside the tensor core and the whole K range accumulates
// in one fp32 TMEM accumulator: there is no per-K-block promotion.  Each
// 1x128 (activation) or 128x128 (weight) scale is used by the four K = 32
// instructions of its K-block.
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles, 16 warps):
//   warp 0      TMA producer: qa tile 128x128 and qb tile 256x128 per K-block
//               into a 4-stage, 192 KB shared-memory ring (128-byte swizzle).
//   warp 1      MMA issuer and TMEM owner: four tcgen05.mma (M=128, N=256,
//               K=32) per K-block into the accumulator, TMEM columns [0, 256),
//               issued by lane 0.
//   warp 2      gatekeeper: does every barrier wait the MMAs depend on
//               (accumulator drained, scale factors written, operands landed)
//               and then meets the issuer warp at a named barrier, once per
//               K-block.  A wait with acquire semantics (an mbarrier test, an
//               acquire load) in a thread that has MMAs in flight stalls it
//               until they complete, ~600 cycles past the 512 a K-block takes;
//               a named barrier does not, and it orders memory between the
//               two warps.  The named barrier has no time limit, so the
//               gatekeeper never leaves its loop early: after a wait runs out it
//               sets an abort flag and keeps meeting the issuer, which then
//               issues nothing.
//   warps 4..7  scale-factor writers, one per TMEM lane quarter: for each
//               group of four K-blocks they convert the scales to UE8M0
//               bytes (byte j = K-block 4g + j, selected per instruction by
//               the descriptor's scale-factor id) and store them with
//               tcgen05.st into a 4-slot ring at TMEM columns [256, 320):
//               A's scale of row m in lane m, column m/32 of the slot; B's
//               scale of weight row n in lane 32q + n%32, column 8 + n/32,
//               in every lane quarter q.  A scale that is not a power of two
//               in [2^-127, 2^127] is reported in the status word.
//   warps 8..15 epilogue, two per lane quarter (128 columns each): once per
//               tile they read the accumulator in three round trips, packing
//               it to bf16, hand TMEM back (the next tile's MMAs start
//               while they store) and write the 32 x 128 block as four 32 x 32
//               TMA stores through a 2 KB shared-memory buffer per warp
//               (64-byte swizzle, so the row-per-thread writes into it are
//               free of bank conflicts).  Stores straight from registers, one
//               16-byte piece of 32 different rows per instruction, slowed the
//               whole kernel by a quarter.  A grouped tile that ends inside an
//               expert stores its rows one by one instead, up to the expert's
//               last row (a TMA store would clip only at M).
// The scale-factor writers and the epilogue sleep in their waits (they are off
// the critical path, and spinning warps slowed the MMA feed by ~5%); the
// producer and the gatekeeper spin.  Every wait is bounded; a wait that runs
// out records a timeout in the status word and the kernel unwinds (waiting,
// bounded, for its own copies and MMAs).
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "codec.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace fp8bs {
namespace mx {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 48 KB
constexpr int STAGES = 4;
constexpr int RING_BYTES = STAGES * STAGE_BYTES;
constexpr int EPI_BUF_BYTES = 32 * 64;           // one 32 x 32 bf16 block per epilogue warp
constexpr int KB_PER_SF = 4;                     // K-blocks per scale-factor group (one byte each)
constexpr int SF_SLOTS = 4;                      // scale-factor groups in flight
constexpr uint32_t SF_COL0 = 256;                // first TMEM column of the scale-factor ring
constexpr uint32_t SF_SLOT_COLS = 16;            // A: columns +0..+3, B: columns +8..+15
constexpr int ISSUE_WARP = 1, GATE_WARP = 2;
constexpr uint32_t kIssueBar = 1;                // named barrier: gatekeeper + issuer warps
constexpr int SF_WARP0 = 4;
constexpr int EPI_WARP0 = 8, EPI_WARPS = 8;
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);   // 512
constexpr int MAX_GROUPS = 1024;
constexpr uint32_t IDESC = idesc_mx_e4m3(BM, BN, 0, 0);
static_assert(SF_COL0 + SF_SLOTS * SF_SLOT_COLS <= 512, "TMEM columns");

// Status word code for a scale that is not an exact power of two (the value
// of FP8_ERR_SCALE_MODE).
constexpr int kStatusBadScale = 4;

struct __align__(16) Ctrl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t sfull[SF_SLOTS];
    uint64_t sempty[SF_SLOTS];
    uint64_t tfull;
    uint64_t tempty;
    uint64_t mma_done;
    uint32_t tmem_base;
    int32_t n_tiles;
    volatile int32_t abort_issue;   // set by the gatekeeper after a wait ran out
    int32_t pad_;
};

constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + (size_t)RING_BYTES + (size_t)EPI_WARPS * EPI_BUF_BYTES +
                               sizeof(Ctrl) + (size_t)(MAX_GROUPS + 1) * sizeof(int32_t);
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");

__device__ __forceinline__ void record(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Two fp32 bit patterns -> a packed bf16 pair (round to nearest even), `lo`
// in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(hi)), "f"(__uint_as_float(lo)));
    return r;
}

// fp32 power of two -> UE8M0 byte (2^(e-127)); 2^-127 is the fp32 subnormal
// 0x00400000, whose exponent field 0 is the right byte.  `bad` is set for
// anything else (zero, negative, non-power-of-two, inf, NaN).
__device__ __forceinline__ uint32_t ue8m0(float s, bool& bad) {
    const uint32_t b = __float_as_uint(s);
    const uint32_t e = b >> 23;
    const bool ok = ((b & 0x7FFFFFu) == 0u && e >= 1u && e <= 254u) || b == 0x00400000u;
    bad |= !ok;
    return ok ? e : 127u;
}

// PER_TENSOR: sa and sb each point at one fp32 scale for the whole operand
// (per-tensor scaling).  The scale factors are then 2^0 (the block-scaled MMA
// is a plain FP8 MMA with fp32 accumulation over all of K) and the epilogue
// multiplies by RN(sa * sb) once.
// Element i of a scale array: fp32, or (e8) a UE8M0 byte widened to the fp32
// power of two it stands for (byte 0 is 2^-127, a subnormal; 255 becomes inf
// and is reported by ue8m0 below).
__device__ __forceinline__ float scale_at(const float* __restrict__ p, size_t i, int e8) {
    if (!e8) return p[i];
    const uint32_t b = reinterpret_cast<const uint8_t*>(p)[i];
    return __uint_as_float(b == 0u ? 0x00400000u : b << 23);
}

// KGROUP (mixture-of-experts weight gradients, per-row B scales): G GEMMs
// C_g [M, N] = A_g B_g^T reducing over each expert's own padded token blocks
// P_g .. P_{g+1}-1 (P_g = sum_{g' < g} ceil(M_g' / 128) over the device
// offsets of kg_tokens tokens), the layout the grouped 128x1 quantiser
// writes; C_g is rows g M .. of the output, zeros for an expert without
// tokens (its tiles issue no MMA and never touch TMEM).
template <bool GROUPED, bool PER_TENSOR = false, bool KGROUP = false>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_mx(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
              const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_q,
              const float* __restrict__ sa, int64_t ldsa, const float* __restrict__ sb, int64_t ldsb,
              uint16_t* __restrict__ c, int64_t ldc, int M, int N, int K, const int32_t* __restrict__ offsets, int G,
              int* status, SplitTail split, QuantOut qo, int e8, int kg_tokens) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* epi_buf = smem + (size_t)RING_BYTES;   // 1024-byte aligned
    Ctrl* ctl = reinterpret_cast<Ctrl*>(epi_buf + (size_t)EPI_WARPS * EPI_BUF_BYTES);
    int32_t* cum = reinterpret_cast<int32_t*>(ctl + 1);

    const int warp = (int)warp_id(), lane = (int)lane_id();
    const int KB = K / BK;
    const int NT = (N + BN - 1) / BN;
    const int NB = N / 128;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int s = 0; s < SF_SLOTS; ++s) {
            mbar_init(&ctl->sfull[s], 4);   // one arrival per scale-factor warp
            mbar_init(&ctl->sempty[s], 1);
        }
        mbar_init(&ctl->tfull, 1);
        mbar_init(&ctl->tempty, EPI_WARPS);
        mbar_init(&ctl->mma_done, 1);
        ctl->abort_issue = 0;
        mbar_init_fence();
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        tma_prefetch_desc(&tm_c);
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == 3) {
        if (GROUPED) {
            const int total = build_group_table<BM>(offsets, G, M, NT, cum);
            if (lane == 0) ctl->n_tiles = total;
        } else if (KGROUP) {
            // cum[g]: the first padded token block of expert g
            build_group_table<BM>(offsets, G, kg_tokens, 1, cum);
            if (lane == 0) ctl->n_tiles = G * ((M + BM - 1) / BM) * NT;
        } else if (lane == 0) {
            ctl->n_tiles = ((M + BM - 1) / BM) * NT;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = ctl->tmem_base;
    const int n_tiles = ctl->n_tiles;
    const int n_items = work_items(n_tiles, split);
    const int tiles_per_expert = ((M + BM - 1) / BM) * NT;   // KGROUP
    // Work item t and its tile (with KGROUP: the expert's K range and tile).
    auto item_at = [&](int t) -> Item {
        Item w = decode_item(t, split, KB);
        if constexpr (KGROUP) {
            const int g = w.tile / tiles_per_expert;
            w.kb0 = cum[g];
            w.kb1 = cum[g + 1];
        }
        return w;
    };
    auto tile_at = [&](const Item& w) -> Tile {
        if constexpr (KGROUP) {
            Tile tl = decode_tile<BM, BN, false>(w.tile % tiles_per_expert, M, N, cum, offsets, G);
            tl.g = w.tile / tiles_per_expert;
            return tl;
        } else {
            return decode_tile<BM, BN, GROUPED>(w.tile, M, N, cum, offsets, G);
        }
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_items && ok; t += gridDim.x) {
                const Item w = item_at(t);
                const Tile tl = tile_at(w);
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (!mbar_wait(&ctl->empty[s], ph ^ 1, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sA = smem + (size_t)s * STAGE_BYTES;
                    mbar_arrive_expect_tx(&ctl->full[s], STAGE_BYTES);
                    tma_load_2d(sA, &tm_a, &ctl->full[s], kb * BK, tl.m0);
                    tma_load_2d(sA + A_BYTES, &tm_b, &ctl->full[s], kb * BK, tl.brow);
                }
            }
            if (!ok) {
                record(status, kStatusTimeout);
                // Let the copies already issued land before the CTA can exit.
                const uint32_t n = it < (uint32_t)STAGES ? it : (uint32_t)STAGES;
                for (uint32_t j = it - n; j < it; ++j)
                    mbar_wait(&ctl->full[j % STAGES], (j / STAGES) & 1, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else if (warp == GATE_WARP) {
        // ------------------------------------------------ gatekeeper
        uint32_t it = 0, gi = 0, tt = 0;   // tt: items that use the accumulator (an empty K range does not)
        bool ok = true;
        for (int t = blockIdx.x; t < n_items; t += gridDim.x) {
            const Item w = item_at(t);
            for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                const uint32_t byte = (uint32_t)(kb - w.kb0) % KB_PER_SF;
                if (lane == 0 && ok) {
                    ok = (kb > w.kb0 || mbar_wait(&ctl->tempty, (tt & 1) ^ 1, kWaitLimitNs)) &&
                         (byte > 0 || mbar_wait(&ctl->sfull[gi % SF_SLOTS], (gi / SF_SLOTS) & 1, kWaitLimitNs)) &&
                         mbar_wait(&ctl->full[it % STAGES], (it / STAGES) & 1, kWaitLimitNs);
                    if (!ok) {
                        ctl->abort_issue = 1;
                        record(status, kStatusTimeout);
                    }
                }
                named_bar_sync(kIssueBar, 64);   // K-block `it` may be issued
                if (byte == KB_PER_SF - 1 || kb == w.kb1 - 1) ++gi;
            }
            if (w.kb1 > w.kb0) ++tt;
        }
    } else if (warp == ISSUE_WARP) {
        // ------------------------------------------------ MMA issuer
        uint32_t it = 0, gi = 0;
        for (int t = blockIdx.x; t < n_items; t += gridDim.x) {
            const Item w = item_at(t);
            for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                const uint32_t s = it % STAGES;
                const uint32_t byte = (uint32_t)(kb - w.kb0) % KB_PER_SF;
                const uint32_t slot = gi % SF_SLOTS;
                named_bar_sync(kIssueBar, 64);
                if (lane == 0 && !ctl->abort_issue) {
                    tc_fence_after_sync();
                    const uint32_t sA = smem_u32(smem + (size_t)s * STAGE_BYTES);
                    const uint64_t adesc = sdesc_kmajor_sw128(sA);
                    const uint64_t bdesc = sdesc_kmajor_sw128(sA + A_BYTES);
                    const uint32_t sfa = tmem_base + SF_COL0 + slot * SF_SLOT_COLS;
                    const uint32_t idesc = IDESC | (byte << 4) | (byte << 29);   // B, A scale-factor byte id
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        umma_mxf8f6f4(tmem_base, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc, sfa,
                                      sfa + 8, (kb > w.kb0 || k > 0) ? 1u : 0u);
                    umma_commit(&ctl->empty[s]);
                    if (byte == KB_PER_SF - 1 || kb == w.kb1 - 1) umma_commit(&ctl->sempty[slot]);
                    if (kb == w.kb1 - 1) umma_commit(&ctl->tfull);
                }
                __syncwarp();
                if (byte == KB_PER_SF - 1 || kb == w.kb1 - 1) ++gi;
            }
        }
        if (lane == 0) {
            // All MMAs this thread issued are complete before TMEM is released.
            umma_commit(&ctl->mma_done);
            mbar_wait(&ctl->mma_done, 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp >= SF_WARP0 && warp < EPI_WARP0) {
        // ------------------------------------------------ scale-factor writers
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        uint32_t gi = 0;
        bool ok = true, bad = false;
        for (int t = blockIdx.x; t < n_items && ok; t += gridDim.x) {
            const Item w = item_at(t);
            const Tile tl = tile_at(w);
            const int m = tl.m0 + q * 32 + lane;
            const bool vrow = m < tl.row_end;
            const int nb0 = tl.n0 / 128;
            const size_t sb0 = ((size_t)tl.g * NB + nb0) * KB;   // index of the tile's first B scale
            for (int kb0 = w.kb0; kb0 < w.kb1; kb0 += KB_PER_SF, ++gi) {
                // Scales first (their latency overlaps the wait for the slot).
                float fa[KB_PER_SF], fb0[KB_PER_SF], fb1[KB_PER_SF];
#pragma unroll
                for (int j = 0; j < KB_PER_SF; ++j) {
                    const int kb = kb0 + j;
                    fa[j] = (!PER_TENSOR && kb < w.kb1 && vrow) ? scale_at(sa, (size_t)kb * ldsa + m, e8) : 1.0f;
                    fb0[j] = (!PER_TENSOR && kb < w.kb1 && ldsb == 0) ? scale_at(sb, sb0 + kb, e8) : 1.0f;
                    fb1[j] = (!PER_TENSOR && kb < w.kb1 && ldsb == 0 && nb0 + 1 < NB) ? scale_at(sb, sb0 + KB + kb, e8)
                                                                                        : 1.0f;
                }
                uint32_t wa = 0, wb0 = 0, wb1 = 0;
#pragma unroll
                for (int j = 0; j < KB_PER_SF; ++j) {
                    wa |= ue8m0(fa[j], bad) << (8 * j);
                    wb0 |= ue8m0(fb0[j], bad) << (8 * j);
                    wb1 |= ue8m0(fb1[j], bad) << (8 * j);
                }
                // B scale-factor column j holds rows n0 + 32 j + lane: the weight
                // block's scale, or with ldsb > 0 each row's own (sb[kb * ldsb + n])
                uint32_t vb[8] = {wb0, wb0, wb0, wb0, wb1, wb1, wb1, wb1};
                if (!PER_TENSOR && ldsb > 0) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int n = tl.n0 + 32 * j + lane;
                        uint32_t wj = 0;
#pragma unroll
                        for (int i = 0; i < KB_PER_SF; ++i) {
                            const int kb = kb0 + i;
                            const float f = (kb < w.kb1 && n < N) ? scale_at(sb, (size_t)kb * ldsb + n, e8) : 1.0f;
                            wj |= ue8m0(f, bad) << (8 * i);
                        }
                        vb[j] = wj;
                    }
                }
                const uint32_t slot = gi % SF_SLOTS;
                bool got = mbar_wait_sleep(&ctl->sempty[slot], ((gi / SF_SLOTS) & 1) ^ 1, kWaitLimitNs);
                got = __all_sync(0xFFFFFFFFu, got);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t col = tmem_base + lane_base + SF_COL0 + slot * SF_SLOT_COLS;
                tmem_st_x1(col + (uint32_t)q, wa);
                tmem_st_x8(col + 8, vb);
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->sfull[slot]);
            }
        }
        if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) record(status, kStatusBadScale);
        if (!ok && lane == 0) record(status, kStatusTimeout);
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int h = (warp - EPI_WARP0) >> 2;   // column half of the tile
        const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 128);
        uint8_t* buf = epi_buf + (size_t)(warp - EPI_WARP0) * EPI_BUF_BYTES;
        // One 32 x 32 bf16 block (16 packed pairs per lane) through this warp's
        // buffer and a TMA store.  Row `lane`, 16-byte piece k goes to offset
        // lane*64 + ((k ^ ((lane >> 1) & 3)) << 4): the 64-byte swizzle the
        // tensor map declares.
        auto store_block = [&](const uint32_t* pk, int col, int row) {
            if (lane == 0) bulk_wait_group_read<0>();   // the previous store has read buf
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint4*>(buf + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                    make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&tm_c, buf, col, row);
                bulk_commit_group();
            }
        };
        // Per-tensor scaling: the whole product's scale, applied to each fp32
        // accumulator before the bf16 rounding.
        const float ts = PER_TENSOR ? sa[0] * sb[0] : 1.0f;
        auto scaled = [&](uint32_t v) -> uint32_t {
            return PER_TENSOR ? __float_as_uint(__uint_as_float(v) * ts) : v;
        };
        uint32_t tt = 0;   // items that used the accumulator so far
        bool ok = true;
        for (int t = blockIdx.x; t < n_items; t += gridDim.x) {
            const Item w = item_at(t);
            const Tile tl = tile_at(w);
            const int m = tl.m0 + q * 32 + lane;
            const int col0 = tl.n0 + h * 128;
            const int crow = (KGROUP ? tl.g * M : 0) + tl.m0 + q * 32;   // first output row of this warp
            if (KGROUP && w.kb1 == w.kb0) {
                // an expert without tokens: its gradient is zero (no MMA, no TMEM)
                if (col0 < N) {
                    uint32_t z[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) z[jj] = 0u;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) store_block(z, col0 + 32 * cc, crow);
                }
                continue;
            }
            bool got = mbar_wait_sleep(&ctl->tfull, tt & 1, kWaitLimitNs);
            ++tt;
            got = __all_sync(0xFFFFFFFFu, got);
            if (!got) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t taddr = tacc;
            uint32_t p[64];   // the warp's 32 x 128 block as bf16 pairs (row `lane`)
            if (w.parts > 1) {
                // A K-split tile of the last wave (this CTA's last item): the fp32
                // part goes straight from TMEM to the workspace, and the warp that
                // completes this slice's ticket adds the parts in part order.
                const bool live = col0 < N;
                float* part0 = split.part + (size_t)(w.tile - split.n_full) * w.parts * (BM * BN) +
                               (size_t)(h * 128) * BM + q * 32 + lane;   // [part][col][row]
                float* dst = part0 + (size_t)w.part * (BM * BN);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t v[32];
                    tmem_ld_x32(taddr + 32 * cc, v);
                    tmem_ld_wait();
                    if (live) {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) __stcg(dst + (cc * 32 + jj) * BM, __uint_as_float(v[jj]));
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty);
                if (!live) continue;
                const int wslot = (w.tile - split.n_full) * EPI_WARPS + (warp - EPI_WARP0);
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) last = atomicAdd(&split.ticket[wslot], 1) == w.parts - 1;
                if (!__shfl_sync(0xFFFFFFFFu, last, 0)) continue;
                __threadfence();
                if (lane == 0) split.ticket[wslot] = 0;   // ready for the next call
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    float sum[32];
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) sum[jj] = 0.0f;
#pragma unroll 1
                    for (int pp = 0; pp < w.parts; ++pp) {
                        const float* src = part0 + (size_t)pp * (BM * BN) + (size_t)(cc * 32) * BM;
                        float v[32];
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) v[jj] = __ldcg(src + jj * BM);
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) sum[jj] += v[jj];
                    }
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        p[16 * cc + jj] = pack_bf16x2(scaled(__float_as_uint(sum[2 * jj])),
                                                      scaled(__float_as_uint(sum[2 * jj + 1])));
                }
                // the summed block goes on like a whole tile's (fused codes, C)
            } else {
                // Three round trips (64, 32 and 32 columns), packed to bf16 pairs as
                // they arrive so that at most 64 raw values are live; TMEM goes back
                // before any store.
                {
                    uint32_t v0[32], v1[32];
                    tmem_ld_x32(taddr, v0);
                    tmem_ld_x32(taddr + 32, v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        p[jj] = pack_bf16x2(scaled(v0[2 * jj]), scaled(v0[2 * jj + 1]));
                        p[16 + jj] = pack_bf16x2(scaled(v1[2 * jj]), scaled(v1[2 * jj + 1]));
                    }
                }
#pragma unroll
                for (int r = 2; r < 4; ++r) {
                    uint32_t v[32];
                    tmem_ld_x32(taddr + 32 * r, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) p[16 * r + jj] = pack_bf16x2(scaled(v[2 * jj]), scaled(v[2 * jj + 1]));
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty);
                if (col0 >= N) continue;   // the half of a 256-wide tile past N
            }
            if (!GROUPED && qo.q != nullptr) {
                // Fused quantisation for the next layer: this warp holds, per row,
                // the whole 128-column block col0 .. col0 + 127 as bf16 pairs, so
                // the row's amax needs no exchange; codes and scale are those the
                // 1x128 activation quantiser gives for these bf16 values.
                uint32_t m2 = 0;
#pragma unroll
                for (int e = 0; e < 64; ++e) m2 = absmax_bf16x2(m2, p[e]);
                const BlockScale bs = make_scale(absmax_pair_to_f32(m2), qo.pow2 != 0);
                if (m < tl.row_end) qo.s[(size_t)(col0 / 128) * qo.lds + m] = bs.s;
                // the product cast for the warp unless a row's factor overflows
                // (a per-pair test of the mode made this cast several times slower)
                const bool all_mul = __all_sync(0xFFFFFFFFu, bs.mode == 1);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
                    with_cast(all_mul, [&](auto cast) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int j0 = 32 * hf + 8 * k;
                            const uint2 c0 =
                                quant8_as<decltype(cast)::mul>(make_uint4(p[j0], p[j0 + 1], p[j0 + 2], p[j0 + 3]), bs);
                            const uint2 c1 = quant8_as<decltype(cast)::mul>(
                                make_uint4(p[j0 + 4], p[j0 + 5], p[j0 + 6], p[j0 + 7]), bs);
                            *reinterpret_cast<uint4*>(buf + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                                make_uint4(c0.x, c0.y, c1.x, c1.y);
                        }
                    });
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tm_q, buf, col0 + 64 * hf, crow);
                        bulk_commit_group();
                    }
                }
                if (!qo.write_c) continue;
            }
            const int rows_here = min(tl.row_end - (tl.m0 + q * 32), 32);
            if (!GROUPED || rows_here == 32) {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) store_block(p + 16 * cc, col0 + 32 * cc, crow);
            } else if (lane < rows_here) {
                uint4* dst = reinterpret_cast<uint4*>(c + (size_t)m * ldc + col0);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    dst[jj] = make_uint4(p[4 * jj], p[4 * jj + 1], p[4 * jj + 2], p[4 * jj + 3]);
            }
        }
        if (lane == 0) bulk_wait_group<0>();   // stores complete before the CTA exits
        if (!ok && lane == 0) record(status, kStatusTimeout);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, 512);
    }
}

template <bool GROUPED, bool PER_TENSOR = false, bool KGROUP = false>
cudaError_t launch(const GemmArgs& a, cudaStream_t st) {
    static DeviceOnce attr_done;     // kernel attributes set on this device
    auto kern = k_gemm_mx<GROUPED, PER_TENSOR, KGROUP>;
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_done.test(dev)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done.set(dev);
    }
    const int64_t NT = (a.N + BN - 1) / BN;
    const int64_t tiles = GROUPED ? (((a.M + BM - 1) / BM) + a.G) * NT
                                  : ((a.M + BM - 1) / BM) * NT * (KGROUP ? a.G : 1);
    SplitTail split{0, 1, nullptr, nullptr};
    if (!GROUPED && !KGROUP) {
        const TailPlan tp = tail_plan(a.M, a.N, a.K, a.sm_count, BN, kMxMaxParts);
        if (tp.parts > 1 && a.workspace && a.ws_bytes >= tp.bytes) {
            split.n_full = (int)tp.n_full;
            split.parts = tp.parts;
            split.ticket = static_cast<int*>(a.workspace);
            split.part = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + tp.ticket_bytes);
        }
    }
    const int64_t items = work_items((int)tiles, split);
    const int grid = (int)(items < a.sm_count ? items : a.sm_count);
    kern<<<grid, THREADS, SMEM_BYTES, st>>>(a.tm_a, a.tm_b, a.tm_c, a.tm_q, a.sa, a.ldsa, a.sb, a.ldsb, static_cast<uint16_t*>(a.c), a.ldc,
                                            (int)a.M, (int)a.N, (int)a.K, a.offsets, a.G, a.status, split, a.qout,
                                            a.scales_e8, (int)a.kg_tokens);
    return cudaGetLastError();
}

}  // namespace mx

cudaError_t launch_gemm_mx(const GemmArgs& a, cudaStream_t st) {
    if (a.M == 0) return cudaSuccess;
    if (a.per_tensor) return a.offsets != nullptr ? cudaErrorInvalidValue : mx::launch<false, true>(a, st);
    if (a.kgroup) {   // per-expert weight gradients over the experts' token blocks
        if (a.offsets == nullptr || a.ldsb <= 0) return cudaErrorInvalidValue;
        return mx::launch<false, false, true>(a, st);
    }
    return a.offsets != nullptr ? mx::launch<true>(a, st) : mx::launch<false>(a, st);
}

}  // namespace fp8bs
