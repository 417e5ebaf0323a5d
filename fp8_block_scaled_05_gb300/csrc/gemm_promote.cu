// Block-scaled FP8 GEMM with per-K-block promotion, dense and grouped (MoE).
//
//   C[m, n] = bf16( sum_kb sA[kb, m] * sB[n/128, kb] * P[m, n, kb] ),
//   P[m, n, kb] = sum_{k in kb} dec(qa[m, k]) dec(qb[n, k])
//
// FP8 linear layers with 1x128 activation and 128x128 weight scales (page
// "NVIDIA NeMo RL достигает ускорения на 48% благодаря сквозному обучению с
// точностью FP8", greentreeone.com, §Технический прорыв), accumulated in
// higher precision than the operands (ai.warp-studio.com end-to-end FP8 RL
// article, §FP8強化学習における精度と安定性の確保).  The grouped form runs
// the same layer per expert of a mixture-of-experts model (upppp.jp NeMo RL
// FP8 article, §まとめ; greentreeone.com page, §Реальные прирост
// производительности, Qwen3-30B).
//
// Design (one CTA per SM, persistent over output tiles of 128 x BN, BN = 128
// or 256):
//   warp 0      TMA producer: qa tile 128x128 and qb tile BNx128 per K-block
//               into a shared-memory ring (128-byte swizzle): 4 stages, 192 KB
//               (3 stages for the weight-gradient form, see WHOLE_OUT).
//   warps 1, 3  MMA issuers, one thread each, taking alternate K-blocks: four
//               tcgen05.mma (M=128, N=BN, K=32) per K-block into one of
//               512/BN BN-column TMEM buffers, the first with accumulate = 0.
//               Two issuers keep the tensor core fed while either waits on a
//               barrier (one thread waiting per K-block leaves the MMA queue
//               empty for the length of the wait).  Warp 1 owns TMEM.
//   warp 2      scale producer: cp.async copies of the 128 activation scales
//               and the weight scale(s) of each K-block into an 8-slot
//               shared-memory ring, so the promotion never waits on a global
//               load.
//   warps 4..   promotion: each K-block's fp32 partial is read from TMEM
//               (tcgen05.ld) and added into registers with the scale product
//               sA*sB; the buffer is handed back right after the read, so the
//               tensor core works on the next K-blocks meanwhile.  Warp w owns
//               TMEM lanes 32*(w%4).. and a column slice of the tile that lies
//               inside one 128-column weight block (one sB per K-block).
//               BN = 128: 16 warps x 32 columns (4 TMEM buffers, 96 registers
//               per thread).  BN = 256: 8 warps x 128 columns (2 buffers); the
//               first warpgroup hands registers to the promotion warpgroups
//               (setmaxnreg 40 / 232 within the 168 per thread of the launch).
// Every wait is bounded; a wait that runs out records a timeout in the status
// word and the kernel unwinds (waiting, bounded, for its own copies and MMAs).
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "codec.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace fp8bs {
namespace promote {

constexpr int BM = 128, BK = 128;
constexpr int EPI_WARP0 = 4;                 // first promotion warp
constexpr int SCALE_WARP = 2;
constexpr uint32_t kBufBar0 = 1;             // named barriers 1.. : TMEM buffer b handed back to its issuer
constexpr int MAX_GROUPS = 1024;
constexpr int SRING = 8;                     // scale ring slots
constexpr int EPI_BLK_BYTES = 32 * 64;       // one 32 x 32 bf16 output block

// WHOLE_OUT (BN 256 only): a 3-stage operand ring (144 KB) leaves room for
// each promotion warp to stage its whole 32 x 128 output (8 KB), so its TMA
// stores drain during the next tile instead of one 2 KB block at a time.
// That pays where the output is large against the work (weight gradients:
// 4-11% faster) and costs the long-K forward GEMMs the fourth stage (5-7%
// slower), so only the per-row-scale (weight-gradient) instantiations use it.
template <int BN_, bool WHOLE_OUT_ = false>
struct Cfg {
    static constexpr int BN = BN_;
    static constexpr bool WHOLE_OUT = WHOLE_OUT_ && BN_ == 256;
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = WHOLE_OUT ? 3 : 4;          // 144 / 192 KB (BN 256) or 128 KB (BN 128)
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int NBUF = 512 / BN;                     // TMEM accumulator buffers
    static constexpr int EPI_WARPS = BN == 128 ? 16 : 8;
    static constexpr int SLICES = EPI_WARPS / 4;              // column slices per TMEM lane quarter
    static constexpr int EPI_COLS = BN / SLICES;              // columns per promotion warp
    static constexpr int CHUNKS = EPI_COLS / 32;
    static constexpr int EPI_BUF_BYTES = (WHOLE_OUT ? CHUNKS : 1) * EPI_BLK_BYTES;   // per promotion warp
    static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
    static constexpr int TBAR_THREADS = 32 * (EPI_WARPS + 1);   // promotion warps + the buffer's issuer warp
    static constexpr bool SPLIT_REGS = BN == 256;
    static constexpr int LAUNCH_REGS = 168;                   // 65536 / 384, rounded to 8 (BN 256)
    static constexpr int REGS_CTRL = 40;                      // warpgroup 0 after setmaxnreg.dec
    static constexpr int REGS_EPI = 232;                      // promotion warpgroups after .inc
    static constexpr uint32_t IDESC = idesc_e4m3_f32(BM, BN);
    static_assert(NBUF % 2 == 0, "each TMEM buffer belongs to one MMA issuer");
    static_assert(STAGES <= 8 && NBUF <= 4, "barrier arrays");
    static_assert(!SPLIT_REGS || (128 * REGS_CTRL + (THREADS - 128) * REGS_EPI <= THREADS * LAUNCH_REGS),
                  "register split exceeds the launch");
};

struct ScaleSlot {
    float sa[BM];
    float sb[2];
    float pad[2];
};

struct __align__(16) Ctrl {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t tfull[4];
    uint64_t tempty[4];
    uint64_t sfull[SRING];
    uint64_t sempty[SRING];
    uint64_t mma_done[2];
    uint32_t tmem_base;
    int32_t n_tiles;
    int32_t abort_flag;
    int32_t pad_;
    ScaleSlot ring[SRING];
};

// ROWB (a scale per B row): a ring of SRING x BN column scales follows the
// group table.
template <int BN, bool ROWB = false>
constexpr size_t smem_bytes() {
    using C = Cfg<BN, ROWB>;
    return 1024 /*align slack*/ + (size_t)C::RING_BYTES + (size_t)C::EPI_WARPS * C::EPI_BUF_BYTES +
           sizeof(Ctrl) + (size_t)(MAX_GROUPS + 4) * sizeof(int32_t) + (ROWB ? (size_t)SRING * BN * sizeof(float) : 0);
}
static_assert(smem_bytes<256, true>() <= 232448 && smem_bytes<128, true>() <= 232448, "shared memory per CTA");

__device__ __forceinline__ void record_timeout(int* status) {
    if (status) atomicCAS(status, 0, kStatusTimeout);
}

// ROWB: sb holds a scale per B row (sb[kb * ldsb + n]), so the promotion
// multiplies by a per-column scale product (dense only).
// KGROUP (with ROWB; mixture-of-experts weight gradients): G independent
// GEMMs C_g [M, N] = A_g B_g^T that reduce over each expert's own tokens:
// the K-blocks of expert g are the padded token blocks P_g .. P_{g+1}-1 (P_g
// = sum_{g' < g} ceil(M_g' / 128), M_g' from the device offsets over
// kg_tokens tokens), the layout the grouped 128x1 quantiser writes.  Tiles
// run expert by expert; C_g is rows g M .. g M + M - 1 of the output (M %
// 128 == 0); an expert without tokens gets zeros.
template <int BN, bool GROUPED, bool ROWB, bool KGROUP = false>
__global__ void __launch_bounds__(Cfg<BN, ROWB>::THREADS, 1)
    k_gemm_promote(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_q,
                   const float* __restrict__ sa, int64_t ldsa, const float* __restrict__ sb, int64_t ldsb,
                   uint16_t* __restrict__ c, int64_t ldc, int M, int N, int K,
                   const int32_t* __restrict__ offsets, int G, int* status, SplitTail split, QuantOut qo,
                   uint64_t wait_ns, int skip_first_load, int kg_tokens) {
    using C = Cfg<BN, ROWB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* epi_buf = smem + (size_t)C::RING_BYTES;   // 1024-byte aligned
    Ctrl* ctl = reinterpret_cast<Ctrl*>(epi_buf + (size_t)C::EPI_WARPS * C::EPI_BUF_BYTES);
    int32_t* cum = reinterpret_cast<int32_t*>(ctl + 1);
    float* sb_ring = reinterpret_cast<float*>(cum + MAX_GROUPS + 4);   // ROWB: [SRING][BN], 16-byte aligned
    static_assert(!(ROWB && GROUPED), "per-row B scales are dense only");
    static_assert(!KGROUP || (ROWB && !GROUPED), "K-grouped tiles are the weight-gradient form");

    const int warp = (int)warp_id(), lane = (int)lane_id();
    const int KB = K / BK;
    const int NT = (N + BN - 1) / BN;
    const int NB = N / 128;
    // How a TMEM buffer goes back to its issuer: the dense forward form uses
    // a named barrier that every participant syncs on (the hand-off is on its
    // critical path: 2-3% faster); the weight-gradient and grouped forms keep
    // the buffer's mbarrier, so that their promotion warps, which bound those
    // forms, never wait for an issuer (the named barrier made them 6-25% slower).
    constexpr bool BAR_HANDOFF = !ROWB && !GROUPED && !KGROUP;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < C::NBUF; ++b) {
            mbar_init(&ctl->tfull[b], 1);
            mbar_init(&ctl->tempty[b], C::EPI_WARPS);
        }
        for (int s = 0; s < SRING; ++s) {
            mbar_init(&ctl->sfull[s], 32);        // one cp.async arrival per lane of the scale warp
            mbar_init(&ctl->sempty[s], C::EPI_WARPS);
        }
        mbar_init(&ctl->mma_done[0], 1);
        mbar_init(&ctl->mma_done[1], 1);
        ctl->abort_flag = 0;
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
    volatile int32_t* abort_flag = &ctl->abort_flag;
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

    if constexpr (C::SPLIT_REGS) {
        if (warp < EPI_WARP0) regs_dealloc<C::REGS_CTRL>();
    }
    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_items && ok; t += gridDim.x) {
                const Item w = item_at(t);
                const Tile tl = tile_at(w);
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    const uint32_t s = it % C::STAGES, ph = (it / C::STAGES) & 1;
                    if (!mbar_wait(&ctl->empty[s], ph ^ 1, wait_ns)) {
                        ok = false;
                        break;
                    }
                    if (skip_first_load && it == 0) continue;   // failure-path test: K-block 0 never lands
                    uint8_t* sA = smem + (size_t)s * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&ctl->full[s], C::STAGE_BYTES);
                    tma_load_2d(sA, &tm_a, &ctl->full[s], kb * BK, tl.m0);
                    tma_load_2d(sA + C::A_BYTES, &tm_b, &ctl->full[s], kb * BK, tl.brow);
                }
            }
            if (!ok) {
                record_timeout(status);
                *abort_flag = 1;
                // Let the copies already issued land before the CTA can exit.
                const uint32_t n = it < (uint32_t)C::STAGES ? it : (uint32_t)C::STAGES;
                for (uint32_t j = it - n; j < it; ++j)
                    mbar_wait(&ctl->full[j % C::STAGES], (j / C::STAGES) & 1, wait_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------ MMA issuers
        if constexpr (BAR_HANDOFF) {
            // A TMEM buffer comes back through a named barrier that the promotion
            // warps and the buffer's issuer warp all sync on (bar.sync wakes within
            // tens of cycles; a polled mbarrier test costs a few hundred, and this
            // wait is on the critical path).  Every participant blocks, so each
            // phase pairs one K-block's promotion with the issue of the next
            // K-block into the same buffer, in K-block order on both sides; after
            // a wait ran out every warp keeps walking the whole schedule (issuing
            // nothing, reading nothing), so no bar.sync is left waiting.
            const uint32_t me = warp == 1 ? 0u : 1u;   // takes K-blocks it with it % 2 == me
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_items; t += gridDim.x) {
                const Item w = item_at(t);
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    if ((it & 1) != me) continue;
                    const uint32_t s = it % C::STAGES, ph = (it / C::STAGES) & 1;
                    const uint32_t b = it % C::NBUF;
                    const uint32_t slot = it % SRING, sph = (it / SRING) & 1;
                    // Operands and scales first (usually ready long before the buffer).
                    // Waiting for the scale slot here means the promotion warps, whose
                    // loop is the critical path, find the scales in place once the
                    // K-block's partial is in TMEM and wait on one barrier only.
                    if (lane == 0 && ok) {
                        ok = mbar_wait(&ctl->full[s], ph, wait_ns) && mbar_wait(&ctl->sfull[slot], sph, wait_ns);
                        if (!ok) {
                            record_timeout(status);
                            *abort_flag = 1;
                        }
                    }
                    // the promotion warps have read buffer b's previous K-block (it - NBUF)
                    if (it >= (uint32_t)C::NBUF) named_bar_sync(kBufBar0 + b, C::TBAR_THREADS);
                    if (lane == 0 && ok) {
                        tc_fence_after_sync();
                        const uint32_t sA = smem_u32(smem + (size_t)s * C::STAGE_BYTES);
                        const uint64_t adesc = sdesc_kmajor_sw128(sA);
                        const uint64_t bdesc = sdesc_kmajor_sw128(sA + C::A_BYTES);
                        const uint32_t d = tmem_base + b * BN;
    #pragma unroll
                        for (int k = 0; k < BK / 32; ++k)
                            umma_f8f6f4(d, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), C::IDESC,
                                        k > 0 ? 1u : 0u);
                        umma_commit(&ctl->empty[s]);
                        umma_commit(&ctl->tfull[b]);
                    }
                    __syncwarp();
                }
            }
            {
                // The promotion of each owned buffer's last K-block is met here,
                // buffer by buffer in the order of those K-blocks (the order in
                // which the promotion warps reach them).  `it` is the CTA's K-block
                // count; buffer b (b < it) last serves K-block b + NBUF*floor((it-1-b)/NBUF).
                constexpr int OWN = C::NBUF / 2;
                int32_t last[OWN];
    #pragma unroll
                for (int i = 0; i < OWN; ++i) {
                    const uint32_t b = me + 2 * i;
                    last[i] = it > b ? (int32_t)(b + C::NBUF * ((it - 1 - b) / C::NBUF)) : -1;
                }
                const int first = (OWN == 2 && last[OWN - 1] >= 0 && last[OWN - 1] < last[0]) ? OWN - 1 : 0;
    #pragma unroll
                for (int r = 0; r < OWN; ++r) {
                    const int i = r == 0 ? first : (OWN - 1) - first;
                    if (last[i] >= 0) named_bar_sync(kBufBar0 + me + 2 * i, C::TBAR_THREADS);
                }
            }
            if (lane == 0) {
                // All MMAs this thread issued are complete before TMEM is released.
                umma_commit(&ctl->mma_done[me]);
                mbar_wait(&ctl->mma_done[me], 0, wait_ns);
            }
            __syncwarp();
        } else {
            if (lane == 0) {
                const uint32_t me = warp == 1 ? 0u : 1u;   // takes K-blocks it with it % 2 == me
                uint32_t it = 0;
                bool ok = true;
                for (int t = blockIdx.x; t < n_items && ok; t += gridDim.x) {
                    const Item w = item_at(t);
                    for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                        if ((it & 1) != me) continue;
                        const uint32_t s = it % C::STAGES, ph = (it / C::STAGES) & 1;
                        const uint32_t b = it % C::NBUF, tph = (it / C::NBUF) & 1;
                        // Operands and scales first (usually ready early), then the TMEM
                        // buffer, so the MMAs go out as soon as the promotion warps release
                        // it.  Waiting for the scale slot here means the promotion warps,
                        // whose loop is the critical path, find the scales in place once
                        // the K-block's partial is in TMEM and wait on one barrier only.
                        const uint32_t slot = it % SRING, sph = (it / SRING) & 1;
                        if (!mbar_wait(&ctl->full[s], ph, wait_ns) ||
                            !mbar_wait(&ctl->sfull[slot], sph, wait_ns) ||
                            !mbar_wait(&ctl->tempty[b], tph ^ 1, wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t sA = smem_u32(smem + (size_t)s * C::STAGE_BYTES);
                        const uint64_t adesc = sdesc_kmajor_sw128(sA);
                        const uint64_t bdesc = sdesc_kmajor_sw128(sA + C::A_BYTES);
                        const uint32_t d = tmem_base + b * BN;
    #pragma unroll
                        for (int k = 0; k < BK / 32; ++k)
                            umma_f8f6f4(d, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), C::IDESC,
                                        k > 0 ? 1u : 0u);
                        umma_commit(&ctl->empty[s]);
                        umma_commit(&ctl->tfull[b]);
                    }
                }
                if (!ok) {
                    record_timeout(status);
                    *abort_flag = 1;
                }
                // All MMAs this thread issued are complete before TMEM is released.
                umma_commit(&ctl->mma_done[me]);
                mbar_wait(&ctl->mma_done[me], 0, wait_ns);
            }
            __syncwarp();
        }
    } else if (warp == SCALE_WARP) {
        // ------------------------------------------------ scale producer
        uint32_t sit = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_items && ok; t += gridDim.x) {
            const Item w = item_at(t);
            const Tile tl = tile_at(w);
            const int nb0 = tl.n0 / 128;
            for (int kb = w.kb0; kb < w.kb1; ++kb, ++sit) {
                const uint32_t slot = sit % SRING, ph = (sit / SRING) & 1;
                bool got = mbar_wait(&ctl->sempty[slot], ph ^ 1, wait_ns);
                got = __all_sync(0xFFFFFFFFu, got);
                if (!got) {
                    ok = false;
                    break;
                }
                ScaleSlot& S = ctl->ring[slot];
                const float* sak = sa + (size_t)kb * ldsa;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = lane + 32 * j, m = tl.m0 + r;
                    const bool v = m < tl.row_end;
                    cp_async_4(&S.sa[r], v ? sak + m : sa, v);
                }
                if constexpr (ROWB) {
                    // the tile's BN column scales, 16 bytes per copy (zero past N)
                    const float* sbk = sb + (size_t)kb * ldsb + tl.n0;
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j) {
                        const int c4 = 4 * (lane + 32 * j);
                        const bool v = tl.n0 + c4 < N;
                        cp_async_16(sb_ring + slot * BN + c4, v ? sbk + c4 : sb, v);
                    }
                } else if (lane < 2) {
                    // BN = 256 spans weight blocks nb0 and nb0 + 1; BN = 128 uses only nb0
                    const int nb = nb0 + (BN == 256 ? lane : 0);
                    const bool v = nb < NB;
                    cp_async_4(&S.sb[lane], v ? sb + ((size_t)tl.g * NB + nb) * KB + kb : sb, v);
                }
                cp_async_arrive_noinc(&ctl->sfull[slot]);
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (!ok && lane == 0) {
            record_timeout(status);
            *abort_flag = 1;
        }
        __syncwarp();
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------ promotion epilogue
        if constexpr (C::SPLIT_REGS) regs_alloc<C::REGS_EPI>();
        const int q = warp & 3;                      // TMEM lane quarter this warp may access
        const int sl = (warp - EPI_WARP0) >> 2;      // column slice of the tile
        const int row_in_tile = q * 32 + lane;
        const int sbi = (sl * C::EPI_COLS) / 128;    // which weight block of the tile (0 or 1)
        uint32_t kbg = 0;
        bool ok = true;
        bool ready = false;   // tfull of K-block kbg already seen complete (early probe)
        // (with BAR_HANDOFF the walk goes on after a wait ran out: the issuers
        // meet every K-block on the buffer barriers)
        for (int t = blockIdx.x; t < n_items && (ok || BAR_HANDOFF); t += gridDim.x) {
            const Item w = item_at(t);
            const Tile tl = tile_at(w);
            const int m = tl.m0 + row_in_tile;
            const int col0 = tl.n0 + sl * C::EPI_COLS;
            const bool vrow = m < tl.row_end;
            const bool vcol = col0 < N;
            float acc[C::CHUNKS][32];
#pragma unroll
            for (int cc = 0; cc < C::CHUNKS; ++cc)
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[cc][j] = 0.0f;
            for (int kb = w.kb0; kb < w.kb1; ++kb, ++kbg) {
                const uint32_t slot = kbg % SRING, sph = (kbg / SRING) & 1;
                const uint32_t b = kbg % C::NBUF, tph = (kbg / C::NBUF) & 1;
                (void)sph;   // the issuer waited for the scale slot before this K-block's MMAs
                bool got = !ok || __all_sync(0xFFFFFFFFu, ready) || mbar_wait(&ctl->tfull[b], tph, wait_ns);
                got = __all_sync(0xFFFFFFFFu, got);
                if (!got) ok = false;
                if (!ok) {
                    if constexpr (!BAR_HANDOFF) break;
                    // gave up: keep meeting the issuers on the buffer barriers
                    named_bar_sync(kBufBar0 + b, C::TBAR_THREADS);
                    continue;
                }
                // ROWB: sA here, the column scales inside the FMAs (the slot is
                // handed back after them)
                const float sc = ROWB ? ctl->ring[slot].sa[row_in_tile]
                                      : ctl->ring[slot].sa[row_in_tile] * ctl->ring[slot].sb[sbi];
                const float* sbv = sb_ring + slot * BN + sl * C::EPI_COLS;
                auto fma_chunk = [&](float (&a)[32], const uint32_t (&v)[32], int cc) {
                    if constexpr (ROWB)
                        fma32_packed_cols(a, v, sc, sbv + cc * 32);
                    else
                        fma32_packed(a, v, sc);
                };
                if constexpr (!ROWB) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->sempty[slot]);
                }
                tc_fence_after_sync();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * BN + sl * C::EPI_COLS;
                uint32_t v0[32], v1[32];
                // The next K-block's partial is probed right after this one's buffer is
                // released; the result is used at the top of the next iteration, so the
                // probe's latency (a barrier test costs ~200 cycles) overlaps the FMAs.
                const uint32_t kn = kbg + 1;
                if constexpr (C::CHUNKS == 1) {
                    tmem_ld_x32(taddr, v0);
                    tmem_ld_wait();
                    tc_fence_before_sync();
                    if constexpr (BAR_HANDOFF) {
                        named_bar_sync(kBufBar0 + b, C::TBAR_THREADS);   // buffer b goes back to its issuer
                    } else {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ctl->tempty[b]);
                    }
                    ready = mbar_test_wait(&ctl->tfull[kn % C::NBUF], (kn / C::NBUF) & 1);
                    fma_chunk(acc[0], v0, 0);
                } else {
                    // two round trips of two 32-column loads each
                    tmem_ld_x32(taddr, v0);
                    tmem_ld_x32(taddr + 32, v1);
                    tmem_ld_wait();
                    fma_chunk(acc[0], v0, 0);
                    fma_chunk(acc[1], v1, 1);
                    tmem_ld_x32(taddr + 64, v0);
                    tmem_ld_x32(taddr + 96, v1);
                    tmem_ld_wait();
                    // all four chunks are in registers: hand the buffer back
                    tc_fence_before_sync();
                    if constexpr (BAR_HANDOFF) {
                        named_bar_sync(kBufBar0 + b, C::TBAR_THREADS);   // buffer b goes back to its issuer
                    } else {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ctl->tempty[b]);
                    }
                    ready = mbar_test_wait(&ctl->tfull[kn % C::NBUF], (kn / C::NBUF) & 1);
                    fma_chunk(acc[2], v0, 2);
                    fma_chunk(acc[3], v1, 3);
                }
                if constexpr (ROWB) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->sempty[slot]);
                }
            }
            if (!ok) {
                if constexpr (BAR_HANDOFF) continue;   // keeps walking the schedule (barriers only)
                break;
            }
            if (!vcol) continue;
            if (w.parts > 1) {
                // A K-split tile of the last wave: publish this part of the
                // warp's 32 x EPI_COLS block, and the warp that completes the
                // block's ticket adds the parts in part order and stores it.
                const int wslot = (w.tile - split.n_full) * C::EPI_WARPS + (warp - EPI_WARP0);
                float* part0 = split.part + (size_t)(w.tile - split.n_full) * w.parts * (BM * BN) +
                               (size_t)(sl * C::EPI_COLS) * BM + q * 32 + lane;   // [part][col][row]
                float* dst = part0 + (size_t)w.part * (BM * BN);
#pragma unroll
                for (int cc = 0; cc < C::CHUNKS; ++cc)
#pragma unroll
                    for (int j = 0; j < 32; ++j) __stcg(dst + (cc * 32 + j) * BM, acc[cc][j]);
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) last = atomicAdd(&split.ticket[wslot], 1) == w.parts - 1;
                if (!__shfl_sync(0xFFFFFFFFu, last, 0)) continue;
                __threadfence();
                if (lane == 0) split.ticket[wslot] = 0;   // ready for the next call
                // every part, this warp's included, is read back and added in part
                // order, one 32-column chunk at a time
#pragma unroll
                for (int cc = 0; cc < C::CHUNKS; ++cc) {
                    float sum[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) sum[j] = 0.0f;
#pragma unroll 1
                    for (int pp = 0; pp < w.parts; ++pp) {
                        const float* src = part0 + (size_t)pp * (BM * BN) + (size_t)(cc * 32) * BM;
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __ldcg(src + j * BM);
#pragma unroll
                        for (int j = 0; j < 32; ++j) sum[j] += v[j];
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) acc[cc][j] = sum[j];
                }
            }
            if constexpr (BN == 256 && !GROUPED) {
                if (qo.q != nullptr) {
                    // Fused quantisation for the next layer: this warp holds, per row,
                    // the whole 128-column block col0 .. col0 + 127, so the row's
                    // amax needs no exchange.  Codes and scale are those the 1x128
                    // activation quantiser gives for the bf16-rounded outputs.
                    uint32_t pk[64];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
                                : "=r"(pk[16 * cc + e])
                                : "f"(acc[cc][2 * e + 1]), "f"(acc[cc][2 * e]));
                    uint32_t m2 = 0;
#pragma unroll
                    for (int e = 0; e < 64; ++e) m2 = absmax_bf16x2(m2, pk[e]);
                    const BlockScale bs = make_scale(absmax_pair_to_f32(m2), qo.pow2 != 0);
                    if (vrow) qo.s[(size_t)(col0 / 128) * qo.lds + m] = bs.s;
                    // the product cast for the warp unless a row's factor
                    // overflows (a per-pair test of the mode made this cast
                    // 3.5x slower: ~3600 against ~1050 cycles per half)
                    const bool all_mul = __all_sync(0xFFFFFFFFu, bs.mode == 1);
                    // two 32 x 64-byte halves through the warp's buffer (64-byte swizzle)
                    uint8_t* qbuf = epi_buf + (size_t)(warp - EPI_WARP0) * C::EPI_BUF_BYTES;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        if (lane == 0) bulk_wait_group_read<0>();
                        __syncwarp();
                        with_cast(all_mul, [&](auto cast) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int j0 = 32 * hf + 8 * k;   // first packed pair of this 16-byte piece
                                const uint2 c0 = quant8_as<decltype(cast)::mul>(
                                    make_uint4(pk[j0], pk[j0 + 1], pk[j0 + 2], pk[j0 + 3]), bs);
                                const uint2 c1 = quant8_as<decltype(cast)::mul>(
                                    make_uint4(pk[j0 + 4], pk[j0 + 5], pk[j0 + 6], pk[j0 + 7]), bs);
                                *reinterpret_cast<uint4*>(qbuf + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                                    make_uint4(c0.x, c0.y, c1.x, c1.y);
                            }
                        });
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tm_q, qbuf, col0 + 64 * hf, tl.m0 + q * 32);
                            bulk_commit_group();
                        }
                    }
                    if (!qo.write_c) continue;
                }
            }
            const int rows_here = min(tl.row_end - (tl.m0 + q * 32), 32);
            if (!GROUPED || rows_here == 32) {
                uint8_t* buf = epi_buf + (size_t)(warp - EPI_WARP0) * C::EPI_BUF_BYTES;
                // One 32 x 32 bf16 sub-block cc into shared memory: row `lane`,
                // 16-byte piece k at lane*64 + ((k ^ ((lane >> 1) & 3)) << 4), the
                // 64-byte swizzle of the output tensor map.  (Stores straight from
                // registers put one 16-byte piece of 32 rows in each instruction
                // and held these warps for thousands of cycles.)
                auto stage_block = [&](uint8_t* dst, int cc) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t p[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int col = 8 * k + 2 * e;
                            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(p[e]) : "f"(acc[cc][col + 1]), "f"(acc[cc][col]));
                        }
                        *reinterpret_cast<uint4*>(dst + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                            make_uint4(p[0], p[1], p[2], p[3]);
                    }
                };
                const int crow = (KGROUP ? tl.g * M : 0) + tl.m0 + q * 32;
                if constexpr (C::WHOLE_OUT) {
                    // all sub-blocks staged, then one TMA store each; they drain
                    // while the warp promotes the next tile
                    if (lane == 0) bulk_wait_group_read<0>();   // the previous tile's stores have read buf
                    __syncwarp();
#pragma unroll
                    for (int cc = 0; cc < C::CHUNKS; ++cc) stage_block(buf + cc * EPI_BLK_BYTES, cc);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
#pragma unroll
                        for (int cc = 0; cc < C::CHUNKS; ++cc)
                            tma_store_2d(&tm_c, buf + cc * EPI_BLK_BYTES, col0 + 32 * cc, crow);
                        bulk_commit_group();
                    }
                } else {
                    // one sub-block at a time through the warp's 2 KB buffer
#pragma unroll
                    for (int cc = 0; cc < C::CHUNKS; ++cc) {
                        if (lane == 0) bulk_wait_group_read<0>();   // the previous store has read buf
                        __syncwarp();
                        stage_block(buf, cc);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tm_c, buf, col0 + 32 * cc, crow);
                            bulk_commit_group();
                        }
                    }
                }
            } else if (vrow) {
                uint4* dst = reinterpret_cast<uint4*>(c + (size_t)m * ldc + col0);
#pragma unroll
                for (int j = 0; j < C::EPI_COLS / 8; ++j) {
                    uint32_t p[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = j * 8 + 2 * e;
                        const float lo = acc[col >> 5][col & 31], hi = acc[(col + 1) >> 5][(col + 1) & 31];
                        uint32_t r;
                        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
                        p[e] = r;
                    }
                    dst[j] = make_uint4(p[0], p[1], p[2], p[3]);
                }
            }
        }
        if (lane == 0) bulk_wait_group<0>();   // stores complete before the CTA exits
        if (!ok) {
            if (lane == 0) {
                record_timeout(status);
                *abort_flag = 1;
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, 512);
    }
}

template <int BN, bool GROUPED, bool ROWB = false, bool KGROUP = false>
cudaError_t launch(const GemmArgs& a, cudaStream_t st) {
    using C = Cfg<BN, ROWB>;
    static DeviceOnce attr_done;     // kernel attributes set on this device
    auto kern = k_gemm_promote<BN, GROUPED, ROWB, KGROUP>;
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_done.test(dev)) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        // The setmaxnreg split is only safe if the CTA really starts with
        // LAUNCH_REGS registers per thread; refuse to launch otherwise.
        if (C::SPLIT_REGS && fa.numRegs != C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<BN, ROWB>());
        if (e != cudaSuccess) return e;
        attr_done.set(dev);
    }
    const int64_t NT = (a.N + BN - 1) / BN;
    const int64_t tiles = GROUPED ? (((a.M + BM - 1) / BM) + a.G) * NT
                                  : ((a.M + BM - 1) / BM) * NT * (KGROUP ? a.G : 1);
    SplitTail split{0, 1, nullptr, nullptr};
    if (!GROUPED && !KGROUP) {
        const TailPlan tp = tail_plan(a.M, a.N, a.K, a.sm_count, BN, kPromoteMaxParts);
        if (tp.parts > 1 && a.workspace && a.ws_bytes >= tp.bytes) {
            split.n_full = (int)tp.n_full;
            split.parts = tp.parts;
            split.ticket = static_cast<int*>(a.workspace);
            split.part = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + tp.ticket_bytes);
        }
    }
    const int64_t items = work_items((int)tiles, split);
    const int grid = (int)(items < a.sm_count ? items : a.sm_count);
    kern<<<grid, C::THREADS, smem_bytes<BN, ROWB>(), st>>>(a.tm_a, a.tm_b, a.tm_c, a.tm_q, a.sa, a.ldsa, a.sb,
                                                           a.ldsb, static_cast<uint16_t*>(a.c), a.ldc, (int)a.M, (int)a.N,
                                                     (int)a.K, a.offsets, a.G, a.status, split, a.qout,
                                                     wait_bound(a), a.skip_first_load, (int)a.kg_tokens);
    return cudaGetLastError();
}

}  // namespace promote

// Split along K (dense).  With at least as many tiles as SMs, `grid` = SMs
// persistent CTAs: the first (tiles / grid) * grid tiles fill whole waves and
// the L left over are split into min(grid / L, KB / 8, max_parts) parts when
// that is at least 2 (promote: 4; MX, whose single accumulator is held while
// a part is written out: 2, and only when L >= grid / 4).  With fewer tiles
// than SMs (small M) every tile is split, into min(SMs / tiles, KB / 8,
// kSingleWaveMaxParts) parts, one per CTA, so that the parts fill the GPU.
TailPlan tail_plan(int64_t M, int64_t N, int64_t K, int sm_count, int bn, int max_parts) {
    TailPlan tp{0, 1, 0, 0};
    if (M <= 0 || bn <= 0 || sm_count <= 0) return tp;
    const int64_t tiles = ((M + 127) / 128) * ((N + bn - 1) / bn);
    int64_t full, left, parts;
    if (tiles < sm_count) {
        full = 0;
        left = tiles;
        parts = sm_count / tiles;
        if (parts > kSingleWaveMaxParts) parts = kSingleWaveMaxParts;
    } else {
        const int64_t grid = sm_count;
        full = (tiles / grid) * grid;
        left = tiles - full;
        if (left == 0) return tp;
        // MX: a last wave under a quarter of the SMs measured slower split than
        // whole (Llama qkv: 8 tiles left, 77 -> 80 us).
        if (max_parts <= kMxMaxParts && left * 4 < grid) return tp;
        parts = grid / left;
        if (parts > max_parts) parts = max_parts;
    }
    // At least 8 K-blocks per part: each extra part costs the warp that
    // completes a tile another 16 KB read of fp32 partials (8 parts of 4
    // K-blocks measured slower than no split).
    if (parts > (K / 128) / 8) parts = (K / 128) / 8;
    if (parts < 2) return tp;
    const int epi_warps = bn == 128 ? 16 : 8;
    if (left * epi_warps > kMaxTickets) return tp;   // more tickets than the region holds: no split
    tp.n_full = full;
    tp.parts = (int)parts;
    tp.ticket_bytes = kTicketBytes;
    tp.bytes = tp.ticket_bytes + (size_t)left * parts * 128 * bn * sizeof(float);
    return tp;
}

// Enough for the last-wave split of either large-M kernel (promote: its tile
// width; MX: 256).
size_t promote_workspace_bytes(int64_t M, int64_t N, int64_t K, int sm_count) {
    const size_t p = tail_plan(M, N, K, sm_count, promote_tile_n(M, N, K, 1), kPromoteMaxParts).bytes;
    const size_t x = tail_plan(M, N, K, sm_count, kMxTileN, kMxMaxParts).bytes;
    return p > x ? p : x;
}

cudaError_t launch_gemm_promote(const GemmArgs& a, cudaStream_t st) {
    if (a.M == 0) return cudaSuccess;
    const bool grouped = a.offsets != nullptr;
    if (a.ldsb > 0 && a.kgroup) {   // per-expert weight gradients over the experts' token blocks
        if (!grouped) return cudaErrorInvalidValue;
        if (a.bn == 128) return promote::launch<128, false, true, true>(a, st);
        if (a.bn == 256) return promote::launch<256, false, true, true>(a, st);
        return cudaErrorInvalidValue;
    }
    if (a.ldsb > 0) {   // a scale per B row (dense only)
        if (grouped) return cudaErrorInvalidValue;
        if (a.bn == 128) return promote::launch<128, false, true>(a, st);
        if (a.bn == 256) return promote::launch<256, false, true>(a, st);
        return cudaErrorInvalidValue;
    }
    if (a.bn == 128) return grouped ? promote::launch<128, true>(a, st) : promote::launch<128, false>(a, st);
    if (a.bn == 256) return grouped ? promote::launch<256, true>(a, st) : promote::launch<256, false>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace fp8bs
