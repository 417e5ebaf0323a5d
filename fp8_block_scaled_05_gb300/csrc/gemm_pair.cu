// Block-scaled FP8 GEMM with per-K-block promotion on CTA pairs
// (tcgen05 cta_group::2), dense, fp32 scales.
//
//   C[m, n] = bf16( sum_kb sA[kb, m] * sB[n/128, kb] * P[m, n, kb] ),
//   P[m, n, kb] = sum_{k in kb} dec(qa[m, k]) dec(qb[n, k])
//
// The same layer as the promote kernel (page "NVIDIA NeMo RL достигает
// ускорения на 48% благодаря сквозному обучению с точностью FP8",
// greentreeone.com, §Технический прорыв: FP8 linear layers with 1x128 and
// 128x128 block scales; ai.warp-studio.com end-to-end FP8 RL article,
// §FP8強化学習における精度と安定性の確保: higher-precision accumulation).
//
// Why pairs.  With fp32 scales every K-block's fp32 partial has to leave TMEM
// for the promotion warps before its buffer can take another K-block: commit,
// barrier, tcgen05.ld and release take longer than the 512 cycles one
// K-block of a 128 x 256 tile keeps the tensor core busy, and 512 TMEM
// columns hold only two such buffers.  A pair of CTAs computes a 256 x 128
// tile instead: each CTA holds its own 128 rows of A and 64 of the tile's 128
// B rows, and the leader's pair MMA (M 256, N 128) reads both CTAs' operands.
// Per SM the tensor core does the same work per byte of operands as a
// 128 x 256 tile, but each CTA's accumulator is 128 x 128, so TMEM holds four
// buffers and the promotion of a K-block has three K-blocks' worth of MMA
// time to hand its buffer back.
//
// Per CTA (both CTAs of a pair have the same warps; only the leader issues):
//   warp 0      TMA producer: its 128 A rows and 64 B rows per K-block into
//               an 8-stage ring; completion is signalled on the leader's
//               stage barrier, which the leader's producer arms with both
//               CTAs' bytes.
//   warps 1, 3  (leader) MMA issuers, alternate K-blocks: four pair MMAs
//               (M 256, N 128, K 32) into one of four 128-column TMEM
//               buffers, then commits multicast to both CTAs' stage-free and
//               buffer-full barriers.  Warp 1 of each CTA owns the pair's TMEM
//               allocation.
//   warp 2      scales: cp.async copies of each K-block's sA of this CTA's 128
//               rows and sB (one per weight block, or with per-row B scales
//               the tile's 128) into a shared-memory ring, well ahead.
//   warps 4-11  promotion: each reads 32 rows x 64 columns of a K-block's
//               partial (two tcgen05.ld), hands the buffer back to the leader
//               (a remote arrive), and adds the partial into registers times
//               the scale product RN(sA sB) (packed FMAs); per tile, bf16 through
//               a swizzled buffer and TMA stores.
// Every wait is bounded; a wait that runs out records a timeout in the status
// word and the kernel unwinds.  Both CTAs meet at a cluster barrier before the
// pair's TMEM is released and before either exits.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace pair {

constexpr int BMP = 256;                         // rows of a pair tile
constexpr int BM = 128;                          // rows per CTA
constexpr int BN = 128;                          // columns of a tile (one weight block)
constexpr int BNH = 64;                          // B rows held by each CTA
constexpr int BK = 128;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BNH * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 24 KB per CTA
constexpr int STAGES = 8;
constexpr int RING_BYTES = STAGES * STAGE_BYTES;
constexpr int NBUF = 4;                          // TMEM accumulator buffers of BN columns
constexpr int SRING = 8;                         // scale-product ring slots
constexpr int SCALE_WARP = 2;
constexpr int EPI_WARP0 = 4, EPI_WARPS = 8;
constexpr int EPI_COLS = 64;                     // columns per promotion warp
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
constexpr int EPI_BUF_BYTES = 32 * 64;           // one 32 x 32 bf16 output block per promotion warp
constexpr uint32_t IDESC = idesc_e4m3_f32(BMP, BN);
constexpr uint16_t PAIR_MASK = 0x3;
static_assert(NBUF * BN <= 512, "TMEM columns");

struct __align__(16) Ctrl {
    uint64_t full[STAGES];     // leader: operands of both CTAs landed
    uint64_t empty[STAGES];    // stage free again (multicast commit)
    uint64_t tfull[NBUF];      // accumulator buffer holds a finished K-block (multicast commit)
    uint64_t tempty[NBUF];     // leader: both CTAs' promotion warps have read the buffer
    uint64_t sfull[SRING];
    uint64_t sempty[SRING];
    uint64_t mma_done[2];
    uint32_t tmem_base;
    int32_t abort_flag;
    int32_t pad_[2];
};

// One K-block's scales: sA of this CTA's 128 rows, and the weight block's sB
// (128x128 blocks) or, with per-row B scales (ROWB), the tile's 128 column
// scales sb[kb * ldsb + n].
struct __align__(16) ScaleSlot {
    float sa[BM];
    float sbc[BN];
    float sb;
    float pad_[3];
};

constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + (size_t)RING_BYTES + (size_t)EPI_WARPS * EPI_BUF_BYTES +
                              sizeof(Ctrl) + (size_t)SRING * sizeof(ScaleSlot);
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");

__device__ __forceinline__ void record_timeout(int* status) {
    if (status) atomicCAS(status, 0, kStatusTimeout);
}

// Pair tile t -> first row of the pair (256 rows) and first column.  With
// M <= N the row tiles vary fastest (pairs running together share B tiles);
// with M > N the column tiles do.
__device__ __forceinline__ void pair_tile(int t, int M, int N, int& m0, int& n0) {
    const int MT = (M + BMP - 1) / BMP, NT = N / BN;
    int mt, nt;
    if (M > N) {
        mt = t / NT;
        nt = t % NT;
    } else {
        mt = t % MT;
        nt = t / MT;
    }
    m0 = mt * BMP;
    n0 = nt * BN;
}

// ROWB: sb holds a scale per B row, sb[kb * ldsb + n] (the weight-gradient
// form), so the promotion multiplies by a per-column scale product.
template <bool ROWB>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_c, const float* __restrict__ sa, int64_t ldsa,
                const float* __restrict__ sb, int64_t ldsb, int M, int N, int K, int* status, uint64_t wait_ns,
                int skip_first_load) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* epi_buf = smem + (size_t)RING_BYTES;   // 1024-byte aligned
    Ctrl* ctl = reinterpret_cast<Ctrl*>(epi_buf + (size_t)EPI_WARPS * EPI_BUF_BYTES);
    ScaleSlot* ring = reinterpret_cast<ScaleSlot*>(ctl + 1);   // 16-byte aligned

    const int warp = (int)warp_id(), lane = (int)lane_id();
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cl = (int)(blockIdx.x >> 1), ncl = (int)(gridDim.x >> 1);
    const int KB = K / BK;
    const int n_tiles = ((M + BMP - 1) / BMP) * (N / BN);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(&ctl->tfull[b], 1);
            mbar_init(&ctl->tempty[b], 2 * EPI_WARPS);
        }
        for (int s = 0; s < SRING; ++s) {
            mbar_init(&ctl->sfull[s], 32);        // every lane of the scale warp
            mbar_init(&ctl->sempty[s], EPI_WARPS);
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
        tmem_alloc_pair(&ctl->tmem_base, NBUF * BN);
        tmem_relinquish_pair();
    }
    // barriers initialised and TMEM allocated in both CTAs before any remote use
    tc_fence_before_sync();
    cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile int32_t* abort_flag = &ctl->abort_flag;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t full_leader = mapa_shared(smem_u32(&ctl->full[0]), 0);
            uint32_t it = 0;
            bool ok = true;
            for (int t = cl; t < n_tiles && ok; t += ncl) {
                int pm0, n0;
                pair_tile(t, M, N, pm0, n0);
                const int m0 = pm0 + (int)rank * BM, brow = n0 + (int)rank * BNH;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (!mbar_wait_cluster(&ctl->empty[s], ph ^ 1, wait_ns)) {
                        ok = false;
                        break;
                    }
                    if (skip_first_load && it == 0) continue;   // failure-path test: K-block 0 never lands
                    uint8_t* st = smem + (size_t)s * STAGE_BYTES;
                    if (leader) mbar_arrive_expect_tx(&ctl->full[s], 2 * STAGE_BYTES);
                    tma_load_2d_pair(st, &tm_a, full_leader + 8u * s, kb * BK, m0);
                    tma_load_2d_pair(st + A_BYTES, &tm_b, full_leader + 8u * s, kb * BK, brow);
                }
            }
            if (!ok) {
                record_timeout(status);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------ MMA issuers (leader)
        if (leader && lane == 0) {
            const uint32_t me = warp == 1 ? 0u : 1u;   // takes K-blocks it with it % 2 == me
            uint32_t it = 0;
            bool ok = true;
            for (int t = cl; t < n_tiles && ok; t += ncl) {
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    if ((it & 1) != me) continue;
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    const uint32_t b = it % NBUF, tph = (it / NBUF) & 1;
                    if (!mbar_wait_cluster(&ctl->full[s], ph, wait_ns) ||
                        !mbar_wait_cluster(&ctl->tempty[b], tph ^ 1, wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sA = smem_u32(smem + (size_t)s * STAGE_BYTES);
                    const uint64_t adesc = sdesc_kmajor_sw128(sA);
                    const uint64_t bdesc = sdesc_kmajor_sw128(sA + A_BYTES);
                    const uint32_t d = tmem_base + b * BN;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        umma_f8f6f4_pair(d, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), IDESC, k > 0 ? 1u : 0u);
                    umma_commit_pair_mc(&ctl->empty[s], PAIR_MASK);
                    umma_commit_pair_mc(&ctl->tfull[b], PAIR_MASK);
                }
            }
            if (!ok) {
                record_timeout(status);
                *abort_flag = 1;
            }
            // All MMAs this thread issued are complete before TMEM is released.
            umma_commit_pair(&ctl->mma_done[me]);
            mbar_wait(&ctl->mma_done[me], 0, wait_ns);
        }
        __syncwarp();
    } else if (warp == SCALE_WARP) {
        // ------------------------------------------------ scales
        // cp.async copies of each K-block's scales into a ring slot; their
        // completion arrives on the slot's barrier (one arrival per lane), so
        // this warp never waits for the data and runs up to SRING K-blocks
        // ahead of the promotion.
        uint32_t sit = 0;
        bool ok = true;
        for (int t = cl; t < n_tiles && ok; t += ncl) {
            int pm0, n0;
            pair_tile(t, M, N, pm0, n0);
            const int m0 = pm0 + (int)rank * BM;
            for (int kb = 0; kb < KB; ++kb, ++sit) {
                const uint32_t slot = sit % SRING, ph = (sit / SRING) & 1;
                bool got = mbar_wait(&ctl->sempty[slot], ph ^ 1, wait_ns);
                got = __all_sync(0xFFFFFFFFu, got);
                if (!got) {
                    ok = false;
                    break;
                }
                ScaleSlot& S = ring[slot];
                const float* sak = sa + (size_t)kb * ldsa;
#pragma unroll
                for (int r = 0; r < BM / 32; ++r) {
                    const int m = m0 + 32 * r + lane;
                    const bool v = m < M;
                    cp_async_4(&S.sa[32 * r + lane], v ? sak + m : sa, v);
                }
                if constexpr (ROWB) {
                    cp_async_16(&S.sbc[4 * lane], sb + (size_t)kb * ldsb + n0 + 4 * lane, true);   // N % 128 == 0
                } else if (lane == 0) {
                    cp_async_4(&S.sb, sb + (size_t)(n0 / 128) * KB + kb, true);
                }
                cp_async_arrive_noinc(&ctl->sfull[slot]);
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (!ok && lane == 0) {
            record_timeout(status);
            *abort_flag = 1;
        }
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------ promotion and output
        const int q = warp & 3;                      // TMEM lane quarter this warp may access
        const int h = (warp - EPI_WARP0) >> 2;       // column half of the tile
        const int row = q * 32 + lane;               // row within this CTA's 128
        const uint32_t tempty_leader = mapa_shared(smem_u32(&ctl->tempty[0]), 0);
        uint8_t* buf = epi_buf + (size_t)(warp - EPI_WARP0) * EPI_BUF_BYTES;
        uint32_t kbg = 0;
        bool ok = true;
        bool ready = false;   // tfull of K-block kbg already seen complete (early probe)
        for (int t = cl; t < n_tiles && ok; t += ncl) {
            int pm0, n0;
            pair_tile(t, M, N, pm0, n0);
            const int m0 = pm0 + (int)rank * BM;
            float acc[2][32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[cc][j] = 0.0f;
            for (int kb = 0; kb < KB; ++kb, ++kbg) {
                const uint32_t b = kbg % NBUF, tph = (kbg / NBUF) & 1;
                const uint32_t slot = kbg % SRING, sph = (kbg / SRING) & 1;
                bool got = __all_sync(0xFFFFFFFFu, ready) || mbar_wait_cluster(&ctl->tfull[b], tph, wait_ns);
                got = __all_sync(0xFFFFFFFFu, got && mbar_wait(&ctl->sfull[slot], sph, wait_ns));
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * BN + h * EPI_COLS;
                uint32_t v0[32], v1[32];
                tmem_ld_x32(taddr, v0);
                tmem_ld_x32(taddr + 32, v1);
                tmem_ld_wait();
                // the partial is in registers: hand the buffer back to the leader
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * b);
                {
                    const uint32_t kn = kbg + 1;
                    ready = mbar_test_wait_cluster(&ctl->tfull[kn % NBUF], (kn / NBUF) & 1);
                }
                const ScaleSlot& S = ring[slot];
                if constexpr (ROWB) {
                    // RN(sA * sB[n]) per column, then the FMA (as the 128x128 form
                    // rounds its single product once)
                    const float sar = S.sa[row];
                    fma32_packed_cols(acc[0], v0, sar, &S.sbc[h * EPI_COLS]);
                    fma32_packed_cols(acc[1], v1, sar, &S.sbc[h * EPI_COLS + 32]);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->sempty[slot]);
                } else {
                    const float sc = S.sa[row] * S.sb;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->sempty[slot]);
                    fma32_packed(acc[0], v0, sc);
                    fma32_packed(acc[1], v1, sc);
                }
            }
            if (!ok) break;
            // 32 x 32 blocks through this warp's 2 KB buffer and TMA stores (row
            // `lane`, 16-byte piece k at lane*64 + ((k ^ ((lane >> 1) & 3)) << 4):
            // the 64-byte swizzle of the output tensor map; rows past M are
            // clipped by the store).
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                if (lane == 0) bulk_wait_group_read<0>();   // the previous store has read buf
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t p[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = 8 * k + 2 * e;
                        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(p[e]) : "f"(acc[cc][col + 1]), "f"(acc[cc][col]));
                    }
                    *reinterpret_cast<uint4*>(buf + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                        make_uint4(p[0], p[1], p[2], p[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tm_c, buf, n0 + h * EPI_COLS + 32 * cc, m0 + q * 32);
                    bulk_commit_group();
                }
            }
        }
        if (lane == 0) bulk_wait_group<0>();   // stores complete before the CTA exits
        if (!ok && lane == 0) {
            record_timeout(status);
            *abort_flag = 1;
        }
    }

    // Both CTAs are done with the pair's TMEM and with each other's shared
    // memory (operands, barriers) before the allocation is released.
    tc_fence_before_sync();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, NBUF * BN);
    }
}

}  // namespace pair

namespace {
constexpr int kPairDevices = 64;
DeviceOnce g_pair_attr;
int g_pair_clusters[kPairDevices];   // co-resident pairs, per device
}  // namespace

// Both instantiations share the launch shape (threads, shared memory), so
// the occupancy of one stands for both.

int pair_max_clusters() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kPairDevices) return 0;
    if (!g_pair_attr.test(dev)) {
        if (cudaFuncSetAttribute(pair::k_gemm_pair<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)pair::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(pair::k_gemm_pair<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)pair::SMEM_BYTES) != cudaSuccess)
            return 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(pair::THREADS);
        cfg.dynamicSmemBytes = pair::SMEM_BYTES;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, pair::k_gemm_pair<false>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        g_pair_clusters[dev] = n;
        g_pair_attr.set(dev);
    }
    return g_pair_clusters[dev];
}

cudaError_t launch_gemm_pair(const GemmArgs& a, cudaStream_t st) {
    if (a.M == 0) return cudaSuccess;
    const int maxc = pair_max_clusters();
    if (maxc < 1) return cudaErrorInvalidConfiguration;
    const int64_t tiles = ((a.M + pair::BMP - 1) / pair::BMP) * (a.N / pair::BN);
    const int ncl = (int)(tiles < maxc ? tiles : maxc);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * ncl));
    cfg.blockDim = dim3(pair::THREADS);
    cfg.dynamicSmemBytes = pair::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (a.ldsb > 0)
        return cudaLaunchKernelEx(&cfg, pair::k_gemm_pair<true>, a.tm_a, a.tm_b, a.tm_c, a.sa, a.ldsa, a.sb, a.ldsb,
                                  (int)a.M, (int)a.N, (int)a.K, a.status, wait_bound(a), a.skip_first_load);
    return cudaLaunchKernelEx(&cfg, pair::k_gemm_pair<false>, a.tm_a, a.tm_b, a.tm_c, a.sa, a.ldsa, a.sb, (int64_t)0,
                              (int)a.M, (int)a.N, (int)a.K, a.status, wait_bound(a), a.skip_first_load);
}

}  // namespace fp8bs
