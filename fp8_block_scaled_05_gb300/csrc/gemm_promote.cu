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
// Design (one CTA per SM, persistent over output tiles of 128 x 256; three
// warpgroups):
//   warp 0      TMA producer: qa tile 128x128 and qb tile 256x128 per K-block
//               into a 4-stage shared-memory ring (128-byte swizzle).
//   warp 1      TMEM owner and MMA issuer: for every K-block, four
//               tcgen05.mma (M=128, N=256, K=32) into one of two 256-column
//               TMEM buffers, the first with accumulate = 0.
//   warps 4..11 promotion: each K-block's fp32 partial is read from TMEM
//               (tcgen05.ld) and added into registers with the scale product
//               sA*sB; the buffer is handed back right after the last read,
//               so the tensor core works on K-block kb+1 while kb is being
//               promoted.  Warp w owns TMEM lanes 32*(w%4).. and one
//               128-column half, i.e. one nb block with a single sB per
//               K-block.  The four 32-column reads of a K-block are pipelined
//               with the FMAs of the previous chunk.
//   Registers: the first warpgroup (producer, MMA, two idle warps) gives its
//   registers to the two promotion warpgroups (setmaxnreg 40 / 232, summing
//   to the 168 per thread the CTA is launched with), which hold 128 fp32
//   accumulators plus two 32-column staging chunks per thread.
// Every wait is bounded; a wait that runs out records a timeout in the status
// word and the kernel unwinds (waiting, bounded, for its own copies and MMAs).
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace promote {

constexpr int BM = 128, BN = kPromoteBN, BK = 128;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 384;
constexpr int EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;                 // first promotion warp (warpgroups 1 and 2)
constexpr int LAUNCH_REGS = 168;             // per thread at launch: 65536 / 384, rounded to 8
constexpr int REGS_CTRL = 40;                // warpgroup 0 after setmaxnreg.dec
constexpr int REGS_EPI = 232;                // warpgroups 1, 2 after setmaxnreg.inc
static_assert(128 * REGS_CTRL + 256 * REGS_EPI <= THREADS * LAUNCH_REGS, "register split exceeds the launch");
constexpr int TMEM_COLS = 512;
constexpr int MAX_GROUPS = 1024;
constexpr uint32_t IDESC = idesc_e4m3_f32(BM, BN);

struct __align__(8) Ctrl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int32_t n_tiles;
    int32_t abort_flag;
};

constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + (size_t)STAGES * STAGE_BYTES + sizeof(Ctrl) +
                              (size_t)3 * (MAX_GROUPS + 1) * sizeof(int32_t);

struct Tile {
    int32_t m0, row_end, brow, n0, g;
};

// Tile t -> coordinates.  Dense: m-tiles vary fastest so that CTAs running at
// the same time share the weight tile.  Grouped: tiles of expert g follow
// those of expert g-1; inside an expert, m-tiles vary fastest.
template <bool GROUPED>
__device__ __forceinline__ Tile decode_tile(int t, int M, int N, const int32_t* cum, const int32_t* glo,
                                            const int32_t* ghi, int G) {
    Tile r;
    if (!GROUPED) {
        const int MT = (M + BM - 1) / BM;
        const int mt = t % MT, nt = t / MT;
        r.m0 = mt * BM;
        r.row_end = M;
        r.brow = nt * BN;
        r.n0 = nt * BN;
        r.g = 0;
    } else {
        int lo = 0, hi = G;   // largest g with cum[g] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cum[mid] <= t) lo = mid; else hi = mid;
        }
        const int g = lo;
        const int local = t - cum[g];
        const int MTg = (ghi[g] - glo[g] + BM - 1) / BM;
        const int mt = local % MTg, nt = local / MTg;
        (void)N;
        r.m0 = glo[g] + mt * BM;
        r.row_end = ghi[g];
        r.brow = g * N + nt * BN;
        r.n0 = nt * BN;
        r.g = g;
    }
    return r;
}

__device__ __forceinline__ void record_timeout(int* status) {
    if (status) atomicCAS(status, 0, kStatusTimeout);
}

template <bool GROUPED>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_promote(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const float* __restrict__ sa, int64_t ldsa, const float* __restrict__ sb,
                   uint16_t* __restrict__ c, int64_t ldc, int M, int N, int K,
                   const int32_t* __restrict__ offsets, int G, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + (size_t)STAGES * STAGE_BYTES);
    int32_t* cum = reinterpret_cast<int32_t*>(ctl + 1);
    int32_t* glo = cum + (MAX_GROUPS + 1);
    int32_t* ghi = glo + (MAX_GROUPS + 1);

    const int warp = (int)warp_id(), lane = (int)lane_id();
    const int KB = K / BK;
    const int NT = (N + BN - 1) / BN;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->tfull[b], 1);
            mbar_init(&ctl->tempty[b], EPI_WARPS);
        }
        mbar_init(&ctl->mma_done, 1);
        ctl->abort_flag = 0;
        mbar_init_fence();
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 2) {
        if (GROUPED) {
            // Per-expert row ranges (clamped to [0, M]) and the running tile count.
            int carry = 0;
            if (lane == 0) cum[0] = 0;
            for (int g0 = 0; g0 < G; g0 += 32) {
                const int g = g0 + lane;
                int lo = 0, hi = 0, tiles = 0;
                if (g < G) {
                    lo = min(max(offsets[g], 0), M);
                    hi = min(max(offsets[g + 1], lo), M);
                    tiles = ((hi - lo + BM - 1) / BM) * NT;
                    glo[g] = lo;
                    ghi[g] = hi;
                }
                int incl = tiles;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                    if (lane >= o) incl += v;
                }
                if (g < G) cum[g + 1] = carry + incl;
                carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
            }
            if (lane == 0) ctl->n_tiles = carry;
        } else if (lane == 0) {
            ctl->n_tiles = ((M + BM - 1) / BM) * NT;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = ctl->tmem_base;
    const int n_tiles = ctl->n_tiles;
    volatile int32_t* abort_flag = &ctl->abort_flag;

    if (warp < EPI_WARP0) regs_dealloc<REGS_CTRL>();
    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile<GROUPED>(t, M, N, cum, glo, ghi, G);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (!mbar_wait(&ctl->empty[s], ph ^ 1, kWaitLimitNs) || *abort_flag) {
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
                record_timeout(status);
                *abort_flag = 1;
                // Let the copies already issued land before the CTA can exit.
                const uint32_t n = it < STAGES ? it : STAGES;
                for (uint32_t j = it - n; j < it; ++j)
                    mbar_wait(&ctl->full[j % STAGES], (j / STAGES) & 1, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, kbg = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                for (int kb = 0; kb < KB; ++kb, ++it, ++kbg) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    const uint32_t b = kbg & 1, tph = (kbg >> 1) & 1;
                    if (!mbar_wait(&ctl->tempty[b], tph ^ 1, kWaitLimitNs) ||
                        !mbar_wait(&ctl->full[s], ph, kWaitLimitNs) || *abort_flag) {
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
                        umma_f8f6f4(d, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), IDESC, k > 0 ? 1u : 0u);
                    umma_commit(&ctl->empty[s]);
                    umma_commit(&ctl->tfull[b]);
                }
            }
            if (!ok) {
                record_timeout(status);
                *abort_flag = 1;
            }
            // All MMAs this thread issued are complete before TMEM is released.
            umma_commit(&ctl->mma_done);
            mbar_wait(&ctl->mma_done, 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------ promotion epilogue
        regs_alloc<REGS_EPI>();
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int h = (warp - EPI_WARP0) >> 2;  // 128-column half of the 256-wide tile
        const int row_in_tile = q * 32 + lane;
        const int NB = N / 128;
        uint32_t kbg = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
            const Tile tl = decode_tile<GROUPED>(t, M, N, cum, glo, ghi, G);
            const int m = tl.m0 + row_in_tile;
            const bool vrow = m < tl.row_end;
            const int nb = tl.n0 / 128 + h;
            const bool vcol = nb < NB;
            const float* sbp = sb + ((size_t)tl.g * NB + (vcol ? nb : 0)) * KB;
            const float* sap = sa + m;
            float acc[4][32];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[cc][j] = 0.0f;
            // scales prefetched two K-blocks ahead
            float sa0 = vrow ? __ldg(sap) : 0.0f, sb0 = vcol ? __ldg(sbp) : 0.0f;
            float sa1 = (vrow && KB > 1) ? __ldg(sap + ldsa) : 0.0f, sb1 = (vcol && KB > 1) ? __ldg(sbp + 1) : 0.0f;
            for (int kb = 0; kb < KB; ++kb, ++kbg) {
                const float sc = sa0 * sb0;
                sa0 = sa1;
                sb0 = sb1;
                if (kb + 2 < KB) {
                    sa1 = vrow ? __ldg(sap + (size_t)(kb + 2) * ldsa) : 0.0f;
                    sb1 = vcol ? __ldg(sbp + kb + 2) : 0.0f;
                }
                const uint32_t b = kbg & 1, tph = (kbg >> 1) & 1;
                bool got = mbar_wait(&ctl->tfull[b], tph, kWaitLimitNs) && !*abort_flag;
                got = __all_sync(0xFFFFFFFFu, got);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * BN + h * 128;
                uint32_t v0[32], v1[32];
                tmem_ld_x32(taddr, v0);
                tmem_ld_wait();
                tmem_ld_x32(taddr + 32, v1);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[0][j] = fmaf(__uint_as_float(v0[j]), sc, acc[0][j]);
                tmem_ld_wait_after(acc[0]);
                tmem_ld_x32(taddr + 64, v0);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[1][j] = fmaf(__uint_as_float(v1[j]), sc, acc[1][j]);
                tmem_ld_wait_after(acc[1]);
                tmem_ld_x32(taddr + 96, v1);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[2][j] = fmaf(__uint_as_float(v0[j]), sc, acc[2][j]);
                tmem_ld_wait_after(acc[2]);
                // all four chunks are in registers: hand the buffer back
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty[b]);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[3][j] = fmaf(__uint_as_float(v1[j]), sc, acc[3][j]);
            }
            if (!ok) break;
            if (vrow && vcol) {
                uint4* dst = reinterpret_cast<uint4*>(c + (size_t)m * ldc + tl.n0 + h * 128);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
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
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace promote

cudaError_t launch_gemm_promote(const GemmArgs& a, cudaStream_t st) {
    using namespace promote;
    if (a.M == 0) return cudaSuccess;
    static int attr_done_mask[2] = {0, 0};   // bit per device ordinal (< 32)
    const bool grouped = a.offsets != nullptr;
    auto kern = grouped ? k_gemm_promote<true> : k_gemm_promote<false>;
    int dev = 0;
    cudaGetDevice(&dev);
    if (!(attr_done_mask[grouped] & (1 << (dev & 31)))) {
        // The setmaxnreg split is only safe if the CTA really starts with
        // LAUNCH_REGS registers per thread; refuse to launch otherwise.
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done_mask[grouped] |= 1 << (dev & 31);
    }
    const int64_t NT = (a.N + BN - 1) / BN;
    int64_t tiles = grouped ? (((a.M + BM - 1) / BM) + a.G) * NT : ((a.M + BM - 1) / BM) * NT;
    const int grid = (int)(tiles < a.sm_count ? tiles : a.sm_count);
    kern<<<grid, THREADS, SMEM_BYTES, st>>>(*a.tm_a, *a.tm_b, a.sa, a.ldsa, a.sb,
                                            static_cast<uint16_t*>(a.c), a.ldc, (int)a.M, (int)a.N,
                                            (int)a.K, a.offsets, a.G, a.status);
    return cudaGetLastError();
}

}  // namespace fp8bs
