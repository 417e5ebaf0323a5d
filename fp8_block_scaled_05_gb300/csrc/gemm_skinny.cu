// Block-scaled FP8 GEMM for decode-sized M (1..256 tokens).
//
// Same operation as the large-M kernel (FP8 linear layer with 1x128 / 128x128
// block scales; page "NVIDIA NeMo RL достигает ускорения на 48% благодаря
// сквозному обучению с точностью FP8", greentreeone.com, §Технический
// прорыв), shaped for generation, where the step is bound by streaming the
// weights (upppp.jp NeMo RL FP8 article, §NeMo RLとは: the generation phase
// is the latency-critical one).
//
// The operands are swapped: 128 weight rows fill the MMA's M side and the
// tokens, padded to NT in {16, 32, 64, 128} (more than 128 tokens run as
// 128-token chunks on the grid's z dimension), are its N side, so
// D[n, m] = sum_k qb[n, k] qa[m, k] lands in TMEM with lane = weight row and
// column = token.  The K-blocks are split over `splits` CTAs per 128-row
// weight tile so that the weight stream is spread over every SM; the last
// CTA of a tile to finish (an atomic ticket in the workspace) adds the fp32
// partials of all splits in split order and writes bf16, so the result does
// not depend on which CTA finishes last.
//
// Per K-block the promotion multiplies column m by sA[kb, m] * sB[nb, kb]:
// sB is one value per CTA and K-block, the NT values of sA travel with the
// operands through the TMA ring (a 2-D fp32 tile, zero-filled past M).
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace skinny {

constexpr int BMW = 128;     // weight rows per CTA (MMA M)
constexpr int BK = 128;
constexpr int EPI_WARP0 = 4;

template <int NT>
struct Cfg {
    static constexpr int W_BYTES = BMW * BK;
    static constexpr int A_BYTES = NT * BK;
    static constexpr int STAGE_BYTES = W_BYTES + A_BYTES;
    static constexpr int STAGES = (200 * 1024) / STAGE_BYTES > 8 ? 8 : (200 * 1024) / STAGE_BYTES;
    // Promotion groups: group g takes the K-blocks i with i % NG == g, each
    // into its own accumulators (combined in group order at the end), so the
    // per-K-block barrier latency of one group overlaps the others' work.
    static constexpr int NG = NT <= 16 ? 4 : (NT <= 64 ? 2 : 1);
    static constexpr int SLICES = NT >= 128 ? 2 : 1;           // column slices per TMEM lane quarter
    static constexpr int GROUP_WARPS = 4 * SLICES;
    static constexpr int EPI_WARPS = NG * GROUP_WARPS;
    static constexpr int CPW = NT / SLICES;                    // token columns per promotion warp
    static constexpr int CHUNK = CPW >= 128 ? 16 : (CPW < 32 ? CPW : 32);
    static constexpr int SA_REGS = (CPW + 31) / 32;            // activation scales held per lane
    static constexpr int NBUF = (512 / NT) < (2 * NG > 4 ? 2 * NG : 4) ? (512 / NT) : (2 * NG > 4 ? 2 * NG : 4);
    static constexpr int TMEM_COLS = NBUF * NT < 32 ? 32 : NBUF * NT;
    static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
    static constexpr uint32_t IDESC = idesc_e4m3_f32(BMW, NT);
    static_assert(NBUF % NG == 0 && NBUF % 2 == 0 && NBUF <= 8, "buffer ownership");
    static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS <= 512, "TMEM allocation");
    static_assert((NG - 1) * NT * BMW * 4 <= STAGES * STAGE_BYTES, "group combine fits the drained ring");
};

constexpr int MAX_KB = 1024;   // K up to 131072: the CTA's weight scales are staged in shared memory

struct __align__(8) Ctrl {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t tfull[8];
    uint64_t tempty[8];
    uint64_t mma_done[2];
    uint32_t tmem_base;
    int32_t abort_flag;
    int32_t last;
    float sw[MAX_KB];          // sB[tile, kb_begin + i]
};

template <int NT>
constexpr size_t smem_bytes() {
    return 1024 + (size_t)Cfg<NT>::STAGES * Cfg<NT>::STAGE_BYTES + sizeof(Ctrl);
}

__device__ __forceinline__ void record_timeout(int* status) {
    if (status) atomicCAS(status, 0, kStatusTimeout);
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
    return r;
}

template <int CHUNK>
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[CHUNK]);
template <>
__device__ __forceinline__ void tmem_ld_chunk<32>(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld_x32(taddr, r); }
template <>
__device__ __forceinline__ void tmem_ld_chunk<16>(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld_x16(taddr, r); }

// Warp roles: 0 TMA producer; 1 and 2 MMA issuers (alternate K-blocks, warp 1
// owns TMEM); 3 idle; 4.. promotion groups of GROUP_WARPS warps.
template <int NT>
__global__ void __launch_bounds__(Cfg<NT>::THREADS, 1)
    k_gemm_skinny(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_a,
                  const float* __restrict__ sa, int64_t ldsa, const float* __restrict__ sb,
                  uint16_t* __restrict__ c, int64_t ldc, int M, int N, int K, int splits,
                  uint8_t* __restrict__ ws, int* status) {
    using C = Cfg<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + (size_t)C::STAGES * C::STAGE_BYTES);

    const int warp = (int)warp_id(), lane = (int)lane_id();
    const int KB = K / BK, NB = N / BMW;
    const int tile = blockIdx.x, split = blockIdx.y;
    // token chunk: tokens tok0 .. tok0 + NT - 1 (M > 128 runs as several chunks)
    const int tok0 = blockIdx.z * NT;
    const int Mc = M - tok0;                         // tokens of this chunk (may exceed NT)
    const int ptile = blockIdx.z * NB + tile;        // tile index of the partials and tickets
    const int kb_begin = (int)((int64_t)split * KB / splits);
    const int kb_end = (int)((int64_t)(split + 1) * KB / splits);
    const int nkb = kb_end - kb_begin;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < C::NBUF; ++b) {
            mbar_init(&ctl->tfull[b], 1);
            mbar_init(&ctl->tempty[b], C::GROUP_WARPS);
        }
        mbar_init(&ctl->mma_done[0], 1);
        mbar_init(&ctl->mma_done[1], 1);
        ctl->abort_flag = 0;
        mbar_init_fence();
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_a);
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile int32_t* abort_flag = &ctl->abort_flag;
    // The prologue above overlaps the previous kernel (programmatic dependent
    // launch); its outputs (the activation codes and scales, usually) are read
    // only from here on.  The next kernel may start its own prologue now.
    griddep_wait();
    griddep_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t evict_first = l2_policy_evict_first();
            uint32_t it = 0;
            bool ok = true;
            for (int i = 0; i < nkb; ++i, ++it) {
                const int kb = kb_begin + i;
                const uint32_t s = it % C::STAGES, ph = (it / C::STAGES) & 1;
                if (!mbar_wait(&ctl->empty[s], ph ^ 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                uint8_t* st = smem + (size_t)s * C::STAGE_BYTES;
                mbar_arrive_expect_tx(&ctl->full[s], C::W_BYTES + C::A_BYTES);
                tma_load_2d_hint(st, &tm_w, &ctl->full[s], kb * BK, tile * BMW, evict_first);
                tma_load_2d(st + C::W_BYTES, &tm_a, &ctl->full[s], kb * BK, tok0);
            }
            if (!ok) {
                record_timeout(status);
                *abort_flag = 1;
                const uint32_t n = it < (uint32_t)C::STAGES ? it : (uint32_t)C::STAGES;
                for (uint32_t j = it - n; j < it; ++j)
                    mbar_wait(&ctl->full[j % C::STAGES], (j / C::STAGES) & 1, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        if (lane == 0) {
            const int me = warp - 1;
            bool ok = true;
            for (int i = me; i < nkb; i += 2) {
                const uint32_t s = i % C::STAGES, ph = (i / C::STAGES) & 1;
                const uint32_t b = i % C::NBUF, tph = (i / C::NBUF) & 1;
                if (!mbar_wait(&ctl->full[s], ph, kWaitLimitNs) ||
                    !mbar_wait(&ctl->tempty[b], tph ^ 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t sw = smem_u32(smem + (size_t)s * C::STAGE_BYTES);
                const uint64_t adesc = sdesc_kmajor_sw128(sw);
                const uint64_t bdesc = sdesc_kmajor_sw128(sw + C::W_BYTES);
                const uint32_t d = tmem_base + b * NT;
#pragma unroll
                for (int k = 0; k < BK / 32; ++k)
                    umma_f8f6f4(d, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), C::IDESC, k > 0 ? 1u : 0u);
                umma_commit(&ctl->empty[s]);
                umma_commit(&ctl->tfull[b]);
            }
            if (!ok) {
                record_timeout(status);
                *abort_flag = 1;
            }
            umma_commit(&ctl->mma_done[me]);
            mbar_wait(&ctl->mma_done[me], 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp >= EPI_WARP0) {
        const int ew = warp - EPI_WARP0;
        const int grp = ew / C::GROUP_WARPS;
        const int q = warp & 3;
        const int sl = (ew % C::GROUP_WARPS) >> 2;   // which CPW-wide column slice
        const int col0 = sl * C::CPW;
        const int row = q * 32 + lane;               // weight row within the tile
        const int n = tile * BMW + row;
        float acc[C::CPW];
#pragma unroll
        for (int j = 0; j < C::CPW; ++j) acc[j] = 0.0f;
        // this CTA's weight scales, loaded once (a dependent global load per
        // K-block would put its latency on the critical path of the pipeline)
        const float* sbp = sb + (size_t)tile * KB + kb_begin;
        for (int i = ew * 32 + lane; i < nkb; i += 32 * C::EPI_WARPS) ctl->sw[i] = __ldg(sbp + i);
        named_bar_sync(1, 32 * C::EPI_WARPS);
        bool ok = true;
        bool ready = false;
        for (int i = grp; i < nkb; i += C::NG) {
            const int kb = kb_begin + i;
            const uint32_t b = i % C::NBUF, tph = (i / C::NBUF) & 1;
            // activation scales of this K-block: lane l holds column col0 + 32 r + l
            float sav[C::SA_REGS];
#pragma unroll
            for (int r = 0; r < C::SA_REGS; ++r) {
                const int col = col0 + 32 * r + lane;
                sav[r] = (col < Mc && 32 * r + lane < C::CPW) ? __ldg(sa + (size_t)kb * ldsa + tok0 + col) : 0.0f;
            }
            const float swv = ctl->sw[i];
            bool got = __all_sync(0xFFFFFFFFu, ready) || mbar_wait(&ctl->tfull[b], tph, kWaitLimitNs);
            got = __all_sync(0xFFFFFFFFu, got);
            if (!got) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * NT + col0;
#pragma unroll
            for (int cc = 0; cc < C::CPW / C::CHUNK; ++cc) {
                uint32_t v[C::CHUNK];
                tmem_ld_chunk<C::CHUNK>(taddr + cc * C::CHUNK, v);
                tmem_ld_wait();
                if (cc == C::CPW / C::CHUNK - 1) {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->tempty[b]);
                    const int in = i + C::NG;
                    ready = mbar_test_wait(&ctl->tfull[in % C::NBUF], (in / C::NBUF) & 1);
                }
#pragma unroll
                for (int j = 0; j < C::CHUNK; ++j) {
                    const int jj = cc * C::CHUNK + j;
                    const float sc = __shfl_sync(0xFFFFFFFFu, sav[jj >> 5], jj & 31) * swv;
                    acc[jj] = fmaf(__uint_as_float(v[j]), sc, acc[jj]);
                }
            }
        }
        if (!ok && lane == 0) {
            record_timeout(status);
            *abort_flag = 1;
        }
        // Every group is done with TMEM and every MMA has completed, so the
        // operand ring is drained: combine the groups through it, in group order.
        named_bar_sync(1, 32 * C::EPI_WARPS);
        ok = !*abort_flag;
        if (C::NG > 1) {
            float* xs = reinterpret_cast<float*>(smem);
            if (grp > 0) {
#pragma unroll
                for (int j = 0; j < C::CPW; ++j) xs[((size_t)(grp - 1) * NT + col0 + j) * BMW + row] = acc[j];
            }
            named_bar_sync(1, 32 * C::EPI_WARPS);
            if (grp == 0) {
                for (int g2 = 1; g2 < C::NG; ++g2) {
#pragma unroll
                    for (int j = 0; j < C::CPW; ++j) acc[j] += xs[((size_t)(g2 - 1) * NT + col0 + j) * BMW + row];
                }
            }
        }
        if (grp == 0 && ok) {
            if (splits == 1) {
                if (n < N) {
#pragma unroll
                    for (int j = 0; j < C::CPW; ++j) {
                        const int m = col0 + j;
                        if (m < Mc) c[(size_t)(tok0 + m) * ldc + n] = f32_to_bf16_rn(acc[j]);
                    }
                }
            } else {
                // Partials: ws layout [tickets: TC*NB int32 in the fixed ticket region]
                //                     [splits][TC*NB][NT][128] fp32 (row fastest, coalesced),
                // TC = gridDim.z token chunks.
                const int PT = gridDim.z * NB;
                int32_t* tickets = reinterpret_cast<int32_t*>(ws);
                float* part = reinterpret_cast<float*>(ws + kTicketBytes);
                float* mine = part + (((size_t)split * PT + ptile) * NT) * BMW;
#pragma unroll
                for (int j = 0; j < C::CPW; ++j) mine[(size_t)(col0 + j) * BMW + row] = acc[j];
                __threadfence();
                named_bar_sync(2, 32 * C::GROUP_WARPS);
                if (ew == 0 && lane == 0) {
                    const int prev = atomicAdd(&tickets[ptile], 1);
                    ctl->last = (prev == splits - 1);
                }
                named_bar_sync(2, 32 * C::GROUP_WARPS);
                if (ctl->last) {
                    __threadfence();
                    // Sum the splits in split order (this CTA's own partial is still in
                    // registers).  Per split and 32-column chunk all loads are issued
                    // before any add, so the chunk costs one L2 round trip.
                    constexpr int RC = C::CPW < 32 ? C::CPW : 32;
#pragma unroll
                    for (int j0 = 0; j0 < C::CPW; j0 += RC) {   // unrolled: acc stays in registers
                        if (col0 + j0 >= Mc) continue;
                        float tot[RC];
#pragma unroll
                        for (int j = 0; j < RC; ++j) tot[j] = 0.0f;
#pragma unroll 1
                        for (int sp = 0; sp < splits; ++sp) {
                            if (sp == split) {
#pragma unroll
                                for (int j = 0; j < RC; ++j) tot[j] += acc[j0 + j];
                            } else {
                                const float* p = part + (((size_t)sp * PT + ptile) * NT + col0 + j0) * BMW + row;
                                float v[RC];
#pragma unroll
                                for (int j = 0; j < RC; ++j) v[j] = __ldcg(p + (size_t)j * BMW);
#pragma unroll
                                for (int j = 0; j < RC; ++j) tot[j] += v[j];
                            }
                        }
                        if (n < N) {
#pragma unroll
                            for (int j = 0; j < RC; ++j) {
                                const int m = col0 + j0 + j;
                                if (m < Mc) c[(size_t)(tok0 + m) * ldc + n] = f32_to_bf16_rn(tot[j]);
                            }
                        }
                    }
                    if (ew == 0 && lane == 0) tickets[ptile] = 0;   // leave the ticket zero for the next call
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int NT>
cudaError_t launch_nt(const GemmArgs& a, cudaStream_t st) {
    using C = Cfg<NT>;
    static DeviceOnce attr_done;     // kernel attributes set on this device
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_done.test(dev)) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_skinny<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem_bytes<NT>());
        if (e != cudaSuccess) return e;
        attr_done.set(dev);
    }
    dim3 grid((unsigned)(a.N / BMW), (unsigned)a.splits, (unsigned)((a.M + NT - 1) / NT));
    if (pdl_for_tokens(a.M))   // programmatic dependent launch: measured faster up to 32 tokens only
        return launch_pdl(k_gemm_skinny<NT>, grid, dim3(C::THREADS), smem_bytes<NT>(), st, a.tm_b, a.tm_a, a.sa,
                          a.ldsa, a.sb, static_cast<uint16_t*>(a.c), a.ldc, (int)a.M, (int)a.N, (int)a.K,
                          a.splits, static_cast<uint8_t*>(a.workspace), a.status);
    k_gemm_skinny<NT><<<grid, C::THREADS, smem_bytes<NT>(), st>>>(
        a.tm_b, a.tm_a, a.sa, a.ldsa, a.sb, static_cast<uint16_t*>(a.c), a.ldc, (int)a.M, (int)a.N, (int)a.K,
        a.splits, static_cast<uint8_t*>(a.workspace), a.status);
    return cudaGetLastError();
}

}  // namespace skinny

int skinny_tile_n(int64_t M) {
    if (M <= 16) return 16;
    if (M <= 32) return 32;
    if (M <= 64) return 64;
    if (M <= 256) return 128;   // 129..256 tokens run as two 128-token chunks
    return 0;
}

static int64_t skinny_chunks(int64_t M) {
    const int nt = skinny_tile_n(M);
    return nt ? (M + nt - 1) / nt : 0;
}

int skinny_splits(int64_t M, int64_t N, int64_t K, int sm_count) {
    const int64_t tiles = (N / 128) * (skinny_chunks(M) > 0 ? skinny_chunks(M) : 1), KB = K / 128;
    if (tiles > kMaxTickets) return 1;   // more tiles than ticket words: no split
    int64_t s = sm_count / (tiles > 0 ? tiles : 1);
    if (s > KB / 2) s = KB / 2;     // at least two K-blocks per split
    if (s > 32) s = 32;
    if (s < 1) s = 1;
    return (int)s;
}

size_t skinny_workspace_bytes(int64_t M, int64_t N, int64_t K, int splits) {
    (void)K;
    const int nt = skinny_tile_n(M);
    if (nt == 0 || splits <= 1) return 0;
    const int64_t PT = (N / 128) * skinny_chunks(M);
    return kTicketBytes + (size_t)splits * PT * nt * 128 * sizeof(float);
}

cudaError_t launch_gemm_skinny(const GemmArgs& a, cudaStream_t st) {
    if (a.M == 0) return cudaSuccess;
    switch (skinny_tile_n(a.M)) {
        case 16: return skinny::launch_nt<16>(a, st);
        case 32: return skinny::launch_nt<32>(a, st);
        case 64: return skinny::launch_nt<64>(a, st);
        case 128: return skinny::launch_nt<128>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------------------
// Skinny GEMM on library-owned scratch (fp8_blockscaled_gemm_skinny_noalloc).
//
// The split-K tickets and fp32 partials live in a fixed array in device
// memory that belongs to the library, so the caller passes no workspace and
// nothing is allocated per call.  Every GPU that loads the library reserves
// the array until the process exits.  All calls share it: two calls that
// overlap on the GPU (different streams, no ordering between them) race on
// it.  The array keeps whatever the last call left; the tickets must start at
// zero, so they are cleared on the stream before every launch (the partials
// are always written before they are read).
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) uint8_t g_skinny_scratch[kNoAllocScratchBytes];

constexpr int kScratchDevices = 64;
std::mutex g_scratch_mu;
uint8_t* g_scratch_addr[kScratchDevices];   // device address of g_skinny_scratch, per device

// Device address of the scratch array on the current device.  In host code
// the array's name only stands for the symbol; the address the kernel needs
// comes from cudaGetSymbolAddress, taken once per device with that device
// current (the first call on a device does this).
cudaError_t scratch_address(uint8_t** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kScratchDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_skinny_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm_skinny_noalloc(GemmArgs a, cudaStream_t st) {
    if (a.M == 0) return cudaSuccess;
    const size_t need = skinny_workspace_bytes(a.M, a.N, a.K, a.splits);
    if (need > kNoAllocScratchBytes) return cudaErrorInvalidValue;   // the caller checked this already
    uint8_t* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return e;
    if (need > 0) {
        // ticket words of the split-K reduction (layout of the kernel's workspace)
        const size_t tickets = ((size_t)(a.N / 128) * skinny_chunks(a.M) * 4 + 255) & ~size_t(255);
        e = cudaMemsetAsync(scratch, 0, tickets, st);   // the part of the ticket region this call uses
        if (e != cudaSuccess) return e;
    }
    a.workspace = scratch;
    a.ws_bytes = kNoAllocScratchBytes;
    return launch_gemm_skinny(a, st);
}

}  // namespace fp8bs
