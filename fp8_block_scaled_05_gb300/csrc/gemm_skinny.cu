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
// 128-token chunks), are its N side, so D[n, m] = sum_k qb[n, k] qa[m, k]
// lands in TMEM with lane = weight row and column = token.
//
// Work division (stream-K): the K-blocks of all output tiles (128 weight rows
// x one token chunk), taken tile after tile, form U = tiles * K/128 units;
// CTA c of P takes units [c U / P, (c+1) U / P), so every CTA streams the
// same number of weight bytes (to within one K-block).  P is a whole multiple
// of the tile count when that fills at least three quarters of the SMs, else
// the SM count.  A CTA's range is cut into segments at tile boundaries.
// A segment that covers a whole tile writes its bf16 output directly; the
// others write an fp32 partial, and the CTA that completes a tile's ticket
// adds the partials of all the tile's segments in CTA order and writes bf16,
// so the result does not depend on which CTA finishes last.
//
// Per K-block the promotion multiplies token column m by sA[kb, m] *
// sB[nb, kb]: a scale warp copies each K-block's scales (cp.async) into a
// shared-memory ring well ahead of the MMAs, and the promotion warps read them
// with broadcast loads, form the products with packed multiplies and fold
// them in with packed FMAs.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdlib>
#include <mutex>

#include "codec.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace skinny {

constexpr int BMW = 128;     // weight rows per tile (MMA M)
constexpr int BK = 128;
constexpr int SCALE_WARP = 3;
constexpr int EPI_WARP0 = 4;
constexpr int SRING = 16;    // scale ring slots (K-blocks of scales in flight)
constexpr int MIN_UNITS = 4; // K-blocks per CTA, at least (when the problem allows)

template <int NT>
struct Cfg {
    static constexpr int W_BYTES = BMW * BK;
    static constexpr int A_BYTES = NT * BK;
    static constexpr int STAGE_BYTES = W_BYTES + A_BYTES;
    // Promotion groups: group g takes the K-blocks i with i % NG == g, each
    // into its own accumulators (added in group order at each segment's end),
    // so a K-block's barrier waits and TMEM round trip overlap the other
    // groups' K-blocks.
    static constexpr int NG = NT <= 16 ? 4 : (NT <= 64 ? 2 : 1);
    static constexpr int SLICES = NT >= 128 ? 2 : 1;           // column slices per TMEM lane quarter
    static constexpr int GROUP_WARPS = 4 * SLICES;
    static constexpr int EPI_WARPS = NG * GROUP_WARPS;
    static constexpr int CPW = NT / SLICES;                    // token columns per promotion warp
    static constexpr int CHUNK = CPW < 32 ? CPW : 32;          // columns per tcgen05.ld
    static constexpr int NBUF = (512 / NT) < 8 ? (512 / NT) : 8;
    static constexpr int TMEM_COLS = NBUF * NT < 32 ? 32 : NBUF * NT;
    static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
    static constexpr int COMBINE_BYTES = (NG - 1) * NT * BMW * 4;   // groups 1.. hand their sums to group 0
    static constexpr int STAGES_FIT = (220 * 1024 - COMBINE_BYTES - 10 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    // reduction: columns per round and segments loaded per round (their
    // loads in flight together); SB * RC values live per thread
    static constexpr int RC = CPW < 32 ? CPW : (THREADS > 256 ? 16 : 32);
    static constexpr int SB = 4;
    static constexpr uint32_t IDESC = idesc_e4m3_f32(BMW, NT);
    static_assert(NBUF % 2 == 0 && NBUF % NG == 0 && NBUF <= 8, "buffer ownership");
    static_assert(SRING % NG == 0, "scale slot ownership");
    static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS <= 512, "TMEM allocation");
    static_assert(CPW % CHUNK == 0 && CPW % 4 == 0 && CPW % RC == 0, "column split");
    static_assert(STAGES >= 4, "operand ring depth");
};

// One K-block's scales: sA[kb, tok0 + j] for the token columns j, and the
// weight block's sB[tile, kb].
struct __align__(16) ScaleSlot {
    float sa[128];
    float sb;
    float pad_[3];
};

struct __align__(16) Ctrl {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t tfull[8];
    uint64_t tempty[8];
    uint64_t sfull[SRING];
    uint64_t sempty[SRING];
    uint64_t mma_done[2];
    uint32_t tmem_base;
    int32_t abort_flag;
    int32_t last;
    int32_t pad_;
    ScaleSlot ring[SRING];
};

template <int NT>
constexpr size_t smem_bytes() {
    return 1024 + (size_t)Cfg<NT>::STAGES * Cfg<NT>::STAGE_BYTES + (size_t)Cfg<NT>::COMBINE_BYTES + sizeof(Ctrl);
}
static_assert(smem_bytes<16>() <= 232448 && smem_bytes<32>() <= 232448 && smem_bytes<64>() <= 232448 &&
                  smem_bytes<128>() <= 232448,
              "shared memory per CTA");

// The stream-K partition: U units (K-blocks, tile-major) over P CTAs.
struct Part {
    int64_t U;
    int32_t P;
    int32_t KB;       // K-blocks per tile
    int32_t T;        // tiles per token chunk (N / 128)
};

// One CTA's segment: global tile tg (chunk * T + tile), K-blocks [kb0, kb1).
struct Seg {
    int32_t tg, kb0, kb1;
};

__device__ __forceinline__ bool next_seg(int64_t& u, int64_t u1, int KB, Seg& s) {
    if (u >= u1) return false;
    s.tg = (int32_t)(u / KB);
    const int64_t base = (int64_t)s.tg * KB;
    s.kb0 = (int32_t)(u - base);
    s.kb1 = (int32_t)((u1 - base) < KB ? (u1 - base) : KB);
    u = base + s.kb1;
    return true;
}

// The CTA whose range holds unit x: the largest c with floor(c U / P) <= x.
__device__ __forceinline__ int cta_of_unit(int64_t x, const Part& p) {
    return (int)(((x + 1) * p.P - 1) / p.U);
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
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t* r);
template <>
__device__ __forceinline__ void tmem_ld_chunk<32>(uint32_t taddr, uint32_t* r) {
    tmem_ld_x32(taddr, *reinterpret_cast<uint32_t(*)[32]>(r));
}
template <>
__device__ __forceinline__ void tmem_ld_chunk<16>(uint32_t taddr, uint32_t* r) {
    tmem_ld_x16(taddr, *reinterpret_cast<uint32_t(*)[16]>(r));
}

// a0 = fma(v0, s0, a0), a1 = fma(v1, s1, a1) as one packed fma.rn.f32x2 (each
// lane an IEEE fma, bit-identical to fmaf).
__device__ __forceinline__ void fma2(float& a0, float& a1, uint32_t v0, uint32_t v1, float s0, float s1) {
    uint64_t a, x, s;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(v0), "r"(v1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(s) : "f"(s0), "f"(s1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(x), "l"(s));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
}

// Warp roles: 0 TMA producer; 1 and 2 MMA issuers (alternate K-blocks, warp 1
// owns TMEM); 3 scale copies; 4.. promotion (EPI_WARPS warps, warp w reads
// TMEM lane quarter w % 4 and a CPW-wide column slice).
template <int NT>
__global__ void __launch_bounds__(Cfg<NT>::THREADS, 1)
    k_gemm_skinny(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_a,
                  const float* __restrict__ sa, int64_t ldsa, const float* __restrict__ sb,
                  uint16_t* __restrict__ c, int64_t ldc, int M, int N, Part part, uint8_t* __restrict__ ws,
                  int* status, uint64_t wait_ns, int skip_first_load) {
    using C = Cfg<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* combine = reinterpret_cast<float*>(smem + (size_t)C::STAGES * C::STAGE_BYTES);   // [NG-1][NT][128]
    Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + (size_t)C::STAGES * C::STAGE_BYTES + C::COMBINE_BYTES);

    const int warp = (int)warp_id(), lane = (int)lane_id();
    const int KB = part.KB, T = part.T;
    const int cta = blockIdx.x;
    const int64_t u0 = (int64_t)cta * part.U / part.P;
    const int64_t u1 = (int64_t)(cta + 1) * part.U / part.P;
    const bool one_chunk = M <= NT;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < C::NBUF; ++b) {
            mbar_init(&ctl->tfull[b], 1);
            mbar_init(&ctl->tempty[b], C::GROUP_WARPS);   // read by one group
        }
        for (int s = 0; s < SRING; ++s) {
            mbar_init(&ctl->sfull[s], 32);     // every lane of the scale warp
            mbar_init(&ctl->sempty[s], C::GROUP_WARPS);
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
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            // A weight tile is read once when there is one token chunk (leave
            // it out of L2's way); with two chunks the second read should hit L2.
            const uint64_t evict_first = l2_policy_evict_first();
            uint32_t it = 0;
            bool ok = true;
            int64_t u = u0;
            Seg sg;
            while (ok && next_seg(u, u1, KB, sg)) {
                const int chunk = sg.tg / T, tile = sg.tg % T;
                for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                    const uint32_t s = it % C::STAGES, ph = (it / C::STAGES) & 1;
                    if (!mbar_wait(&ctl->empty[s], ph ^ 1, wait_ns)) {
                        ok = false;
                        break;
                    }
                    if (skip_first_load && it == 0) continue;   // failure-path test: K-block 0 never lands
                    uint8_t* st = smem + (size_t)s * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&ctl->full[s], C::W_BYTES + C::A_BYTES);
                    if (one_chunk)
                        tma_load_2d_hint(st, &tm_w, &ctl->full[s], kb * BK, tile * BMW, evict_first);
                    else
                        tma_load_2d(st, &tm_w, &ctl->full[s], kb * BK, tile * BMW);
                    tma_load_2d(st + C::W_BYTES, &tm_a, &ctl->full[s], kb * BK, chunk * NT);
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
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------ MMA issuers
        if (lane == 0) {
            const uint32_t me = warp - 1;
            const uint32_t nkb = (uint32_t)(u1 - u0);   // K-blocks of this CTA, all segments
            bool ok = true;
            for (uint32_t i = me; i < nkb; i += 2) {
                const uint32_t s = i % C::STAGES, ph = (i / C::STAGES) & 1;
                const uint32_t b = i % C::NBUF, tph = (i / C::NBUF) & 1;
                if (!mbar_wait(&ctl->full[s], ph, wait_ns) ||
                    !mbar_wait(&ctl->tempty[b], tph ^ 1, wait_ns)) {
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
            mbar_wait(&ctl->mma_done[me], 0, wait_ns);
        }
        __syncwarp();
    } else if (warp == SCALE_WARP) {
        // ------------------------------------------------ scales
        // cp.async copies of each K-block's activation scales and weight scale
        // into a ring slot; the copies' completion arrives on the slot's
        // barrier (one arrival per lane), so this warp never waits for the
        // data and runs up to SRING K-blocks ahead of the promotion.
        uint32_t it = 0;
        bool ok = true;
        int64_t u = u0;
        Seg sg;
        while (ok && next_seg(u, u1, KB, sg)) {
            const int tok0 = (sg.tg / T) * NT, tile = sg.tg % T;
            for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                const uint32_t slot = it % SRING, ph = (it / SRING) & 1;
                bool got = mbar_wait(&ctl->sempty[slot], ph ^ 1, wait_ns);
                got = __all_sync(0xFFFFFFFFu, got);
                if (!got) {
                    ok = false;
                    break;
                }
                ScaleSlot& S = ctl->ring[slot];
                const float* sak = sa + (size_t)kb * ldsa + tok0;
#pragma unroll
                for (int r = 0; r < (NT + 31) / 32; ++r) {
                    const int j = 32 * r + lane;
                    if (j < NT) {
                        const bool v = tok0 + j < M;
                        cp_async_4(&S.sa[j], v ? sak + j : sa, v);
                    }
                }
                if (lane == 0) cp_async_4(&S.sb, sb + (size_t)tile * KB + kb, true);
                cp_async_arrive_noinc(&ctl->sfull[slot]);
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (!ok && lane == 0) {
            record_timeout(status);
            *abort_flag = 1;
        }
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------ promotion
        const int ew = warp - EPI_WARP0;
        const int grp = ew / C::GROUP_WARPS;
        const int q = warp & 3;
        const int col0 = ((ew % C::GROUP_WARPS) >> 2) * C::CPW;   // this warp's token columns
        const int row = q * 32 + lane;                           // weight row within the tile
        int32_t* tickets = reinterpret_cast<int32_t*>(ws);
        float* parts = reinterpret_cast<float*>(ws + kTicketBytes);
        uint32_t kbg = 0;
        bool ok = true;
        bool ready = false;   // tfull of this group's next K-block already seen complete (early probe)
        int64_t u = u0;
        Seg sg;
        while (next_seg(u, u1, KB, sg)) {
            const int tok0 = (sg.tg / T) * NT, tile = sg.tg % T;
            const int n = tile * BMW + row;
            float acc[C::CPW];
#pragma unroll
            for (int j = 0; j < C::CPW; ++j) acc[j] = 0.0f;
            for (int kb = sg.kb0; kb < sg.kb1 && ok; ++kb, ++kbg) {
                if ((int)(kbg % C::NG) != grp) continue;
                const uint32_t b = kbg % C::NBUF, tph = (kbg / C::NBUF) & 1;
                const uint32_t slot = kbg % SRING, sph = (kbg / SRING) & 1;
                bool got = __all_sync(0xFFFFFFFFu, ready) || mbar_wait(&ctl->tfull[b], tph, wait_ns);
                got = __all_sync(0xFFFFFFFFu, got && mbar_wait(&ctl->sfull[slot], sph, wait_ns));
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * NT + col0;
                uint32_t v[C::CPW];
#pragma unroll
                for (int cc = 0; cc < C::CPW / C::CHUNK; ++cc) tmem_ld_chunk<C::CHUNK>(taddr + cc * C::CHUNK, v + cc * C::CHUNK);
                tmem_ld_wait();
                // the partial is in registers: hand the buffer back, probe this
                // group's next K-block
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty[b]);
                {
                    const uint32_t kn = kbg + C::NG;
                    ready = mbar_test_wait(&ctl->tfull[kn % C::NBUF], (kn / C::NBUF) & 1);
                }
                // scale products RN(sA * sB) per token column (packed multiplies;
                // every lane reads the same addresses), then the packed FMAs
                const ScaleSlot& S = ctl->ring[slot];
                const float swv = S.sb;
#pragma unroll
                for (int g = 0; g < C::CPW / 4; ++g) {
                    const float4 a4 = *reinterpret_cast<const float4*>(&S.sa[col0 + 4 * g]);
                    float p0, p1, p2, p3;
                    mul2(a4.x, a4.y, swv, p0, p1);
                    mul2(a4.z, a4.w, swv, p2, p3);
                    fma2(acc[4 * g], acc[4 * g + 1], v[4 * g], v[4 * g + 1], p0, p1);
                    fma2(acc[4 * g + 2], acc[4 * g + 3], v[4 * g + 2], v[4 * g + 3], p2, p3);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->sempty[slot]);
            }
            // Every promotion warp reaches this barrier, failed or not, and all
            // take the same decision: give up together if any wait ran out.
            if (named_bar_red_or(1, 32 * C::EPI_WARPS, !ok || *abort_flag != 0)) {
                ok = false;
                break;
            }
            if (C::NG > 1) {
                // groups 1.. hand their sums to group 0, which adds them in group order
                if (grp > 0) {
#pragma unroll
                    for (int j = 0; j < C::CPW; ++j) combine[((size_t)(grp - 1) * NT + col0 + j) * BMW + row] = acc[j];
                }
                named_bar_sync(1, 32 * C::EPI_WARPS);
                if (grp > 0) continue;   // group 0 finishes the segment
                for (int g2 = 1; g2 < C::NG; ++g2) {
#pragma unroll
                    for (int j = 0; j < C::CPW; ++j) acc[j] += combine[((size_t)(g2 - 1) * NT + col0 + j) * BMW + row];
                }
            }
            if (sg.kb0 == 0 && sg.kb1 == KB) {
                // the whole tile in this segment: bf16 straight out
#pragma unroll
                for (int j = 0; j < C::CPW; ++j) {
                    const int m = tok0 + col0 + j;
                    if (m < M) c[(size_t)m * ldc + n] = f32_to_bf16_rn(acc[j]);
                }
                continue;
            }
            // A piece of a tile: publish the fp32 partial in slot (cta + tile),
            // unique per (CTA, tile) pair, laid out [column][row].  The CTA that
            // completes the tile's ticket adds every segment in CTA order.
            const int c_first = cta_of_unit((int64_t)sg.tg * KB, part);
            const int c_last = cta_of_unit((int64_t)sg.tg * KB + KB - 1, part);
            {
                float* mine = parts + ((size_t)(cta + sg.tg) * NT + col0) * BMW + row;
#pragma unroll
                for (int j = 0; j < C::CPW; ++j) __stcg(mine + (size_t)j * BMW, acc[j]);
            }
            __threadfence();
            named_bar_sync(2, 32 * C::GROUP_WARPS);
            if (ew == 0 && lane == 0) {
                const int prev = atomicAdd(&tickets[sg.tg], 1);
                ctl->last = (prev == c_last - c_first);
            }
            named_bar_sync(2, 32 * C::GROUP_WARPS);
            if (!ctl->last) continue;
            __threadfence();
            // Every segment's partial is in the workspace (this CTA's too, still
            // in L2): add them in CTA order, SB segments' loads in flight per round.
#pragma unroll 1
            for (int j0 = 0; j0 < C::CPW; j0 += C::RC) {
                if (tok0 + col0 + j0 >= M) break;
                float tot[C::RC];
#pragma unroll
                for (int j = 0; j < C::RC; ++j) tot[j] = 0.0f;
#pragma unroll 1
                for (int cs = c_first; cs <= c_last; cs += C::SB) {
                    float ld[C::SB][C::RC];
#pragma unroll
                    for (int k = 0; k < C::SB; ++k) {
                        const int c2 = cs + k <= c_last ? cs + k : c_last;   // past the end: re-read the last, unused
                        const float* p = parts + ((size_t)(c2 + sg.tg) * NT + col0 + j0) * BMW + row;
#pragma unroll
                        for (int j = 0; j < C::RC; ++j) ld[k][j] = __ldcg(p + (size_t)j * BMW);
                    }
#pragma unroll
                    for (int k = 0; k < C::SB; ++k) {
                        if (cs + k > c_last) break;
#pragma unroll
                        for (int j = 0; j < C::RC; ++j) tot[j] += ld[k][j];
                    }
                }
#pragma unroll
                for (int j = 0; j < C::RC; ++j) {
                    const int m = tok0 + col0 + j0 + j;
                    if (m < M) c[(size_t)m * ldc + n] = f32_to_bf16_rn(tot[j]);
                }
            }
            if (ew == 0 && lane == 0) tickets[sg.tg] = 0;   // leave the ticket zero for the next call
        }
        if (!ok && lane == 0) {
            record_timeout(status);
            *abort_flag = 1;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace skinny

int skinny_tile_n(int64_t M) {
    if (M <= 16) return 16;
    if (M <= 32) return 32;
    if (M <= 64) return 64;
    if (M <= 256) return 128;   // 129..256 tokens run as two 128-token chunks
    return 0;
}

namespace {

struct SkinnyPlan {
    int nt = 0;
    int64_t tiles = 0;     // output tiles, all token chunks
    int64_t U = 0;         // units (K-blocks of all tiles)
    int P = 1;             // CTAs
    bool split = false;    // some tile is shared by several CTAs
};

SkinnyPlan make_plan(int64_t M, int64_t N, int64_t K, int sm_count) {
    SkinnyPlan p;
    p.nt = skinny_tile_n(M);
    if (p.nt == 0 || N < 128 || K < 128) return p;
    const int64_t KB = K / 128;
    p.tiles = (N / 128) * ((M + p.nt - 1) / p.nt);
    p.U = p.tiles * KB;
    int64_t P = p.U / skinny::MIN_UNITS;
    if (P > sm_count) P = sm_count;
    // A whole number of CTAs per tile when that still fills three quarters of
    // the SMs: every CTA's range then lies inside one tile (one segment, one
    // partial), which measured faster than ranges straddling tile boundaries
    // (M 64, N 4096, K 14336: 28.7 against 33.3 us).
    if (p.tiles <= sm_count) {
        const int64_t aligned = p.tiles * (sm_count / p.tiles);
        if (4 * aligned >= 3 * (int64_t)sm_count && aligned <= p.U / skinny::MIN_UNITS) P = aligned;
    }
    // FP8BS_SKINNY_CTAS=n caps the CTA count (for tuning); with n a multiple
    // of the tile count every CTA's range stays inside one tile
    static const int64_t cap = [] {
        const char* e = std::getenv("FP8BS_SKINNY_CTAS");
        return e ? (int64_t)std::atoll(e) : (int64_t)0;
    }();
    if (cap > 0 && P > cap) P = cap;
    if (P < 1) P = 1;
    if (p.tiles > kMaxTickets) P = p.tiles;   // more tiles than ticket words: whole tiles per CTA
    p.P = (int)P;
    for (int64_t c = 1; c < P && !p.split; ++c) p.split = ((c * p.U / P) % KB) != 0;
    return p;
}

}  // namespace

int skinny_splits(int64_t M, int64_t N, int64_t K, int sm_count) { return make_plan(M, N, K, sm_count).P; }

size_t skinny_workspace_bytes(int64_t M, int64_t N, int64_t K, int splits) {
    (void)splits;
    // the plan depends only on the sizes and the CTA count; recompute it from
    // the CTA count the caller was given by skinny_splits
    SkinnyPlan p;
    p.nt = skinny_tile_n(M);
    if (p.nt == 0 || N < 128 || K < 128 || splits < 1) return 0;
    const int64_t KB = K / 128;
    p.tiles = (N / 128) * ((M + p.nt - 1) / p.nt);
    p.U = p.tiles * KB;
    for (int64_t c = 1; c < splits && !p.split; ++c) p.split = ((c * p.U / splits) % KB) != 0;
    if (!p.split) return 0;
    return kTicketBytes + (size_t)(splits + p.tiles - 1) * p.nt * 128 * sizeof(float);
}

namespace skinny {

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
    Part p;
    p.KB = (int32_t)(a.K / BK);
    p.T = (int32_t)(a.N / BMW);
    p.U = (int64_t)p.T * ((a.M + NT - 1) / NT) * p.KB;
    p.P = a.splits;
    if (p.P < 1 || p.P > p.U) return cudaErrorInvalidValue;
    dim3 grid((unsigned)p.P);
    if (pdl_for_tokens(a.M))   // programmatic dependent launch: measured faster up to 32 tokens only
        return launch_pdl(k_gemm_skinny<NT>, grid, dim3(C::THREADS), smem_bytes<NT>(), st, a.tm_b, a.tm_a, a.sa,
                          a.ldsa, a.sb, static_cast<uint16_t*>(a.c), a.ldc, (int)a.M, (int)a.N, p,
                          static_cast<uint8_t*>(a.workspace), a.status, wait_bound(a),
                          a.skip_first_load);
    k_gemm_skinny<NT><<<grid, C::THREADS, smem_bytes<NT>(), st>>>(a.tm_b, a.tm_a, a.sa, a.ldsa, a.sb,
                                                                   static_cast<uint16_t*>(a.c), a.ldc, (int)a.M,
                                                                   (int)a.N, p, static_cast<uint8_t*>(a.workspace),
                                                                   a.status, wait_bound(a), a.skip_first_load);
    return cudaGetLastError();
}

}  // namespace skinny

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
        // ticket words of the split reduction, one per output tile (layout of
        // the kernel's workspace): the part of the ticket region this call uses
        const int nt = skinny_tile_n(a.M);
        const size_t tiles = (size_t)(a.N / 128) * (size_t)((a.M + nt - 1) / nt);
        const size_t tickets = (tiles * 4 + 255) & ~size_t(255);
        e = cudaMemsetAsync(scratch, 0, tickets, st);
        if (e != cudaSuccess) return e;
    }
    a.workspace = scratch;
    a.ws_bytes = kNoAllocScratchBytes;
    return launch_gemm_skinny(a, st);
}

}  // namespace fp8bs
