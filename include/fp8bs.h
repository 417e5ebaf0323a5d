/*
 * fp8bs.h -- C ABI of the GB300 (sm_103a) block-scaled FP8 linear layer.
 *
 * The operation (page "NVIDIA NeMo RL достигает ускорения на 48% благодаря
 * сквозному обучению с точностью FP8", greentreeone.com, §Технический
 * прорыв): linear layers compute on FP8 E4M3 codes, with activations
 * quantised in 1x128 blocks and weights in 128x128 blocks, each block
 * carrying its own scale; attention, normalisation and non-linearities stay
 * bf16 and are not part of this library.  The scale is recomputed from the
 * block's current amax on every call because the policy's weights change
 * after each optimizer step (upppp.jp NeMo RL FP8 article,
 * §KVキャッシュとAttentionにも拡張).  A power-of-two scale option exists
 * (upppp.jp article, §設定方法).  Accumulation is kept in higher precision
 * than the FP8 operands (ai.warp-studio.com end-to-end FP8 RL article,
 * §FP8強化学習における精度と安定性の確保).
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" must be device (or managed) memory of the
 *    current CUDA device; the caller owns every buffer, the library never
 *    frees or keeps them.  Sizes and leading dimensions are in ELEMENTS.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  A returned FP8_OK means "validated and
 *    enqueued", not "finished".
 *  - Arguments are validated on the host before anything touches the GPU:
 *    a call that returns an error has enqueued nothing.
 *  - Kernels never trap.  Every wait inside a kernel has a time limit; a
 *    wait that runs out records FP8_ERR_TIMEOUT in a per-device status word
 *    (read it with fp8_last_device_status) and the kernel returns.
 *  - Non-finite inputs (NaN, Inf) are outside the contract: the calls run,
 *    the codes they produce are unspecified.
 *  - E4M3 is the OCP OFP8 "fn" variant: bias 7, no infinities, NaN = S.1111.111,
 *    largest finite magnitude 448.  Conversion rounds to nearest, ties to
 *    even, and saturates to +-448.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FP8BS_API __attribute__((visibility("default")))
#else
#define FP8BS_API
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *fp8_stream_t;

typedef enum {
    FP8_OK = 0,
    FP8_ERR_NULL = 1,            /* a required pointer is NULL */
    FP8_ERR_SHAPE = 2,           /* sizes out of range, or a leading dimension too small */
    FP8_ERR_ALIGN = 3,           /* a pointer or a row pitch breaks the 16-byte rule */
    FP8_ERR_SCALE_MODE = 4,      /* unknown scale mode or flag bits */
    FP8_ERR_WORKSPACE = 5,       /* workspace missing or smaller than fp8_gemm_workspace_size() */
    FP8_ERR_ARCH = 6,            /* no CUDA device, or the current device is not sm_103 */
    FP8_ERR_CUDA = 7,            /* a CUDA runtime/driver call failed (launch, descriptor) */
    FP8_ERR_TIMEOUT = 8,         /* a kernel wait ran out of time (device status word only) */
    FP8_ERR_NOT_IMPLEMENTED = 9  /* the requested path is not built */
} fp8_status;

/*
 * Scale rules.  Each block has a stored scale s (dequantisation: x ~ dec(q) s)
 * and a cast factor r: the codes are q = e4m3(RN_fp32(x r)), rounded to
 * nearest even and saturated at +-448.  The pages give the scale as amax/448
 * and leave open whether the cast divides by it or multiplies by the
 * reciprocal; the library multiplies (the usual FP8 cast), with r =
 * RN_fp32(448 / amax).  Where that reciprocal overflows fp32 (amax below
 * 448 * 2^-128) the cast divides, q = e4m3(RN_fp32(x / s)).
 */
typedef enum {
    /* s = RN_fp32(amax / 448), r = RN_fp32(448 / amax); an all-zero block
     * gets s = r = 1. */
    FP8_SCALE_FP32_AMAX = 0,
    /* s = 2^e, e = ceil(log2(amax / 448)) clamped to [-127, 127], r = 2^-e
     * (so x r is the exact quotient x / s); an all-zero block gets s = 1. */
    FP8_SCALE_POW2 = 1
} fp8_scale_mode;

/* GEMM flags. */
#define FP8_GEMM_SCALES_POW2   0x1u  /* caller promises every sA, sB is an exact power of two
                                        in [2^-127, 2^127] (as FP8_SCALE_POW2 produces); lets the
                                        hardware block-scaled (UE8M0) path run */
#define FP8_GEMM_SCALES_E8     0x2u  /* sA and sB are UE8M0 bytes (2^(b-127), as the _e8 quantisers
                                        write them) at the indices of the fp32 arrays; MX path only
                                        (AUTO picks it; PROMOTE and SKINNY return NOT_IMPLEMENTED) */
#define FP8_GEMM_PATH_MASK     0xF0u /* kernel selection; 0 = automatic */
#define FP8_GEMM_PATH_AUTO     0x00u
#define FP8_GEMM_PATH_PROMOTE  0x10u /* large-M kernel, fp32 scale promotion per K-block */
#define FP8_GEMM_PATH_MX       0x20u /* large-M kernel, hardware UE8M0 block scaling (needs SCALES_POW2) */
#define FP8_GEMM_PATH_SKINNY   0x30u /* M <= 256: weights as the MMA's M side, K split over all SMs */

/*
 * 1x128 activation quantisation.
 *
 *   for every row m < M and K-block kb < K/128:
 *     amax      = max_{k in kb} |x[m, k]|
 *     s[kb, m]  = scale(amax)           (see fp8_scale_mode)
 *     q[m, k]   = e4m3( RN_fp32(x[m, k] * r(amax)) )   (see fp8_scale_mode)
 *
 * x   device, bf16 [M, K] row-major, row pitch ldx (>= K, ldx % 8 == 0, x 16-byte aligned)
 * q   device, uint8 E4M3 codes [M, K] row-major, row pitch ldq (>= K, ldq % 16 == 0, 16-byte aligned)
 * s   device, fp32 [K/128][lds]: the scale of row m, K-block kb is s[kb * lds + m]
 *     (K-block-major so that a GEMM reads the scales of consecutive rows
 *     contiguously); lds >= M, lds % 4 == 0, 16-byte aligned.
 * M >= 0 (M == 0 is a no-op; M < 2^31), 0 < K <= 2^26 and K % 128 == 0.
 */
FP8BS_API fp8_status fp8_quant_act_1x128(const void *x, int64_t M, int64_t K, int64_t ldx,
                               uint8_t *q, int64_t ldq, float *s, int64_t lds,
                               fp8_scale_mode mode, fp8_stream_t stream);

/*
 * 1x128 activation quantisation with power-of-two scales stored as UE8M0
 * bytes (OCP Microscaling E8M0: byte b means 2^(b - 127)): the codes are
 * those of fp8_quant_act_1x128(..., FP8_SCALE_POW2) and s[kb * lds + m] is the
 * byte of the scale that call writes as fp32 -- a quarter of the scale bytes,
 * in the form the MX GEMM path takes (FP8_GEMM_SCALES_E8).
 * s  device, uint8 [K/128][lds] (lds >= M, lds % 4 == 0; any address);
 * everything else as fp8_quant_act_1x128.
 */
FP8BS_API fp8_status fp8_quant_act_1x128_e8(const void *x, int64_t M, int64_t K, int64_t ldx,
                                            uint8_t *q, int64_t ldq, uint8_t *s, int64_t lds,
                                            fp8_stream_t stream);

/*
 * 128x128 weight quantisation with power-of-two scales stored as UE8M0 bytes:
 * codes as fp8_quant_weight_128x128(..., FP8_SCALE_POW2), s uint8 [N/128][K/128]
 * (contiguous, any address).
 */
FP8BS_API fp8_status fp8_quant_weight_128x128_e8(const void *w, int64_t N, int64_t K, int64_t ldw,
                                                 uint8_t *q, int64_t ldq, uint8_t *s,
                                                 fp8_stream_t stream);

/*
 * 128x128 weight quantisation (run after every optimizer step).
 *
 *   for every tile (nb, kb), nb < N/128, kb < K/128:
 *     amax        = max over the 128x128 tile of |w|
 *     s[nb, kb]   = scale(amax)
 *     q[n, k]     = e4m3( RN_fp32(w[n, k] * r(amax of the tile)) )
 *
 * w   device, bf16 [N, K] row-major, row pitch ldw (>= K, ldw % 8 == 0, 16-byte aligned)
 * q   device, uint8 [N, K] row-major, row pitch ldq (>= K, ldq % 16 == 0, 16-byte aligned)
 * s   device, fp32 [N/128][K/128] row-major, contiguous, 4-byte aligned (so that
 *     one expert's block of a [G][N/128][K/128] array can be passed)
 * N, K > 0, both multiples of 128.
 */
FP8BS_API fp8_status fp8_quant_weight_128x128(const void *w, int64_t N, int64_t K, int64_t ldw,
                                    uint8_t *q, int64_t ldq, float *s,
                                    fp8_scale_mode mode, fp8_stream_t stream);

/*
 * A layer's two quantisations in one launch: exactly fp8_quant_act_1x128(x,
 * M, K, ...) and fp8_quant_weight_128x128(w, N, K, ...) (same codes, same
 * scales, same layouts and argument rules), the activations and weights of a
 * linear layer y = x W^T sharing K.  One grid covers both, so the two HBM
 * streams share one ramp-up and one tail instead of paying each (the weights
 * are re-quantised every step, greentreeone.com NeMo RL FP8 page,
 * §Реальные прирост производительности).  M may be 0 (weights only).
 */
FP8BS_API fp8_status fp8_quant_act_weight(const void *x, int64_t M, int64_t K, int64_t ldx,
                                          uint8_t *qa, int64_t ldqa, float *sa, int64_t ldsa,
                                          const void *w, int64_t N, int64_t ldw, uint8_t *qw,
                                          int64_t ldqw, float *sw, fp8_scale_mode mode,
                                          fp8_stream_t stream);

/*
 * Training-side operands.  The pages run FP8 through training as well as
 * generation (greentreeone.com NeMo RL FP8 page, §Технический прорыв;
 * ai.warp-studio.com end-to-end FP8 RL article, opening section: activations,
 * gradients and updates).  For a linear layer y = x W^T the backward GEMMs
 * are dX = dY W (dgrad) and dW = dY^T X (wgrad); every operand is blocked by
 * 128 along the dimension its GEMM reduces over:
 *   dgrad: A = dY codes from fp8_quant_act_1x128 (blocks along the output
 *          features), B = W^T codes from fp8_quant_weight_128x128_t, run
 *          through fp8_blockscaled_gemm with M = tokens, N = in-features,
 *          K = out-features;
 *   wgrad: A = dY^T and B = X^T codes from fp8_quant_act_128x1 (128x1 blocks:
 *          128 tokens of one column), run through fp8_blockscaled_gemm_wgrad
 *          with M = out-features, N = in-features, K = tokens.
 */

/*
 * 128x1 activation quantisation, written transposed (the wgrad operand):
 *
 *   for every column k < K and token block mb < M/128:
 *     amax          = max_{m in mb} |x[m, k]|
 *     st[mb, k]     = scale(amax)
 *     qt[k, m]      = e4m3( RN_fp32(x[m, k] * r(amax of the block)) )
 *
 * i.e. exactly what fp8_quant_act_1x128 writes for x^T.  Optionally (q and s
 * both non-NULL) the same pass also writes the 1x128 codes and scales of x
 * itself, as fp8_quant_act_1x128(x) would: one read of x for both layouts.
 *
 * x   device, bf16 [M, K] row-major, row pitch ldx (>= K, % 8 == 0)
 * qt  device, uint8 [K, Mp] row-major (token-contiguous), row pitch ldqt (>= Mp, % 16 == 0),
 *     Mp = M rounded up to a multiple of 128
 * st  device, fp32 [Mp/128][ldst]: the scale of column k, token block mb is
 *     st[mb * ldst + k] (ldst >= K, % 4 == 0) -- the layout a GEMM's sA/sB takes
 * q, s  optional (both NULL, or both set): as fp8_quant_act_1x128 (ldq, lds)
 * M >= 0 (0 is a no-op); a last token block of fewer than 128 rows is padded
 * with zero rows (they change no block's amax and add nothing to dW; their
 * codes in qt are zero), Mp/128 <= 65535; K > 0, K % 128 == 0.  Pointers
 * 16-byte aligned.
 */
FP8BS_API fp8_status fp8_quant_act_128x1(const void *x, int64_t M, int64_t K, int64_t ldx,
                                         uint8_t *qt, int64_t ldqt, float *st, int64_t ldst,
                                         uint8_t *q, int64_t ldq, float *s, int64_t lds,
                                         fp8_scale_mode mode, fp8_stream_t stream);

/*
 * 128x128 weight quantisation written for W^T (the dgrad operand): the
 * blocks of W^T are W's blocks transposed, with the same scales, so
 *
 *   qt[k, n]       = q[n, k]        (q as fp8_quant_weight_128x128 defines it)
 *   st[kb, nb]     = s[nb, kb]
 *
 * Optionally (q and s both non-NULL) W's own codes and scales come from the
 * same pass, exactly as fp8_quant_weight_128x128 writes them.
 *
 * w   device, bf16 [N, K] row-major, row pitch ldw (>= K, % 8 == 0)
 * qt  device, uint8 [K, N] row-major, row pitch ldqt (>= N, % 16 == 0)
 * st  device, fp32 [K/128][N/128] row-major, contiguous
 * q, s  optional: uint8 [N, K] (ldq >= K, % 16 == 0) and fp32 [N/128][K/128]
 * N, K > 0, both multiples of 128, N/128 <= 65535.  Pointers 16-byte aligned.
 */
FP8BS_API fp8_status fp8_quant_weight_128x128_t(const void *w, int64_t N, int64_t K, int64_t ldw,
                                                uint8_t *q, int64_t ldq, float *s,
                                                uint8_t *qt, int64_t ldqt, float *st,
                                                fp8_scale_mode mode, fp8_stream_t stream);

/*
 * Block-scaled FP8 GEMM, C = A * B^T ("TN": both operands K-major):
 *
 *   C[m, n] = bf16_RN( sum_kb  sA[kb, m] * sB[n/128, kb] * P[m, n, kb] ),
 *   P[m, n, kb] = sum_{k in kb} dec(qa[m, k]) * dec(qb[n, k])
 *
 * Promote and skinny paths: each K-block's partial P is accumulated in fp32
 * by the tensor cores and promoted into an fp32 running sum with the scale
 * product.  MX path (power-of-two scales only): the tensor core applies the
 * scales itself as UE8M0 block scale factors and accumulates the whole K range
 * in fp32.  The order of the fp32 additions is not specified; results agree
 * with an exact evaluation to fp32 accumulation error plus bf16 output
 * rounding.
 *
 * Path choice with FP8_GEMM_PATH_AUTO: M <= 128 -> skinny; otherwise MX when
 * FP8_GEMM_SCALES_POW2 is set, else promote.  FP8_GEMM_PATH_MX without
 * FP8_GEMM_SCALES_POW2 returns FP8_ERR_SCALE_MODE.  On the MX path a scale that
 * is not a power of two in [2^-127, 2^127] breaks the promise: the output is
 * unspecified and the device status word reads FP8_ERR_SCALE_MODE.
 *
 * qa  device, uint8 [M, K], row pitch lda (>= K, % 16 == 0)
 * sa  device, fp32 [K/128][ldsa] as written by fp8_quant_act_1x128 (ldsa >= M, % 4 == 0)
 * qb  device, uint8 [N, K], row pitch ldb (>= K, % 16 == 0)
 * sb  device, fp32 [N/128][K/128] contiguous, as written by fp8_quant_weight_128x128
 * c   device, bf16 [M, N], row pitch ldc (>= N, % 8 == 0)
 * M >= 0 (0 is a no-op), N, K > 0 and multiples of 128.  All pointers 16-byte aligned.
 * flags: FP8_GEMM_SCALES_POW2 | one FP8_GEMM_PATH_* value.
 * workspace: device scratch of fp8_gemm_workspace_size(M, N, K, 1) bytes (may be
 *     NULL when that size is 0).  Its first 64 KiB hold split-K semaphores
 *     that must be zero before the first use; every completed call leaves them
 *     zero again (allocate it zero-filled once and reuse it, for any shapes).
 *     Calls that share a workspace must not run concurrently.
 *     - Skinny path (M <= 256): required when the size is not 0 (the
 *       K-blocks of all output tiles are shared evenly by up to one CTA per
 *       SM, so a tile may be computed in pieces whose fp32 partials are then
 *       added in CTA order); smaller or NULL returns FP8_ERR_WORKSPACE.
 *     - Promote and MX paths: optional.  With it, when the output tiles do
 *       not fill whole waves of the GPU's SMs, the tiles of the last wave (or,
 *       with fewer tiles than SMs, every tile) are split along K and their
 *       fp32 parts added in a fixed order; without it (or if it is too small)
 *       every tile is computed whole.
 */
FP8BS_API fp8_status fp8_blockscaled_gemm(const uint8_t *qa, int64_t lda, const float *sa, int64_t ldsa,
                                const uint8_t *qb, int64_t ldb, const float *sb,
                                void *c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                uint32_t flags, void *workspace, size_t ws_bytes,
                                fp8_stream_t stream);

/*
 * Mixture-of-experts weight gradients in two launches per operand pair
 * (end-to-end FP8 training of the MoE models the recipe covers: upppp.jp
 * NeMo RL FP8 article, §まとめ; greentreeone.com page, §Технический прорыв).
 * For each expert g with token rows offsets[g] .. offsets[g+1]-1 of the
 * expert-sorted dY [T, M] and X [T, N]:  dW_g [M, N] = dY_g^T X_g, every
 * operand quantised in 128x1 blocks of that expert's own tokens (the last
 * block padded with zero rows).
 *
 * fp8_quant_act_128x1_grouped: the 128x1 codes of each expert's tokens,
 * transposed, in padded token slots: with P_g = sum_{g' < g} ceil(M_g' / 128),
 * expert g's blocks are slots 128 P_g .. 128 P_{g+1} - 1, i.e. qt columns,
 * and their scales rows P_g .. P_{g+1} - 1 of st.  Slots past P_G are not
 * written.
 *   x        device, bf16 [T, K] (row pitch ldx), tokens sorted by expert
 *   offsets  device, int32 [G+1] (as fp8_blockscaled_grouped_gemm); G <= 1024
 *   qt       device, uint8 [K][ldqt], ldqt >= 128 * (ceil(T/128) + G), % 16 == 0
 *   st       device, fp32 [ceil(T/128) + G][ldst], ldst >= K, % 4 == 0
 *   K % 128 == 0; ceil(T/128) + G <= 65535.
 *
 * fp8_blockscaled_grouped_gemm_wgrad: all G weight gradients in one launch,
 *   C[g M + m, n] = bf16( sum over expert g's slots kb of
 *                         sA[kb, m] sB[kb, n] sum_{k in kb} dec(qa[m, k]) dec(qb[n, k]) )
 *   qa, sa   the grouped quantiser's output for dY (M rows of qa, ldsa >= M)
 *   qb, sb   the same for X (N rows, ldsb >= N)
 *   c        device, bf16 [G * M, N] (row pitch ldc): dW_g at rows g M ..; an
 *            expert without tokens gets zeros
 *   M, N multiples of 128 (0: nothing to do); T and offsets as given to the quantiser;
 *   lda, ldb >= 128 * (ceil(T/128) + G).  flags: FP8_GEMM_PATH_AUTO runs
 *   the per-K-block promotion kernel, or with FP8_GEMM_SCALES_POW2 (every
 *   scale an exact power of two) the hardware block-scaled kernel, which
 *   accumulates each expert's whole token range in TMEM; _PROMOTE and _MX
 *   force one (_MX needs the pow2 promise: FP8_ERR_SCALE_MODE otherwise);
 *   _SKINNY and FP8_GEMM_SCALES_E8 return FP8_ERR_NOT_IMPLEMENTED.
 */
FP8BS_API fp8_status fp8_quant_act_128x1_grouped(const void *x, int64_t T, int64_t K, int64_t ldx,
                                                 const int32_t *offsets, int32_t G, uint8_t *qt, int64_t ldqt,
                                                 float *st, int64_t ldst, fp8_scale_mode mode,
                                                 fp8_stream_t stream);
FP8BS_API fp8_status fp8_blockscaled_grouped_gemm_wgrad(const uint8_t *qa, int64_t lda, const float *sa,
                                                        int64_t ldsa, const uint8_t *qb, int64_t ldb,
                                                        const float *sb, int64_t ldsb, const int32_t *offsets,
                                                        int32_t G, int64_t T, void *c, int64_t ldc, int64_t M,
                                                        int64_t N, uint32_t flags, fp8_stream_t stream);

/*
 * Per-tensor dynamic scaling: one scale for the whole tensor, recomputed from
 * its current amax so that every value fits the FP8 range (ai.warp-studio.com
 * end-to-end FP8 RL article, §FP8強化学習における精度と安定性の確保).
 *
 *   amax           = max over the whole tensor of |x[m, k]|
 *   s              = scale(amax)        (see fp8_scale_mode; the block rule
 *                                        applied to one block, the tensor)
 *   q[m, k]        = e4m3( RN_fp32(x[m, k] * r(amax)) )
 *
 * Two kernels on `stream` (an amax reduction, then the cast); the call also
 * clears the amax word first.
 * x          device, bf16 [M, K] row-major, row pitch ldx (>= K, % 8 == 0)
 * q          device, uint8 [M, K] row-major, row pitch ldq (>= K, % 16 == 0)
 * scale_amax device, 2 floats, 8-byte aligned: [0] receives s, [1] the amax
 *            (overwritten; both valid once the stream reaches the call's end)
 * M >= 0 (0 is a no-op: nothing written), K > 0, K % 8 == 0.
 */
FP8BS_API fp8_status fp8_quant_per_tensor(const void *x, int64_t M, int64_t K, int64_t ldx,
                                          uint8_t *q, int64_t ldq, float *scale_amax,
                                          fp8_scale_mode mode, fp8_stream_t stream);

/*
 * FP8 KV cache and decode attention (upppp.jp NeMo RL FP8 article,
 * §KVキャッシュとAttentionにも拡張): during rollout the KV cache and the
 * attention run in FP8; the Q, K and V scales are recomputed at the end of
 * each training step (the policy changes) and used for the next rollout.
 * Calibration is fp8_quant_per_tensor's amax (scale_amax[0] = amax/448 of
 * the calibration Q, K or V activations); the cache and the queries are cast
 * with fp8_quant_with_scale; fp8_decode_attention runs one decode step.
 */

/*
 * Cast under a given scale:  q[m, k] = e4m3( RN_fp32(x[m, k] * RN_fp32(1 / s)) ),
 * s = scale[0] (the division x / s if 1 / s overflows fp32).
 * Values beyond +-448 s saturate to the largest code (a calibrated scale can
 * be exceeded by later activations).
 * x      device, bf16 [M, K] row-major, row pitch ldx (>= K, % 8 == 0)
 * q      device, uint8 [M, K], row pitch ldq (>= K, % 16 == 0)
 * scale  device, one fp32; must be a positive normal number (it is read on
 *        the device; nothing checks it)
 * M >= 0 (0 is a no-op), K > 0, K % 8 == 0.  x, q 16-byte aligned.
 */
FP8BS_API fp8_status fp8_quant_with_scale(const void *x, int64_t M, int64_t K, int64_t ldx,
                                          uint8_t *q, int64_t ldq, const float *scale,
                                          fp8_stream_t stream);

/*
 * Cache append of one decode step: for every sequence b and KV head g,
 *   k_cache[b, g, seq_lens[b], :] = e4m3( RN_fp32(k_new[b, g, :] * RN_fp32(1 / sk[0])) )
 * and likewise v with sv[0] (values beyond +-448 s saturate).  Rows whose
 * slot seq_lens[b] is outside [0, T) are skipped; seq_lens is not changed
 * (the caller advances it after the step's attention).
 * k_new, v_new  device, bf16 [B, Hkv, D], contiguous
 * sk, sv        device, one fp32 each (positive normal numbers)
 * k_cache, v_cache  device, uint8 [B, Hkv, T, D]
 * D == 128; B >= 0 (0 is a no-op).  Tensors 16-byte aligned.
 */
FP8BS_API fp8_status fp8_kv_cache_append(const void *k_new, const void *v_new, const float *sk,
                                         const float *sv, const int32_t *seq_lens, uint8_t *k_cache,
                                         uint8_t *v_cache, int64_t B, int64_t Hkv, int64_t T, int64_t D,
                                         fp8_stream_t stream);

/*
 * One decode step of grouped-query attention over an FP8 KV cache:
 *
 *   o[b, h, :] = sum_t p_t * dec(v[b, g, t, :]) * sv,   g = h / (Hq / Hkv),
 *   p = softmax_t( (dec(q[b, h, :]) sq) . (dec(k[b, g, t, :]) sk) / sqrt(D) ),
 *   t = 0 .. seq_lens[b] - 1   (a sequence with no keys gets zeros)
 *
 * computed in fp32 (online softmax over key splits of 512, merged in a
 * second kernel when T > 512), output rounded to bf16.
 * q        device, uint8 [B, Hq, D] codes (scale sq[0])
 * k_cache  device, uint8 [B, Hkv, T, D] codes (sk[0]); v_cache likewise (sv[0])
 * seq_lens device, int32 [B]; values are clamped to [0, T]
 * out      device, bf16 [B, Hq, D]
 * workspace device scratch of fp8_decode_attention_workspace_size(B, Hq, T)
 *          bytes (NULL when that is 0); no state is kept between calls.
 * D == 128; Hq % Hkv == 0 with Hq / Hkv in {1, 2, 4, 8}; T > 0.
 * B >= 0 (0 is a no-op).  q, caches, out and workspace 16-byte aligned.
 */
FP8BS_API size_t fp8_decode_attention_workspace_size(int64_t B, int64_t Hq, int64_t T);
FP8BS_API fp8_status fp8_decode_attention(const uint8_t *q, const float *sq,
                                          const uint8_t *k_cache, const float *sk,
                                          const uint8_t *v_cache, const float *sv,
                                          const int32_t *seq_lens, int64_t B, int64_t Hq,
                                          int64_t Hkv, int64_t T, int64_t D, void *out,
                                          void *workspace, size_t ws_bytes, fp8_stream_t stream);

/*
 * FP8 GEMM with one scale per operand (per-tensor scaling):
 *
 *   C[m, n] = bf16_RN( RN_fp32(sa * sb) * sum_k dec(qa[m, k]) dec(qb[n, k]) )
 *
 * with the sum accumulated in fp32 by the tensor core over the whole K range
 * (no per-K-block promotion is needed: the scales do not change along K).
 * Runs the MX kernel with unit scale factors.
 * qa, lda, qb, ldb, c, ldc, M, N, K, workspace: as fp8_blockscaled_gemm.
 * sa, sb  device, one fp32 each (e.g. scale_amax[0] of fp8_quant_per_tensor).
 * flags: FP8_GEMM_PATH_AUTO or FP8_GEMM_PATH_MX (FP8_GEMM_SCALES_POW2 is
 *     accepted and changes nothing); _PROMOTE and _SKINNY return
 *     FP8_ERR_NOT_IMPLEMENTED.
 */
FP8BS_API fp8_status fp8_tensorscaled_gemm(const uint8_t *qa, int64_t lda, const float *sa,
                                           const uint8_t *qb, int64_t ldb, const float *sb,
                                           void *c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                           uint32_t flags, void *workspace, size_t ws_bytes,
                                           fp8_stream_t stream);

/*
 * Block-scaled FP8 GEMM with a scale per row of B as well (the wgrad form,
 * dW = dY^T X with both operands from fp8_quant_act_128x1):
 *
 *   C[m, n] = bf16_RN( sum_kb  sA[kb, m] * sB[kb, n] * P[m, n, kb] )
 *
 * qa, sa, lda, ldsa, c, ldc, M, N, K, workspace: as fp8_blockscaled_gemm
 *     (K is the token count here, a multiple of 128).
 * qb  device, uint8 [N, K], row pitch ldb (>= K, % 16 == 0)
 * sb  device, fp32 [K/128][ldsb]: the scale of row n of B, K-block kb is
 *     sb[kb * ldsb + n] (ldsb >= N, % 4 == 0, 16-byte aligned)
 * flags: FP8_GEMM_SCALES_POW2 | FP8_GEMM_PATH_AUTO, _PROMOTE or _MX (AUTO:
 *     MX with FP8_GEMM_SCALES_POW2, else promote); FP8_GEMM_PATH_SKINNY
 *     returns FP8_ERR_NOT_IMPLEMENTED.  On the promote kernel each K-block's
 *     partial is multiplied by RN(sA * sB) per element (one more multiply per
 *     element than the 128x128 form); the MX kernel takes the per-row scales
 *     as its B scale factors at no extra cost.
 */
FP8BS_API fp8_status fp8_blockscaled_gemm_wgrad(const uint8_t *qa, int64_t lda, const float *sa, int64_t ldsa,
                                                const uint8_t *qb, int64_t ldb, const float *sb, int64_t ldsb,
                                                void *c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                                uint32_t flags, void *workspace, size_t ws_bytes,
                                                fp8_stream_t stream);

/*
 * Block-scaled FP8 GEMM with the next layer's activation quantisation fused
 * into its epilogue.  The pages project a gain from fusing the quantisation
 * kernels (upppp.jp NeMo RL FP8 article, §重要度サンプリングで精度を保つ).
 *
 * Computes C as fp8_blockscaled_gemm does (the promote kernel, or the MX
 * kernel for power-of-two scales), rounds it to bf16, and writes the E4M3
 * codes and 1x128 scales that
 * fp8_quant_act_1x128(C_bf16, ..., out_mode) would produce from it: qc and sc
 * are bit-identical to running the GEMM and then the activation quantiser on
 * its output, without the bf16 round trip through memory.
 *
 * qa, sa, qb, sb, M, N, K, workspace: as fp8_blockscaled_gemm.
 * c   optional (NULL: not written); bf16 [M, N], row pitch ldc (>= N, % 8 == 0).
 * qc  device, uint8 [M, N], row pitch ldqc (>= N, % 16 == 0), 16-byte aligned.
 * sc  device, fp32 [N/128][ldsc]: scale of row m, column block j at sc[j * ldsc + m]
 *     (ldsc >= M, % 4 == 0, 16-byte aligned) -- the layout the next GEMM's sa takes.
 * flags: FP8_GEMM_SCALES_POW2 (about sa, sb) | FP8_GEMM_PATH_AUTO, _PROMOTE or
 *     _MX (AUTO: MX with FP8_GEMM_SCALES_POW2, else promote); the skinny path
 *     returns FP8_ERR_NOT_IMPLEMENTED.  On the promote kernel the cast runs
 *     on the warps that bound its speed and measured slower than the separate
 *     quantiser; on the MX kernel it runs on otherwise idle epilogue warps.
 * out_mode: the scale rule of qc/sc (FP8_SCALE_FP32_AMAX or FP8_SCALE_POW2).
 */
FP8BS_API fp8_status fp8_blockscaled_gemm_quant(const uint8_t *qa, int64_t lda, const float *sa, int64_t ldsa,
                                                const uint8_t *qb, int64_t ldb, const float *sb,
                                                void *c, int64_t ldc, uint8_t *qc, int64_t ldqc,
                                                float *sc, int64_t ldsc, int64_t M, int64_t N, int64_t K,
                                                uint32_t flags, fp8_scale_mode out_mode,
                                                void *workspace, size_t ws_bytes, fp8_stream_t stream);

/*
 * Grouped (mixture-of-experts) block-scaled GEMM: for each expert g < G,
 * rows offsets[g] .. offsets[g+1]-1 of A (tokens sorted by expert) times
 * expert g's weights:
 *
 *   C[m, n] = bf16( sum_kb sA[kb, m] * sB[g][n/128, kb] * P_g[m, n, kb] )
 *
 * qa       device, uint8 [M_total, K], row pitch lda;  sa device fp32 [K/128][ldsa]
 * offsets  device, int32 [G+1], non-decreasing, offsets[0] == 0,
 *          offsets[G] == M_total.  Read on the device, so no host sync is
 *          needed; values that break these rules are outside the contract
 *          (the kernel clamps them to [0, M_total] and never reads or
 *          writes out of bounds).
 * qb       device, uint8 [G][N][K] contiguous;  sb device fp32 [G][N/128][K/128] contiguous
 * c        device, bf16 [M_total, N], row pitch ldc
 * Empty experts are allowed.  G >= 1, N and K multiples of 128.
 * flags: FP8_GEMM_SCALES_POW2 | FP8_GEMM_PATH_AUTO, _PROMOTE or _MX (AUTO picks
 *     MX when FP8_GEMM_SCALES_POW2 is set, else promote);
 *     FP8_GEMM_PATH_SKINNY returns FP8_ERR_NOT_IMPLEMENTED.
 */
FP8BS_API fp8_status fp8_blockscaled_grouped_gemm(const uint8_t *qa, int64_t lda, const float *sa, int64_t ldsa,
                                        const int32_t *offsets, int32_t G, int64_t M_total,
                                        const uint8_t *qb, const float *sb,
                                        void *c, int64_t ldc, int64_t N, int64_t K,
                                        uint32_t flags, void *workspace, size_t ws_bytes,
                                        fp8_stream_t stream);

/*
 * Decode-sized GEMM (M <= 256) that allocates nothing and takes no workspace.
 *
 * The web pages have no counterpart: this is an interface convenience.  It
 * computes the same C as fp8_blockscaled_gemm on the skinny path (same
 * kernels, same division of the K-blocks over the CTAs, same fixed-order
 * reduction, so the output is bit-identical), but keeps the reduction's
 * tickets and fp32 partials in an 8 MiB array inside the library's own
 * device memory instead of a caller-provided workspace.  It is meant for
 * callers that cannot call cudaMalloc: plugins hosted by a runtime that
 * reserves all device memory at start-up and fails or mis-accounts later
 * allocations, and decode loops where cudaMalloc/cudaFree would synchronise
 * the device.  Inputs and output are passed exactly as for
 * fp8_blockscaled_gemm.
 *
 * - Every GPU that loads the library holds the 8 MiB array until the process
 *   exits.
 * - The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any
 *   stream capture.
 * - All calls share the array, and it keeps what the last call left in it.
 *   The call clears the ticket words on `stream` before its launch.  Calls
 *   that overlap on the GPU (unordered streams) race on the array: order them.
 * - The scratch needed is the skinny path's: 0 when every output tile is
 *   computed by one CTA, else 65536 bytes of tickets plus
 *   (P + T - 1) * NT * 128 * 4 bytes of partials, where NT = M rounded up to
 *   16, 32, 64 or 128 (128 for M > 64), T = (N/128) * ceil(M / NT) output
 *   tiles (tokens beyond 128 run as further 128-token chunks), and P is the
 *   CTA count fp8_gemm_plan reports for FP8_GEMM_PATH_SKINNY (it is at most
 *   fp8_gemm_workspace_size(M, N, K, 1)).  Sizes that need more than 8 MiB return
 *   FP8_ERR_WORKSPACE without launching.
 *   M > 256 returns FP8_ERR_SHAPE.
 * - flags: FP8_GEMM_PATH_AUTO or FP8_GEMM_PATH_SKINNY (plus FP8_GEMM_SCALES_POW2);
 *   FP8_GEMM_SCALES_E8 returns FP8_ERR_NOT_IMPLEMENTED (fp32 scales only).
 * - The array's address is looked up once per device and kept for the life of
 *   the process: after cudaDeviceReset (or anything else that replaces the
 *   device's primary context) this entry point must not be called again.
 */
FP8BS_API fp8_status fp8_blockscaled_gemm_skinny_noalloc(const uint8_t *qa, int64_t lda, const float *sa,
                                                         int64_t ldsa, const uint8_t *qb, int64_t ldb,
                                                         const float *sb, void *c, int64_t ldc, int64_t M,
                                                         int64_t N, int64_t K, uint32_t flags,
                                                         fp8_stream_t stream);

/* Bytes of workspace fp8_blockscaled_gemm (G == 1) or
 * fp8_blockscaled_grouped_gemm (G > 1) needs for these sizes, whatever path
 * the flags choose or force (the largest of the paths' needs); 0 when none. */
FP8BS_API size_t fp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int32_t G);

/* Static, human-readable name of a status code. */
FP8BS_API const char *fp8_status_string(fp8_status status);

/*
 * Failure-path test hook (the pages have no counterpart).  Until called
 * again, GEMMs launched by this process on the promote and skinny
 * kernels bound every wait inside the kernel by `wait_limit_ns` nanoseconds
 * (0: the default of 2 s; at most 2 s), and with skip_first_load != 0 their
 * TMA producer leaves out the first K-block's operands, so the waits on them
 * run out: the kernel records FP8_ERR_TIMEOUT in the status word, releases
 * its TMEM and returns; its output is unspecified.  The CUDA context stays
 * usable.  fp8_debug_inject(0, 0) restores normal operation.  A workspace
 * used by such a call may hold non-zero tickets afterwards: zero it again.
 * Returns FP8_ERR_SHAPE for a limit above 2 s.
 */
FP8BS_API fp8_status fp8_debug_inject(int32_t skip_first_load, uint64_t wait_limit_ns);

/* Synchronises `stream`, returns the current device's status word (FP8_OK
 * or the first error a kernel recorded, e.g. FP8_ERR_TIMEOUT) and clears it. */
FP8BS_API fp8_status fp8_last_device_status(fp8_stream_t stream);

/* Which kernel fp8_blockscaled_gemm would run for these arguments
 * (one of the FP8_GEMM_PATH_* values, never AUTO), and, through
 * `splits` (may be NULL), for the skinny path the number of CTAs P that
 * share the K-blocks of all output tiles (stream-K: CTA c takes K-blocks
 * [c U / P, (c+1) U / P) of the U = tiles * K/128, tile after tile), else 1. */
FP8BS_API uint32_t fp8_gemm_plan(int64_t M, int64_t N, int64_t K, uint32_t flags, int32_t *splits);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
