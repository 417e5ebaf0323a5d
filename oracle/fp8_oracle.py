"""CPU oracle for the block-scaled FP8 linear layer.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain reference that the
CUDA library is checked against.  Only the test suite, the package's smoke
entry point and the benchmark's CPU-baseline leg may import it; the product
path never does, and it shares no code, tables or helpers with the CUDA
kernels.

What it computes, and where each step comes from:

* The element format is FP8 E4M3 and the blocks are 1x128 for activations and
  128x128 for weights -- page "NVIDIA NeMo RL достигает ускорения на 48%
  благодаря сквозному обучению с точностью FP8" (greentreeone.com),
  §Технический прорыв.  The pages do not spell out the bit layout; it is taken
  from the public OCP 8-bit Floating Point specification (OFP8, 2023), E4M3:
  1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
  S.1111.111 is NaN, largest finite magnitude 448.
* A power-of-two scale option -- page "NVIDIA NeMo RL FP8" (upppp.jp),
  §設定方法, and the greentreeone.com page, §Почему это важно.
* Scales are recomputed from the current tensor on every call (weights are
  re-quantised after each optimizer step) -- upppp.jp page,
  §KVキャッシュとAttentionにも拡張; greentreeone.com page,
  §Реальные прирост производительности.
* Linear layers do their arithmetic on the FP8 codes with higher-precision
  accumulation -- page "エンドツーエンドFP8精度で実現する高スループット強化学習
  トレーニング" (ai.warp-studio.com), §FP8強化学習における精度と安定性の確保.

Readings where the pages are silent (each also listed in the design notes):
scale = amax/448 rounded to fp32; an all-zero block gets scale 1; the cast
multiplies by the reciprocal factor r = 448/amax rounded to fp32 (RN(x r),
then E4M3 with round-to-nearest-even and saturation at +-448) -- the pages
give the scale as amax/448 and leave open whether the cast divides by it or
multiplies by its reciprocal; where 448/amax overflows fp32 (amax below
448 * 2**-128) the cast divides by the scale instead.  A cast with a given
scale s (not from an amax) multiplies by RN(1/s), or divides where that
overflows.  The power-of-two scale is 2**ceil(log2(amax/448)) with the
exponent clamped to [-127, 127], and its cast multiplies by 2**-e, which is
the quotient exactly.  The GEMM reference is dequantise-then-multiply in
fp64.

Every function below is pinned by the CPU tests in tests/test_oracle_pins.py
and (training-side functions) tests/test_oracle_pins_training.py, (per-tensor
scaling and UE8M0 scale bytes) tests/test_oracle_pins_per_tensor.py, (KV-cache attention)
tests/test_oracle_pins_attention.py against
facts that do not come from this file (the OCP code table, library
casts, exact rational arithmetic, brute force, PyTorch autograd and closed
forms).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0        # largest finite E4M3 magnitude (OCP OFP8, E4M3 row)
QBLOCK = 128            # block edge: 1x128 activations, 128x128 weights

__all__ = [
    "E4M3_MAX", "QBLOCK",
    "e4m3_decode", "e4m3_encode", "bf16_bits_to_f32",
    "block_amax_act", "block_amax_weight",
    "scale_from_amax_fp32", "scale_from_amax_pow2", "scale_from_amax", "recip_from_amax", "recip_from_scale",
    "quant_act_1x128", "quant_weight_128x128",
    "dequant_act", "dequant_weight",
    "gemm_ref", "gemm_ref_rows", "grouped_gemm_ref",
    "block_amax_col", "quant_act_128x1", "quant_weight_128x128_t",
    "dgrad_ref", "wgrad_ref", "wgrad_ref_rows", "moe_wgrad_ref",
    "quant_per_tensor", "gemm_per_tensor_ref",
    "quant_with_scale", "decode_attention_ref",
    "scale_to_ue8m0", "ue8m0_to_scale",
]


# --------------------------------------------------------------------------
# Element format
# --------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 byte as float64 (NaN for the two NaN codes).

    OCP OFP8 E4M3: sign = bit 7, exponent field E = bits 6..3 (bias 7),
    mantissa m = bits 2..0.  E == 0 is subnormal, value m * 2**-9; otherwise
    (1 + m/8) * 2**(E-7).  E == 15 with m == 7 is NaN; there is no infinity.
    """
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    sub = m.astype(np.float64) * 2.0 ** -9
    nrm = (1.0 + m.astype(np.float64) / 8.0) * np.exp2((e - 7).astype(np.float64))
    val = sign * np.where(e == 0, sub, nrm)
    return np.where((e == 15) & (m == 7), np.nan, val)


# The 127 non-negative finite codes 0x00..0x7E; their values increase with the
# code, so a sorted search over this table finds the two neighbours of |y|.
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = e4m3_decode(_POS_CODES)


def e4m3_encode(y) -> np.ndarray:
    """E4M3 code of each finite float32 value: round to nearest, ties to the
    even code, magnitudes at or above 448 saturate to 448 (code 0x7E).

    The sign bit of the input becomes the sign bit of the code, so -0.0 maps
    to 0x80.  Between two neighbouring representable values lo <= |y| < hi the
    nearer one wins; on an exact tie the code whose last bit is 0 wins (the
    even mantissa).  The distances are exact in float64 because |y| is a
    float32 and lo, hi are E4M3 values.  Non-finite inputs are outside the
    contract.
    """
    y = np.asarray(y, dtype=np.float32)
    neg = np.signbit(y)
    a = np.abs(y.astype(np.float64))
    sat = a >= E4M3_MAX
    a_in = np.where(sat, 0.0, a)
    lo_idx = np.searchsorted(_POS_VALUES, a_in, side="right") - 1
    lo_idx = np.clip(lo_idx, 0, 125)
    hi_idx = lo_idx + 1
    d_lo = a_in - _POS_VALUES[lo_idx]
    d_hi = _POS_VALUES[hi_idx] - a_in
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi_idx % 2 == 0))
    mag = np.where(pick_hi, hi_idx, lo_idx)
    mag = np.where(sat, 0x7E, mag).astype(np.uint8)
    return (mag | (neg.astype(np.uint8) << 7)).astype(np.uint8)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) to the float32 values they denote (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


# --------------------------------------------------------------------------
# Block statistics and scales
# --------------------------------------------------------------------------
def _check_mult(n, what):
    if n % QBLOCK:
        raise ValueError(f"{what}={n} is not a multiple of {QBLOCK}")


def block_amax_act(x: np.ndarray) -> np.ndarray:
    """max |x| over each 1x128 block of a [M, K] float32 matrix -> [M, K/128]."""
    M, K = x.shape
    _check_mult(K, "K")
    return np.abs(x).reshape(M, K // QBLOCK, QBLOCK).max(axis=2).astype(np.float32)


def block_amax_weight(w: np.ndarray) -> np.ndarray:
    """max |w| over each 128x128 tile of a [N, K] float32 matrix -> [N/128, K/128]."""
    N, K = w.shape
    _check_mult(N, "N")
    _check_mult(K, "K")
    t = np.abs(w).reshape(N // QBLOCK, QBLOCK, K // QBLOCK, QBLOCK)
    return t.max(axis=(1, 3)).astype(np.float32)


def scale_from_amax_fp32(amax) -> np.ndarray:
    """fp32 scale s = amax / 448 (IEEE float32 division); s = 1 for amax == 0."""
    amax = np.asarray(amax, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        s = amax / np.float32(E4M3_MAX)
    return np.where(amax > 0, s, np.float32(1.0)).astype(np.float32)


def scale_from_amax_pow2(amax) -> np.ndarray:
    """Power-of-two scale 2**e with e = ceil(log2(amax / 448)).

    amax = F * 2**E with F in [1, 2) (frexp, which also normalises
    subnormals).  Because 448 = 1.75 * 2**8, amax / 448 = (F / 1.75) * 2**(E-8)
    with F / 1.75 in [4/7, 8/7), so the ceiling of its log2 is E - 8 when
    F <= 1.75 and E - 7 when F > 1.75.  e is clamped to [-127, 127] (the range
    an 8-bit power-of-two exponent can hold); amax == 0 gives e = 0.
    """
    amax = np.asarray(amax, dtype=np.float32).astype(np.float64)
    f, E = np.frexp(amax)          # amax = f * 2**E, f in [0.5, 1)
    F = 2.0 * f
    E = E - 1
    e = E - 8 + (F > 1.75).astype(np.int64)
    e = np.clip(e, -127, 127)
    e = np.where(amax > 0, e, 0)
    return np.ldexp(np.float64(1.0), e).astype(np.float32)


def scale_from_amax(amax, pow2: bool) -> np.ndarray:
    return scale_from_amax_pow2(amax) if pow2 else scale_from_amax_fp32(amax)


def recip_from_amax(amax, pow2: bool) -> np.ndarray:
    """The cast's factor r: fp32 mode RN(448 / amax) (IEEE float32 division;
    +inf where it overflows), 1 for amax == 0; power-of-two mode 2**-e, the
    exact reciprocal of the scale."""
    amax = np.asarray(amax, dtype=np.float32)
    if pow2:
        return (np.float64(1.0) / scale_from_amax_pow2(amax).astype(np.float64)).astype(np.float32)
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        r = np.float32(E4M3_MAX) / amax
    return np.where(amax > 0, r, np.float32(1.0)).astype(np.float32)


def recip_from_scale(s) -> np.ndarray:
    """The cast's factor for a given scale s: RN(1 / s) (+inf where it overflows)."""
    with np.errstate(divide="ignore", over="ignore"):
        return (np.float32(1.0) / np.asarray(s, dtype=np.float32)).astype(np.float32)


# --------------------------------------------------------------------------
# Quantisers
# --------------------------------------------------------------------------
def _cast(x: np.ndarray, s_broadcast: np.ndarray, r_broadcast: np.ndarray) -> np.ndarray:
    """codes = e4m3(RN_fp32(x * r)) elementwise (IEEE float32 multiply), or
    e4m3(RN_fp32(x / s)) where r is not finite (IEEE float32 division)."""
    x = x.astype(np.float32)
    r = r_broadcast.astype(np.float32)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        prod = (x * r).astype(np.float32)
        quot = (x / s_broadcast.astype(np.float32)).astype(np.float32)
    return e4m3_encode(np.where(np.isfinite(r), prod, quot))


def quant_act_1x128(x: np.ndarray, pow2: bool = False):
    """1x128 activation quantisation.

    x: float32 [M, K] (bf16 values).  Returns (q uint8 [M, K],
    s float32 [M, K/128]) where s[m, kb] is the scale of row m, columns
    kb*128 .. kb*128+127, and q = e4m3(RN(x r)) with r = RN(448 / amax) of
    the block (the quotient x / s where r overflows; x 2**-e exactly for
    power-of-two scales).  (The library stores the
    scales K-block-major, s[kb][m]; that is a layout choice, the values are
    these.)
    """
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    amax = block_amax_act(x)
    s = scale_from_amax(amax, pow2)
    r = recip_from_amax(amax, pow2)
    return _cast(x, np.repeat(s, QBLOCK, axis=1), np.repeat(r, QBLOCK, axis=1)), s


def quant_weight_128x128(w: np.ndarray, pow2: bool = False):
    """128x128 weight quantisation.

    w: float32 [N, K] (bf16 values).  Returns (q uint8 [N, K],
    s float32 [N/128, K/128]) with q the cast of quant_act_1x128 tile by tile.
    """
    w = np.asarray(w, dtype=np.float32)
    amax = block_amax_weight(w)
    s = scale_from_amax(amax, pow2)
    r = recip_from_amax(amax, pow2)
    grow = lambda t: np.repeat(np.repeat(t, QBLOCK, axis=0), QBLOCK, axis=1)  # noqa: E731
    return _cast(w, grow(s), grow(r)), s


# --------------------------------------------------------------------------
# GEMM reference: dequantise, then multiply in fp64
# --------------------------------------------------------------------------
def dequant_act(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """dec(q[m, k]) * s[m, k // 128] in float64 (exact: <= 4 + 24 bits)."""
    return e4m3_decode(q) * np.repeat(np.asarray(s, np.float64), QBLOCK, axis=1)


def dequant_weight(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """dec(q[n, k]) * s[n // 128, k // 128] in float64 (exact)."""
    sb = np.repeat(np.repeat(np.asarray(s, np.float64), QBLOCK, axis=0), QBLOCK, axis=1)
    return e4m3_decode(q) * sb


def gemm_ref(qa, sa, qw, sw) -> np.ndarray:
    """C[m, n] = sum_k deqA[m, k] * deqW[n, k] in float64 (C = A W^T).

    Equal, up to fp64 rounding order, to sum over K-blocks kb of
    sA[m, kb] * sW[n/128, kb] * sum_{k in kb} dec(qA[m, k]) dec(qW[n, k]).
    """
    return dequant_act(qa, sa) @ dequant_weight(qw, sw).T


def gemm_ref_rows(qa, sa, qw, sw, rows) -> np.ndarray:
    """gemm_ref restricted to the given output rows (for sampled checks)."""
    rows = np.asarray(rows)
    return dequant_act(qa[rows], sa[rows]) @ dequant_weight(qw, sw).T


def grouped_gemm_ref(qa, sa, offsets, qw_groups, sw_groups, rows=None) -> np.ndarray:
    """Per-expert GEMM: rows offsets[g] .. offsets[g+1]-1 of A times W_g^T.

    qw_groups: uint8 [G, N, K]; sw_groups: float32 [G, N/128, K/128].
    Empty groups contribute no rows.  With `rows`, only those output rows are
    computed (returned in the order given).
    """
    offsets = np.asarray(offsets, dtype=np.int64)
    G = len(offsets) - 1
    N = qw_groups.shape[1]
    M = qa.shape[0]
    want = np.arange(M) if rows is None else np.asarray(rows)
    out = np.zeros((len(want), N), dtype=np.float64)
    grp = np.searchsorted(offsets, want, side="right") - 1
    for g in range(G):
        sel = np.nonzero(grp == g)[0]
        if sel.size == 0:
            continue
        r = want[sel]
        out[sel] = dequant_act(qa[r], sa[r]) @ dequant_weight(qw_groups[g], sw_groups[g]).T
    return out


# --------------------------------------------------------------------------
# Training-side operands and GEMMs
#
# The pages apply FP8 to training as well as generation ("end-to-end FP8":
# page "NVIDIA NeMo RL достигает ускорения на 48% благодаря сквозному обучению
# с точностью FP8", §Технический прорыв; page "エンドツーエンドFP8精度で実現
# する高スループット強化学習トレーニング", the opening section: parameters,
# activations, gradients and optimizer updates).  For a linear layer
# y = x W^T the backward pass computes dX = dY W and dW = dY^T X.  The pages
# name only the 1x128 (activations) and 128x128 (weights) blocks; the reading
# taken here is that every operand is quantised in blocks of 128 along the
# dimension its GEMM reduces over:
#   dgrad  dX = dY W   : dY in 1x128 blocks along its rows (reduction over
#                        output features), W in its 128x128 blocks;
#   wgrad  dW = dY^T X : dY and X in 128x1 blocks (128 consecutive tokens of
#                        one column), the reduction being over tokens.
# --------------------------------------------------------------------------
def block_amax_col(x: np.ndarray) -> np.ndarray:
    """max |x| over each 128x1 block (128 consecutive rows of one column) of a
    [M, K] float32 matrix -> [M/128, K]."""
    M, K = x.shape
    _check_mult(M, "M")
    return np.abs(x).reshape(M // QBLOCK, QBLOCK, K).max(axis=1).astype(np.float32)


def quant_act_128x1(x: np.ndarray, pow2: bool = False):
    """128x1 (column-wise) activation quantisation, the wgrad operand.

    x: float32 [M, K] (bf16 values), M tokens.  The block of column k, tokens
    mb*128 .. mb*128+127 gets scale s[mb, k] from its own amax, and q[m, k]
    is x[m, k] cast with that block's scale (as in quant_act_1x128).
    Returned transposed, the way the
    wgrad GEMM reads them (token-contiguous rows): (qt uint8 [K, Mp] with
    qt[k, m] = q[m, k], st float32 [K, Mp/128] with st[k, mb] = s[mb, k]).
    A token count M that is not a multiple of 128 is padded with zero rows
    to Mp (zero rows change no block's amax and add nothing to dW; their
    codes are zero).
    """
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    if M % QBLOCK:
        xp = np.zeros(((M + QBLOCK - 1) // QBLOCK * QBLOCK, K), np.float32)
        xp[:M] = x
        x = xp
    amax = block_amax_col(x)
    s = scale_from_amax(amax, pow2)
    r = recip_from_amax(amax, pow2)
    q = _cast(x, np.repeat(s, QBLOCK, axis=0), np.repeat(r, QBLOCK, axis=0))
    return np.ascontiguousarray(q.T), np.ascontiguousarray(s.T)


def quant_weight_128x128_t(w: np.ndarray, pow2: bool = False):
    """The 128x128 quantisation of W seen from W^T, the dgrad operand.

    A 128x128 block of W^T is the transpose of a block of W and has the same
    amax, so its codes and scale are those of W's block, transposed:
    (qt uint8 [K, N] = q^T, st float32 [K/128, N/128] = s^T).
    """
    q, s = quant_weight_128x128(w, pow2)
    return np.ascontiguousarray(q.T), np.ascontiguousarray(s.T)


def dgrad_ref(q_dy, s_dy, q_w, s_w) -> np.ndarray:
    """Input gradient of y = x W^T: dX[m, k] = sum_n deq(dY)[m, n] deq(W)[n, k]
    in float64.

    q_dy uint8 [M, N] with 1x128 scales s_dy [M, N/128] (blocks along n, the
    reduction); q_w uint8 [N, K] with 128x128 scales s_w [N/128, K/128].
    """
    return dequant_act(q_dy, s_dy) @ dequant_weight(q_w, s_w)


def wgrad_ref(qt_dy, st_dy, qt_x, st_x) -> np.ndarray:
    """Weight gradient of y = x W^T: dW[n, k] = sum_m deq(dY)[m, n] deq(X)[m, k]
    in float64.

    Both operands come as quant_act_128x1 returns them: qt_dy uint8 [N, M]
    (row n = column n of dY, token-contiguous) with st_dy [N, M/128], and
    qt_x uint8 [K, M] with st_x [K, M/128].
    """
    return dequant_act(qt_dy, st_dy) @ dequant_act(qt_x, st_x).T


def moe_wgrad_ref(dy, x, offsets, pow2: bool = False) -> np.ndarray:
    """Weight gradients of a mixture-of-experts layer: for each expert g,
    dW_g = dY_g^T X_g over its token rows offsets[g] .. offsets[g+1]-1, each
    operand quantised in 128x1 blocks of that expert's own tokens (the last
    block zero-padded).  dy [T, N], x [T, K] float32; returns [G, N, K]."""
    offsets = np.asarray(offsets, np.int64)
    G = len(offsets) - 1
    out = np.zeros((G, dy.shape[1], x.shape[1]), np.float64)
    for g in range(G):
        lo, hi = int(offsets[g]), int(offsets[g + 1])
        if hi > lo:
            qg, sg = quant_act_128x1(dy[lo:hi], pow2)
            qx, sx = quant_act_128x1(x[lo:hi], pow2)
            out[g] = wgrad_ref(qg, sg, qx, sx)
    return out


def wgrad_ref_rows(qt_dy, st_dy, qt_x, st_x, rows) -> np.ndarray:
    """wgrad_ref restricted to the given output rows n (for sampled checks)."""
    rows = np.asarray(rows)
    return dequant_act(qt_dy[rows], st_dy[rows]) @ dequant_act(qt_x, st_x).T


# --------------------------------------------------------------------------
# Per-tensor dynamic scaling
#
# One scale for the whole tensor, recomputed from the tensor's current amax
# so that every value fits the FP8 range (page "エンドツーエンドFP8精度で実現
# する高スループット強化学習トレーニング", ai.warp-studio.com,
# §FP8強化学習における精度と安定性の確保: dynamic scaling factors per tensor).
# The scale rule and the cast are the block quantisers' (amax/448 rounded to
# fp32, or the power of two), applied to a single block that is the tensor.
# --------------------------------------------------------------------------
def quant_per_tensor(x: np.ndarray, pow2: bool = False):
    """Per-tensor quantisation of a float32 matrix (bf16 values).

    Returns (q uint8 of x's shape, s float32 scalar): s from max |x| over the
    whole tensor, q the block cast with that scale (x times RN(448/amax)).
    """
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    s = scale_from_amax(np.array([amax], np.float32), pow2)[0]
    r = recip_from_amax(np.array([amax], np.float32), pow2)[0]
    return _cast(x, np.full(x.shape, s, np.float32), np.full(x.shape, r, np.float32)), np.float32(s)


def gemm_per_tensor_ref(qa, sa, qb, sb) -> np.ndarray:
    """C = sA * sB * (dec(qa) @ dec(qb)^T) in float64, one scale per operand."""
    return (e4m3_decode(qa) @ e4m3_decode(qb).T) * (np.float64(np.float32(sa)) * np.float64(np.float32(sb)))


# --------------------------------------------------------------------------
# FP8 KV cache and attention (decode)
#
# Page "NVIDIA NeMo RL FP8" (upppp.jp), §KVキャッシュとAttentionにも拡張:
# the KV cache and the attention run in FP8 too; because the policy's weights
# change every step, the Q, K and V scales are recomputed at the end of each
# training step (from training prompts and responses) and handed to the
# rollout engine.  Readings: one fp32 scale per tensor for each of Q, K and V
# (the per-tensor rule above applied to the calibration activations); the
# cache holds E4M3 codes cast with those fixed scales (values beyond the
# calibrated range saturate at +-448 codes); the attention dequantises and
# computes softmax(q.K^T / sqrt(D)) V, here in float64.
# --------------------------------------------------------------------------
def quant_with_scale(x: np.ndarray, s) -> np.ndarray:
    """Codes of x under a given fp32 scale: e4m3(RN_fp32(x * RN(1/s))), or
    e4m3(RN_fp32(x / s)) where 1/s overflows."""
    x = np.asarray(x, dtype=np.float32)
    r = recip_from_scale(np.float32(s))
    return _cast(x, np.full(x.shape, np.float32(s), np.float32), np.full(x.shape, r, np.float32))


def decode_attention_ref(q, sq, k_cache, sk, v_cache, sv, seq_lens) -> np.ndarray:
    """One decode step of grouped-query attention over an FP8 KV cache.

    q       uint8 [B, Hq, D] codes of the new tokens' queries (scale sq)
    k_cache uint8 [B, Hkv, T, D] codes (scale sk); v_cache likewise (sv)
    seq_lens int [B]: keys 0 .. seq_lens[b]-1 of sequence b are attended
    Query head h reads KV head h // (Hq / Hkv).  Returns float64 [B, Hq, D];
    a sequence with no keys gets zeros.
    """
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), np.float64)
    qd = e4m3_decode(q) * np.float64(np.float32(sq))
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        for h in range(Hq):
            g = h // G
            kd = e4m3_decode(k_cache[b, g, :L]) * np.float64(np.float32(sk))
            vd = e4m3_decode(v_cache[b, g, :L]) * np.float64(np.float32(sv))
            scores = kd @ qd[b, h] / np.sqrt(np.float64(D))
            p = np.exp(scores - scores.max())
            out[b, h] = (p / p.sum()) @ vd
    return out


# --------------------------------------------------------------------------
# Power-of-two scales stored as UE8M0 bytes
#
# A power-of-two scale 2^e (e in [-127, 127], the power-of-two rule above)
# needs only its exponent.  The byte format is UE8M0 of the OCP Microscaling
# (MX) specification v1.0: 8 exponent bits, bias 127, no sign or mantissa,
# 0xFF reserved for NaN; byte b means 2^(b - 127).
# --------------------------------------------------------------------------
def scale_to_ue8m0(s) -> np.ndarray:
    """Byte e + 127 of each power-of-two scale 2^e (ValueError otherwise)."""
    s = np.asarray(s, dtype=np.float64)
    e = np.log2(s)
    if not np.all(np.isfinite(e)) or not np.array_equal(e, np.round(e)) or np.any(np.abs(e) > 127):
        raise ValueError("not a power of two in [2^-127, 2^127]")
    return (np.round(e).astype(np.int64) + 127).astype(np.uint8)


def ue8m0_to_scale(b) -> np.ndarray:
    """2^(b - 127) as float32 (b < 255)."""
    b = np.asarray(b, dtype=np.int64)
    return np.ldexp(np.float64(1.0), b - 127).astype(np.float32)
