"""Pins of the oracle's training-side functions (the backward GEMMs of a
linear layer y = x W^T and their operand quantisers) against facts that do
not come from the oracle: exact rational arithmetic, brute-force code
search, Python integer products, PyTorch autograd's derivative of the
forward GEMM, and one-hot closed forms.  Each mutant at the end plants one
plausible mistake in a copy of an oracle routine and must be rejected.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.fp8_oracle as O
from tests.test_oracle_pins import (CODE_0, CODE_M1, CODE_P1, FINITE_CODES, TIE_AMAX, TIE_X, _bf16_round,
                                    brute_force_encode, expected_cast)


# ---------------------------------------------------------------- 128x1 activation quantiser
def _col_sample(seed=31, M=256, K=40):
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[7, :] *= 40                              # one token dominates its blocks
    x[128:256, 3] = 0.0                        # an all-zero block
    x[:128, 4] = 0.0
    x[9, 4] = -2.0 ** -130                     # a block whose amax is a bf16 subnormal
    x[:128, 5] *= 1e-30
    x[:128, 6] = np.clip(x[:128, 6] * 0.25, -0.9, 0.9)
    x[0, 6], x[1, 6] = TIE_AMAX, TIE_X         # separates multiply-by-RN(448/amax) from x/s
    return _bf16_round(x)


def check_col_quant(quant_col):
    """Codes and scales of every 128x1 block against exact arithmetic: the
    scale from the block's amax, each code the nearest-even E4M3 rounding of
    the cast value of expected_cast; outputs transposed (qt[k, m])."""
    x = _col_sample()
    M, K = x.shape
    for pow2 in (False, True):
        qt, st = quant_col(x, pow2=pow2)
        if qt.shape != (K, M) or st.shape != (K, M // 128):
            return False
        rule = O.scale_from_amax_pow2 if pow2 else O.scale_from_amax_fp32
        for k in range(K):
            for mb in range(M // 128):
                blk = x[mb * 128:(mb + 1) * 128, k]
                amax = float(np.max(np.abs(blk)))
                si = float(st[k, mb])
                if si != float(rule(np.array([amax], np.float32))[0]):
                    return False
                q32 = expected_cast(blk, si, amax=amax, pow2=pow2)
                if not np.array_equal(qt[k, mb * 128:(mb + 1) * 128], brute_force_encode(q32)):
                    return False
    return True


def check_col_geometry(quant_col):
    """A planted large value at (token m, column k) moves only the scale of
    its own 128x1 block: st[k, m // 128]."""
    rng = np.random.Generator(np.random.PCG64(32))
    x = _bf16_round(rng.uniform(-1, 1, (384, 24)).astype(np.float32))
    _, s0 = quant_col(x)
    x2 = x.copy()
    x2[200, 17] = 1000.0
    _, s1 = quant_col(x2)
    return np.argwhere(s0 != s1).tolist() == [[17, 1]]


def test_col_quant_exact():
    assert check_col_quant(O.quant_act_128x1)


def test_col_geometry():
    assert check_col_geometry(O.quant_act_128x1)


def test_col_quant_is_row_quant_of_the_transpose():
    # The 128x1 blocks of x are the 1x128 blocks of x^T.
    x = _col_sample(seed=33, M=384, K=256)
    for pow2 in (False, True):
        qt, st = O.quant_act_128x1(x, pow2)
        q1, s1 = O.quant_act_1x128(np.ascontiguousarray(x.T), pow2)
        assert np.array_equal(qt, q1) and np.array_equal(st, s1)


def test_col_quant_ragged_tokens_pad_with_zeros():
    # 300 tokens: the last block holds 44 real rows; its scales and codes are
    # those of the block padded with zero rows, and the pad codes are zero.
    x = _col_sample(seed=34, M=384, K=40)
    x[300:] = 0.0
    qt, st = O.quant_act_128x1(x[:300])
    qt_full, st_full = O.quant_act_128x1(x)
    assert qt.shape == (40, 384) and np.array_equal(qt, qt_full) and np.array_equal(st, st_full)
    assert np.all(qt[:, 300:] == 0)


def test_moe_wgrad_is_per_expert_wgrad_and_autograd():
    """Per expert: dL/dW_g of L = sum_g sum(G_g * (X_g W_g^T)) on the
    dequantised (zero-padded) operands, by PyTorch autograd; an empty expert
    gets zeros."""
    rng = np.random.Generator(np.random.PCG64(40))
    offs = [0, 70, 70, 300]
    N, K = 128, 256
    x = _bf16_round(rng.standard_normal((300, K)).astype(np.float32))
    dy = _bf16_round((rng.standard_normal((300, N)) * 1e-3).astype(np.float32))
    got = O.moe_wgrad_ref(dy, x, offs)
    assert got.shape == (3, N, K) and np.all(got[1] == 0)
    for g in (0, 2):
        lo, hi = offs[g], offs[g + 1]
        qg, sg = O.quant_act_128x1(dy[lo:hi])
        qx, sx = O.quant_act_128x1(x[lo:hi])
        Gc = _deq(qg, sg).T.contiguous()
        Xc = _deq(qx, sx).T.contiguous()
        W = torch.zeros((N, K), dtype=torch.float64, requires_grad=True)
        (Gc * (Xc @ W.T)).sum().backward()
        assert np.max(np.abs(got[g] - W.grad.numpy())) <= 1e-12 * np.max(np.abs(got[g]))


# ---------------------------------------------------------------- W^T operand
def test_weight_t_is_quantisation_of_the_transpose():
    # Quantising W^T directly (its own 128x128 blocks) gives the same codes
    # and scales as transposing W's.
    rng = np.random.Generator(np.random.PCG64(34))
    w = _bf16_round((rng.standard_normal((384, 256)) * 0.02).astype(np.float32))
    w[5, 200] = 3.0
    for pow2 in (False, True):
        qt, st = O.quant_weight_128x128_t(w, pow2)
        q2, s2 = O.quant_weight_128x128(np.ascontiguousarray(w.T), pow2)
        assert qt.shape == (256, 384) and st.shape == (2, 3)
        assert np.array_equal(qt, q2) and np.array_equal(st, s2)
    # a value planted in block (n 0, k 1) of W moves scale (k 1, n 0) of W^T only
    flat = np.full((384, 256), 0.5, np.float32)
    _, s0 = O.quant_weight_128x128_t(flat)
    flat[5, 200] = 100.0
    _, s1 = O.quant_weight_128x128_t(flat)
    assert np.argwhere(s0 != s1).tolist() == [[1, 0]]


# ---------------------------------------------------------------- backward GEMMs
def _deq(q, s):
    """Plain dequantisation through PyTorch's own E4M3 type, 1x128 scales."""
    return torch.from_numpy(q).view(torch.float8_e4m3fn).double() * \
        torch.from_numpy(np.asarray(s, np.float32)).double().repeat_interleave(128, 1)


def _deq_w(q, s):
    sb = torch.from_numpy(np.asarray(s, np.float32)).double().repeat_interleave(128, 0).repeat_interleave(128, 1)
    return torch.from_numpy(q).view(torch.float8_e4m3fn).double() * sb


def check_backward_autograd(dgrad, wgrad):
    """PyTorch autograd differentiates L = sum(G * (X W^T)) in fp64 on the
    dequantised operands; dgrad must give dL/dX and wgrad dL/dW."""
    rng = np.random.Generator(np.random.PCG64(35))
    M, N, K = 256, 384, 256
    x = _bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    w = _bf16_round((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    g = _bf16_round((rng.standard_normal((M, N)) * 1e-3).astype(np.float32))
    # dgrad operands: G in 1x128 blocks along n, W in its 128x128 blocks
    q_g, s_g = O.quant_act_1x128(g)
    q_w, s_w = O.quant_weight_128x128(w)
    X = torch.zeros((M, K), dtype=torch.float64, requires_grad=True)
    W = _deq_w(q_w, s_w).requires_grad_(False)
    G = _deq(q_g, s_g)
    (G * (X @ W.T)).sum().backward()
    got = dgrad(q_g, s_g, q_w, s_w)
    ref = X.grad.numpy()
    if got.shape != ref.shape or np.max(np.abs(got - ref)) > 1e-12 * np.max(np.abs(ref)):
        return False
    # wgrad operands: G and X in 128x1 blocks along tokens
    qt_g, st_g = O.quant_act_128x1(g)
    qt_x, st_x = O.quant_act_128x1(x)
    Gc = _deq(qt_g, st_g).T.contiguous()          # [M, N]
    Xc = _deq(qt_x, st_x).T.contiguous()          # [M, K]
    Wv = torch.zeros((N, K), dtype=torch.float64, requires_grad=True)
    (Gc * (Xc @ Wv.T)).sum().backward()
    got = wgrad(qt_g, st_g, qt_x, st_x)
    ref = Wv.grad.numpy()
    return got.shape == ref.shape and np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def check_backward_one_hot(dgrad, wgrad):
    """One-hot gradients give closed forms: dY = e_(m0, n0) makes row m0 of
    dX the dequantised row n0 of W; dY = e_(t, n0) and X = e_(t, k0) make dW
    the single entry (n0, k0) = sdy * sx."""
    rng = np.random.Generator(np.random.PCG64(36))
    M, N, K = 130, 256, 384
    q_w = rng.choice(FINITE_CODES, (N, K)).astype(np.uint8)
    s_w = rng.uniform(0.5, 2, (N // 128, K // 128)).astype(np.float32)
    m0, n0 = 129, 200
    q_dy = np.zeros((M, N), np.uint8)
    q_dy[m0, n0] = CODE_P1
    s_dy = np.ones((M, N // 128), np.float32)
    got = dgrad(q_dy, s_dy, q_w, s_w)
    want = np.zeros((M, K))
    want[m0] = O.e4m3_decode(q_w[n0]) * np.repeat(s_w[n0 // 128].astype(np.float64), 128)
    if not np.array_equal(got, want):
        return False
    T, t, k0 = 256, 140, 300
    qt_dy = np.zeros((N, T), np.uint8)
    qt_x = np.zeros((K, T), np.uint8)
    qt_dy[n0, t] = CODE_M1
    qt_x[k0, t] = CODE_P1
    st_dy = np.full((N, T // 128), 0.25, np.float32)
    st_x = np.full((K, T // 128), 8.0, np.float32)
    got = wgrad(qt_dy, st_dy, qt_x, st_x)
    want = np.zeros((N, K))
    want[n0, k0] = -2.0
    return np.array_equal(got, want)


def check_wgrad_integer(wgrad):
    """Codes decoding to {-1, 0, 1}, power-of-two scales per (row, token
    block): dW against Python integer sums."""
    rng = np.random.Generator(np.random.PCG64(37))
    N, K, T = 128, 128, 256
    enc = {1: CODE_P1, -1: CODE_M1, 0: CODE_0}
    ig = rng.integers(-1, 2, (N, T))
    ix = rng.integers(-1, 2, (K, T))
    eg = rng.integers(-3, 4, (N, T // 128))
    ex = rng.integers(-3, 4, (K, T // 128))
    qt_dy = np.vectorize(enc.get)(ig).astype(np.uint8)
    qt_x = np.vectorize(enc.get)(ix).astype(np.uint8)
    got = wgrad(qt_dy, np.exp2(eg).astype(np.float32), qt_x, np.exp2(ex).astype(np.float32))
    for n in range(0, N, 7):
        for k in range(0, K, 5):
            tot = Fraction(0)
            for tb in range(T // 128):
                p = sum(int(ig[n, i]) * int(ix[k, i]) for i in range(tb * 128, (tb + 1) * 128))
                tot += Fraction(2) ** int(eg[n, tb]) * Fraction(2) ** int(ex[k, tb]) * p
            if Fraction(float(got[n, k])) != tot:
                return False
    return True


def check_wgrad_rational(wgrad):
    """Random codes and fp32 scales on both operands, against an exact
    rational evaluation of sum_tb sdy[n, tb] * sx[k, tb] * sum_t dec * dec."""
    rng = np.random.Generator(np.random.PCG64(38))
    N, K, T = 3, 128, 256
    qt_dy = rng.choice(FINITE_CODES, (N, T)).astype(np.uint8)
    qt_x = rng.choice(FINITE_CODES, (K, T)).astype(np.uint8)
    st_dy = rng.uniform(0.01, 3, (N, T // 128)).astype(np.float32)
    st_x = rng.uniform(0.01, 3, (K, T // 128)).astype(np.float32)
    dec = {int(c): Fraction(float(v)) for c, v in zip(FINITE_CODES, O.e4m3_decode(FINITE_CODES))}
    got = wgrad(qt_dy, st_dy, qt_x, st_x)
    for n in range(N):
        for k in range(0, K, 13):
            tot = Fraction(0)
            for tb in range(T // 128):
                p = sum(dec[int(qt_dy[n, i])] * dec[int(qt_x[k, i])] for i in range(tb * 128, (tb + 1) * 128))
                tot += Fraction(float(st_dy[n, tb])) * Fraction(float(st_x[k, tb])) * p
            if abs(Fraction(float(got[n, k])) - tot) > abs(tot) * Fraction(1, 10 ** 13) + Fraction(1, 10 ** 300):
                return False
    return True


def test_backward_autograd():
    assert check_backward_autograd(O.dgrad_ref, O.wgrad_ref)


def test_backward_one_hot():
    assert check_backward_one_hot(O.dgrad_ref, O.wgrad_ref)


def test_wgrad_integer_exact():
    assert check_wgrad_integer(O.wgrad_ref)


def test_wgrad_rational():
    assert check_wgrad_rational(O.wgrad_ref)


def test_wgrad_rows_subset():
    rng = np.random.Generator(np.random.PCG64(39))
    qt_dy = rng.choice(FINITE_CODES, (256, 256)).astype(np.uint8)
    qt_x = rng.choice(FINITE_CODES, (128, 256)).astype(np.uint8)
    st_dy = rng.uniform(0.5, 2, (256, 2)).astype(np.float32)
    st_x = rng.uniform(0.5, 2, (128, 2)).astype(np.float32)
    rows = np.array([255, 0, 100])
    full = O.wgrad_ref(qt_dy, st_dy, qt_x, st_x)[rows]
    got = O.wgrad_ref_rows(qt_dy, st_dy, qt_x, st_x, rows)
    assert np.max(np.abs(got - full)) <= 1e-13 * np.max(np.abs(full))


# ---------------------------------------------------------------- mutations
def _col_quant_whole_slab(x, pow2=False):
    # mistake: one amax for the whole 128-token slab instead of one per column
    x = np.asarray(x, np.float32)
    M, K = x.shape
    amax = np.abs(x).reshape(M // 128, 128 * K).max(axis=1, keepdims=True)
    s = O.scale_from_amax(np.broadcast_to(amax, (M // 128, K)), pow2)
    q = O.e4m3_encode((x / np.repeat(s, 128, axis=0)).astype(np.float32))
    return np.ascontiguousarray(q.T), np.ascontiguousarray(s.T)


def _col_quant_untransposed_scales(x, pow2=False):
    # mistake: scale grid of the next token block
    qt, st = O.quant_act_128x1(x, pow2)
    return qt, np.roll(st, 1, axis=1)


def _dgrad_w_transposed(q_dy, s_dy, q_w, s_w):
    # mistake: W's rows taken from the wrong end (a transposition slip in the operand)
    return O.dequant_act(q_dy, s_dy) @ O.dequant_weight(q_w, s_w)[::-1]


def _wgrad_scale_of_other_block(qt_dy, st_dy, qt_x, st_x):
    # mistake: X's scales taken from the other token block
    return O.dequant_act(qt_dy, st_dy) @ O.dequant_act(qt_x, st_x[:, ::-1]).T


def _wgrad_drops_last_block(qt_dy, st_dy, qt_x, st_x):
    qt_x = qt_x.copy()
    qt_x[:, -128:] = 0
    return O.wgrad_ref(qt_dy, st_dy, qt_x, st_x)


def _col_quant_divides(x, pow2=False):
    # mistake: the cast divides by the stored scale
    x = np.asarray(x, np.float32)
    s = O.scale_from_amax(O.block_amax_col(x), pow2)
    q = O.e4m3_encode((x / np.repeat(s, 128, axis=0)).astype(np.float32))
    return np.ascontiguousarray(q.T), np.ascontiguousarray(s.T)


@pytest.mark.parametrize("mutant", [_col_quant_whole_slab, _col_quant_untransposed_scales, _col_quant_divides])
def test_mutant_col_quantisers_are_caught(mutant):
    assert not (check_col_quant(mutant) and check_col_geometry(mutant))


def test_mutant_dgrad_is_caught():
    assert not (check_backward_autograd(_dgrad_w_transposed, O.wgrad_ref) and
                check_backward_one_hot(_dgrad_w_transposed, O.wgrad_ref))


@pytest.mark.parametrize("mutant", [_wgrad_scale_of_other_block, _wgrad_drops_last_block])
def test_mutant_wgrads_are_caught(mutant):
    checks = [check_wgrad_integer(mutant), check_wgrad_rational(mutant),
              check_backward_autograd(O.dgrad_ref, mutant), check_backward_one_hot(O.dgrad_ref, mutant)]
    assert not all(checks)
