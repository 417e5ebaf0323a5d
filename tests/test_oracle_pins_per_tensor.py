"""Pins of the oracle's per-tensor scaling functions against facts that do
not come from the oracle's per-tensor code: exact rational arithmetic and the
brute-force encoder, the reduction to the 1x128 quantiser when the tensor is
one block, invariance under power-of-two rescaling, and Python-integer GEMMs.
Mutants at the end must be rejected.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest

import oracle.fp8_oracle as O
from tests.test_oracle_pins import (CODE_0, CODE_M1, CODE_P1, FINITE_CODES, TIE_AMAX, TIE_X, _bf16_round,
                                    brute_force_encode, expected_cast)


def _sample(seed=51, shape=(37, 300)):
    rng = np.random.Generator(np.random.PCG64(seed))
    x = np.clip(rng.standard_normal(shape).astype(np.float32) * 0.2, -0.9, 0.9)
    x[3, 7] = TIE_AMAX * 64             # the tensor's amax
    x[3, 8] = TIE_X * 64                # an exact E4M3 tie under RN(448/amax), not under x/s
    x[5, :] = 0.0
    x[6, 11] = -2.0 ** -130             # bf16 subnormal
    return _bf16_round(x)


def check_per_tensor_exact(quant):
    """One scale from the whole tensor's amax (exact rational check of the
    scale rule) and every code the nearest-even E4M3 rounding of
    RN(x RN(448/amax)) (fp32 scale) or of x/s (power of two); see
    expected_cast."""
    x = _sample()
    for pow2 in (False, True):
        q, s = quant(x, pow2=pow2)
        if q.shape != x.shape or np.ndim(s) != 0:
            return False
        amax = float(np.max(np.abs(x)))
        rule = O.scale_from_amax_pow2 if pow2 else O.scale_from_amax_fp32
        if float(s) != float(rule(np.array([amax], np.float32))[0]):
            return False
        if not pow2 and Fraction(float(s)) != Fraction(amax) / 448 and \
                abs(Fraction(float(s)) - Fraction(amax) / 448) > Fraction(float(s)) / 2 ** 24:
            return False
        q32 = expected_cast(x, s, amax=amax, pow2=pow2)
        if not np.array_equal(q, brute_force_encode(q32.ravel()).reshape(x.shape)):
            return False
        if not pow2 and not np.all((q[np.abs(x) == amax] & 0x7F) == 0x7E):
            return False
    return True


def check_per_tensor_single_block(quant):
    """A [1, 128] tensor is one 1x128 block: the per-tensor and 1x128
    quantisers agree."""
    rng = np.random.Generator(np.random.PCG64(52))
    x = _bf16_round(rng.standard_normal((1, 128)).astype(np.float32) * 3)
    for pow2 in (False, True):
        q, s = quant(x, pow2=pow2)
        q1, s1 = O.quant_act_1x128(x, pow2)
        if not (np.array_equal(q, q1) and float(s) == float(s1[0, 0])):
            return False
    return True


def check_per_tensor_pow2_invariance(quant):
    """x * 2^k has the same codes and a scale 2^k times larger (while no
    value leaves the normal fp32 range)."""
    x = _sample(seed=53)
    for pow2 in (False, True):
        q, s = quant(x, pow2=pow2)
        q2, s2 = quant(x * np.float32(2.0 ** 9), pow2=pow2)
        if not (np.array_equal(q, q2) and float(s2) == float(s) * 2.0 ** 9):
            return False
    return True


def check_per_tensor_gemm(gemm):
    """Codes decoding to {-1, 0, 1} and power-of-two scales: C is a Python
    integer product times sA * sB; random codes and fp32 scales: exact
    rational evaluation."""
    rng = np.random.Generator(np.random.PCG64(54))
    enc = {1: CODE_P1, -1: CODE_M1, 0: CODE_0}
    ia = rng.integers(-1, 2, (5, 256))
    ib = rng.integers(-1, 2, (7, 256))
    qa = np.vectorize(enc.get)(ia).astype(np.uint8)
    qb = np.vectorize(enc.get)(ib).astype(np.uint8)
    got = gemm(qa, np.float32(0.25), qb, np.float32(8.0))
    want = np.array([[2 * sum(int(ia[m, k]) * int(ib[n, k]) for k in range(256)) for n in range(7)]
                     for m in range(5)], np.float64)
    if not np.array_equal(got, want):
        return False
    qa = rng.choice(FINITE_CODES, (2, 128)).astype(np.uint8)
    qb = rng.choice(FINITE_CODES, (3, 128)).astype(np.uint8)
    sa, sb = np.float32(0.37), np.float32(1.9)
    dec = {int(c): Fraction(float(v)) for c, v in zip(FINITE_CODES, O.e4m3_decode(FINITE_CODES))}
    got = gemm(qa, sa, qb, sb)
    for m in range(2):
        for n in range(3):
            tot = Fraction(float(sa)) * Fraction(float(sb)) * sum(dec[int(qa[m, k])] * dec[int(qb[n, k])]
                                                                  for k in range(128))
            if abs(Fraction(float(got[m, n])) - tot) > abs(tot) * Fraction(1, 10 ** 13) + Fraction(1, 10 ** 300):
                return False
    return True


def test_per_tensor_exact():
    assert check_per_tensor_exact(O.quant_per_tensor)


def test_per_tensor_single_block():
    assert check_per_tensor_single_block(O.quant_per_tensor)


def test_per_tensor_pow2_invariance():
    assert check_per_tensor_pow2_invariance(O.quant_per_tensor)


def test_per_tensor_gemm():
    assert check_per_tensor_gemm(O.gemm_per_tensor_ref)


def test_per_tensor_gemm_equals_block_gemm_with_constant_scales():
    # With every block scale equal to the tensor scale the block-scaled
    # reference is the per-tensor one.
    rng = np.random.Generator(np.random.PCG64(55))
    qa = rng.choice(FINITE_CODES, (9, 256)).astype(np.uint8)
    qb = rng.choice(FINITE_CODES, (128, 256)).astype(np.uint8)
    sa, sb = np.float32(0.013), np.float32(2.5)
    ref = O.gemm_ref(qa, np.full((9, 2), sa, np.float32), qb, np.full((1, 2), sb, np.float32))
    got = O.gemm_per_tensor_ref(qa, sa, qb, sb)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


# ---------------------------------------------------------------- mutations
def _per_row_amax(x, pow2=False):
    # mistake: the amax of the first row instead of the whole tensor
    x = np.asarray(x, np.float32)
    s = O.scale_from_amax(np.array([np.max(np.abs(x[0]))], np.float32), pow2)[0]
    return O.e4m3_encode((x / s).astype(np.float32)), np.float32(s)


def _divide_by_scale(x, pow2=False):
    # mistake: divide by the stored scale instead of multiplying by RN(448/amax)
    x = np.asarray(x, np.float32)
    amax = np.float32(np.max(np.abs(x)))
    s = O.scale_from_amax(np.array([amax], np.float32), pow2)[0]
    return O.e4m3_encode((x / s).astype(np.float32)), np.float32(s)


def _gemm_one_scale(qa, sa, qb, sb):
    return (O.e4m3_decode(qa) @ O.e4m3_decode(qb).T) * np.float64(sa)


@pytest.mark.parametrize("mutant", [_per_row_amax, _divide_by_scale])
def test_mutant_per_tensor_quantisers_are_caught(mutant):
    assert not (check_per_tensor_exact(mutant) and check_per_tensor_single_block(mutant))


def test_mutant_per_tensor_gemm_is_caught():
    assert not check_per_tensor_gemm(_gemm_one_scale)


# ---------------------------------------------------------------- UE8M0 scale bytes
def test_ue8m0_landmarks():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "ue8m0_ocp_mx_landmarks.txt")
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        b, v = line.split()
        assert float(O.ue8m0_to_scale(int(b, 16))) == float(v)
        assert int(O.scale_to_ue8m0(np.float32(float(v)))) == int(b, 16)


def test_ue8m0_roundtrip_of_every_pow2_scale():
    # every exponent the power-of-two rule can produce, and the scales that
    # rule gives for a sweep of amax values
    e = np.arange(-127, 128)
    s = np.ldexp(np.float64(1.0), e).astype(np.float32)
    b = O.scale_to_ue8m0(s)
    assert np.array_equal(b.astype(np.int64), e + 127)
    assert np.array_equal(O.ue8m0_to_scale(b), s)
    amax = np.exp2(np.arange(-140, 127, 0.37)).astype(np.float32)      # all finite in float32
    sp = O.scale_from_amax_pow2(amax[amax > 0])
    assert np.array_equal(O.ue8m0_to_scale(O.scale_to_ue8m0(sp)), sp)


def test_ue8m0_rejects_non_powers_of_two():
    with pytest.raises(ValueError):
        O.scale_to_ue8m0(np.float32(0.75))
    with pytest.raises(ValueError):
        O.scale_to_ue8m0(np.float32(2.0 ** -130))
