"""Pins for the CPU oracle, against facts that do not come from the oracle.

Each check is a function taking the oracle routine under test, so that the
mutation tests at the end can hand it a copy of the oracle with a planted
mistake and confirm that at least one pin fails.  Sources of truth used here:
the OCP OFP8 code table (tests/golden/e4m3_ocp_landmarks.txt), the library
casts torch.float8_e4m3fn and ml_dtypes.float8_e4m3fn, exact rational
arithmetic (fractions.Fraction), brute force over the 254 finite codes, and
closed forms (integer GEMMs, power-of-two bounds).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.fp8_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ALL_CODES = np.arange(256, dtype=np.uint8)


def _finite_bf16_f32():
    """Every finite bf16 value as float32."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = O.bf16_bits_to_f32(bits)
    return f[np.isfinite(f)]


# ---------------------------------------------------------------- decode
def check_decode_landmarks(decode):
    for line in open(os.path.join(GOLDEN, "e4m3_ocp_landmarks.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code_s, val_s = line.split()
        got = float(decode(np.array([int(code_s, 16)], np.uint8))[0])
        if val_s == "nan":
            if not math.isnan(got):
                return False
        else:
            want = float(val_s)
            if got != want or math.copysign(1, got) != math.copysign(1, want):
                return False
    return True


def check_decode_vs_libraries(decode):
    ours = decode(ALL_CODES)
    t = torch.from_numpy(ALL_CODES.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ml = pytest.importorskip("ml_dtypes")
    m = ALL_CODES.view(ml.float8_e4m3fn).astype(np.float64)
    for ref in (t, m):
        nan_ok = np.array_equal(np.isnan(ours), np.isnan(ref))
        fin = ~np.isnan(ref)
        if not nan_ok or not np.array_equal(ours[fin], ref[fin]):
            return False
        if not np.array_equal(np.signbit(ours[fin]), np.signbit(ref[fin])):
            return False
    return True


def test_decode_landmarks():
    assert check_decode_landmarks(O.e4m3_decode)


def test_decode_matches_torch_and_ml_dtypes():
    assert check_decode_vs_libraries(O.e4m3_decode)


def test_decode_counts():
    v = O.e4m3_decode(ALL_CODES)
    assert np.isnan(v).sum() == 2
    assert np.isfinite(v).sum() == 254
    assert np.nanmax(v) == 448.0 and np.nanmin(v) == -448.0
    # code order equals value order over the non-negative finite codes
    assert np.all(np.diff(v[:127]) > 0)


# ---------------------------------------------------------------- encode
FINITE_CODES = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)


def brute_force_encode(y32: np.ndarray) -> np.ndarray:
    """argmin over the 254 finite codes of |dec(c) - y| in exact float64;
    ties go to the code with an even last bit; |y| >= 448 saturates; the code
    carries the sign bit of y.  Independent of the oracle's search."""
    vals = np.array([float(Fraction(int(c & 7) + 8, 8) * Fraction(2) ** (int((c >> 3) & 15) - 7))
                     if (c >> 3) & 15 else float(Fraction(int(c & 7), 512))
                     for c in range(127)])
    a = np.abs(y32.astype(np.float64))
    out = np.empty(a.shape, np.uint8)
    for i in range(0, a.size, 4096):
        blk = a[i:i + 4096]
        d = np.abs(blk[:, None] - vals[None, :])
        best = d.min(axis=1, keepdims=True)
        cand = d == best
        # among tied candidates prefer even codes; at most two tie
        even = cand & (np.arange(127)[None, :] % 2 == 0)
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        out[i:i + 4096] = pick
    out = np.where(a >= 448.0, 0x7E, out).astype(np.uint8)
    return out | (np.signbit(y32).astype(np.uint8) << 7)


def _probe_values():
    """Finite bf16 values, all E4M3 values, and every midpoint between
    neighbouring E4M3 values together with its float32 neighbours."""
    vals = O.e4m3_decode(FINITE_CODES).astype(np.float32)
    pos = np.sort(np.unique(np.abs(vals)))
    mids = ((pos[:-1].astype(np.float64) + pos[1:]) / 2).astype(np.float32)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    extra = np.array([464.0, 465.0, 480.0, 1e30, 2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -149,
                      2.0 ** -126, 447.99997], np.float32)
    core = np.concatenate([vals, mids, up, dn, extra])
    return np.concatenate([_finite_bf16_f32(), core, -core])


def check_encode_bruteforce(encode):
    y = _probe_values()
    return np.array_equal(encode(y), brute_force_encode(y))


def check_encode_vs_torch(encode):
    y = _probe_values()
    y = y[np.abs(y) <= 464.0]           # torch's cast is not saturating above 464
    t = torch.from_numpy(y.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return np.array_equal(encode(y), t)


def check_encode_roundtrip(encode):
    return np.array_equal(encode(O.e4m3_decode(FINITE_CODES).astype(np.float32)), FINITE_CODES)


def check_encode_special(encode):
    # (a list, not a dict: -0.0 and 0.0 are equal keys)
    cases = [(1e30, 0x7E), (-1e30, 0xFE), (448.0, 0x7E), (464.0, 0x7E), (465.0, 0x7E),
             (2.0 ** -10, 0x00), (-(2.0 ** -10), 0x80), (3 * 2.0 ** -11, 0x01),
             (-0.0, 0x80), (0.0, 0x00), (2.0 ** -149, 0x00), (1.0, 0x38),
             # ties between two normals go to the even code: 1.0625 is between
             # 1.0 (0x38) and 1.125 (0x39) -> 0x38; 1.1875 between 0x39, 0x3A -> 0x3A
             (1.0625, 0x38), (1.1875, 0x3A)]
    y = np.array([c[0] for c in cases], np.float32)
    return np.array_equal(encode(y), np.array([c[1] for c in cases], np.uint8))


def test_encode_roundtrip():
    assert check_encode_roundtrip(O.e4m3_encode)


def test_encode_bruteforce():
    assert check_encode_bruteforce(O.e4m3_encode)


def test_encode_vs_torch():
    assert check_encode_vs_torch(O.e4m3_encode)


def test_encode_special_cases():
    assert check_encode_special(O.e4m3_encode)


# ---------------------------------------------------------------- scales
def _amax_samples():
    rng = np.random.Generator(np.random.PCG64(11))
    f = _finite_bf16_f32()
    pos = np.unique(np.abs(f[f != 0]))
    # every positive bf16 value is a possible amax; add a random subset twice
    return np.concatenate([pos, rng.choice(pos, 2000)])


def _f32_ulp(x: float) -> Fraction:
    x = abs(float(np.float32(x)))
    if x < 2.0 ** -126:
        return Fraction(2) ** -149
    e = math.frexp(x)[1] - 1
    return Fraction(2) ** (e - 23)


def check_scale_fp32(scale_fn):
    amax = _amax_samples()
    s = scale_fn(amax)
    for a, si in zip(amax[::7], s[::7]):
        exact = Fraction(float(a)) / 448
        err = abs(Fraction(float(si)) - exact)
        # correctly rounded: within half an ulp of the exact quotient, and the
        # float32 neighbours are no closer
        if err > _f32_ulp(si) / 2:
            return False
        for nb in (np.nextafter(si, np.float32(0)), np.nextafter(si, np.float32(np.inf))):
            if abs(Fraction(float(nb)) - exact) < err:
                return False
    return bool(scale_fn(np.array([0.0], np.float32))[0] == 1.0)


def check_scale_pow2(scale_fn):
    amax = _amax_samples()
    s = scale_fn(amax)
    for a, si in zip(amax, s):
        sf = Fraction(float(si))
        # a power of two: numerator and denominator are both powers of two
        if sf.numerator & (sf.numerator - 1) or sf.denominator & (sf.denominator - 1):
            return False
        e = sf.numerator.bit_length() - 1 - (sf.denominator.bit_length() - 1)
        r = Fraction(float(a)) / 448
        if -127 < e < 127:
            # e = ceil(log2(amax/448)): 2**(e-1) < amax/448 <= 2**e
            if not (Fraction(2) ** (e - 1) < r <= Fraction(2) ** e):
                return False
        elif e == -127:
            if not r <= Fraction(2) ** -127:
                return False
        else:
            return False
    return bool(scale_fn(np.array([0.0], np.float32))[0] == 1.0)


def test_scale_fp32_correctly_rounded():
    assert check_scale_fp32(O.scale_from_amax_fp32)


def test_scale_pow2_is_ceil_power_of_two():
    assert check_scale_pow2(O.scale_from_amax_pow2)


# ---------------------------------------------------------------- quantisers
def _bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def expected_cast(x, s, amax=None, pow2=False) -> np.ndarray:
    """The float32 value the cast rounds to E4M3, from exact arithmetic.

    Power-of-two scale: the quotient x / s (exact in float64, rounded once).
    fp32 scale: r = RN(448 / amax) when the scale comes from an amax (amax 0:
    r = 1), r = RN(1 / s) for a given scale -- a float64 quotient rounded to
    float32 is the correctly rounded float32 quotient (Figueroa: 53 >= 2*24 +
    2) -- then RN(x r), the float64 product of two float32 values being exact.
    Where r overflows float32 the quotient x / s, rounded once."""
    x64 = np.asarray(x, np.float32).astype(np.float64)
    if pow2:
        return (x64 / np.float64(s)).astype(np.float32)
    with np.errstate(over="ignore"):
        if amax is None:
            r = np.float32(np.float64(1.0) / np.float64(s))
        else:
            r = np.float32(1.0) if amax == 0 else np.float32(np.float64(448.0) / np.float64(amax))
    if np.isfinite(r):
        return (x64 * np.float64(r)).astype(np.float32)
    return (x64 / np.float64(s)).astype(np.float32)


# amax 1.0 and the element 2**-16: 2**-16 * 448 = 3.5 * 2**-9 is an exact
# E4M3 tie (rounds to the even code 0x04), while 2**-16 / RN(1/448) lies just
# off it, so a cast that divides by the stored scale gives another code here.
TIE_AMAX, TIE_X = 1.0, 2.0 ** -16


def _act_sample(seed=3, M=37, K=640):
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[:, 5] *= 40
    x[3, 128:256] = 0.0                       # an all-zero block
    x[4, 256:384] = 0.0
    x[4, 300] = -2.0 ** -130                  # a block whose amax is a bf16 subnormal
    x[5, :128] *= 1e-30
    x[6, :128] = np.clip(x[6, :128] * 0.25, -0.9, 0.9)
    x[6, 0], x[6, 1] = TIE_AMAX, TIE_X        # the cast multiplies by RN(448/amax), not divides
    return _bf16_round(x)


def check_act_quant(quant):
    """Codes against exact arithmetic, block by block: amax element -> +-448
    (fp32 mode), and every code equals the nearest-even E4M3 rounding of
    RN(x RN(448/amax)) (fp32 scales; the quotient x/s where the reciprocal
    overflows) or of x/s (power-of-two scales), see expected_cast."""
    x = _act_sample()
    for pow2 in (False, True):
        q, s = quant(x, pow2=pow2)
        M, K = x.shape
        if q.shape != x.shape or s.shape != (M, K // 128):
            return False
        for m in range(M):
            for kb in range(K // 128):
                blk = x[m, kb * 128:(kb + 1) * 128]
                amax = float(np.max(np.abs(blk)))
                si = float(s[m, kb])
                want_s = (O.scale_from_amax_pow2 if pow2 else O.scale_from_amax_fp32)(
                    np.array([amax], np.float32))[0]
                if si != float(want_s):
                    return False
                q32 = expected_cast(blk, si, amax=amax, pow2=pow2)
                if not np.array_equal(q[m, kb * 128:(kb + 1) * 128], brute_force_encode(q32)):
                    return False
                if amax > 0 and not pow2:
                    at = np.abs(blk) == amax
                    if not np.all((q[m, kb * 128:(kb + 1) * 128][at] & 0x7F) == 0x7E):
                        return False
                if amax > 0 and pow2 and amax >= 448 * 2.0 ** -127:
                    at = np.abs(blk) == amax
                    mags = q[m, kb * 128:(kb + 1) * 128][at] & 0x7F
                    if not np.all((mags >= 0x76) & (mags <= 0x7E)):
                        return False
    return True


def test_act_quant_exact():
    assert check_act_quant(O.quant_act_1x128)


def check_block_geometry(quant_act, quant_w):
    """A single planted large value moves exactly one scale: the one of its
    own 1x128 block (activations) or 128x128 tile (weights)."""
    rng = np.random.Generator(np.random.PCG64(5))
    x = _bf16_round(rng.uniform(-1, 1, (6, 512)).astype(np.float32))
    _, s0 = quant_act(x)
    x2 = x.copy()
    x2[4, 300] = 1000.0
    _, s1 = quant_act(x2)
    changed = np.argwhere(s0 != s1)
    if changed.tolist() != [[4, 300 // 128]]:
        return False
    w = _bf16_round(rng.uniform(-1, 1, (256, 384)).astype(np.float32))
    _, t0 = quant_w(w)
    w2 = w.copy()
    w2[200, 70] = 1000.0
    _, t1 = quant_w(w2)
    return np.argwhere(t0 != t1).tolist() == [[1, 0]]


def test_block_geometry():
    assert check_block_geometry(O.quant_act_1x128, O.quant_weight_128x128)


def test_weight_quant_matches_per_tile_act_quant():
    # A 128x128 tile quantised with one scale equals the element cast with
    # that tile's scale; checked against exact arithmetic on one tile.
    rng = np.random.Generator(np.random.PCG64(9))
    w = _bf16_round((rng.standard_normal((256, 256)) * 0.02).astype(np.float32))
    q, s = O.quant_weight_128x128(w)
    for nb in range(2):
        for kb in range(2):
            t = w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            amax = np.float32(np.max(np.abs(t)))
            assert Fraction(float(s[nb, kb])) == Fraction(float(np.float32(
                np.float64(amax) / 448.0)))
            q32 = expected_cast(t, s[nb, kb], amax=float(amax))
            assert np.array_equal(q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128],
                                  brute_force_encode(q32.ravel()).reshape(128, 128))


# ---------------------------------------------------------------- GEMM
CODE_P1, CODE_M1, CODE_0 = 0x38, 0xB8, 0x00


def check_gemm_integer(gemm):
    """Codes decoding to {-1, 0, 1}, unit scales: the GEMM is an integer
    matrix product, computed here with Python integers."""
    rng = np.random.Generator(np.random.PCG64(21))
    for K in (128, 256):
        ia = rng.integers(-1, 2, (5, K))
        iw = rng.integers(-1, 2, (128, K))
        enc = {1: CODE_P1, -1: CODE_M1, 0: CODE_0}
        qa = np.vectorize(enc.get)(ia).astype(np.uint8)
        qw = np.vectorize(enc.get)(iw).astype(np.uint8)
        want = [[sum(int(ia[m, k]) * int(iw[n, k]) for k in range(K)) for n in range(128)]
                for m in range(5)]
        for j in (0, -3, 4):                 # powers of two keep it exact
            sa = np.full((5, K // 128), 2.0 ** j, np.float32)
            sw = np.full((1, K // 128), 2.0 ** -j, np.float32)
            got = gemm(qa, sa, qw, sw)
            if not np.array_equal(got, np.array(want, np.float64)):
                return False
    return True


def check_gemm_rational(gemm):
    """Random codes and fp32 scales on a tiny problem, against an exact
    rational evaluation of sum_kb sA*sW*sum_k dec(a)dec(w)."""
    rng = np.random.Generator(np.random.PCG64(22))
    M, N, K = 2, 128, 256
    fin = FINITE_CODES
    qa = rng.choice(fin, (M, K)).astype(np.uint8)
    qw = rng.choice(fin, (N, K)).astype(np.uint8)
    sa = rng.uniform(0.01, 3, (M, K // 128)).astype(np.float32)
    sw = rng.uniform(0.01, 3, (N // 128, K // 128)).astype(np.float32)
    dec = {int(c): Fraction(float(v)) for c, v in zip(fin, O.e4m3_decode(fin))}
    got = gemm(qa, sa, qw, sw)
    for m in range(M):
        for n in range(0, N, 17):
            tot = Fraction(0)
            for kb in range(K // 128):
                p = sum(dec[int(qa[m, k])] * dec[int(qw[n, k])]
                        for k in range(kb * 128, (kb + 1) * 128))
                tot += Fraction(float(sa[m, kb])) * Fraction(float(sw[n // 128, kb])) * p
            if abs(Fraction(float(got[m, n])) - tot) > abs(tot) * Fraction(1, 10 ** 13) + Fraction(1, 10 ** 300):
                return False
    return True


def check_gemm_orientation(gemm):
    """C = A W^T: with W row n holding a single 1 at column pi(n), column n of
    C is column pi(n) of the dequantised A (scaled)."""
    rng = np.random.Generator(np.random.PCG64(23))
    M, N, K = 3, 128, 256
    qa = rng.choice(FINITE_CODES, (M, K)).astype(np.uint8)
    sa = np.array([[1.0, 2.0]] * M, np.float32)
    perm = rng.permutation(K)[:N]
    qw = np.zeros((N, K), np.uint8)
    qw[np.arange(N), perm] = CODE_P1
    sw = np.array([[1.0, 0.5]], np.float32)
    got = gemm(qa, sa, qw, sw)
    deqa = O.e4m3_decode(qa) * np.repeat(sa.astype(np.float64), 128, axis=1)
    want = deqa[:, perm] * np.where(perm < 128, 1.0, 0.5)[None, :]
    return np.array_equal(got, want)


def test_gemm_integer_exact():
    assert check_gemm_integer(O.gemm_ref)


def test_gemm_rational():
    assert check_gemm_rational(O.gemm_ref)


def test_gemm_orientation():
    assert check_gemm_orientation(O.gemm_ref)


def test_gemm_matches_torch_fp64():
    rng = np.random.Generator(np.random.PCG64(24))
    x = _bf16_round(rng.standard_normal((64, 384)).astype(np.float32))
    w = _bf16_round((rng.standard_normal((256, 384)) * 0.02).astype(np.float32))
    qa, sa = O.quant_act_1x128(x)
    qw, sw = O.quant_weight_128x128(w)
    a = torch.from_numpy(qa).view(torch.float8_e4m3fn).double() * torch.from_numpy(sa).double().repeat_interleave(128, 1)
    b = torch.from_numpy(qw).view(torch.float8_e4m3fn).double() * torch.from_numpy(sw).double().repeat_interleave(128, 0).repeat_interleave(128, 1)
    ref = (a @ b.T).numpy()
    got = O.gemm_ref(qa, sa, qw, sw)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_gemm_rows_subset():
    rng = np.random.Generator(np.random.PCG64(25))
    x = _bf16_round(rng.standard_normal((50, 256)).astype(np.float32))
    w = _bf16_round(rng.standard_normal((128, 256)).astype(np.float32))
    qa, sa = O.quant_act_1x128(x)
    qw, sw = O.quant_weight_128x128(w)
    rows = np.array([49, 0, 17])
    full = O.gemm_ref(qa, sa, qw, sw)[rows]
    # BLAS may block the two calls differently: equal up to fp64 rounding
    assert np.max(np.abs(O.gemm_ref_rows(qa, sa, qw, sw, rows) - full)) <= 1e-13 * np.max(np.abs(full))


def test_grouped_gemm_matches_per_group_and_empty_groups():
    rng = np.random.Generator(np.random.PCG64(26))
    offs = np.array([0, 5, 5, 12, 12, 20])        # groups 1 and 3 empty
    G, N, K = 5, 128, 256
    x = _bf16_round(rng.standard_normal((20, K)).astype(np.float32))
    w = _bf16_round((rng.standard_normal((G, N, K)) * 0.02).astype(np.float32))
    qa, sa = O.quant_act_1x128(x)
    qws, sws = zip(*[O.quant_weight_128x128(w[g]) for g in range(G)])
    qw, sw = np.stack(qws), np.stack(sws)
    got = O.grouped_gemm_ref(qa, sa, offs, qw, sw)
    scale = np.max(np.abs(got))
    for g in range(G):
        r = slice(offs[g], offs[g + 1])
        if offs[g + 1] > offs[g]:
            assert np.max(np.abs(got[r] - O.gemm_ref(qa[r], sa[r], qw[g], sw[g]))) <= 1e-13 * scale
    rows = np.array([19, 3, 11])
    assert np.max(np.abs(O.grouped_gemm_ref(qa, sa, offs, qw, sw, rows=rows) - got[rows])) <= 1e-13 * scale


# ---------------------------------------------------------------- mutations
# Each mutant plants one plausible mistake in a copy of an oracle routine;
# at least one pin above must reject it.
def _enc_ties_away(y):
    y = np.asarray(y, np.float32)
    vals = O.e4m3_decode(np.arange(127, dtype=np.uint8))
    a = np.abs(y.astype(np.float64))
    idx = np.clip(np.searchsorted(vals, np.minimum(a, 447), side="right") - 1, 0, 125)
    pick = np.where(vals[idx + 1] - a <= a - vals[idx], idx + 1, idx)
    pick = np.where(a >= 448, 0x7E, pick).astype(np.uint8)
    return pick | (np.signbit(y).astype(np.uint8) << 7)


def _enc_truncate(y):
    y = np.asarray(y, np.float32)
    vals = O.e4m3_decode(np.arange(127, dtype=np.uint8))
    a = np.abs(y.astype(np.float64))
    idx = np.clip(np.searchsorted(vals, a, side="right") - 1, 0, 126).astype(np.uint8)
    return idx | (np.signbit(y).astype(np.uint8) << 7)


def _enc_no_signed_zero(y):
    c = O.e4m3_encode(y)
    return np.where((c & 0x7F) == 0, 0, c).astype(np.uint8)


def _dec_bias8(codes):
    return O.e4m3_decode(codes) / 2.0


def _pow2_floor(amax):
    a = np.asarray(amax, np.float32).astype(np.float64)
    f, E = np.frexp(a)
    e = np.clip(E - 1 - 8, -127, 127)
    return np.where(a > 0, np.ldexp(1.0, e), 1.0).astype(np.float32)


def _scale_mul_recip(amax):
    a = np.asarray(amax, np.float32)
    return np.where(a > 0, a * np.float32(1.0 / 448.0), 1.0).astype(np.float32)


def _gemm_transposed_w(qa, sa, qw, sw):
    # mistake: output columns indexed from the wrong end of W
    return O.dequant_act(qa, sa) @ O.dequant_weight(qw, sw)[::-1].T


def _gemm_scale_wrong_block(qa, sa, qw, sw):
    return O.dequant_act(qa, sa[:, ::-1]) @ O.dequant_weight(qw, sw).T


def _gemm_drops_last_kblock(qa, sa, qw, sw):
    qa = qa.copy()
    qa[:, -128:] = 0
    return O.gemm_ref(qa, sa, qw, sw)


def _quant_act_transposed_blocks(x, pow2=False):
    q, s = O.quant_act_1x128(x, pow2)
    x2 = np.asarray(x, np.float32)
    amax = np.abs(x2).reshape(x2.shape[0], -1, 128).max(axis=2)
    # mistake: amax taken over 128 rows of a column-slab instead of the row's block
    return q, O.scale_from_amax(np.roll(amax, 1, axis=0), pow2)


def _quant_act_divides(x, pow2=False):
    # mistake: the cast divides by the stored scale instead of multiplying by
    # RN(448/amax)
    x = np.asarray(x, np.float32)
    s = O.scale_from_amax(O.block_amax_act(x), pow2)
    return O.e4m3_encode((x / np.repeat(s, 128, axis=1)).astype(np.float32)), s


def _quant_act_recip_of_scale(x, pow2=False):
    # mistake: the factor is RN(1/s) of the rounded scale instead of RN(448/amax)
    x = np.asarray(x, np.float32)
    s = O.scale_from_amax(O.block_amax_act(x), pow2)
    with np.errstate(over="ignore", divide="ignore", invalid="ignore"):
        r = (np.float32(1.0) / s).astype(np.float32)
        return O.e4m3_encode((x * np.repeat(r, 128, axis=1)).astype(np.float32)), s


def _quant_w_wrong_tile(w, pow2=False):
    w = np.asarray(w, np.float32)
    N, K = w.shape
    t = np.abs(w).reshape(N // 128, 128, K // 128, 128).max(axis=(1, 2))  # wrong axes
    s = O.scale_from_amax(np.broadcast_to(t.max(axis=1, keepdims=True), (N // 128, K // 128)), pow2)
    return O.quant_weight_128x128(w, pow2)[0], s


@pytest.mark.parametrize("mutant,checks", [
    (_enc_ties_away, [check_encode_bruteforce, check_encode_vs_torch, check_encode_special]),
    (_enc_truncate, [check_encode_bruteforce, check_encode_roundtrip]),
    (_enc_no_signed_zero, [check_encode_special, check_encode_bruteforce]),
])
def test_mutant_encoders_are_caught(mutant, checks):
    assert not all(c(mutant) for c in checks)


def test_mutant_decoder_is_caught():
    assert not check_decode_landmarks(_dec_bias8)
    assert not check_decode_vs_libraries(_dec_bias8)


def test_mutant_scales_are_caught():
    assert not check_scale_pow2(_pow2_floor)
    assert not check_scale_fp32(_scale_mul_recip)


@pytest.mark.parametrize("mutant", [_gemm_transposed_w, _gemm_scale_wrong_block, _gemm_drops_last_kblock])
def test_mutant_gemms_are_caught(mutant):
    checks = [check_gemm_integer, check_gemm_rational, check_gemm_orientation]
    assert not all(c(mutant) for c in checks)


@pytest.mark.parametrize("mutant", [_quant_act_divides, _quant_act_recip_of_scale])
def test_mutant_casts_are_caught(mutant):
    assert not check_act_quant(mutant)


def test_the_planted_tie_separates_the_two_readings():
    # independent of the oracle: multiplying by RN(448/amax) gives the exact
    # tie 3.5 * 2**-9, rounded to the even code 4; dividing by RN(amax/448)
    # does not land on it
    s = np.float32(np.float64(TIE_AMAX) / 448.0)
    by_mul = expected_cast(np.array([TIE_X], np.float32), s, amax=TIE_AMAX)
    by_div = (np.float64(TIE_X) / np.float64(s)).astype(np.float32)
    assert Fraction(float(by_mul[0])) == Fraction(7, 2 ** 10)
    assert brute_force_encode(by_mul)[0] == 0x04
    assert brute_force_encode(np.array([by_div], np.float32))[0] != 0x04


def test_mutant_block_geometry_is_caught():
    assert not check_block_geometry(_quant_act_transposed_blocks, O.quant_weight_128x128)
    assert not check_block_geometry(O.quant_act_1x128, _quant_w_wrong_tile)
