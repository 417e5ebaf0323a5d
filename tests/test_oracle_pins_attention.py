"""Pins of the oracle's FP8 KV-cache attention against facts that do not
come from it: PyTorch's scaled_dot_product_attention in float64 on the
dequantised tensors, closed forms (one key, identical keys), invariance under
permuting the keys, the grouped-query head mapping, and the cast under a
given scale against exact arithmetic.  Mutants at the end must be rejected.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.fp8_oracle as O
from tests.test_oracle_pins import FINITE_CODES, _bf16_round, brute_force_encode, expected_cast


def _case(seed=61, B=3, Hq=8, Hkv=2, T=40, D=128):
    rng = np.random.Generator(np.random.PCG64(seed))
    fin = FINITE_CODES[np.abs(O.e4m3_decode(FINITE_CODES)) <= 8]   # moderate magnitudes
    q = rng.choice(fin, (B, Hq, D)).astype(np.uint8)
    k = rng.choice(fin, (B, Hkv, T, D)).astype(np.uint8)
    v = rng.choice(fin, (B, Hkv, T, D)).astype(np.uint8)
    return q, k, v, np.array([T, 1, 17][:B])


def _sdpa(q, sq, k, sk, v, sv, lens):
    B, Hq, D = q.shape
    G = Hq // k.shape[1]
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(lens[b])
        qt = torch.from_numpy(O.e4m3_decode(q[b]) * sq)[:, None, :]                 # [Hq, 1, D]
        kt = torch.from_numpy(O.e4m3_decode(k[b, :, :L]) * sk).repeat_interleave(G, 0)
        vt = torch.from_numpy(O.e4m3_decode(v[b, :, :L]) * sv).repeat_interleave(G, 0)
        out[b] = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, 0, :].numpy()
    return out


def check_attention_vs_torch(attn):
    q, k, v, lens = _case()
    sq, sk, sv = 0.05, 0.02, 0.3
    got = attn(q, sq, k, sk, v, sv, lens)
    ref = _sdpa(q, np.float32(sq), k, np.float32(sk), v, np.float32(sv), lens)
    return got.shape == ref.shape and np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def check_attention_closed_forms(attn):
    """One key: the output is that key's value row.  Identical keys: the
    output is the mean of the value rows.  No keys: zeros."""
    q, k, v, _ = _case(seed=62, B=3, Hq=4, Hkv=4, T=8)
    got = attn(q, 1.0, k, 1.0, v, 0.5, np.array([1, 8, 0]))
    want0 = O.e4m3_decode(v[0, :, 0]) * 0.5                                        # [Hkv=Hq, D]
    if not np.array_equal(got[0], want0):
        return False
    k2 = k.copy()
    k2[1] = k2[1, :, :1]                                                           # all keys of b=1 equal
    got = attn(q, 1.0, k2, 1.0, v, 0.5, np.array([1, 8, 0]))
    want1 = (O.e4m3_decode(v[1]) * 0.5).mean(axis=1)
    return np.max(np.abs(got[1] - want1)) <= 1e-12 * np.max(np.abs(want1)) and np.all(got[2] == 0)


def check_attention_permutation_and_groups(attn):
    """Permuting the attended keys (with their values) changes nothing; query
    heads of one group read that group's KV head only."""
    q, k, v, _ = _case(seed=63, B=1, Hq=8, Hkv=2, T=30)
    lens = np.array([30])
    base = attn(q, 0.05, k, 0.02, v, 0.3, lens)
    perm = np.random.Generator(np.random.PCG64(64)).permutation(30)
    if np.max(np.abs(attn(q, 0.05, k[:, :, perm], 0.02, v[:, :, perm], 0.3, lens) - base)) > 1e-12 * np.max(np.abs(base)):
        return False
    v2 = v.copy()
    v2[0, 1] = 0                                                                   # KV head 1 -> heads 4..7
    got = attn(q, 0.05, k, 0.02, v2, 0.3, lens)
    return np.array_equal(got[0, :4], base[0, :4]) and np.all(got[0, 4:] == 0)


def test_attention_vs_torch_sdpa():
    assert check_attention_vs_torch(O.decode_attention_ref)


def test_attention_closed_forms():
    assert check_attention_closed_forms(O.decode_attention_ref)


def test_attention_permutation_and_groups():
    assert check_attention_permutation_and_groups(O.decode_attention_ref)


def test_quant_with_scale_exact():
    rng = np.random.Generator(np.random.PCG64(65))
    x = _bf16_round(rng.standard_normal((6, 256)).astype(np.float32) * 3)
    x[2, 5] = 900.0                                  # beyond the calibrated range: saturates
    x[3, 9] = 0.000732421875                         # 3 * 2**-12: x RN(1/0.03) and x / 0.03 round apart
    for s in (np.float32(0.0123), np.float32(2.0 ** -4), np.float32(0.03)):
        q = O.quant_with_scale(x, s)
        q32 = expected_cast(x, s)
        assert np.array_equal(q, brute_force_encode(q32.ravel()).reshape(x.shape))
    assert (O.quant_with_scale(x, np.float32(0.0123))[2, 5] & 0x7F) == 0x7E
    # the planted element tells the multiply from the division
    s = np.float32(0.03)
    by_div = (np.float64(x[3, 9]) / np.float64(s)).astype(np.float32)
    assert brute_force_encode(np.array([by_div], np.float32))[0] != O.quant_with_scale(x, s)[3, 9]


# ---------------------------------------------------------------- mutations
def _attn_no_sqrt(q, sq, k, sk, v, sv, lens):
    # mistake: scores not divided by sqrt(D)
    return O.decode_attention_ref(q, sq * np.sqrt(128.0), k, sk, v, sv, lens)


def _attn_wrong_group(q, sq, k, sk, v, sv, lens):
    # mistake: head h reads KV head h % Hkv instead of h // (Hq / Hkv)
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    perm = [h % Hkv for h in range(Hq)]
    out = np.zeros((B, Hq, D))
    for h in range(Hq):
        kk = k[:, perm[h]:perm[h] + 1]
        vv = v[:, perm[h]:perm[h] + 1]
        out[:, h] = O.decode_attention_ref(q[:, h:h + 1], sq, kk, sk, vv, sv, lens)[:, 0]
    return out


def _attn_all_keys(q, sq, k, sk, v, sv, lens):
    # mistake: attends to every slot of the cache, not just the sequence's keys
    return O.decode_attention_ref(q, sq, k, sk, v, sv, np.full_like(lens, k.shape[2]))


@pytest.mark.parametrize("mutant", [_attn_no_sqrt, _attn_wrong_group, _attn_all_keys])
def test_mutant_attention_is_caught(mutant):
    checks = [check_attention_vs_torch(mutant), check_attention_closed_forms(mutant),
              check_attention_permutation_and_groups(mutant)]
    assert not all(checks)
