"""FP8 KV cache and decode attention on the GPU against the oracle: the
casts under calibrated scales bit for bit, the attention output within the
GEMM tolerance of tests/helpers.py (fp32 arithmetic against the oracle's
fp64), across head-group sizes, key splits, ragged and empty sequences, and
a full-size Qwen3-8B decode step on sampled sequences.

Inputs: q, K, V ~ N(0, 1) rounded to bf16; the scales are calibrated as the
pages describe (per-tensor amax / 448 of the same activations, from the
oracle's per-tensor rule)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.fp8_oracle as O
from fp8_block_scaled_05_gb300 import inputs as I
from tests.helpers import assert_gemm_close, bf16_to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_05_gb300 import build, ops as _ops
    build.build()
    return _ops


def _sync_ok(ops):
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0


def _setup(ops, B, Hq, Hkv, T, seed, q_gain=1.0):
    D = 128
    q = (I.normal_bf16(I.stream(seed, 1), (B, Hq, D)).float() * q_gain).to(torch.bfloat16)
    k = I.normal_bf16(I.stream(seed, 2), (B, Hkv, T, D))
    v = I.normal_bf16(I.stream(seed, 3), (B, Hkv, T, D))
    scales = {}
    codes = {}
    for name, x in (("q", q), ("k", k), ("v", v)):
        xn = bf16_to_np(x).reshape(-1, D)
        _, s = O.quant_per_tensor(xn)                          # calibration: amax / 448
        sd = torch.tensor([s], dtype=torch.float32, device="cuda")
        qd = torch.empty(xn.shape, dtype=torch.uint8, device="cuda")
        ops.fp8_quant_with_scale(x.reshape(-1, D).cuda(), qd, sd)
        scales[name] = (np.float32(s), sd)
        codes[name] = (O.quant_with_scale(xn, s).reshape(x.shape), qd.reshape(x.shape))
    _sync_ok(ops)
    for name in codes:
        assert np.array_equal(codes[name][1].cpu().numpy(), codes[name][0]), name
    return scales, codes


def _check(ops, scales, codes, lens, what):
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = ops.decode_attention(codes["q"][1], scales["q"][1], codes["k"][1], scales["k"][1], codes["v"][1],
                               scales["v"][1], lens_d)
    _sync_ok(ops)
    ref = O.decode_attention_ref(codes["q"][0], scales["q"][0], codes["k"][0], scales["k"][0], codes["v"][0],
                                 scales["v"][0], np.array(lens))
    got = bf16_to_np(out)
    empty = [b for b, L in enumerate(lens) if L == 0]
    for b in empty:
        assert np.all(got[b] == 0)
    keep = [b for b in range(len(lens)) if lens[b] > 0]
    assert_gemm_close(got[keep].reshape(-1, 128), ref[keep].reshape(-1, 128), what)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (8, 2), (16, 2)])
def test_decode_attention_single_split(ops, Hq, Hkv):
    scales, codes = _setup(ops, 3, Hq, Hkv, 300, seed=Hq * 10 + Hkv)
    _check(ops, scales, codes, [300, 1, 77], f"attention G={Hq // Hkv}")


def test_decode_attention_splits_and_edges(ops):
    """T = 1500: three key splits of 512; lengths at and around the split
    boundaries, one key, and an empty sequence."""
    lens = [1500, 700, 0, 513, 512, 1]
    scales, codes = _setup(ops, len(lens), 32, 8, 1500, seed=5)
    _check(ops, scales, codes, lens, "attention splits")


def test_decode_attention_sharp_softmax(ops):
    """Queries 8x larger: the softmax concentrates on few keys (exercises the
    running-max rescaling)."""
    scales, codes = _setup(ops, 2, 8, 2, 1100, seed=6, q_gain=8.0)
    _check(ops, scales, codes, [1100, 1025], "attention sharp")


def test_decode_attention_saturating_cache(ops):
    """Values beyond the calibrated range saturate in the cache: the cast and
    the attention still agree with the oracle."""
    scales, codes = _setup(ops, 2, 8, 2, 200, seed=7)
    D = 128
    k = I.normal_bf16(I.stream(7, 2), (2, 2, 200, D)).float() * 3.0         # 3x past the calibration
    kn = k.to(torch.bfloat16)
    s = scales["k"][0]
    qk = torch.empty((2 * 2 * 200, D), dtype=torch.uint8, device="cuda")
    ops.fp8_quant_with_scale(kn.reshape(-1, D).cuda(), qk, scales["k"][1])
    _sync_ok(ops)
    ref_codes = O.quant_with_scale(bf16_to_np(kn).reshape(-1, D), s)
    assert np.array_equal(qk.cpu().numpy(), ref_codes)
    assert np.any((ref_codes & 0x7F) == 0x7E)
    codes["k"] = (ref_codes.reshape(2, 2, 200, D), qk.reshape(2, 2, 200, D))
    _check(ops, scales, codes, [200, 150], "attention saturated cache")


def test_decode_attention_qwen8b_full_size_sampled(ops):
    """Qwen3-8B attention shape (32 query heads, 8 KV heads, D 128), 16
    sequences of up to 4096 cached tokens; 4 sequences checked against the
    oracle."""
    B, Hq, Hkv, T = 16, 32, 8, 4096
    rng = np.random.Generator(np.random.PCG64(9))
    lens = rng.integers(1, T + 1, B)
    lens[0] = T
    scales, codes = _setup(ops, B, Hq, Hkv, T, seed=8)
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = ops.decode_attention(codes["q"][1], scales["q"][1], codes["k"][1], scales["k"][1], codes["v"][1],
                               scales["v"][1], lens_d)
    _sync_ok(ops)
    pick = [0, 3, 9, 15]
    ref = O.decode_attention_ref(codes["q"][0][pick], scales["q"][0], codes["k"][0][pick], scales["k"][0],
                                 codes["v"][0][pick], scales["v"][0], lens[pick])
    assert_gemm_close(bf16_to_np(out)[pick].reshape(-1, 128), ref.reshape(-1, 128), "attention qwen8b")


def test_kv_cache_append_then_attend(ops):
    """Three decode steps: each appends the new token's K/V rows at every
    sequence's current length (one sequence already full: skipped), then
    attends; the cache rows and the outputs against the oracle, the other
    cache slots untouched."""
    B, Hq, Hkv, T, D = 3, 8, 2, 64, 128
    scales, codes = _setup(ops, B, Hq, Hkv, T, seed=11)
    lens = np.array([10, 0, T])
    kc_o, vc_o = codes["k"][0].copy(), codes["v"][0].copy()
    kc_d, vc_d = codes["k"][1].clone(), codes["v"][1].clone()
    for step in range(3):
        kn = I.normal_bf16(I.stream(20 + step, 1), (B, Hkv, D))
        vn = I.normal_bf16(I.stream(20 + step, 2), (B, Hkv, D))
        lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
        ops.fp8_kv_cache_append(kn.cuda(), vn.cuda(), scales["k"][1], scales["v"][1], lens_d, kc_d, vc_d)
        for b in range(B):
            if lens[b] < T:
                kc_o[b, :, lens[b]] = O.quant_with_scale(bf16_to_np(kn[b]), scales["k"][0])
                vc_o[b, :, lens[b]] = O.quant_with_scale(bf16_to_np(vn[b]), scales["v"][0])
        lens = np.minimum(lens + 1, T)
        lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
        out = ops.decode_attention(codes["q"][1], scales["q"][1], kc_d, scales["k"][1], vc_d, scales["v"][1], lens_d)
        _sync_ok(ops)
        assert np.array_equal(kc_d.cpu().numpy(), kc_o) and np.array_equal(vc_d.cpu().numpy(), vc_o)
        ref = O.decode_attention_ref(codes["q"][0], scales["q"][0], kc_o, scales["k"][0], vc_o, scales["v"][0], lens)
        assert_gemm_close(bf16_to_np(out).reshape(-1, D), ref.reshape(-1, D), f"append step {step}")
