"""Per-tensor scaling on the GPU against the oracle: the two-pass quantiser
(amax reduction, then the cast) bit for bit, and the per-tensor-scaled GEMM
(the MX kernel with unit scale factors and the scale product applied in the
epilogue) within the GEMM tolerance of tests/helpers.py."""
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


def _act(seed, shape):
    a = I.normal_bf16(I.stream(seed, 8), shape)
    if shape[1] >= 256:
        a, _ = I.with_outlier_columns(a, I.stream(seed, 9), max(1, shape[1] // 100), 30.0)
    return a


@pytest.mark.parametrize("M,K", [(1, 128), (37, 640), (1000, 4096), (3, 16), (4096, 14336)])
@pytest.mark.parametrize("pow2", [False, True])
def test_quant_per_tensor_matches_oracle(ops, M, K, pow2):
    x = _act(M + K, (M, K))
    q, sa = ops.quant_tensor(x.cuda(), pow2)
    _sync_ok(ops)
    q_o, s_o = O.quant_per_tensor(bf16_to_np(x), pow2)
    assert float(sa[1]) == float(np.max(np.abs(bf16_to_np(x))))
    assert float(sa[0]) == float(s_o)
    assert np.array_equal(q.cpu().numpy(), q_o)


@pytest.mark.parametrize("pow2", [False, True])
def test_quant_per_tensor_edge_values(ops, pow2):
    # all zeros (scale 1, signed zero codes), a subnormal amax, a huge amax,
    # and a pitched input
    z = torch.zeros((5, 256), dtype=torch.bfloat16)
    z[2, 3] = -0.0
    q, sa = ops.quant_tensor(z.cuda(), pow2)
    _sync_ok(ops)
    q_o, s_o = O.quant_per_tensor(bf16_to_np(z), pow2)
    assert float(sa[0]) == float(s_o) == 1.0 and float(sa[1]) == 0.0
    assert np.array_equal(q.cpu().numpy(), q_o)
    for amax in (2.0 ** -130, 3.0e38):
        x = bf16_to_np(_act(7, (9, 384))).copy() * 0.0
        x[4, 100] = -amax
        x[1, 5] = amax / 3
        xt = torch.from_numpy(x).to(torch.bfloat16)
        q, sa = ops.quant_tensor(xt.cuda(), pow2)
        _sync_ok(ops)
        q_o, s_o = O.quant_per_tensor(bf16_to_np(xt), pow2)
        assert float(sa[0]) == float(s_o) and np.array_equal(q.cpu().numpy(), q_o)
    big = _act(11, (64, 1024)).cuda()
    xp = torch.empty((64, 1024 + 64), dtype=torch.bfloat16, device="cuda")
    xp[:, :1024] = big
    xp[:, 1024:] = 1.0e4                               # outside the view: must not count
    q = torch.empty((64, 1024 + 32), dtype=torch.uint8, device="cuda")
    sa = torch.empty(2, dtype=torch.float32, device="cuda")
    ops.fp8_quant_per_tensor(xp[:, :1024], q[:, :1024], sa, ops.FP8_SCALE_POW2 if pow2 else 0)
    _sync_ok(ops)
    q_o, s_o = O.quant_per_tensor(bf16_to_np(big.cpu()), pow2)
    assert float(sa[0]) == float(s_o) and np.array_equal(q[:, :1024].cpu().numpy(), q_o)


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (300, 384, 640), (1, 256, 256), (4096, 1536, 4096)])
def test_tensorscaled_gemm_matches_oracle(ops, M, N, K):
    """Ragged M, a half-empty 256-wide tile (N = 384), M = 1, and a last-wave
    K split (4096 x 1536: 32 x 6 = 192 tiles of 128 x 256; on 152 SMs the 40
    left over are split in two along K)."""
    a = _act(M + N, (M, K))
    w = I.normal_bf16(I.stream(N + K, 3), (N, K), std=0.02)
    qa, sa = ops.quant_tensor(a.cuda())
    qw, sw = ops.quant_tensor(w.cuda())
    c = ops.gemm_tensor(qa, sa, qw, sw)
    _sync_ok(ops)
    qa_o, sa_o = O.quant_per_tensor(bf16_to_np(a))
    qw_o, sw_o = O.quant_per_tensor(bf16_to_np(w))
    assert np.array_equal(qa.cpu().numpy(), qa_o) and np.array_equal(qw.cpu().numpy(), qw_o)
    assert_gemm_close(bf16_to_np(c), O.gemm_per_tensor_ref(qa_o, sa_o, qw_o, sw_o), f"per-tensor {M}x{N}x{K}")


def test_tensorscaled_gemm_exact_integer(ops):
    """Codes decoding to {-1, 0, 1}, sA = 0.25, sB = 8: every output is twice
    an integer of at most 8 significant bits, exact in bf16."""
    rng = np.random.Generator(np.random.PCG64(57))
    M, N, K = 200, 384, 256
    lut = np.array([0x00, 0x38, 0xB8], np.uint8)
    qa = lut[rng.integers(0, 3, (M, K))]
    qb = lut[rng.integers(0, 3, (N, K))]
    ref = O.gemm_per_tensor_ref(qa, np.float32(0.25), qb, np.float32(8.0))
    sa = torch.tensor([0.25, 0.0], dtype=torch.float32, device="cuda")
    sb = torch.tensor([8.0, 0.0], dtype=torch.float32, device="cuda")
    c = ops.gemm_tensor(torch.from_numpy(qa).cuda(), sa, torch.from_numpy(qb).cuda(), sb)
    _sync_ok(ops)
    assert np.array_equal(bf16_to_np(c), ref)


def test_tensorscaled_gemm_llama_qkv_full_size_sampled(ops):
    case = I.llama8b_layers(layers=["qkv"])[0]
    qa, sa = ops.quant_tensor(case.a.cuda())
    qw, sw = ops.quant_tensor(case.w.cuda())
    c = ops.gemm_tensor(qa, sa, qw, sw)
    _sync_ok(ops)
    qa_o, sa_o = O.quant_per_tensor(bf16_to_np(case.a))
    qw_o, sw_o = O.quant_per_tensor(bf16_to_np(case.w))
    assert np.array_equal(qa.cpu().numpy(), qa_o) and float(sa[0]) == float(sa_o)
    assert np.array_equal(qw.cpu().numpy(), qw_o) and float(sw[0]) == float(sw_o)
    rows = np.sort(np.random.Generator(np.random.PCG64(58)).choice(case.a.shape[0], 16, replace=False))
    ref = O.gemm_per_tensor_ref(qa_o[rows], sa_o, qw_o, sw_o)
    assert_gemm_close(bf16_to_np(c[rows]), ref, "per-tensor qkv")
