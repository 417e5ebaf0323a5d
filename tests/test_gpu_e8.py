"""Power-of-two scales stored as UE8M0 bytes on the GPU: the _e8 quantisers
write the codes of the power-of-two quantisers and the bytes of their scales
(against the oracle), and the MX GEMM fed the bytes (FP8_GEMM_SCALES_E8) gives
bit for bit the output it gives with the fp32 scales -- the same arithmetic."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.fp8_oracle as O
from fp8_block_scaled_05_gb300 import inputs as I
from tests.helpers import bf16_to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_05_gb300 import build, ops as _ops
    build.build()
    return _ops


def _sync_ok(ops):
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0


def _quant_e8(ops, a, w):
    M, K = a.shape
    N = w.shape[0]
    qa = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.empty((K // 128, ops.round_up(M, 4)), dtype=torch.uint8, device="cuda")
    qw = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty((N // 128, K // 128), dtype=torch.uint8, device="cuda")
    ops.fp8_quant_act_1x128_e8(a.cuda(), qa, sa)
    ops.fp8_quant_weight_128x128_e8(w.cuda(), qw, sw)
    return qa, sa, qw, sw


@pytest.mark.parametrize("M,N,K", [(300, 384, 640), (4096, 1536, 4096), (1, 256, 256)])
def test_e8_quantisers_and_gemm(ops, M, N, K):
    a = I.normal_bf16(I.stream(M + K, 1), (M, K))
    w = I.normal_bf16(I.stream(N + K, 3), (N, K), std=0.02)
    an = bf16_to_np(a).copy()
    an[0, :128] *= 2.0 ** -120                         # scales near the bottom of the UE8M0 range
    a = torch.from_numpy(an).to(torch.bfloat16)
    qa8, sa8, qw8, sw8 = _quant_e8(ops, a, w)
    qa, sa = ops.quant_act(a.cuda(), True)
    qw, sw = ops.quant_weight(w.cuda(), True)
    _sync_ok(ops)
    # codes identical to the fp32-scale quantisers, bytes = UE8M0 of their scales
    assert torch.equal(qa8, qa) and torch.equal(qw8, qw)
    qa_o, sa_o = O.quant_act_1x128(bf16_to_np(a), True)
    qw_o, sw_o = O.quant_weight_128x128(bf16_to_np(w), True)
    assert np.array_equal(qa8.cpu().numpy(), qa_o)
    assert np.array_equal(sa8[:, :M].cpu().numpy(), O.scale_to_ue8m0(sa_o.T))
    assert np.array_equal(sw8.cpu().numpy(), O.scale_to_ue8m0(sw_o))
    # the MX GEMM on the bytes equals the MX GEMM on the fp32 scales, bit for bit
    c8 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ops.fp8_blockscaled_gemm(qa8, sa8, qw8, sw8, c8, ops.FP8_GEMM_SCALES_E8, ops.workspace_for(M, N, K, 1, "cuda"))
    c = ops.gemm(qa, sa, qw, sw, pow2=True, path="mx")
    _sync_ok(ops)
    assert torch.equal(c8, c)


def test_e8_grouped_gemm(ops):
    offs = [0, 5, 5, 140, 300]
    G, N, K = 4, 384, 256
    a = I.normal_bf16(I.stream(1, 1), (offs[-1], K))
    w = I.normal_bf16(I.stream(1, 3), (G, N, K), std=0.02)
    qa8 = torch.empty((offs[-1], K), dtype=torch.uint8, device="cuda")
    sa8 = torch.empty((K // 128, ops.round_up(offs[-1], 4)), dtype=torch.uint8, device="cuda")
    ops.fp8_quant_act_1x128_e8(a.cuda(), qa8, sa8)
    qw8 = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
    sw8 = torch.empty((G, N // 128, K // 128), dtype=torch.uint8, device="cuda")
    qw = torch.empty_like(qw8)
    sw = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device="cuda")
    for g in range(G):
        ops.fp8_quant_weight_128x128_e8(w[g].cuda(), qw8[g], sw8[g])
        ops.fp8_quant_weight_128x128(w[g].cuda(), qw[g], sw[g], ops.FP8_SCALE_POW2)
    qa, sa = ops.quant_act(a.cuda(), True)
    offs_d = torch.tensor(offs, dtype=torch.int32, device="cuda")
    c8 = torch.empty((offs[-1], N), dtype=torch.bfloat16, device="cuda")
    ops.fp8_blockscaled_grouped_gemm(qa8, sa8, offs_d, qw8, sw8, c8, ops.FP8_GEMM_SCALES_E8)
    c = ops.grouped_gemm(qa, sa, offs_d, qw, sw, True, "mx")
    _sync_ok(ops)
    assert torch.equal(qw8, qw) and torch.equal(c8, c)
