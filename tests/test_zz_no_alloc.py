"""The decode GEMM entry point that allocates nothing,
fp8_blockscaled_gemm_skinny_noalloc, checked against the regular
fp8_blockscaled_gemm (skinny path, caller-provided workspace).

The no-allocation entry point is for callers that cannot call cudaMalloc:
plugins inside a runtime that reserved all device memory at start-up (a late
allocation fails or escapes the runtime's accounting), and decode loops where
an allocation would synchronise the device.  It keeps its split-K scratch in
a fixed array that the library owns, shared by every call.

This file is named so that pytest collects it last: a run that stops at the
first failure has then already run every other test.
"""
from __future__ import annotations

import pytest
import torch

from fp8_block_scaled_05_gb300 import inputs as I
from tests.helpers import assert_gemm_close, bf16_to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_05_gb300 import build, ops as _ops
    build.build()
    return _ops


def _operands(ops, M, N, K, seed):
    a = I.normal_bf16(I.stream(seed, 1), (M, K)).cuda()
    w = I.normal_bf16(I.stream(seed, 2), (N, K), std=0.02).cuda()
    qa, sa = ops.quant_act(a)
    qw, sw = ops.quant_weight(w)
    return qa, sa, qw, sw


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(ops):
    # Two different decode problems; both fit the 8 MiB scratch (the second
    # needs ~4 MiB of partials), and the second call reuses the scratch the
    # first one left behind.
    cases = [(8, 6144, 4096, 1), (64, 4096, 14336, 2)]
    operands = [_operands(ops, M, N, K, seed) for M, N, K, seed in cases]
    outs = []
    for (M, N, K, _), (qa, sa, qw, sw) in zip(cases, operands):
        c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        ops.fp8_blockscaled_gemm_skinny_noalloc(qa, sa, qw, sw, c)
        outs.append(c)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    for (M, N, K, _), (qa, sa, qw, sw), c in zip(cases, operands, outs):
        ref = ops.gemm(qa, sa, qw, sw, path="skinny")
        torch.cuda.synchronize()
        assert ops.fp8_last_device_status() == 0
        assert_gemm_close(bf16_to_np(c), bf16_to_np(ref).astype("float64"), f"no-alloc M={M} N={N} K={K}")


def test_noalloc_rejects_problems_larger_than_its_scratch(ops):
    # M = 128, N = 2048, K = 16384 splits K nine ways: ~9.4 MB of split-K
    # partials, more than the fixed scratch, so the call must refuse before
    # launching.
    M, N, K = 128, 2048, 16384
    qa = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.ones((K // 128, M), dtype=torch.float32, device="cuda")
    qw = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    sw = torch.ones((N // 128, K // 128), dtype=torch.float32, device="cuda")
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.FP8Error) as e:
        ops.fp8_blockscaled_gemm_skinny_noalloc(qa, sa, qw, sw, c)
    assert e.value.status == 5   # FP8_ERR_WORKSPACE
