"""The decode GEMM entry point that allocates nothing,
fp8_blockscaled_gemm_skinny_noalloc, checked against the regular
fp8_blockscaled_gemm (skinny path, caller-provided workspace) and against the
oracle.

The no-allocation entry point is for callers that cannot call cudaMalloc:
plugins inside a runtime that reserved all device memory at start-up (a late
allocation fails or escapes the runtime's accounting), and decode loops where
an allocation would synchronise the device.  It keeps its reduction scratch in
a fixed array that the library owns, shared by every call.

Both entry points run the same kernel with the same division of the K-blocks
over the CTAs and the same fixed-order reduction, so their outputs must be
bit-identical; the output is also checked against the oracle's fp64
reference on the oracle's own quantisation of the inputs.

This file is named so that pytest collects it last: a run that stops at the
first failure has then already run every other test.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.fp8_oracle as O
from fp8_block_scaled_05_gb300 import inputs as I
from tests.helpers import assert_gemm_close, bf16_to_np

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_05_gb300 import build, ops as _ops
    build.build()
    return _ops


def _skinny_scratch(ops, M, N, K):
    """The skinny path's reduction scratch as the header states it: 0 when no
    output tile is shared by two CTAs, else 64 KiB of tickets plus
    (P + T - 1) * NT * 128 fp32 partials, with P the CTA count fp8_gemm_plan
    reports for the skinny path on this GPU."""
    path, P = ops.fp8_gemm_plan(M, N, K, ops.FP8_GEMM_PATH_SKINNY)
    assert path == ops.FP8_GEMM_PATH_SKINNY
    nt = 16 if M <= 16 else 32 if M <= 32 else 64 if M <= 64 else 128
    KB = K // 128
    T = (N // 128) * -(-M // nt)
    U = T * KB
    shared = any((c * U // P) % KB for c in range(1, P))
    return 65536 + (P + T - 1) * nt * 128 * 4 if shared else 0


def _operands(M, N, K, seed):
    """Oracle quantisation of seeded inputs, and the same codes and scales as
    device tensors in the library's layouts."""
    a = I.normal_bf16(I.stream(seed, 1), (M, K))
    w = I.normal_bf16(I.stream(seed, 2), (N, K), std=0.02)
    qa, sa = O.quant_act_1x128(bf16_to_np(a))
    qw, sw = O.quant_weight_128x128(bf16_to_np(w))
    lds = (M + 3) // 4 * 4
    sa_dev = torch.zeros((K // 128, lds), dtype=torch.float32)
    sa_dev[:, :M] = torch.from_numpy(np.ascontiguousarray(sa.T))
    dev = (torch.from_numpy(qa).cuda(), sa_dev.cuda(), torch.from_numpy(qw).cuda(),
           torch.from_numpy(np.ascontiguousarray(sw)).cuda())
    return (qa, sa, qw, sw), dev


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(ops):
    # Decode problems of different tile layouts, run back to back so that each
    # call finds the scratch as the previous one left it: one token chunk
    # (M = 8, 64) and two 128-token chunks (M = 200); every one of them
    # shares some output tiles between CTAs, so the reduction's tickets and
    # partials are used.
    cases = [(8, 6144, 4096, 1), (64, 4096, 14336, 2), (200, 256, 4096, 3), (8, 6144, 4096, 1)]
    for M, N, K, _ in cases:
        need = _skinny_scratch(ops, M, N, K)
        assert 0 < need <= SCRATCH_BYTES, (M, N, K, need)
        assert need <= ops.fp8_gemm_workspace_size(M, N, K, 1)
    operands = {seed: _operands(M, N, K, seed) for M, N, K, seed in cases}
    outs = []
    for M, N, K, seed in cases:
        _, (qa, sa, qw, sw) = operands[seed]
        c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        ops.fp8_blockscaled_gemm_skinny_noalloc(qa, sa, qw, sw, c)
        outs.append(c)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    for (M, N, K, seed), c in zip(cases, outs):
        (qa_o, sa_o, qw_o, sw_o), (qa, sa, qw, sw) = operands[seed]
        ref = ops.gemm(qa, sa, qw, sw, path="skinny")
        torch.cuda.synchronize()
        assert ops.fp8_last_device_status() == 0
        assert torch.equal(c, ref), f"no-alloc differs from the workspace path, M={M} N={N} K={K}"
        assert_gemm_close(bf16_to_np(c), O.gemm_ref(qa_o, sa_o, qw_o, sw_o), f"no-alloc M={M} N={N} K={K}")


def test_noalloc_rejects_problems_larger_than_its_scratch(ops):
    # The first of these decode shapes whose reduction scratch, from the CTA
    # count the library plans on this GPU, exceeds the fixed array: the call
    # must refuse before launching.
    shapes = [(256, 4096, 14336), (256, 8192, 14336), (256, 16384, 16384), (256, 65536, 16384)]
    big = [s for s in shapes if _skinny_scratch(ops, *s) > SCRATCH_BYTES]
    assert big, "no candidate shape needs more scratch than the array holds"
    M, N, K = big[0]
    qa = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.ones((K // 128, M), dtype=torch.float32, device="cuda")
    qw = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    sw = torch.ones((N // 128, K // 128), dtype=torch.float32, device="cuda")
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.FP8Error) as e:
        ops.fp8_blockscaled_gemm_skinny_noalloc(qa, sa, qw, sw, c)
    assert e.value.status == 5   # FP8_ERR_WORKSPACE
