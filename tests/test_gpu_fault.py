"""Failure detection inside the GEMM kernels, exercised without a GPU fault.

Every wait inside the kernels is bounded; a wait that runs out records
FP8_ERR_TIMEOUT in the device status word, the kernel releases its TMEM and
returns.  Here the bound is shortened to 20 ms and the TMA producer leaves
out the first K-block's operands (fp8_debug_inject), so the waits on them run
out for certain: the status word must read FP8_ERR_TIMEOUT, and afterwards a
normal call on the same CUDA context must still compute the right result.
Covered: the promote kernel (plain and with its fused output quantisation)
and the decode (skinny) kernel with one and two token chunks.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.fp8_oracle as O
from fp8_block_scaled_05_gb300 import inputs as I
from tests.helpers import assert_gemm_close, bf16_to_np

pytestmark = pytest.mark.gpu

FP8_ERR_TIMEOUT = 8
SHORT_WAIT_NS = 20_000_000


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_05_gb300 import build, ops as _ops
    build.build()
    return _ops


def _operands(M, N, K, seed):
    a = I.normal_bf16(I.stream(seed, 1), (M, K))
    w = I.normal_bf16(I.stream(seed, 2), (N, K), std=0.02)
    qa, sa = O.quant_act_1x128(bf16_to_np(a))
    qw, sw = O.quant_weight_128x128(bf16_to_np(w))
    lds = (M + 3) // 4 * 4
    sa_dev = torch.zeros((K // 128, lds), dtype=torch.float32)
    sa_dev[:, :M] = torch.from_numpy(np.ascontiguousarray(sa.T))
    dev = (torch.from_numpy(qa).cuda(), sa_dev.cuda(), torch.from_numpy(qw).cuda(),
           torch.from_numpy(np.ascontiguousarray(sw)).cuda())
    return dev, O.gemm_ref(qa, sa, qw, sw)


@pytest.mark.parametrize("kernel,M,N,K", [("promote", 384, 512, 1024), ("promote_fused", 384, 512, 1024),
                                          ("skinny", 8, 1024, 2048), ("skinny", 200, 512, 4096)])
def test_wait_timeout_is_reported_and_the_context_survives(ops, kernel, M, N, K):
    (qa, sa, qw, sw), ref = _operands(M, N, K, seed=M + K)
    ws = ops.workspace_for(M, N, K, 1, "cuda")
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    if kernel == "promote_fused":
        # the promote kernel with the next layer's quantisation in its epilogue
        qc = torch.empty((M, N), dtype=torch.uint8, device="cuda")
        sc = torch.empty((N // 128, (M + 3) // 4 * 4), dtype=torch.float32, device="cuda")

        def run():
            ops.fp8_blockscaled_gemm_quant(qa, sa, qw, sw, c, qc, sc, ops.FP8_GEMM_PATH_PROMOTE, 0, ws)
    else:
        flags = ops.FP8_GEMM_PATH_SKINNY if kernel == "skinny" else ops.FP8_GEMM_PATH_PROMOTE

        def run():
            ops.fp8_blockscaled_gemm(qa, sa, qw, sw, c, flags, ws)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    ops.fp8_debug_inject(True, SHORT_WAIT_NS)
    try:
        run()
        torch.cuda.synchronize()
        assert ops.fp8_last_device_status() == FP8_ERR_TIMEOUT
    finally:
        ops.fp8_debug_inject(False, 0)
    if ws is not None:
        ws.zero_()   # the aborted call may have left reduction tickets behind
    # the context is still usable: the same call now computes the layer
    c.fill_(float("nan"))
    run()
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    assert_gemm_close(bf16_to_np(c), ref, f"{kernel} after an injected timeout")


def test_inject_rejects_a_limit_above_the_default(ops):
    with pytest.raises(ops.FP8Error):
        ops.fp8_debug_inject(False, 3_000_000_000)
    ops.fp8_debug_inject(False, 0)
