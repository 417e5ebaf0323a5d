"""The pieced, parallel application of the oracle used by the whole-output
GPU tests (tests/oracle_par.py) returns exactly what the oracle returns for
the whole tensor: quantisers by row, 128-row band and column ranges, and the
fp64 GEMM reference by column blocks."""
from __future__ import annotations

import numpy as np
import pytest

import oracle.fp8_oracle as O
from fp8_block_scaled_05_gb300 import inputs as I
from tests import oracle_par as par
from tests.helpers import bf16_to_np


@pytest.fixture(scope="module")
def pool():
    par.pool()
    yield
    par.shutdown()


@pytest.mark.parametrize("pow2", [False, True])
def test_pieces_equal_the_whole(pool, pow2):
    x = bf16_to_np(I.normal_bf16(I.stream(3, 1), (1000, 1024)))
    x[5, :128] = 0.0
    x[7, 3] = 3.0e38
    w = bf16_to_np(I.normal_bf16(I.stream(3, 2), (640, 1024), std=0.02))
    for got, want in ((par.quant_act_1x128(x, pow2), O.quant_act_1x128(x, pow2)),
                      (par.quant_weight_128x128(w, pow2), O.quant_weight_128x128(w, pow2)),
                      (par.quant_act_128x1(x[:700], pow2), O.quant_act_128x1(x[:700], pow2))):
        assert all(np.array_equal(g, h) for g, h in zip(got, want))
    qa, sa = O.quant_act_1x128(x, pow2)
    qw, sw = O.quant_weight_128x128(w, pow2)
    assert np.array_equal(par.gemm_ref(qa, sa, qw, sw, cols=256), O.gemm_ref(qa, sa, qw, sw))
