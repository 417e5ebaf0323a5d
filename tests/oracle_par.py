"""The CPU oracle's block quantisers and GEMM reference applied to whole
full-size tensors, in pieces.

The quantisers run in spawned worker processes (spawned, so no worker
inherits a CUDA context) over independent ranges: a 1x128 block lies in one
row, a 128x128 tile in one band of 128 rows, and a 128x1 block in one
column, so the pieces, put back together, are exactly what the oracle
returns for the whole tensor.  The fp64 GEMM reference runs in this process
(numpy's BLAS is multi-threaded) over column blocks of the output, each a
call of the oracle's own reference on the operands' matching rows.

Test infrastructure only; nothing here computes anything the oracle does not.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np

import oracle.fp8_oracle as O

_pool = None
_workers = 1


def pool() -> ProcessPoolExecutor:
    global _pool, _workers
    if _pool is None:
        _workers = max(1, min(16, len(os.sched_getaffinity(0))))
        _pool = ProcessPoolExecutor(max_workers=_workers, mp_context=mp.get_context("spawn"))
    return _pool


def shutdown() -> None:
    global _pool
    if _pool is not None:
        _pool.shutdown()
        _pool = None


def _ranges(n: int, align: int, pieces: int):
    step = max(align, -(-n // pieces) // align * align or align)
    return [(i, min(n, i + step)) for i in range(0, n, step)]


def _qa(args):
    x, pow2 = args
    return O.quant_act_1x128(x, pow2)


def _qw(args):
    w, pow2 = args
    return O.quant_weight_128x128(w, pow2)


def _qt(args):
    x, pow2 = args
    return O.quant_act_128x1(x, pow2)


def quant_act_1x128(x: np.ndarray, pow2: bool = False):
    """O.quant_act_1x128 of x [M, K], by row ranges."""
    p = pool()
    parts = list(p.map(_qa, [(x[a:b], pow2) for a, b in _ranges(x.shape[0], 1, 4 * _workers)]))
    return np.concatenate([q for q, _ in parts]), np.concatenate([s for _, s in parts])


def quant_weight_128x128(w: np.ndarray, pow2: bool = False):
    """O.quant_weight_128x128 of w [N, K], by bands of 128-row multiples."""
    p = pool()
    parts = list(p.map(_qw, [(w[a:b], pow2) for a, b in _ranges(w.shape[0], 128, 4 * _workers)]))
    return np.concatenate([q for q, _ in parts]), np.concatenate([s for _, s in parts])


def quant_act_128x1(x: np.ndarray, pow2: bool = False):
    """O.quant_act_128x1 of x [M, K] (returned transposed: qt [K, Mp], st
    [K, Mp/128]), by column ranges."""
    p = pool()
    parts = list(p.map(_qt, [(np.ascontiguousarray(x[:, a:b]), pow2)
                             for a, b in _ranges(x.shape[1], 1, 4 * _workers)]))
    return np.concatenate([q for q, _ in parts]), np.concatenate([s for _, s in parts])


def gemm_ref(qa, sa, qw, sw, cols: int = 4096) -> np.ndarray:
    """O.gemm_ref(qa, sa, qw, sw) [M, N] in fp64, one block of `cols` output
    columns (weight rows, a multiple of 128) at a time."""
    M, N = qa.shape[0], qw.shape[0]
    out = np.empty((M, N), np.float64)
    for n0 in range(0, N, cols):
        n1 = min(N, n0 + cols)
        out[:, n0:n1] = O.gemm_ref(qa, sa, qw[n0:n1], sw[n0 // 128:(n1 + 127) // 128])
    return out


def _moe_wgrad_expert(args):
    dy, x, pow2 = args
    qg, sg = O.quant_act_128x1(dy, pow2)
    qx, sx = O.quant_act_128x1(x, pow2)
    return qg, sg, qx, sx, O.wgrad_ref(qg, sg, qx, sx)


def moe_wgrad_experts(dy: np.ndarray, x: np.ndarray, offsets, pow2: bool = False):
    """Yields (g, qt_dy, st_dy, qt_x, st_x, dW_g) for every expert with
    tokens: O.quant_act_128x1 of the expert's rows of dy and x, and
    O.wgrad_ref of them (fp64), one expert per task."""
    offsets = [int(v) for v in offsets]
    live = [g for g in range(len(offsets) - 1) if offsets[g + 1] > offsets[g]]
    tasks = ((dy[offsets[g]:offsets[g + 1]], x[offsets[g]:offsets[g + 1]], pow2) for g in live)
    for g, r in zip(live, pool().map(_moe_wgrad_expert, tasks)):
        yield (g,) + tuple(r)

