"""GPU parity of the two quantisers with the CPU oracle: codes and scales
bit-exact, on the workload inputs, exhaustive bf16 plantings, ragged and
degenerate shapes."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.fp8_oracle as O
from fp8_block_scaled_05_gb300 import inputs as I
from tests.helpers import amax_sweep, bf16_to_np, planted_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_05_gb300 import build, ops as _ops
    build.build()
    return _ops


def _act_gpu(ops, x_bf16_cpu: torch.Tensor, pow2: bool, ldx_pad=0, lds_pad=0, ldq_pad=0):
    M, K = x_bf16_cpu.shape
    xb = torch.zeros((M, K + ldx_pad), dtype=torch.bfloat16, device="cuda")
    xb[:, :K] = x_bf16_cpu.cuda()
    x = xb[:, :K]
    qb = torch.full((M, K + ldq_pad), 0xAA, dtype=torch.uint8, device="cuda")
    q = qb[:, :K]
    lds = ops.round_up(max(M, 1), 4) + lds_pad
    s = torch.full((K // 128, lds), -7.0, dtype=torch.float32, device="cuda")
    ops.fp8_quant_act_1x128(x, q, s, ops.FP8_SCALE_POW2 if pow2 else 0)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    return qb.cpu().numpy(), s.cpu().numpy()


def _check_act(ops, x_cpu: torch.Tensor, pow2: bool, **pads):
    M, K = x_cpu.shape
    qb, s = _act_gpu(ops, x_cpu, pow2, **pads)
    qo, so = O.quant_act_1x128(bf16_to_np(x_cpu), pow2)
    assert np.array_equal(qb[:, :K], qo), "codes differ"
    assert np.array_equal(s[:, :M].T.view(np.uint32), so.view(np.uint32)), "scales differ"
    # nothing written outside the logical extents
    if qb.shape[1] > K:
        assert np.all(qb[:, K:] == 0xAA)
    if s.shape[1] > M:
        assert np.all(s[:, M:] == -7.0)


@pytest.mark.parametrize("pow2", [False, True])
def test_act_tiny(ops, pow2):
    _check_act(ops, I.tiny().a, pow2)


@pytest.mark.parametrize("pow2", [False, True])
def test_act_exhaustive_bf16(ops, pow2):
    x = planted_rows(amax_sweep(7), 128, 8)
    _check_act(ops, torch.from_numpy(x).to(torch.bfloat16), pow2)


@pytest.mark.parametrize("M,K", [(1, 128), (3, 256), (33, 1152), (127, 640), (129, 384)])
@pytest.mark.parametrize("pow2", [False, True])
def test_act_ragged(ops, M, K, pow2):
    g = I.stream(1, M * 7 + K)
    x = I.normal_bf16(g, (M, K))
    x[0, :128] = 0.0                                 # all-zero block
    if K >= 256:
        x[-1, 128:256] = torch.tensor(2.0 ** -130).to(torch.bfloat16)   # subnormal amax
    _check_act(ops, x, pow2, ldx_pad=8, lds_pad=4, ldq_pad=16)


def test_act_empty(ops):
    q = torch.empty((0, 256), dtype=torch.uint8, device="cuda")
    s = torch.empty((2, 4), dtype=torch.float32, device="cuda")
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    ops.fp8_quant_act_1x128(x, q, s)


@pytest.mark.parametrize("layer", ["qkv", "down"])
def test_act_llama_full_size_sampled_rows(ops, layer):
    case = I.llama8b_layers(layers=[layer])[0]
    x = case.a.cuda()
    q, s = ops.quant_act(x)
    torch.cuda.synchronize()
    rows = np.sort(np.random.Generator(np.random.PCG64(3)).choice(x.shape[0], 48, replace=False))
    qo, so = O.quant_act_1x128(bf16_to_np(case.a[rows]))
    assert np.array_equal(q[rows].cpu().numpy(), qo)
    assert np.array_equal(s[:, rows].T.cpu().numpy().view(np.uint32), so.view(np.uint32))


# ------------------------------------------------------------------ weights
def _check_w(ops, w_cpu: torch.Tensor, pow2: bool, ldw_pad=0, ldq_pad=0):
    N, K = w_cpu.shape
    wb = torch.zeros((N, K + ldw_pad), dtype=torch.bfloat16, device="cuda")
    wb[:, :K] = w_cpu.cuda()
    qb = torch.full((N, K + ldq_pad), 0xAA, dtype=torch.uint8, device="cuda")
    s = torch.empty((N // 128, K // 128), dtype=torch.float32, device="cuda")
    ops.fp8_quant_weight_128x128(wb[:, :K], qb[:, :K], s, ops.FP8_SCALE_POW2 if pow2 else 0)
    torch.cuda.synchronize()
    qo, so = O.quant_weight_128x128(bf16_to_np(w_cpu), pow2)
    qn = qb.cpu().numpy()
    assert np.array_equal(qn[:, :K], qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    if ldq_pad:
        assert np.all(qn[:, K:] == 0xAA)


@pytest.mark.parametrize("pow2", [False, True])
def test_weight_tiny(ops, pow2):
    _check_w(ops, I.tiny().w, pow2)


@pytest.mark.parametrize("pow2", [False, True])
def test_weight_exhaustive_bf16(ops, pow2):
    # each 128x128 tile holds 16384 planted values with one amax
    rows = planted_rows(amax_sweep(13), 128 * 128, 1)           # [tiles, 16384]
    tiles = rows.reshape(-1, 128, 128)
    nt = tiles.shape[0]
    cols = 4
    nt_pad = (-nt) % cols
    if nt_pad:
        tiles = np.concatenate([tiles, tiles[:nt_pad]])
    w = tiles.reshape(-1, cols, 128, 128).transpose(0, 2, 1, 3).reshape(-1, cols * 128)
    _check_w(ops, torch.from_numpy(np.ascontiguousarray(w)).to(torch.bfloat16), pow2)


@pytest.mark.parametrize("N,K", [(128, 128), (384, 640), (256, 1152)])
def test_weight_ragged(ops, N, K):
    w = I.normal_bf16(I.stream(2, N + K), (N, K), std=0.02)
    w[:128, :128] = 0.0
    _check_w(ops, w, False, ldw_pad=16, ldq_pad=32)


def test_weight_llama_full_size_sampled_tiles(ops):
    case = I.llama8b_layers(layers=["gate_up"])[0]
    w = case.w.cuda()
    q, s = ops.quant_weight(w)
    torch.cuda.synchronize()
    rng = np.random.Generator(np.random.PCG64(4))
    NB, KB = w.shape[0] // 128, w.shape[1] // 128
    for nb, kb in zip(rng.integers(0, NB, 12), rng.integers(0, KB, 12)):
        t = case.w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
        qo, so = O.quant_weight_128x128(bf16_to_np(t))
        assert np.array_equal(q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128].cpu().numpy(), qo)
        assert s[nb, kb].item() == float(so[0, 0])


# ------------------------------------------------------------ one launch for a layer
def _layer_gpu(ops, x, w, pow2):
    """fp8_quant_act_weight on device copies of x [M, K] and w [N, K]; the
    output buffers are pre-filled so that a missed write shows."""
    M, K = x.shape
    N = w.shape[0]
    qa = torch.full((M, K), 0xAA, dtype=torch.uint8, device="cuda")
    sa = torch.full((K // 128, ops.round_up(max(M, 1), 4)), -7.0, dtype=torch.float32, device="cuda")
    qw = torch.full((N, K), 0xAA, dtype=torch.uint8, device="cuda")
    sw = torch.full((N // 128, K // 128), -7.0, dtype=torch.float32, device="cuda")
    ops.fp8_quant_act_weight(x.cuda(), qa, sa, w.cuda(), qw, sw, ops.FP8_SCALE_POW2 if pow2 else 0)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    return qa, sa, qw, sw


@pytest.mark.parametrize("M,N,K", [(300, 384, 640), (1, 128, 128), (0, 256, 256), (129, 1152, 384)])
@pytest.mark.parametrize("pow2", [False, True])
def test_act_weight_one_launch_ragged(ops, M, N, K, pow2):
    """The layer quantiser writes what the oracle's two quantisers give, and
    nothing outside the activations' M rows."""
    x = I.normal_bf16(I.stream(M + 3, 1), (max(M, 1), K))[:M].contiguous()
    w = I.normal_bf16(I.stream(N + 5, 2), (N, K), std=0.02)
    qa, sa, qw, sw = _layer_gpu(ops, x, w, pow2)
    qw_o, sw_o = O.quant_weight_128x128(bf16_to_np(w), pow2)
    assert np.array_equal(qw.cpu().numpy(), qw_o) and np.array_equal(sw.cpu().numpy(), sw_o)
    if M:
        qa_o, sa_o = O.quant_act_1x128(bf16_to_np(x), pow2)
        assert np.array_equal(qa.cpu().numpy(), qa_o)
        s = sa.cpu().numpy()
        assert np.array_equal(s[:, :M].T, sa_o) and np.all(s[:, M:] == -7.0)


@pytest.mark.parametrize("pow2", [False, True])
def test_act_weight_one_launch_equals_two_launches_llama(ops, pow2):
    """All three Llama-3.1-8B layers at full size: codes and scales of the one
    launch are bit-identical to the two separate quantisers' (which the
    whole-output tests compare with the oracle)."""
    mode = ops.FP8_SCALE_POW2 if pow2 else 0
    for c in I.llama8b_layers(0):
        x, w = c.a.cuda(), c.w.cuda()
        qa, sa, qw, sw = _layer_gpu(ops, c.a, c.w, pow2)
        qa2, sa2 = torch.empty_like(qa), torch.empty_like(sa)
        qw2, sw2 = torch.empty_like(qw), torch.empty_like(sw)
        ops.fp8_quant_act_1x128(x, qa2, sa2, mode)
        ops.fp8_quant_weight_128x128(w, qw2, sw2, mode)
        torch.cuda.synchronize()
        M = x.shape[0]
        assert torch.equal(qa, qa2) and torch.equal(sa[:, :M], sa2[:, :M]), c.name
        assert torch.equal(qw, qw2) and torch.equal(sw, sw2), c.name
