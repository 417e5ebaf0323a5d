"""Training-side path on the GPU against the oracle: the transposing
quantisers (128x1 activations, W^T), the dgrad GEMM (dX = dY W through the
ordinary block-scaled GEMM on W^T codes) and the wgrad GEMM (dW = dY^T X with
1x128 scales on both operands), on both large-M kernels.

Codes and scales are compared bit for bit; GEMM outputs within the GEMM
tolerance of tests/helpers.py.  Gradients dY are heavy-tailed and small
(Student-t, nu = 4, times 1e-4), activations normal with outlier columns,
weights normal (std 0.02).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.fp8_oracle as O
from fp8_block_scaled_05_gb300 import inputs as I
from tests.helpers import assert_gemm_close, bf16_to_np, sample_block_rows, weight_block_cols

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_05_gb300 import build, ops as _ops
    build.build()
    return _ops


def _grad(seed, shape):
    g = I.student_t_bf16(I.stream(seed, 7), shape, nu=4.0)
    return (g.float() * 1e-4).to(torch.bfloat16)


def _act(seed, shape):
    a = I.normal_bf16(I.stream(seed, 8), shape)
    if shape[1] >= 256:
        a, _ = I.with_outlier_columns(a, I.stream(seed, 9), max(1, shape[1] // 100), 30.0)
    return a


def _edge_act(M, K, seed):
    """Activations with the 128x1 edge cases planted: an all-zero token block
    of a column, a block whose amax is a bf16 subnormal, a tiny block, and a
    huge value."""
    x = bf16_to_np(_act(seed, (M, K))).copy()
    x[:128, 3] = 0.0
    x[:128, 4] = 0.0
    x[7, 4] = -2.0 ** -130
    x[:128, 5] *= 1e-30
    x[M - 1, K - 1] = 3.0e38
    return torch.from_numpy(x).to(torch.bfloat16)


def _sync_ok(ops):
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0


# ---------------------------------------------------------------- quantisers
@pytest.mark.parametrize("M,K", [(128, 128), (256, 384), (384, 640), (1024, 256)])
@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("rowwise", [False, True])
def test_quant_act_128x1_matches_oracle(ops, M, K, pow2, rowwise):
    x = _edge_act(M, K, seed=M + K)
    out = ops.quant_act_t(x.cuda(), pow2, rowwise=rowwise)
    _sync_ok(ops)
    qt_o, st_o = O.quant_act_128x1(bf16_to_np(x), pow2)
    assert np.array_equal(out[0].cpu().numpy(), qt_o)
    assert np.array_equal(out[1][:, :K].cpu().numpy(), st_o.T)
    if rowwise:
        q_o, s_o = O.quant_act_1x128(bf16_to_np(x), pow2)
        assert np.array_equal(out[2].cpu().numpy(), q_o)
        assert np.array_equal(out[3][:, :M].cpu().numpy(), s_o.T)
        # and the same bytes as the 1x128 quantiser's own kernel
        q1, s1 = ops.quant_act(x.cuda(), pow2)
        _sync_ok(ops)
        assert torch.equal(out[2], q1) and torch.equal(out[3][:, :M], s1[:, :M])


def test_quant_act_128x1_padded_pitches(ops):
    # qt rows and st rows longer than the data: the pitches are honoured and
    # the padding is left alone.
    M, K = 256, 256
    x = _act(5, (M, K)).cuda()
    qt = torch.full((K, M + 32), 0xAB, dtype=torch.uint8, device="cuda")
    st = torch.full((M // 128, K + 12), -1.0, dtype=torch.float32, device="cuda")
    ops.fp8_quant_act_128x1(x, qt[:, :M], st[:, :K])
    _sync_ok(ops)
    qt_o, st_o = O.quant_act_128x1(bf16_to_np(x.cpu()))
    assert np.array_equal(qt[:, :M].cpu().numpy(), qt_o)
    assert torch.all(qt[:, M:] == 0xAB) and torch.all(st[:, K:] == -1.0)
    assert np.array_equal(st[:, :K].cpu().numpy(), st_o.T)


@pytest.mark.parametrize("N,K", [(128, 128), (384, 256), (256, 640)])
@pytest.mark.parametrize("pow2", [False, True])
def test_quant_weight_t_matches_oracle(ops, N, K, pow2):
    w = I.normal_bf16(I.stream(N + K, 3), (N, K), std=0.02)
    wn = bf16_to_np(w).copy()
    wn[5, K - 3] = 2.0          # one block with a larger amax
    wn[128:256, :128] = 0.0     # an all-zero block (no-op when N = 128)
    w = torch.from_numpy(wn).to(torch.bfloat16)
    qt, st, q, s = ops.quant_weight_t(w.cuda(), pow2, with_w=True)
    _sync_ok(ops)
    qt_o, st_o = O.quant_weight_128x128_t(wn, pow2)
    assert np.array_equal(qt.cpu().numpy(), qt_o) and np.array_equal(st.cpu().numpy(), st_o)
    q1, s1 = ops.quant_weight(w.cuda(), pow2)
    _sync_ok(ops)
    assert torch.equal(q, q1) and torch.equal(s, s1)
    qt2, st2 = ops.quant_weight_t(w.cuda(), pow2)        # without W's own codes
    _sync_ok(ops)
    assert torch.equal(qt, qt2) and torch.equal(st, st2)


# ---------------------------------------------------------------- dgrad / wgrad
@pytest.mark.parametrize("T,N,K", [(128, 128, 128), (256, 384, 640), (300, 256, 384)])
@pytest.mark.parametrize("pow2", [False, True])
def test_dgrad_matches_oracle(ops, T, N, K, pow2):
    """dX [T, K] = dY [T, N] W [N, K] on W^T codes; T ragged in one case."""
    dy = _grad(T + N, (T, N))
    w = I.normal_bf16(I.stream(N + K, 3), (N, K), std=0.02)
    q_dy, s_dy = ops.quant_act(dy.cuda(), pow2)
    qt_w, st_w = ops.quant_weight_t(w.cuda(), pow2)
    dx = ops.gemm(q_dy, s_dy, qt_w, st_w, pow2=pow2, path="mx" if pow2 else "promote")
    _sync_ok(ops)
    q_o, s_o = O.quant_act_1x128(bf16_to_np(dy), pow2)
    qw_o, sw_o = O.quant_weight_128x128(bf16_to_np(w), pow2)
    assert_gemm_close(bf16_to_np(dx), O.dgrad_ref(q_o, s_o, qw_o, sw_o), f"dgrad {T}x{N}x{K}")


@pytest.mark.parametrize("T,N,K", [(128, 128, 128), (256, 384, 640), (512, 256, 384), (1024, 640, 256)])
@pytest.mark.parametrize("path,pow2", [("promote", False), ("promote", True), ("mx", True)])
def test_wgrad_matches_oracle(ops, T, N, K, path, pow2):
    """dW [N, K] = dY^T X from the 128x1 quantiser's outputs; N = 384 and 640
    leave a half-empty 256-wide tile."""
    dy = _grad(T + N, (T, N))
    x = _act(T + K, (T, K))
    qt_dy, st_dy = ops.quant_act_t(dy.cuda(), pow2)
    qt_x, st_x = ops.quant_act_t(x.cuda(), pow2)
    dw = ops.wgrad(qt_dy, st_dy, qt_x, st_x, pow2=pow2, path=path)
    _sync_ok(ops)
    qg_o, sg_o = O.quant_act_128x1(bf16_to_np(dy), pow2)
    qx_o, sx_o = O.quant_act_128x1(bf16_to_np(x), pow2)
    assert np.array_equal(qt_dy.cpu().numpy(), qg_o) and np.array_equal(qt_x.cpu().numpy(), qx_o)
    assert_gemm_close(bf16_to_np(dw), O.wgrad_ref(qg_o, sg_o, qx_o, sx_o), f"wgrad {path} {T}x{N}x{K}")


@pytest.mark.parametrize("path,pow2", [("promote", False), ("mx", True)])
def test_wgrad_ragged_rows_random_codes(ops, path, pow2):
    """Random codes and per-row scales, M = 200 output rows (a ragged tile),
    N = 384, K = 512: the kernel against the oracle's wgrad."""
    rng = np.random.Generator(np.random.PCG64(41))
    M, N, K = 200, 384, 512
    fin = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    qa = rng.choice(fin, (M, K)).astype(np.uint8)
    qb = rng.choice(fin, (N, K)).astype(np.uint8)
    if pow2:
        sa = np.exp2(rng.integers(-20, 5, (M, K // 128))).astype(np.float32)
        sb = np.exp2(rng.integers(-20, 5, (N, K // 128))).astype(np.float32)
    else:
        sa = rng.uniform(1e-6, 1e-3, (M, K // 128)).astype(np.float32)
        sb = rng.uniform(1e-6, 1e-3, (N, K // 128)).astype(np.float32)
    sa_dev = torch.zeros((K // 128, 200), dtype=torch.float32)
    sa_dev[:, :M] = torch.from_numpy(np.ascontiguousarray(sa.T))
    sb_dev = torch.from_numpy(np.ascontiguousarray(sb.T))
    c = ops.wgrad(torch.from_numpy(qa).cuda(), sa_dev.cuda(), torch.from_numpy(qb).cuda(), sb_dev.cuda(),
                  pow2=pow2, path=path)
    _sync_ok(ops)
    assert_gemm_close(bf16_to_np(c), O.wgrad_ref(qa, sa, qb, sb), f"wgrad ragged {path}")


@pytest.mark.parametrize("path", ["promote", "mx"])
def test_wgrad_exact_integer(ops, path):
    """Codes decoding to {-1, 0, 1}, K = 256 tokens, and power-of-two scales
    per (row, token block) chosen so that both token blocks of a row pair
    share one scale product: every output is an integer in [-256, 256] times a
    power of two, exact in bf16; the GPU must reproduce it exactly."""
    rng = np.random.Generator(np.random.PCG64(43))
    M, N, K = 256, 384, 256
    lut = np.array([0x00, 0x38, 0xB8], np.uint8)
    qa = lut[rng.integers(0, 3, (M, K))]
    qb = lut[rng.integers(0, 3, (N, K))]
    ea = rng.integers(-3, 3, (M, 1))
    eb = rng.integers(-3, 3, (N, 1))
    sa = np.repeat(np.exp2(ea), 2, axis=1).astype(np.float32)
    sb = np.repeat(np.exp2(eb), 2, axis=1).astype(np.float32)
    ref = O.wgrad_ref(qa, sa, qb, sb)
    ints = ref / np.exp2(ea + eb.T)
    assert np.array_equal(ints, np.round(ints)) and np.all(np.abs(ints) <= 256)
    c = ops.wgrad(torch.from_numpy(qa).cuda(), torch.from_numpy(np.ascontiguousarray(sa.T)).cuda(),
                  torch.from_numpy(qb).cuda(), torch.from_numpy(np.ascontiguousarray(sb.T)).cuda(),
                  pow2=True, path=path)
    _sync_ok(ops)
    assert np.array_equal(bf16_to_np(c), ref)


def test_wgrad_last_wave_split(ops):
    """A wgrad shape whose last wave of tiles is split along K (the token
    axis) when a workspace is given: same tolerance as the whole-tile run."""
    T, N, K = 4096, 1280, 4096     # 10 x 16 = 160 tiles of 128 x 256 on 152 SMs: 8 left over
    dy = _grad(51, (T, N))
    x = _act(52, (T, K))
    qt_dy, st_dy = ops.quant_act_t(dy.cuda())
    qt_x, st_x = ops.quant_act_t(x.cuda())
    dw = ops.wgrad(qt_dy, st_dy, qt_x, st_x)
    dw_whole = torch.empty_like(dw)
    ops.fp8_blockscaled_gemm_wgrad(qt_dy, st_dy, qt_x, st_x, dw_whole, ops.FP8_GEMM_PATH_PROMOTE, None)
    _sync_ok(ops)
    rows = np.sort(np.random.Generator(np.random.PCG64(53)).choice(N, 24, replace=False))
    qg_o, sg_o = O.quant_act_128x1(bf16_to_np(dy))
    qx_o, sx_o = O.quant_act_128x1(bf16_to_np(x))
    ref = O.wgrad_ref_rows(qg_o, sg_o, qx_o, sx_o, rows)
    assert_gemm_close(bf16_to_np(dw[rows]), ref, "wgrad split")
    assert_gemm_close(bf16_to_np(dw_whole[rows]), ref, "wgrad whole")


# ---------------------------------------------------------------- one whole layer
@pytest.mark.parametrize("pow2", [False, True])
def test_linear_layer_forward_and_backward(ops, pow2):
    """y = x W^T, dX = dY W, dW = dY^T X for one layer, with every operand
    produced by the dual-layout quantisers (one read of x, W and dY each)."""
    T, N, K = 512, 384, 640
    x = _act(61, (T, K))
    w = I.normal_bf16(I.stream(62, 3), (N, K), std=0.02)
    dy = _grad(63, (T, N))
    qt_x, st_x, q_x, s_x = ops.quant_act_t(x.cuda(), pow2, rowwise=True)
    qt_w, st_w, q_w, s_w = ops.quant_weight_t(w.cuda(), pow2, with_w=True)
    qt_dy, st_dy, q_dy, s_dy = ops.quant_act_t(dy.cuda(), pow2, rowwise=True)
    y = ops.gemm(q_x, s_x, q_w, s_w, pow2=pow2)
    dx = ops.gemm(q_dy, s_dy, qt_w, st_w, pow2=pow2)
    dw = ops.wgrad(qt_dy, st_dy, qt_x, st_x, pow2=pow2)
    _sync_ok(ops)
    xn, wn, gn = bf16_to_np(x), bf16_to_np(w), bf16_to_np(dy)
    qx_o, sx_o = O.quant_act_1x128(xn, pow2)
    qw_o, sw_o = O.quant_weight_128x128(wn, pow2)
    qg_o, sg_o = O.quant_act_1x128(gn, pow2)
    assert_gemm_close(bf16_to_np(y), O.gemm_ref(qx_o, sx_o, qw_o, sw_o), "forward")
    assert_gemm_close(bf16_to_np(dx), O.dgrad_ref(qg_o, sg_o, qw_o, sw_o), "dgrad")
    qtg_o, stg_o = O.quant_act_128x1(gn, pow2)
    qtx_o, stx_o = O.quant_act_128x1(xn, pow2)
    assert_gemm_close(bf16_to_np(dw), O.wgrad_ref(qtg_o, stg_o, qtx_o, stx_o), "wgrad")


@pytest.mark.parametrize("pow2", [False, True])
def test_llama_gate_up_backward_full_size_sampled(ops, pow2):
    """Llama-3.1-8B gate+up projection backward at full size (4096 tokens,
    4096 -> 28672): dgrad and wgrad on sampled output rows against the
    oracle; the 128x1 quantiser on sampled columns."""
    case = I.llama8b_layers(layers=["gate_up"])[0]
    T, K = case.a.shape
    N = case.w.shape[0]
    dy = _grad(71, (T, N))
    x_d, w_d, dy_d = case.a.cuda(), case.w.cuda(), dy.cuda()
    qt_x, st_x = ops.quant_act_t(x_d, pow2)
    qt_w, st_w = ops.quant_weight_t(w_d, pow2)
    qt_dy, st_dy, q_dy, s_dy = ops.quant_act_t(dy_d, pow2, rowwise=True)
    dx = ops.gemm(q_dy, s_dy, qt_w, st_w, pow2=pow2)
    dw = ops.wgrad(qt_dy, st_dy, qt_x, st_x, pow2=pow2)
    _sync_ok(ops)
    rng = np.random.Generator(np.random.PCG64(72))
    # dgrad: sampled tokens x a few 128-column blocks of W (each block column
    # of W is quantised on its own, so the oracle needs only those)
    rows = np.sort(rng.choice(T, 8, replace=False))
    qg_o, sg_o = O.quant_act_1x128(bf16_to_np(dy[rows]), pow2)
    cols, qw_o, sw_o = weight_block_cols(case.w, sample_block_rows(K, 4, 73), pow2)
    assert np.array_equal(qt_w[torch.from_numpy(cols)].cpu().numpy(), qw_o.T)
    assert_gemm_close(bf16_to_np(dx[rows])[:, cols], O.dgrad_ref(qg_o, sg_o, qw_o, sw_o), "dgrad full size")
    # wgrad rows (output features): their dY columns, all of X
    nrows = np.sort(rng.choice(N, 8, replace=False))
    qtg_o, stg_o = O.quant_act_128x1(bf16_to_np(dy[:, nrows]), pow2)
    qtx_o, stx_o = O.quant_act_128x1(bf16_to_np(case.a), pow2)
    assert np.array_equal(qt_dy[nrows].cpu().numpy(), qtg_o)
    assert np.array_equal(st_dy[:, nrows].cpu().numpy(), stg_o.T)
    assert np.array_equal(qt_x.cpu().numpy(), qtx_o)
    assert_gemm_close(bf16_to_np(dw[nrows]), O.wgrad_ref(qtg_o, stg_o, qtx_o, stx_o), "wgrad full size")


@pytest.mark.parametrize("pow2", [False, True])
def test_quant_act_128x1_ragged_tokens(ops, pow2):
    """300 tokens: the last 128x1 block holds 44 real rows and is padded with
    zeros inside the kernel (codes of the pad are zero)."""
    x = _edge_act(384, 256, seed=77)[:300].contiguous()
    qt, st, q, s = ops.quant_act_t(x.cuda(), pow2, rowwise=True)
    _sync_ok(ops)
    qt_o, st_o = O.quant_act_128x1(bf16_to_np(x), pow2)
    assert qt.shape == (256, 384) and np.array_equal(qt.cpu().numpy(), qt_o)
    assert np.array_equal(st[:, :256].cpu().numpy(), st_o.T)
    q_o, s_o = O.quant_act_1x128(bf16_to_np(x), pow2)
    assert np.array_equal(q.cpu().numpy(), q_o) and np.array_equal(s[:, :300].cpu().numpy(), s_o.T)


@pytest.mark.parametrize("pow2", [False, True])
def test_moe_wgrad(ops, pow2):
    """MoE weight gradients over Zipf-routed, expert-sorted tokens with ragged
    and empty experts (each expert's token blocks padded with zeros)."""
    offs = [0, 5, 5, 140, 140, 300, 301, 557]
    N, K = 256, 384
    T = offs[-1]
    x = _act(81, (T, K))
    dy = _grad(82, (T, N))
    dw = ops.moe_wgrad(dy.cuda(), x.cuda(), offs, pow2)
    _sync_ok(ops)
    ref = O.moe_wgrad_ref(bf16_to_np(dy), bf16_to_np(x), offs, pow2)
    got = bf16_to_np(dw)
    for g in range(len(offs) - 1):
        if offs[g + 1] == offs[g]:
            assert np.all(got[g] == 0)
        else:
            assert_gemm_close(got[g], ref[g], f"moe wgrad expert {g}")


@pytest.mark.parametrize("pow2", [False, True])
def test_quant_act_128x1_grouped_layout(ops, pow2):
    """The grouped 128x1 quantiser: expert g's tokens go to padded slots
    128 P_g .. 128 P_{g+1} - 1 (P_g = blocks of the experts before it), each
    expert's last block padded with zero codes; codes and scales bit-exact
    with the oracle's per-expert quantisation.  Experts: empty, 5 tokens,
    exactly 128, 256, 39, 1 and 256 tokens; the edge-case columns (an all-zero
    block, a subnormal amax, a tiny block, a huge value) are planted."""
    offs = [0, 0, 5, 133, 389, 389, 428, 429, 685]
    T, K = offs[-1], 384
    x = _edge_act(768, K, seed=91)[:T].contiguous()
    qt, st = ops.quant_act_t_grouped(x.cuda(), torch.tensor(offs, dtype=torch.int32, device="cuda"), pow2)
    _sync_ok(ops)
    qt, st = qt.cpu().numpy(), st.cpu().numpy()
    xn = bf16_to_np(x)
    P = 0
    for g in range(len(offs) - 1):
        lo, hi = offs[g], offs[g + 1]
        nb = (hi - lo + 127) // 128
        if nb:
            q_o, s_o = O.quant_act_128x1(xn[lo:hi], pow2)
            assert np.array_equal(qt[:, 128 * P:128 * (P + nb)], q_o), f"codes of expert {g}"
            assert np.array_equal(st[P:P + nb, :K], s_o.T), f"scales of expert {g}"
        P += nb


def test_moe_wgrad_one_expert_matches_dense_wgrad(ops):
    """With a single expert holding every token the grouped path is the dense
    weight gradient: the same codes, scales and (to the bit) the same dW."""
    T, N, K = 300, 256, 384
    x = _act(93, (T, K)).cuda()
    dy = _grad(94, (T, N)).cuda()
    dw = ops.moe_wgrad(dy, x, [0, T])
    qt_dy, st_dy = ops.quant_act_t(dy)
    qt_x, st_x = ops.quant_act_t(x)
    ref = ops.wgrad(qt_dy, st_dy, qt_x, st_x)
    _sync_ok(ops)
    assert torch.equal(dw[0].view(torch.int16), ref.view(torch.int16))


def test_moe_wgrad_no_tokens(ops):
    """T = 0: nothing to quantise, every expert's gradient is zero."""
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    dy = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    dw = ops.moe_wgrad(dy, x, [0, 0, 0, 0])
    _sync_ok(ops)
    assert dw.shape == (3, 128, 256) and not torch.any(dw.float() != 0)

