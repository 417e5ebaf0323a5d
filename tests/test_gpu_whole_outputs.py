"""Whole-output parity at the workloads' full sizes.

Every FP8 code, every scale and every output element the GPU writes is
compared with the oracle on the same seeded inputs -- not a sample of rows or
blocks: the tile schedules, the last-wave K split of the large-M kernels, the
stream-K division of the decode kernel and the grouped kernel's tile table
all write parts of these outputs, and a fault confined to some tiles would
show up here.

Workloads (seeded synthetic inputs of the shapes and value distributions of
the layers the pages measure on):
  * Llama-3.1-8B linear layers, M = 4096: qkv, gate+up, down, both scale
    modes (codes, scales, whole C);
  * Qwen3-8B prefill, M = 16384: codes and scales of all three layers, whole
    C of o_proj, both modes;
  * decode, M in {1, 8, 64, 256} at both shapes: whole weight codes and C;
  * Qwen3-30B-A3B experts (Zipf routing): codes, scales and whole C of both
    grouped GEMMs, both modes; the gate+up experts' weight gradients (grouped
    128x1 quantisers and the grouped wgrad GEMM), both modes;
  * Llama gate+up backward: the dual-layout quantisers' codes and scales,
    whole dX (dgrad on W^T codes) and whole dW (wgrad on 128x1 operands),
    both modes.

Codes and scales must be bit-exact; GEMM outputs meet the GEMM tolerance of
tests/helpers.py on every element.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.fp8_oracle as O
from fp8_block_scaled_05_gb300 import inputs as I
from tests import oracle_par as par
from tests.helpers import assert_gemm_close_whole, bf16_to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_05_gb300 import build, ops as _ops
    build.build()
    par.pool()
    yield _ops
    par.shutdown()


def _sync_ok(ops):
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0


def _same_act(q, s, q_o, s_o, what):
    """Device 1x128 codes [M, K] and K-block-major scales [K/128, lds] equal the
    oracle's ([M, K], [M, K/128])."""
    M = q_o.shape[0]
    assert np.array_equal(q.cpu().numpy(), q_o), f"{what}: activation codes"
    assert np.array_equal(s[:, :M].cpu().numpy(), s_o.T), f"{what}: activation scales"


def _same_weight(q, s, q_o, s_o, what):
    assert np.array_equal(q.cpu().numpy(), q_o), f"{what}: weight codes"
    assert np.array_equal(s.cpu().numpy(), s_o), f"{what}: weight scales"


# ------------------------------------------------------------ Llama-3.1-8B, M = 4096
@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("layer", ["qkv", "gate_up", "down"])
def test_llama_whole_layer(ops, layer, pow2):
    case = I.llama8b_layers(layers=[layer])[0]
    y, (qa, sa), (qw, sw) = ops.linear(case.a.cuda(), case.w.cuda(), pow2=pow2)
    _sync_ok(ops)
    qa_o, sa_o = par.quant_act_1x128(bf16_to_np(case.a), pow2)
    qw_o, sw_o = par.quant_weight_128x128(bf16_to_np(case.w), pow2)
    _same_act(qa, sa, qa_o, sa_o, f"llama {layer}")
    _same_weight(qw, sw, qw_o, sw_o, f"llama {layer}")
    del qa, sa, qw, sw
    assert_gemm_close_whole(y, par.gemm_ref(qa_o, sa_o, qw_o, sw_o), f"llama {layer} pow2={pow2}")


# ------------------------------------------------------------ Qwen3-8B prefill, M = 16384
@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("layer", ["gate_up", "down", "o_proj"])
def test_qwen_prefill_whole_codes(ops, layer, pow2):
    """Codes and scales of the whole prefill layer; for o_proj also the whole
    output (its GEMM, 550 GFLOP, is the one the oracle can afford)."""
    case = I.qwen_prefill_layers(layers=[layer])[0]
    a, w = case.a.cuda(), case.w.cuda()
    qa, sa = ops.quant_act(a, pow2)
    qw, sw = ops.quant_weight(w, pow2)
    y = ops.gemm(qa, sa, qw, sw, pow2=pow2) if layer == "o_proj" else None
    _sync_ok(ops)
    del a, w
    qa_o, sa_o = par.quant_act_1x128(bf16_to_np(case.a), pow2)
    qw_o, sw_o = par.quant_weight_128x128(bf16_to_np(case.w), pow2)
    _same_act(qa, sa, qa_o, sa_o, f"qwen {layer}")
    _same_weight(qw, sw, qw_o, sw_o, f"qwen {layer}")
    if y is not None:
        del qa, sa, qw, sw
        assert_gemm_close_whole(y, par.gemm_ref(qa_o, sa_o, qw_o, sw_o), f"qwen o_proj pow2={pow2}")


# ------------------------------------------------------------ decode-sized, M <= 256
_decode_w = {}


def _decode_weights(ops, K, N):
    """Whole weight of a decode shape, quantised on the device and by the
    oracle (once per shape), codes compared."""
    if (K, N) not in _decode_w:
        w = I.decode_case(1, K, N).w
        qw, sw = ops.quant_weight(w.cuda())
        _sync_ok(ops)
        qw_o, sw_o = par.quant_weight_128x128(bf16_to_np(w))
        _same_weight(qw, sw, qw_o, sw_o, f"decode weight K={K} N={N}")
        _decode_w[(K, N)] = (qw, sw, qw_o, sw_o)
    return _decode_w[(K, N)]


@pytest.mark.parametrize("K,N", [(14336, 4096), (4096, 6144)])
@pytest.mark.parametrize("M,path", [(1, "auto"), (8, "auto"), (64, "auto"), (256, "auto"), (256, "skinny")])
def test_decode_whole_output(ops, M, path, K, N):
    # automatic path: the skinny kernel up to 128 rows, the promote kernel with
    # every tile split along K at 256; the skinny kernel forced at 256 (two
    # 128-token chunks per weight tile)
    qw, sw, qw_o, sw_o = _decode_weights(ops, K, N)
    a = I.decode_case(M, K, N).a
    qa, sa = ops.quant_act(a.cuda())
    y = ops.gemm(qa, sa, qw, sw, path=path)
    _sync_ok(ops)
    qa_o, sa_o = O.quant_act_1x128(bf16_to_np(a))
    _same_act(qa, sa, qa_o, sa_o, f"decode M={M}")
    assert_gemm_close_whole(y, O.gemm_ref(qa_o, sa_o, qw_o, sw_o), f"decode M={M} K={K} N={N} path={path}")


# ------------------------------------------------------------ Qwen3-30B-A3B experts
_moe = {}


def _moe_case():
    if "case" not in _moe:
        _moe["case"] = I.moe_case()
    return _moe["case"]


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("proj", ["gate_up", "down"])
def test_moe_whole_grouped_output(ops, proj, pow2):
    m = _moe_case()
    a, w = (m.a_gate_up, m.w_gate_up) if proj == "gate_up" else (m.a_down, m.w_down)
    G, N, K = w.shape
    mode = ops.FP8_SCALE_POW2 if pow2 else ops.FP8_SCALE_FP32_AMAX
    qa, sa = ops.quant_act(a.cuda(), pow2)
    qw = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device="cuda")
    # all experts in one launch: a 128x128 tile never straddles two experts
    ops.fp8_quant_weight_128x128(w.cuda().view(G * N, K), qw.view(G * N, K), sw.view(G * N // 128, K // 128), mode)
    c = ops.grouped_gemm(qa, sa, torch.from_numpy(m.offsets).cuda(), qw, sw, pow2)
    _sync_ok(ops)
    qa_o, sa_o = par.quant_act_1x128(bf16_to_np(a), pow2)
    qw_o, sw_o = par.quant_weight_128x128(bf16_to_np(w).reshape(G * N, K), pow2)
    _same_act(qa, sa, qa_o, sa_o, f"moe {proj}")
    _same_weight(qw.view(G * N, K), sw.view(G * N // 128, K // 128), qw_o, sw_o, f"moe {proj}")
    del qa, sa, qw, sw
    ref = O.grouped_gemm_ref(qa_o, sa_o, m.offsets, qw_o.reshape(G, N, K), sw_o.reshape(G, N // 128, K // 128))
    assert_gemm_close_whole(c, ref, f"moe {proj} pow2={pow2}")


@pytest.mark.parametrize("pow2", [False, True])
def test_moe_wgrad_whole(ops, pow2):
    """Weight gradients of the gate+up experts, dW_g = dY_g^T X_g over the
    Zipf-routed expert-sorted rows (65536 rows, 128 experts): both grouped
    128x1 quantisers and the grouped wgrad GEMM, every code, scale and dW
    element of every expert against the oracle's per-expert quantisation and
    wgrad (dY ~ Student-t, nu = 4, x 1e-4)."""
    m = _moe_case()
    x = m.a_gate_up
    T, K = x.shape
    N = m.w_gate_up.shape[1]
    G = len(m.offsets) - 1
    dy = (I.student_t_bf16(I.stream(7, 85), (T, N), nu=4.0).float() * 1e-4).to(torch.bfloat16)
    offs = torch.from_numpy(m.offsets.astype(np.int32)).cuda()
    qt_dy, st_dy = ops.quant_act_t_grouped(dy.cuda(), offs, pow2)
    qt_x, st_x = ops.quant_act_t_grouped(x.cuda(), offs, pow2)
    dw = torch.empty((G, N, K), dtype=torch.bfloat16, device="cuda")
    ops.fp8_blockscaled_grouped_gemm_wgrad(qt_dy, st_dy, qt_x, st_x, offs, T, dw,
                                           ops.FP8_GEMM_SCALES_POW2 if pow2 else 0)
    _sync_ok(ops)
    live = set()
    blocks = np.cumsum([0] + [(int(m.offsets[g + 1]) - int(m.offsets[g]) + 127) // 128 for g in range(G)])
    for g, qg, sg, qx, sx, ref in par.moe_wgrad_experts(bf16_to_np(dy), bf16_to_np(x), m.offsets, pow2):
        live.add(g)
        b0, b1 = int(blocks[g]), int(blocks[g + 1])
        assert torch.equal(qt_dy[:, 128 * b0:128 * b1].cpu(), torch.from_numpy(qg)), f"dY codes, expert {g}"
        assert torch.equal(qt_x[:, 128 * b0:128 * b1].cpu(), torch.from_numpy(qx)), f"X codes, expert {g}"
        assert np.array_equal(st_dy[b0:b1, :N].cpu().numpy(), sg.T), f"dY scales, expert {g}"
        assert np.array_equal(st_x[b0:b1, :K].cpu().numpy(), sx.T), f"X scales, expert {g}"
        assert_gemm_close_whole(dw[g], ref, f"moe wgrad expert {g} pow2={pow2}")
    for g in set(range(G)) - live:
        assert not torch.any(dw[g].float() != 0), f"expert {g} has no tokens"


# ------------------------------------------------------------ Llama gate+up backward
@pytest.mark.parametrize("pow2", [False, True])
def test_llama_gate_up_backward_whole(ops, pow2):
    """Gradients dY [4096, 28672] ~ Student-t (nu = 4) x 1e-4: the 1x128 and
    128x1 codes of dY and X, W^T's codes, whole dX = dY W and whole
    dW = dY^T X against the oracle."""
    case = I.llama8b_layers(layers=["gate_up"])[0]
    T, K = case.a.shape
    N = case.w.shape[0]
    dy = (I.student_t_bf16(I.stream(71, 7), (T, N), nu=4.0).float() * 1e-4).to(torch.bfloat16)
    qt_x, st_x = ops.quant_act_t(case.a.cuda(), pow2)
    qt_w, st_w = ops.quant_weight_t(case.w.cuda(), pow2)
    qt_dy, st_dy, q_dy, s_dy = ops.quant_act_t(dy.cuda(), pow2, rowwise=True)
    dx = ops.gemm(q_dy, s_dy, qt_w, st_w, pow2=pow2)
    dw = ops.wgrad(qt_dy, st_dy, qt_x, st_x, pow2=pow2)
    _sync_ok(ops)
    xn, wn, gn = bf16_to_np(case.a), bf16_to_np(case.w), bf16_to_np(dy)
    # dgrad operands and output
    qg_o, sg_o = par.quant_act_1x128(gn, pow2)
    qw_o, sw_o = par.quant_weight_128x128(wn, pow2)
    _same_act(q_dy, s_dy, qg_o, sg_o, "dY 1x128")
    assert np.array_equal(qt_w.cpu().numpy(), qw_o.T), "W^T codes"
    assert np.array_equal(st_w.cpu().numpy(), sw_o.T), "W^T scales"
    assert_gemm_close_whole(dx, O.dgrad_ref(qg_o, sg_o, qw_o, sw_o), f"dgrad pow2={pow2}")
    del qg_o, sg_o, qw_o, sw_o, dx
    # wgrad operands and output
    qtg_o, stg_o = par.quant_act_128x1(gn, pow2)
    qtx_o, stx_o = par.quant_act_128x1(xn, pow2)
    assert np.array_equal(qt_dy.cpu().numpy(), qtg_o), "dY 128x1 codes"
    assert np.array_equal(st_dy[:, :N].cpu().numpy(), stg_o.T), "dY 128x1 scales"
    assert np.array_equal(qt_x.cpu().numpy(), qtx_o), "X 128x1 codes"
    assert np.array_equal(st_x[:, :K].cpu().numpy(), stx_o.T), "X 128x1 scales"
    ref = np.empty((N, K), np.float64)
    for n0 in range(0, N, 4096):   # output rows in blocks (the oracle's wgrad on those dY columns)
        ref[n0:n0 + 4096] = O.wgrad_ref(qtg_o[n0:n0 + 4096], stg_o[n0:n0 + 4096], qtx_o, stx_o)
    assert_gemm_close_whole(dw, ref, f"wgrad pow2={pow2}")
