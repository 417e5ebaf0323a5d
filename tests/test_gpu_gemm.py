"""GPU parity of the block-scaled GEMMs (large-M promote kernel, skinny
split-K kernel, grouped MoE kernel) with the oracle's fp64
dequantise-then-multiply reference; operands come from the oracle's own
quantisers on the same seeded inputs, so the GEMM is checked on its own."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.fp8_oracle as O
from fp8_block_scaled_05_gb300 import inputs as I
from tests.helpers import assert_gemm_close, bf16_to_np, sample_block_rows, weight_block_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from fp8_block_scaled_05_gb300 import build, ops as _ops
    build.build()
    return _ops


def _to_dev(qa, sa_mk, qw, sw):
    """Oracle operands -> device tensors in the library's layouts."""
    M = qa.shape[0]
    lds = max(4, (M + 3) // 4 * 4)
    sa_dev = torch.zeros((sa_mk.shape[1], lds), dtype=torch.float32)
    sa_dev[:, :M] = torch.from_numpy(np.ascontiguousarray(sa_mk.T))
    return (torch.from_numpy(qa).cuda(), sa_dev.cuda(), torch.from_numpy(qw).cuda(),
            torch.from_numpy(np.ascontiguousarray(sw)).cuda())


def _case(M, N, K, seed, pow2=False, outliers=True):
    a = I.normal_bf16(I.stream(seed, 1), (M, K))
    if outliers and K >= 256:
        a, _ = I.with_outlier_columns(a, I.stream(seed, 2), max(1, K // 100), 30.0)
    w = I.normal_bf16(I.stream(seed, 3), (N, K), std=0.02)
    qa, sa = O.quant_act_1x128(bf16_to_np(a), pow2)
    qw, sw = O.quant_weight_128x128(bf16_to_np(w), pow2)
    return qa, sa, qw, sw


def _run(ops, qa, sa, qw, sw, path, pow2=False):
    dqa, dsa, dqw, dsw = _to_dev(qa, sa, qw, sw)
    c = ops.gemm(dqa, dsa, dqw, dsw, pow2=pow2, path=path)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    return bf16_to_np(c)


@pytest.mark.parametrize("path,pow2", [("promote", False), ("promote", True), ("skinny", False),
                                       ("skinny", True), ("mx", True)])
def test_tiny(ops, path, pow2):
    case = I.tiny()
    qa, sa = O.quant_act_1x128(bf16_to_np(case.a), pow2)
    qw, sw = O.quant_weight_128x128(bf16_to_np(case.w), pow2)
    c = _run(ops, qa, sa, qw, sw, path, pow2)
    assert_gemm_close(c, O.gemm_ref(qa, sa, qw, sw), f"tiny/{path}/{pow2}")


@pytest.mark.parametrize("M,N,K", [(300, 640, 1152), (128, 256, 128), (129, 128, 256), (513, 384, 512),
                                   (1000, 1280, 384)])
def test_promote_ragged(ops, M, N, K):
    qa, sa, qw, sw = _case(M, N, K, seed=M + N)
    c = _run(ops, qa, sa, qw, sw, "promote")
    assert_gemm_close(c, O.gemm_ref(qa, sa, qw, sw), f"promote {M}x{N}x{K}")


@pytest.mark.parametrize("path,M", [("promote", 1200), ("promote", 1280), ("mx", 1500), ("mx", 1536)])
def test_last_wave_split(ops, M, path):
    """Output tiles that do not fill whole waves of 152 SMs: promote, 10 x 16 =
    160 tiles, the 8 of the last wave split along K into 2 parts (16 K-blocks,
    at least 8 per part); MX, 12 x 16 = 192 tiles, the 40 of the last wave (at
    least a quarter of the SMs) split into 2.  The fp32 parts are added in
    part order.  Checked against the oracle, bit-identical on a second call
    (fixed order), and within tolerance without a workspace (no split)."""
    N, K = 4096, 2048
    pow2 = path == "mx"
    qa, sa, qw, sw = _case(M, N, K, seed=M, pow2=pow2)
    ref = O.gemm_ref(qa, sa, qw, sw)
    dqa, dsa, dqw, dsw = _to_dev(qa, sa, qw, sw)
    assert ops.fp8_gemm_workspace_size(M, N, K, 1) > 0
    c1 = ops.gemm(dqa, dsa, dqw, dsw, pow2=pow2, path=path)
    c2 = ops.gemm(dqa, dsa, dqw, dsw, pow2=pow2, path=path)
    c0 = torch.empty_like(c1)
    flags = ops.PATHS[path] | (ops.FP8_GEMM_SCALES_POW2 if pow2 else 0)
    ops.fp8_blockscaled_gemm(dqa, dsa, dqw, dsw, c0, flags, None)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    assert torch.equal(c1, c2)
    assert_gemm_close(bf16_to_np(c1), ref, f"{path} split M={M}")
    assert_gemm_close(bf16_to_np(c0), ref, f"{path} unsplit M={M}")


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("M", [127, 128, 129, 130])
def test_auto_path_at_the_row_threshold(ops, M, pow2):
    """The automatic path takes the skinny kernel up to 128 rows and the
    large-M kernels (every tile split along K here: 2 x 8 tiles on 152 SMs)
    from 129: on both sides of the threshold the plan names the expected
    kernel and the whole output is within tolerance of the oracle."""
    N, K = 1024, 4096
    flags = ops.FP8_GEMM_SCALES_POW2 if pow2 else 0
    path, _ = ops.fp8_gemm_plan(M, N, K, flags)
    want = ops.FP8_GEMM_PATH_SKINNY if M <= 128 else (ops.FP8_GEMM_PATH_MX if pow2 else ops.FP8_GEMM_PATH_PROMOTE)
    assert path == want
    qa, sa, qw, sw = _case(M, N, K, seed=3 * M + pow2, pow2=pow2)
    c = _run(ops, qa, sa, qw, sw, "auto", pow2)
    assert_gemm_close(c, O.gemm_ref(qa, sa, qw, sw), f"auto path M={M} pow2={pow2}")


@pytest.mark.parametrize("path,M,N,K", [("promote", 300, 1024, 4096), ("mx", 300, 1024, 4096),
                                        ("promote", 64, 2048, 8192), ("mx", 200, 1536, 4096),
                                        ("promote", 1, 768, 2048), ("mx", 8, 4096, 14336)])
def test_single_wave_split(ops, path, M, N, K):
    """Fewer output tiles than SMs: every tile is split along K, one part per
    CTA (on 152 SMs: 12 tiles x 4 parts, 8 x 8, 12 x 4, 3 x 2 and 16 x 9,
    the parts at least 8 K-blocks long).  Checked against the oracle,
    bit-identical on a second call (parts added in part order), within
    tolerance without a workspace (no split), and the tickets are left at
    zero."""
    pow2 = path == "mx"
    qa, sa, qw, sw = _case(M, N, K, seed=M + 7 * N, pow2=pow2)
    ref = O.gemm_ref(qa, sa, qw, sw)
    dqa, dsa, dqw, dsw = _to_dev(qa, sa, qw, sw)
    flags = ops.PATHS[path] | (ops.FP8_GEMM_SCALES_POW2 if pow2 else 0)
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    outs = []
    for w in (ws, ws, None):
        c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        ops.fp8_blockscaled_gemm(dqa, dsa, dqw, dsw, c, flags, w)
        torch.cuda.synchronize()
        assert ops.fp8_last_device_status() == 0
        outs.append(c)
    assert torch.equal(outs[0], outs[1])
    assert_gemm_close(bf16_to_np(outs[0]), ref, f"{path} single-wave split {M}x{N}x{K}")
    assert_gemm_close(bf16_to_np(outs[2]), ref, f"{path} unsplit {M}x{N}x{K}")
    assert int(ws[:65536].view(torch.int32).abs().sum()) == 0


def test_workspace_shared_across_shapes(ops):
    """One zero-initialised workspace reused, in sequence, by calls of several
    shapes and paths whose tickets and partials differ in size (split-K decode,
    last-wave splits of both large-M kernels): each call's partials must never
    land on the tickets a later call relies on.  Every result is checked
    against the oracle."""
    seq = [("promote", 1280, 4096, 2048), ("promote", 1536, 4096, 2048), ("skinny", 8, 640, 2048),
           ("mx", 1536, 4096, 2048), ("skinny", 64, 4096, 4096), ("promote", 1280, 4096, 2048),
           ("skinny", 8, 640, 2048), ("mx", 1536, 4096, 2048)]
    cache = {}
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    for path, M, N, K in seq:
        pow2 = path == "mx"
        key = (M, N, K, pow2)
        if key not in cache:
            qa, sa, qw, sw = _case(M, N, K, seed=M + N, pow2=pow2)
            cache[key] = (_to_dev(qa, sa, qw, sw), O.gemm_ref(qa, sa, qw, sw))
        (dqa, dsa, dqw, dsw), ref = cache[key]
        assert ops.fp8_gemm_workspace_size(M, N, K, 1) <= ws.numel()
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ops.fp8_blockscaled_gemm(dqa, dsa, dqw, dsw, c, ops.PATHS[path] | (ops.FP8_GEMM_SCALES_POW2 if pow2 else 0), ws)
        torch.cuda.synchronize()
        assert ops.fp8_last_device_status() == 0
        assert_gemm_close(bf16_to_np(c), ref, f"shared workspace {path} {M}x{N}x{K}")
    assert int(ws[:65536].view(torch.int32).abs().sum()) == 0   # tickets left at zero


@pytest.mark.parametrize("M,N,K", [(200, 384, 512), (300, 1024, 1152), (129, 256, 128), (1, 512, 256),
                                   (1280, 4096, 2048), (1536, 4096, 2048), (200, 1024, 4096)])
@pytest.mark.parametrize("pow2,out_pow2", [(False, False), (True, True), (False, True), (True, False)])
def test_gemm_quant_fused(ops, M, N, K, pow2, out_pow2):
    """GEMM with the next layer's 1x128 quantisation fused into the epilogue:
    the codes and scales must be exactly those of fp8_quant_act_1x128 (and of
    the oracle's quantiser) applied to the bf16 C the same call writes; C is
    within tolerance of the oracle; without C the codes and scales are the
    same.  Covers a half-empty last tile (N = 384), ragged M, K = 128, M = 1
    and the last-wave K split (M = 1280 and 1536, N = 4096: the promote
    kernel splits the 8 and 40 left-over tiles, the MX kernel the 40, the
    codes coming from the summed parts), and fewer tiles than SMs (M = 200,
    N = 1024, K = 4096: every tile split along K).  Power-of-two input scales take the
    MX kernel, the others the promote kernel."""
    qa, sa, qw, sw = _case(M, N, K, seed=M + K, pow2=pow2)
    ref = O.gemm_ref(qa, sa, qw, sw)
    dqa, dsa, dqw, dsw = _to_dev(qa, sa, qw, sw)
    c, qc, sc = ops.gemm_quant(dqa, dsa, dqw, dsw, pow2=pow2, out_pow2=out_pow2)
    _, qc2, sc2 = ops.gemm_quant(dqa, dsa, dqw, dsw, pow2=pow2, out_pow2=out_pow2, with_c=False)
    qa_gpu, sa_gpu = ops.quant_act(c, out_pow2)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    assert_gemm_close(bf16_to_np(c), ref, f"gemm_quant C {M}x{N}x{K}")
    assert torch.equal(qc, qa_gpu) and torch.equal(sc[:, :M], sa_gpu[:, :M])
    assert torch.equal(qc, qc2) and torch.equal(sc[:, :M], sc2[:, :M])
    q_o, s_o = O.quant_act_1x128(bf16_to_np(c), out_pow2)
    assert np.array_equal(qc.cpu().numpy(), q_o)
    assert np.array_equal(sc[:, :M].cpu().numpy(), s_o.T)


@pytest.mark.parametrize("path,out_pow2", [("promote", False), ("promote", True), ("mx", False), ("mx", True)])
def test_gemm_quant_fused_exact_output(ops, path, out_pow2):
    """Operands whose product is exact in bf16 (codes decoding to {-1, 0, 1},
    power-of-two scales shared by both K-blocks): C equals the oracle's C, so
    the fused codes and scales must equal the oracle quantiser applied to the
    oracle's C -- no value of the device path enters the expected result."""
    rng = np.random.Generator(np.random.PCG64(33))
    M, N, K = 300, 512, 256
    lut = np.array([0x00, 0x38, 0xB8], np.uint8)
    qa = lut[rng.integers(0, 3, (M, K))]
    qw = lut[rng.integers(0, 3, (N, K))]
    sa = np.repeat(2.0 ** rng.integers(-3, 3, (M, 1)), K // 128, axis=1).astype(np.float32)
    sw = np.repeat(2.0 ** rng.integers(-2, 2, (N // 128, 1)), K // 128, axis=1).astype(np.float32)
    ref = O.gemm_ref(qa, sa, qw, sw)
    dqa, dsa, dqw, dsw = _to_dev(qa, sa, qw, sw)
    c, qc, sc = ops.gemm_quant(dqa, dsa, dqw, dsw, pow2=True, out_pow2=out_pow2) if path == "mx" else \
        _gemm_quant_path(ops, dqa, dsa, dqw, dsw, ops.FP8_GEMM_PATH_PROMOTE | ops.FP8_GEMM_SCALES_POW2, out_pow2)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    assert np.array_equal(bf16_to_np(c), ref)
    q_o, s_o = O.quant_act_1x128(ref.astype(np.float32), out_pow2)
    assert np.array_equal(qc.cpu().numpy(), q_o)
    assert np.array_equal(sc[:, :M].cpu().numpy(), s_o.T)


@pytest.mark.parametrize("path", ["promote", "mx"])
def test_gemm_quant_fused_rows_whose_factor_overflows(ops, path):
    """The fused cast's rare path: rows whose bf16 outputs are so small that
    448/amax overflows fp32 are cast by division (x / s), and a warp holding
    one takes the per-pair choice for all its rows.  Exact operands as above;
    rows 0-31 (a whole lane quarter) and every 37th row get sA = 2^-124 with
    sB = 2^-2, so C there is an integer times 2^-126 (normal, exact in bf16)
    and amax stays below 448 / FLT_MAX; the other rows keep ordinary scales.
    Codes and scales must equal the oracle's quantiser on the oracle's C."""
    rng = np.random.Generator(np.random.PCG64(35))
    M, N, K = 300, 512, 256
    lut = np.array([0x00, 0x38, 0xB8], np.uint8)
    qa = lut[rng.integers(0, 3, (M, K))]
    qw = lut[rng.integers(0, 3, (N, K))]
    ea = rng.integers(-3, 3, (M, 1)).astype(np.float64)
    tiny = np.zeros(M, bool)
    tiny[:32] = True
    tiny[::37] = True
    ea[tiny] = -124
    sa = np.repeat(2.0 ** ea, K // 128, axis=1).astype(np.float32)
    sw = np.full((N // 128, K // 128), 0.25, np.float32)
    ref = O.gemm_ref(qa, sa, qw, sw)
    amax_tiny = np.abs(ref[tiny]).max()
    assert 0 < amax_tiny < 448.0 / np.finfo(np.float32).max   # the division path is reached
    dqa, dsa, dqw, dsw = _to_dev(qa, sa, qw, sw)
    flags = (ops.FP8_GEMM_PATH_MX if path == "mx" else ops.FP8_GEMM_PATH_PROMOTE) | ops.FP8_GEMM_SCALES_POW2
    c, qc, sc = _gemm_quant_path(ops, dqa, dsa, dqw, dsw, flags, False)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    assert np.array_equal(bf16_to_np(c), ref)
    q_o, s_o = O.quant_act_1x128(ref.astype(np.float32), False)
    assert np.array_equal(qc.cpu().numpy(), q_o)
    assert np.array_equal(sc[:, :M].cpu().numpy(), s_o.T)


def _gemm_quant_path(ops, qa, sa, qw, sw, flags, out_pow2):
    M, N = qa.shape[0], qw.shape[0]
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    qc = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    sc = torch.empty((N // 128, ops.round_up(M, 4)), dtype=torch.float32, device="cuda")
    ops.fp8_blockscaled_gemm_quant(qa, sa, qw, sw, c, qc, sc, flags,
                                   ops.FP8_SCALE_POW2 if out_pow2 else ops.FP8_SCALE_FP32_AMAX,
                                   ops.workspace_for(M, N, qa.shape[1], 1, qa.device))
    return c, qc, sc


@pytest.mark.parametrize("pow2", [False, True])
def test_gemm_quant_fused_llama_gate_up_sampled_rows(ops, pow2):
    """Full-size Llama-3.1-8B gate+up GEMM with its output quantised in the
    epilogue (promote kernel with fp32 scales, MX kernel with power-of-two
    scales): sampled rows' C against the oracle, codes and scales against the
    oracle's quantiser of the same bf16 rows."""
    case = I.llama8b_layers(layers=["gate_up"])[0]
    qa, sa = ops.quant_act(case.a.cuda(), pow2)
    qw, sw = ops.quant_weight(case.w.cuda(), pow2)
    c, qc, sc = ops.gemm_quant(qa, sa, qw, sw, pow2=pow2, out_pow2=pow2)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    rows = np.sort(np.random.Generator(np.random.PCG64(23)).choice(case.a.shape[0], 16, replace=False))
    qa_o, sa_o = O.quant_act_1x128(bf16_to_np(case.a[rows]), pow2)
    wrows, qw_o, sw_o = weight_block_rows(case.w, sample_block_rows(case.w.shape[0], 6, 24), pow2)
    ref = O.gemm_ref(qa_o, sa_o, qw_o, sw_o)
    c_rows = bf16_to_np(c[rows])
    assert_gemm_close(c_rows[:, wrows], ref, "gemm_quant llama gate_up")
    q_o, s_o = O.quant_act_1x128(c_rows, pow2)
    assert np.array_equal(qc[rows].cpu().numpy(), q_o)
    assert np.array_equal(sc[:, rows].cpu().numpy(), s_o.T)


@pytest.mark.parametrize("M", [1, 2, 8, 16, 17, 33, 64, 100, 128, 200, 256])
def test_skinny_ragged(ops, M):
    N, K = 640, 2048
    qa, sa, qw, sw = _case(M, N, K, seed=M)
    c = _run(ops, qa, sa, qw, sw, "skinny")
    assert_gemm_close(c, O.gemm_ref(qa, sa, qw, sw), f"skinny M={M}")


@pytest.mark.parametrize("path", ["promote", "skinny", "mx"])
def test_exact_integer_gemm(ops, path):
    """Codes decoding to {-1, 0, 1}, K = 256, and a power-of-two scale that is
    the same for both K-blocks of a row (and of a weight tile row): every
    output is an integer in [-256, 256] (at most 8 significant bits) times a
    power of two, exact in bf16; the GPU must reproduce it exactly."""
    rng = np.random.Generator(np.random.PCG64(31))
    M, N, K = 200, 384, 256
    lut = np.array([0x00, 0x38, 0xB8], np.uint8)
    qa = lut[rng.integers(0, 3, (M, K))]
    qw = lut[rng.integers(0, 3, (N, K))]
    sa = np.repeat(2.0 ** rng.integers(-3, 3, (M, 1)), K // 128, axis=1).astype(np.float32)
    sw = np.repeat(2.0 ** rng.integers(-2, 2, (N // 128, 1)), K // 128, axis=1).astype(np.float32)
    ref = O.gemm_ref(qa, sa, qw, sw)
    ints = ref / (sa[:, :1].astype(np.float64) * np.repeat(sw[:, 0], 128)[None, :])
    assert np.array_equal(ints, np.round(ints)) and np.all(np.abs(ints) <= 256)
    c = _run(ops, qa, sa, qw, sw, path, pow2=path == "mx")
    assert np.array_equal(c, ref)


# ------------------------------------------------------------ MX (pow2 scales)
@pytest.mark.parametrize("M,N,K", [(300, 640, 1152), (128, 256, 128), (129, 128, 256), (513, 384, 512),
                                   (1000, 1280, 384), (257, 768, 640), (1, 256, 256), (64, 512, 2048)])
def test_mx_ragged(ops, M, N, K):
    """Ragged M, N = 128 mod 256 (half-empty last tile), K-block counts that
    are not multiples of the four scale bytes per TMEM word, M below 256."""
    qa, sa, qw, sw = _case(M, N, K, seed=M + N + 1, pow2=True)
    c = _run(ops, qa, sa, qw, sw, "mx", pow2=True)
    assert_gemm_close(c, O.gemm_ref(qa, sa, qw, sw), f"mx {M}x{N}x{K}")


def test_mx_matches_promote_on_pow2_scales(ops):
    """Both large-M kernels compute the same C from the same power-of-two
    operands; each is within tolerance of the oracle and of the other."""
    qa, sa, qw, sw = _case(384, 1024, 2048, seed=5, pow2=True)
    ref = O.gemm_ref(qa, sa, qw, sw)
    c_mx = _run(ops, qa, sa, qw, sw, "mx", pow2=True)
    c_pr = _run(ops, qa, sa, qw, sw, "promote", pow2=True)
    assert_gemm_close(c_mx, ref, "mx")
    assert_gemm_close(c_pr, ref, "promote")
    assert_gemm_close(c_mx, c_pr.astype(np.float64), "mx vs promote")


def test_mx_extreme_scale_range(ops):
    """Rows whose magnitudes span 2^-60 .. 2^60 (activation scales from
    2^-69 to 2^52) against weights of 2^-20 .. 2^20 per 128-row block: the
    hardware's UE8M0 exponents must reach both ends.  Checked row by row so
    that small rows are not hidden behind large ones."""
    M, N, K = 256, 512, 512
    a = I.normal_bf16(I.stream(41, 1), (M, K)).float() * torch.exp2(torch.linspace(-60, 60, M).round())[:, None]
    w = I.normal_bf16(I.stream(41, 2), (N, K)).float() * torch.exp2(torch.tensor([-20.0, -7.0, 9.0, 20.0])
                                                                    ).repeat_interleave(128)[:, None]
    qa, sa = O.quant_act_1x128(bf16_to_np(a.to(torch.bfloat16)), True)
    qw, sw = O.quant_weight_128x128(bf16_to_np(w.to(torch.bfloat16)), True)
    ref = O.gemm_ref(qa, sa, qw, sw)
    c = _run(ops, qa, sa, qw, sw, "mx", pow2=True)
    for r in range(M):
        for nb in range(N // 128):
            cols = slice(128 * nb, 128 * nb + 128)
            assert_gemm_close(c[r, cols], ref[r, cols], f"mx row {r} block {nb}")


@pytest.mark.parametrize("where", ["sa", "sb"])
def test_mx_reports_a_scale_that_is_not_a_power_of_two(ops, where):
    qa, sa, qw, sw = _case(256, 256, 512, seed=3, pow2=True)
    dqa, dsa, dqw, dsw = _to_dev(qa, sa, qw, sw)
    (dsa if where == "sa" else dsw).view(-1)[1] *= 0.75
    ops.gemm(dqa, dsa, dqw, dsw, pow2=True, path="mx")
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 4   # FP8_ERR_SCALE_MODE
    assert ops.fp8_last_device_status() == 0   # reading clears it


def test_rejects_bad_arguments(ops):
    qa = torch.zeros((4, 2048), dtype=torch.uint8, device="cuda")
    sa = torch.ones((16, 4), dtype=torch.float32, device="cuda")
    qw = torch.zeros((128, 2048), dtype=torch.uint8, device="cuda")
    sw = torch.ones((1, 16), dtype=torch.float32, device="cuda")
    c = torch.empty((4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.FP8Error) as e:
        ops.fp8_blockscaled_gemm(qa[:, :200], sa, qw[:, :200], sw, c)
    assert e.value.status == 2
    with pytest.raises(ops.FP8Error) as e:
        ops.fp8_blockscaled_gemm(qa, sa, qw, sw, c, flags=ops.FP8_GEMM_PATH_SKINNY, workspace=None)
    assert e.value.status == 5


# ------------------------------------------------------------ full sizes
@pytest.mark.parametrize("layer,pow2", [("qkv", False), ("down", False), ("gate_up", True), ("down", True)])
def test_llama_full_size_sampled_rows(ops, layer, pow2):
    """Llama-3.1-8B layer shapes, whole path on the GPU (quantisers + GEMM;
    power-of-two scales take the MX kernel), checked on sampled output rows
    against the oracle."""
    case = I.llama8b_layers(layers=[layer])[0]
    y, (qa, sa), (qw, sw) = ops.linear(case.a.cuda(), case.w.cuda(), pow2=pow2)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    rows = np.sort(np.random.Generator(np.random.PCG64(8)).choice(case.a.shape[0], 24, replace=False))
    qa_o, sa_o = O.quant_act_1x128(bf16_to_np(case.a[rows]), pow2)
    assert np.array_equal(qa[rows].cpu().numpy(), qa_o)
    nbs = sample_block_rows(case.w.shape[0], 6, 9)
    wrows, qw_o, sw_o = weight_block_rows(case.w, nbs, pow2)
    assert np.array_equal(qw[torch.from_numpy(wrows)].cpu().numpy(), qw_o)
    assert np.array_equal(sw[torch.from_numpy(nbs)].cpu().numpy(), sw_o)
    ref = O.gemm_ref(qa_o, sa_o, qw_o, sw_o)
    assert_gemm_close(bf16_to_np(y[rows])[:, wrows], ref, f"llama {layer}")


@pytest.mark.parametrize("layer", ["gate_up", "down", "o_proj"])
@pytest.mark.parametrize("pow2", [False, True])
def test_qwen_prefill_full_size_sampled_rows(ops, layer, pow2):
    """Qwen3-8B-shaped prefill (M 16384, Student-t nu = 4 activations), both
    scale modes: fp32 scales take the promote kernel, power-of-two scales the
    MX kernel.  Whole path on the GPU, checked on sampled output rows."""
    case = I.qwen_prefill_layers(layers=[layer])[0]
    y, (qa, sa), (qw, sw) = ops.linear(case.a.cuda(), case.w.cuda(), pow2=pow2)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    M = case.a.shape[0]
    rows = np.unique(np.concatenate([np.random.Generator(np.random.PCG64(11)).choice(M, 24, replace=False),
                                     [0, 127, 128, M - 1]]))
    qa_o, sa_o = O.quant_act_1x128(bf16_to_np(case.a[rows]), pow2)
    assert np.array_equal(qa[rows].cpu().numpy(), qa_o)
    nbs = sample_block_rows(case.w.shape[0], 6, 12)
    wrows, qw_o, sw_o = weight_block_rows(case.w, nbs, pow2)
    assert np.array_equal(qw[torch.from_numpy(wrows)].cpu().numpy(), qw_o)
    ref = O.gemm_ref(qa_o, sa_o, qw_o, sw_o)
    assert_gemm_close(bf16_to_np(y[rows])[:, wrows], ref, f"qwen prefill {layer} pow2={pow2}")


@pytest.mark.parametrize("M", [1, 8, 32])
def test_decode_layer_chain(ops, M):
    """Decode steps as a model runs them: for each of three layers the
    activation quantiser and then the skinny GEMM, back to back on one stream
    with no synchronisation (up to 32 tokens both launch as programmatic
    dependents, so each kernel's prologue overlaps the previous kernel), the
    next layer's input being written by the host copy in between.  Every
    layer's codes and output are checked against the oracle."""
    K, N = 4096, 2048
    layers = []
    for i in range(3):
        x = I.normal_bf16(I.stream(90 + i, M), (M, K))
        w = I.normal_bf16(I.stream(95 + i, M), (N, K), std=0.02)
        qw, sw = ops.quant_weight(w.cuda())
        layers.append((x, w, qw, sw))
    torch.cuda.synchronize()
    outs = []
    for x, _, qw, sw in layers:
        qa, sa = ops.quant_act(x.cuda())
        outs.append((ops.gemm(qa, sa, qw, sw), qa, sa))
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    for (x, w, qw, sw), (y, qa, sa) in zip(layers, outs):
        qa_o, sa_o = O.quant_act_1x128(bf16_to_np(x))
        assert np.array_equal(qa.cpu().numpy(), qa_o)
        qw_o, sw_o = O.quant_weight_128x128(bf16_to_np(w), False)
        assert np.array_equal(qw.cpu().numpy(), qw_o)
        ref = O.gemm_ref(qa_o, sa_o, qw_o, sw_o)
        assert_gemm_close(bf16_to_np(y), ref, f"decode chain M={M}")


@pytest.mark.parametrize("K,N", [(14336, 4096), (4096, 6144)])
@pytest.mark.parametrize("M", [1, 8, 64, 256])
def test_decode_full_size(ops, M, K, N):
    case = I.decode_case(M, K, N)
    y, (qa, sa), (qw, sw) = ops.linear(case.a.cuda(), case.w.cuda())
    torch.cuda.synchronize()
    qa_o, sa_o = O.quant_act_1x128(bf16_to_np(case.a))
    assert np.array_equal(qa.cpu().numpy(), qa_o)
    wrows, qw_o, sw_o = weight_block_rows(case.w, sample_block_rows(N, 6, M + K), False)
    assert np.array_equal(qw[torch.from_numpy(wrows)].cpu().numpy(), qw_o)
    ref = O.gemm_ref(qa_o, sa_o, qw_o, sw_o)
    assert_gemm_close(bf16_to_np(y)[:, wrows], ref, f"decode M={M}")


# ------------------------------------------------------------ grouped
def _grouped_ref_blocks(qw_dev, w, grp, qa_o, sa_o, N, pow2, seed):
    """Oracle reference of sampled grouped-GEMM rows (row i in expert grp[i])
    on a few 128-row blocks of each expert's weight, quantised by the oracle
    (and checked against the device's codes for those blocks).  Returns the
    output columns covered and the reference [rows, columns]."""
    nbs = sample_block_rows(N, 2, seed)
    ref = []
    for i, g in enumerate(grp):
        wrows, q, s = weight_block_rows(w[int(g)], nbs, pow2)
        if i == 0 or g != grp[i - 1]:
            assert np.array_equal(qw_dev[int(g)][torch.from_numpy(wrows)].cpu().numpy(), q)
        ref.append(O.gemm_ref(qa_o[i:i + 1], sa_o[i:i + 1], q, s)[0])
    return wrows, np.stack(ref)


def _grouped_inputs(offsets, N, K, seed, pow2=False):
    G = len(offsets) - 1
    M = int(offsets[-1])
    a = I.normal_bf16(I.stream(seed, 1), (M, K))
    w = I.normal_bf16(I.stream(seed, 2), (G, N, K), std=0.02)
    qa, sa = O.quant_act_1x128(bf16_to_np(a), pow2)
    qs = [O.quant_weight_128x128(bf16_to_np(w[g]), pow2) for g in range(G)]
    qw = np.stack([q for q, _ in qs])
    sw = np.stack([s for _, s in qs])
    return qa, sa, qw, sw


def _run_grouped(ops, qa, sa, offsets, qw, sw, pow2=False, path="auto"):
    dqa, dsa, _, _ = _to_dev(qa, sa, qw[0], sw[0])
    c = ops.grouped_gemm(dqa, dsa, torch.tensor(offsets, dtype=torch.int32, device="cuda"),
                         torch.from_numpy(qw).cuda(), torch.from_numpy(sw).cuda(), pow2, path)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    return bf16_to_np(c)


@pytest.mark.parametrize("path", ["promote", "mx"])
@pytest.mark.parametrize("offsets", [[0, 5, 5, 140, 140, 300, 301], [0, 0, 0, 128], [0, 1000],
                                     [0, 129, 258, 387, 516]])
def test_grouped_ragged_with_empty_experts(ops, offsets, path):
    # N = 384: the MX kernel's 256-wide tiles end half outside an expert's
    # weights (the extra rows belong to the next expert or lie past the end).
    N, K = 384, 512
    pow2 = path == "mx"
    qa, sa, qw, sw = _grouped_inputs(offsets, N, K, seed=len(offsets), pow2=pow2)
    c = _run_grouped(ops, qa, sa, offsets, qw, sw, pow2, path)
    assert_gemm_close(c, O.grouped_gemm_ref(qa, sa, offsets, qw, sw), f"grouped {path} {offsets}")


@pytest.mark.parametrize("pow2", [False, True])
def test_grouped_moe_full_size_sampled_rows(ops, pow2):
    """Qwen3-30B-A3B-shaped experts (gate+up: K 2048, N 1536), Zipf routing;
    power-of-two scales take the MX kernel."""
    m = I.moe_case(with_weights=False)
    G, N, K = 128, 1536, 2048
    w = I.normal_bf16(I.stream(0, 82), (G, N, K), std=0.02)
    x = m.a_gate_up.cuda()
    qa, sa = ops.quant_act(x, pow2)
    qw = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device="cuda")
    wd = w.cuda()
    mode = ops.FP8_SCALE_POW2 if pow2 else ops.FP8_SCALE_FP32_AMAX
    for g in range(G):
        ops.fp8_quant_weight_128x128(wd[g], qw[g], sw[g], mode)
    offs = torch.from_numpy(m.offsets).cuda()
    c = ops.grouped_gemm(qa, sa, offs, qw, sw, pow2)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    rng = np.random.Generator(np.random.PCG64(9))
    rows = np.sort(rng.choice(x.shape[0], 32, replace=False))
    # include the first and last row of a few experts (tile edges)
    rows = np.unique(np.concatenate([rows, m.offsets[1:6] - 1, m.offsets[:5]]))
    rows = rows[rows < x.shape[0]]
    qa_o, sa_o = O.quant_act_1x128(bf16_to_np(m.a_gate_up[rows]), pow2)
    assert np.array_equal(qa[rows].cpu().numpy(), qa_o)
    grp = np.searchsorted(m.offsets, rows, side="right") - 1
    wrows, ref = _grouped_ref_blocks(qw, w, grp, qa_o, sa_o, N, pow2, seed=10)
    assert_gemm_close(bf16_to_np(c[rows])[:, wrows], ref, "moe gate_up")


@pytest.mark.parametrize("pow2", [False, True])
def test_grouped_moe_down_full_size_sampled_rows(ops, pow2):
    """Qwen3-30B-A3B-shaped expert down projection (K 768: six K-blocks, so the
    MX kernel's last scale-factor group is partial; N 2048), Zipf routing."""
    m = I.moe_case(with_weights=False)
    G, N, K = 128, 2048, 768
    w = I.normal_bf16(I.stream(0, 83), (G, N, K), std=0.02)
    x = m.a_down.cuda()
    qa, sa = ops.quant_act(x, pow2)
    qw = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device="cuda")
    wd = w.cuda()
    mode = ops.FP8_SCALE_POW2 if pow2 else ops.FP8_SCALE_FP32_AMAX
    for g in range(G):
        ops.fp8_quant_weight_128x128(wd[g], qw[g], sw[g], mode)
    offs = torch.from_numpy(m.offsets).cuda()
    c = ops.grouped_gemm(qa, sa, offs, qw, sw, pow2)
    torch.cuda.synchronize()
    assert ops.fp8_last_device_status() == 0
    rng = np.random.Generator(np.random.PCG64(19))
    rows = np.sort(rng.choice(x.shape[0], 32, replace=False))
    rows = np.unique(np.concatenate([rows, m.offsets[1:6] - 1, m.offsets[:5]]))
    rows = rows[rows < x.shape[0]]
    qa_o, sa_o = O.quant_act_1x128(bf16_to_np(m.a_down[rows]), pow2)
    assert np.array_equal(qa[rows].cpu().numpy(), qa_o)
    grp = np.searchsorted(m.offsets, rows, side="right") - 1
    wrows, ref = _grouped_ref_blocks(qw, w, grp, qa_o, sa_o, N, pow2, seed=20)
    assert_gemm_close(bf16_to_np(c[rows])[:, wrows], ref, "moe down")
