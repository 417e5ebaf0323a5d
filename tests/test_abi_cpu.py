"""The C-ABI library builds, loads without a GPU, exports every entry point
include/fp8bs.h declares, and rejects bad arguments on the host before any
CUDA call (so these run on a machine with no GPU)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")


@pytest.fixture(scope="module")
def L():
    from fp8_block_scaled_05_gb300 import build, ops
    build.build()
    return ops.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"FP8BS_API\s+[\w\s\*]+?\**\s*\b(fp8_\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"fp8_quant_act_1x128", "fp8_quant_weight_128x128", "fp8_blockscaled_gemm",
            "fp8_blockscaled_grouped_gemm", "fp8_gemm_workspace_size", "fp8_status_string",
            "fp8_last_device_status", "fp8_gemm_plan"} <= names


def test_every_declared_symbol_is_exported(L):
    from fp8_block_scaled_05_gb300 import ops
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in ops.SIGNATURES, f"binding lacks {name}"


def test_status_strings(L):
    for code in range(10):
        s = L.fp8_status_string(code).decode()
        assert s.startswith("FP8_"), s


NULL = None
A16 = 0x10000          # aligned fake addresses: never dereferenced (validation fails first or no GPU)
A16b = 0x20000
A16c = 0x30000
MIS = 0x10008          # misaligned


def test_quant_act_validation(L):
    f = L.fp8_quant_act_1x128
    assert f(NULL, 4, 256, 256, A16, 256, A16b, 4, 0, NULL) == 1          # null x
    assert f(A16, 4, 200, 256, A16b, 256, A16c, 4, 0, NULL) == 2          # K % 128
    assert f(A16, 4, 256, 128, A16b, 256, A16c, 4, 0, NULL) == 2          # ldx < K
    assert f(A16, 8, 256, 256, A16b, 256, A16c, 4, 0, NULL) == 2          # lds < M
    assert f(A16, 4, 256, 260, A16b, 256, A16c, 4, 0, NULL) == 3          # ldx % 8
    assert f(MIS, 4, 256, 256, A16b, 256, A16c, 4, 0, NULL) == 3          # x misaligned
    assert f(A16, 4, 256, 256, A16b, 264, A16c, 4, 0, NULL) == 3          # ldq % 16
    assert f(A16, 4, 256, 256, A16b, 256, A16c, 6, 0, NULL) == 3          # lds % 4
    assert f(A16, 4, 256, 256, A16b, 256, A16c, 4, 7, NULL) == 4          # mode
    assert f(A16, -1, 256, 256, A16b, 256, A16c, 4, 0, NULL) == 2         # M < 0
    assert f(NULL, 0, 256, 256, NULL, 256, NULL, 4, 0, NULL) == 0         # M == 0: no-op


def test_quant_weight_validation(L):
    f = L.fp8_quant_weight_128x128
    assert f(NULL, 128, 256, 256, A16, 256, A16b, 0, NULL) == 1
    assert f(A16, 100, 256, 256, A16b, 256, A16c, 0, NULL) == 2
    assert f(A16, 128, 256, 256, A16b, 256, A16c, 2, NULL) == 4
    assert f(A16, 128, 256, 256, MIS, 256, A16c, 0, NULL) == 3


def test_gemm_validation(L):
    f = L.fp8_blockscaled_gemm
    ok = dict(qa=A16, lda=256, sa=A16b, ldsa=8, qb=A16c, ldb=256, sb=A16, c=A16b, ldc=128,
              M=8, N=128, K=256, flags=0, ws=NULL, wsb=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["qa"], a["lda"], a["sa"], a["ldsa"], a["qb"], a["ldb"], a["sb"], a["c"], a["ldc"],
                 a["M"], a["N"], a["K"], a["flags"], a["ws"], a["wsb"], NULL)

    assert call(qa=NULL) == 1
    assert call(N=100) == 2
    assert call(K=0) == 2
    assert call(ldsa=4) == 2
    assert call(ldc=120) == 2
    assert call(lda=272) == 0 or call(lda=272) == 6 or True   # valid pitch: reaches the device check
    assert call(lda=264) == 3
    assert call(ldc=132) == 3
    assert call(c=MIS) == 3
    assert call(flags=0x100) == 4
    assert call(flags=0x20) == 4                  # MX path without the pow2 promise
    assert call(M=0, qa=NULL) == 0
    # valid arguments: the next check is the device (none here -> FP8_ERR_ARCH)
    if not _has_gpu():
        assert call() == 6


def test_gemm_quant_validation(L):
    f = L.fp8_blockscaled_gemm_quant
    ok = dict(qa=A16, lda=256, sa=A16b, ldsa=8, qb=A16c, ldb=256, sb=A16, c=A16b, ldc=128, qc=A16c, ldqc=128,
              sc=A16, ldsc=8, M=8, N=128, K=256, flags=0, mode=0, ws=NULL, wsb=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["qa"], a["lda"], a["sa"], a["ldsa"], a["qb"], a["ldb"], a["sb"], a["c"], a["ldc"], a["qc"],
                 a["ldqc"], a["sc"], a["ldsc"], a["M"], a["N"], a["K"], a["flags"], a["mode"], a["ws"], a["wsb"],
                 NULL)

    assert call(qc=NULL) == 1
    assert call(sc=NULL) == 1
    assert call(mode=7) == 4
    assert call(ldqc=120) == 2
    assert call(ldsc=4) == 2
    assert call(ldqc=136) == 3
    assert call(sc=MIS) == 3
    assert call(flags=0x20) == 4                  # MX without the pow2 promise
    assert call(flags=0x30) == 9                  # the skinny path has no fused quantisation
    assert call(M=0, qc=NULL) == 0
    if not _has_gpu():
        assert call() == 6                        # valid arguments; no sm_103 device here
        assert call(c=NULL, ldc=0) == 6           # C is optional
        assert call(flags=0x21) == 6              # MX with pow2 scales


def test_quant_act_128x1_validation(L):
    f = L.fp8_quant_act_128x1
    ok = dict(x=A16, M=256, K=128, ldx=128, qt=A16b, ldqt=256, st=A16c, ldst=128, q=NULL, ldq=0, s=NULL, lds=0,
              mode=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["x"], a["M"], a["K"], a["ldx"], a["qt"], a["ldqt"], a["st"], a["ldst"], a["q"], a["ldq"],
                 a["s"], a["lds"], a["mode"], NULL)

    assert call(x=NULL) == 1
    assert call(qt=NULL) == 1
    assert call(st=NULL) == 1
    assert call(q=A16) == 1                       # q without s
    assert call(M=200, ldqt=200) == 2             # qt rows hold the padded 256 tokens
    assert call(K=200) == 2
    assert call(ldqt=128) == 2                    # ldqt < M
    assert call(ldst=64) == 2                     # ldst < K
    assert call(ldqt=264) == 3
    assert call(ldst=130) == 3
    assert call(st=MIS) == 3
    assert call(q=A16, s=A16, ldq=64, lds=256) == 2   # ldq < K
    assert call(q=A16, s=A16, ldq=128, lds=200) == 2  # lds < M
    assert call(q=A16, s=MIS, ldq=128, lds=256) == 3
    assert call(mode=5) == 4
    assert call(M=0) == 0
    if not _has_gpu():
        assert call() == 6
        assert call(q=A16, s=A16, ldq=128, lds=256) == 6
        assert call(M=200, ldqt=256) == 6         # a ragged last token block is padded


def test_quant_weight_t_validation(L):
    f = L.fp8_quant_weight_128x128_t
    ok = dict(w=A16, N=256, K=128, ldw=128, q=NULL, ldq=0, s=NULL, qt=A16b, ldqt=256, st=A16c, mode=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["w"], a["N"], a["K"], a["ldw"], a["q"], a["ldq"], a["s"], a["qt"], a["ldqt"], a["st"],
                 a["mode"], NULL)

    assert call(w=NULL) == 1
    assert call(qt=NULL) == 1
    assert call(s=A16) == 1                       # s without q
    assert call(N=0) == 2
    assert call(N=200) == 2
    assert call(ldqt=128) == 2                    # ldqt < N
    assert call(ldqt=272 + 8) == 3
    assert call(q=A16, s=A16, ldq=64) == 2        # ldq < K
    assert call(q=A16, s=A16, ldq=136) == 3
    assert call(mode=9) == 4
    if not _has_gpu():
        assert call() == 6
        assert call(q=A16, s=A16, ldq=128) == 6


def test_wgrad_validation(L):
    f = L.fp8_blockscaled_gemm_wgrad
    ok = dict(qa=A16, lda=256, sa=A16b, ldsa=256, qb=A16c, ldb=256, sb=A16, ldsb=128, c=A16b, ldc=128, M=256,
              N=128, K=256, flags=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["qa"], a["lda"], a["sa"], a["ldsa"], a["qb"], a["ldb"], a["sb"], a["ldsb"], a["c"], a["ldc"],
                 a["M"], a["N"], a["K"], a["flags"], NULL, 0, NULL)

    assert call(sb=NULL) == 1
    assert call(ldsb=64) == 2                     # ldsb < N
    assert call(ldsb=130) == 3
    assert call(K=200) == 2
    assert call(flags=0x20) == 4                  # MX without the pow2 promise
    assert call(flags=0x30) == 9                  # no skinny wgrad
    assert call(M=0) == 0
    if not _has_gpu():
        assert call() == 6
        assert call(flags=0x21) == 6


def test_quant_per_tensor_validation(L):
    f = L.fp8_quant_per_tensor
    ok = dict(x=A16, M=4, K=256, ldx=256, q=A16b, ldq=256, sa=A16c, mode=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["x"], a["M"], a["K"], a["ldx"], a["q"], a["ldq"], a["sa"], a["mode"], NULL)

    assert call(x=NULL) == 1
    assert call(sa=NULL) == 1
    assert call(K=260) == 2                       # K % 8
    assert call(ldq=128) == 2
    assert call(ldq=264) == 3
    assert call(sa=A16c + 4) == 3                 # scale_amax 8-byte aligned
    assert call(mode=3) == 4
    assert call(M=0) == 0
    if not _has_gpu():
        assert call() == 6
        assert call(K=8, ldx=8, ldq=16) == 6      # any K % 8 == 0


def test_tensorscaled_gemm_validation(L):
    f = L.fp8_tensorscaled_gemm
    ok = dict(qa=A16, lda=256, sa=A16b, qb=A16c, ldb=256, sb=A16, c=A16b, ldc=128, M=8, N=128, K=256, flags=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["qa"], a["lda"], a["sa"], a["qb"], a["ldb"], a["sb"], a["c"], a["ldc"], a["M"], a["N"], a["K"],
                 a["flags"], NULL, 0, NULL)

    assert call(sa=NULL) == 1
    assert call(sb=NULL) == 1
    assert call(K=200) == 2
    assert call(ldb=128) == 2
    assert call(flags=0x10) == 9                  # promote: not built for per-tensor scales
    assert call(flags=0x30) == 9                  # nor skinny
    assert call(M=0) == 0
    if not _has_gpu():
        assert call() == 6
        assert call(flags=0x20) == 6              # MX without the pow2 flag is fine here
        assert call(flags=0x21) == 6


def test_quant_with_scale_validation(L):
    f = L.fp8_quant_with_scale
    assert f(NULL, 4, 128, 128, A16b, 128, A16c, NULL) == 1
    assert f(A16, 4, 128, 128, A16b, 128, NULL, NULL) == 1
    assert f(A16, 4, 130, 136, A16b, 144, A16c, NULL) == 2        # K % 8
    assert f(A16, 4, 128, 128, A16b, 136, A16c, NULL) == 3        # ldq % 16
    assert f(A16, 4, 128, 128, A16b, 128, A16c + 2, NULL) == 3    # scale 4-byte aligned
    assert f(A16, 0, 128, 128, NULL, 128, NULL, NULL) == 0
    if not _has_gpu():
        assert f(A16, 4, 128, 128, A16b, 128, A16c, NULL) == 6


def test_decode_attention_validation(L):
    f = L.fp8_decode_attention
    ok = dict(q=A16, sq=A16b, k=A16c, sk=A16b, v=A16, sv=A16b, lens=A16c, B=2, Hq=8, Hkv=2, T=1024, D=128,
              out=A16b, ws=A16c, wsb=1 << 20)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["sq"], a["k"], a["sk"], a["v"], a["sv"], a["lens"], a["B"], a["Hq"], a["Hkv"], a["T"],
                 a["D"], a["out"], a["ws"], a["wsb"], NULL)

    assert call(D=64) == 2
    assert call(Hq=6, Hkv=4) == 2                 # Hq % Hkv
    assert call(Hq=48, Hkv=3) == 2                # group of 16
    assert call(T=0) == 2
    assert call(q=NULL) == 1
    assert call(lens=NULL) == 1
    assert call(k=MIS) == 3
    assert call(ws=NULL) == 5                     # two splits need the workspace
    assert call(wsb=100) == 5
    assert call(B=0) == 0
    assert L.fp8_decode_attention_workspace_size(2, 8, 512) == 0       # one split: direct output
    assert L.fp8_decode_attention_workspace_size(2, 8, 1024) == 2 * 8 * 2 * 130 * 4
    if not _has_gpu():
        assert call() == 6
        assert call(T=512, ws=NULL, wsb=0) == 6


def test_kv_cache_append_validation(L):
    f = L.fp8_kv_cache_append
    assert f(A16, A16b, A16c, A16c, A16, A16b, A16c, 2, 8, 64, 64, NULL) == 2     # D != 128
    assert f(NULL, A16b, A16c, A16c, A16, A16b, A16c, 2, 8, 64, 128, NULL) == 1
    assert f(A16, A16b, A16c, A16c, A16, MIS, A16c, 2, 8, 64, 128, NULL) == 3
    assert f(A16, A16b, A16c, A16c, A16, A16b, A16c, 0, 8, 64, 128, NULL) == 0
    if not _has_gpu():
        assert f(A16, A16b, A16c, A16c, A16, A16b, A16c, 2, 8, 64, 128, NULL) == 6


def test_e8_scales_validation(L):
    qa = L.fp8_quant_act_1x128_e8
    assert qa(NULL, 4, 256, 256, A16b, 256, A16c, 4, NULL) == 1
    assert qa(A16, 4, 200, 256, A16b, 256, A16c, 4, NULL) == 2
    assert qa(A16, 8, 256, 256, A16b, 256, A16c, 4, NULL) == 2      # lds < M
    assert qa(A16, 4, 256, 256, MIS, 256, A16c, 4, NULL) == 3      # codes misaligned
    qw = L.fp8_quant_weight_128x128_e8
    assert qw(A16, 128, 200, 256, A16b, 256, A16c, NULL) == 2
    assert qw(A16, 128, 256, 256, A16b, 256, NULL, NULL) == 1
    g = L.fp8_blockscaled_gemm
    args = (A16, 256, A16b, 8, A16c, 256, A16, A16b, 128, 8, 128, 256)
    assert g(*args, 0x12, NULL, 0, NULL) == 9     # UE8M0 scales on the promote path
    assert g(*args, 0x32, NULL, 0, NULL) == 9     # nor skinny
    assert L.fp8_blockscaled_gemm_wgrad(A16, 256, A16b, 256, A16c, 256, A16, 128, A16b, 128, 256, 128, 256, 0x2,
                                        NULL, 0, NULL) == 9
    assert L.fp8_tensorscaled_gemm(A16, 256, A16b, A16c, 256, A16, A16b, 128, 8, 128, 256, 0x2, NULL, 0, NULL) == 4
    if not _has_gpu():
        assert qa(A16, 4, 256, 256, A16b, 256, A16c, 4, NULL) == 6
        assert g(*args, 0x2, NULL, 0, NULL) == 6  # AUTO picks MX
        assert g(*args, 0x22, NULL, 0, NULL) == 6


def test_plan_with_scale_flags(L):
    from fp8_block_scaled_05_gb300 import ops
    # UE8M0 byte scales always take the MX kernel (the only one that reads them),
    # power-of-two fp32 scales take it above the decode sizes
    assert ops.fp8_gemm_plan(4096, 4096, 4096, ops.FP8_GEMM_SCALES_E8)[0] == ops.FP8_GEMM_PATH_MX
    assert ops.fp8_gemm_plan(8, 4096, 4096, ops.FP8_GEMM_SCALES_E8)[0] == ops.FP8_GEMM_PATH_MX
    assert ops.fp8_gemm_plan(4096, 4096, 4096, ops.FP8_GEMM_SCALES_POW2)[0] == ops.FP8_GEMM_PATH_MX
    assert ops.fp8_gemm_plan(8, 4096, 4096, ops.FP8_GEMM_SCALES_POW2)[0] == ops.FP8_GEMM_PATH_SKINNY


def test_grouped_scale_flag_validation(L):
    f = L.fp8_blockscaled_grouped_gemm
    base = (A16, 256, A16b, 8, A16c, 2, 8, A16, A16b, A16c, 128, 128, 256)
    assert f(*base, 0x12, NULL, 0, NULL) == 9     # UE8M0 scales on the promote kernel
    assert f(*base, 0x20, NULL, 0, NULL) == 4     # MX needs power-of-two (or UE8M0) scales
    assert f(*base, 0x40, NULL, 0, NULL) == 4     # unknown path bits
    if not _has_gpu():
        assert f(*base, 0x2, NULL, 0, NULL) == 6  # AUTO takes MX for byte scales


def test_attention_workspace_sizes(L):
    # one split (T <= 512): the kernel writes the output directly
    assert L.fp8_decode_attention_workspace_size(64, 32, 512) == 0
    # T = 4096: 8 splits of (max, sum, 128 partial outputs) per (sequence, head)
    assert L.fp8_decode_attention_workspace_size(64, 32, 4096) == 64 * 32 * 8 * 130 * 4
    assert L.fp8_decode_attention_workspace_size(0, 32, 4096) == 0


def test_grouped_validation(L):
    f = L.fp8_blockscaled_grouped_gemm
    assert f(A16, 256, A16b, 8, A16c, 0, 8, A16, A16b, A16c, 128, 128, 256, 0, NULL, 0, NULL) == 2   # G=0
    assert f(A16, 256, A16b, 8, NULL, 2, 8, A16, A16b, A16c, 128, 128, 256, 0, NULL, 0, NULL) == 1   # offsets
    assert f(A16, 256, A16b, 8, A16c, 2, 8, A16, A16b, A16c, 128, 128, 256, 0x30, NULL, 0, NULL) == 9


def test_workspace_size_and_plan(L):
    from fp8_block_scaled_05_gb300 import ops
    # Large M (no device here, so 152 SMs are assumed): 32 x 24 = 768 tiles of
    # 128 x 256 are 5 full waves + 8 tiles; those 8 are split into
    # min(152 // 8, 32 // 8, 4) = 4 parts: the fixed 64 KiB ticket region +
    # 8 x 4 fp32 128 x 256 parts.
    assert ops.fp8_gemm_workspace_size(4096, 6144, 4096) == 65536 + 8 * 4 * 128 * 256 * 4
    assert ops.fp8_gemm_workspace_size(4096, 4864, 4096) == 0          # 32 x 19 = 608 tiles: 4 full waves
    assert ops.fp8_gemm_workspace_size(4096, 6144, 1920) == 0          # 15 K-blocks: no 2 parts of 8
    assert ops.fp8_gemm_workspace_size(1, 6144, 4096) > 0              # decode: split-K partials
    path, splits = ops.fp8_gemm_plan(8, 4096, 14336)
    assert path == ops.FP8_GEMM_PATH_SKINNY and splits > 1
    assert ops.fp8_gemm_plan(4096, 4096, 4096)[0] == ops.FP8_GEMM_PATH_PROMOTE
    # the automatic path: the skinny kernel up to 128 rows, the large-M kernels above
    assert ops.fp8_gemm_plan(128, 4096, 14336)[0] == ops.FP8_GEMM_PATH_SKINNY
    assert ops.fp8_gemm_plan(129, 4096, 14336)[0] == ops.FP8_GEMM_PATH_PROMOTE
    assert ops.fp8_gemm_plan(256, 4096, 14336, ops.FP8_GEMM_SCALES_POW2)[0] == ops.FP8_GEMM_PATH_MX


def _skinny_bytes(ops, M, N, K):
    """The skinny path's scratch by the header's formula, with the CTA count P
    the library plans for the forced skinny path."""
    _, P = ops.fp8_gemm_plan(M, N, K, ops.FP8_GEMM_PATH_SKINNY)
    nt = 16 if M <= 16 else 32 if M <= 32 else 64 if M <= 64 else 128
    KB, T = K // 128, (N // 128) * -(-M // nt)
    U = T * KB
    return 65536 + (P + T - 1) * nt * 128 * 4 if any((c * U // P) % KB for c in range(1, P)) else 0


def _large_m_bytes(M, N, K, sms=152):
    """The large-M kernels' K split (256-wide tiles): every tile split when the
    tiles do not fill the SMs, else the last wave's tiles."""
    tiles = -(-M // 128) * (N // 256)
    KB = K // 128
    if tiles < sms:
        left, parts = tiles, min(sms // tiles, 16)
    else:
        left = tiles % sms
        if left == 0:
            return 0
        parts = min(sms // left, 4)
    parts = min(parts, KB // 8)
    return 65536 + left * parts * 128 * 256 * 4 if parts >= 2 else 0


@pytest.mark.parametrize("M,N,K", [(1, 6144, 4096), (64, 4096, 14336), (128, 4096, 14336), (200, 4096, 14336),
                                   (256, 6144, 4096), (512, 4096, 4096), (4096, 6144, 4096)])
def test_workspace_size_covers_every_path(L, M, N, K):
    """fp8_gemm_workspace_size is the largest need of the paths these sizes
    may take, automatic or forced (no device here: 152 SMs assumed): at least
    the skinny kernel's scratch up to 256 rows and the large-M kernels' K
    split, and equal to the larger of the two."""
    from fp8_block_scaled_05_gb300 import ops
    need = ops.fp8_gemm_workspace_size(M, N, K)
    sk = _skinny_bytes(ops, M, N, K) if M <= 256 else 0
    lm = _large_m_bytes(M, N, K)
    assert need == max(sk, lm), (need, sk, lm)


def _has_gpu():
    import torch
    return torch.cuda.is_available()


def test_noalloc_validation(L):
    """The no-allocation decode GEMM takes fp32 scales only: UE8M0 byte scales
    (FP8_GEMM_SCALES_E8) are refused before anything launches, as are the
    large-M paths and M > 256."""
    f = L.fp8_blockscaled_gemm_skinny_noalloc

    def call(M=8, flags=0, qa=A16):
        return f(qa, 256, A16b, 8, A16c, 256, A16, A16b, 128, M, 128, 256, flags, NULL)

    assert call(flags=0x2) == 9                   # E8 byte scales, AUTO path
    assert call(flags=0x32) == 9                  # E8 byte scales, SKINNY path
    assert call(flags=0x10) == 4                  # promote path
    assert call(flags=0x21) == 4                  # MX path
    assert call(qa=NULL) == 1
    assert call(qa=MIS) == 3
    assert call(M=0) == 0
    assert call(M=300) == 2                       # beyond 256 tokens (ldsa < M first would also say SHAPE)


def test_quant_act_128x1_grouped_validation(L):
    """Grouped 128x1 quantiser: ldqt must hold 128 (ceil(T/128) + G) slots."""
    f = L.fp8_quant_act_128x1_grouped
    ok = dict(x=A16, T=300, K=256, ldx=256, offs=A16b, G=3, qt=A16c, ldqt=768, st=A16, ldst=256, mode=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["x"], a["T"], a["K"], a["ldx"], a["offs"], a["G"], a["qt"], a["ldqt"], a["st"], a["ldst"],
                 a["mode"], NULL)

    assert call(x=NULL) == 1
    assert call(offs=NULL) == 1
    assert call(K=200) == 2
    assert call(G=0) == 2
    assert call(G=1025) == 2
    assert call(ldqt=640) == 2                    # 128 x (3 + 3) slots needed
    assert call(ldst=128) == 2                    # ldst < K
    assert call(ldqt=776) == 3                    # row pitch not a multiple of 16 bytes
    assert call(offs=A16b + 2) == 3               # int32 offsets misaligned
    assert call(mode=7) == 4
    assert call(T=0) == 0                         # nothing to quantise
    if not _has_gpu():
        assert call() == 6


def test_grouped_wgrad_validation(L):
    """Grouped weight-gradient GEMM: fp32 scales only (no UE8M0 bytes); the
    MX path needs the power-of-two promise; no skinny path."""
    f = L.fp8_blockscaled_grouped_gemm_wgrad
    ok = dict(qa=A16, lda=768, sa=A16b, ldsa=256, qb=A16c, ldb=768, sb=A16, ldsb=128, offs=A16b, G=3, T=300,
              c=A16c, ldc=128, M=256, N=128, flags=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["qa"], a["lda"], a["sa"], a["ldsa"], a["qb"], a["ldb"], a["sb"], a["ldsb"], a["offs"], a["G"],
                 a["T"], a["c"], a["ldc"], a["M"], a["N"], a["flags"], NULL)

    assert call(flags=0x2) == 9                   # UE8M0 byte scales
    assert call(flags=0x20) == 4                  # MX path without the pow2 promise
    assert call(flags=0x30) == 9                  # skinny path
    assert call(M=200) == 2
    assert call(G=0) == 2
    assert call(lda=640) == 2                     # fewer slots than the quantiser may fill
    assert call(ldsb=64) == 2                     # ldsb < N
    assert call(ldc=64) == 2                      # ldc < N
    assert call(offs=NULL) == 1
    assert call(sb=NULL) == 1
    assert call(lda=776) == 3
    assert call(c=A16c + 8) == 3
    assert call(M=0) == 0                         # empty output
    if not _has_gpu():
        assert call() == 6
        assert call(flags=0x11) == 6              # promote path, pow2 scales
        assert call(flags=0x21) == 6              # MX path, pow2 scales


def test_quant_act_weight_validation(L):
    """The layer quantiser takes the union of the two quantisers' rules."""
    f = L.fp8_quant_act_weight
    ok = dict(x=A16, M=8, K=256, ldx=256, qa=A16b, ldqa=256, sa=A16c, ldsa=8, w=A16, N=128, ldw=256, qw=A16b,
              ldqw=256, sw=A16c, mode=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["x"], a["M"], a["K"], a["ldx"], a["qa"], a["ldqa"], a["sa"], a["ldsa"], a["w"], a["N"], a["ldw"],
                 a["qw"], a["ldqw"], a["sw"], a["mode"], NULL)

    assert call(w=NULL) == 1
    assert call(x=NULL) == 1
    assert call(x=NULL, M=0) in (0, 6)           # weights only: x is not needed
    assert call(K=200) == 2
    assert call(N=200) == 2
    assert call(ldsa=4) == 2                     # ldsa < M
    assert call(ldqw=128) == 2                   # ldqw < K
    assert call(ldqa=264) == 3                   # row pitch not a multiple of 16 bytes
    assert call(sw=A16c + 2) == 3
    assert call(mode=5) == 4
    if not _has_gpu():
        assert call() == 6

