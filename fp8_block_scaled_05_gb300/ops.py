"""ctypes binding of libfp8bs.so (include/fp8bs.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of the library.  Functions named like the C entry points take torch
CUDA tensors (PyTorch supplies device memory and streams) and raise
``FP8Error`` on any non-OK status.  ``quant_act``, ``quant_weight``, ``gemm``,
``grouped_gemm`` and ``linear`` are conveniences that allocate their outputs
with torch and then make the same calls.

There is no CPU fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8bs.so")

FP8_OK = 0
STATUS_NAMES = {
    0: "FP8_OK", 1: "FP8_ERR_NULL", 2: "FP8_ERR_SHAPE", 3: "FP8_ERR_ALIGN", 4: "FP8_ERR_SCALE_MODE",
    5: "FP8_ERR_WORKSPACE", 6: "FP8_ERR_ARCH", 7: "FP8_ERR_CUDA", 8: "FP8_ERR_TIMEOUT",
    9: "FP8_ERR_NOT_IMPLEMENTED",
}
FP8_SCALE_FP32_AMAX = 0
FP8_SCALE_POW2 = 1
FP8_GEMM_SCALES_POW2 = 0x1
FP8_GEMM_SCALES_E8 = 0x2
FP8_GEMM_PATH_AUTO = 0x00
FP8_GEMM_PATH_PROMOTE = 0x10
FP8_GEMM_PATH_MX = 0x20
FP8_GEMM_PATH_SKINNY = 0x30
PATHS = {"auto": FP8_GEMM_PATH_AUTO, "promote": FP8_GEMM_PATH_PROMOTE, "mx": FP8_GEMM_PATH_MX,
         "skinny": FP8_GEMM_PATH_SKINNY}

# Every function the header declares, with its ctypes signature.
_i64, _u32, _i32, _vp, _sz = ctypes.c_int64, ctypes.c_uint32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
SIGNATURES = {
    "fp8_quant_act_1x128": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, ctypes.c_int, _vp]),
    "fp8_quant_weight_128x128": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, ctypes.c_int, _vp]),
    "fp8_quant_act_weight": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i64, _vp, _i64,
                                            _vp, ctypes.c_int, _vp]),
    "fp8_blockscaled_gemm": (ctypes.c_int, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i64, _i64, _i64, _i64,
                                            _u32, _vp, _sz, _vp]),
    "fp8_blockscaled_grouped_gemm": (ctypes.c_int, [_vp, _i64, _vp, _i64, _vp, _i32, _i64, _vp, _vp, _vp, _i64,
                                                    _i64, _i64, _u32, _vp, _sz, _vp]),
    "fp8_blockscaled_gemm_skinny_noalloc": (ctypes.c_int, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i64, _i64,
                                                           _i64, _i64, _u32, _vp]),
    "fp8_blockscaled_gemm_quant": (ctypes.c_int, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i64, _vp, _i64, _vp,
                                                  _i64, _i64, _i64, _i64, _u32, ctypes.c_int, _vp, _sz, _vp]),
    "fp8_quant_act_128x1": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                                           ctypes.c_int, _vp]),
    "fp8_quant_weight_128x128_t": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _i64, _vp,
                                                  ctypes.c_int, _vp]),
    "fp8_blockscaled_gemm_wgrad": (ctypes.c_int, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i64,
                                                  _i64, _i64, _u32, _vp, _sz, _vp]),
    "fp8_quant_act_1x128_e8": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp]),
    "fp8_quant_weight_128x128_e8": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp]),
    "fp8_quant_per_tensor": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, ctypes.c_int, _vp]),
    "fp8_tensorscaled_gemm": (ctypes.c_int, [_vp, _i64, _vp, _vp, _i64, _vp, _vp, _i64, _i64, _i64, _i64, _u32,
                                             _vp, _sz, _vp]),
    "fp8_quant_with_scale": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp]),
    "fp8_kv_cache_append": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp]),
    "fp8_decode_attention_workspace_size": (_sz, [_i64, _i64, _i64]),
    "fp8_decode_attention": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _vp,
                                            _vp, _sz, _vp]),
    "fp8_gemm_workspace_size": (_sz, [_i64, _i64, _i64, _i32]),
    "fp8_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fp8_last_device_status": (ctypes.c_int, [_vp]),
    "fp8_gemm_plan": (_u32, [_i64, _i64, _i64, _u32, ctypes.POINTER(_i32)]),
    "fp8_debug_inject": (ctypes.c_int, [_i32, ctypes.c_uint64]),
    "fp8_quant_act_128x1_grouped": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i32, _vp, _i64, _vp, _i64,
                                                   ctypes.c_int, _vp]),
    "fp8_blockscaled_grouped_gemm_wgrad": (ctypes.c_int, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i32,
                                                          _i64, _vp, _i64, _i64, _i64, _u32, _vp]),
}

_lib = None
_lock = threading.Lock()


class FP8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once; raises if it was never built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is not built: run `python -m fp8_block_scaled_05_gb300.build` "
                        "(there is no CPU fallback)")
                L = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    f = getattr(L, name)
                    f.restype = res
                    f.argtypes = args
                _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().fp8_status_string(int(status)).decode()
    except Exception:  # noqa: BLE001 - only used for messages
        return STATUS_NAMES.get(int(status), f"status {status}")


def _check(status: int, where: str):
    if status != FP8_OK:
        raise FP8Error(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, dtype, name: str, rows_major: bool = True):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if rows_major and t.dim() >= 1 and t.shape[-1] > 1 and t.stride(-1) != 1:
        raise ValueError(f"{name} must have unit stride in its last dimension")


# ----------------------------------------------------------- C entry points
def fp8_quant_act_1x128(x: torch.Tensor, q: torch.Tensor, s: torch.Tensor, mode: int = FP8_SCALE_FP32_AMAX,
                        stream=None) -> None:
    """x bf16 [M, K]; q uint8 [M, K]; s fp32 [K/128, lds] with lds >= M."""
    _need(x, torch.bfloat16, "x")
    _need(q, torch.uint8, "q")
    _need(s, torch.float32, "s")
    M, K = x.shape
    _check(lib().fp8_quant_act_1x128(_ptr(x), M, K, x.stride(0), _ptr(q), q.stride(0), _ptr(s), s.stride(0),
                                     int(mode), _stream(stream)), "fp8_quant_act_1x128")


def fp8_quant_weight_128x128(w: torch.Tensor, q: torch.Tensor, s: torch.Tensor,
                             mode: int = FP8_SCALE_FP32_AMAX, stream=None) -> None:
    """w bf16 [N, K]; q uint8 [N, K]; s fp32 [N/128, K/128] contiguous."""
    _need(w, torch.bfloat16, "w")
    _need(q, torch.uint8, "q")
    _need(s, torch.float32, "s")
    if not s.is_contiguous():
        raise ValueError("s must be contiguous")
    N, K = w.shape
    _check(lib().fp8_quant_weight_128x128(_ptr(w), N, K, w.stride(0), _ptr(q), q.stride(0), _ptr(s), int(mode),
                                          _stream(stream)), "fp8_quant_weight_128x128")


def fp8_quant_act_weight(x: torch.Tensor, qa: torch.Tensor, sa: torch.Tensor, w: torch.Tensor, qw: torch.Tensor,
                         sw: torch.Tensor, mode: int = FP8_SCALE_FP32_AMAX, stream=None) -> None:
    """fp8_quant_act_1x128(x, qa, sa) and fp8_quant_weight_128x128(w, qw, sw)
    in one launch; x bf16 [M, K], w bf16 [N, K]."""
    for t, dt, n in ((x, torch.bfloat16, "x"), (qa, torch.uint8, "qa"), (sa, torch.float32, "sa"),
                     (w, torch.bfloat16, "w"), (qw, torch.uint8, "qw"), (sw, torch.float32, "sw")):
        _need(t, dt, n)
    if not sw.is_contiguous():
        raise ValueError("sw must be contiguous")
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("x and w must share K")
    _check(lib().fp8_quant_act_weight(_ptr(x), M, K, x.stride(0), _ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0),
                                      _ptr(w), N, w.stride(0), _ptr(qw), qw.stride(0), _ptr(sw), int(mode),
                                      _stream(stream)), "fp8_quant_act_weight")


def fp8_quant_act_128x1(x: torch.Tensor, qt: torch.Tensor, st: torch.Tensor, q: torch.Tensor | None = None,
                        s: torch.Tensor | None = None, mode: int = FP8_SCALE_FP32_AMAX, stream=None) -> None:
    """x bf16 [M, K] (M % 128 == 0); qt uint8 [K, M] (128x1 codes, transposed);
    st fp32 [M/128, ldst >= K]; optionally q uint8 [M, K] and s fp32
    [K/128, lds >= M] (the 1x128 codes of x from the same pass)."""
    _need(x, torch.bfloat16, "x")
    _need(qt, torch.uint8, "qt")
    _need(st, torch.float32, "st")
    if q is not None:
        _need(q, torch.uint8, "q")
    if s is not None:
        _need(s, torch.float32, "s")
    M, K = x.shape
    _check(lib().fp8_quant_act_128x1(_ptr(x), M, K, x.stride(0), _ptr(qt), qt.stride(0), _ptr(st), st.stride(0),
                                     _ptr(q), q.stride(0) if q is not None else 0, _ptr(s),
                                     s.stride(0) if s is not None else 0, int(mode), _stream(stream)),
           "fp8_quant_act_128x1")


def fp8_quant_weight_128x128_t(w: torch.Tensor, qt: torch.Tensor, st: torch.Tensor, q: torch.Tensor | None = None,
                               s: torch.Tensor | None = None, mode: int = FP8_SCALE_FP32_AMAX,
                               stream=None) -> None:
    """w bf16 [N, K]; qt uint8 [K, N] (W^T codes); st fp32 [K/128, N/128]
    contiguous; optionally q uint8 [N, K] and s fp32 [N/128, K/128] (W's own)."""
    _need(w, torch.bfloat16, "w")
    _need(qt, torch.uint8, "qt")
    _need(st, torch.float32, "st")
    if not st.is_contiguous() or (s is not None and not s.is_contiguous()):
        raise ValueError("st and s must be contiguous")
    if q is not None:
        _need(q, torch.uint8, "q")
    if s is not None:
        _need(s, torch.float32, "s")
    N, K = w.shape
    _check(lib().fp8_quant_weight_128x128_t(_ptr(w), N, K, w.stride(0), _ptr(q),
                                            q.stride(0) if q is not None else 0, _ptr(s), _ptr(qt), qt.stride(0),
                                            _ptr(st), int(mode), _stream(stream)), "fp8_quant_weight_128x128_t")


def fp8_blockscaled_gemm_wgrad(qa, sa, qb, sb, c, flags: int = 0, workspace: torch.Tensor | None = None,
                               stream=None) -> None:
    """C[M, N] (bf16) = qa[M, K] * qb[N, K]^T with 1x128 scales on both
    operands: sa fp32 [K/128, >= M], sb fp32 [K/128, >= N]."""
    _need(qa, torch.uint8, "qa")
    _need(qb, torch.uint8, "qb")
    _need(sa, torch.float32, "sa")
    _need(sb, torch.float32, "sb")
    _need(c, torch.bfloat16, "c")
    M, K = qa.shape
    N = qb.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fp8_blockscaled_gemm_wgrad(_ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0), _ptr(qb), qb.stride(0),
                                            _ptr(sb), sb.stride(0), _ptr(c), c.stride(0), M, N, K, int(flags),
                                            _ptr(workspace), ws_bytes, _stream(stream)),
           "fp8_blockscaled_gemm_wgrad")


def fp8_quant_act_128x1_grouped(x: torch.Tensor, offsets: torch.Tensor, qt: torch.Tensor, st: torch.Tensor,
                                mode: int = FP8_SCALE_FP32_AMAX, stream=None) -> None:
    """x bf16 [T, K] expert-sorted; offsets int32 [G+1] (device); qt uint8
    [K, >= 128 (ceil(T/128) + G)]; st fp32 [ceil(T/128) + G, >= K]."""
    _need(x, torch.bfloat16, "x")
    _need(offsets, torch.int32, "offsets")
    _need(qt, torch.uint8, "qt")
    _need(st, torch.float32, "st")
    T, K = x.shape
    _check(lib().fp8_quant_act_128x1_grouped(_ptr(x), T, K, x.stride(0), _ptr(offsets), offsets.numel() - 1,
                                             _ptr(qt), qt.stride(0), _ptr(st), st.stride(0), int(mode),
                                             _stream(stream)), "fp8_quant_act_128x1_grouped")


def fp8_blockscaled_grouped_gemm_wgrad(qa, sa, qb, sb, offsets, T: int, c, flags: int = 0, stream=None) -> None:
    """c bf16 [G, M, N] (or [G M, N]) = per-expert dY^T X from the grouped
    128x1 operands (qa [M, slots], qb [N, slots])."""
    _need(qa, torch.uint8, "qa")
    _need(qb, torch.uint8, "qb")
    _need(sa, torch.float32, "sa")
    _need(sb, torch.float32, "sb")
    _need(offsets, torch.int32, "offsets")
    _need(c, torch.bfloat16, "c")
    M, N = qa.shape[0], qb.shape[0]
    _check(lib().fp8_blockscaled_grouped_gemm_wgrad(_ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0), _ptr(qb),
                                                    qb.stride(0), _ptr(sb), sb.stride(0), _ptr(offsets),
                                                    offsets.numel() - 1, T, _ptr(c), c.stride(-2), M, N, int(flags),
                                                    _stream(stream)), "fp8_blockscaled_grouped_gemm_wgrad")


def fp8_quant_act_1x128_e8(x: torch.Tensor, q: torch.Tensor, s: torch.Tensor, stream=None) -> None:
    """Power-of-two 1x128 quantisation with UE8M0 scale bytes: s uint8 [K/128, lds >= M]."""
    _need(x, torch.bfloat16, "x")
    _need(q, torch.uint8, "q")
    _need(s, torch.uint8, "s")
    M, K = x.shape
    _check(lib().fp8_quant_act_1x128_e8(_ptr(x), M, K, x.stride(0), _ptr(q), q.stride(0), _ptr(s), s.stride(0),
                                        _stream(stream)), "fp8_quant_act_1x128_e8")


def fp8_quant_weight_128x128_e8(w: torch.Tensor, q: torch.Tensor, s: torch.Tensor, stream=None) -> None:
    """Power-of-two 128x128 quantisation with UE8M0 scale bytes: s uint8 [N/128, K/128] contiguous."""
    _need(w, torch.bfloat16, "w")
    _need(q, torch.uint8, "q")
    _need(s, torch.uint8, "s")
    if not s.is_contiguous():
        raise ValueError("s must be contiguous")
    N, K = w.shape
    _check(lib().fp8_quant_weight_128x128_e8(_ptr(w), N, K, w.stride(0), _ptr(q), q.stride(0), _ptr(s),
                                             _stream(stream)), "fp8_quant_weight_128x128_e8")


def fp8_quant_per_tensor(x: torch.Tensor, q: torch.Tensor, scale_amax: torch.Tensor,
                         mode: int = FP8_SCALE_FP32_AMAX, stream=None) -> None:
    """x bf16 [M, K]; q uint8 [M, K]; scale_amax fp32 [2] (scale, amax) on the device."""
    _need(x, torch.bfloat16, "x")
    _need(q, torch.uint8, "q")
    _need(scale_amax, torch.float32, "scale_amax")
    if scale_amax.numel() < 2 or not scale_amax.is_contiguous():
        raise ValueError("scale_amax must be a contiguous fp32 tensor of 2 elements")
    M, K = x.shape
    _check(lib().fp8_quant_per_tensor(_ptr(x), M, K, x.stride(0), _ptr(q), q.stride(0), _ptr(scale_amax), int(mode),
                                      _stream(stream)), "fp8_quant_per_tensor")


def fp8_quant_with_scale(x: torch.Tensor, q: torch.Tensor, scale: torch.Tensor, stream=None) -> None:
    """q = e4m3(RN(x * RN(1 / scale[0]))); x bf16 [M, K] (or any 2-D view), q uint8 of the same shape."""
    _need(x, torch.bfloat16, "x")
    _need(q, torch.uint8, "q")
    _need(scale, torch.float32, "scale")
    M, K = x.shape
    _check(lib().fp8_quant_with_scale(_ptr(x), M, K, x.stride(0), _ptr(q), q.stride(0), _ptr(scale),
                                      _stream(stream)), "fp8_quant_with_scale")


def fp8_kv_cache_append(k_new, v_new, sk, sv, seq_lens, k_cache, v_cache, stream=None) -> None:
    """k_new / v_new bf16 [B, Hkv, D]; caches uint8 [B, Hkv, T, D]; writes slot seq_lens[b]."""
    for t, dt, n in ((k_new, torch.bfloat16, "k_new"), (v_new, torch.bfloat16, "v_new"),
                     (sk, torch.float32, "sk"), (sv, torch.float32, "sv"), (seq_lens, torch.int32, "seq_lens"),
                     (k_cache, torch.uint8, "k_cache"), (v_cache, torch.uint8, "v_cache")):
        _need(t, dt, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    B, Hkv, T, D = k_cache.shape
    if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D) or v_cache.shape != k_cache.shape:
        raise ValueError("shapes do not match the cache")
    _check(lib().fp8_kv_cache_append(_ptr(k_new), _ptr(v_new), _ptr(sk), _ptr(sv), _ptr(seq_lens), _ptr(k_cache),
                                     _ptr(v_cache), B, Hkv, T, D, _stream(stream)), "fp8_kv_cache_append")


def fp8_decode_attention_workspace_size(B: int, Hq: int, T: int) -> int:
    return int(lib().fp8_decode_attention_workspace_size(B, Hq, T))


def fp8_decode_attention(q, sq, k_cache, sk, v_cache, sv, seq_lens, out, workspace=None, stream=None) -> None:
    """q uint8 [B, Hq, D]; k_cache / v_cache uint8 [B, Hkv, T, D]; sq, sk, sv
    one-element fp32 device tensors; seq_lens int32 [B]; out bf16 [B, Hq, D]."""
    for t, dt, n in ((q, torch.uint8, "q"), (k_cache, torch.uint8, "k_cache"), (v_cache, torch.uint8, "v_cache"),
                     (sq, torch.float32, "sq"), (sk, torch.float32, "sk"), (sv, torch.float32, "sv"),
                     (seq_lens, torch.int32, "seq_lens"), (out, torch.bfloat16, "out")):
        _need(t, dt, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    B, Hq, D = q.shape
    Hkv, T = k_cache.shape[1], k_cache.shape[2]
    if v_cache.shape != k_cache.shape or k_cache.shape[0] != B or k_cache.shape[3] != D:
        raise ValueError("cache shapes do not match q")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fp8_decode_attention(_ptr(q), _ptr(sq), _ptr(k_cache), _ptr(sk), _ptr(v_cache), _ptr(sv),
                                      _ptr(seq_lens), B, Hq, Hkv, T, D, _ptr(out), _ptr(workspace), ws_bytes,
                                      _stream(stream)), "fp8_decode_attention")


def fp8_tensorscaled_gemm(qa, sa, qb, sb, c, flags: int = 0, workspace: torch.Tensor | None = None,
                          stream=None) -> None:
    """C[M, N] (bf16) = sa * sb * qa[M, K] qb[N, K]^T; sa, sb one-element fp32 device tensors."""
    _need(qa, torch.uint8, "qa")
    _need(qb, torch.uint8, "qb")
    _need(sa, torch.float32, "sa")
    _need(sb, torch.float32, "sb")
    _need(c, torch.bfloat16, "c")
    M, K = qa.shape
    N = qb.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fp8_tensorscaled_gemm(_ptr(qa), qa.stride(0), _ptr(sa), _ptr(qb), qb.stride(0), _ptr(sb), _ptr(c),
                                       c.stride(0), M, N, K, int(flags), _ptr(workspace), ws_bytes, _stream(stream)),
           "fp8_tensorscaled_gemm")


def fp8_blockscaled_gemm(qa, sa, qb, sb, c, flags: int = 0, workspace: torch.Tensor | None = None,
                         stream=None) -> None:
    """C[M, N] (bf16) = block-scaled qa[M, K] * qb[N, K]^T (sa, sb uint8 UE8M0
    bytes with FP8_GEMM_SCALES_E8, else fp32)."""
    sdt = torch.uint8 if flags & FP8_GEMM_SCALES_E8 else torch.float32
    _need(qa, torch.uint8, "qa")
    _need(qb, torch.uint8, "qb")
    _need(sa, sdt, "sa")
    _need(sb, sdt, "sb")
    _need(c, torch.bfloat16, "c")
    M, K = qa.shape
    N = qb.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fp8_blockscaled_gemm(_ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0), _ptr(qb), qb.stride(0),
                                      _ptr(sb), _ptr(c), c.stride(0), M, N, K, int(flags), _ptr(workspace),
                                      ws_bytes, _stream(stream)), "fp8_blockscaled_gemm")


def fp8_blockscaled_gemm_quant(qa, sa, qb, sb, c, qc, sc, flags: int = 0, out_mode: int = FP8_SCALE_FP32_AMAX,
                               workspace: torch.Tensor | None = None, stream=None) -> None:
    """C = block-scaled GEMM, and the 1x128 E4M3 quantisation of bf16(C) for
    the next layer: qc uint8 [M, N], sc fp32 [N/128, >= M]; c (bf16 [M, N])
    may be None."""
    _need(qa, torch.uint8, "qa")
    _need(qb, torch.uint8, "qb")
    _need(sa, torch.float32, "sa")
    _need(sb, torch.float32, "sb")
    _need(qc, torch.uint8, "qc")
    _need(sc, torch.float32, "sc")
    if c is not None:
        _need(c, torch.bfloat16, "c")
    M, K = qa.shape
    N = qb.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fp8_blockscaled_gemm_quant(_ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0), _ptr(qb), qb.stride(0),
                                            _ptr(sb), _ptr(c), c.stride(0) if c is not None else 0, _ptr(qc),
                                            qc.stride(0), _ptr(sc), sc.stride(0), M, N, K, int(flags),
                                            int(out_mode), _ptr(workspace), ws_bytes, _stream(stream)),
           "fp8_blockscaled_gemm_quant")


def fp8_blockscaled_grouped_gemm(qa, sa, offsets, qb, sb, c, flags: int = 0,
                                 workspace: torch.Tensor | None = None, stream=None) -> None:
    """Per-expert GEMM; offsets int32 [G+1] on the device; qb uint8 [G, N, K]
    (sa, sb uint8 UE8M0 bytes with FP8_GEMM_SCALES_E8, else fp32)."""
    sdt = torch.uint8 if flags & FP8_GEMM_SCALES_E8 else torch.float32
    _need(qa, torch.uint8, "qa")
    _need(qb, torch.uint8, "qb")
    _need(sa, sdt, "sa")
    _need(sb, sdt, "sb")
    _need(c, torch.bfloat16, "c")
    _need(offsets, torch.int32, "offsets")
    if not (qb.is_contiguous() and sb.is_contiguous() and offsets.is_contiguous()):
        raise ValueError("qb, sb and offsets must be contiguous")
    M, K = qa.shape
    G, N = qb.shape[0], qb.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fp8_blockscaled_grouped_gemm(_ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0), _ptr(offsets), G,
                                              M, _ptr(qb), _ptr(sb), _ptr(c), c.stride(0), N, K, int(flags),
                                              _ptr(workspace), ws_bytes, _stream(stream)),
           "fp8_blockscaled_grouped_gemm")


def fp8_blockscaled_gemm_skinny_noalloc(qa, sa, qb, sb, c, flags: int = 0, stream=None) -> None:
    """Decode-sized (M <= 256) GEMM on the library's own scratch: no
    workspace argument and no allocation (see include/fp8bs.h)."""
    _need(qa, torch.uint8, "qa")
    _need(qb, torch.uint8, "qb")
    _need(sa, torch.float32, "sa")
    _need(sb, torch.float32, "sb")
    _need(c, torch.bfloat16, "c")
    M, K = qa.shape
    N = qb.shape[0]
    _check(lib().fp8_blockscaled_gemm_skinny_noalloc(_ptr(qa), qa.stride(0), _ptr(sa), sa.stride(0), _ptr(qb),
                                                     qb.stride(0), _ptr(sb), _ptr(c), c.stride(0), M, N, K,
                                                     int(flags), _stream(stream)),
           "fp8_blockscaled_gemm_skinny_noalloc")


def fp8_gemm_workspace_size(M: int, N: int, K: int, G: int = 1) -> int:
    return int(lib().fp8_gemm_workspace_size(M, N, K, G))


def fp8_gemm_plan(M: int, N: int, K: int, flags: int = 0):
    sp = ctypes.c_int32(0)
    path = lib().fp8_gemm_plan(M, N, K, flags, ctypes.byref(sp))
    return int(path), int(sp.value)


def fp8_debug_inject(skip_first_load: bool = False, wait_limit_ns: int = 0) -> None:
    """Failure-path test hook: shortened kernel waits and a skipped first
    K-block for the GEMMs launched after it (see include/fp8bs.h)."""
    _check(lib().fp8_debug_inject(1 if skip_first_load else 0, int(wait_limit_ns)), "fp8_debug_inject")


def fp8_last_device_status(stream=None) -> int:
    return int(lib().fp8_last_device_status(_stream(stream)))


# ----------------------------------------------------------- conveniences
def round_up(v: int, m: int) -> int:
    return (v + m - 1) // m * m


def quant_act(x: torch.Tensor, pow2: bool = False, stream=None):
    """Returns (q uint8 [M, K], s fp32 [K/128, round_up(M, 4)])."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((K // 128, max(round_up(M, 4), 4)), dtype=torch.float32, device=x.device)
    fp8_quant_act_1x128(x, q, s, FP8_SCALE_POW2 if pow2 else FP8_SCALE_FP32_AMAX, stream)
    return q, s


def quant_weight(w: torch.Tensor, pow2: bool = False, stream=None):
    """Returns (q uint8 [N, K], s fp32 [N/128, K/128])."""
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    fp8_quant_weight_128x128(w, q, s, FP8_SCALE_POW2 if pow2 else FP8_SCALE_FP32_AMAX, stream)
    return q, s


def quant_act_t(x: torch.Tensor, pow2: bool = False, rowwise: bool = False, stream=None):
    """128x1 quantisation of x [M, K], transposed: returns (qt uint8 [K, Mp],
    st fp32 [Mp/128, round_up(K, 4)]) with Mp = M rounded up to 128 (the pad
    tokens are zeros), and with rowwise=True also (q, s) as quant_act(x)
    returns them, from the same pass."""
    M, K = x.shape
    Mp = round_up(M, 128)
    qt = torch.empty((K, Mp), dtype=torch.uint8, device=x.device)
    st = torch.empty((Mp // 128, max(round_up(K, 4), 4)), dtype=torch.float32, device=x.device)
    q = s = None
    if rowwise:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
        s = torch.empty((K // 128, max(round_up(M, 4), 4)), dtype=torch.float32, device=x.device)
    fp8_quant_act_128x1(x, qt, st, q, s, FP8_SCALE_POW2 if pow2 else FP8_SCALE_FP32_AMAX, stream)
    return (qt, st, q, s) if rowwise else (qt, st)


def quant_weight_t(w: torch.Tensor, pow2: bool = False, with_w: bool = False, stream=None):
    """W^T operand of the dgrad GEMM: returns (qt uint8 [K, N], st fp32
    [K/128, N/128]), and with with_w=True also (q, s) as quant_weight(w)."""
    N, K = w.shape
    qt = torch.empty((K, N), dtype=torch.uint8, device=w.device)
    st = torch.empty((K // 128, N // 128), dtype=torch.float32, device=w.device)
    q = s = None
    if with_w:
        q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
        s = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    fp8_quant_weight_128x128_t(w, qt, st, q, s, FP8_SCALE_POW2 if pow2 else FP8_SCALE_FP32_AMAX, stream)
    return (qt, st, q, s) if with_w else (qt, st)


def quant_tensor(x: torch.Tensor, pow2: bool = False, stream=None):
    """Per-tensor quantisation: returns (q uint8 [M, K], scale_amax fp32 [2])."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    sa = torch.empty(2, dtype=torch.float32, device=x.device)
    fp8_quant_per_tensor(x, q, sa, FP8_SCALE_POW2 if pow2 else FP8_SCALE_FP32_AMAX, stream)
    return q, sa


_ws: dict[int, torch.Tensor] = {}


def workspace_for(M: int, N: int, K: int, G: int, device) -> torch.Tensor | None:
    """A zero-initialised workspace of at least the needed size, kept per device."""
    need = fp8_gemm_workspace_size(M, N, K, G)
    if need == 0:
        return None
    dev = torch.device(device).index or 0
    ws = _ws.get(dev)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(round_up(need, 1 << 20), dtype=torch.uint8, device=device)
        _ws[dev] = ws
    return ws


def gemm(qa, sa, qb, sb, pow2: bool = False, path: str = "auto", out: torch.Tensor | None = None, stream=None):
    """C = block-scaled GEMM of quantised operands; allocates C (bf16 [M, N])
    and, for the split-K path, a zero-filled workspace kept per device."""
    M, K = qa.shape
    N = qb.shape[0]
    c = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=qa.device)
    flags = PATHS[path] | (FP8_GEMM_SCALES_POW2 if pow2 else 0)
    # The size query follows the automatic plan: for M <= 128 the split-K
    # skinny kernel, above it the large-M kernels' last-wave split (optional,
    # so a plan mismatch only costs that split).
    ws = workspace_for(M, N, K, 1, qa.device)
    fp8_blockscaled_gemm(qa, sa, qb, sb, c, flags, ws, stream)
    return c


def grouped_gemm(qa, sa, offsets, qb, sb, pow2: bool = False, path: str = "auto", out=None, stream=None):
    """Grouped (per-expert) block-scaled GEMM; allocates C (bf16 [M, N])."""
    M, K = qa.shape
    N = qb.shape[1]
    c = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=qa.device)
    flags = PATHS[path] | (FP8_GEMM_SCALES_POW2 if pow2 else 0)
    fp8_blockscaled_grouped_gemm(qa, sa, offsets, qb, sb, c, flags, None, stream)
    return c


def gemm_quant(qa, sa, qb, sb, pow2: bool = False, out_pow2: bool = False, with_c: bool = True, stream=None):
    """Block-scaled GEMM with the next layer's 1x128 quantisation fused in.
    Returns (c or None, qc, sc) with sc in the [N/128, round_up(M, 4)] layout
    of quant_act's scales."""
    M, K = qa.shape
    N = qb.shape[0]
    c = torch.empty((M, N), dtype=torch.bfloat16, device=qa.device) if with_c else None
    qc = torch.empty((M, N), dtype=torch.uint8, device=qa.device)
    sc = torch.empty((N // 128, round_up(M, 4)), dtype=torch.float32, device=qa.device)
    ws = workspace_for(M, N, K, 1, qa.device)
    fp8_blockscaled_gemm_quant(qa, sa, qb, sb, c, qc, sc, FP8_GEMM_SCALES_POW2 if pow2 else 0,
                               FP8_SCALE_POW2 if out_pow2 else FP8_SCALE_FP32_AMAX, ws, stream)
    return c, qc, sc


def wgrad(qt_dy, st_dy, qt_x, st_x, pow2: bool = False, path: str = "auto", out=None, stream=None):
    """dW [N, K] (bf16) = dY^T X from the transposed 128x1 operands
    (quant_act_t of dY [T, N] and of X [T, K])."""
    N, T = qt_dy.shape
    K = qt_x.shape[0]
    c = out if out is not None else torch.empty((N, K), dtype=torch.bfloat16, device=qt_dy.device)
    ws = workspace_for(N, K, T, 1, qt_dy.device)
    fp8_blockscaled_gemm_wgrad(qt_dy, st_dy, qt_x, st_x, c, PATHS[path] | (FP8_GEMM_SCALES_POW2 if pow2 else 0),
                               ws, stream)
    return c


def gemm_tensor(qa, sa, qb, sb, out=None, stream=None):
    """C = per-tensor-scaled GEMM; sa, sb the scale_amax tensors of quant_tensor
    (their element 0 is the scale)."""
    M, K = qa.shape
    N = qb.shape[0]
    c = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=qa.device)
    fp8_tensorscaled_gemm(qa, sa[:1], qb, sb[:1], c, 0, workspace_for(M, N, K, 1, qa.device), stream)
    return c


def decode_attention(q, sq, k_cache, sk, v_cache, sv, seq_lens, stream=None):
    """One FP8 decode-attention step; allocates the bf16 output and the
    split workspace.  sq, sk, sv: fp32 device tensors whose element 0 is the scale."""
    B, Hq, D = q.shape
    T = k_cache.shape[2]
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    need = fp8_decode_attention_workspace_size(B, Hq, T)
    ws = torch.empty(need, dtype=torch.uint8, device=q.device) if need else None
    fp8_decode_attention(q, sq[:1], k_cache, sk[:1], v_cache, sv[:1], seq_lens, out, ws, stream)
    return out


def quant_act_t_grouped(x: torch.Tensor, offsets: torch.Tensor, pow2: bool = False, stream=None):
    """Grouped 128x1 quantisation of expert-sorted x [T, K]: returns (qt uint8
    [K, 128 (ceil(T/128) + G)], st fp32 [ceil(T/128) + G, round_up(K, 4)])."""
    T, K = x.shape
    nb = (T + 127) // 128 + offsets.numel() - 1
    qt = torch.empty((K, 128 * nb), dtype=torch.uint8, device=x.device)
    st = torch.empty((nb, max(round_up(K, 4), 4)), dtype=torch.float32, device=x.device)
    fp8_quant_act_128x1_grouped(x, offsets, qt, st, FP8_SCALE_POW2 if pow2 else FP8_SCALE_FP32_AMAX, stream)
    return qt, st


def moe_wgrad(dy: torch.Tensor, x: torch.Tensor, offsets, pow2: bool = False, stream=None):
    """Weight gradients of a mixture-of-experts layer, dW_g = dY_g^T X_g for
    the expert-sorted token rows offsets[g] .. offsets[g+1]-1 (offsets: an
    int32 device tensor or a host sequence of G+1 ints).  Each expert's rows
    are quantised in 128x1 blocks of its own tokens (the last block padded
    with zeros) by one grouped quantiser launch per operand, and one grouped
    GEMM launch computes every expert's gradient.  Returns bf16 [G, N, K];
    experts without tokens get zeros."""
    if not isinstance(offsets, torch.Tensor):
        offsets = torch.tensor([int(v) for v in offsets], dtype=torch.int32)
    offsets = offsets.to(device=dy.device, dtype=torch.int32)
    G = offsets.numel() - 1
    T, N = dy.shape
    K = x.shape[1]
    qt_dy, st_dy = quant_act_t_grouped(dy, offsets, pow2, stream)
    qt_x, st_x = quant_act_t_grouped(x, offsets, pow2, stream)
    dw = torch.empty((G, N, K), dtype=torch.bfloat16, device=dy.device)
    fp8_blockscaled_grouped_gemm_wgrad(qt_dy, st_dy, qt_x, st_x, offsets, T, dw,
                                       FP8_GEMM_SCALES_POW2 if pow2 else 0, stream)
    return dw


def linear(x: torch.Tensor, w: torch.Tensor, pow2: bool = False, stream=None):
    """bf16 y = FP8 linear layer: quantise x (1x128) and w (128x128) in one
    launch, then the block-scaled GEMM.  Returns (y, (qa, sa), (qw, sw))."""
    M, K = x.shape
    N = w.shape[0]
    qa = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    sa = torch.empty((K // 128, max(round_up(M, 4), 4)), dtype=torch.float32, device=x.device)
    qw = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    fp8_quant_act_weight(x, qa, sa, w, qw, sw, FP8_SCALE_POW2 if pow2 else FP8_SCALE_FP32_AMAX, stream)
    return gemm(qa, sa, qw, sw, pow2, stream=stream), (qa, sa), (qw, sw)
