"""Per-kernel micro-benchmark of the library.

Runs one entry point on one shape, `--warmup` times untimed and `--iters`
times timed with CUDA events on the launching stream (L2 flushed before each
timed launch unless --no-flush; the call is replayed from a CUDA graph and all
iterations are enqueued before one synchronize, so host launch overhead does
not land inside the event pairs), and prints one JSON line with the mean time
and the achieved rate (algorithmic bytes or FLOPs).  Also the command used for
ncu captures of a single kernel.

  python -m fp8_block_scaled_05_gb300.kbench --kernel gemm --M 4096 --N 28672 --K 4096
  python -m fp8_block_scaled_05_gb300.kbench --kernel quant_act --M 4096 --K 14336
"""
from __future__ import annotations

import argparse
import json

import torch

from . import build as _build
from . import ops
from .timing import L2Flush


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--kernel", required=True,
                   choices=["quant_act", "quant_weight", "gemm", "grouped", "quant_act_t", "quant_weight_t", "wgrad",
                            "pt_gemm", "attention", "moe_wgrad", "quant_layer"])
    p.add_argument("--dual", action="store_true", help="quant_act_t / quant_weight_t: also the other layout")
    p.add_argument("--M", type=int, default=4096)
    p.add_argument("--N", type=int, default=4096)
    p.add_argument("--K", type=int, default=4096)
    p.add_argument("--G", type=int, default=128, help="experts (grouped)")
    p.add_argument("--moe", choices=["gate_up", "down"], default=None,
                   help="grouped, moe_wgrad: the Qwen3-30B-A3B expert shapes and Zipf(1.1) top-8 routing of "
                        "8192 tokens (overrides M, N, K, G)")
    p.add_argument("--pow2", action="store_true")
    p.add_argument("--path", default="auto", choices=list(ops.PATHS))
    p.add_argument("--iters", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--no-flush", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="launch through the Python wrapper every iteration")
    a = p.parse_args(argv)

    _build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    M, N, K = a.M, a.N, a.K
    mode = ops.FP8_SCALE_POW2 if a.pow2 else ops.FP8_SCALE_FP32_AMAX
    flush = None if a.no_flush else L2Flush(dev)

    if a.kernel == "quant_act":
        x = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
        q = torch.empty((M, K), dtype=torch.uint8, device=dev)
        s = torch.empty((K // 128, ops.round_up(M, 4)), dtype=torch.float32, device=dev)
        run = lambda: ops.fp8_quant_act_1x128(x, q, s, mode)  # noqa: E731
        work, unit = 3.0 * M * K + 4.0 * M * (K // 128), "GB/s"
    elif a.kernel == "quant_layer":
        # activations x [M, K] (1x128) and weights w [N, K] (128x128) in one launch
        x = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
        w = (torch.randn((N, K), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
        sa = torch.empty((K // 128, ops.round_up(M, 4)), dtype=torch.float32, device=dev)
        qw = torch.empty((N, K), dtype=torch.uint8, device=dev)
        sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev)
        run = lambda: ops.fp8_quant_act_weight(x, qa, sa, w, qw, sw, mode)  # noqa: E731
        work, unit = 3.0 * (M + N) * K + 4.0 * M * (K // 128) + 4.0 * (N // 128) * (K // 128), "GB/s"
    elif a.kernel == "quant_weight":
        w = (torch.randn((N, K), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        q = torch.empty((N, K), dtype=torch.uint8, device=dev)
        s = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev)
        run = lambda: ops.fp8_quant_weight_128x128(w, q, s, mode)  # noqa: E731
        work, unit = 3.0 * N * K + 4.0 * (N // 128) * (K // 128), "GB/s"
    elif a.kernel == "quant_act_t":
        # x [M, K] -> 128x1 codes transposed (+ 1x128 codes with --dual)
        x = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
        qt = torch.empty((K, M), dtype=torch.uint8, device=dev)
        st = torch.empty((M // 128, ops.round_up(K, 4)), dtype=torch.float32, device=dev)
        q = torch.empty((M, K), dtype=torch.uint8, device=dev) if a.dual else None
        s = torch.empty((K // 128, ops.round_up(M, 4)), dtype=torch.float32, device=dev) if a.dual else None
        run = lambda: ops.fp8_quant_act_128x1(x, qt, st, q, s, mode)  # noqa: E731
        work, unit = (4.0 if a.dual else 3.0) * M * K + (8.0 if a.dual else 4.0) * M * K / 128, "GB/s"
    elif a.kernel == "quant_weight_t":
        w = (torch.randn((N, K), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        qt = torch.empty((K, N), dtype=torch.uint8, device=dev)
        st = torch.empty((K // 128, N // 128), dtype=torch.float32, device=dev)
        q = torch.empty((N, K), dtype=torch.uint8, device=dev) if a.dual else None
        s = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev) if a.dual else None
        run = lambda: ops.fp8_quant_weight_128x128_t(w, qt, st, q, s, mode)  # noqa: E731
        work, unit = (4.0 if a.dual else 3.0) * N * K, "GB/s"
    elif a.kernel == "wgrad":
        # C [M, N] = A [M, K] B [N, K]^T with 1x128 scales on both (K = tokens)
        qa, sa = ops.quant_act(torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16), a.pow2)
        qb, sb = ops.quant_act(torch.randn((N, K), generator=g, device=dev).to(torch.bfloat16), a.pow2)
        c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        run = lambda: ops.wgrad(qa, sa, qb, sb, a.pow2, a.path, out=c)  # noqa: E731
        work, unit = 2.0 * M * N * K, "TFLOP/s"
    elif a.kernel == "pt_gemm":
        # per-tensor scaled GEMM (one scale per operand)
        qa, sa = ops.quant_tensor(torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16))
        qw, sw = ops.quant_tensor((torch.randn((N, K), generator=g, device=dev) * 0.02).to(torch.bfloat16))
        c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        run = lambda: ops.gemm_tensor(qa, sa, qw, sw, out=c)  # noqa: E731
        work, unit = 2.0 * M * N * K, "TFLOP/s"
    elif a.kernel == "attention":
        # decode attention over an FP8 KV cache: M sequences, N query heads
        # (N / 4 KV heads), K cached tokens each, D = 128
        B, Hq, T, D = M, N, K, 128
        Hkv = max(1, Hq // 4)
        kv = torch.randn((B * Hkv * T, D), generator=g, device=dev).to(torch.bfloat16)
        kc, ssk = ops.quant_tensor(kv)
        del kv
        vc = kc.flip(0).contiguous()
        qc, ssq = ops.quant_tensor(torch.randn((B * Hq, D), generator=g, device=dev).to(torch.bfloat16))
        lens = torch.full((B,), T, dtype=torch.int32, device=dev)
        kc4, vc4, qc3 = kc.view(B, Hkv, T, D), vc.view(B, Hkv, T, D), qc.view(B, Hq, D)
        run = lambda: ops.decode_attention(qc3, ssq, kc4, ssk, vc4, ssk, lens)  # noqa: E731
        work, unit = 2.0 * B * Hkv * T * D + 3.0 * B * Hq * D, "GB/s"
    elif a.kernel == "moe_wgrad":
        # grouped weight gradients dW_g [M, N] = dY_g^T X_g of the expert
        # projection (gate_up: M 1536, N 2048; down: M 2048, N 768) over the
        # Zipf-routed expert-sorted rows; operands from the grouped quantiser
        from . import inputs as I
        mc = I.moe_case(with_weights=False)
        G, T = len(mc.offsets) - 1, int(mc.offsets[-1])
        M, N = (1536, 2048) if (a.moe or "gate_up") == "gate_up" else (2048, 768)
        K = T
        offs = torch.from_numpy(mc.offsets).to(dev)
        dy = (torch.randn((T, M), generator=g, device=dev) * 1e-4).to(torch.bfloat16)
        x = torch.randn((T, N), generator=g, device=dev).to(torch.bfloat16)
        qg, sg = ops.quant_act_t_grouped(dy, offs, a.pow2)
        qx, sx = ops.quant_act_t_grouped(x, offs, a.pow2)
        del dy, x
        c = torch.empty((G, M, N), dtype=torch.bfloat16, device=dev)
        flags = ops.FP8_GEMM_SCALES_POW2 if a.pow2 else 0
        run = lambda: ops.fp8_blockscaled_grouped_gemm_wgrad(qg, sg, qx, sx, offs, T, c, flags)  # noqa: E731
        work, unit = 2.0 * M * N * K, "TFLOP/s"
    elif a.kernel == "gemm":
        qa, sa = ops.quant_act(torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16), a.pow2)
        qw, sw = ops.quant_weight((torch.randn((N, K), generator=g, device=dev) * 0.02).to(torch.bfloat16), a.pow2)
        c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        run = lambda: ops.gemm(qa, sa, qw, sw, a.pow2, a.path, out=c)  # noqa: E731
        work, unit = 2.0 * M * N * K, "TFLOP/s"
    else:
        G = a.G
        if a.moe:
            from . import inputs as I
            mc = I.moe_case(with_weights=False)
            G, M = len(mc.offsets) - 1, int(mc.offsets[-1])
            N, K = (1536, 2048) if a.moe == "gate_up" else (2048, 768)
            offs = torch.from_numpy(mc.offsets).to(dev)
        else:
            sizes = torch.full((G,), M // G, dtype=torch.int64)
            sizes[: M - int(sizes.sum())] += 1
            offs = torch.zeros(G + 1, dtype=torch.int32)
            offs[1:] = torch.cumsum(sizes, 0)
            offs = offs.to(dev)
        qa, sa = ops.quant_act(torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16), a.pow2)
        qw = torch.randint(0, 0x7E, (G, N, K), dtype=torch.uint8, device=dev, generator=g)
        sw = torch.rand((G, N // 128, K // 128), generator=g, device=dev) * 1e-3
        if a.pow2:
            sw = torch.exp2(torch.ceil(torch.log2(sw)))
        c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        run = lambda: ops.grouped_gemm(qa, sa, offs, qw, sw, a.pow2, a.path, out=c)  # noqa: E731
        work, unit = 2.0 * M * N * K, "TFLOP/s"

    for _ in range(max(a.warmup, 1)):
        run()
    torch.cuda.synchronize()
    timed = run
    if not a.no_graph:
        # The library call is captured once into a CUDA graph (its one-time
        # set-up already happened in the warm-up), so a timed iteration costs
        # the host one replay: the host stays ahead of the GPU and no launch
        # gap lands inside the event pair (the Python wrapper alone takes
        # longer than a decode-sized kernel).
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run()
        timed = graph.replay
        timed()
        torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.iters)]
    for e0, e1 in evs:
        if flush is not None:
            flush()
        e0.record()
        timed()
        e1.record()
    torch.cuda.synchronize()
    times = [e0.elapsed_time(e1) for e0, e1 in evs]
    st = ops.fp8_last_device_status()
    ms = sum(times) / len(times)
    rate = work / (ms / 1e3) / (1e9 if unit == "GB/s" else 1e12)
    plan = ops.fp8_gemm_plan(M, N, K, ops.PATHS[a.path]) if a.kernel == "gemm" else None
    print(json.dumps({"kernel": a.kernel, "M": M, "N": N, "K": K, "pow2": a.pow2, "path": a.path, "plan": plan,
                      "ms": ms, "min_ms": min(times), unit: rate, "status": st}))
    return 0 if st == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
