#!/usr/bin/env python
"""Benchmark of the block-scaled FP8 linear layer at Llama-3.1-8B shapes.

One step = the whole hot path over one batch: for each of the three linear
layers of a Llama-3.1-8B block at M = 4096 tokens (QKV K=4096 N=6144,
gate+up K=4096 N=28672, down K=14336 N=4096): 1x128 activation quantisation,
128x128 weight re-quantisation (weights change every optimizer step) and the
block-scaled FP8 GEMM, all in libfp8bs.so's kernels, fp32 amax/448 scales.

metric: quant+GEMM TFLOP/s = sum(2 M N K) / (t_quantA + t_quantW + t_gemm).

Timing: W untimed warm-up steps, then exactly K steps, each preceded (outside
its CUDA-event interval) by a 256 MB write that flushes the 129 MB L2 and
a 256 MB read that leaves it holding clean lines;
barrier + synchronize around the timed region; max over ranks.  N > 1 runs
independent replicas (the path has no exchange step): value is the work of
all ranks divided by the slowest rank's time.

--impl reference times the CPU oracle (oracle/) on a bounded sample of the
same workload instead; under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-scaled FP8 quant+GEMM TFLOP/s at Llama-8B shapes; % FP8 peak / HBM"
UNIT = "TFLOP/s"
WORKLOAD = "llama3.1-8b linear layers, M=4096 tokens: qkv(K4096,N6144) gate_up(K4096,N28672) down(K14336,N4096)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0          # nominal dense ratio (4.5 / 2.25 PFLOP/s)
L2_FLUSH_BYTES = 256 << 20
# bounded oracle sample per layer: rows of A and rows of W
CPU_SAMPLE_ROWS_A = 128
CPU_SAMPLE_ROWS_W = 512


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-pow2", action="store_true", help="skip the power-of-two scale-mode measurement")
    p.add_argument("--no-fused", action="store_true", help="skip the fused GEMM + quantisation measurement")
    p.add_argument("--no-training", action="store_true", help="skip the training-step (forward + backward) "
                                                                "measurement")
    p.add_argument("--no-per-tensor", action="store_true", help="skip the per-tensor scaling measurement")
    p.add_argument("--no-attention", action="store_true", help="skip the FP8 KV-cache decode attention measurement")
    p.add_argument("--no-qwen", action="store_true", help="skip the Qwen3-8B prefill (M = 16384) measurement")
    p.add_argument("--no-decode", action="store_true", help="skip the decode-sized (M <= 256) measurement")
    p.add_argument("--no-moe", action="store_true", help="skip the Qwen3-30B-A3B grouped MoE measurement")
    a = p.parse_args(argv)
    a.warmup = max(a.warmup, 3) if a.impl == "ours" else max(a.warmup, 0)
    return a


# ------------------------------------------------------------------ peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        hbm = float(d.get("hbm_gbs") or 0) or None
        bf16 = float(d.get("bf16_tflops") or 0) or None
        bf16_s = float(d.get("bf16_tflops_sustained") or 0) or None
        if hbm and bf16:
            return {"hbm_gbs": hbm, "bf16_tflops": bf16, "bf16_tflops_sustained": bf16_s or bf16,
                    "source": "measured"}
    except (OSError, ValueError, TypeError):
        pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ dist
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist


def reduce_max(value: float, world: int, device) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ oracle sample
def oracle_sample(layers, rows_a=CPU_SAMPLE_ROWS_A, rows_w=CPU_SAMPLE_ROWS_W, parts=None):
    """Time the CPU oracle on a bounded sample of each layer (first rows_a rows
    of A, first rows_w rows of W): quant A, quant W, GEMM.  Returns
    (flops of the sample, seconds); with a dict `parts`, also fills in each
    step's own rate (quantisers in GB/s of 3 bytes per element, the GEMM in
    GFLOP/s) over the sample."""
    import numpy as np
    import oracle.fp8_oracle as O
    flops = 0.0
    tq = [0.0, 0.0, 0.0]
    nq = [0.0, 0.0]
    t0 = time.perf_counter()
    for a, w in layers:
        xa = a[:rows_a].float().numpy()
        xw = w[:rows_w].float().numpy()
        t1 = time.perf_counter()
        qa, sa = O.quant_act_1x128(xa)
        t2 = time.perf_counter()
        qw, sw = O.quant_weight_128x128(xw)
        t3 = time.perf_counter()
        c = O.gemm_ref(qa, sa, qw, sw)
        t4 = time.perf_counter()
        assert np.isfinite(c).all()
        tq[0] += t2 - t1
        tq[1] += t3 - t2
        tq[2] += t4 - t3
        nq[0] += xa.size
        nq[1] += xw.size
        flops += 2.0 * xa.shape[0] * xw.shape[0] * xa.shape[1]
    secs = time.perf_counter() - t0
    if parts is not None:
        parts["quant_act"] = {"GB/s": 3.0 * nq[0] / tq[0] / 1e9, "seconds": tq[0]}
        parts["quant_weight"] = {"GB/s": 3.0 * nq[1] / tq[1] / 1e9, "seconds": tq[1]}
        parts["gemm"] = {"GFLOP/s": flops / tq[2] / 1e9, "seconds": tq[2]}
    return flops, secs


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:  # noqa: BLE001
        pass
    return len(os.sched_getaffinity(0))


def sample_desc():
    return (f"oracle (numpy, fp64 GEMM) on the first {CPU_SAMPLE_ROWS_A} rows of A and first "
            f"{CPU_SAMPLE_ROWS_W} rows of W of each of the 3 layers (quant A + quant W + GEMM); "
            f"value = sample FLOPs / sample time")


# ------------------------------------------------------------------ reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return 0
    from fp8_block_scaled_05_gb300 import inputs as I
    layers = [(c.a, c.w) for c in I.llama8b_layers(args.seed)]
    for _ in range(args.warmup):
        oracle_sample(layers)
    flops = secs = 0.0
    for _ in range(args.steps):
        f, s = oracle_sample(layers)
        flops += f
        secs += s
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample_desc()},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                         "sample": sample_desc()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
def traffic_for(kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it
    was taken on the current sources; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        from fp8_block_scaled_05_gb300 import build as B
        if d.get("source_stamp") != B.source_stamp():
            return None
        return d.get("kernels", {}).get(kernel)
    except (OSError, ValueError, AttributeError):
        return None


def run_ours(args, world, rank, local):
    import torch
    from fp8_block_scaled_05_gb300 import build as B
    from fp8_block_scaled_05_gb300 import inputs as I
    from fp8_block_scaled_05_gb300 import ops

    B.build()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    stream = torch.cuda.Stream(device=dev)
    cases = I.llama8b_layers(args.seed)

    layers = []
    for c in cases:
        M, N, K = c.shape
        a = c.a.to(dev)
        w = c.w.to(dev)
        L = dict(name=c.name.split(".")[1], M=M, N=N, K=K, a=a, w=w,
                 qa=torch.empty((M, K), dtype=torch.uint8, device=dev),
                 sa=torch.empty((K // 128, ops.round_up(M, 4)), dtype=torch.float32, device=dev),
                 qw=torch.empty((N, K), dtype=torch.uint8, device=dev),
                 sw=torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev),
                 c=torch.empty((M, N), dtype=torch.bfloat16, device=dev),
                 ws=ops.workspace_for(M, N, K, 1, dev))
        layers.append(L)
    flops_step = sum(2.0 * L["M"] * L["N"] * L["K"] for L in layers)
    from fp8_block_scaled_05_gb300.timing import L2Flush
    flush = L2Flush(dev, L2_FLUSH_BYTES)
    launches_per_step = 2 * len(layers)

    def step(events=None, pow2=False):
        # per layer: the activation and weight quantisers in one launch, then the GEMM
        mode = ops.FP8_SCALE_POW2 if pow2 else ops.FP8_SCALE_FP32_AMAX
        flags = ops.FP8_GEMM_SCALES_POW2 if pow2 else 0
        for i, L in enumerate(layers):
            if events is not None:
                events[2 * i].record(stream)
            ops.fp8_quant_act_weight(L["a"], L["qa"], L["sa"], L["w"], L["qw"], L["sw"], mode, stream)
            if events is not None:
                events[2 * i + 1].record(stream)
            ops.fp8_blockscaled_gemm(L["qa"], L["sa"], L["qw"], L["sw"], L["c"], flags, L["ws"], stream)
        if events is not None:
            events[2 * len(layers)].record(stream)

    def timed(pow2, steps):
        """Runs `steps` flushed steps; returns (per-step ms, per-kernel mean ms)."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(layers) + 1)] for _ in range(steps)]
        with torch.cuda.stream(stream):
            for k in range(steps):
                flush()
                step(evs[k], pow2)
        torch.cuda.synchronize(dev)
        step_ms = [evs[k][0].elapsed_time(evs[k][-1]) for k in range(steps)]
        kern = {}
        for i, L in enumerate(layers):
            for j, kname in enumerate(("quant", "gemm")):
                ms = [evs[k][2 * i + j].elapsed_time(evs[k][2 * i + j + 1]) for k in range(steps)]
                kern[f"{L['name']}.{kname}"] = sum(ms) / len(ms)
        return step_ms, kern

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush()
            step()
    torch.cuda.synchronize(dev)
    st = ops.fp8_last_device_status(stream)
    if st != 0:
        raise SystemExit(f"device status after warm-up: {ops.status_string(st)}")

    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    step_ms, kern = timed(False, args.steps)
    clk = clocks.stop()
    barrier(world)
    total_ms = reduce_max(sum(step_ms), world, dev)
    value = flops_step * args.steps * world / (total_ms / 1e3) / 1e12

    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    # dominant kernel: the GEMM with the largest time share
    gemms = {L["name"]: (kern[f"{L['name']}.gemm"], 2.0 * L["M"] * L["N"] * L["K"]) for L in layers}
    dom = max(gemms, key=lambda n: gemms[n][0])
    dom_ms, dom_flops = gemms[dom]
    achieved = dom_flops / (dom_ms / 1e3) / 1e12
    traffic = traffic_for(f"gemm.{dom}")
    kernels_out = {}
    qbytes = {}
    for L in layers:
        n = L["name"]
        qa_bytes = 2 * L["M"] * L["K"] + L["M"] * L["K"] + 4 * L["M"] * L["K"] // 128
        qw_bytes = 2 * L["N"] * L["K"] + L["N"] * L["K"] + 4 * (L["N"] // 128) * (L["K"] // 128)
        qbytes[n] = (qa_bytes, qw_bytes)
        q_ms = kern[f"{n}.quant"]
        kernels_out[f"{n}.quant"] = {"what": "1x128 activations and 128x128 weights in one launch",
                                     "ms": q_ms, "GB/s": (qa_bytes + qw_bytes) / q_ms / 1e6,
                                     "frac_hbm": (qa_bytes + qw_bytes) / q_ms / 1e6 / peaks["hbm_gbs"]}
        gf = 2.0 * L["M"] * L["N"] * L["K"]
        kernels_out[f"{n}.gemm"] = {"ms": kern[f"{n}.gemm"], "TFLOP/s": gf / kern[f"{n}.gemm"] / 1e9,
                                    "frac_fp8": gf / kern[f"{n}.gemm"] / 1e9 / fp8_peak}
    gemm_ms = sum(kern[f"{L['name']}.gemm"] for L in layers)

    # each quantiser alone (one launch each), for the per-kernel rooflines
    qcalls = []
    for L in layers:
        qcalls += [lambda L=L: ops.fp8_quant_act_1x128(L["a"], L["qa"], L["sa"], 0, stream),
                   lambda L=L: ops.fp8_quant_weight_128x128(L["w"], L["qw"], L["sw"], 0, stream)]
    qper, _ = time_calls(args, stream, dev, flush, qcalls)
    quantisers = {"what": "the two quantisers of each layer launched on their own (fp32 scales), flushed L2"}
    for i, L in enumerate(layers):
        n = L["name"]
        for j, (kn, nbytes) in enumerate(zip(("quant_act", "quant_weight"), qbytes[n])):
            ms = qper[2 * i + j]
            quantisers[f"{n}.{kn}"] = {"ms": ms, "GB/s": nbytes / ms / 1e6,
                                       "frac_hbm": nbytes / ms / 1e6 / peaks["hbm_gbs"]}

    # ---------------- end to end: pinned host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        host = [(L["a"].cpu().pin_memory(), L["w"].cpu().pin_memory(),
                 torch.empty((L["M"], L["N"]), dtype=torch.bfloat16).pin_memory()) for L in layers]
        h2d = sum(a.numel() * 2 + w.numel() * 2 for a, w, _ in host)
        d2h = sum(c.numel() * 2 for _, _, c in host)
        e2e_steps = max(3, args.steps // 4)
        # Three streams: host->device copies, the library's kernels, and
        # device->host copies, ordered per layer by events, so that one
        # layer's transfers overlap another layer's kernels.  Every step still
        # copies its inputs in from pinned host memory and its results out.
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        nl = len(layers)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        prev_done = [None] * nl     # kernels of layer i (previous step) finished reading a_i, w_i
        prev_out = [None] * nl      # previous step's result of layer i copied out

        def e2e_step():
            for i, (L, (ah, wh, ch)) in enumerate(zip(layers, host)):
                if prev_done[i] is not None:
                    s_in.wait_event(prev_done[i])
                with torch.cuda.stream(s_in):
                    L["a"].copy_(ah, non_blocking=True)
                    L["w"].copy_(wh, non_blocking=True)
                    e_in = ev()
                    e_in.record(s_in)
                stream.wait_event(e_in)
                if prev_out[i] is not None:
                    stream.wait_event(prev_out[i])
                ops.fp8_quant_act_weight(L["a"], L["qa"], L["sa"], L["w"], L["qw"], L["sw"], 0, stream)
                ops.fp8_blockscaled_gemm(L["qa"], L["sa"], L["qw"], L["sw"], L["c"], 0, L["ws"], stream)
                e_k = ev()
                e_k.record(stream)
                prev_done[i] = e_k
                s_out.wait_event(e_k)
                with torch.cuda.stream(s_out):
                    ch.copy_(L["c"], non_blocking=True)
                    e_o = ev()
                    e_o.record(s_out)
                prev_out[i] = e_o

        e2e_step()
        torch.cuda.synchronize(dev)
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        stream.wait_event(e0)
        s_out.wait_event(e0)
        for _ in range(e2e_steps):
            e2e_step()
        stream.wait_event(prev_out[-1])
        for e in prev_out:
            stream.wait_event(e)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = reduce_max(e0.elapsed_time(e1), world, dev)
        e2e = {"value": flops_step * e2e_steps * world / (e2e_ms / 1e3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "ms_per_step": e2e_ms / e2e_steps,
               "pipelining": "host->device copies, kernels and device->host copies on three streams, "
                             "ordered per layer by events"}

    # ---------------- the optional power-of-two scale mode on the same workload:
    # quantisers in pow2 mode, GEMM with the pow2 promise (the MX kernel).  A
    # separate timed region, reported beside the headline.
    pow2 = None
    if not args.no_pow2:
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                flush()
                step(None, True)
        torch.cuda.synchronize(dev)
        barrier(world)
        p_ms, p_kern = timed(True, args.steps)
        barrier(world)
        p_total = reduce_max(sum(p_ms), world, dev)
        p_gemm_ms = sum(p_kern[f"{L['name']}.gemm"] for L in layers)
        plan = ops.fp8_gemm_plan(layers[0]["M"], layers[0]["N"], layers[0]["K"], ops.FP8_GEMM_SCALES_POW2)[0]
        pow2 = {"scale": "pow2 (2^ceil(log2(amax/448)))", "gemm_path": {v: k for k, v in ops.PATHS.items()}[plan],
                "value": flops_step * args.steps * world / (p_total / 1e3) / 1e12, "unit": UNIT,
                "ms_per_step": p_total / args.steps,
                "gemm_only_tflops": flops_step / (p_gemm_ms / 1e3) / 1e12,
                "gemm_frac_fp8": flops_step / (p_gemm_ms / 1e3) / 1e12 / fp8_peak,
                "kernels_ms": p_kern, "gpu_launches": launches_per_step * args.steps}

    # ---------------- the GEMM with the next layer's quantisation fused into its
    # epilogue, against the GEMM followed by the activation quantiser of its
    # output (same inputs; each variant timed per layer over flushed steps).
    fused = None
    if not args.no_fused:
        fl = {}
        for L, pw in [(L, pw) for pw in (False, True) for L in layers]:
            M, N = L["M"], L["N"]
            qc = torch.empty((M, N), dtype=torch.uint8, device=dev)
            sc = torch.empty((N // 128, ops.round_up(M, 4)), dtype=torch.float32, device=dev)
            mode = ops.FP8_SCALE_POW2 if pw else ops.FP8_SCALE_FP32_AMAX
            flags = ops.FP8_GEMM_SCALES_POW2 if pw else 0
            # operands in the matching scale mode
            with torch.cuda.stream(stream):
                ops.fp8_quant_act_1x128(L["a"], L["qa"], L["sa"], mode, stream)
                ops.fp8_quant_weight_128x128(L["w"], L["qw"], L["sw"], mode, stream)

            def unfused():
                ops.fp8_blockscaled_gemm(L["qa"], L["sa"], L["qw"], L["sw"], L["c"], flags, L["ws"], stream)
                ops.fp8_quant_act_1x128(L["c"], qc, sc, mode, stream)

            def fused_c():
                ops.fp8_blockscaled_gemm_quant(L["qa"], L["sa"], L["qw"], L["sw"], L["c"], qc, sc, flags, mode,
                                               L["ws"], stream)

            def fused_noc():
                ops.fp8_blockscaled_gemm_quant(L["qa"], L["sa"], L["qw"], L["sw"], None, qc, sc, flags, mode,
                                               L["ws"], stream)

            res = {"gemm_kernel": "mx" if pw else "promote"}
            for name, fn in (("unfused_ms", unfused), ("fused_ms", fused_c), ("fused_no_c_ms", fused_noc)):
                with torch.cuda.stream(stream):
                    for _ in range(args.warmup):
                        flush()
                        fn()
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(args.steps)]
                with torch.cuda.stream(stream):
                    for e0, e1 in evs:
                        flush()
                        e0.record(stream)
                        fn()
                        e1.record(stream)
                torch.cuda.synchronize(dev)
                res[name] = sum(e0.elapsed_time(e1) for e0, e1 in evs) / len(evs)
            res["speedup"] = res["unfused_ms"] / res["fused_ms"]
            res["speedup_no_c"] = res["unfused_ms"] / res["fused_no_c_ms"]
            fl[L["name"] + (".pow2" if pw else ".fp32")] = res
        fused = {"what": "GEMM then 1x128 quantisation of its bf16 output (unfused) vs the quantisation fused "
                         "into the GEMM epilogue, with and without writing the bf16 output",
                 "layers": fl}

    # ---------------- the same step with per-tensor dynamic scaling: one amax
    # per tensor (two passes: reduction, then cast) and the GEMM with one scale
    # per operand (MX kernel, unit scale factors, scale product in the epilogue).
    per_tensor = None
    if not args.no_per_tensor:
        per_tensor = per_tensor_measure(args, layers, ops, stream, dev, flush, flops_step, fp8_peak)

    # ---------------- one decode step of attention over an FP8 KV cache
    # ---------------- the other workloads of the layer: Qwen3-8B long-rollout
    # prefill (M = 16384, both scale modes), decode-sized GEMMs (M <= 256,
    # weight-stream bound) and the Qwen3-30B-A3B grouped expert GEMMs.
    qwen = None
    if not args.no_qwen:
        qwen = qwen_measure(args, ops, stream, dev, flush, fp8_peak)
    decode = None
    if not args.no_decode:
        decode = decode_measure(args, ops, stream, dev, flush, peaks["hbm_gbs"])
    moe = None
    if not args.no_moe:
        moe = moe_measure(args, ops, stream, dev, flush, fp8_peak, peaks["hbm_gbs"])

    attention = None
    if not args.no_attention:
        attention = attention_measure(args, ops, stream, dev, flush, peaks["hbm_gbs"])

    # ---------------- a training step of each layer: forward y = x W^T and the
    # backward GEMMs dX = dY W, dW = dY^T X, every operand from the dual-layout
    # quantisers (x, W and dY are each read once for both of their layouts).
    training = None
    if not args.no_training:
        training = train_measure(args, layers, ops, stream, dev, flush, fp8_peak, peaks["hbm_gbs"])

    st = ops.fp8_last_device_status(stream)
    if st != 0:
        raise SystemExit(f"device status after the timed region: {ops.status_string(st)}")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        layers_cpu = [(c.a, c.w) for c in cases]
        parts = {}
        f, s = oracle_sample(layers_cpu, parts=parts)
        cpu = {"value": f / s / 1e12, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": sample_desc(), "seconds": s, "per_step": parts}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e4m3 -> fp32 accumulate, bf16 out",
            "data": "synthetic (seeded numpy PCG64: A ~ N(0,1) with 1% outlier channels x30, W ~ N(0,0.02))",
            "config": {"workload": WORKLOAD, "M": 4096, "scale": "fp32 amax/448",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "flushed before every timed step (256 MB write, then a 256 MB read of a second buffer so the "
                             "lines left are clean; outside the step's events)"},
            "roofline": {"bound": "tensor", "kernel": f"gemm.{dom}", "achieved": achieved, "peak": fp8_peak,
                         "unit": "TFLOP/s", "frac": achieved / fp8_peak, "traffic": traffic,
                         "peak_source": f"{peaks['source']}: bf16 {peaks['bf16_tflops']} TFLOP/s x {FP8_OVER_BF16} "
                                        f"(fp8/bf16 nominal ratio)",
                         "hbm_peak_gbs": peaks["hbm_gbs"]},
            "gemm_only_tflops": sum(g[1] for g in gemms.values()) / (gemm_ms / 1e3) / 1e12,
            "kernels": kernels_out,
            "quantisers": quantisers,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "pow2": pow2,
            "fused_quant": fused,
            "training": training,
            "per_tensor": per_tensor,
            "attention": attention,
            "qwen_prefill": qwen,
            "decode": decode,
            "moe": moe,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    return 0


def per_tensor_measure(args, layers, ops, stream, dev, flush, flops_step, fp8_peak):
    """The bench step with per-tensor scaling, timed per call with CUDA events
    over flushed steps (same inputs and shapes as the block-scaled step)."""
    import torch

    bufs = [dict(sa=torch.empty(2, dtype=torch.float32, device=dev), sw=torch.empty(2, dtype=torch.float32, device=dev))
            for _ in layers]
    names = ("quant_act", "quant_weight", "gemm")

    def pstep(evs):
        for i, (L, B) in enumerate(zip(layers, bufs)):
            calls = (lambda: ops.fp8_quant_per_tensor(L["a"], L["qa"], B["sa"], 0, stream),
                     lambda: ops.fp8_quant_per_tensor(L["w"], L["qw"], B["sw"], 0, stream),
                     lambda: ops.fp8_tensorscaled_gemm(L["qa"], B["sa"][:1], L["qw"], B["sw"][:1], L["c"], 0, L["ws"],
                                                       stream))
            for j, call in enumerate(calls):
                if evs is not None:
                    evs[3 * i + j].record(stream)
                call()
        if evs is not None:
            evs[3 * len(layers)].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush()
            pstep(None)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3 * len(layers) + 1)] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            flush()
            pstep(evs[k])
    torch.cuda.synchronize(dev)
    total = sum(evs[k][0].elapsed_time(evs[k][-1]) for k in range(args.steps))
    kern, gemm_ms = {}, 0.0
    for i, L in enumerate(layers):
        for j, kn in enumerate(names):
            ms = sum(evs[k][3 * i + j].elapsed_time(evs[k][3 * i + j + 1]) for k in range(args.steps)) / args.steps
            kern[f"{L['name']}.{kn}"] = ms
            if kn == "gemm":
                gemm_ms += ms
    return {"scale": "one fp32 amax/448 per tensor (two passes: amax reduction, then cast)",
            "gemm_path": "mx (unit scale factors, scale product in the epilogue)",
            "value": flops_step * args.steps / (total / 1e3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": total / args.steps, "gemm_only_tflops": flops_step / (gemm_ms / 1e3) / 1e12,
            "gemm_frac_fp8": flops_step / (gemm_ms / 1e3) / 1e12 / fp8_peak, "kernels_ms": kern,
            "gpu_launches": 5 * len(layers) * args.steps}


def time_calls(args, stream, dev, flush, calls, graph=False):
    """Mean CUDA-event time (ms) of each callable in `calls` (a list of
    zero-argument functions run back to back on `stream`), over args.steps
    flushed steps after args.warmup untimed ones; returns (per-call ms,
    whole-sequence ms).  With graph=True the sequence is captured once into a
    CUDA graph and each call replayed from its own graph, so that host launch
    overhead does not land inside the event pairs of short kernels."""
    import torch

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush()
            for f in calls:
                f()
    torch.cuda.synchronize(dev)
    runs = calls
    if graph:
        runs = []
        for f in calls:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                f()
            runs.append(g.replay)
        with torch.cuda.stream(stream):
            for r in runs:
                r()
        torch.cuda.synchronize(dev)
    n = len(runs)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            flush()
            for i, r in enumerate(runs):
                evs[k][i].record(stream)
                r()
            evs[k][n].record(stream)
    torch.cuda.synchronize(dev)
    per = [sum(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps)) / args.steps for i in range(n)]
    total = sum(evs[k][0].elapsed_time(evs[k][n]) for k in range(args.steps)) / args.steps
    return per, total


def qwen_measure(args, ops, stream, dev, flush, fp8_peak):
    """Qwen3-8B-shaped long-rollout prefill, M = 16384 tokens (Student-t nu = 4
    activations, seeded host draws; W ~ N(0, 0.02)): per layer the 1x128
    activation quantiser, the 128x128 weight quantiser and the GEMM, timed per
    call over flushed steps, in both scale modes (fp32 scales: promote
    kernel; power-of-two scales: MX kernel)."""
    import torch

    from fp8_block_scaled_05_gb300 import inputs as I

    out = {"workload": "qwen3-8b prefill, M=16384: gate_up(K4096,N24576) down(K12288,N4096) o_proj(K4096,N4096)",
           "inputs": "A ~ Student-t(nu=4), W ~ N(0,0.02), seeded PCG64", "modes": {}}
    layers = []
    for case in I.qwen_prefill_layers(args.seed):
        M, N, K = case.shape
        layers.append(dict(name=case.name.split(".")[1], M=M, N=N, K=K, a=case.a.to(dev), w=case.w.to(dev),
                           qa=torch.empty((M, K), dtype=torch.uint8, device=dev),
                           sa=torch.empty((K // 128, ops.round_up(M, 4)), dtype=torch.float32, device=dev),
                           qw=torch.empty((N, K), dtype=torch.uint8, device=dev),
                           sw=torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev),
                           c=torch.empty((M, N), dtype=torch.bfloat16, device=dev),
                           ws=ops.workspace_for(M, N, K, 1, dev)))
    flops = sum(2.0 * L["M"] * L["N"] * L["K"] for L in layers)
    for pow2 in (False, True):
        mode = ops.FP8_SCALE_POW2 if pow2 else ops.FP8_SCALE_FP32_AMAX
        flags = ops.FP8_GEMM_SCALES_POW2 if pow2 else 0
        calls = []
        for L in layers:
            calls += [lambda L=L: ops.fp8_quant_act_weight(L["a"], L["qa"], L["sa"], L["w"], L["qw"], L["sw"], mode,
                                                           stream),
                      lambda L=L: ops.fp8_blockscaled_gemm(L["qa"], L["sa"], L["qw"], L["sw"], L["c"], flags,
                                                           L["ws"], stream)]
        per, total = time_calls(args, stream, dev, flush, calls)
        rows, gemm_ms = {}, 0.0
        for i, L in enumerate(layers):
            q_ms, g_ms = per[2 * i:2 * i + 2]
            gf = 2.0 * L["M"] * L["N"] * L["K"]
            gemm_ms += g_ms
            rows[L["name"]] = {"quant_ms": q_ms, "gemm_ms": g_ms,
                               "quant_gemm_tflops": gf / ((q_ms + g_ms) / 1e3) / 1e12,
                               "gemm_tflops": gf / (g_ms / 1e3) / 1e12,
                               "gemm_frac_fp8": gf / (g_ms / 1e3) / 1e12 / fp8_peak}
        out["modes"]["pow2" if pow2 else "fp32"] = {
            "gemm_kernel": "mx" if pow2 else "promote", "ms_per_step": total,
            "quant_gemm_tflops": flops / (total / 1e3) / 1e12, "gemm_only_tflops": flops / (gemm_ms / 1e3) / 1e12,
            "gemm_frac_fp8": flops / (gemm_ms / 1e3) / 1e12 / fp8_peak, "layers": rows,
            "gpu_launches": 2 * len(layers) * args.steps}
    return out


def decode_measure(args, ops, stream, dev, flush, hbm_peak):
    """Decode-sized layers: M in {1, 8, 64, 256} tokens at (K, N) = (4096,
    6144) and (14336, 4096), weights pre-quantised 128x128 (fp32 scales).  A
    decode step is the 1x128 quantiser of the bf16 activations and the GEMM on
    the automatic path (the skinny kernel up to 128 tokens, the promote kernel
    with every tile split along K above); each is replayed from a CUDA graph
    with the L2 flushed before every step.  Algorithmic bytes of the step: N K (weight codes) + 4 N K / 16384
    (weight scales) + 2 M K (bf16 activations) + 2 M N (bf16 output); of the
    GEMM alone the activations count as M K codes + 4 M K / 128 scales."""
    import torch

    from fp8_block_scaled_05_gb300 import inputs as I

    out = {"what": "quant_act (bf16 A -> E4M3 1x128) + GEMM (automatic path) on pre-quantised weights, "
                   "CUDA-graph replays, L2 flushed before each step", "points": {}}
    path_name = {v: k for k, v in ops.PATHS.items()}
    fracs = []
    for K, N in I.DECODE_SHAPES:
        w = I.decode_case(1, K, N, args.seed).w.to(dev)
        qw, sw = ops.quant_weight(w)
        del w
        for M in I.DECODE_TOKENS:
            a = I.decode_case(M, K, N, args.seed).a.to(dev)
            qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
            sa = torch.empty((K // 128, max(ops.round_up(M, 4), 4)), dtype=torch.float32, device=dev)
            c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = ops.workspace_for(M, N, K, 1, dev)

            def step():
                ops.fp8_quant_act_1x128(a, qa, sa, 0, stream)
                ops.fp8_blockscaled_gemm(qa, sa, qw, sw, c, 0, ws, stream)

            def gemm_only():
                ops.fp8_blockscaled_gemm(qa, sa, qw, sw, c, 0, ws, stream)

            (step_ms,), _ = time_calls(args, stream, dev, flush, [step], graph=True)
            (gemm_ms,), _ = time_calls(args, stream, dev, flush, [gemm_only], graph=True)
            wbytes = N * K + 4.0 * N * K / 16384
            step_bytes = wbytes + 2.0 * M * K + 2.0 * M * N
            gemm_bytes = wbytes + M * K + 4.0 * M * K / 128 + 2.0 * M * N
            path, ctas = ops.fp8_gemm_plan(M, N, K)
            pt = {"step_us": step_ms * 1e3, "step_GB/s": step_bytes / (step_ms / 1e3) / 1e9,
                  "step_frac_hbm": step_bytes / (step_ms / 1e3) / 1e9 / hbm_peak,
                  "gemm_us": gemm_ms * 1e3, "gemm_GB/s": gemm_bytes / (gemm_ms / 1e3) / 1e9,
                  "gemm_frac_hbm": gemm_bytes / (gemm_ms / 1e3) / 1e9 / hbm_peak,
                  "gemm_tflops": 2.0 * M * N * K / (gemm_ms / 1e3) / 1e12, "path": path_name.get(path, path),
                  "skinny_ctas": ctas if path == ops.FP8_GEMM_PATH_SKINNY else None}
            fracs.append(pt["step_frac_hbm"])
            out["points"][f"M{M}.K{K}.N{N}"] = pt
    out["min_step_frac_hbm"] = min(fracs)
    out["gpu_launches"] = 3 * len(fracs) * args.steps
    return out


def moe_measure(args, ops, stream, dev, flush, fp8_peak, hbm_peak):
    """Qwen3-30B-A3B-shaped mixture-of-experts layer: 8192 tokens, top-8 of 128
    experts with Zipf(1.1) popularity (seeded Gumbel-top-8), rows sorted by
    expert (65536 rows); expert gate+up (K 2048, N 1536) and down (K 768,
    N 2048).  Per projection: the 1x128 quantiser of the expert-sorted
    activations and the 128x128 quantiser of all experts' weights in one
    launch (the weights as the [G N, K] view; no tile straddles two experts
    since N % 128 == 0), then the grouped GEMM with device-side offsets, in
    both scale modes.  FLOPs
    are 2 sum(M_e) N K; the weight stream is G N K code bytes."""
    import numpy as np
    import torch

    from fp8_block_scaled_05_gb300 import inputs as I

    m = I.moe_case(args.seed)
    G = m.w_gate_up.shape[0]
    offs = torch.from_numpy(m.offsets).to(dev)
    projs = []
    for name, a, w in (("gate_up", m.a_gate_up, m.w_gate_up), ("down", m.a_down, m.w_down)):
        Mt, K = a.shape
        N = w.shape[1]
        projs.append(dict(name=name, M=Mt, N=N, K=K, a=a.to(dev), w=w.to(dev).view(G * N, K),
                          qa=torch.empty((Mt, K), dtype=torch.uint8, device=dev),
                          sa=torch.empty((K // 128, ops.round_up(Mt, 4)), dtype=torch.float32, device=dev),
                          qw=torch.empty((G, N, K), dtype=torch.uint8, device=dev),
                          sw=torch.empty((G, N // 128, K // 128), dtype=torch.float32, device=dev),
                          c=torch.empty((Mt, N), dtype=torch.bfloat16, device=dev)))
    sizes = m.offsets[1:] - m.offsets[:-1]
    out = {"workload": "qwen3-30b-a3b MoE: 8192 tokens, 128 experts, top-8, Zipf(1.1) routing; "
                       "gate_up (K2048,N1536), down (K768,N2048) per expert",
           "rows_per_expert": {"min": int(sizes.min()), "median": float(np.median(sizes)), "max": int(sizes.max())},
           "modes": {}}
    for pow2 in (False, True):
        mode = ops.FP8_SCALE_POW2 if pow2 else ops.FP8_SCALE_FP32_AMAX
        flags = ops.FP8_GEMM_SCALES_POW2 if pow2 else 0
        calls = []
        for P in projs:
            calls += [lambda P=P: ops.fp8_quant_act_weight(P["a"], P["qa"], P["sa"], P["w"], P["qw"].view(-1, P["K"]),
                                                           P["sw"].view(-1, P["K"] // 128), mode, stream),
                      lambda P=P: ops.fp8_blockscaled_grouped_gemm(P["qa"], P["sa"], offs, P["qw"], P["sw"], P["c"],
                                                                   flags, None, stream)]
        per, total = time_calls(args, stream, dev, flush, calls)
        rows = {}
        for i, P in enumerate(projs):
            q_ms, g_ms = per[2 * i:2 * i + 2]
            gf = 2.0 * P["M"] * P["N"] * P["K"]
            wbytes = G * P["N"] * P["K"]
            rows[P["name"]] = {"quant_ms": q_ms, "gemm_ms": g_ms,
                               "gemm_tflops": gf / (g_ms / 1e3) / 1e12,
                               "gemm_frac_fp8": gf / (g_ms / 1e3) / 1e12 / fp8_peak,
                               "weight_stream_GB/s": wbytes / (g_ms / 1e3) / 1e9,
                               "weight_stream_frac_hbm": wbytes / (g_ms / 1e3) / 1e9 / hbm_peak,
                               "quant_gemm_tflops": gf / ((q_ms + g_ms) / 1e3) / 1e12}
        flops = sum(2.0 * P["M"] * P["N"] * P["K"] for P in projs)
        out["modes"]["pow2" if pow2 else "fp32"] = {
            "gemm_kernel": "mx (grouped)" if pow2 else "promote (grouped)", "ms_per_step": total,
            "quant_gemm_tflops": flops / (total / 1e3) / 1e12, "projections": rows,
            "gpu_launches": 2 * len(projs) * args.steps}
    out["wgrad"] = moe_wgrad_measure(args, ops, stream, dev, flush, fp8_peak, m, projs, offs)
    return out


def moe_wgrad_measure(args, ops, stream, dev, flush, fp8_peak, m, projs, offs):
    """Weight gradients of the same experts, dW_g = dY_g^T X_g over each
    expert's rows: the grouped 128x1 quantiser of dY and of X (each expert's
    last token block padded with zeros) and the grouped wgrad GEMM, three
    launches per projection for all 128 experts.  dY is drawn on the device
    (N(0,1) x 1e-4; only the timing matters here, parity is tested
    separately).  FLOPs are 2 T N K (T = 65536 expert-sorted rows)."""
    import torch

    G = len(m.offsets) - 1
    offs32 = offs.to(torch.int32)
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed + 91)
    nb = (projs[0]["M"] + 127) // 128 + G
    W = []
    for P in projs:
        T, N, K = P["M"], P["N"], P["K"]
        dy = (torch.randn((T, N), generator=gen, device=dev) * 1e-4).to(torch.bfloat16)
        W.append(dict(name=P["name"], T=T, N=N, K=K, dy=dy, x=P["a"],
                      qg=torch.empty((N, 128 * nb), dtype=torch.uint8, device=dev),
                      sg=torch.empty((nb, ops.round_up(N, 4)), dtype=torch.float32, device=dev),
                      qx=torch.empty((K, 128 * nb), dtype=torch.uint8, device=dev),
                      sx=torch.empty((nb, ops.round_up(K, 4)), dtype=torch.float32, device=dev),
                      dw=torch.empty((G, N, K), dtype=torch.bfloat16, device=dev)))
    out = {"what": "per projection: grouped 128x1 quantiser of dY and of X, grouped wgrad GEMM (per-expert K "
                   "ranges from device offsets; promote kernel for fp32 scales, MX kernel for pow2 scales); "
                   "3 launches for all experts",
           "modes": {}}
    for pow2 in (False, True):
        mode = ops.FP8_SCALE_POW2 if pow2 else ops.FP8_SCALE_FP32_AMAX
        flags = ops.FP8_GEMM_SCALES_POW2 if pow2 else 0
        calls = []
        for P in W:
            calls += [lambda P=P: ops.fp8_quant_act_128x1_grouped(P["dy"], offs32, P["qg"], P["sg"], mode, stream),
                      lambda P=P: ops.fp8_quant_act_128x1_grouped(P["x"], offs32, P["qx"], P["sx"], mode, stream),
                      lambda P=P: ops.fp8_blockscaled_grouped_gemm_wgrad(P["qg"], P["sg"], P["qx"], P["sx"], offs32,
                                                                         P["T"], P["dw"], flags, stream)]
        per, total = time_calls(args, stream, dev, flush, calls)
        rows = {}
        for i, P in enumerate(W):
            qg_ms, qx_ms, g_ms = per[3 * i:3 * i + 3]
            gf = 2.0 * P["T"] * P["N"] * P["K"]
            rows[P["name"]] = {"quant_dy_ms": qg_ms, "quant_x_ms": qx_ms, "wgrad_ms": g_ms,
                               "wgrad_tflops": gf / (g_ms / 1e3) / 1e12,
                               "wgrad_frac_fp8": gf / (g_ms / 1e3) / 1e12 / fp8_peak,
                               "quant_wgrad_tflops": gf / ((qg_ms + qx_ms + g_ms) / 1e3) / 1e12}
        flops = sum(2.0 * P["T"] * P["N"] * P["K"] for P in W)
        out["modes"]["pow2" if pow2 else "fp32"] = {
            "wgrad_kernel": "mx (K-grouped)" if pow2 else "promote (K-grouped)",
            "ms_per_step": total, "quant_wgrad_tflops": flops / (total / 1e3) / 1e12, "projections": rows,
            "gpu_launches": 3 * len(W) * args.steps}
    return out


def attention_measure(args, ops, stream, dev, flush, hbm_peak):
    """One decode step of grouped-query attention over an FP8 KV cache at the
    Qwen3-8B attention shape (32 query heads, 8 KV heads, D 128): 64
    sequences with 4096 cached tokens each.  The cache holds seeded random
    codes of N(0, 1) activations under calibrated per-tensor scales (drawn on
    the device: only the timing matters here; parity is tested separately)."""
    import torch

    B, Hq, Hkv, T, D = 64, 32, 8, 4096, 128
    g = torch.Generator(device=dev)
    g.manual_seed(args.seed + 77)
    kv = torch.randn((B * Hkv * T, D), generator=g, device=dev).to(torch.bfloat16)
    qx = torch.randn((B * Hq, D), generator=g, device=dev).to(torch.bfloat16)
    sa = torch.empty(2, dtype=torch.float32, device=dev)
    kc = torch.empty((B * Hkv * T, D), dtype=torch.uint8, device=dev)
    vc = torch.empty_like(kc)
    qc = torch.empty((B * Hq, D), dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        ops.fp8_quant_per_tensor(kv, kc, sa, 0, stream)          # calibration + cast
        vc.copy_(kc.flip(0))
        ops.fp8_quant_per_tensor(qx, qc, sa, 0, stream)
    torch.cuda.synchronize(dev)
    del kv
    sq = sa[:1].clone()
    sk = sa[:1].clone()
    lens = torch.full((B,), T, dtype=torch.int32, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    need = ops.fp8_decode_attention_workspace_size(B, Hq, T)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    kc4, vc4, qc3 = kc.view(B, Hkv, T, D), vc.view(B, Hkv, T, D), qc.view(B, Hq, D)

    def run():
        ops.fp8_decode_attention(qc3, sq, kc4, sk, vc4, sk, lens, out, ws, stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush()
            run()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            flush()
            e0.record(stream)
            run()
            e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / len(evs)
    kv_bytes = 2.0 * B * Hkv * T * D            # FP8 K and V read once
    alg = kv_bytes + B * Hq * D + 2.0 * B * Hq * D
    return {"workload": "decode attention, Qwen3-8B heads (Hq 32, Hkv 8, D 128), 64 sequences x 4096 cached tokens",
            "kv_cache": "E4M3 codes, per-tensor calibrated K and V scales", "ms": ms,
            "GB/s": alg / (ms / 1e3) / 1e9, "frac_hbm": alg / (ms / 1e3) / 1e9 / hbm_peak,
            "bf16_cache_bytes_ratio": 2.0, "kernels_per_step": 2 if need else 1}


TRAIN_KERNELS = ("quant_x", "quant_w", "fprop", "quant_dy", "dgrad", "wgrad")


def train_measure(args, layers, ops, stream, dev, flush, fp8_peak, hbm_peak):
    """Times one training step per layer (forward + backward of y = x W^T) in
    both scale modes, per kernel with CUDA events over flushed steps.
    Gradients dY: Student-t (nu = 4) x 1e-4, seeded."""
    import torch

    from fp8_block_scaled_05_gb300 import inputs as I
    out = {"what": "per layer: dual quantisers of x (1x128 + 128x1), W (W + W^T) and dY (1x128 + 128x1); "
                   "fprop y = x W^T, dgrad dX = dY W (W^T codes), wgrad dW = dY^T X (1x128 scales on both)",
           "grad_recipe": "dY ~ Student-t(nu=4) x 1e-4, seeded PCG64", "modes": {}}
    bufs = []
    for L in layers:
        M, N, K = L["M"], L["N"], L["K"]
        dy = I.student_t_bf16(I.stream(args.seed + 500, N), (M, N), nu=4.0)
        dy = (dy.float() * 1e-4).to(torch.bfloat16).to(dev)
        B = dict(dy=dy,
                 qt_x=torch.empty((K, M), dtype=torch.uint8, device=dev),
                 st_x=torch.empty((M // 128, ops.round_up(K, 4)), dtype=torch.float32, device=dev),
                 qt_w=torch.empty((K, N), dtype=torch.uint8, device=dev),
                 st_w=torch.empty((K // 128, N // 128), dtype=torch.float32, device=dev),
                 q_dy=torch.empty((M, N), dtype=torch.uint8, device=dev),
                 s_dy=torch.empty((N // 128, ops.round_up(M, 4)), dtype=torch.float32, device=dev),
                 qt_dy=torch.empty((N, M), dtype=torch.uint8, device=dev),
                 st_dy=torch.empty((M // 128, ops.round_up(N, 4)), dtype=torch.float32, device=dev),
                 dx=torch.empty((M, K), dtype=torch.bfloat16, device=dev),
                 dw=torch.empty((N, K), dtype=torch.bfloat16, device=dev),
                 ws_d=ops.workspace_for(M, K, N, 1, dev), ws_w=ops.workspace_for(N, K, M, 1, dev))
        bufs.append(B)
    nk = len(TRAIN_KERNELS)

    def tstep(evs, pow2):
        mode = ops.FP8_SCALE_POW2 if pow2 else ops.FP8_SCALE_FP32_AMAX
        flags = ops.FP8_GEMM_SCALES_POW2 if pow2 else 0
        for i, (L, B) in enumerate(zip(layers, bufs)):
            calls = (
                lambda: ops.fp8_quant_act_128x1(L["a"], B["qt_x"], B["st_x"], L["qa"], L["sa"], mode, stream),
                lambda: ops.fp8_quant_weight_128x128_t(L["w"], B["qt_w"], B["st_w"], L["qw"], L["sw"], mode, stream),
                lambda: ops.fp8_blockscaled_gemm(L["qa"], L["sa"], L["qw"], L["sw"], L["c"], flags, L["ws"], stream),
                lambda: ops.fp8_quant_act_128x1(B["dy"], B["qt_dy"], B["st_dy"], B["q_dy"], B["s_dy"], mode, stream),
                lambda: ops.fp8_blockscaled_gemm(B["q_dy"], B["s_dy"], B["qt_w"], B["st_w"], B["dx"], flags,
                                                 B["ws_d"], stream),
                lambda: ops.fp8_blockscaled_gemm_wgrad(B["qt_dy"], B["st_dy"], B["qt_x"], B["st_x"], B["dw"], flags,
                                                       B["ws_w"], stream),
            )
            for j, call in enumerate(calls):
                if evs is not None:
                    evs[nk * i + j].record(stream)
                call()
        if evs is not None:
            evs[nk * len(layers)].record(stream)

    flops = sum(6.0 * L["M"] * L["N"] * L["K"] for L in layers)
    for pow2 in (False, True):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                flush()
                tstep(None, pow2)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nk * len(layers) + 1)] for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                flush()
                tstep(evs[k], pow2)
        torch.cuda.synchronize(dev)
        step_ms = sum(evs[k][0].elapsed_time(evs[k][-1]) for k in range(args.steps)) / args.steps
        per = {}
        for i, L in enumerate(layers):
            M, N, K = L["M"], L["N"], L["K"]
            ms = {kn: sum(evs[k][nk * i + j].elapsed_time(evs[k][nk * i + j + 1]) for k in range(args.steps))
                  / args.steps for j, kn in enumerate(TRAIN_KERNELS)}
            qbytes = {"quant_x": 4.0 * M * K + 8.0 * M * K / 128, "quant_w": 4.0 * N * K + 8.0 * N * K / 16384,
                      "quant_dy": 4.0 * M * N + 8.0 * M * N / 128}
            row = {"ms": ms}
            for kn, b in qbytes.items():
                row[kn + "_gbs"] = b / (ms[kn] / 1e3) / 1e9
                row[kn + "_frac_hbm"] = row[kn + "_gbs"] / hbm_peak
            for kn in ("fprop", "dgrad", "wgrad"):
                row[kn + "_tflops"] = 2.0 * M * N * K / (ms[kn] / 1e3) / 1e12
                row[kn + "_frac_fp8"] = row[kn + "_tflops"] / fp8_peak
            per[L["name"]] = row
        out["modes"]["pow2" if pow2 else "fp32"] = {
            "gemm_kernel": "mx" if pow2 else "promote", "ms_per_step": step_ms,
            "tflops": flops / (step_ms / 1e3) / 1e12, "layers": per,
            "gpu_launches": nk * len(layers) * args.steps}
    return out


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
