"""Throughput of the fused linear cross-entropy forward+backward on GB300.

One step = lce_forward + lce_backward over one batch (every strip of the vocabulary: logits and
online log-sum-exp fold, strip combine, finalize; recomputed logits and gradient, dH and dW
contractions), through the C ABI, on inputs already resident in HBM.  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--strip-V S]
                  [--impl lce|reference] [--no-cpu-baseline]

Under torchrun (N > 1) every rank runs its own batch of the same workload (weak scaling, no
collective on the data path); rank 0 prints max-over-ranks timing.  ``--impl reference`` times
the float64 CPU oracle on a bounded sample of the same workload (the reference arm).
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from memory_bounded_linear_gb300 import api, full_logits_bytes  # noqa: E402
from memory_bounded_linear_gb300 import _lib  # noqa: E402
from memory_bounded_linear_gb300.workloads import HEADLINE, WORKLOADS, make_inputs  # noqa: E402

METRIC = "fused linear-CE fwd+bwd tokens/s and TFLOP/s vs GB300 bf16 dense peak; peak MB"
L2_BYTES = 129 * 1024 * 1024
# FLOPs per step of each contraction kernel, in units of N*d*V, summed over its launches: the
# forward logits (2); the backward's gradient launches (recomputed logits: 2) and dH + dW launches
# (4), or, for small backward steps, the overlapped launches that run all three (6); the fp32
# engine's four separate kernels.
GEMM_FLOP_FACTOR = {"tc_fwd_lse": 2, "tc_bwd_grad": 2, "tc_dh_dw": 4, "tc_bwd": 6,
                    "simt_fwd_lse": 2, "simt_bwd_grad": 2, "simt_dh": 2, "simt_dw": 2}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest value of x over all ranks (the slowest rank's time); x itself when alone."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def tokens_per_second(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own batch of tokens_per_rank per step."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of each tensor-core
# kernel, from one ncu capture of this benchmark's timed step at full size (one pass per
# kernel), keyed by workload, strip width, kernel and arithmetic.  They describe the source whose
# SHA-256 is KERNEL_SOURCE_SHA256; once the source differs they no longer apply (traffic: null).
KERNEL_SOURCES = ("memory_bounded_linear_gb300/csrc/lce_tc.cu",
                  "memory_bounded_linear_gb300/csrc/ptx.cuh",
                  "memory_bounded_linear_gb300/csrc/lce_internal.h",
                  "memory_bounded_linear_gb300/csrc/lce_api.cu")  # launch structure
KERNEL_SOURCE_SHA256 = "649966d7e5fcd986904d7a1bde41bc8be0ff22df4e4985d2f313c6bd396c7890"
MEASURED_TRAFFIC = {
    # N=32768 d=6144 V=151552, strip 16384 (ten strips of 15360 columns, the last 13312): the
    # timed step's 21 launches -- the forward over the whole vocabulary, then per strip the
    # gradient launch and the dW + dH launch (each averaged over its 10 launches)
    ("n32768-d6144-v151552-outliers", 16384, "tc_fwd_lse", "bf16"): 30406000000,
    ("n32768-d6144-v151552-outliers", 16384, "tc_bwd_grad", "bf16"): 4437000000,
    ("n32768-d6144-v151552-outliers", 16384, "tc_dh_dw", "bf16"): 20225000000,
    # N=16384 d=7168 V=200000 fp32, three-product tf32, strip 16384 (13 strips of 15616 columns,
    # the last 12608): the timed step's 39 tensor-core launches -- 13 forward strips, then per
    # strip the gradient launch and the dH + dW launch (each averaged over its 13 launches)
    ("n16384-d7168-v200000-fp32", 16384, "tc_fwd_lse", "tf32x3"): 14557000000,
    ("n16384-d7168-v200000-fp32", 16384, "tc_bwd_grad", "tf32x3"): 18253000000,
    ("n16384-d7168-v200000-fp32", 16384, "tc_dh_dw", "tf32x3"): 46299000000,
}


def kernel_source_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload: str, strip_V: int, kernel: str, dtype: str):
    """Bytes per launch measured for this kernel source, else None."""
    if KERNEL_SOURCE_SHA256 is None or kernel_source_sha256() != KERNEL_SOURCE_SHA256:
        return None
    return MEASURED_TRAFFIC.get((workload, strip_V, kernel, dtype))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


def cpu_baseline(w, H, W, y, target_s=15.0, min_tokens=16):
    """Time the float64 oracle (as it stands) on a bounded token sample of the same workload:
    one block of tokens through logits, lse, loss, dH rows and the block's dW contribution."""
    import numpy as np

    import oracle

    Wn = W.cpu().to(torch.float64).numpy()
    valid = (y != -100)
    n_valid = int(valid.sum().item())
    scale = (1.0 / max(n_valid, 1)) if w.reduction == "mean" else 1.0

    def run(n):
        Hb = H[:n].cpu().to(torch.float64).numpy()
        yb = y[:n].cpu().numpy()
        t0 = time.perf_counter()
        oracle.token_block_fwd_bwd(Hb, Wn, yb, scale)
        return time.perf_counter() - t0

    # grow the sample until it takes at least 2/3 of target_s (the first, small runs also warm up
    # the BLAS thread pool), never beyond the batch
    n = min_tokens
    t = run(n)
    for _ in range(3):
        if t >= target_s * 2 / 3 or n >= w.N:
            break
        n = int(min(w.N, max(n + 1, n * target_s / max(t, 1e-3))))
        t = run(n)
    cores = len(os.sched_getaffinity(0))
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", os.environ.get("OMP_NUM_THREADS", cores)))
    del np
    return {"value": n / t, "unit": "tokens/s", "cores": min(cores, threads), "kind": "oracle",
            "seconds": t,
            "sample": f"{n} tokens x full vocabulary ({w.V}) x d={w.d}, float64 numpy: "
                      f"logits, lse, loss, dH rows and the block's dW contribution"}


def run_reference(args, w):
    """Reference arm: the float64 CPU oracle, timed on host cores, each step a bounded sample."""
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle

    H, W, y = make_inputs(w, "cpu", seed=0)
    Wn = W.to(torch.float64).numpy()
    n = args.ref_tokens
    Hb = H[:n].to(torch.float64).numpy()
    yb = y[:n].numpy()
    n_valid = int((y != -100).sum().item())
    scale = (1.0 / max(n_valid, 1)) if w.reduction == "mean" else 1.0
    for _ in range(args.warmup):
        oracle.token_block_fwd_bwd(Hb, Wn, yb, scale)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.token_block_fwd_bwd(Hb, Wn, yb, scale)
    dt = (time.perf_counter() - t0) / args.steps
    value = n / dt
    cores = len(os.sched_getaffinity(0))
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "N": w.N, "d": w.d, "V": w.V, "strip_V": args.strip_V,
                   "reduction": w.reduction, "sample_tokens": n},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} tokens of the workload per step, full vocabulary"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--strip-V", dest="strip_V", type=int, default=None)
    ap.add_argument("--impl", default="lce", choices=["lce", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ref-tokens", type=int, default=64)
    ap.add_argument("--tile-config", type=int, default=0, choices=[0, 1, 2],
                    help="tensor-core tile variant: 0 automatic, 1 single-CTA, 2 CTA pairs")
    ap.add_argument("--f32-mode", dest="f32_mode", default="exact", choices=["exact", "tf32x3"],
                    help="arithmetic for fp32 workloads: exact FFMA, or three tf32 tensor-core "
                         "products per fp32 product")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override N (same d, V, strip and distributions; for small profiling runs)")
    ap.add_argument("--vocab", type=int, default=None,
                    help="override V (same N, d, strip and distributions; for small profiling runs)")
    args = ap.parse_args()
    w = WORKLOADS[args.workload]
    if args.tokens:
        w = w.with_sizes(N=args.tokens)
    if args.vocab:
        w = w.with_sizes(V=args.vocab)
    args.strip_V = args.strip_V or w.strip_V
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        run_reference(args, w)
        return

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    lib = _lib.load()
    _lib.check(lib.lce_set_tile_config(args.tile_config), "lce_set_tile_config")

    N, d, V, S = w.N, w.d, w.V, args.strip_V
    fm = args.f32_mode
    dt = "tf32x3" if (w.dtype == "f32" and fm == "tf32x3") else w.dtype
    H, W, y = make_inputs(w, dev, seed=rank)
    ws_bytes = api.lce_workspace_size(N, d, V, S, dt)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    loss = torch.empty((), device=dev)
    lse = torch.empty(N, device=dev)
    nv = torch.empty((), dtype=torch.int64, device=dev)
    dH = torch.empty(N, d, device=dev)
    dW = torch.empty(V, d, device=dev)
    one = torch.ones((), device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        api.lce_forward(H, W, y, strip_V=S, reduction=w.reduction, workspace=ws,
                        out=(loss, lse, nv), stream=stream, f32_mode=fm)
        api.lce_backward(H, W, y, lse, nv, one, strip_V=S, reduction=w.reduction, workspace=ws,
                         dH=dH, dW=dW, stream=stream, f32_mode=fm)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    # warm-up; peak memory of one forward+backward measured here
    in_out_bytes = sum(t.numel() * t.element_size() for t in (H, W, y, lse, dH, dW))
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    for _ in range(args.warmup):
        step()
    barrier()
    api.lce_check_error(ws)
    peak = torch.cuda.max_memory_allocated(dev)

    # per-launch trace buffers (events recorded around every launch on the launching stream)
    per_step = 7 * ((V + S - 1) // S) + 4  # at most: splits, GEMMs, combines, finalize
    cap = per_step * args.steps + 16
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(cap)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(cap)]
    for e in starts + stops:
        e.record(stream)
    torch.cuda.synchronize(dev)
    arr = ctypes.c_void_p * cap
    st_arr = arr(*[e.cuda_event for e in starts])
    sp_arr = arr(*[e.cuda_event for e in stops])
    ids = (ctypes.c_int32 * cap)()

    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clocks:
        barrier()
        launches0 = lib.lce_launch_count()
        _lib.check(lib.lce_trace_begin(st_arr, sp_arr, ids, cap), "lce_trace_begin")
        t_start.record(stream)
        for _ in range(args.steps):
            step()
        t_stop.record(stream)
        n_traced = lib.lce_trace_end()
        launches = lib.lce_launch_count() - launches0
        barrier()
    ms_total = max_over_ranks(t_start.elapsed_time(t_stop), world, dev)
    ms = ms_total / args.steps
    tokens_s = tokens_per_second(world, N, ms)
    tflops = world * w.flops / (ms / 1e3) / 1e12
    api.lce_check_error(ws)

    # per-kernel device time from the trace (same timed region)
    agg = {}
    for i in range(n_traced):
        name = lib.lce_kernel_name(ids[i]).decode()
        a = agg.setdefault(name, [0, 0.0])
        a[0] += 1
        a[1] += starts[i].elapsed_time(stops[i])
    if "tc_bwd" in agg:
        # small backward steps: the first launch computes the first strip's gradient alone and the
        # last one dW and dH of the last strip alone; with the overlapped launches between them
        # they make up the backward's 6*N*d*V, so they are counted together
        for k in ("tc_bwd_grad", "tc_dh_dw"):
            if k in agg:
                n_k, t_k = agg.pop(k)
                agg["tc_bwd"][0] += n_k
                agg["tc_bwd"][1] += t_k
    dominant = max((k for k in agg if k in GEMM_FLOP_FACTOR), key=lambda k: agg[k][1])
    n_launch, t_kernel = agg[dominant]
    peaks, peak_src = measured_peaks()
    # three-product tf32: the tensor pipe runs three tf32 products per fp32 product, so the
    # kernel's tensor work is 3x its fp32 GEMM FLOPs, set against the tf32 peak (the measured bf16
    # peak x the nominal dense tf32 / bf16 ratio, 18 / 36 PFLOP/s per 8 GPUs)
    x3_factor = 3 if dt == "tf32x3" else 1
    # The sustained peak (back-to-back GEMMs held at the power cap) when the power cap was active
    # during the timed region, else the burst peak (a GEMM below the cap).
    clk = clocks.summary()
    capped = "sw_power_cap" in (clk.get("reasons") or [])
    bf16_key = "bf16_tflops_sustained" if capped else "bf16_tflops"
    if dt == "bf16":
        peak_tf, peak_name = peaks[bf16_key], f"{bf16_key} ({peak_src})"
    elif dt == "tf32x3":
        peak_tf = peaks[bf16_key] * 0.5
        peak_name = f"tf32 dense = {bf16_key} ({peak_src}) x nominal tf32/bf16 ratio 0.5"
    else:
        # exact fp32 runs on the FFMA units: 152 SMs x 128 fp32 lanes x 2 FLOP x max SM clock
        mhz = peaks.get("sm_max_mhz", 2070.0)
        peak_tf = 152 * 128 * 2 * mhz * 1e6 / 1e12
        peak_name = f"derived fp32 FFMA peak: 152 SMs x 128 lanes x 2 FLOP x {mhz:.0f} MHz"
    # algorithmic FLOPs of that kernel per step: factor * N * d * V (2 per contraction it runs,
    # summed over its launches -- every strip, tail strip included)
    kernel_flops_step = GEMM_FLOP_FACTOR[dominant] * N * d * V * x3_factor
    achieved = kernel_flops_step * args.steps / (t_kernel / 1e3) / 1e12
    roofline = {"kernel": dominant, "bound": "alu" if dt == "f32" else "tensor",
                "achieved": achieved, "peak": peak_tf,
                "unit": "TFLOP/s", "frac": (achieved / peak_tf) if peak_tf else None,
                "traffic": (None if (args.tokens or args.vocab)
                            else measured_traffic(w.name, S, dominant, dt)),
                "launches": n_launch,
                "avg_launch_ms": t_kernel / n_launch,
                "peak_source": peak_name,
                "per_kernel_ms_per_step": {k: v[1] / args.steps for k, v in sorted(agg.items())},
                # every contraction kernel's algorithmic rate (the dominant one is above)
                "per_kernel_tflops": {k: GEMM_FLOP_FACTOR[k] * N * d * V * x3_factor * args.steps
                                         / (v[1] / 1e3) / 1e12
                                      for k, v in sorted(agg.items()) if k in GEMM_FLOP_FACTOR}}
    if dt != "f32" and clk.get("sm_mhz") and clk.get("samples", 0) >= 10:
        # Context for the fraction above: the dense tensor rate per SM and clock (8192 bf16 or
        # 4096 tf32 FLOP per cycle, the per-SM rate behind the nominal 2.25 / 1.1 PFLOP/s) at the
        # median SM clock sampled during the timed region.  Under the power cap the tf32 MMAs hold
        # a higher clock than the bf16 GEMMs behind the measured peak, so against that peak x 0.5
        # a tf32 kernel can read above 1.  Only with at least 10 clock samples (2 s of timed work).
        per_clk = 8192 if dt == "bf16" else 4096
        p_clk = 152 * per_clk * clk["sm_mhz"] * 1e6 / 1e12
        roofline["peak_at_sampled_clock"] = p_clk
        roofline["frac_at_sampled_clock"] = achieved / p_clk

    # End to end through the C ABI with HOST buffers (lce_forward_backward_host), two variants,
    # each timed over K steps:
    #  * e2e (every result back): each step's call copies H, W, labels and dloss from pinned host
    #    memory into its device buffer, runs forward+backward, and copies EVERY output (loss, lse,
    #    n_valid, dH, dW, error flags) back to pinned host memory -- the library used as a
    #    host-to-host operator;
    #  * e2e_loss_only (the training-loop figure): the same calls, but only the loss and the error
    #    flags come back; dH and dW stay on the device, where the previous layer's backward and the
    #    optimizer would use them.
    # Consecutive steps rotate over three device buffers and three streams, and each step's kernels
    # wait for the previous step's (compute_after / compute_done): the kernels run one step at a
    # time while the copies in of one step and the copies out of another proceed beside them on
    # the two copy directions.
    e2e = e2e_loss = None
    if not args.no_e2e:
        Hh = H.cpu().pin_memory()
        Wh = W.cpu().pin_memory()
        yh = y.cpu().pin_memory()
        dl = torch.ones((), dtype=torch.float32).pin_memory()
        in_bytes = sum(t.numel() * t.element_size() for t in (Hh, Wh, yh, dl))
        hb = api.lce_host_buffer_size(N, d, V, S, dt)
        NB = 3
        dbufs = [torch.empty(hb, dtype=torch.uint8, device=dev) for _ in range(NB)]
        streams = [torch.cuda.Stream(dev) for _ in range(NB)]
        houts = [{"loss": torch.empty((), dtype=torch.float32).pin_memory(),
                  "lse": torch.empty(N, dtype=torch.float32).pin_memory(),
                  "n_valid": torch.empty((), dtype=torch.int64).pin_memory(),
                  "dH": torch.empty(N, d, dtype=torch.float32).pin_memory(),
                  "dW": torch.empty(V, d, dtype=torch.float32).pin_memory(),
                  "flags": torch.zeros(1, dtype=torch.int32).pin_memory()} for _ in range(NB)]

        done = [torch.cuda.Event() for _ in range(NB)]

        def run_steps(k, results_back):
            for i in range(k):
                o = houts[i % NB]
                outs = o if results_back else {"loss": o["loss"], "flags": o["flags"]}
                # this step's kernels start after the previous step's have finished
                api.lce_forward_backward_host(Hh, Wh, yh, dl, device_buffer=dbufs[i % NB],
                                              strip_V=S, reduction=w.reduction, f32_mode=fm,
                                              stream=streams[i % NB],
                                              compute_after=done[(i - 1) % NB] if i else None,
                                              compute_done=done[i % NB], **outs)

        def time_e2e(results_back):
            run_steps(NB, results_back)
            barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            k2 = max(3, args.steps)
            e0.record(stream)
            for st in streams:
                st.wait_event(e0)
            run_steps(k2, results_back)
            for st in streams:
                stream.wait_stream(st)
            e1.record(stream)
            barrier()
            if any(int(o["flags"].item()) != 0 for o in houts):
                raise RuntimeError("device error flags set during the end-to-end steps")
            return max_over_ranks(e0.elapsed_time(e1) / k2, world, dev)

        out_bytes = sum(t.numel() * t.element_size() for t in houts[0].values())

        def copy_gbs():
            """The box's pinned-memory copy rate, copies alone (no kernels), with the same pinned
            buffers: dH and dW back (device to host), H and W in (host to device)."""
            st = streams[0]
            as_bytes = [t.reshape(-1).view(torch.uint8)
                        for t in (houts[0]["dH"], houts[0]["dW"], Hh, Wh)]
            pairs_d2h = [(o, dbufs[0][:o.numel()]) for o in as_bytes[:2]]
            pairs_h2d = [(dbufs[0][:t.numel()], t) for t in as_bytes[2:]]
            rates = {}
            for name, pairs in (("d2h", pairs_d2h), ("h2d", pairs_h2d)):
                nbytes = sum(dst.numel() for dst, _ in pairs)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(st):
                    for dst, src in pairs:
                        dst.copy_(src, non_blocking=True)
                    e0.record(st)
                    for _ in range(3):
                        for dst, src in pairs:
                            dst.copy_(src, non_blocking=True)
                    e1.record(st)
                st.synchronize()
                rates[name] = 3 * nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9
            return rates

        copy_rates = copy_gbs()
        e_ms = time_e2e(True)
        e2e = {"value": tokens_per_second(world, N, e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
               "ms_per_step": e_ms, "api": "lce_forward_backward_host",
               "results": "loss, lse, n_valid, dH, dW and error flags copied back to pinned host "
                          "memory every step",
               "overlap": "three device buffers and streams rotating by step; each step's kernels "
                          "wait for the previous step's (compute_after / compute_done)",
               "copy_gbs_alone": copy_rates}
        l_ms = time_e2e(False)
        e2e_loss = {"value": tokens_per_second(world, N, l_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": 4 + 4,
                    "ms_per_step": l_ms, "api": "lce_forward_backward_host",
                    "results": "loss and error flags only; dH and dW stay on the device "
                               "(training-loop figure)",
                    "overlap": "three device buffers and streams rotating by step; each step's "
                               "kernels wait for the previous step's"}
        del dbufs, houts

    # Delayed weight gradient (lce_backward_parts): the dgrad-only and wgrad-only backward calls
    # against the fused backward on the same inputs and workspace, CUDA events on the launching
    # stream, after the timed region.  Each part recomputes its strips' logits.
    def time_backward(parts, n):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier()
        e0.record(stream)
        for _ in range(n):
            api.lce_backward(H, W, y, lse, nv, one, strip_V=S, reduction=w.reduction,
                             workspace=ws, dH=dH, dW=dW, stream=stream, f32_mode=fm, parts=parts)
        e1.record(stream)
        barrier()
        return max_over_ranks(e0.elapsed_time(e1) / n, world, dev)

    n_bwd = max(1, min(5, int(2000.0 / max(time_backward("both", 1), 1e-3))))
    bwd_ms = {p: time_backward(p, n_bwd) for p in ("both", "dh", "dw")}
    api.lce_check_error(ws)
    delayed_wgrad = {"backward_ms": bwd_ms["both"], "dgrad_only_ms": bwd_ms["dh"],
                     "wgrad_only_ms": bwd_ms["dw"], "iterations": n_bwd,
                     "critical_path_fraction": bwd_ms["dh"] / bwd_ms["both"]}

    # The same step captured once into a CUDA graph and replayed K times (no host work per step):
    # any launch overhead the direct calls above pay would show as the difference.
    def step_current_stream():
        api.lce_forward(H, W, y, strip_V=S, reduction=w.reduction, workspace=ws,
                        out=(loss, lse, nv), f32_mode=fm)
        api.lce_backward(H, W, y, lse, nv, one, strip_V=S, reduction=w.reduction, workspace=ws,
                         dH=dH, dW=dW, f32_mode=fm)

    # (thread-local capture: other threads of the process -- e.g. a process group's watchdog --
    # may keep using CUDA meanwhile)
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            step_current_stream()
        graph.replay()
        graph_err = None
    except RuntimeError as ex:
        graph, graph_err = None, str(ex).splitlines()[0][:200]
    # every rank times the replays, or none does (the barriers below must match across ranks)
    if max_over_ranks(0.0 if graph_err is None else 1.0, world, dev) > 0.0:
        graph_err = graph_err or "capture failed on another rank"
        graph = None
    barrier()
    if graph is not None:
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        g1.record(stream)
        barrier()
        api.lce_check_error(ws)
        t_graph = g0.elapsed_time(g1) / args.steps
        del graph
    else:
        t_graph = float("nan")
    graph_ms = max_over_ranks(t_graph, world, dev)
    cuda_graph = ({"ms_per_step": graph_ms, "value": tokens_per_second(world, N, graph_ms),
                   "unit": "tokens/s"} if graph_err is None else {"unavailable": graph_err})

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, H, W, y)

    if rank == 0:
        line = {
            "metric": METRIC, "value": tokens_s, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dt, "data": "synthetic",
            "config": {"workload": w.name, "N": N, "d": d, "V": V, "strip_V": S,
                       "reduction": w.reduction, "parallelism": f"independent batch per GPU x{world}",
                       "tile_config": ["auto", "single-cta", "cta-pair"][args.tile_config],
                       "l2": "inputs larger than L2 (H+W = %.0f MB > 129 MB), no flush"
                             % ((H.numel() * H.element_size() + W.numel() * W.element_size()) / 1e6)},
            "tflops": tflops,
            "frac_of_peak": x3_factor * tflops / peak_tf if peak_tf else None,
            "peak_mb": peak / 1e6,
            "peak_minus_inputs_outputs_mb": (peak - in_out_bytes) / 1e6,
            "workspace_mb": ws_bytes / 1e6,
            "full_logits_mb_avoided": full_logits_bytes(N, V) / 1e6,
            "gpu_launches": launches,
            "roofline": roofline,
            "clocks": clk,
            "e2e": e2e,
            "e2e_loss_only": e2e_loss,
            "delayed_wgrad": delayed_wgrad,
            "cuda_graph": cuda_graph,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
