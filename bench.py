"""Benchmark of fused linear cross-entropy forward+backward on GB300.

One step = one call of flce_forward_backward (loss, lse, dH, dW) over one batch
of the Llama-3-8B-shaped head workload: N = 8192 tokens (B=2, S=4096),
D = 4096, V = 128256, H ~ N(0,1), W ~ N(0, 0.02^2) in bf16, Zipf(1.1) labels,
10% ignored tokens. Inputs are seeded synthetic data.

Reported (one JSON line on rank 0):
  value      tokens/s over all ranks, inputs resident in device memory
  tflops     8*N*V*D flops per step / step time (forward, recompute, two gradient GEMMs)
  e2e        tokens/s through the public API with host buffers: H, W and labels
             copied from pinned host memory and the loss read back, every step
  roofline   the dominant tcgen05 GEMM kernel (dW and dH launches) and each of the
             four products against the measured bf16 matmul peak (burst; the
             sustained peak beside it)
  cpu_baseline  the float64 CPU oracle timed on a bounded sample of the workload, a
                labelled extrapolation to the full step, and the tiny workload on
                one core
  peak_extra_hbm_bytes  the library's workspace (its whole extra device memory)
                        next to the N*V*4 bytes of fp32 logits an unfused head holds

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
For N > 1 the driver launches one process per GPU with torch.distributed.run;
every rank runs the same workload (replicas, weak scaling) and the slowest
rank's time is reported.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import flce_inputs  # noqa: E402

METRIC = "FLCE fwd+bwd tokens/s & TFLOP/s vs GB300 BF16 peak; peak extra HBM bytes"
UNIT = "tokens/s"


KERNEL_SOURCES = ("flce_gemm.cuh", "flce_gemm_params.h", "ptx.cuh")


def kernel_source_sha() -> str:
    """sha256 over the GEMM kernel's sources with comments and blank space
    removed: a DRAM-traffic figure measured with ncu applies only while the code
    is unchanged (editing a comment does not invalidate it)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "linear_cross_entropy_flce_gb300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)   # block comments
        src = re.sub(r"//[^\n]*", " ", src)                   # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


TRAFFIC_RECORDS = os.path.join(ROOT, "profiles", "dram_traffic.json")


def measured_traffic(kernel: str, workload: str, v_chunk: int):
    """DRAM bytes per launch of `kernel` on `workload` from the committed record of
    ncu captures (profiles/dram_traffic.json); None when absent, when the plan
    differs, or when the kernel sources changed since the counters were taken."""
    if not os.path.exists(TRAFFIC_RECORDS):
        return None
    sha = kernel_source_sha()
    with open(TRAFFIC_RECORDS) as f:
        records = json.load(f).get("records", [])
    for r in records:
        if r.get("kernel") == kernel and r.get("workload") == workload \
                and r.get("kernel_sha") == sha and int(r.get("v_chunk", -1)) == int(v_chunk):
            return float(r["bytes_per_launch"])
    return None


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Replicas:
    """Host-side coordination of independent replicas: a barrier and the max of
    a per-rank time. No data of the computation crosses ranks."""

    def __init__(self, world: int, rank: int):
        self.world, self.rank = world, rank
        self.pg = None
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


_SAMPLE_CACHE = {}


def cpu_oracle_sample(wl, tokens: int) -> dict:
    """The float64 oracle, as it stands, on the first `tokens` tokens of the
    workload (full V and D): loss, lse, dH for those tokens and dW from them.
    Only the oracle call is timed; the seeded draw is made once per sample size."""
    import oracle
    key = (wl.name, tokens)
    if key not in _SAMPLE_CACHE:
        Hb, Wb, y = flce_inputs.make_inputs(wl, N=tokens)
        _SAMPLE_CACHE.clear()
        _SAMPLE_CACHE[key] = (flce_inputs.bf16_bits_to_f32(Hb), flce_inputs.bf16_bits_to_f32(Wb), y)
    H, W, y = _SAMPLE_CACHE[key]
    t0 = time.perf_counter()
    oracle.flce(H, W, y)
    dt = time.perf_counter() - t0
    return {"seconds": dt, "tokens": tokens}


def oracle_tiny_single_core() -> dict:
    """The float64 oracle on the whole tiny workload (64 x 128 x 1000), fwd+bwd, in a
    child process whose BLAS is limited to one thread (best of 5 after a warm-up)."""
    code = ("import time, flce_inputs, oracle\n"
            "wl = flce_inputs.get('tiny')\n"
            "Hb, Wb, y = flce_inputs.make_inputs(wl)\n"
            "H, W = flce_inputs.bf16_bits_to_f64(Hb), flce_inputs.bf16_bits_to_f64(Wb)\n"
            "oracle.flce(H, W, y)\n"
            "best = 1e9\n"
            "for _ in range(5):\n"
            "    t0 = time.perf_counter(); oracle.flce(H, W, y); best = min(best, time.perf_counter() - t0)\n"
            "print(best)\n")
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=120, cwd=ROOT)
        sec = float(r.stdout.strip().splitlines()[-1])
    except Exception as e:   # reported, never fatal
        return {"error": str(e)[:200]}
    N = flce_inputs.get("tiny").N
    return {"seconds": sec, "tokens_per_s": N / sec, "cores": 1,
            "sample": "the whole tiny workload (N=64, D=128, V=1000), float64 fwd+bwd, best of 5"}


def fp8_reference_tflops(H8, W8, sh, sw, stream, reps: int = 10) -> dict:
    """cuBLASLt's E4M3 GEMM (torch._scaled_mm, bf16 output) on the same operands,
    Z = H8 W8^T at the LSE product's shape: the measured FP8 denominator."""
    import torch
    M, K = H8.shape
    Nn = W8.shape[0]
    try:
        a = H8.view(torch.float8_e4m3fn)
        b = W8.view(torch.float8_e4m3fn).t()   # [K, N] column-major
        s_a, s_b = sh[0:1].reshape(()), sw[0:1].reshape(())
        out = torch.empty(M, Nn, dtype=torch.bfloat16, device=H8.device)
        with torch.cuda.stream(stream):
            for _ in range(3):
                torch._scaled_mm(a, b, scale_a=s_a, scale_b=s_b, out_dtype=torch.bfloat16, out=out)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            best = 1e9
            for _ in range(reps):
                e0.record()
                torch._scaled_mm(a, b, scale_a=s_a, scale_b=s_b, out_dtype=torch.bfloat16, out=out)
                e1.record()
                e1.synchronize()
                best = min(best, e0.elapsed_time(e1))
        del out
        return {"tflops": 2.0 * M * Nn * K / (best * 1e-3) / 1e12, "ms_best": best,
                "how": f"torch._scaled_mm E4M3 x E4M3 -> bf16, {M} x {Nn} x {K}, best of {reps}"}
    except Exception as e:
        return {"tflops": None, "error": str(e)[:300]}


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args, wl, world, rank):
    """The reference arm: the float64 CPU oracle, each step a bounded sample."""
    if rank != 0:
        return 0
    tokens = min(args.ref_tokens, wl.N)  # a sample of the workload, never more
    for _ in range(args.warmup):
        cpu_oracle_sample(wl, tokens)
    times = [cpu_oracle_sample(wl, tokens)["seconds"] for _ in range(args.steps)]
    total = sum(times)
    value = tokens * args.steps / total
    sample = (f"first {tokens} tokens of the {wl.name} workload per step, full V={wl.V} and "
              f"D={wl.D}, float64 fwd+bwd (loss, lse, dH, dW)")
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_block(wl, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_forward_only(args, wl, world, rank, local):
    """The evaluation path: flce_forward (LSE GEMM, merge, reduce), 2*N*V*D flops."""
    import torch
    import linear_cross_entropy_flce_gb300 as flce
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rep = Replicas(world, rank)
    peaks = load_peaks()
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H = torch.from_numpy(Hb.view(np.int16)).to(dev).view(torch.bfloat16)
    W = torch.from_numpy(Wb.view(np.int16)).to(dev).view(torch.bfloat16)
    lab = torch.from_numpy(y).to(dev)
    N, D, V = wl.N, wl.D, wl.V
    ws = torch.empty(flce.forward_workspace_size(N, D, V), dtype=torch.uint8, device=dev)
    out = {"loss": torch.empty(1, dtype=torch.float32, device=dev),
           "lse": torch.empty(N, dtype=torch.float32, device=dev)}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        flce.forward(H, W, lab, out=out, workspace=ws, status=status, stream=stream.cuda_stream)

    for _ in range(args.warmup):
        step()
    if flce.check_status(status, stream.cuda_stream) != flce.FLCE_OK:
        raise RuntimeError("device status error")
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        rep.barrier()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        rep.barrier()
    ms = rep.max(ev0.elapsed_time(ev1) / args.steps)
    tflops = 2.0 * N * V * D / (ms / 1e3) / 1e12
    burst = peaks["bf16_tflops"]
    sustained = peaks.get("bf16_tflops_sustained", burst)
    line = {"metric": "FLCE forward (loss + lse) tokens/s", "value": N * world / (ms / 1e3),
            "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded; no dataset or weights)",
            "config": config_block(wl, world), "tflops": tflops, "frac_bf16_peak": tflops / burst,
            "frac_bf16_peak_sustained": tflops / sustained,
            "gpu_launches": 3 * args.steps, "clocks": clk.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    rep.close()
    return 0


def run_ce_logits(args, wl, world, rank, local):
    """Cross-entropy over given logits [N, V]: one step = loss, lse and the
    gradient written to a second buffer (flce_ce_logits). HBM-bound: the
    algorithmic bytes are one read and one write of the logits."""
    import torch
    import linear_cross_entropy_flce_gb300 as flce
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rep = Replicas(world, rank)
    peaks = load_peaks()
    N, V = wl.N, wl.V
    sigma = wl.h_scale * wl.w_std * (wl.D ** 0.5)   # logit std of the fused workload
    g = np.random.Generator(np.random.Philox(np.random.SeedSequence([wl.seed, 90])))
    dt = torch.float32 if args.ce_logits == "float32" else torch.bfloat16
    Z = torch.empty(N, V, dtype=dt, device=dev)
    rows = 1024
    for r0 in range(0, N, rows):
        r1 = min(N, r0 + rows)
        blk = g.standard_normal((r1 - r0, V), dtype=np.float32) * np.float32(sigma)
        Z[r0:r1].copy_(torch.from_numpy(blk))
    lab = torch.from_numpy(flce_inputs.make_labels(wl)).to(dev)
    elt = Z.element_size()
    out = {"loss": torch.empty(1, dtype=torch.float32, device=dev),
           "lse": torch.empty(N, dtype=torch.float32, device=dev),
           "dlogits": torch.empty_like(Z)}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(**kw):
        flce.ce_logits(Z, lab, out=out, status=status, stream=stream.cuda_stream, **kw)

    for _ in range(args.warmup):
        step()
    if flce.check_status(status, stream.cuda_stream) != flce.FLCE_OK:
        raise RuntimeError("device status error")
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        rep.barrier()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        rep.barrier()
    ms = rep.max(ev0.elapsed_time(ev1) / args.steps)
    # per-kernel: count, rows, reduce
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in evs:
        e.record(stream)
    torch.cuda.synchronize(dev)
    rows_ms = 0.0
    for _ in range(args.steps):
        step(trace_events=evs)
        torch.cuda.synchronize(dev)
        rows_ms += evs[1].elapsed_time(evs[2]) / args.steps
    algo = 2.0 * N * V * elt + N * 12
    achieved = algo / (rows_ms / 1e3) / 1e9
    line = {"metric": "cross-entropy over given logits (loss + gradient) tokens/s",
            "value": N * world / (ms / 1e3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if elt == 4 else "bf16", "data": "synthetic (seeded normal logits)",
            "config": {"workload": f"logits [{N}, {V}] {args.ce_logits}, labels of {wl.name}",
                       "N": N, "V": V, "l2": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "unit": "GB/s", "kernel": "ce_rows_kernel",
                         "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "frac": achieved / peaks["hbm_gbs"], "ms_per_launch": rows_ms,
                         "algorithmic_bytes_per_launch": algo, "traffic": None},
            "gpu_launches": 3 * args.steps, "clocks": clk.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    rep.close()
    return 0


OTHER_WORKLOADS = ("llama2", "qwen2_7b", "long_seq")


def time_steps(step, steps, stream, dev, local, flush=None) -> dict:
    """Device time of `steps` calls of step(), each bracketed by its own CUDA events
    on `stream`; with `flush` (a device buffer larger than L2) the buffer is
    overwritten before every step, outside the events, so each step starts with
    cold L2."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with ClockSampler(local) as clk:
        torch.cuda.synchronize(dev)
        for a, b in evs:
            if flush is not None:
                flush.zero_()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
    times = sorted(a.elapsed_time(b) for a, b in evs)
    c = clk.summary()
    return {"ms_per_step": sum(times) / steps, "ms_median": times[len(times) // 2],
            "steps": steps, "sm_mhz": c.get("sm_mhz"), "reasons": c.get("reasons")}


def other_workloads(args, flce, H, W, lab, wl_main, dev, local, stream, peaks) -> dict:
    """The 'workloads' block of the default line: every other head of the
    benchmark set (forward + backward, default plan), and the Llama-3-8B head's
    forward-only and FP8 steps, each timed in this run. The heads' inputs are
    drawn by the same seeded recipe; L2 is flushed before every timed step. An
    entry that fails records its error instead of stopping the run."""
    import torch
    burst = peaks["bf16_tflops"]
    steps, warmup = max(1, args.other_steps), 3
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # 2x L2
    block = {"note": ("each entry timed in this run after the main measurement: seeded "
                      "inputs by the same recipe, default plan, CUDA events per step on the "
                      "launching stream, L2 flushed (256 MB written) before every step")}

    def check(status):
        code = flce.check_status(status, stream.cuda_stream)
        if code != flce.FLCE_OK:
            raise RuntimeError(f"device status {code}: {flce.status_string(code)}")

    for name in OTHER_WORKLOADS:
        try:
            wl = flce_inputs.get(name)
            Hb, Wb, y = flce_inputs.make_inputs(wl)
            Hx = torch.from_numpy(Hb.view(np.int16)).to(dev).view(torch.bfloat16)
            Wx = torch.from_numpy(Wb.view(np.int16)).to(dev).view(torch.bfloat16)
            lx = torch.from_numpy(y).to(dev)
            del Hb, Wb
            N, D, V = wl.N, wl.D, wl.V
            ws_bytes = flce.workspace_size(N, D, V)
            ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
            out = {"loss": torch.empty(1, dtype=torch.float32, device=dev),
                   "lse": torch.empty(N, dtype=torch.float32, device=dev),
                   "dH": torch.empty(N, D, dtype=torch.bfloat16, device=dev),
                   "dW": torch.empty(V, D, dtype=torch.float32, device=dev)}
            status = torch.zeros(1, dtype=torch.int32, device=dev)

            def step():
                flce.forward_backward(Hx, Wx, lx, out=out, workspace=ws, status=status,
                                      stream=stream.cuda_stream)
            for _ in range(warmup):
                step()
            check(status)
            t = time_steps(step, steps, stream, dev, local, flush)
            check(status)
            tf = 8.0 * N * V * D / (t["ms_per_step"] * 1e-3) / 1e12
            block[name] = {"workload": config_block(wl, 1)["workload"], **t,
                           "tokens_per_s": N / (t["ms_per_step"] * 1e-3), "tflops_8nvd": tf,
                           "frac_of_burst_bf16": tf / burst, "workspace_bytes": ws_bytes,
                           "logits_bytes_unfused": N * V * 4}
            del Hx, Wx, lx, ws, out
        except Exception as e:   # keep the main line
            block[name] = {"error": str(e)[:300]}

    N, D, V = wl_main.N, wl_main.D, wl_main.V
    try:   # forward only (loss and lse), the evaluation path
        ws = torch.empty(flce.forward_workspace_size(N, D, V), dtype=torch.uint8, device=dev)
        out = {"loss": torch.empty(1, dtype=torch.float32, device=dev),
               "lse": torch.empty(N, dtype=torch.float32, device=dev)}
        status = torch.zeros(1, dtype=torch.int32, device=dev)

        def fstep():
            flce.forward(H, W, lab, out=out, workspace=ws, status=status,
                         stream=stream.cuda_stream)
        for _ in range(warmup):
            fstep()
        check(status)
        t = time_steps(fstep, steps, stream, dev, local, flush)
        check(status)
        tf = 2.0 * N * V * D / (t["ms_per_step"] * 1e-3) / 1e12
        block[f"{wl_main.name}_forward_only"] = {
            **t, "tokens_per_s": N / (t["ms_per_step"] * 1e-3), "tflops_2nvd": tf,
            "frac_of_burst_bf16": tf / burst, "workspace_bytes": ws.numel()}
        del ws, out
    except Exception as e:
        block[f"{wl_main.name}_forward_only"] = {"error": str(e)[:300]}

    try:   # E4M3 logits products, H and W quantised on the device every step
        q = (torch.empty(N, D, dtype=torch.uint8, device=dev),
             torch.empty(2, dtype=torch.float32, device=dev),
             torch.empty(V, D, dtype=torch.uint8, device=dev),
             torch.empty(2, dtype=torch.float32, device=dev))
        ws = torch.empty(flce.workspace_size(N, D, V), dtype=torch.uint8, device=dev)
        out = {"loss": torch.empty(1, dtype=torch.float32, device=dev),
               "lse": torch.empty(N, dtype=torch.float32, device=dev),
               "dH": torch.empty(N, D, dtype=torch.bfloat16, device=dev),
               "dW": torch.empty(V, D, dtype=torch.float32, device=dev)}
        status = torch.zeros(1, dtype=torch.int32, device=dev)

        def qstep():
            flce.quantize_e4m3(H, q=q[0], out=q[1], stream=stream.cuda_stream)
            flce.quantize_e4m3(W, q=q[2], out=q[3], stream=stream.cuda_stream)
            flce.forward_backward_fp8(q[0], q[1], q[2], q[3], lab, H, W, out=out, workspace=ws,
                                      status=status, stream=stream.cuda_stream)
        for _ in range(warmup):
            qstep()
        check(status)
        t = time_steps(qstep, steps, stream, dev, local, flush)
        check(status)
        block[f"{wl_main.name}_fp8"] = {
            **t, "tokens_per_s": N / (t["ms_per_step"] * 1e-3),
            "tflops_8nvd_effective": 8.0 * N * V * D / (t["ms_per_step"] * 1e-3) / 1e12,
            "note": "E4M3 logits products (forward, recompute), bf16 dH and dW products; "
                    "each step quantises H and W on the device first"}
        del q, ws, out
    except Exception as e:
        block[f"{wl_main.name}_fp8"] = {"error": str(e)[:300]}
    del flush
    torch.cuda.empty_cache()
    return block


def small_pass_bytes(N, D, plan) -> dict:
    """Algorithmic HBM bytes per step of the passes around the GEMMs (one read of
    what each reads, one write of what each writes): the merge reads the
    (max, sum) partials of every vocabulary range plus the target logits and the
    labels and writes lse, the NLL and the per-token (max, 1 / sum, 1 - p, 0) of
    the backward; the loss reduction reads the NLL and the labels; the rounding of
    the fp32 dH accumulator (several chunks only) reads it and writes bf16 dH."""
    npad = -(-N // 256) * 256
    out = {"lse_merge": 8 * plan["v_splits"] * npad + 8 * N + 24 * N,
           "loss_reduce": 8 * N}
    if plan["n_chunks"] > 1:
        out["dh_round"] = 6 * N * D
    return out


def make_roofline(N, V, D, kernel_ms, n_kind, per_kind, steps, peaks, traffic,
                  hbm_bytes_per_step=None) -> dict:
    """The roofline block of the JSON line from the per-kernel CUDA-event times.

    kernel_ms: ms per step of each kernel kind; n_kind / per_kind: launches and
    total ms of each kind over `steps` traced steps. The dominant kernel is the
    tcgen05 GEMM with the fp32 epilogue, whose one launch per chunk computes both
    dW = G^T H and dH = G W (two 2 N c D products): half of the step's flops and
    the largest time share. The kernels are timed as launches inside a step well
    under a second long, so the burst cuBLAS peak is the denominator; the
    sustained one is reported beside it. Every fraction is a quotient of the
    block's own numbers and the peaks. hbm_bytes_per_step (small_pass_bytes) adds
    to the HBM-bound passes their algorithmic GB/s and its fraction of the
    measured copy bandwidth."""
    burst = peaks["bf16_tflops"]
    sustained = peaks.get("bf16_tflops_sustained", burst)
    gemm_flops = 2.0 * N * V * D   # per step, for each of the four products

    def rate(ms_per_step):
        return gemm_flops / (ms_per_step / 1e3) / 1e12 if ms_per_step > 0 else None

    mult = {"dwdh_gemm": 2.0}
    f32_ms = kernel_ms["dwdh_gemm"]
    f32_launches = n_kind["dwdh_gemm"]
    achieved = 2.0 * gemm_flops / (f32_ms / 1e3) / 1e12
    products = {}
    for name, k in (("lse", "lse_gemm"), ("gradient", "grad_gemm"), ("dW + dH", "dwdh_gemm")):
        r = mult.get(k, 1.0) * rate(kernel_ms[k])
        products[name] = {"kernel": k, "tflops": r, "frac": r / burst,
                          "frac_of_sustained": r / sustained}
    total = sum(kernel_ms.values())
    kernels = {k: {"ms_per_step": kernel_ms[k],
                   "ms_per_launch": per_kind[k] / max(n_kind[k], 1),
                   "launches_per_step": n_kind[k] // steps,
                   "tflops": mult.get(k, 1.0) * rate(kernel_ms[k]) if k.endswith("gemm") else None,
                   "share": kernel_ms[k] / total}
               for k in ["lse_gemm", "lse_merge", "loss_reduce", "grad_gemm", "dwdh_gemm",
                         "dh_round"] if k in kernel_ms}
    for k, nbytes in (hbm_bytes_per_step or {}).items():
        if k in kernels and kernels[k]["ms_per_step"] > 0:
            gbs = nbytes / (kernels[k]["ms_per_step"] / 1e3) / 1e9
            kernels[k].update({"bound": "hbm", "algorithmic_bytes_per_step": nbytes, "gbs": gbs,
                               "frac_of_hbm": gbs / peaks["hbm_gbs"]})
    return {
        "bound": "tensor", "unit": "TFLOP/s",
        "kernel": "flce_gemm_kernel<EPI_F32> (tcgen05, 256 x 512 tiles: dW = G^T H and dH = G W, one launch per chunk)",
        "achieved": achieved, "peak": burst, "frac": achieved / burst,
        "peak_kind": f"bf16 cuBLAS burst, {peaks.get('source', 'measured')} (MEASURED_PEAKS.json bf16_tflops)",
        "peak_sustained": sustained, "frac_of_sustained": achieved / sustained,
        "products": products,
        "launches_per_step": f32_launches // steps,
        "flops_per_launch_avg": 2.0 * gemm_flops / (f32_launches / steps),
        "ms_per_launch_avg": per_kind["dwdh_gemm"] / max(f32_launches, 1),
        "traffic": traffic,
        "traffic_source": "profiles/dram_traffic.json (ncu dram__bytes_read.sum + "
                          "dram__bytes_write.sum per launch; null if the kernel changed)",
        "kernel_sha": kernel_source_sha(),
        "kernels": kernels,
    }


def config_block(wl, world) -> dict:
    return {"workload": f"{wl.name}: FLCE head N={wl.N} tokens, D={wl.D}, V={wl.V}, "
                        f"labels {wl.labels}, {int(round(wl.p_ignore * 100))}% ignore_index=-100",
            "N": wl.N, "D": wl.D, "V": wl.V, "global_batch_tokens": wl.N * world,
            "l2": "inputs larger than L2 (W alone is %.2f GB > 129 MB)" % (wl.V * wl.D * 2 / 1e9),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="llama3_8b", choices=sorted(flce_inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=1024,
                    help="tokens in the CPU-oracle baseline sample")
    ap.add_argument("--ref-tokens", type=int, default=256,
                    help="tokens per step of the reference (oracle) arm")
    ap.add_argument("--vocab", type=int, default=0,
                    help="override V (smaller profiling cases with the workload's other laws)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override N (smaller or tile-aligned cases with the workload's other laws)")
    ap.add_argument("--v-chunk", type=int, default=0, help="plan override: vocabulary ids per G chunk")
    ap.add_argument("--n-block", type=int, default=0, help="plan override: tokens per block")
    ap.add_argument("--forward-only", action="store_true",
                    help="time flce_forward (loss and lse, the evaluation path) instead")
    ap.add_argument("--ce-logits", choices=["float32", "bfloat16"], default=None,
                    help="time the cross-entropy over given [N, V] logits (loss + gradient) instead")
    ap.add_argument("--fp8", action="store_true",
                    help="FP8 operand variant: E4M3 H and W (per-tensor scales) for the two "
                         "logits products, bf16 H and W for the gradient products")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the 'workloads' block (the other heads, forward only, FP8) "
                         "that the default Llama-3-8B run adds to its line")
    ap.add_argument("--other-steps", type=int, default=10,
                    help="timed steps per entry of the 'workloads' block")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)

    wl = flce_inputs.get(args.workload)
    if args.vocab:
        import dataclasses
        wl = dataclasses.replace(wl, name=f"{wl.name}_V{args.vocab}", V=args.vocab)
    if args.tokens:
        import dataclasses
        wl = dataclasses.replace(wl, name=f"{wl.name}_N{args.tokens}", N=args.tokens)
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, wl, world, rank)
    if args.forward_only:
        return run_forward_only(args, wl, world, rank, local)
    if args.ce_logits:
        return run_ce_logits(args, wl, world, rank, local)
    if args.fp8:
        args.no_e2e = True
        args.no_cpu_baseline = True

    import torch
    import linear_cross_entropy_flce_gb300 as flce

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rep = Replicas(world, rank)
    peaks = load_peaks()

    # Inputs: seeded host draw, pinned host copy (e2e) and device copy (resident).
    Hb, Wb, y = flce_inputs.make_inputs(wl)
    H_host = torch.from_numpy(Hb.view(np.int16)).view(torch.bfloat16)
    W_host = torch.from_numpy(Wb.view(np.int16)).view(torch.bfloat16)
    y_host = torch.from_numpy(y)
    if not args.no_e2e:   # page-locked host buffers for the end-to-end leg
        H_host, W_host, y_host = H_host.pin_memory(), W_host.pin_memory(), y_host.pin_memory()
    H = H_host.to(dev)
    W = W_host.to(dev)
    lab = y_host.to(dev)
    N, D, V = wl.N, wl.D, wl.V
    fp8 = None
    if args.fp8:   # E4M3 operand buffers, quantised from H and W on the device every step
        fp8 = (torch.empty(N, D, dtype=torch.uint8, device=dev),
               torch.empty(2, dtype=torch.float32, device=dev),   # [scale_h, amax_h]
               torch.empty(V, D, dtype=torch.uint8, device=dev),
               torch.empty(2, dtype=torch.float32, device=dev))   # [scale_w, amax_w]

    plan_kw = {"v_chunk": args.v_chunk, "n_block": args.n_block}
    opts = flce.make_options(**plan_kw)
    plan = flce.get_plan(N, D, V, opts)
    ws_bytes = flce.workspace_size(N, D, V, opts)
    out = {"loss": torch.empty(1, dtype=torch.float32, device=dev),
           "lse": torch.empty(N, dtype=torch.float32, device=dev),
           "dH": torch.empty(N, D, dtype=torch.bfloat16, device=dev),
           "dW": torch.empty(V, D, dtype=torch.float32, device=dev)}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # Peak extra device memory of a call, seen by the caching allocator: inputs
    # and outputs already exist, the library allocates nothing itself, so the
    # growth is the workspace the caller hands it.
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    free0 = torch.cuda.mem_get_info(dev)[0]   # cross-check through cudaMemGetInfo
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def call(**kw):
        if fp8 is not None:
            flce.forward_backward_fp8(fp8[0], fp8[1], fp8[2], fp8[3], lab, H, W, out=out,
                                      workspace=ws, status=status, stream=stream.cuda_stream,
                                      **plan_kw, **kw)
        else:
            flce.forward_backward(H, W, lab, out=out, workspace=ws, status=status,
                                  stream=stream.cuda_stream, **plan_kw, **kw)

    def quantize():
        # per-tensor E4M3 operands and their scales, made on the device; the FP8
        # entry points read the scales from device memory (no host round trip)
        flce.quantize_e4m3(H, q=fp8[0], out=fp8[1], stream=stream.cuda_stream)
        flce.quantize_e4m3(W, q=fp8[2], out=fp8[3], stream=stream.cuda_stream)

    def step():
        if fp8 is not None:
            quantize()
        call()

    for _ in range(args.warmup):
        step()
    code = flce.check_status(status, stream.cuda_stream)
    if code != flce.FLCE_OK:
        raise RuntimeError(f"device status {code}: {flce.status_string(code)}")
    peak_delta = torch.cuda.max_memory_allocated(dev) - base
    torch.cuda.synchronize(dev)
    # device memory that left the free pool over the workspace allocation and the
    # warm-up calls (the allocator's 2 MB segment rounding and the first launch's
    # module loading included)
    free_delta = free0 - torch.cuda.mem_get_info(dev)[0]

    # ---- device-timed steps (inputs resident) ----
    # an event between consecutive steps (recorded on the same stream, no
    # synchronisation) gives each step's time for the median and the minimum
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev_step = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps - 1)]
    with ClockSampler(local) as clk:
        rep.barrier()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for k in range(args.steps):
            step()
            if k < args.steps - 1:
                ev_step[k].record(stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        rep.barrier()
    ms_local = ev0.elapsed_time(ev1) / args.steps
    ms = rep.max(ms_local)
    bounds = [ev0] + ev_step + [ev1]
    per_step = sorted(bounds[k].elapsed_time(bounds[k + 1]) for k in range(args.steps))
    step_stats = {"median": per_step[len(per_step) // 2], "min": per_step[0], "max": per_step[-1]}
    code = flce.check_status(status, stream.cuda_stream)
    if code != flce.FLCE_OK:
        raise RuntimeError(f"device status {code}: {flce.status_string(code)}")

    # ---- per-kernel durations: CUDA events the library records on this stream
    # before its first kernel and after each kernel of a call ----
    n_launch = plan["kernel_launches"]
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_launch + 1)]
    for e in evs:
        e.record(stream)  # creates the event handles
    torch.cuda.synchronize(dev)
    # per token block: each chunk's gradient GEMM and its one launch of the dW and
    # dH products, then (several chunks) the bf16 rounding of the block's fp32 dH
    # accumulator
    per_block = ["grad_gemm", "dwdh_gemm"] * plan["n_chunks"] + \
        (["dh_round"] if plan["n_chunks"] > 1 else [])
    kinds = ["lse_gemm", "lse_merge", "loss_reduce"] + per_block * plan["n_blocks"]
    assert len(kinds) == n_launch, (len(kinds), n_launch)
    per_kind = {k: 0.0 for k in kinds}
    n_kind = {k: 0 for k in kinds}
    for _ in range(args.steps):
        call(trace_events=evs)
        torch.cuda.synchronize(dev)
        for k in range(n_launch):
            per_kind[kinds[k]] += evs[k].elapsed_time(evs[k + 1])
            n_kind[kinds[k]] += 1
    kernel_ms = {k: per_kind[k] / args.steps for k in per_kind}      # per step
    quant_ms = None
    if fp8 is not None:   # the two device quantisations of a step, timed alone
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            quantize()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        quant_ms = ev0.elapsed_time(ev1) / args.steps

    # ---- end to end through the public API with host buffers ----
    # Every step copies its inputs (H, W, labels) from pinned host memory and
    # reads its loss back. The copies of step i+1 run on a copy stream into the
    # second of two device input buffers while step i computes.
    e2e = None
    if not args.no_e2e:
        copy_stream = torch.cuda.Stream(dev)
        bufs = [(H, W, lab), (torch.empty_like(H), torch.empty_like(W), torch.empty_like(lab))]
        copied = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]
        loss_host = torch.empty(args.steps + args.warmup, dtype=torch.float32).pin_memory()

        def run_e2e(nsteps, slot0):
            for i in range(nsteps):
                b = i % 2
                Hd, Wd, yd = bufs[b]
                copy_stream.wait_event(consumed[b])      # buffer b no longer in use
                with torch.cuda.stream(copy_stream):
                    Hd.copy_(H_host, non_blocking=True)
                    Wd.copy_(W_host, non_blocking=True)
                    yd.copy_(y_host, non_blocking=True)
                copied[b].record(copy_stream)
                stream.wait_event(copied[b])
                flce.forward_backward(Hd, Wd, yd, out=out, workspace=ws, status=status,
                                      stream=stream.cuda_stream, **plan_kw)
                consumed[b].record(stream)
                with torch.cuda.stream(stream):  # ordered after this step's kernels
                    loss_host[slot0 + i:slot0 + i + 1].copy_(out["loss"], non_blocking=True)

        run_e2e(args.warmup, 0)
        torch.cuda.synchronize(dev)
        # one step's host-to-device copies on their own, for reference
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(copy_stream)
        with torch.cuda.stream(copy_stream):
            bufs[1][0].copy_(H_host, non_blocking=True)
            bufs[1][1].copy_(W_host, non_blocking=True)
            bufs[1][2].copy_(y_host, non_blocking=True)
        c1.record(copy_stream)
        torch.cuda.synchronize(dev)
        h2d_alone_ms = c0.elapsed_time(c1)
        rep.barrier()
        with ClockSampler(local) as clk_e2e:
            t0 = time.perf_counter()
            ev0.record(copy_stream)
            run_e2e(args.steps, args.warmup)
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            wall = (time.perf_counter() - t0) / args.steps
        rep.barrier()
        code = flce.check_status(status, stream.cuda_stream)
        if code != flce.FLCE_OK:
            raise RuntimeError(f"device status {code}: {flce.status_string(code)}")
        ev_ms = ev0.elapsed_time(ev1) / args.steps
        e2e_ms = rep.max(max(ev_ms, 1e3 * wall))
        h2d = H_host.numel() * 2 + W_host.numel() * 2 + y_host.numel() * 4
        e2e = {"value": N * world / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": 4, "ms_per_step": e2e_ms,
               "overlap": "copies of step i+1 on a second stream during step i",
               "ms_device_events": ev_ms, "ms_host_wall": 1e3 * wall,
               "h2d_ms_one_step_alone": h2d_alone_ms,
               "clocks": clk_e2e.summary()}
        del bufs

    flops = 8.0 * N * V * D
    tflops = flops / (ms / 1e3) / 1e12
    value = N * world / (ms / 1e3)
    burst = peaks["bf16_tflops"]
    sustained = peaks.get("bf16_tflops_sustained", burst)
    roofline = make_roofline(N, V, D, kernel_ms, n_kind, per_kind, args.steps, peaks,
                             measured_traffic("flce_gemm_kernel<EPI_F32>", wl.name,
                                              plan["v_chunk"]),
                             hbm_bytes_per_step=small_pass_bytes(N, D, plan))
    products = roofline["products"]
    clocks = clk.summary()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:   # N = 1 only
        r = cpu_oracle_sample(wl, min(args.cpu_tokens, wl.N))
        full_s = r["seconds"] * wl.N / r["tokens"]
        cpu = {"value": r["tokens"] / r["seconds"], "unit": UNIT, "cores": blas_threads(),
               "kind": "oracle", "seconds": r["seconds"],
               "sample": f"first {r['tokens']} tokens of the {wl.name} workload, full V={V} "
                         f"and D={D}, float64 fwd+bwd (loss, lse, dH, dW)",
               "extrapolated_full": {
                   "seconds_per_step": full_s, "tokens_per_s": wl.N / full_s,
                   "method": f"EXTRAPOLATED, not measured: sample seconds x N / sample tokens "
                             f"({wl.N} / {r['tokens']}); the oracle's work is linear in N at "
                             f"fixed V and D (logits, lse, dH and dW passes: about 8 N V D "
                             f"float64 flops)"},
               "tiny_single_core": oracle_tiny_single_core()}

    others = None
    if (rank == 0 and world == 1 and fp8 is None and not args.no_other_workloads
            and wl.name == "llama3_8b"):
        others = other_workloads(args, flce, H, W, lab, wl, dev, local, stream, peaks)

    if fp8 is not None:
        # the two logits products run on E4M3 operands: their denominator is cuBLASLt's
        # own E4M3 GEMM (torch._scaled_mm) timed in this process at the LSE product's
        # shape; the nominal FP8/bf16 ratio (4.5 / 2.25 PFLOP/s dense) x the measured
        # bf16 peak only if that GEMM cannot run here
        fp8_ref = fp8_reference_tflops(fp8[0], fp8[2], fp8[1], fp8[3], stream)
        fp8_peak = fp8_ref["tflops"] if fp8_ref.get("tflops") else 2.0 * burst
        for name, k in (("lse", "lse_gemm"), ("gradient", "grad_gemm")):
            roofline["kernels"][k]["peak_fp8"] = fp8_peak
            roofline["kernels"][k]["frac_of_fp8_peak"] = roofline["kernels"][k]["tflops"] / fp8_peak
            products[name]["frac"] = products[name]["tflops"] / fp8_peak
            products[name]["peak"] = fp8_peak
        roofline["fp8_reference"] = fp8_ref
        roofline["note_fp8"] = ("lse_gemm and grad_gemm use E4M3 operands (kind::f8f6f4); their "
                                "fractions are against fp8_reference (cuBLASLt E4M3 GEMM at the "
                                "LSE shape, same process); each step first quantises H and W "
                                "on the device (amax + E4M3 kernels, 2 launches per tensor)")
        q_bytes = (N + V) * D * (2 + 2 + 1)   # amax read, quantise read + write
        roofline["quantize"] = {"ms_per_step": quant_ms, "algorithmic_bytes": q_bytes,
                                "gbs": q_bytes / (quant_ms * 1e-3) / 1e9}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 logits products + bf16 gradient products" if fp8 else "bf16", "data": "synthetic (seeded; no dataset or weights)",
        "config": config_block(wl, world),
        "tflops": tflops, "frac_bf16_peak": tflops / burst,
        "frac_bf16_peak_sustained": tflops / sustained,
        "ms_per_step_stats": step_stats,
        "peak_extra_hbm_bytes": int(peak_delta),
        "workspace_bytes": ws_bytes, "allocator_peak_delta_bytes": int(peak_delta),
        "cuda_free_bytes_delta": int(free_delta),
        "logits_bytes_unfused": N * V * 4,
        "plan": plan,
        "gpu_launches": (plan["kernel_launches"] + (4 if fp8 is not None else 0)) * args.steps,
        "e2e": e2e, "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks,
    }
    if others is not None:
        line["workloads"] = others
    if rank == 0:
        print(json.dumps(line), flush=True)
    rep.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
