"""Benchmark of the quantized weight-streaming decode step on GB300.

Default workload: the Bonsai-27B-shaped PQ2_0 decode weight stream (401
ternary projections, 6.80 GB of packed weights, one activation vector per
projection), run as one persistent-kernel decode step per iteration through
the C ABI.  Metric: weight-stream GB/s = (packed weight bytes + fp32
activation bytes read + fp32 output bytes written) / device time per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kq|reference]

--impl reference times the FP64 CPU oracle on a bounded sample of the same
workload (rows sampled from every projection) on the host cores.  With N > 1
(torchrun, one rank per GPU) every rank streams its own full replica (weak
scaling, no collective on the data path); rank 0 prints one JSON line.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "bonsai_27b_pq2_0_step"
SECONDARY = "qwen3_4b_q8_0_step"
METRIC = "quantized GEMV weight-stream GB/s (% of GB300 HBM peak); us per decode step"
FALLBACK_HBM_GBS = 6800.0


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_code_sha256(path):
    """sha256 of a source file's code: every line, stripped, except empty
    lines and whole-line // comments, so that comment edits keep it."""
    import hashlib

    keep = [ln.strip() for ln in open(path, encoding="utf-8") if ln.strip() and not ln.strip().startswith("//")]
    return hashlib.sha256("\n".join(keep).encode()).hexdigest()


def _traffic(workload):
    """DRAM bytes per launch of the stream kernel from the committed ncu summary,
    or None when the kernel code changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "stream_kernel_traffic.txt")
    src = os.path.join(ROOT, "quantized_weight_streaming_gb300", "csrc", "kq_stream.cu")
    try:
        kv = {}
        for line in open(path):
            line = line.split("#", 1)[0].strip()
            if "=" in line:
                k, v = (t.strip() for t in line.split("=", 1))
                kv[k] = v
        if kv.get("source_code_sha256") != source_code_sha256(src):
            return None
        return float(kv[workload + ".dram_read_bytes"]) + float(kv[workload + ".dram_write_bytes"])
    except Exception:
        return None


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.reader.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# libkq arm
# ----------------------------------------------------------------------------

def _time_steps(fn, steps, stream):
    import torch

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3  # seconds


def _step_stats(fn, n, stream):
    """Per-step device times of n more steps, each between its own pair of
    CUDA events on the stream: median, median absolute deviation, min, max (us)."""
    import torch

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    t = np.array([a.elapsed_time(b) * 1e3 for a, b in ev])
    med = float(np.median(t))
    return {"n": n, "median_us": round(med, 2), "mad_us": round(float(np.median(np.abs(t - med))), 2),
            "min_us": round(float(t.min()), 2), "max_us": round(float(t.max()), 2)}


def max_over_ranks(value, device=None):
    """Largest `value` over all ranks of the default process group (the value
    itself without one).  Used for the timed seconds: the job is as slow as its
    slowest replica."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_step, steps, seconds_max, world):
    """Whole-job throughput: every replica streams bytes_per_step per step, the
    job takes as long as its slowest rank."""
    return bytes_per_step * steps * world / seconds_max / 1e9


def _decode_measure(kq, wl_mod, config, steps, warmup, stream, sampler_gpu=None, world=1, limit=None, linked=False,
                    e2e=True, rotation=None, stats=False):
    import torch

    W = wl_mod.DecodeWorkload(config, seed=0, limit=limit, linked=linked, rotation=rotation)
    bytes_per_step = W.weight_bytes + W.activation_bytes
    for _ in range(warmup):
        W.step(stream)
    torch.cuda.synchronize()
    if kq.kq_device_status(True) != kq.KQ_OK:
        raise RuntimeError("device status not ok after warm-up")
    clocks = None
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    if sampler_gpu is not None:
        with ClockSampler(sampler_gpu) as cs:
            secs = _time_steps(lambda: W.step(stream), steps, stream)
        clocks = cs.summary()
    else:
        secs = _time_steps(lambda: W.step(stream), steps, stream)
    if world > 1:
        secs = max_over_ranks(secs, device="cuda")
    if kq.kq_device_status(True) != kq.KQ_OK:
        raise RuntimeError("device status not ok after the timed region")
    step_stats = _step_stats(lambda: W.step(stream), min(steps, 50), stream) if stats else None
    per_step = secs / steps
    if not e2e:
        out = {"config": config, "matrices": len(W.mats_spec), "weight_bytes": W.weight_bytes,
               "bytes_per_step": bytes_per_step, "seconds": secs, "per_step_s": per_step,
               "gbs": bytes_per_step / per_step / 1e9, "stages": W.plan.stages,
               "split_matrices": W.plan.split_matrices}
        W.close()
        del W
        torch.cuda.empty_cache()
        return out
    # end to end: activations from pinned host memory, outputs back to pinned host memory
    xh = torch.empty(W.x.numel(), dtype=torch.float32, pin_memory=True)
    xh.copy_(W.x.cpu())
    yh = torch.empty(W.y.numel(), dtype=torch.float32, pin_memory=True)

    # the public host-buffer call on one stream: the activations copied in, then the step,
    # whose outputs reach the pinned yh (stored there by the kernel for a one-stage plan,
    # copied back otherwise)
    def e2e_step():
        W.plan.step_host(xh, yh, W.x, W.y, W.ws, stream=stream)

    for _ in range(3):
        e2e_step()
    e2e_steps = max(3, steps // 4)
    e2e_secs = _time_steps(e2e_step, e2e_steps, stream)
    out = {
        "config": config,
        "matrices": len(W.mats_spec),
        "weight_bytes": W.weight_bytes,
        "activation_bytes": W.activation_bytes,
        "bytes_per_step": bytes_per_step,
        "seconds": secs,
        "per_step_s": per_step,
        "gbs": bytes_per_step / per_step / 1e9,
        "e2e_per_step_s": e2e_secs / e2e_steps,
        "e2e_gbs": bytes_per_step / (e2e_secs / e2e_steps) / 1e9,
        "h2d_bytes": xh.numel() * 4,
        "d2h_bytes": yh.numel() * 4,
        "clocks": clocks,
        "step_stats": step_stats,
    }
    W.close()
    del W
    torch.cuda.empty_cache()
    return out


def _gemv_graph_measure(kq, wl_mod, fmt, n, k, m, stream, replays=20):
    """Per-launch time of a GEMV / small-M GEMM over enough rotated weight copies
    that the working set is at least four times the L2, launched from a CUDA graph."""
    import torch
    import synth

    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    W0 = wl_mod.build_matrix(fmt, n, k, 0, synth.stream_id("small_m" if m > 1 else
                                                             ("q8_0_gemv" if fmt == "q8_0" else "pq2_0_gemv"), 0, 0))
    copies = max(2, int(np.ceil(4 * l2 / W0.weight_bytes)))
    mats = [W0]
    for _ in range(copies - 1):
        Wc = kq.QMatrix(fmt, n, k)
        Wc.codes.copy_(W0.codes)
        Wc.scales.copy_(W0.scales)
        mats.append(Wc)
    X = wl_mod.build_activation(k, 0, 12345, rows=m)
    Y = torch.empty(m * n, dtype=torch.float32, device="cuda")
    nb = kq.kq_gemv_workspace_bytes(W0, m)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda") if nb else None

    gemv = {"pq2_0": kq.kq_gemv_pq2_0, "q8_0": kq.kq_gemv_q8_0, "scale4": kq.kq_gemv_scale4}[fmt]

    def launch(Wm, st):
        if m == 1:
            gemv(Wm, X, Y, ws, stream=st)
        else:
            kq.kq_gemm_small_m(Wm, X, m, Y, ws, stream=st)

    for Wm in mats[:3]:
        launch(Wm, stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for Wm in mats:
                launch(Wm, s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(replays):
        g.replay()
    end.record()
    torch.cuda.synchronize()
    per_launch = start.elapsed_time(end) / 1e3 / (replays * len(mats))
    nbytes = W0.weight_bytes + 4 * m * (k + n)
    if m >= (9 if fmt == "scale4" else 5):  # kq_gemm_small_m runs the tensor-core GEMM: prologue, GEMM, split pass
        split = kq.kq_gemm_tc_workspace_bytes(W0, m, 0) > kq.kq_gemm_tc_workspace_bytes(W0, m, 1)
        path, launches = "tcgen05", 2 + (1 if split else 0)
    else:
        path, launches = "stream", ((m + 3) // 4) * (1 + (1 if nb else 0))
        if m == 1 and ((fmt == "q8_0" and k <= 4096 and n * k <= 20 << 20) or
                       (fmt == "pq2_0" and k <= 5376 and n * k // 4 <= 16 << 20)):  # the library's one-launch GEMVs
            path = "direct"
    out = {"fmt": fmt, "n": n, "k": k, "m": m, "path": path, "us_per_call": per_launch * 1e6,
           "gbs": nbytes / per_launch / 1e9, "copies": copies, "launches_per_call": launches}
    if m > 1:
        out["tflops"] = 2.0 * m * n * k / per_launch / 1e12
    del g, mats
    torch.cuda.empty_cache()
    return out


CONTROL_RINGS = ((34816, 4), (69632, 2), (65536, 3))  # the Q8_0 and PQ2_0 stream-kernel rings, and a deeper one


def _control_measure(kq, nbytes, stream, reps=10):
    """Read-only streaming control (kq_stream_read) over nbytes, the same byte
    count as one decode step: the in-harness ceiling of a kernel that reads
    each byte once through shared memory.  Best of the ring shapes above; each
    timed over `reps` launches after warm-up (input far larger than L2)."""
    import torch

    nbytes = nbytes // 16 * 16
    src = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    src.fill_(0x5A)
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    by_ring = {}
    for stage_bytes, stages in CONTROL_RINGS:
        run = lambda: kq.kq_stream_read(src, nbytes, sink, stage_bytes=stage_bytes, stages=stages, stream=stream)
        for _ in range(3):
            run()
        secs = _time_steps(run, reps, stream)
        by_ring[f"{stages}x{stage_bytes}"] = round(nbytes / (secs / reps) / 1e9, 1)
    if kq.kq_device_status(True) != kq.KQ_OK:
        raise RuntimeError("device status not ok after the control kernel")
    del src
    torch.cuda.empty_cache()
    best = max(by_ring, key=by_ring.get)
    return {"kernel": "kq::stream_read_kernel (kq_stream_read)", "gbs": by_ring[best], "ring": best,
            "bytes": nbytes, "by_ring": by_ring}


def _head_kernel(args):
    if args.workload == SECONDARY:
        return "kq::stream_kernel<Q8_0,1> (one launch per step)"
    if args.pq2_0_consumer == "tcgen05":
        return "kq::tcs::tcs_kernel (tcgen05.mma kind::f8f6f4; one launch per step)"
    return "kq::stream_kernel<PQ2_0,1> (one launch per step)"


def run_kq(args):
    import torch

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import quantized_weight_streaming_gb300 as kq
    import workloads

    ver = kq.kq_kernel_binary_version()
    if ver != 103:
        raise SystemExit(f"refusing to measure: kernels loaded as sm_{ver}, not sm_103a")
    kq.kq_device_status(True)
    if args.pq2_0_consumer == "tcgen05":  # the headline line under the opt-in consumer (profiling cases)
        kq.kq_set_pq2_0_consumer(kq.KQ_PQ2_0_TCGEN05)
    stream = torch.cuda.current_stream()
    gpu_index = torch.cuda.current_device()
    head = _decode_measure(kq, workloads, args.workload, args.steps, args.warmup, stream, sampler_gpu=gpu_index,
                           world=world, limit=args.matrices, stats=True)
    peak, peak_kind = _peaks()
    control = _control_measure(kq, head["bytes_per_step"], stream) if rank == 0 else None
    extras = {}
    if not args.no_extras and rank == 0:
        sec = _decode_measure(kq, workloads, SECONDARY if args.workload != SECONDARY else HEADLINE,
                              max(3, args.steps // 2), args.warmup, stream)
        extras["decode_steps"] = {sec["config"]: {
            "gbs": round(sec["gbs"], 1), "us_per_step": round(sec["per_step_s"] * 1e6, 2),
            "frac_of_measured_hbm": round(sec["gbs"] / peak, 4),
            "frac_of_control": round(sec["gbs"] / control["gbs"], 4), "e2e_gbs": round(sec["e2e_gbs"], 1),
            "weight_bytes": sec["weight_bytes"], "matrices": sec["matrices"]}}
        # the same projections with the model's dependencies: stage by stage
        # (q/k/v -> o -> gate/up -> down -> next layer), one cooperative launch
        chain = {}
        for cfg in (HEADLINE, SECONDARY):
            ch = _decode_measure(kq, workloads, cfg, max(3, args.steps // 4), args.warmup, stream, linked=True,
                                 e2e=False)
            chain[cfg] = {"gbs": round(ch["gbs"], 1), "us_per_step": round(ch["per_step_s"] * 1e6, 2),
                          "frac_of_measured_hbm": round(ch["gbs"] / peak, 4),
                          "frac_of_control": round(ch["gbs"] / control["gbs"], 4), "stages": ch["stages"],
                          "split_matrices": ch["split_matrices"], "matrices": ch["matrices"]}
        extras["decode_chain"] = chain
        # more decode streams: the Qwen3-4B projections in scale4_gs32, and the
        # Bonsai step with the page's own rotation (n = 1024, a sign vector per K width)
        more = {}
        for key, cfg, rot in (("qwen3_4b_scale4_step", "qwen3_4b_scale4_step", None),
                              ("bonsai_27b_pq2_0_step_page_rotation", HEADLINE, "page")):
            r = _decode_measure(kq, workloads, cfg, max(3, args.steps // 4), args.warmup, stream, e2e=False,
                                rotation=rot)
            more[key] = {"gbs": round(r["gbs"], 1), "us_per_step": round(r["per_step_s"] * 1e6, 2),
                         "frac_of_measured_hbm": round(r["gbs"] / peak, 4),
                         "frac_of_control": round(r["gbs"] / control["gbs"], 4), "weight_bytes": r["weight_bytes"],
                         "matrices": r["matrices"]}
        # the same Bonsai step with the opt-in tcgen05 consumer of PQ2_0 at one row
        kq.kq_set_pq2_0_consumer(kq.KQ_PQ2_0_TCGEN05)
        try:
            r = _decode_measure(kq, workloads, HEADLINE, max(3, args.steps // 4), args.warmup, stream, e2e=False)
        finally:
            kq.kq_set_pq2_0_consumer(kq.KQ_PQ2_0_MMA_SYNC)
        more["bonsai_27b_pq2_0_step_tcgen05_consumer"] = {
            "gbs": round(r["gbs"], 1), "us_per_step": round(r["per_step_s"] * 1e6, 2),
            "frac_of_measured_hbm": round(r["gbs"] / peak, 4), "frac_of_control": round(r["gbs"] / control["gbs"], 4),
            "kernel": "kq::tcs::tcs_kernel (tcgen05.mma kind::f8f6f4)", "weight_bytes": r["weight_bytes"],
            "matrices": r["matrices"]}
        extras["decode_steps"].update(more)
        gemv = []
        for fmt, n, k, m in (("q8_0", 1024, 2560, 1), ("pq2_0", 10240, 5120, 1), ("q8_0", 9728, 2560, 1),
                             ("q8_0", 9728, 2560, 4), ("q8_0", 9728, 2560, 16), ("q8_0", 9728, 2560, 64),
                             ("pq2_0", 17408, 5120, 1), ("pq2_0", 17408, 5120, 4), ("pq2_0", 17408, 5120, 16),
                             ("pq2_0", 17408, 5120, 64), ("scale4", 9728, 2560, 1), ("scale4", 9728, 2560, 4),
                             ("scale4", 9728, 2560, 16), ("scale4", 9728, 2560, 64)):
            r = _gemv_graph_measure(kq, workloads, fmt, n, k, m, stream)
            gemv.append({key: (round(v, 3) if isinstance(v, float) else v) for key, v in r.items()})
        extras["gemv_graph"] = gemv
    per_gpu_gbs = head["gbs"]
    value = aggregate_gbs(head["bytes_per_step"], args.steps, head["seconds"], world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, budget_s=args.cpu_seconds)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(head["per_step_s"] * 1e3, 5),
        "us_per_step": round(head["per_step_s"] * 1e6, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": args.workload + (f" (first {args.matrices} projections)" if args.matrices else ""),
                   "matrices": head["matrices"], "weight_bytes": head["weight_bytes"],
                   "activation_bytes": head["activation_bytes"], "bytes_per_step": head["bytes_per_step"],
                   "l2": "inputs larger than L2 (weights streamed once per step, 50x the L2)",
                   "parallelism": f"replicas x{world}", "seed": 0, "pq2_0_consumer": args.pq2_0_consumer},
        "frac_of_measured_hbm": round(per_gpu_gbs / peak, 4),
        "frac_of_nominal_8tbs": round(per_gpu_gbs / 8000.0, 4),
        "frac_of_control": round(per_gpu_gbs / control["gbs"], 4) if control else None,
        "control": control,
        "roofline": {"bound": "hbm", "achieved": round(per_gpu_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(per_gpu_gbs / peak, 4),
                     "traffic": args.traffic if args.traffic is not None else (
                         _traffic(args.workload) if "stream_kernel" in _head_kernel(args) else None),
                     "peak_kind": peak_kind, "kernel": _head_kernel(args)},
        "e2e": {"value": round(head["e2e_gbs"] * world, 2), "unit": "GB/s", "h2d_bytes_per_step": head["h2d_bytes"],
                "d2h_bytes_per_step": head["d2h_bytes"], "us_per_step": round(head["e2e_per_step_s"] * 1e6, 2)},
        "gpu_launches": args.steps,
        "clocks": head["clocks"],
        "step_stats": head["step_stats"],
        "cpu_baseline": cpu,
    }
    if extras:
        line["extras"] = extras
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# oracle (CPU) arm
# ----------------------------------------------------------------------------

class OracleSample:
    """A bounded sample of a decode-step workload for the FP64 oracle: `rows`
    rows of every `stride`-th projection, quantized once (untimed); one step
    dequantizes the sampled rows, transforms the activation (PQ2_0) and runs
    the FP64 GEMV of each sampled projection."""

    def __init__(self, config, rows_per_matrix, stride=1, seed=0):
        import oracle
        import synth

        self.oracle = oracle
        self.config = config
        self.spec = synth.workload(config)
        self.rows = rows_per_matrix
        self.stride = stride
        self.items = []
        self.bytes = 0
        for i, (_, fmt, n, k) in enumerate(self.spec):
            if i % stride:
                continue
            rows = np.linspace(0, n - 1, num=min(rows_per_matrix, n)).astype(np.int64)
            w = synth.matrix_rows_host(n, k, rows, seed, synth.stream_id(config, synth.ROLE_W, i))
            x = synth.fill_host("x", k, seed, synth.stream_id(config, synth.ROLE_X, i))
            if fmt == "pq2_0":
                blocks = oracle.pq2_0_quantize(oracle.rotate_rows(w)[1])
            else:
                blocks = oracle.q8_0_quantize(w)
            self.items.append((fmt, rows.size, k, blocks, x))
            bs = 128 if fmt == "pq2_0" else 32
            self.bytes += rows.size * (k // (4 if fmt == "pq2_0" else 1) + 2 * k // bs) + 4 * (k + rows.size)

    def describe(self):
        which = "every projection" if self.stride == 1 else f"one projection in {self.stride}"
        return (f"{self.rows} rows of {len(self.items)} of the {len(self.spec)} projections of {self.config} "
                f"({which}; {self.bytes / 1e6:.2f} MB of the step's bytes)")

    def step(self):
        o = self.oracle
        for fmt, r, k, blocks, x in self.items:
            if fmt == "pq2_0":
                deq = o.pq2_0_dequant(blocks, r, k)
                x64 = o.rotate_rows(x)[0]
            else:
                deq = o.q8_0_dequant(blocks, r, k)
                x64 = x.astype(np.float64)
            o.gemv(deq, x64)


# One sizing rule for every timing of the oracle (the reference arm and the
# cpu_baseline leg): rows of every projection, as many as the step budget
# allows, at most this many (building a sample costs more than stepping it).
ORACLE_MAX_ROWS = 128


def _sized_sample(config, step_budget_s, max_rows=ORACLE_MAX_ROWS):
    """OracleSample whose step takes about step_budget_s on this host.  The
    per-row cost comes from two small probes (1 and 4 rows of every
    projection), so only one more sample is built; rows are capped at
    max_rows."""
    def timed(sample):
        sample.step()
        t0 = time.perf_counter()
        sample.step()
        return time.perf_counter() - t0

    t1 = timed(OracleSample(config, 1, 1))
    if t1 > step_budget_s:
        return OracleSample(config, 1, int(np.ceil(t1 / step_budget_s)))
    t4 = timed(OracleSample(config, 4, 1))
    per_row = max((t4 - t1) / 3.0, 1e-6)
    rows = int((step_budget_s - (t1 - per_row)) / per_row)
    return OracleSample(config, max(1, min(max_rows, rows)), 1)


def _step_bytes(config):
    """Algorithmic bytes of one whole step of a workload: packed weights (codes and
    fp16 scales) plus fp32 activations read and outputs written."""
    import synth

    total = 0
    for _, fmt, n, k in synth.workload(config):
        bs = 128 if fmt == synth.PQ2_0 else 32
        code = {synth.PQ2_0: n * k // 4, synth.Q8_0: n * k, synth.SCALE4: n * k // 2}[fmt]
        total += code + 2 * n * (k // bs) + 4 * (n + k)
    return total


def _cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform

    return platform.machine()


def cpu_baseline(config, budget_s=15.0):
    """The oracle as it stands, timed on the host cores on a bounded sample."""
    import oracle

    sample = _sized_sample(config, budget_s / 8)
    sample.step()
    reps, t0 = 0, time.perf_counter()
    while True:
        sample.step()
        reps += 1
        el = time.perf_counter() - t0
        if el > budget_s / 2 or reps >= 50:
            break
    per = el / reps
    out = {"value": round(sample.bytes / per / 1e9, 5), "unit": "GB/s", "cores": oracle.max_threads(),
           "kind": "oracle", "cpu_model": _cpu_model(),
           "s_per_step_equivalent": round(per * _step_bytes(config) / sample.bytes, 1),
           "sample": f"{sample.describe()}, {reps} timed passes of {per * 1e3:.1f} ms each "
                     f"(FP64 dequantize + transform + GEMV)"}
    # the same code on one core, on a sample sized for it
    cores = oracle.max_threads()
    oracle.set_threads(1)
    try:
        one = _sized_sample(config, budget_s / 16)
        one.step()
        reps, t0 = 0, time.perf_counter()
        while True:
            one.step()
            reps += 1
            el = time.perf_counter() - t0
            if el > budget_s / 4 or reps >= 20:
                break
    finally:
        oracle.set_threads(cores)
    per = el / reps
    out["single_core"] = {"value": round(one.bytes / per / 1e9, 5), "unit": "GB/s", "cores": 1,
                          "sample": f"{one.describe()}, {reps} timed passes of {per * 1e3:.1f} ms each"}
    return out


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle

    # size each step so that warm-up plus timed steps take about a minute
    sample = _sized_sample(args.workload, max(0.02, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        sample.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sample.step()
    secs = time.perf_counter() - t0
    per = secs / args.steps
    value = sample.bytes / per / 1e9
    desc = sample.describe() + " per step"
    rows = sample.rows
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(per * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "sample_rows_per_matrix": rows, "sample_matrix_stride": sample.stride,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle", "cores": oracle.max_threads(),
                         "cpu_model": _cpu_model(), "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def profile_gemm(spec):
    """Three kq_gemm_small_m calls on one synthetic matrix (for ncu captures of
    the GEMM kernels: -k regex:tc_gemm_kernel -s 2 -c 1)."""
    import torch
    import synth
    import quantized_weight_streaming_gb300 as kq
    import workloads

    fmt, n, k, m = spec.split(",")
    n, k, m = int(n), int(k), int(m)
    torch.cuda.set_device(0)
    W = workloads.build_matrix(fmt, n, k, 0, synth.stream_id("small_m", 0, 0))
    X = workloads.build_activation(k, 0, synth.stream_id("small_m", 1, 0), rows=m)
    Y = torch.empty(m * n, dtype=torch.float32, device="cuda")
    nbytes = kq.kq_gemv_workspace_bytes(W, m)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        kq.kq_gemm_small_m(W, X, m, Y, ws)
    torch.cuda.synchronize()
    if kq.kq_device_status(True) != kq.KQ_OK:
        raise SystemExit("device status not OK")
    print(json.dumps({"profile_gemm": spec, "ok": True}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("kq", "reference"), default="kq")
    ap.add_argument("--workload", default=HEADLINE, choices=(HEADLINE, SECONDARY))
    ap.add_argument("--no-extras", action="store_true", help="skip the secondary workload and GEMV lines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--matrices", type=int, default=None,
                    help="only the first N projections of the workload (small profiling cases)")
    ap.add_argument("--pq2-0-consumer", choices=("mma_sync", "tcgen05"), default="mma_sync",
                    help="consumer of PQ2_0 products at one activation row for the headline line")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the stream kernel from an ncu capture (reported as is)")
    ap.add_argument("--profile-gemm", default=None, metavar="FMT,N,K,M",
                    help="profiling case: build one N x K matrix and run kq_gemm_small_m with M rows three times")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.profile_gemm:
        profile_gemm(args.profile_gemm)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_kq(args)


if __name__ == "__main__":
    main()
