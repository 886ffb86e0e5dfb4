"""Benchmark of the codec's hot path on one GB300 (or N independent replicas).

One step = one pass of the whole path over one batch of synthetic input:
  K1  taco_compress       all simulated TP ranks (one launch, DELAYED dual-scale)
  K23 qar_reduce_requant  dequantize the N code planes, sum in FP32 and
                          requantize for the gather stage (one kernel); with
                          --path split: K2 qar_reduce + K3 qar_requant
  K4  taco_decompress     the gathered codes back to the 16-bit dtype
      taco_update_scale   both stages' per-tensor scales (one launch)
Metric: GB/s of 16-bit input processed (2 bytes x elements x ranks / step
time); "roofline" gives the fraction of the measured HBM bandwidth the
dominant kernel (K1) reaches.  The timed steps replay the step captured as
a CUDA graph (--no-graph: eager launches).  Per-kernel times come from a
graph of the same steps with a timing event between every two kernels,
replayed after the timed region (eager launches if that is unavailable).

The default run measures every target workload: the headline (--workload,
default the largest: 8 x [16384 x 8192] bf16, block-symmetric INT8) with
the end-to-end, CPU-baseline and roofline reports, then each other target
workload as its own report under "per_config" (the Qwen-style gradient
workload as 16 drifting per-step inputs resident in HBM and cycled), and
the K0 copy kernel on 1 GiB beside the measured copy peak.  The compress's
SM cap is chosen per workload from whole steps unless --k1-sms fixes it.
Optional reports: --ring (EQuARX adder chains and the hop kernels), --hop
(the hop kernels alone), --sm-sweep, --choose-block.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--per-config auto|none|a,b] [--impl qta|reference]

--gpus N without torchrun starts N local replica processes (one per GPU).
--impl reference times the CPU oracle (the plain single-threaded reference
implementation of the same path) on a bounded row sample of the workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import glob
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "fused compress + dequant-reduce GB/s of bf16 input; % of GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0

# Per-launch DRAM traffic (bytes read + written) of the dominant kernel from
# one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum), keyed by
# (kernel, workload) together with the digest of the CUDA sources it was
# measured on; a changed source makes it stale (null).
NCU_TRAFFIC = {
    ("taco_compress", "gpt_tp"): {"bytes": 536912128 + 236075264, "src": "ab617c98ab5262bf"},
    # captured on 4096 of the 16384 rows per rank; the input is read and the
    # codes written once per row, so a full launch moves four times as much
    ("taco_compress", "equarx_int8"): {"bytes": 4 * (536902912 + 250640896), "src": "ab617c98ab5262bf"},
    ("taco_compress", "qwen_grad"): {"bytes": 335590912 + 133776128, "src": "ab617c98ab5262bf"},
    # captured with the compress on all SMs; the bench runs it on 128, which
    # moves the same bytes
    ("taco_compress", "flash_int4"): {"bytes": 1073914368 + 265253376, "src": "ab617c98ab5262bf"},
}


def _roofline(w, kern, alg, peak_info) -> dict:
    """K1 against the measured copy peak: algorithmic bytes / event time, with
    the ncu DRAM traffic of one launch while the sources keep its digest."""
    peak, peak_kind = peak_info
    achieved = alg["K1"] / (kern["K1"]["ms"] * 1e-3) / 1e9
    tr = NCU_TRAFFIC.get(("taco_compress", w.name))
    traffic = tr["bytes"] if tr and tr.get("src") == _src_digest() else None
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "kernel": "K1 taco_compress", "peak_source": f"{peak_kind} hbm_gbs",
            "algorithmic_bytes": alg["K1"]}


def _src_digest() -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "quantized_tensor_activation_gb300", "csrc", "*"))):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    return ws, rank


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        if self.idx is None:
            return
        try:
            fd, self.path = tempfile.mkstemp(prefix="qta_clocks_", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.STDOUT)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            raw = f.read()
        for line in raw.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"error": "no nvidia-smi samples", "gpu": str(self.idx), "output": raw[:200]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def _smi_gpu_id(torch, local: int) -> str:
    """The identifier nvidia-smi needs for the device this process uses."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        tok = vis.split(",")[local].strip()
        if tok:
            return tok
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        return str(local)


def max_over_ranks(value: float, device="cpu") -> float:
    """The largest value over all ranks of the process group (the value itself
    without one): the job's step time is that of its slowest replica."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: float, ms_step_max: float, world_size: int) -> float:
    """Whole-job GB/s of 16-bit input: every replica processes its own batch
    in the same (slowest-rank) step time."""
    return bytes_per_rank_step * world_size / (ms_step_max * 1e-3) / 1e9


def _cpu_oracle_path(w: workloads.Workload, rows: int, seed: int = 0):
    """The oracle's full path over a row sample of every rank; returns
    (seconds, 16-bit input bytes processed, threads used)."""
    import numpy as np
    import torch

    import oracle as orc
    torch.set_num_threads(1)
    x = workloads.make_rank_inputs(w, rows=rows, seed=seed)
    xb = x.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    sch = {"taco_fp8": orc.TACO_FP8, "int8_sym": orc.INT8_SYM, "int4_asym": orc.INT4_ASYM,
           "int8_asym": orc.INT8_ASYM}
    s1, s2 = sch[w.scheme], sch[w.gather_scheme]
    N, C, B, gB = w.ranks, w.cols, w.block, w.gather_block
    dt = orc.BF16 if w.dtype == "bf16" else orc.FP16
    E = rows * C
    t0 = time.perf_counter()
    st = np.zeros(2 * N, dtype=np.float32) if s1 == orc.TACO_FP8 else None
    c, s, z = orc.compress(s1, B, xb, dt, N, rows, C, st, orc.CURRENT)
    t1 = time.perf_counter()
    cb = E // 2 if s1 == orc.INT4_ASYM else E
    nb = E // B
    shards = [(c[r * cb:(r + 1) * cb], s[r * nb:(r + 1) * nb], None if z is None else z[r * nb:(r + 1) * nb],
               None if st is None else st[2 * r:2 * r + 2]) for r in range(N)]
    gr = max(1, rows // N)
    st2 = np.zeros(2 * N, dtype=np.float32) if s2 == orc.TACO_FP8 else None
    c2, sc2, z2 = orc.reduce_requant(s1, B, shards, rows, C, 0, N * gr, s2, gB, N, st2, orc.CURRENT)
    t2 = time.perf_counter()
    orc.decompress(s2, gB, c2, sc2, z2, st2, N, gr, C, dt)
    t3 = time.perf_counter()
    _cpu_oracle_path.stages = {"compress_s": t1 - t0, "reduce_requant_s": t2 - t1, "decompress_s": t3 - t2}
    return t3 - t0, 2 * E * N, 1


def _host_cpu():
    """The host's logical CPU count and model name (for the CPU-baseline report)."""
    model = platform.processor() or platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model}


def run_reference(args, w):
    ws, rank = _dist()
    if rank != 0:
        return
    rows = args.ref_rows
    _cpu_oracle_path(w, 8)  # build / warm the oracle
    times = []
    for i in range(args.warmup + args.steps):
        dt_s, nbytes, threads = _cpu_oracle_path(w, rows, seed=i)
        if i >= args.warmup:
            times.append(dt_s)
    t = sum(times) / len(times)
    val = nbytes / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": _config(w),
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} of {w.rows} rows of each of the {w.ranks} ranks per step "
                                   f"({w.ranks * rows * w.cols} elements), full path",
                         "stages": dict(_cpu_oracle_path.stages), "host": _host_cpu()},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(w):
    return {"workload": f"{w.name}: {w.description}", "ranks": w.ranks, "rows": w.rows, "cols": w.cols,
            "input_dtype": w.dtype, "scheme": w.scheme, "block": w.block, "gather_scheme": w.gather_scheme,
            "gather_block": w.gather_block,
            "l2": "inputs larger than L2 (%.0f MB of 16-bit input per step)" % (2 * w.elems_per_rank * w.ranks / 1e6)}


def algorithmic_bytes(w):
    """Bytes each kernel must move once per step (inputs read once, outputs
    written once)."""
    E, N = w.elems_per_rank, w.ranks

    def codes(s):
        return 0.5 if s == "int4_asym" else 1.0

    def meta(s, b):
        return {"taco_fp8": 1.0, "int8_sym": 4.0, "int4_asym": 4.0, "int8_asym": 4.0}[s] / b

    k1 = N * E * (2 + codes(w.scheme) + meta(w.scheme, w.block))
    k2 = N * E * (codes(w.scheme) + meta(w.scheme, w.block)) + E * 4
    k3 = E * (4 + codes(w.gather_scheme) + meta(w.gather_scheme, w.gather_block))
    k23 = k2 - E * 4 + k3 - E * 4
    k4 = E * (codes(w.gather_scheme) + meta(w.gather_scheme, w.gather_block) + 2)
    return {"K1": k1, "K2": k2, "K3": k3, "K23": k23, "K4": k4}


def ring_report(qta, w, x, steps: int, peak: float):
    """EQuARX full-loop and semi-loop adder chains (ring reduce-scatter with
    the partial sum requantized at every hop, then the quantized all-gather)
    over the workload's ranks: time of the reduce-scatter chains (CUDA events,
    eager launches) and mean squared errors against the float64 sums."""
    import torch
    from quantized_tensor_activation_gb300 import ring

    N, R, C = x.shape
    d = qta.desc(w.scheme, w.block, R, C)
    rc = R // N
    exact = x.double().sum(dim=0)
    out = {"ranks": N, "shape": [R, C], "scheme": w.scheme, "block": w.block,
           "note": "chunk j owned by rank j; CURRENT scale per hop for TACO; MSE vs the float64 sum"}
    for semi in (False, True):
        name = "semi_loop" if semi else "full_loop"
        ring.reduce_scatter(d, x, semi)                      # warm-up
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            ring.reduce_scatter(d, x, semi)
        b.record()
        torch.cuda.synchronize()
        s, y = ring.allreduce(d, x, semi, torch.float32)
        e_rs = s.double() - exact
        e_ar = y.double() - exact
        out[name] = {"reduce_scatter_ms": a.elapsed_time(b) / steps,
                     "requantizations_per_chunk": max(len(c) for c in ring.chunk_orders(N, 0, semi)),
                     "reduce_scatter_mse": float((e_rs * e_rs).mean()),
                     "allreduce_mse": float((e_ar * e_ar).mean())}
        del s, y, e_rs, e_ar
    # error of the full-loop partial sums after each hop
    parts = []
    ring.reduce_scatter(d, x, False, hop_partials=parts)
    per_hop = []
    for k, p in enumerate(parts):
        err = 0.0
        for j in range(N):
            ranks = [(j + i) % N for i in range(1, k + 2)]
            ex = x[ranks, j * rc:(j + 1) * rc].double().sum(dim=0)
            e = p[j * rc:(j + 1) * rc].double() - ex
            err += float((e * e).sum())
        per_hop.append(err / (R * C))
    out["full_loop"]["mse_after_hop"] = per_hop
    del parts
    out["hop_kernel"] = hop_kernel_report(qta, w, x, peak)
    assert qta.qta_device_error() == 0
    return out


def hop_kernel_report(qta, w, x, peak: float, iters: int = 10):
    """The ring's inner call on a whole rank tensor, for its roofline: rank
    1's codes as the incoming partial sum, rank 0's tensor as the local
    addend.  CUDA events around each call; a 256 MB write between calls
    flushes L2.  Algorithmic bytes: the incoming codes and metadata, the local
    tensor, and the output (codes and metadata, or the FP32 sum)."""
    import torch

    N, R, C = x.shape
    dev = x.device
    dt = {torch.bfloat16: qta.BF16, torch.float16: qta.FP16, torch.float32: qta.FP32}[x.dtype]
    d = qta.desc(w.scheme, w.block, R, C)
    qin = qta.alloc_qtensor(d, dev)
    qta.taco_compress(d, x[1], dt, qin, qta.SCALE_CURRENT)
    qout = qta.alloc_qtensor(d, dev)
    qta.qar_dequant_add_requant(d, qin, x[0], dt, qout, qta.SCALE_CURRENT)
    if qout.state is not None:
        qta.taco_update_scale(qout.state, 1)        # S from this tensor: DELAYED from here on
    s = torch.empty((R, C), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    E = R * C
    q_bytes = qta.codes_bytes(d) + qta.scales_bytes(d) + qta.zeros_bytes(d)
    x_bytes = E * x.element_size()
    calls = {
        "qar_dequant_add_requant": (lambda: qta.qar_dequant_add_requant(d, qin, x[0], dt, qout, qta.SCALE_DELAYED),
                                    2 * q_bytes + x_bytes),
        "qar_dequant_add": (lambda: qta.qar_dequant_add(d, qin, x[0], dt, s), q_bytes + x_bytes + 4 * E),
    }
    rep = {"shape": [R, C], "note": "one call over a whole rank tensor; L2 flushed between calls"}
    for name, (fn, nbytes) in calls.items():
        fn()
        total = 0.0
        for _ in range(iters):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            total += a.elapsed_time(b)
        ms = total / iters
        rep[name] = {"ms": ms, "gb_s": nbytes / (ms * 1e-3) / 1e9, "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / peak,
                     "algorithmic_bytes": nbytes}
    del flush, s, qin, qout
    return rep


def _cpu_rows(w, target_elems: int) -> int:
    """Rows per rank of a bounded oracle sample of about target_elems
    elements over all ranks (a multiple of the rank count, at least one row
    per gather shard)."""
    rows = max(w.ranks, int(target_elems // (w.ranks * w.cols)))
    rows = min(w.rows, rows - rows % w.ranks)
    return max(rows, w.ranks)


def cpu_baseline(w, rows: int, seed: int, min_s: float = 0.0, max_reps: int = 8):
    """The oracle's whole path on a row sample of every rank, repeated on new
    seeds until min_s seconds of CPU work are reached (at most max_reps)."""
    total_s, total_b, reps = 0.0, 0, 0
    stages = {}
    while reps < max_reps and (reps == 0 or total_s < min_s):
        dt_s, nbytes, threads = _cpu_oracle_path(w, rows, seed=seed + reps)
        total_s += dt_s
        total_b += nbytes
        reps += 1
        for k, v in _cpu_oracle_path.stages.items():
            stages[k] = stages.get(k, 0.0) + v
    return {"value": total_b / total_s / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} of {w.rows} rows of each of the {w.ranks} ranks "
                      f"({w.ranks * rows * w.cols} elements), full path, {reps} pass(es) on different seeds, "
                      f"{total_s:.1f} s",
            "stages": stages, "host": _host_cpu()}


def measure_workload(qta, w, args, dev, ws: int, local: int, headline: bool) -> dict:
    """Time the whole hot path on one workload: K1 taco_compress (all ranks),
    K23 qar_reduce_requant (or K2 + K3), K4 taco_decompress and the state
    update, as one captured CUDA graph per step.  A workload with a per-step
    magnitude drift keeps one input per step resident in HBM and cycles
    through them, so every timed step compresses a new tensor with the
    per-tensor scales the previous step left.  Returns the per-workload
    report (times are the max over ranks)."""
    import torch

    sch = qta.SCHEMES
    N, R, C = w.ranks, w.rows, w.cols
    in_dt = qta.BF16 if w.dtype == "bf16" else qta.FP16
    tdt = w.torch_dtype
    n_in = max(1, w.steps)
    # inputs resident in HBM: [N, R, C] per step
    xs = [workloads.make_rank_inputs(w, device=dev, seed=args.seed, step=k) for k in range(n_in)]
    d_in = qta.desc(sch[w.scheme], w.block, R, C, batch=N, max_sms=max(args.k1_sms, 0))
    d_sh = qta.desc(sch[w.scheme], w.block, R, C)
    d_g = qta.desc(sch[w.gather_scheme], w.gather_block, R // N, C, batch=N)
    taco1 = w.scheme == "taco_fp8"
    taco2 = w.gather_scheme == "taco_fp8"
    q = qta.alloc_qtensor(d_in, dev)
    g = qta.alloc_qtensor(d_g, dev)
    # both stages' per-tensor states live in one buffer so that one
    # taco_update_scale launch ends the step
    n_state = (N if taco1 else 0) + (N if taco2 else 0)
    states = torch.zeros(2 * max(n_state, 1), dtype=torch.float32, device=dev)
    states[0::2] = 1.0
    off = 0
    if taco1:
        q.state = states[0:2 * N]
        off = 2 * N
    if taco2:
        g.state = states[off:off + 2 * N]
    shards = [q.shard(r) for r in range(N)]
    ssum = torch.empty((R, C), dtype=torch.float32, device=dev)
    y = torch.empty((R, C), dtype=tdt, device=dev)
    stream = torch.cuda.current_stream()
    launches = [0]
    counter = [0]            # steps issued so far: step i compresses input i mod n_in

    def step(first=False, ev=None, fused=True, i=None):
        # each compress uses the per-tensor scale left by the previous step and
        # accumulates this step's amax; the receiving side dequantizes with the
        # same scale, so the states are updated once, at the end of the step.
        # Events go on the current stream (the capture stream while a CUDA
        # graph of the step is recorded).
        if i is None:
            i = counter[0]
            counter[0] += 1
        x = xs[i % n_in]
        mode = qta.SCALE_CURRENT if first else qta.SCALE_DELAYED
        if ev:
            ev[0].record()
        qta.taco_compress(d_in, x, in_dt, q, mode)
        if ev:
            ev[1].record()
        if fused:
            qta.qar_reduce_requant(d_sh, shards, 0, R, d_g, g, mode)
            if ev:
                ev[2].record()
                ev[3].record()
        else:
            qta.qar_reduce(d_sh, shards, 0, R, ssum)
            if ev:
                ev[2].record()
            qta.qar_requant(d_g, ssum, g, mode)
            if ev:
                ev[3].record()
        qta.taco_decompress(d_g, g, y, in_dt)
        if ev:
            ev[4].record()
        if n_state:
            qta.taco_update_scale(states, n_state)
        if ev:
            ev[5].record()
            ev[6].record()          # an interval with no kernel: the cost of the event nodes themselves
        launches[0] += (3 if fused else 4) + int(n_state > 0)

    fused = args.path == "fused"
    # warm-up (first step in CURRENT mode, the rest as timed), both paths
    step(first=True, fused=fused)
    for _ in range(max(args.warmup, 3) - 1):
        step(fused=fused)
        step(fused=not fused)
    torch.cuda.synchronize()
    assert qta.qta_device_error() == 0

    # the compress's SM cap (qta_desc.max_sms): fixed by --k1-sms >= 0, else
    # the fastest of a few candidates on whole eager steps (inside the step
    # the compress overlaps the write-back of the previous kernels' dirty L2
    # lines, and leaving some SMs idle can shorten it)
    k1_tune = None
    if args.k1_sms < 0:
        k1_tune = {}
        for _ in range(2):
            for cap in (0, 144, 136, 128):
                d_in.max_sms = cap
                step(fused=fused)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(5):
                    step(fused=fused)
                b.record(stream)
                torch.cuda.synchronize()
                ms = a.elapsed_time(b) / 5
                k1_tune[cap] = min(ms, k1_tune.get(cap, ms))
        d_in.max_sms = min(k1_tune, key=lambda c: (k1_tune[c], c != 0))
    k1_cap = d_in.max_sms

    # a load window of about 0.6 s on each side of the timed region, so that
    # nvidia-smi samples the clocks under the same continuous load
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(3):
        step(fused=fused)
    b.record(stream)
    torch.cuda.synchronize()
    pad = 0 if args.no_clocks else max(1, int(600.0 / max(a.elapsed_time(b) / 3, 1e-3)))

    def timed(fused_path):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        launches[0] = 0
        t0.record(stream)
        for i in range(args.steps):
            step(ev=evs[i], fused=fused_path)
        t1.record(stream)
        return evs, t0, t1, launches[0]

    # the step as CUDA graphs, one per resident input (kernel parameters,
    # tensor maps included, are fixed at capture; every replay recomputes
    # the whole step)
    graphs = None
    if not args.no_graph:
        graphs = []
        for k in range(n_in):
            gr_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr_):
                step(fused=fused, i=k)
            graphs.append(gr_)
        for gr_ in graphs:
            gr_.replay()
        torch.cuda.synchronize()
    replays = [0]

    def run_step():
        if graphs is not None:
            graphs[replays[0] % n_in].replay()
            replays[0] += 1
        else:
            step(fused=fused)

    # the timed steps as one CUDA graph with a timing event between every two
    # kernels (event record nodes): the per-kernel times then come from steps
    # like the timed ones, free of host launch gaps
    graph_event_error = [None]

    def graph_with_events(fused_path):
        try:
            evl = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(7)]
                   for _ in range(args.steps)]
            gr_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr_):
                for i in range(args.steps):
                    step(ev=evl[i], fused=fused_path, i=i)
            gr_.replay()
            torch.cuda.synchronize()
            evl[0][0].elapsed_time(evl[0][1])
            return gr_, evl
        except (TypeError, RuntimeError) as e:
            graph_event_error[0] = f"{type(e).__name__}: {str(e).splitlines()[0][:160]}"
            return None, None

    tgraph, tevs = (None, None) if args.no_graph else graph_with_events(fused)

    # ---- timed region: inputs resident in HBM
    clocks = ClockSampler(None if args.no_clocks else _smi_gpu_id(torch, local))
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    if not args.no_clocks:
        time.sleep(0.3)
    for _ in range(pad):
        run_step()
    if ws > 1:
        torch.cuda.synchronize()
        torch.distributed.barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        run_step()
    t_end.record(stream)
    n_launch = args.steps * ((3 if fused else 4) + int(n_state > 0))
    for _ in range(pad):
        run_step()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if clk is not None:
        clk["window"] = (f"sampled every 100 ms over {2 * pad + args.steps} back-to-back steps around and "
                         f"including the timed ones")
    ms_step = max_over_ranks(t_start.elapsed_time(t_end) / args.steps, dev)
    events_ms = None
    if tgraph is not None:
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        tgraph.replay()
        p1.record(stream)
        torch.cuda.synchronize()
        events_ms = p0.elapsed_time(p1) / args.steps

    # per-kernel times: from the event graph, else from eager steps with events
    evs, e0, e1, _ = timed(fused)
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / args.steps
    if tevs is not None:
        evs = tevs
    # the other path (two calls, FP32 sum through HBM), for comparison
    g2, evs2 = (None, None) if args.no_graph else graph_with_events(not fused)
    if g2 is not None:
        s2a, s2b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2a.record(stream)
        g2.replay()
        s2b.record(stream)
    else:
        evs2, s2a, s2b, _ = timed(not fused)
    torch.cuda.synchronize()
    other_ms = s2a.elapsed_time(s2b) / args.steps
    del g2
    assert qta.qta_device_error() == 0

    # the same step with every call capped to a number of SMs (eager launches)
    sweep_raw = []
    if headline and args.sm_sweep:
        for n_sms in [int(v) for v in args.sm_sweep.split(",")]:
            for dd in (d_in, d_sh, d_g):
                dd.max_sms = n_sms
            timed(fused)
            evs3, s3a, s3b, _ = timed(fused)
            torch.cuda.synchronize()
            sweep_raw.append((n_sms, s3a.elapsed_time(s3b) / args.steps, evs3))
        d_in.max_sms, d_sh.max_sms, d_g.max_sms = k1_cap, 0, 0
        assert qta.qta_device_error() == 0

    # ---- end to end through the public API with host buffers (headline)
    e2e = None
    if headline and not args.no_e2e:
        xh = [x.cpu().pin_memory() for x in xs]
        yh = [torch.empty((R, C), dtype=tdt).pin_memory() for _ in range(2)]
        # double-buffered: the upload of step i+1 runs on its own copy stream
        # while step i computes and downloads its result
        xd = [torch.empty_like(xs[0]) for _ in range(2)]
        yd = [y, torch.empty_like(y)]
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        x_free = [torch.cuda.Event() for _ in range(2)]    # the step that last read xd[b] has compressed it
        y_free = [torch.cuda.Event() for _ in range(2)]    # yd[b] has been copied to the host
        for ev in x_free + y_free:
            ev.record(stream)
        torch.cuda.synchronize()

        def e2e_step(i):
            bi = i % 2
            h2d.wait_event(x_free[bi])
            with torch.cuda.stream(h2d):
                xd[bi].copy_(xh[i % n_in], non_blocking=True)
            arrived = torch.cuda.Event()
            arrived.record(h2d)
            stream.wait_event(arrived)
            qta.taco_compress(d_in, xd[bi], in_dt, q, qta.SCALE_DELAYED)
            x_free[bi].record(stream)
            if fused:
                qta.qar_reduce_requant(d_sh, shards, 0, R, d_g, g, qta.SCALE_DELAYED)
            else:
                qta.qar_reduce(d_sh, shards, 0, R, ssum)
                qta.qar_requant(d_g, ssum, g, qta.SCALE_DELAYED)
            stream.wait_event(y_free[bi])
            qta.taco_decompress(d_g, g, yd[bi], in_dt)
            if n_state:
                qta.taco_update_scale(states, n_state)
            done = torch.cuda.Event()
            done.record(stream)
            d2h.wait_event(done)
            with torch.cuda.stream(d2h):
                yh[bi].copy_(yd[bi], non_blocking=True)
            y_free[bi].record(d2h)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k = max(4, args.steps // 2)
        a.record(stream)
        h2d.wait_event(a)
        for i in range(k):
            e2e_step(i)
        for ev in y_free:
            stream.wait_event(ev)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / k, dev)
        e2e = {"value": 2 * N * R * C / (e2e_ms * 1e-3) / 1e9 * ws, "unit": "GB/s",
               "h2d_bytes_per_step": xs[0].numel() * xs[0].element_size(),
               "d2h_bytes_per_step": y.numel() * y.element_size(), "ms_per_step": e2e_ms,
               "pipeline": "inputs and outputs double-buffered: the upload of step i+1 overlaps step i's "
                           "kernels and download; each step copies its own inputs in and its result out"}
        del xh, yh, xd, yd

    in_bytes = 2 * N * R * C
    value = job_throughput(in_bytes, ms_step, ws)
    peak, peak_kind = _peaks()
    alg = algorithmic_bytes(w)

    def kernel_table(ev_list, fused_path):
        per_k = {k: [] for k in ("K1", "K2", "K3", "K4", "U", "E")}
        for e in ev_list:
            for j, k in enumerate(per_k):
                per_k[k].append(e[j].elapsed_time(e[j + 1]))
        ev_ms = statistics.mean(per_k["E"])
        names = {"K1": "taco_compress", "K2": "qar_reduce_requant" if fused_path else "qar_reduce",
                 "K3": None if fused_path else "qar_requant", "K4": "taco_decompress"}
        table = {}
        for k in ("K1", "K2", "K3", "K4"):
            if names[k] is None:
                continue
            ms = statistics.mean(per_k[k])
            nbytes = alg["K23"] if (k == "K2" and fused_path) else alg[k]
            net = max(ms - ev_ms, 1e-6)
            table[k] = {"call": names[k], "ms": ms, "gb_s": nbytes / (ms * 1e-3) / 1e9,
                        "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / peak, "algorithmic_bytes": nbytes,
                        "frac_of_hbm_net": nbytes / (net * 1e-3) / 1e9 / peak}
        table["U"] = {"call": "taco_update_scale" if n_state else None, "ms": statistics.mean(per_k["U"])}
        table["event_interval_ms"] = ev_ms
        table["note"] = ("ms: between the kernel's two event nodes; event_interval_ms: two consecutive event "
                         "nodes with no kernel between them, in the same graph; frac_of_hbm_net uses ms minus it")
        return table

    kern = kernel_table(evs, fused)
    step_bytes = alg["K1"] + alg["K4"] + (alg["K23"] if fused else alg["K2"] + alg["K3"])

    # reconstruction error of one step's output against the exact sum of the
    # ranks' inputs (float64), and of one rank's compress -> decompress
    recon = None
    if not args.no_recon:
        step(fused=fused, i=0)
        with torch.no_grad():
            x0 = xs[0]
            exact = x0.double().sum(dim=0)
            err = y.double() - exact
            mse = float((err * err).mean())
            d0 = qta.desc(sch[w.scheme], w.block, R, C)
            y0 = torch.empty((R, C), dtype=torch.float32, device=dev)
            qta.taco_decompress(d0, shards[0], y0, qta.FP32)
            e0 = y0.double() - x0[0].double()
            recon = {"allreduce_mse": mse, "allreduce_nmse": mse / float((exact * exact).mean()),
                     "stage1_mse_rank0": float((e0 * e0).mean()),
                     "stage1_nmse_rank0": float((e0 * e0).mean()) / float((x0[0].double() ** 2).mean()),
                     "note": "output of one step (input 0, DELAYED scales) vs the float64 sum of the 16-bit "
                             "inputs"}
            del exact, err, e0, y0
        torch.cuda.synchronize()
        assert qta.qta_device_error() == 0

    # K4 beside the plain copy kernel K0 moving the same number of bytes (half
    # read, half written), both timed the same way: single launches after an
    # L2 flush that only reads (so that no dirty lines are left to write
    # back), mean of 40 CUDA-event intervals each
    k4_copy = None
    if not getattr(args, "no_k0", False):
        nb = (int(alg["K4"]) // 2) & ~4095
        csrc_ = torch.empty(nb, dtype=torch.uint8, device=dev)
        cdst = torch.empty_like(csrc_)
        flush_buf = torch.ones(64 << 20, dtype=torch.float32, device=dev)

        def single_ms(fn, reps=40):
            fn()
            ts = []
            for _ in range(reps):
                flush_buf.sum()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
            return statistics.mean(ts)

        k4_ms = single_ms(lambda: qta.taco_decompress(d_g, g, y, in_dt))
        k0_ms = single_ms(lambda: qta.qta_copy(csrc_, cdst, nb))
        k4_copy = {"k4_bytes": alg["K4"], "k4_ms": k4_ms, "k4_gb_s": alg["K4"] / (k4_ms * 1e-3) / 1e9,
                   "k0_bytes": 2 * nb, "k0_ms": k0_ms, "k0_gb_s": 2 * nb / (k0_ms * 1e-3) / 1e9,
                   "note": "single launches after a 256 MB read-only L2 flush, mean of 40 CUDA-event intervals; "
                           "K0 (qta_copy) copies k0_bytes / 2"}
        del csrc_, cdst, flush_buf
        assert qta.qta_device_error() == 0

    rep = {
        "config": _config(w),
        "ms_per_step": ms_step,
        "value": value,
        "unit": "GB/s",
        "step_frac_of_hbm": step_bytes / (ms_step * 1e-3) / 1e9 / peak,
        "kernels": kern,
        "k1_sms": {"k1_max_sms": k1_cap or "all",
                   "k1_sms_choice": ("fixed" if k1_tune is None else
                                     "fastest eager step of " + ", ".join(
                                         f"{c or 'all'}: {t * 1e3:.1f} us" for c, t in k1_tune.items()))},
        "path": "fused reduce+requant (qar_reduce_requant)" if fused else "qar_reduce + qar_requant",
        "launch": (f"CUDA graph of one step, replayed ({n_in} graphs, one per resident input)" if n_in > 1
                   else "CUDA graph of one step, replayed") if graphs is not None else "eager",
        "kernel_times": ("events between the kernels inside a CUDA graph of the same steps, replayed after "
                         "the timed region" if tevs is not None else
                         "eager step with events" + (f" (graph events unavailable: {graph_event_error[0]})"
                                                     if graph_event_error[0] else "")),
        "ms_per_step_graph_with_events": events_ms,
        "eager_ms_per_step": eager_ms,
        "other_path": {"path": "qar_reduce + qar_requant" if fused else "qar_reduce_requant",
                       "ms_per_step": other_ms, "value": in_bytes / (other_ms * 1e-3) / 1e9 * ws,
                       "kernels": kernel_table(evs2, not fused)},
        "recon": recon,
        "k4_beside_copy": k4_copy,
        "clocks": clk,
        "gpu_launches": n_launch,
        "inputs": (f"{n_in} per-step inputs resident in HBM ({n_in * in_bytes / 1e9:.2f} GB), cycled: step i "
                   f"compresses input i mod {n_in}, each drawn with its own magnitude factor" if n_in > 1
                   else f"one input resident in HBM ({in_bytes / 1e9:.2f} GB of 16-bit values)"),
        "_alg": alg, "_peak": (peak, peak_kind), "_e2e": e2e, "_sweep": sweep_raw,
        "_kernel_table": kernel_table, "_fused": fused,
    }
    if headline:
        rep["_keep"] = (xs, shards, q)
    else:
        del xs, q, g, shards, ssum, y, states
    del graphs, tgraph
    return rep


def ash_report(qta, dev, names=("gpt_tp", "flash_int4"), iters: int = 10) -> dict:
    """The adaptive rescaling of the ASH transform against the plain one: on
    each workload's full-size rank tensors, compressed with TACO FP8 (B = 128,
    CURRENT scale), the per-channel factors from the channel amax over all
    ranks; MSE of one rank's round trip and of the all-reduce (compress all
    ranks, fused reduce + requant into the gather stage, decompress) against
    the float64 inputs / sum, with and without the factors, and the compress
    time with and without them (CUDA events, 10 calls)."""
    import torch

    out = {"note": "TACO FP8 B128 on the workload's tensors (whatever its own scheme); factors from "
                   "taco_channel_amax over all ranks + taco_ash_update"}
    for name in names:
        w = workloads.WORKLOADS[name]
        N, R, C = w.ranks, w.rows, w.cols
        dt = qta.BF16 if w.dtype == "bf16" else qta.FP16
        x = workloads.make_rank_inputs(w, device=dev, seed=3)
        d = qta.desc(qta.TACO_FP8, 128, R, C, batch=N)
        chan = qta.alloc_chan(C, dev)
        qta.taco_channel_amax(d, x, dt, chan)
        qta.taco_ash_update(chan, C)
        e = torch.log2(chan[C:2 * C]).round().to(torch.int64).cpu()
        rep = {"channels_rescaled": int((e > 0).sum()), "factor_histogram": torch.bincount(e, minlength=4).tolist()}
        exact = x.double().sum(dim=0)
        for tag, ch in (("plain", None), ("rescaled", chan)):
            q = qta.alloc_qtensor(d, dev)
            q.chan = ch
            qta.taco_compress(d, x, dt, q, qta.SCALE_CURRENT)
            y0 = torch.empty((R, C), dtype=torch.float32, device=dev)
            qta.taco_decompress(qta.desc(qta.TACO_FP8, 128, R, C), q.shard(0), y0, qta.FP32)
            dg = qta.desc(qta.TACO_FP8, 128, R // N, C, batch=N)
            g = qta.alloc_qtensor(dg, dev)
            g.chan = ch
            qta.qar_reduce_requant(qta.desc(qta.TACO_FP8, 128, R, C), [q.shard(r) for r in range(N)], 0, R, dg, g,
                                   qta.SCALE_CURRENT)
            y = torch.empty((R, C), dtype=torch.float32, device=dev)
            qta.taco_decompress(dg, g, y, qta.FP32)
            e0 = y0.double() - x[0].double()
            ea = y.double() - exact
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(iters):
                qta.taco_compress(d, x, dt, q, qta.SCALE_DELAYED)
            b.record()
            torch.cuda.synchronize()
            rep[tag] = {"round_trip_mse_rank0": float((e0 * e0).mean()), "allreduce_mse": float((ea * ea).mean()),
                        "compress_ms": a.elapsed_time(b) / iters}
            del q, g, y0, y, e0, ea
        rep["round_trip_mse_ratio"] = rep["rescaled"]["round_trip_mse_rank0"] / rep["plain"]["round_trip_mse_rank0"]
        rep["allreduce_mse_ratio"] = rep["rescaled"]["allreduce_mse"] / rep["plain"]["allreduce_mse"]
        out[name] = rep
        del x, exact, chan
        torch.cuda.empty_cache()
    assert qta.qta_device_error() == 0
    return out


def copy_probe(qta, dev, nbytes: int = 1 << 30, iters: int = 10) -> dict:
    """K0: the plain copy kernel (qta_copy) over nbytes (larger than L2),
    mean of iters calls timed with CUDA events after warm-up."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    src.random_(0, 255)
    dst = torch.empty_like(src)
    for _ in range(3):
        qta.qta_copy(src, dst, nbytes)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        qta.qta_copy(src, dst, nbytes)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / iters
    ok = bool(torch.equal(src, dst))
    del src, dst
    peak, kind = _peaks()
    gbs = 2 * nbytes / (ms * 1e-3) / 1e9
    return {"kernel": "K0 qta_copy", "bytes_copied": nbytes, "ms": ms, "gb_s": gbs,
            "frac_of_peak": gbs / peak, "peak": peak, "peak_source": f"{kind} hbm_gbs (a torch copy, driver-measured)",
            "copy_correct": ok, "note": "read + write bytes per call / mean CUDA-event time of 10 calls"}


def run_qta(args, w):
    import torch

    import quantized_tensor_activation_gb300 as qta

    ws, rank = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    qta.build()

    head = measure_workload(qta, w, args, dev, ws, local, headline=True)
    xs, shards, q = head.pop("_keep")
    alg, (peak, peak_kind) = head.pop("_alg"), head.pop("_peak")
    e2e, sweep_raw = head.pop("_e2e"), head.pop("_sweep")
    kernel_table, fused = head.pop("_kernel_table"), head.pop("_fused")
    kern = head["kernels"]

    N, R, C = w.ranks, w.rows, w.cols
    in_bytes = 2 * N * R * C
    x = xs[0]
    ring_rep = ring_report(qta, w, x, 3, peak) if args.ring else None
    hop_rep = hop_kernel_report(qta, w, x, peak) if (args.hop and not args.ring) else None
    block_choice = None
    if args.choose_block:
        from quantized_tensor_activation_gb300 import calib
        best, errs = calib.choose_block(x[0])
        block_choice = {"tensor": "rank 0", "chosen_block": best, "workload_block": w.block,
                        "mse": {str(b): e / x[0].numel() for b, e in errs.items()}}
    sm_sweep = None
    if sweep_raw:
        sm_sweep = []
        for n_sms, ms, evs3 in sweep_raw:
            t = kernel_table(evs3, fused)
            sm_sweep.append({"max_sms": n_sms, "eager_ms_per_step": ms,
                             "value": in_bytes / (ms * 1e-3) / 1e9 * ws,
                             "kernels_ms": {k: v["ms"] for k, v in t.items() if isinstance(v, dict)},
                             "kernels_frac_of_hbm": {k: v["frac_of_hbm"] for k, v in t.items()
                                                     if isinstance(v, dict) and "frac_of_hbm" in v}})
    del xs, shards, q, x
    torch.cuda.empty_cache()

    # the other target workloads, each measured the same way
    per_config = {}
    for name in args.per_config:
        wc = workloads.WORKLOADS[name]
        rep = measure_workload(qta, wc, args, dev, ws, local, headline=False)
        rep["roofline"] = _roofline(wc, rep["kernels"], rep["_alg"], rep["_peak"])
        for k in ("_alg", "_peak", "_e2e", "_sweep", "_kernel_table", "_fused"):
            rep.pop(k)
        per_config[name] = rep
        torch.cuda.empty_cache()

    k0 = None if args.no_k0 else copy_probe(qta, dev)
    ash = None if args.no_ash else ash_report(qta, dev)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_rows or _cpu_rows(w, 4e8), args.seed, min_s=10.0)
        for name, rep in per_config.items():
            wc = workloads.WORKLOADS[name]
            rep["cpu_baseline"] = cpu_baseline(wc, _cpu_rows(wc, 6e7), args.seed)

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return

    line = {
        "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": head["config"],
        "k1_sms": head["k1_sms"],
        "roofline": _roofline(w, kern, alg, (peak, peak_kind)),
        "path": head["path"],
        "launch": head["launch"],
        "kernel_times": head["kernel_times"],
        "ms_per_step_graph_with_events": head["ms_per_step_graph_with_events"],
        "eager_ms_per_step": head["eager_ms_per_step"],
        "kernels": kern,
        "step_frac_of_hbm": head["step_frac_of_hbm"],
        "other_path": head["other_path"],
        "recon": head["recon"],
        "inputs": head["inputs"],
        "ring": ring_rep,
        "hop_kernel": hop_rep,
        "sm_sweep": sm_sweep,
        "block_choice": block_choice,
        "cpu_baseline": cpu,
        "clocks": head["clocks"],
        "e2e": e2e,
        "gpu_launches": head["gpu_launches"],
        "k0_copy": k0,
        "ash_rescaling": ash,
        "per_config": per_config or None,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def _free_port() -> int:
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def launch_replicas(n: int, argv) -> int:
    """--gpus N without torchrun: start N local processes, one per GPU, with
    the rendezvous variables torchrun would set (127.0.0.1), and return the
    worst exit code.  Rank 0 prints the JSON line."""
    port = _free_port()
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n), LOCAL_WORLD_SIZE=str(n),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__), *argv], env=env))
    rcs = [p.wait() for p in procs]
    return max(rcs, key=abs)


TARGET_CONFIGS = ["gpt_tp", "qwen_grad", "equarx_int8", "flash_int4"]


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="equarx_int8", choices=sorted(workloads.WORKLOADS),
                    help="the headline workload (default: the largest, 8 x [16384 x 8192] bf16)")
    ap.add_argument("--per-config", default="auto",
                    help="comma-separated workloads measured after the headline, each as its own report under "
                         "per_config ('auto': the other target workloads; 'none': no others)")
    ap.add_argument("--impl", default="qta", choices=["qta", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-rows", type=int, default=0,
                    help="oracle row sample per rank of the headline's CPU baseline (0: about 4e8 elements)")
    ap.add_argument("--ref-rows", type=int, default=1024)
    ap.add_argument("--rows", type=int, default=0,
                    help="rows per rank of the headline workload (0: the workload's own; profiling captures of a "
                         "smaller case)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-k0", action="store_true", help="skip the K0 copy-kernel probe")
    ap.add_argument("--no-ash", action="store_true",
                    help="skip the adaptive-rescaling report (TACO with per-channel factors vs plain)")
    ap.add_argument("--no-clocks", action="store_true", help="skip the nvidia-smi clock window (profiling runs)")
    ap.add_argument("--no-recon", action="store_true", help="skip the reconstruction-error report")
    ap.add_argument("--k1-sms", type=int, default=-1,
                    help="SMs the compress (K1) may occupy (qta_desc.max_sms; 0: all; -1: the fastest of "
                         "all, 144, 136, 128 on whole steps)")
    ap.add_argument("--sm-sweep", default="",
                    help="comma-separated SM counts: time the step with every call capped to that many SMs")
    ap.add_argument("--choose-block", action="store_true",
                    help="add the reconstruction error of rank 0's tensor for TACO blocks 64/128/256")
    ap.add_argument("--hop", action="store_true",
                    help="time the ring's hop kernels alone on a whole rank tensor (roofline; no adder chains)")
    ap.add_argument("--ring", action="store_true",
                    help="add the ring adder-chain report (full loop / semi loop) of the workload")
    ap.add_argument("--no-graph", action="store_true", help="launch the timed steps eagerly instead of as a CUDA graph")
    ap.add_argument("--path", default="fused", choices=["fused", "split"],
                    help="fused: qar_reduce_requant; split: qar_reduce then qar_requant (FP32 sum in HBM)")
    args = ap.parse_args(argv)
    if args.per_config == "auto":
        args.per_config = [c for c in TARGET_CONFIGS if c != args.workload]
    elif args.per_config in ("", "none"):
        args.per_config = []
    else:
        args.per_config = [c.strip() for c in args.per_config.split(",") if c.strip()]
        bad = [c for c in args.per_config if c not in workloads.WORKLOADS]
        if bad:
            ap.error(f"unknown workloads in --per-config: {bad}")
    w = workloads.WORKLOADS[args.workload]
    if args.rows:
        # a smaller case of the same workload (profiling captures): rows per rank
        if args.rows % w.ranks:
            ap.error("--rows must be a multiple of the workload's rank count")
        w = dataclasses.replace(w, rows=args.rows)
    ws, _ = _dist()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # N independent replicas, one process per GPU, as torchrun would start them
        if args.impl == "qta":
            import torch
            have = torch.cuda.device_count()
            if have < args.gpus:
                print(f"bench.py: --gpus {args.gpus} asks for more GPUs than the {have} visible", file=sys.stderr)
                return 2
        return launch_replicas(args.gpus, argv)
    if args.gpus > 1 and ws != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={ws}", file=sys.stderr)
        return 2
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_qta(args, w)
    return 0


if __name__ == "__main__":
    sys.exit(main())
