"""Benchmark of the differential-attention head forward on GB300.

One step = one pass of the whole hot path (the fused bf16 forward, including
the head-norm epilogue) over one batch of the needle-style causal workload
B=2, H=16, N=4096, d=64 (value width 128).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload needle_4k|small_causal|mid_causal|long_16k|rising_4k|decode_16k]
                  [--scaling strong|weak]

--workload picks another measured shape (default needle_4k, the headline).
wide_4k is the forward with query/key halves of width d = 128 (B=2, H=8,
N=4096, causal; value width 256).  needle_4k_fp8 is the headline shape with
q1, k1, q2, k2 in fp8 e4m3 (v and out bf16).
needle_4k_bwd times the backward pass (diffattn_bwd given the saved
activations of diffattn_fwd_train) on the needle_4k shape, at 20*d
algorithmic flops per visible pair; wide_4k_bwd the same on the wide_4k
shape (d = 128).
decode_16k is one decoding step of 32 heads (B=1, H=32, one query each)
against a 16384-key cache through diffattn_fwd_kv with the library's split
count; it is bound by HBM, so its metric is algorithmic GB/s (the cache read
once, queries in, outputs out).

rising_4k is the headline shape with logits that climb along the key axis
(an adversarial case for the softmax's running maximum).

Metric: algorithmic TFLOP/s with 8*d flops per visible (query, key) pair
(2*d for each of the two Q K^T maps, 4*d for one combined map times V of
width 2d) and the causal half convention B*H*N^2/2 pairs.  Every launch is
bracketed by CUDA events: value is from the whole timed region, and the line
also reports the median per-launch time.

Several GPUs (--gpus N; launched under torchrun, or relaunched under it when
started without one): every (batch, head) is independent and the head norm is
per token, so the forward needs no collective.  --scaling strong (the default)
partitions the workload's B*H heads into N contiguous, balanced slices, one per
rank, each run as its own forward (the caller would gather the output
slices); --scaling weak runs the whole workload on every rank.  value = flops
of all ranks / max over ranks of the timed region.  The key/value-cache and
backward workloads always run weak.
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
import torch  # noqa: E402

WORKLOAD = "needle_4k"
METRIC = "diff-attn fwd TFLOP/s (causal, bf16) and % of GB300 tensor peak, 1 GPU"
UNIT = "TFLOP/s"
SPEC_BF16_TFLOPS = 2250.0  # GB300 nominal dense bf16 rate (context next to the measured peak)
L2_BYTES = 129 * 1024 * 1024
PROFILES = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = ["differential_attention_attn_gb300/csrc/fwd_bf16_sm103.cu",
                  "differential_attention_attn_gb300/csrc/ptx.cuh"]


def alg_flops(B, H, N, d, causal=True) -> float:
    pairs = B * H * N * N * (0.5 if causal else 1.0)
    return 8.0 * d * pairs


def alg_bytes(B, H, N, d, elem=2, qk_elem=None) -> float:
    # q1, k1, q2, k2 (4 * d) + v (2d) in, out (2d) out, per token per head
    qk = elem if qk_elem is None else qk_elem
    return float(B * H * N * (4 * d * qk + (2 * d + 2 * d) * elem))


def row_flops(i, d, causal=True) -> float:
    return 8.0 * d * ((i + 1) if causal else 1)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic(workload: str):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary,
    or None if that summary was taken on a different kernel source."""
    path = os.path.join(PROFILES, f"traffic_fwd_bf16_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#") and " " in line:
                k, v = line.split(None, 1)
                vals[k] = v.strip()
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks/throttle sampling in the background (100 ms period)."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t_start = time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    @staticmethod
    def _ts(s):
        from datetime import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.strptime(s.strip(), fmt).timestamp()
            except ValueError:
                pass
        return None

    def summary(self, t0: float, t1: float):
        rows = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append((self._ts(f[0]), float(f[2]), float(f[3]), f[5:10]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "none"}
        inside = [r for r in rows if r[0] is not None and t0 - 0.1 <= r[0] <= t1 + 0.1]
        window = "timed"
        if not inside:
            inside, window = rows, "whole run (timed region shorter than the sampling period)"
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": sorted(reasons),
                "samples": len(inside), "window": window}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def max_over_ranks(values, dist=None, device="cpu"):
    """The job's times are its slowest rank's: the element-wise maximum of every
    rank's values (an all-reduce when a process group is given)."""
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def head_slice(BH: int, world: int, rank: int):
    """Contiguous, balanced slice [lo, hi) of the BH flattened (batch, head)
    pairs for `rank` of `world`: slice sizes differ by at most one head and the
    slices tile [0, BH) in rank order."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world")
    return rank * BH // world, (rank + 1) * BH // world


def timed_launches(step, steps: int, stream):
    """Run step(0 .. steps-1) with an event before every launch and one after
    the last.  Returns (ms from first to last event, per-launch ms, wall-clock
    start, wall-clock end)."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    t_wall0 = time.time()
    for i in range(steps):
        ev[i].record(stream)
        step(i)
    ev[steps].record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    per_launch = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return ev[0].elapsed_time(ev[steps]), per_launch, t_wall0, t_wall1


def cpu_baseline(w, seconds: float, seed: int = 3):
    """Time the float64 oracle on a bounded, seeded sample of the workload's rows.

    Rows are drawn uniformly over (head, query) so that their mean causal length
    matches the workload's; the value is algorithmic TFLOP/s of those rows."""
    import oracle
    from tests import harness

    args, kw = harness.oracle_args(w)
    rng = np.random.default_rng(seed)
    BH, N = w.B * w.H, w.N
    cores = oracle.max_threads(0)

    def run(n):
        bh = rng.integers(0, BH, size=n)
        ri = rng.integers(0, N, size=n)
        t = time.perf_counter()
        oracle.fwd_rows(*args, bh, ri, **kw)
        dt = time.perf_counter() - t
        return dt, float(sum(row_flops(int(i), w.d, w.causal) for i in ri))

    n = 2 * cores
    dt, fl = run(n)
    while dt < 0.5 and n < 1 << 20:
        n *= 4
        dt, fl = run(n)
    n_final = max(n, int(n * seconds / max(dt, 1e-6)))
    dt, fl = run(n_final)
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n_final} query rows drawn uniformly over the {BH} heads x {N} rows "
                      f"of {w.name} (causal), full float64 oracle per row; {dt:.1f} s"}


def run_reference(args):
    """The oracle as the reference arm: rank 0 only, host cores, bounded samples."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from differential_attention_attn_gb300 import workloads as W
    from tests import harness

    if args.workload in DECODE:
        w = decode_workload(args.workload)
        base = decode_cpu_baseline(w, 1.0)
        line = {"impl": "reference", "metric": DECODE_METRIC, "value": base["value"],
                "unit": "GB/s", "n_gpus": world, "steps": 1, "warmup": 0,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic",
                "config": {"workload": args.workload, "B": w.B, "H": w.H, "Nq": w.N,
                           "Nkv": w.n_kv, "d": w.d},
                "cpu_baseline": base,
                "e2e": {"value": base["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    WORKLOAD = args.workload
    w = W.make(WORKLOAD)
    oargs, kw = harness.oracle_args(w)
    rng = np.random.default_rng(11)
    BH, N = w.B * w.H, w.N
    cores = oracle.max_threads(0)

    def step(n):
        bh = rng.integers(0, BH, size=n)
        ri = rng.integers(0, N, size=n)
        t = time.perf_counter()
        oracle.fwd_rows(*oargs, bh, ri, **kw)
        return time.perf_counter() - t, float(sum(row_flops(int(i), w.d) for i in ri))

    n = 2 * cores
    dt, _ = step(n)
    target = 1.0  # seconds of CPU work per step
    n = max(n, int(n * target / max(dt, 1e-6)))
    for _ in range(max(args.warmup, 0)):
        step(n)
    tot_t, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        dt, fl = step(n)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dv": 2 * w.d,
                   "causal": True, "headnorm": True,
                   "sample_per_step": f"{n} query rows drawn uniformly over heads x rows"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{n} rows per step x {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


DECODE = {"decode_16k": dict(B=1, H=32, Nq=1, Nkv=16384, layer=24)}
DECODE_METRIC = "diff-attn decode GB/s (1 query per head vs a 16K-key cache, bf16), 1 GPU"


def decode_bytes(B, H, Nq, Nkv, d=64, elem=2) -> float:
    # k1, k2 (2 * d) + v (2d) per cached key; q1, q2 (2 * d) in and out (2d) per query
    return float(B * H * (Nkv * 4 * d + Nq * 4 * d) * elem)


def decode_workload(name, seed_offset=0):
    from differential_attention_attn_gb300 import workloads as W
    c = DECODE[name]
    return W.kv_cache(2000 + seed_offset, B=c["B"], H=c["H"], Nq=c["Nq"], Nkv=c["Nkv"],
                      causal=True, layer=c["layer"], random_w=False)


def run_decode(args):
    """One decoding step per timed step, through diffattn_fwd_kv (split-KV + combine)."""
    from differential_attention_attn_gb300 import ops

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    ops.load()
    w = decode_workload(args.workload, seed_offset=rank)
    B, H, Nq, Nkv, d = w.B, w.H, w.N, w.n_kv, w.d
    li = float(np.float32(ops.lambda_init(w.layer)))
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device=dev)
    host = [t.contiguous() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    set_bytes = sum(t.numel() * t.element_size() for t in host)
    n_sets = max(2, -(-2 * L2_BYTES // set_bytes) + 1)
    sets = [[t.to(dev) for t in host] for _ in range(n_sets)]
    out = torch.empty((B, H, Nq, 2 * d), dtype=torch.bfloat16, device=dev)
    splits, ws_bytes = ops.fwd_kv_plan(B, H, Nq, Nkv, causal=True, splits=0)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    kw = dict(causal=True, headnorm=True, eps=float(np.float32(w.eps)), lambda_init=li,
              splits=splits, workspace=ws, stream=stream)

    def step(ins, o):
        ops.fwd_kv(*ins, lam, out=o, **kw)

    for i in range(args.warmup):
        step(sets[i % n_sets], out)
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ms_total, per_launch, t_wall0, t_wall1 = timed_launches(
        lambda i: step(sets[i % n_sets], out), args.steps, stream)
    if dist:
        dist.barrier()
    if sampler:
        time.sleep(0.15)
        sampler.stop()

    # e2e: the step's queries come from pinned host memory and the outputs go back;
    # the key/value cache is state that stays resident on the device.
    q_host = [w.q1.contiguous().pin_memory(), w.q2.contiguous().pin_memory()]
    cache = sets[0]
    q_dev = [torch.empty_like(t, device=dev) for t in q_host]
    host_out = torch.empty((B, H, Nq, 2 * d), dtype=torch.bfloat16).pin_memory()

    def e2e_step():
        for dst, src in zip(q_dev, q_host):
            dst.copy_(src, non_blocking=True)
        step([q_dev[0], cache[1], q_dev[1], cache[3], cache[4]], out)
        host_out.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = f0.elapsed_time(f1)
    med_ms = statistics.median(per_launch)
    ms_total, e2e_ms, med_ms = max_over_ranks([ms_total, e2e_ms, med_ms], dist, dev)
    nbytes = decode_bytes(B, H, Nq, Nkv, d)
    value = world * nbytes * args.steps / (ms_total * 1e-3) / 1e9
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    peaks, peak_src = read_peaks()
    peak = float(peaks["hbm_gbs"])
    launch_ms = ms_total / args.steps
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": launch_ms,
        "median_ms_per_launch": med_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "H": H, "Nq": Nq, "Nkv": Nkv, "d": d,
                   "dv": 2 * d, "causal": True, "headnorm": True, "splits": splits,
                   "workspace_bytes": ws_bytes,
                   "bytes_convention": "k1, k2, v of the cache once + q1, q2 in + out",
                   "l2": f"rotating {n_sets} caches of {set_bytes / 1e6:.1f} MB: a step's set was last "
                         f"used {(n_sets - 1) * set_bytes / 1e6:.0f} MB of other sets earlier "
                         f"(L2 {L2_BYTES / 1e6:.0f} MB)",
                   "parallelism": f"weak x{world} (one full workload per rank)"},
        "roofline": {"bound": "hbm", "achieved": nbytes / (launch_ms * 1e-3) / 1e9,
                     "peak": peak, "unit": "GB/s",
                     "frac": nbytes / (launch_ms * 1e-3) / 1e9 / peak,
                     "peak_source": f"{peak_src} hbm_gbs (copy)",
                     "kernel": "diffattn_fwd_bf16_sm103_kernel (split-KV partial) + "
                               "diffattn_splitkv_combine_kernel, timed together per step",
                     "alg_bytes_per_launch": nbytes, "traffic": None},
        "e2e": {"value": world * nbytes * args.steps / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in q_host)),
                "d2h_bytes_per_step": int(host_out.numel() * host_out.element_size())},
        "gpu_launches": args.steps * (2 if splits > 1 else 1),
        "clocks": sampler.summary(t_wall0, t_wall1) if sampler else None,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = decode_cpu_baseline(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def decode_cpu_baseline(w, seconds: float):
    """The float64 oracle on whole decoding steps, repeated for about `seconds`."""
    import oracle
    from tests import harness

    args, kw = harness.oracle_args(w)
    cores = oracle.max_threads(0)
    nbytes = decode_bytes(w.B, w.H, w.N, w.n_kv, w.d)
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < seconds or n == 0:
        oracle.fwd_kv(*args, **kw)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": n * nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} whole decoding steps of {w.name}, float64 oracle; {dt:.1f} s"}


BWD_METRIC = "diff-attn bwd TFLOP/s (causal, bf16), 1 GPU"


def run_bwd(args):
    """One backward pass per step (diffattn_bwd given diffattn_fwd_train's saved
    activations) on the needle_4k shape (wide_4k_bwd: the wide_4k shape, d = 128);
    20*d algorithmic flops per visible pair."""
    from differential_attention_attn_gb300 import ops
    from differential_attention_attn_gb300 import workloads as W

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    ops.load()
    wide = args.workload == "wide_4k_bwd"
    if wide:
        w = W.custom(3000 + rank, B=2, H=8, N=4096, d=128, causal=True, headnorm=True,
                     random_w=True, layer=12)
    else:
        w = W.make("needle_4k", seed_offset=rank)
    B, H, N, d = w.B, w.H, w.N, w.d
    li = float(np.float32(ops.lambda_init(w.layer) if wide else w.lambda_init_override))
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device=dev)
    nw = torch.tensor(np.asarray(w.w, dtype=np.float32), device=dev) if wide else None
    kw = dict(causal=True, headnorm=True, norm_w=nw, eps=float(np.float32(w.eps)),
              lambda_init=li)
    rng = np.random.default_rng(77 + rank)
    dy_host = torch.from_numpy(rng.standard_normal((B, H, N, 2 * d))).to(torch.bfloat16)
    host = [t.contiguous() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    saved_bytes, ws_bytes = ops.train_sizes(B, H, N, d=d)
    set_bytes = sum(t.numel() * t.element_size() for t in host) + saved_bytes + \
        dy_host.numel() * 2
    n_sets = max(2, -(-2 * L2_BYTES // set_bytes) + 1)
    sets = []
    for _ in range(n_sets):
        ins = [t.to(dev) for t in host]
        _, saved = ops.fwd_train(*ins, lam, **kw)
        sets.append((ins, saved, dy_host.to(dev)))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    grads = {k: torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
             for k in ("dq1", "dk1", "dq2", "dk2")}
    grads["dv"] = torch.empty((B, H, N, 2 * d), dtype=torch.bfloat16, device=dev)
    grads["dlam"] = torch.empty(H, dtype=torch.float32, device=dev)
    grads["dw"] = torch.empty((H, 2 * d), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        ins, saved, dy = sets[i % n_sets]
        ops.bwd(*ins, lam, saved, dy, workspace=ws, grads=grads, stream=stream, **kw)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ms_total, per_launch, t_wall0, t_wall1 = timed_launches(step, args.steps, stream)
    if dist:
        dist.barrier()
    if sampler:
        time.sleep(0.15)
        sampler.stop()
    med_ms = statistics.median(per_launch)
    ms_total, med_ms = max_over_ranks([ms_total, med_ms], dist, dev)
    flops_step = alg_flops(B, H, N, d) * 20.0 / 8.0
    value = world * flops_step * args.steps / (ms_total * 1e-3) / 1e12
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    peaks, peak_src = read_peaks()
    peak = float(peaks["bf16_tflops"])
    launch_ms = ms_total / args.steps
    line = {
        "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": launch_ms,
        "median_ms_per_launch": med_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "H": H, "N": N, "d": d, "dv": 2 * d,
                   "causal": True, "headnorm": True,
                   "flops_convention": "20*d per visible pair (S1, S2, dW, dV, dQ, dK), "
                                       "B*H*N^2/2 pairs",
                   "l2": f"rotating {n_sets} sets of {set_bytes / 1e6:.1f} MB: a step's set was last "
                         f"used {(n_sets - 1) * set_bytes / 1e6:.0f} MB of other sets earlier "
                         f"(L2 {L2_BYTES / 1e6:.0f} MB)",
                   "parallelism": f"weak x{world} (one full workload per rank)"},
        "roofline": {"bound": "tensor", "achieved": flops_step / (launch_ms * 1e-3) / 1e12,
                     "peak": peak, "unit": UNIT,
                     "frac": flops_step / (launch_ms * 1e-3) / 1e12 / peak,
                     "peak_source": f"{peak_src} bf16_tflops (burst, cuBLAS bf16 GEMM)",
                     "kernel": ("diffattn_bwd_pre_d128_kernel + diffattn_bwd_d128_sm103_kernel"
                                "<dV> + <dK/dQ> + diffattn_bwd_finish_d128_kernel (+ 3 memsets)"
                                if wide else
                                "diffattn_bwd_pre_kernel + diffattn_bwd_bf16_sm103_kernel + "
                                "diffattn_bwd_finish_kernel (+ 4 memsets)") + ", timed together",
                     "alg_flops_per_launch": flops_step, "traffic": None},
        "gpu_launches": args.steps * (4 if wide else 3),
        "clocks": sampler.summary(t_wall0, t_wall1) if sampler else None,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_ours(args):
    from differential_attention_attn_gb300 import ops
    from differential_attention_attn_gb300 import workloads as W

    if args.workload in DECODE:
        return run_decode(args)
    if args.workload in ("needle_4k_bwd", "wide_4k_bwd"):
        return run_bwd(args)
    WORKLOAD = args.workload

    world, rank, local = dist_env()
    strong = args.scaling == "strong"
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    ops.load()

    fp8 = WORKLOAD == "needle_4k_fp8"
    if WORKLOAD == "wide_4k":  # d = 128 per half (value width 256)
        w = W.custom(3000 + rank, B=2, H=8, N=4096, d=128, causal=True, headnorm=True,
                     random_w=True, layer=12)
    elif fp8:  # the needle inputs with q1, k1, q2, k2 rounded to e4m3
        w = W.make("needle_4k", seed_offset=rank)
        for name in ("q1", "k1", "q2", "k2"):
            setattr(w, name, getattr(w, name).float().to(torch.float8_e4m3fn))
    else:
        w = W.make(WORKLOAD, seed_offset=0 if strong else rank)
    B, H, N, d = w.B, w.H, w.N, w.d
    li = float(np.float32(w.lambda_init_override if w.layer is None
                          else ops.lambda_init(w.layer)))
    lam_all = np.asarray(w.lambdas(li), dtype=np.float32)
    w_all = None if w.w is None else np.asarray(w.w, dtype=np.float32)
    host = [t.contiguous() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    bh_lo, bh_hi = 0, B * H
    if strong:
        # This rank's heads: a contiguous slice of the flattened (batch, head)
        # pairs, run as one batch of hi - lo heads with their own lambda and
        # norm weights (head h of batch b is flattened index b * H + h).
        bh_lo, bh_hi = head_slice(B * H, world, rank)
        heads = np.arange(bh_lo, bh_hi) % H
        host = [t.reshape(B * H, N, -1)[bh_lo:bh_hi].reshape(1, bh_hi - bh_lo, N, -1).contiguous()
                for t in host]
        lam_all = lam_all[heads]
        w_all = None if w_all is None else w_all[heads]
        B, H = 1, bh_hi - bh_lo
    lam = torch.tensor(lam_all, dtype=torch.float32, device=dev)
    norm_w = None if w_all is None else torch.tensor(w_all, dtype=torch.float32, device=dev)
    set_bytes = sum(t.numel() * t.element_size() for t in host) + B * H * N * 2 * d * 2
    n_sets = max(2, -(-2 * L2_BYTES // set_bytes) + 1)
    sets = []
    for _ in range(n_sets):
        ins = [t.to(dev) for t in host]
        out = torch.empty((B, H, N, 2 * d), dtype=torch.bfloat16, device=dev)
        sets.append((ins, out))
    stream = torch.cuda.current_stream()
    kw = dict(causal=True, headnorm=True, norm_w=norm_w, eps=float(np.float32(w.eps)),
              lambda_init=li, stream=stream)

    fwd = ops.fwd_fp8 if fp8 else ops.fwd

    def step(i):
        ins, out = sets[i % n_sets]
        fwd(*ins, lam, out=out, **kw)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ms_total, per_launch, t_wall0, t_wall1 = timed_launches(step, args.steps, stream)
    if dist:
        dist.barrier()
    if sampler:
        time.sleep(0.15)
        sampler.stop()

    # e2e: the same forward through the C-ABI entry that takes host buffers
    # (diffattn_fwd_host): every step copies its five inputs from pinned host
    # memory into device staging, runs the kernel and copies the output back, all
    # inside the call.  Consecutive steps alternate two streams (each with its own
    # staging buffer and host output), so one step's copies overlap the other's
    # kernel, as a serving loop would.  The e4m3 variant keeps torch copies around
    # diffattn_fwd (the host entry takes bf16 and fp32 tensors).
    pinned = [t.pin_memory() for t in host]
    e2e_streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    e2e_path = "diffattn_fwd_host (C ABI): pinned host inputs and output, device staging, " \
               "two alternating streams"
    if not fp8:
        need = ops.fwd_host_staging_bytes(B, H, N, d)
        staging = [torch.empty(need, dtype=torch.uint8, device=dev) for _ in range(2)]
        host_outs = [torch.empty((B, H, N, 2 * d), dtype=torch.bfloat16).pin_memory()
                     for _ in range(2)]
        host_out = host_outs[0]

        kw_host = {k: v for k, v in kw.items() if k != "stream"}

        def e2e_step(i):
            s = i % 2
            ops.fwd_host(*pinned, lam, out=host_outs[s], staging=staging[s],
                         stream=e2e_streams[s], **kw_host)

        def e2e_fence():  # the compute stream waits for both streams
            for st_ in e2e_streams:
                stream.wait_stream(st_)
        h2d_stream, d2h_stream = e2e_streams
    else:
        e2e_path = "torch copies from pinned host memory around diffattn_fwd (e4m3 inputs)"
        dev_in = [[torch.empty_like(t, device=dev) for t in host] for _ in range(2)]
        dev_out = [torch.empty((B, H, N, 2 * d), dtype=torch.bfloat16, device=dev)
                   for _ in range(2)]
        host_out = torch.empty((B, H, N, 2 * d), dtype=torch.bfloat16).pin_memory()
        h2d_stream, d2h_stream = e2e_streams
        in_ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]      # kernel of the buffer set finished
        out_read = [torch.cuda.Event() for _ in range(2)]  # its output copied back

        def e2e_step(i):
            s = i % 2
            with torch.cuda.stream(h2d_stream):
                h2d_stream.wait_event(done[s])  # the inputs of step i - 2 are consumed
                for dst, src in zip(dev_in[s], pinned):
                    dst.copy_(src, non_blocking=True)
                in_ready[s].record(h2d_stream)
            stream.wait_event(in_ready[s])
            stream.wait_event(out_read[s])  # the output of step i - 2 is copied back
            fwd(*dev_in[s], lam, out=dev_out[s], **kw)
            done[s].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(done[s])
                host_out.copy_(dev_out[s], non_blocking=True)
                out_read[s].record(d2h_stream)

        def e2e_fence():  # the compute stream waits for both copy streams
            ev_a, ev_b = torch.cuda.Event(), torch.cuda.Event()
            ev_a.record(h2d_stream)
            ev_b.record(d2h_stream)
            stream.wait_event(ev_a)
            stream.wait_event(ev_b)

    for i in range(max(2, min(args.warmup, 3))):
        e2e_step(i)
    e2e_fence()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, args.steps)
    f0.record(stream)
    h2d_stream.wait_stream(stream)  # no copy of the timed steps starts before f0
    d2h_stream.wait_stream(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    e2e_fence()
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = f0.elapsed_time(f1)

    med_ms = statistics.median(per_launch)
    ms_total, e2e_ms, med_ms = max_over_ranks([ms_total, e2e_ms, med_ms], dist, dev)
    flops_step = alg_flops(B, H, N, d)  # this rank's launch
    # One step of the job: the whole workload once (strong) or once per rank (weak).
    job_flops = alg_flops(w.B, w.H, N, d) * (1 if strong else world)
    value = job_flops * args.steps / (ms_total * 1e-3) / 1e12
    e2e_value = job_flops * e2e_steps / (e2e_ms * 1e-3) / 1e12
    launch_ms = ms_total / args.steps
    achieved = flops_step / (launch_ms * 1e-3) / 1e12

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    peaks, peak_src = read_peaks()
    peak = float(peaks["bf16_tflops"])
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    if strong and world > 1:
        par = (f"strong x{world}: the {w.B * w.H} (batch, head) pairs in contiguous slices of "
               f"{w.B * w.H // world} to {-(-w.B * w.H // world)}, one per rank; no collective")
    else:
        par = f"weak x{world} (one full workload per rank)"
    line = {
        "metric": METRIC.replace("bf16", "e4m3 q/k, bf16 v") if fp8 else METRIC,
        "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_total / args.steps, "higher_is_better": True,
        "scaling": "strong" if (strong and world > 1) else "weak", "vs_baseline": None,
        "median_ms_per_launch": med_ms,
        "value_at_median": job_flops / (med_ms * 1e-3) / 1e12,
        "dtype": "e4m3 q/k, bf16 v/out" if fp8 else "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": w.B, "H": w.H, "N": N, "d": d, "dv": 2 * d,
                   "causal": True, "headnorm": True,
                   "flops_convention": "8*d per visible pair, B*H*N^2/2 pairs",
                   "l2": f"rotating {n_sets} input sets of {set_bytes / 1e6:.1f} MB: a step's set was last "
                         f"used {(n_sets - 1) * set_bytes / 1e6:.0f} MB of other sets earlier "
                         f"(L2 {L2_BYTES / 1e6:.0f} MB)",
                   "parallelism": par},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak,
                     "spec_peak": SPEC_BF16_TFLOPS, "frac_of_spec": achieved / SPEC_BF16_TFLOPS,
                     "peak_source": f"{peak_src} bf16_tflops (burst, cuBLAS bf16 GEMM)",
                     "kernel": ("diffattn_fwd_d128_sm103_kernel" if d == 128
                                else "diffattn_fwd_bf16_sm103_kernel"),
                     "alg_flops_per_launch": flops_step,
                     "alg_bytes_per_launch": alg_bytes(B, H, N, d, qk_elem=1 if fp8 else 2),
                     "achieved_gbs": alg_bytes(B, H, N, d, qk_elem=1 if fp8 else 2)
                     / (launch_ms * 1e-3) / 1e9,
                     "traffic": read_traffic(WORKLOAD) if d == 64 and not fp8 else None},
        "e2e": {"value": e2e_value, "unit": UNIT,
                "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in host)),
                "d2h_bytes_per_step": int(host_out.numel() * host_out.element_size()),
                "path": e2e_path},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if strong and world > 1:
        line["config"]["heads_rank0"] = [bh_lo, bh_hi]
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def relaunch(gpus: int):
    """Run this same command as `gpus` ranks under torch.distributed.run (one
    process per GPU of this node, rendezvous on 127.0.0.1) and exit with its
    status."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={gpus}", "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__), *sys.argv[1:]]
    raise SystemExit(subprocess.call(cmd))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["needle_4k", "small_causal", "mid_causal", "long_16k", "rising_4k",
                             *DECODE, "needle_4k_bwd", "wide_4k_bwd", "wide_4k",
                             "needle_4k_fp8"])
    ap.add_argument("--scaling", choices=["strong", "weak"], default="strong",
                    help="with several GPUs: partition the heads (strong) or replicate (weak)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # timing rule: at least 3 untimed warm-up steps
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        relaunch(args.gpus)  # does not return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch one rank per GPU")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
