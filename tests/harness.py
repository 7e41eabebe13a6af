"""Run one workload through the CUDA path (C ABI) and through the oracle.

The two sides share only the seeded inputs from workloads.py.  Each side
evaluates lambda_init with its own code (library: diffattn_lambda_init;
oracle: oracle_lambda_init), and both receive the float32-rounded lambda,
norm weight and eps that the kernel sees.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from differential_attention_attn_gb300 import ops


def lambda_init_for(w, side: str) -> float:
    if w.layer is None:
        li = w.lambda_init_override or 0.0
    elif side == "gpu":
        li = ops.lambda_init(w.layer)
    else:
        li = oracle.lambda_init(w.layer)
    return float(np.float32(li))


def run_gpu(w, *, out=None, status=None, device="cuda"):
    li = lambda_init_for(w, "gpu")
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device=device)
    nw = None if w.w is None else torch.tensor(w.w, dtype=torch.float32, device=device)
    dev = [t.to(device) for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    o = ops.fwd(*dev, lam, causal=w.causal, headnorm=w.headnorm, norm_w=nw,
                eps=float(np.float32(w.eps)), lambda_init=li, out=out, status=status)
    torch.cuda.synchronize()
    return o


def run_gpu_kv(w, *, splits=0, workspace=None, out=None, status=None, device="cuda",
               raw_status=False):
    """The workload through diffattn_fwd_kv (queries against its key/value rows)."""
    li = lambda_init_for(w, "gpu")
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device=device)
    nw = None if w.w is None else torch.tensor(w.w, dtype=torch.float32, device=device)
    dev = [t.to(device) for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    o = ops.fwd_kv(*dev, lam, causal=w.causal, headnorm=w.headnorm, norm_w=nw,
                   eps=float(np.float32(w.eps)), lambda_init=li, splits=splits,
                   workspace=workspace, out=out, status=status, raw_status=raw_status)
    torch.cuda.synchronize()
    return o


def run_oracle_kv(w, bh_idx=None, row_idx=None):
    args, kw = oracle_args(w)
    return oracle.fwd_kv(*args, bh_idx=bh_idx, row_idx=row_idx, **kw)


def oracle_args(w):
    li = lambda_init_for(w, "oracle")
    f = w.f64
    return (f(w.q1), f(w.k1), f(w.q2), f(w.k2), f(w.v), w.lambdas(li)), dict(
        causal=w.causal, headnorm=w.headnorm, w=w.w, eps=float(np.float32(w.eps)),
        lambda_init_value=li)


def run_oracle(w):
    args, kw = oracle_args(w)
    return oracle.fwd(*args, **kw)


def run_oracle_rows(w, bh_idx, row_idx):
    args, kw = oracle_args(w)
    return oracle.fwd_rows(*args, bh_idx, row_idx, **kw)


def sample_rows(w, n_random_per_head: int, full_heads=(), seed: int = 5):
    """(bh, row) pairs: every row of `full_heads`, plus rows 0, N-1 and random rows of
    every other head (and the needle query rows when the workload has them)."""
    rng = np.random.default_rng(seed)
    BH, N = w.B * w.H, w.N
    bh, ri = [], []
    for f in full_heads:
        bh += [f] * N
        ri += list(range(N))
    extra = list(w.meta.get("needle_query", []))
    for x in range(BH):
        if x in full_heads:
            continue
        rows = set([0, N - 1] + extra + list(rng.integers(0, N, size=n_random_per_head)))
        bh += [x] * len(rows)
        ri += sorted(rows)
    return np.array(bh, dtype=np.int64), np.array(ri, dtype=np.int64)


def bf16_tolerance(ref: np.ndarray) -> float:
    """max-abs bound for bf16 outputs: 2e-2 * max|ref|."""
    return 2e-2 * float(np.max(np.abs(ref))) if ref.size else 0.0
