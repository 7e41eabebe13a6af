"""Seeded synthetic inputs for the differential-attention head.

This module draws random inputs and nothing else: it holds none of the
method's arithmetic (no softmax, no lambda_init formula, no normalisation), so
that the CUDA path and the float64 oracle can both be fed from it without
sharing any computation.  Where a workload's lambda is defined relative to
lambda_init(l), the workload returns the layer index and the random offsets;
each side evaluates lambda_init with its own code.

Workloads (shapes and value recipes follow the five synthetic configurations
this library is measured on; the worked example is the one printed on the
"Differential Transformer" glossary page, section "How differential attention
works"):

  pages_example  fp32, B=H=1, N=6, d=8, non-causal, lambda=0.8, no head norm;
                 drawn exactly as the page's snippet does
                 (torch.manual_seed(0); randn(4, 6, 8); randn(6, 16)).
  small_causal   bf16, B=1, H=4,  N=512,   d=64, causal, layer 1,
                 lambda_h ~ U[0.1, 0.9], norm weight 1.
  mid_causal     bf16, B=4, H=16, N=2048,  d=64, causal, Q/K ~ 0.5 N(0,1),
                 layer 12, lambda_h = lambda_init + U[-0.05, 0.05],
                 norm weight ~ 1 + 0.02 N(0,1) of shape [H, 2d].
  needle_4k      bf16, B=2, H=16, N=4096,  d=64, causal, six "needle" keys per
                 head: K1[p_k] = 4 * Q1[N - 6 + k] for p_k drawn without
                 replacement from [0, N - 6); lambda = 0.8, lambda_init = 0.8.
  long_16k       bf16, B=1, H=32, N=16384, d=64, causal, layer 24,
                 lambda_h ~ U[0.6, 0.9], norm weight 1.
  rising_4k      bf16, B=2, H=16, N=4096, d=64, causal, logits that climb
                 along the key axis (see rising()); layer 8,
                 lambda_h ~ U[0.3, 0.9], norm weight 1.  An adversarial case
                 for softmax kernels that keep a stale running maximum.

Random source: numpy.random.default_rng(1000 + workload number) drawing in
float64 in the order Q1, K1, Q2, K2, V, [needle positions], lambda, w; the
float64 draws are rounded to the storage dtype (bf16 round-to-nearest-even via
torch).  The oracle is given exactly the rounded values.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

WORKLOADS = ("pages_example", "small_causal", "mid_causal", "needle_4k", "long_16k",
             "rising_4k")
WORKLOAD_NUMBER = {name: i + 1 for i, name in enumerate(WORKLOADS)}


@dataclass
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: torch.dtype
    causal: bool
    headnorm: bool
    eps: float
    q1: torch.Tensor  # [B, H, N, d] on the CPU, storage dtype
    k1: torch.Tensor
    q2: torch.Tensor
    k2: torch.Tensor
    v: torch.Tensor   # [B, H, N, 2d]
    lam_offset: np.ndarray            # [H] float64
    lam_plus_lambda_init: bool        # lambda_h = offset (+ lambda_init if True)
    layer: int | None                 # layer index for lambda_init, or None
    lambda_init_override: float | None  # fixed lambda_init when layer is None
    w: np.ndarray | None              # [H, 2d] float64 or None (ones)
    meta: dict = field(default_factory=dict)
    n_kv: int | None = None           # key/value rows when they differ from N (k1, k2, v)

    @property
    def dv(self) -> int:
        return 2 * self.d

    def lambdas(self, lambda_init_value: float) -> np.ndarray:
        """Per-head lambda, float32-rounded, given this side's lambda_init."""
        lam = self.lam_offset + (lambda_init_value if self.lam_plus_lambda_init else 0.0)
        return lam.astype(np.float32).astype(np.float64)

    def f64(self, t: torch.Tensor) -> np.ndarray:
        return t.to(torch.float64).numpy()


def _normal(rng, shape, scale=1.0):
    return rng.standard_normal(size=shape) * scale


def _to_storage(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).contiguous()


def random_heads(seed: int, B: int, H: int, N: int, d: int, *, dtype=torch.bfloat16,
                 qk_scale: float = 1.0, v_scale: float = 1.0):
    """Q1, K1, Q2, K2 ~ qk_scale * N(0,1) [B,H,N,d] and V ~ v_scale * N(0,1) [B,H,N,2d]."""
    rng = np.random.default_rng(seed)
    qk = [_to_storage(_normal(rng, (B, H, N, d), qk_scale), dtype) for _ in range(4)]
    v = _to_storage(_normal(rng, (B, H, N, 2 * d), v_scale), dtype)
    return rng, qk, v


def pages_example() -> Workload:
    """The page's worked example, drawn with the page's own recipe."""
    g = torch.Generator().manual_seed(0)
    n, d = 6, 8
    q1, k1, q2, k2 = torch.randn(4, n, d, generator=g)
    v = torch.randn(n, 2 * d, generator=g)
    r = lambda t: t.reshape(1, 1, *t.shape).contiguous()
    return Workload("pages_example", 1, 1, n, d, torch.float32, False, False, 1e-5,
                    r(q1), r(k1), r(q2), r(k2), r(v), np.array([0.8]), False, None, None,
                    None)


def make(name: str, *, seed_offset: int = 0) -> Workload:
    """Build one named workload (CPU tensors)."""
    if name == "pages_example":
        return pages_example()
    seed = 1000 + WORKLOAD_NUMBER[name] + seed_offset
    if name == "small_causal":
        B, H, N, d = 1, 4, 512, 64
        rng, (q1, k1, q2, k2), v = random_heads(seed, B, H, N, d)
        lam = rng.uniform(0.1, 0.9, size=H)
        return Workload(name, B, H, N, d, torch.bfloat16, True, True, 1e-5, q1, k1, q2, k2, v,
                        lam, False, 1, None, None)
    if name == "mid_causal":
        B, H, N, d = 4, 16, 2048, 64
        rng, (q1, k1, q2, k2), v = random_heads(seed, B, H, N, d, qk_scale=0.5)
        lam = rng.uniform(-0.05, 0.05, size=H)
        w = 1.0 + 0.02 * rng.standard_normal(size=(H, 2 * d))
        w = w.astype(np.float32).astype(np.float64)
        return Workload(name, B, H, N, d, torch.bfloat16, True, True, 1e-5, q1, k1, q2, k2, v,
                        lam, True, 12, None, w)
    if name == "needle_4k":
        return needle(seed, B=2, H=16, N=4096, d=64)
    if name == "long_16k":
        B, H, N, d = 1, 32, 16384, 64
        rng, (q1, k1, q2, k2), v = random_heads(seed, B, H, N, d)
        lam = rng.uniform(0.6, 0.9, size=H)
        return Workload(name, B, H, N, d, torch.bfloat16, True, True, 1e-5, q1, k1, q2, k2, v,
                        lam, False, 24, None, None)
    if name == "rising_4k":
        return rising(seed, B=2, H=16, N=4096, d=64)
    raise KeyError(f"unknown workload {name!r}; known: {WORKLOADS}")


def needle(seed: int, *, B: int, H: int, N: int, d: int, n_needles: int = 6,
           gain: float = 4.0, dtype=torch.bfloat16) -> Workload:
    """Needle-style causal inputs: per head, n_needles key rows of K1 are set to
    gain * the Q1 row of a matching query near the end of the sequence, so that
    map1 is sharply peaked on those rows while map2 (K2 untouched) stays diffuse.
    Needle k pairs with query N - n_needles + k; its key position is drawn
    without replacement from [0, N - n_needles)."""
    if N <= 2 * n_needles:
        raise ValueError("needle workload needs N > 2 * n_needles")
    rng = np.random.default_rng(seed)
    q1 = _normal(rng, (B, H, N, d))
    k1 = _normal(rng, (B, H, N, d))
    q2 = _normal(rng, (B, H, N, d))
    k2 = _normal(rng, (B, H, N, d))
    v = _normal(rng, (B, H, N, 2 * d))
    pos = np.zeros((B, H, n_needles), dtype=np.int64)
    for b in range(B):
        for h in range(H):
            p = rng.choice(N - n_needles, size=n_needles, replace=False)
            pos[b, h] = p
            for k in range(n_needles):
                k1[b, h, p[k]] = gain * q1[b, h, N - n_needles + k]
    t = lambda x: _to_storage(x, dtype)
    return Workload("needle_4k" if (B, H, N, d) == (2, 16, 4096, 64) else "needle", B, H, N, d,
                    dtype, True, True, 1e-5, t(q1), t(k1), t(q2), t(k2), t(v),
                    np.full(H, 0.8), False, None, 0.8, None,
                    meta={"needle_pos": pos, "needle_query": N - n_needles + np.arange(n_needles)})


def rising(seed: int, *, B: int, H: int, N: int, d: int, slope: float = 3.5,
           q_gain: float = 4.0, dtype=torch.bfloat16, name: str | None = None) -> Workload:
    """Causal inputs whose logits climb along the key axis, for both maps.

    Per head and map a random unit direction u is drawn; queries are
    q_gain * u + 0.5 N(0,1) and key j is (0.5 + slope * j / 128) * u + N(0,1).
    With the defaults (|q . u| = 4, d = 64) the mean logit q . k_j / sqrt(d)
    grows by about 1.75 natural units (2.5 in base 2) per 128 keys, so every
    key tile of a row lies a few base-2 units above the one before and the row
    maximum moves on nearly every tile.  V ~ N(0,1).  Draw order: u1, u2, the
    noise of Q1, K1, Q2, K2, then V, lambda."""
    rng = np.random.default_rng(seed)
    u = [rng.standard_normal(size=(B, H, 1, d)) for _ in range(2)]
    u = [x / np.linalg.norm(x, axis=-1, keepdims=True) for x in u]
    pos = (0.5 + slope * np.arange(N) / 128.0).reshape(1, 1, N, 1)
    out = []
    for k in range(2):
        q = q_gain * u[k] + 0.5 * _normal(rng, (B, H, N, d))
        key = pos * u[k] + _normal(rng, (B, H, N, d))
        out += [q, key]
    v = _normal(rng, (B, H, N, 2 * d))
    lam = rng.uniform(0.3, 0.9, size=H)
    t = lambda x: _to_storage(x, dtype)
    nm = name or ("rising_4k" if (B, H, N, d) == (2, 16, 4096, 64) else f"rising_B{B}H{H}N{N}")
    return Workload(nm, B, H, N, d, dtype, True, True, 1e-5, t(out[0]), t(out[1]), t(out[2]),
                    t(out[3]), t(v), lam, False, 8, None, None)


def custom(seed: int, *, B: int, H: int, N: int, d: int, causal: bool, headnorm: bool = True,
           dtype=torch.bfloat16, lam_range=(0.1, 0.9), qk_scale: float = 1.0,
           random_w: bool = False, layer: int | None = 1, eps: float = 1e-5) -> Workload:
    """Arbitrary-shape inputs for parity sweeps (tile edges, ragged tails)."""
    rng, (q1, k1, q2, k2), v = random_heads(seed, B, H, N, d, dtype=dtype, qk_scale=qk_scale)
    lam = rng.uniform(lam_range[0], lam_range[1], size=H)
    w = None
    if random_w:
        w = (1.0 + 0.1 * rng.standard_normal(size=(H, 2 * d))).astype(np.float32).astype(np.float64)
    return Workload(f"custom_B{B}H{H}N{N}d{d}", B, H, N, d, dtype, causal, headnorm, eps,
                    q1, k1, q2, k2, v, lam, False, layer, None if layer else 0.0, w)


def kv_cache(seed: int, *, B: int, H: int, Nq: int, Nkv: int, d: int = 64, causal: bool = True,
             headnorm: bool = True, lam_range=(0.1, 0.9), random_w: bool = True,
             layer: int | None = 4, eps: float = 1e-5) -> Workload:
    """Queries against a key/value cache: Q1, Q2 [B, H, Nq, d], K1, K2 [B, H, Nkv, d],
    V [B, H, Nkv, 2d], all N(0,1) in bf16; the queries are the last Nq positions.
    Draw order: K1, K2, V, Q1, Q2, lambda, w."""
    rng = np.random.default_rng(seed)
    k1, k2 = (_to_storage(_normal(rng, (B, H, Nkv, d), 1.0), torch.bfloat16) for _ in range(2))
    v = _to_storage(_normal(rng, (B, H, Nkv, 2 * d), 1.0), torch.bfloat16)
    q1, q2 = (_to_storage(_normal(rng, (B, H, Nq, d), 1.0), torch.bfloat16) for _ in range(2))
    lam = rng.uniform(lam_range[0], lam_range[1], size=H)
    w = None
    if random_w:
        w = (1.0 + 0.1 * rng.standard_normal(size=(H, 2 * d))).astype(np.float32).astype(np.float64)
    return Workload(f"kv_B{B}H{H}Nq{Nq}Nkv{Nkv}", B, H, Nq, d, torch.bfloat16, causal, headnorm,
                    eps, q1, k1, q2, k2, v, lam, False, layer, None if layer else 0.0, w,
                    n_kv=Nkv)
