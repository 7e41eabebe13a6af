"""Pins for the float64 oracle: facts fixed by the page and by mathematics.

Each pin takes a loaded oracle library handle and returns (ok, detail).  They
are gathered here so that the same checks run against the real oracle
(``test_oracle.py``: every pin must hold) and against deliberately broken copies
of it (``test_oracle_mutants.py``: every planted mistake must trip at least one
pin).  Sources, all on the "Differential Transformer" glossary page (Ultralytics;
ja/pt/ar editions), section "How differential attention works":

  * the worked example and its printed result (row sums 0.20, 13 of 36
    weights negative);
  * each softmax map sums to 1, so each row of map1 - lambda map2 sums to
    1 - lambda, and weights may be negative;
  * each map is ordinary softmax attention (so lambda = 0, or identical maps,
    reduce to ordinary scaled-dot-product attention);
  * each head's output is normalised on its own and then multiplied by
    (1 - lambda_init), lambda_init(l) = 0.8 - 0.6 exp(-0.3 (l - 1)).
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from tests import bruteforce

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(None, 1)
            vals[k] = v
    return vals


def _rand(seed, B, H, N, d):
    rng = np.random.default_rng(seed)
    q1, k1, q2, k2 = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    v = rng.standard_normal((B, H, N, 2 * d))
    return rng, q1, k1, q2, k2, v


def _sdpa(q, k, v, causal):
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x))
    return F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=causal).numpy()


def pin_pages_example(lib):
    """The page's worked example: rows sum to 0.20 and 13 of 36 weights are negative."""
    g = _read_golden("pages_example.txt")
    gen = torch.Generator().manual_seed(int(g["seed"]))
    n, d, lam = int(g["n"]), int(g["d"]), float(g["lambda"])
    q1, k1, q2, k2 = torch.randn(4, n, d, generator=gen).double().numpy()
    wmap = oracle.diff_map(q1, k1, q2, k2, lam, causal=False, lib=lib)
    sums = wmap.sum(-1)
    neg = int((wmap < 0).sum())
    ok = (np.all(np.abs(sums - float(g["row_sum"])) < 1e-12) and neg == int(g["negative"])
          and wmap.size == int(g["total"]))
    return ok, f"row sums {sums}, negatives {neg} of {wmap.size}"


def pin_row_sum(lib):
    """Every row of map1 - lambda map2 sums to 1 - lambda (causal or not)."""
    _, q1, k1, q2, k2, _ = _rand(11, 1, 1, 37, 16)
    worst = 0.0
    for causal in (False, True):
        for lam in (0.0, 0.37, 0.8, 1.0, 1.6):
            wmap = oracle.diff_map(q1[0, 0], k1[0, 0], q2[0, 0], k2[0, 0], lam, causal=causal,
                                   lib=lib)
            worst = max(worst, float(np.max(np.abs(wmap.sum(-1) - (1.0 - lam)))))
            if causal and np.any(np.triu(wmap, 1) != 0.0):
                return False, "masked weight is nonzero"
    return worst < 1e-12, f"max |row sum - (1 - lambda)| = {worst:.3e}"


def pin_lambda_zero_is_sdpa(lib):
    """lambda = 0 leaves map1 V alone: ordinary softmax attention with scale 1/sqrt(d)."""
    _, q1, k1, q2, k2, v = _rand(12, 2, 3, 33, 16)
    worst = 0.0
    for causal in (False, True):
        o = oracle.fwd(q1, k1, q2, k2, v, np.zeros(3), causal=causal, headnorm=False, lib=lib)
        worst = max(worst, float(np.max(np.abs(o - _sdpa(q1, k1, v, causal)))))
    return worst < 1e-12, f"max err vs SDPA {worst:.3e}"


def pin_identical_maps(lib):
    """q2 = q1, k2 = k1 gives (1 - lambda_h) times ordinary attention, per head."""
    rng, q1, k1, _, _, v = _rand(13, 2, 3, 29, 8)
    lam = rng.uniform(-0.5, 1.5, size=3)
    worst = 0.0
    for causal in (False, True):
        o = oracle.fwd(q1, k1, q1, k1, v, lam, causal=causal, headnorm=False, lib=lib)
        ref = (1.0 - lam)[None, :, None, None] * _sdpa(q1, k1, v, causal)
        worst = max(worst, float(np.max(np.abs(o - ref))))
    return worst < 1e-12, f"max err {worst:.3e}"


def pin_headnorm_lambda_free(lib):
    """With identical maps and eps = 0 the normalised head output does not depend on
    lambda (< 1): the (1 - lambda) factor cancels in the RMS normalisation."""
    rng, q1, k1, _, _, v = _rand(14, 1, 2, 21, 8)
    w = rng.uniform(0.5, 1.5, size=(2, 16))
    outs = [oracle.fwd(q1, k1, q1, k1, v, np.full(2, lam), causal=True, headnorm=True, w=w,
                       eps=0.0, lambda_init_value=0.35, lib=lib) for lam in (0.0, 0.3, 0.9)]
    worst = max(float(np.max(np.abs(o - outs[0]))) for o in outs[1:])
    return worst < 1e-11, f"max spread over lambda {worst:.3e}"


def pin_causal_edges(lib):
    """Causal: row 0 sees only key 0, so o_0 = (1 - lambda) v_0; the last row sees all
    keys, so it equals the non-causal last row."""
    rng, q1, k1, q2, k2, v = _rand(15, 1, 2, 19, 8)
    lam = np.array([0.8, 0.25])
    oc = oracle.fwd(q1, k1, q2, k2, v, lam, causal=True, headnorm=False, lib=lib)
    on = oracle.fwd(q1, k1, q2, k2, v, lam, causal=False, headnorm=False, lib=lib)
    e0 = float(np.max(np.abs(oc[0, :, 0] - (1.0 - lam)[:, None] * v[0, :, 0])))
    e1 = float(np.max(np.abs(oc[0, :, -1] - on[0, :, -1])))
    differs = float(np.max(np.abs(oc[0, :, 1:-1] - on[0, :, 1:-1])))
    return e0 < 1e-14 and e1 < 1e-12 and differs > 1e-3, f"row0 {e0:.1e} last {e1:.1e}"


def pin_headnorm_is_rms_norm(lib):
    """The head normalisation equals torch rms_norm over the 2d channels with the
    head's weight, times (1 - lambda_init); checked through the full forward and
    through the standalone normalisation entry."""
    rng, q1, k1, q2, k2, v = _rand(16, 2, 3, 17, 8)
    lam = rng.uniform(0.1, 0.9, size=3)
    w = rng.uniform(0.5, 1.5, size=(3, 16))
    li = 0.6
    worst = 0.0
    for eps in (1e-5, 0.3):
        raw = oracle.fwd(q1, k1, q2, k2, v, lam, causal=True, headnorm=False, lib=lib)
        y = oracle.fwd(q1, k1, q2, k2, v, lam, causal=True, headnorm=True, w=w, eps=eps,
                       lambda_init_value=li, lib=lib)
        ref = np.empty_like(raw)
        for h in range(3):
            ref[:, h] = F.rms_norm(torch.from_numpy(raw[:, h]), (16,), torch.from_numpy(w[h]),
                                   eps).numpy() * (1.0 - li)
        worst = max(worst, float(np.max(np.abs(y - ref))))
        flat = raw.reshape(-1, 16)
        hidx = np.tile(np.repeat(np.arange(3), 17), 2)
        y2 = oracle.headnorm(flat, hidx, w, H=3, eps=eps, lambda_init_value=li, lib=lib)
        worst = max(worst, float(np.max(np.abs(y2 - ref.reshape(-1, 16)))))
    return worst < 1e-12, f"max err vs rms_norm {worst:.3e}"


def pin_headnorm_closed_form(lib):
    """With weight 1: mean_c y^2 = (1 - lambda_init)^2 ms / (ms + eps), ms = mean_c o^2."""
    rng, q1, k1, q2, k2, v = _rand(17, 1, 2, 23, 8)
    lam = np.array([0.5, 0.9])
    eps, li = 0.05, 0.25
    raw = oracle.fwd(q1, k1, q2, k2, v, lam, causal=False, headnorm=False, lib=lib)
    y = oracle.fwd(q1, k1, q2, k2, v, lam, causal=False, headnorm=True, eps=eps,
                   lambda_init_value=li, lib=lib)
    ms = (raw ** 2).mean(-1)
    err = float(np.max(np.abs((y ** 2).mean(-1) - (1 - li) ** 2 * ms / (ms + eps))))
    return err < 1e-12, f"max err {err:.3e}"


def pin_permutation(lib):
    """Non-causal: permuting the rows of K1, K2 and V together leaves the output unchanged."""
    rng, q1, k1, q2, k2, v = _rand(18, 1, 2, 25, 8)
    lam = np.array([0.7, 0.2])
    perm = rng.permutation(25)
    o = oracle.fwd(q1, k1, q2, k2, v, lam, causal=False, headnorm=False, lib=lib)
    op = oracle.fwd(q1, k1[:, :, perm], q2, k2[:, :, perm], v[:, :, perm], lam, causal=False,
                    headnorm=False, lib=lib)
    err = float(np.max(np.abs(o - op)))
    return err < 1e-12, f"max err {err:.3e}"


def pin_linear_in_v(lib):
    """Without the normalisation the output is linear in V."""
    rng, q1, k1, q2, k2, v = _rand(19, 1, 2, 14, 8)
    v2 = rng.standard_normal(v.shape)
    lam = np.array([0.8, 0.4])
    f = lambda vv: oracle.fwd(q1, k1, q2, k2, vv, lam, causal=True, headnorm=False, lib=lib)
    err = float(np.max(np.abs(f(2.5 * v - 0.75 * v2) - (2.5 * f(v) - 0.75 * f(v2)))))
    return err < 1e-12, f"max err {err:.3e}"


def pin_zero_queries(lib):
    """Zero queries give uniform maps: o_i = (1 - lambda) mean of the visible v_j."""
    rng, _, k1, _, k2, v = _rand(20, 1, 2, 11, 8)
    q = np.zeros_like(k1)
    lam = np.array([0.8, -0.3])
    worst = 0.0
    for causal in (False, True):
        o = oracle.fwd(q, k1, q, k2, v, lam, causal=causal, headnorm=False, lib=lib)
        if causal:
            ref = np.cumsum(v, axis=2) / np.arange(1, 12)[None, None, :, None]
        else:
            ref = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
        ref = (1.0 - lam)[None, :, None, None] * ref
        worst = max(worst, float(np.max(np.abs(o - ref))))
    return worst < 1e-13, f"max err {worst:.3e}"


def pin_bruteforce(lib):
    """Pure-Python loops on tiny shapes agree to 1e-12."""
    worst = 0.0
    for seed, (B, H, N, d), causal in [(21, (1, 1, 1, 1), True), (22, (1, 2, 5, 3), False),
                                       (23, (2, 2, 16, 8), True), (24, (1, 3, 9, 4), False)]:
        rng, q1, k1, q2, k2, v = _rand(seed, B, H, N, d)
        lam = rng.uniform(-0.2, 1.2, size=H)
        w = rng.uniform(0.5, 1.5, size=(H, 2 * d))
        for headnorm in (False, True):
            o = oracle.fwd(q1, k1, q2, k2, v, lam, causal=causal, headnorm=headnorm, w=w,
                           eps=1e-3, lambda_init_value=0.45, lib=lib)
            for b in range(B):
                for h in range(H):
                    ref = bruteforce.head_forward(q1[b, h].tolist(), k1[b, h].tolist(),
                                                  q2[b, h].tolist(), k2[b, h].tolist(),
                                                  v[b, h].tolist(), float(lam[h]), causal,
                                                  headnorm, w[h].tolist(), 1e-3, 0.45)
                    worst = max(worst, float(np.max(np.abs(o[b, h] - np.array(ref)))))
    return worst < 1e-12, f"max err {worst:.3e}"


def pin_lambda_init(lib):
    """lambda_init(1) = 0.8 - 0.6 = 0.2; it rises with depth towards 0.8."""
    vals = [oracle.lambda_init(l, lib=lib) for l in range(1, 60)]
    ok = (abs(vals[0] - 0.2) < 1e-15 and all(b > a for a, b in zip(vals, vals[1:]))
          and abs(oracle.lambda_init(400, lib=lib) - 0.8) < 1e-15
          and abs(vals[1] - (0.8 - 0.6 / math.e ** 0.3)) < 1e-15)
    return ok, f"l=1 {vals[0]!r}, l=2 {vals[1]!r}, l=59 {vals[-1]!r}"


def pin_rows_match_full(lib):
    """The selected-rows entry computes the same rows as the full forward."""
    rng, q1, k1, q2, k2, v = _rand(25, 2, 3, 20, 8)
    lam = rng.uniform(0.1, 0.9, size=3)
    w = rng.uniform(0.5, 1.5, size=(3, 16))
    kw = dict(causal=True, headnorm=True, w=w, eps=1e-5, lambda_init_value=0.3, lib=lib)
    full = oracle.fwd(q1, k1, q2, k2, v, lam, **kw)
    bh = rng.integers(0, 6, size=40)
    ri = rng.integers(0, 20, size=40)
    rows = oracle.fwd_rows(q1, k1, q2, k2, v, lam, bh, ri, **kw)
    err = float(np.max(np.abs(rows - full.reshape(6, 20, 16)[bh, ri])))
    return err == 0.0, f"max err {err:.3e}"


def _rand_kv(seed, B, H, Nq, Nkv, d):
    rng = np.random.default_rng(seed)
    q1, q2 = (rng.standard_normal((B, H, Nq, d)) for _ in range(2))
    k1, k2 = (rng.standard_normal((B, H, Nkv, d)) for _ in range(2))
    v = rng.standard_normal((B, H, Nkv, 2 * d))
    return rng, q1, k1, q2, k2, v


def pin_kv_bruteforce(lib):
    """Key/value-cache form (fewer queries than keys, queries at the last positions)
    agrees with pure-Python loops to 1e-12, full and selected rows."""
    worst = 0.0
    for seed, (B, H, Nq, Nkv, d), causal in [(41, (1, 2, 3, 7, 4), True),
                                             (42, (2, 1, 5, 9, 3), False),
                                             (43, (1, 1, 1, 6, 2), True),
                                             (44, (1, 2, 4, 4, 3), True),
                                             (45, (2, 2, 2, 11, 4), True)]:
        rng, q1, k1, q2, k2, v = _rand_kv(seed, B, H, Nq, Nkv, d)
        lam = rng.uniform(-0.2, 1.2, size=H)
        w = rng.uniform(0.5, 1.5, size=(H, 2 * d))
        for headnorm in (False, True):
            kw = dict(causal=causal, headnorm=headnorm, w=w, eps=1e-3, lambda_init_value=0.45,
                      lib=lib)
            o = oracle.fwd_kv(q1, k1, q2, k2, v, lam, **kw)
            bh = rng.integers(0, B * H, size=7)
            ri = rng.integers(0, Nq, size=7)
            rows = oracle.fwd_kv(q1, k1, q2, k2, v, lam, bh_idx=bh, row_idx=ri, **kw)
            for b in range(B):
                for h in range(H):
                    ref = np.array(bruteforce.head_forward(
                        q1[b, h].tolist(), k1[b, h].tolist(), q2[b, h].tolist(),
                        k2[b, h].tolist(), v[b, h].tolist(), float(lam[h]), causal, headnorm,
                        w[h].tolist(), 1e-3, 0.45))
                    worst = max(worst, float(np.max(np.abs(o[b, h] - ref))))
                    sel = bh == b * H + h
                    if sel.any():
                        worst = max(worst, float(np.max(np.abs(rows[sel] - ref[ri[sel]]))))
    return worst < 1e-12, f"max err {worst:.3e}"


def pin_kv_last_rows(lib):
    """Attending with the last Nq queries against the whole key/value sequence gives
    exactly the last Nq rows of the full (square) forward."""
    worst = 0.0
    for seed, causal in [(46, True), (47, False)]:
        rng, q1, k1, q2, k2, v = _rand(seed, 2, 2, 13, 4)
        lam = rng.uniform(0.1, 0.9, size=2)
        kw = dict(causal=causal, headnorm=True, eps=1e-5, lambda_init_value=0.3, lib=lib)
        full = oracle.fwd(q1, k1, q2, k2, v, lam, **kw)
        for nq in (1, 5, 13):
            o = oracle.fwd_kv(q1[:, :, -nq:], k1, q2[:, :, -nq:], k2, v, lam, **kw)
            worst = max(worst, float(np.max(np.abs(o - full[:, :, -nq:]))))
    return worst == 0.0, f"max err {worst:.3e}"


def pin_kv_zero_queries(lib):
    """Zero queries give uniform maps, so causal query i of Nq against Nkv keys is
    (1 - lambda) times the mean of v_0 .. v_{Nkv - Nq + i}."""
    rng = np.random.default_rng(48)
    Nq, Nkv, d = 4, 10, 3
    q = np.zeros((1, 2, Nq, d))
    k1, k2 = rng.standard_normal((2, 1, 2, Nkv, d))
    v = rng.standard_normal((1, 2, Nkv, 2 * d))
    lam = np.array([0.25, -0.5])
    o = oracle.fwd_kv(q, k1, q, k2, v, lam, causal=True, headnorm=False, lib=lib)
    ref = np.cumsum(v, axis=2)[:, :, Nkv - Nq:] / np.arange(Nkv - Nq + 1, Nkv + 1)[:, None]
    ref = (1.0 - lam)[None, :, None, None] * ref
    err = float(np.max(np.abs(o - ref)))
    return err < 1e-13, f"max err {err:.3e}"


def _fd_grads(lib, tensors, lam, w, dy, causal, headnorm, eps, li, h=1e-6):
    """Central differences of L = sum(y * dy) through the forward oracle."""
    names = ["q1", "k1", "q2", "k2", "v"]
    params = dict(zip(names, [t.copy() for t in tensors]))
    params["lam"] = lam.copy()
    params["w"] = w.copy()

    def loss():
        y = oracle.fwd(*(params[n] for n in names), params["lam"], causal=causal,
                       headnorm=headnorm, w=params["w"], eps=eps, lambda_init_value=li,
                       lib=lib)
        return float(np.sum(y * dy))

    grads = {}
    for n, arr in params.items():
        g = np.zeros_like(arr)
        flat, gflat = arr.reshape(-1), g.reshape(-1)
        for idx in range(flat.size):
            keep = flat[idx]
            flat[idx] = keep + h
            lp = loss()
            flat[idx] = keep - h
            lm = loss()
            flat[idx] = keep
            gflat[idx] = (lp - lm) / (2 * h)
        grads[n] = g
    return grads


def pin_bwd_finite_differences(lib):
    """Every gradient of the backward oracle matches central differences of the
    forward oracle (loss sum(y * dy)), causal or not, without the norm and with
    either form of it (RMS, group)."""
    worst = 0.0
    for seed, causal, headnorm in [(61, True, 1), (62, False, 1), (63, True, 0),
                                   (64, False, 0), (65, True, 2), (66, False, 2)]:
        rng, q1, k1, q2, k2, v = _rand(seed, 1, 2, 5, 3)
        lam = rng.uniform(-0.3, 1.2, size=2)
        w = rng.uniform(0.5, 1.5, size=(2, 6))
        dy = rng.standard_normal(v.shape)
        eps, li = 1e-2, 0.35
        g = oracle.bwd(q1, k1, q2, k2, v, lam, dy, causal=causal, headnorm=headnorm, w=w,
                       eps=eps, lambda_init_value=li, lib=lib)
        fd = _fd_grads(lib, [q1, k1, q2, k2, v], lam, w, dy, causal, headnorm, eps, li)
        pairs = [("dq1", "q1"), ("dk1", "k1"), ("dq2", "q2"), ("dk2", "k2"), ("dv", "v"),
                 ("dlam", "lam"), ("dw", "w")]
        for gn, pn in pairs:
            scale = max(1.0, float(np.max(np.abs(fd[pn]))))
            worst = max(worst, float(np.max(np.abs(g[gn] - fd[pn]))) / scale)
    return worst < 1e-7, f"max rel err {worst:.3e}"


def pin_bwd_lambda_zero_is_sdpa_grad(lib):
    """lambda = 0, no norm: map 2 gets no gradient and the rest is the float64 autograd
    gradient of torch scaled_dot_product_attention (an independent implementation)."""
    worst = 0.0
    for seed, causal in [(65, True), (66, False)]:
        rng, q1, k1, q2, k2, v = _rand(seed, 2, 2, 9, 4)
        dy = rng.standard_normal(v.shape)
        g = oracle.bwd(q1, k1, q2, k2, v, np.zeros(2), dy, causal=causal, headnorm=False,
                       lib=lib)
        tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_() for x in (q1, k1, v))
        out = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
        out.backward(torch.from_numpy(dy))
        worst = max(worst, float(np.max(np.abs(g["dq1"] - tq.grad.numpy()))),
                    float(np.max(np.abs(g["dk1"] - tk.grad.numpy()))),
                    float(np.max(np.abs(g["dv"] - tv.grad.numpy()))),
                    float(np.max(np.abs(g["dq2"]))), float(np.max(np.abs(g["dk2"]))))
    return worst < 1e-12, f"max err {worst:.3e}"


def pin_bwd_d128_is_sdpa_grad(lib):
    """The backward oracle at the d = 128 head width (values 256 wide): with lambda = 0
    and no norm, map 1's gradients and dv are the float64 autograd gradient of torch
    scaled_dot_product_attention, map 2's are zero; with lambda = 1 and identical maps
    the output (1 - lambda) SDPA is identically zero, so dv and the two maps' summed dq
    and dk vanish, while dlambda = -sum(SDPA * dy)."""
    worst = 0.0
    for seed, causal in [(68, True), (69, False)]:
        rng, q1, k1, q2, k2, v = _rand(seed, 1, 2, 6, 128)
        dy = rng.standard_normal(v.shape)
        g = oracle.bwd(q1, k1, q2, k2, v, np.zeros(2), dy, causal=causal, headnorm=False,
                       lib=lib)
        tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_() for x in (q1, k1, v))
        out = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
        out.backward(torch.from_numpy(dy))
        worst = max(worst, float(np.max(np.abs(g["dq1"] - tq.grad.numpy()))),
                    float(np.max(np.abs(g["dk1"] - tk.grad.numpy()))),
                    float(np.max(np.abs(g["dv"] - tv.grad.numpy()))),
                    float(np.max(np.abs(g["dq2"]))), float(np.max(np.abs(g["dk2"]))))
        g = oracle.bwd(q1, k1, q1, k1, v, np.ones(2), dy, causal=causal, headnorm=False,
                       lib=lib)
        dlam_ref = -np.sum(_sdpa(q1, k1, v, causal) * dy, axis=(0, 2, 3))
        worst = max(worst, float(np.max(np.abs(g["dv"]))),
                    float(np.max(np.abs(g["dlam"] - dlam_ref))),
                    float(np.max(np.abs(g["dq1"] + g["dq2"]))),
                    float(np.max(np.abs(g["dk1"] + g["dk2"]))))
    return worst < 1e-11, f"max err {worst:.3e}"


def pin_bwd_identical_maps_lambda(lib):
    """q2 = q1, k2 = k1, no norm: y = (1 - lambda) SDPA, so dL/dlambda = -sum(SDPA * dy)."""
    rng, q1, k1, _, _, v = _rand(67, 2, 3, 7, 4)
    lam = rng.uniform(0.1, 0.9, size=3)
    dy = rng.standard_normal(v.shape)
    g = oracle.bwd(q1, k1, q1, k1, v, lam, dy, causal=True, headnorm=False, lib=lib)
    ref = -np.sum(_sdpa(q1, k1, v, True) * dy, axis=(0, 2, 3))
    err = float(np.max(np.abs(g["dlam"] - ref)))
    return err < 1e-12, f"max err {err:.3e}"


def pin_groupnorm_is_torch_group_norm(lib):
    """headnorm = 2 equals torch group_norm with one group over the 2d channels of each
    (batch, head, token) and the head's weight, times (1 - lambda_init); also through the
    standalone entry."""
    rng, q1, k1, q2, k2, v = _rand(71, 2, 3, 10, 4)
    lam = rng.uniform(0.1, 0.9, size=3)
    w = rng.uniform(0.5, 1.5, size=(3, 8))
    eps, li = 1e-3, 0.4
    raw = oracle.fwd(q1, k1, q2, k2, v, lam, causal=True, headnorm=0, lib=lib)
    got = oracle.fwd(q1, k1, q2, k2, v, lam, causal=True, headnorm=2, w=w, eps=eps,
                     lambda_init_value=li, lib=lib)
    worst = 0.0
    for h in range(3):
        x = torch.from_numpy(raw[:, h].reshape(-1, 8, 1).copy())
        ref = F.group_norm(x, 1, weight=torch.from_numpy(w[h].copy()), eps=eps).numpy()
        ref = ref.reshape(raw[:, h].shape) * (1 - li)
        worst = max(worst, float(np.max(np.abs(got[:, h] - ref))))
    hidx = np.tile(np.repeat(np.arange(3), 10), 2)
    alone = oracle.groupnorm(raw.reshape(-1, 8), hidx, w, H=3, eps=eps, lambda_init_value=li,
                             lib=lib)
    worst = max(worst, float(np.max(np.abs(alone - got.reshape(-1, 8)))))
    return worst < 1e-12, f"max err {worst:.3e}"


def pin_groupnorm_shift_invariance(lib):
    """Adding the same constant to every entry of V shifts each o channel by
    (1 - lambda) times it (rows of map1 - lambda map2 sum to 1 - lambda), which the
    mean-subtracting norm removes; the RMS norm does not."""
    rng, q1, k1, q2, k2, v = _rand(72, 1, 2, 9, 4)
    lam = np.array([0.3, 0.6])
    w = rng.uniform(0.5, 1.5, size=(2, 8))
    kw = dict(causal=True, w=w, eps=1e-4, lambda_init_value=0.25, lib=lib)
    a = oracle.fwd(q1, k1, q2, k2, v, lam, headnorm=2, **kw)
    b = oracle.fwd(q1, k1, q2, k2, v + 3.0, lam, headnorm=2, **kw)
    r1 = oracle.fwd(q1, k1, q2, k2, v, lam, headnorm=1, **kw)
    r2 = oracle.fwd(q1, k1, q2, k2, v + 3.0, lam, headnorm=1, **kw)
    err = float(np.max(np.abs(a - b)))
    rms_moves = float(np.max(np.abs(r1 - r2)))
    return err < 1e-10 and rms_moves > 1e-3, f"group shift err {err:.3e}, rms moves {rms_moves:.3e}"


def pin_groupnorm_closed_form(lib):
    """With weight 1, each output row has mean 0 and mean square
    (1 - lambda_init)^2 var / (var + eps), var = the row's variance of o."""
    rng, q1, k1, q2, k2, v = _rand(73, 1, 2, 12, 4)
    lam = np.array([0.5, 0.7])
    eps, li = 1e-2, 0.3
    raw = oracle.fwd(q1, k1, q2, k2, v, lam, causal=False, headnorm=0, lib=lib)
    y = oracle.fwd(q1, k1, q2, k2, v, lam, causal=False, headnorm=2, eps=eps,
                   lambda_init_value=li, lib=lib)
    var = raw.var(axis=-1)
    e1 = float(np.max(np.abs(y.mean(axis=-1))))
    e2 = float(np.max(np.abs((y ** 2).mean(axis=-1) - (1 - li) ** 2 * var / (var + eps))))
    return max(e1, e2) < 1e-13, f"mean err {e1:.3e}, ms err {e2:.3e}"


PINS = {name[4:]: fn for name, fn in sorted(globals().items()) if name.startswith("pin_")}


def run_pins(lib):
    """Run every pin; returns {name: (ok, detail)}.  An exception counts as a failure."""
    res = {}
    for name, fn in PINS.items():
        try:
            with np.errstate(all="ignore"):
                ok, detail = fn(lib)
            res[name] = (bool(ok), detail)
        except Exception as e:  # a crash is a failed pin
            res[name] = (False, f"{type(e).__name__}: {e}")
    return res
