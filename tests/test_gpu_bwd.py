"""Backward pass on the GPU (diffattn_fwd_train + diffattn_bwd) against the float64
oracle's gradients.

Tolerance per gradient tensor: max-abs <= 2e-2 * max|oracle| (bf16 inputs, P, dS and
do on the tensor cores, fp32 accumulation; bf16 dq, dk, dv outputs).  dlambda =
-sum_rows do . o_2 cancels heavily (the head norm leaves do nearly orthogonal to o), so
its error is a sum of random-sign rounding errors of the rows' terms (the forward's
bf16 P in o_k): it grows with the square root of the row width, and its bound is
2e-2 * sqrt(d / 64) * max|oracle| (the d = 64 bound at d = 64).
"""
import numpy as np
import pytest
import torch

import oracle
from differential_attention_attn_gb300 import ops
from differential_attention_attn_gb300 import workloads as W
from tests import harness

pytestmark = pytest.mark.gpu

GRADS = ("dq1", "dk1", "dq2", "dk2", "dv", "dlam", "dw")


def _dy(w, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.standard_normal((w.B, w.H, w.N, 2 * w.d))).to(torch.bfloat16)


def _run(w, dy, *, status=None):
    li = harness.lambda_init_for(w, "gpu")
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device="cuda")
    nw = None if w.w is None else torch.tensor(w.w, dtype=torch.float32, device="cuda")
    dev = [t.cuda() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    kw = dict(causal=w.causal, headnorm=w.headnorm, norm_w=nw, eps=float(np.float32(w.eps)),
              lambda_init=li)
    out, saved = ops.fwd_train(*dev, lam, status=status, **kw)
    g = ops.bwd(*dev, lam, saved, dy.cuda(), status=status, **kw)
    torch.cuda.synchronize()
    return out, g


def _oracle(w, dy):
    args, kw = harness.oracle_args(w)
    return oracle.bwd(*args, dy.double().numpy(), **kw)


def _cmp(g, ref, what, names=GRADS):
    d = g["dq1"].shape[-1]
    for k in names:
        got = g[k].double().cpu().numpy()
        assert np.all(np.isfinite(got)), f"{what} {k}: non-finite"
        mx = float(np.max(np.abs(ref[k])))
        err = float(np.max(np.abs(got - ref[k])))
        rel = 2e-2 * (np.sqrt(d / 64) if k == "dlam" else 1.0)
        assert err <= rel * mx + 1e-6, f"{what} {k}: max-abs err {err:.3g} > {rel:.3g} * {mx:.3g}"


@pytest.mark.parametrize("N", [1, 7, 128, 129, 200, 256, 384])
@pytest.mark.parametrize("causal", [True, False])
def test_bwd_tile_edges(N, causal):
    w = W.custom(500 + N, B=2, H=2, N=N, d=64, causal=causal, headnorm=True, random_w=True,
                 layer=6)
    dy = _dy(w, N)
    _, g = _run(w, dy)
    _cmp(g, _oracle(w, dy), f"N={N} causal={causal}")


# With the head norm, lambda = 1 is left out: a causal row whose maps agree (row 0
# sees only key 0, so o1 = o2 = v_0) has o = o1 - o2 = 0, and rows near it nearly
# cancel; the norm divides by rms(o), amplifying the bf16 rounding of P by
# |o1| / |o| without bound.  Without the norm nothing amplifies, so lambda = 1 is
# tested there.
@pytest.mark.parametrize("lam,headnorm", [(0.0, True), (0.8, True), (-0.5, True),
                                          (0.0, False), (1.0, False), (-0.5, False)])
def test_bwd_lambda_and_norm(lam, headnorm):
    w = W.custom(17, B=1, H=3, N=320, d=64, causal=True, headnorm=headnorm, random_w=True,
                 layer=3)
    w.lam_offset = np.full(w.H, lam)
    dy = _dy(w, 5)
    _, g = _run(w, dy)
    names = GRADS if headnorm else GRADS[:-1]
    _cmp(g, _oracle(w, dy), f"lambda={lam} headnorm={headnorm}", names)
    if not headnorm:
        assert float(g["dw"].abs().max()) == 0.0


def test_bwd_larger_many_items():
    """Eight key tiles per head, 128 work items: B=2, H=4, N=1024 (every row)."""
    w = W.custom(23, B=2, H=4, N=1024, d=64, causal=True, headnorm=True, random_w=True,
                 layer=8)
    dy = _dy(w, 23)
    _, g = _run(w, dy)
    _cmp(g, _oracle(w, dy), "B2H4N1024")


@pytest.mark.parametrize("B,H,N,causal", [(8, 16, 384, True), (4, 16, 256, False),
                                          (2, 8, 1408, True), (5, 8, 333, True)])
def test_bwd_several_items_per_cta(B, H, N, causal):
    """More (key tile, head, map) work items than a GB300 has SMs (152), so the
    persistent gradient kernel walks several items per CTA: accumulators handed
    from one item's epilogue to the next item's MMAs, K and V reloaded, and the
    last dQ tile of one item drained during the next.  Items of different
    lengths (causal) and ragged key tiles (N = 333, 1408) meet in one CTA."""
    assert 2 * B * H * -(-N // 128) > 152
    w = W.custom(900 + N, B=B, H=H, N=N, d=64, causal=causal, headnorm=True, random_w=True,
                 layer=5)
    dy = _dy(w, 900 + N)
    _, g = _run(w, dy)
    _cmp(g, _oracle(w, dy), f"B{B}H{H}N{N} causal={causal}")


def test_fwd_train_output_is_the_forward():
    w = W.custom(29, B=1, H=2, N=300, d=64, causal=True, headnorm=True, random_w=True, layer=2)
    out, _ = _run(w, _dy(w, 1))
    assert torch.equal(out, harness.run_gpu(w))


def test_bwd_status_clear_and_repeatable():
    w = W.custom(31, B=1, H=2, N=512, d=64, causal=True, headnorm=True, layer=4)
    dy = _dy(w, 2)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, a = _run(w, dy, status=status)
    _, b = _run(w, dy, status=status)
    assert int(status.item()) == 0
    for k in ("dk1", "dk2", "dlam"):  # written without cross-CTA accumulation order effects
        if k == "dlam":
            assert torch.allclose(a[k], b[k], rtol=1e-5, atol=1e-5)
        else:
            assert torch.equal(a[k], b[k])
    for k in ("dq1", "dq2", "dv"):  # fp32 atomics: order may differ, values agree closely
        assert torch.allclose(a[k].float(), b[k].float(), rtol=2e-2, atol=1e-2)


@pytest.mark.parametrize("N,causal", [(7, True), (200, True), (256, False), (384, True)])
@pytest.mark.parametrize("lam", [0.8, -0.5])
def test_bwd_group_norm(N, causal, lam):
    """headnorm = 2 (the page's GroupNorm, mean-subtracting): every gradient, including
    the norm weight's, against the oracle; the training forward's output equals the
    plain forward's bitwise."""
    w = W.custom(700 + N, B=2, H=2, N=N, d=64, causal=causal, headnorm=2, random_w=True,
                 layer=5)
    w.lam_offset = np.full(w.H, lam)
    dy = _dy(w, N + 1)
    out, g = _run(w, dy)
    _cmp(g, _oracle(w, dy), f"group norm N={N} causal={causal} lambda={lam}")
    assert torch.equal(out, harness.run_gpu(w))


def _bnhd(t):
    """A [B, H, N, w] view of [B, N, H, w] storage holding the same values."""
    return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)


@pytest.mark.parametrize("causal,headnorm,N,d", [(True, 1, 333, 64), (False, 2, 256, 64),
                                                 (True, 0, 130, 64), (True, 1, 200, 128),
                                                 (False, 2, 256, 128)])
def test_train_strided_matches_contiguous(causal, headnorm, N, d):
    """fwd_train_strided / bwd_strided on [B, N, H, .] storage (inputs, dy and every
    gradient): out, saved and dk bitwise equal to the contiguous calls; dq, dv,
    dlambda and dw up to the order of their fp32 atomic sums; and the gradients within
    the oracle tolerance."""
    w = W.custom(900 + N, B=2, H=3, N=N, d=d, causal=causal, headnorm=headnorm,
                 random_w=True, layer=5)
    dy = _dy(w, 31)
    li = harness.lambda_init_for(w, "gpu")
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device="cuda")
    nw = None if w.w is None else torch.tensor(w.w, dtype=torch.float32, device="cuda")
    dev = [t.cuda() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    kw = dict(causal=causal, headnorm=headnorm, norm_w=nw, eps=float(np.float32(w.eps)),
              lambda_init=li)
    out_c, saved_c = ops.fwd_train(*dev, lam, **kw)
    g_c = ops.bwd(*dev, lam, saved_c, dy.cuda(), **kw)

    views = [_bnhd(t) for t in dev]
    assert not views[0].is_contiguous()
    out_s = _bnhd(torch.empty_like(out_c))
    out_s, saved_s = ops.fwd_train_strided(*views, lam, out=out_s, **kw)
    grads = {k: _bnhd(torch.empty_like(g_c[k])) for k in ("dq1", "dk1", "dq2", "dk2", "dv")}
    grads["dlam"] = torch.empty_like(g_c["dlam"])
    grads["dw"] = torch.zeros_like(g_c["dw"])
    g_s = ops.bwd_strided(*views, lam, saved_s, _bnhd(dy.cuda()), grads=grads, **kw)
    torch.cuda.synchronize()

    assert torch.equal(out_s, out_c)
    assert torch.equal(saved_s, saved_c)
    for k in ("dk1", "dk2"):
        assert torch.equal(g_s[k], g_c[k]), k
    for k in ("dq1", "dq2", "dv", "dlam", "dw"):
        a, b = g_s[k].float(), g_c[k].float()
        tol = 2 ** -7 * float(b.abs().max()) + 1e-6
        assert float((a - b).abs().max()) <= tol, k
    names = GRADS if headnorm else GRADS[:-1]
    _cmp({k: v.contiguous() for k, v in g_s.items()}, _oracle(w, dy), f"strided N={N} d={d}",
         names)


@pytest.mark.parametrize("N,causal,headnorm", [(2, True, 1), (7, False, 2), (128, True, 1),
                                               (200, True, 1), (256, False, 2), (384, True, 0),
                                               (130, False, 1)])
def test_bwd_d128(N, causal, headnorm):
    """d = 128 (values 256 wide): the saving forward's output equals the plain
    forward's bitwise, and every gradient is within the oracle tolerance.

    N = 2 rather than 1: with one key every dq and dk is exactly zero (dS = dW - D
    cancels), and the d = 128 path rebuilds o_1 = o + lambda o_2 from the forward's
    bf16-weighted accumulator, so they come out at rounding level (about 1e-5) with no
    scale for a relative bound; at N = 2 row 0 is that degenerate row and row 1 gives
    the tensor its scale.  N = 1 runs in the bounds-checked build."""
    w = W.custom(1100 + N, B=2, H=2, N=N, d=128, causal=causal, headnorm=headnorm,
                 random_w=True, layer=5)
    dy = _dy(w, N + 3)
    out, g = _run(w, dy)
    names = GRADS if headnorm else GRADS[:-1]
    _cmp(g, _oracle(w, dy), f"d=128 N={N} causal={causal} headnorm={headnorm}", names)
    assert torch.equal(out, harness.run_gpu(w))


@pytest.mark.parametrize("causal", [True, False])
def test_bwd_d128_many_items(causal):
    """d = 128 with more dV and dK/dQ items than SMs (B=3, H=4, N=1100: 9 key tiles, a
    ragged last one, 108 dV and 216 dK/dQ items; non-causal, every item the same length)."""
    w = W.custom(1200, B=3, H=4, N=1100, d=128, causal=causal, headnorm=1, random_w=True,
                 layer=7)
    dy = _dy(w, 1200)
    _, g = _run(w, dy)
    _cmp(g, _oracle(w, dy), f"d=128 B3H4N1100 causal={causal}")


@pytest.mark.parametrize("lam,headnorm", [(0.0, 1), (-0.5, 1), (0.8, 2), (1.0, 0), (-0.5, 0)])
def test_bwd_d128_lambda_and_norm(lam, headnorm):
    """d = 128 with lambda at 0, negative, and 1 (without the norm, as at d = 64: with it a
    row whose maps agree has o = 0 and the norm amplifies P's rounding without bound)."""
    w = W.custom(19, B=1, H=3, N=320, d=128, causal=True, headnorm=headnorm, random_w=True,
                 layer=3)
    w.lam_offset = np.full(w.H, lam)
    dy = _dy(w, 6)
    _, g = _run(w, dy)
    names = GRADS if headnorm else GRADS[:-1]
    _cmp(g, _oracle(w, dy), f"d=128 lambda={lam} headnorm={headnorm}", names)
    if not headnorm:
        assert float(g["dw"].abs().max()) == 0.0


@pytest.mark.parametrize("N,causal", [(200, True), (130, False)])
def test_saved_d128_matches_oracle(N, causal):
    """The d = 128 saved activations themselves: the pre-norm o = o_1 - lambda o_2 (the
    oracle's forward without the norm), o_2 (its forward with lambda = 0 and the query/key
    pairs swapped) and each map's log2-sum-exp, log2 sum_j 2^(q.k_j log2e / sqrt(d)) over
    the visible keys, written out in float64 here."""
    w = W.custom(1300 + N, B=2, H=2, N=N, d=128, causal=causal, headnorm=1, random_w=True,
                 layer=4)
    li = harness.lambda_init_for(w, "gpu")
    lam_np = np.asarray(w.lambdas(li), dtype=np.float32)
    lam = torch.tensor(lam_np, device="cuda")
    nw = torch.tensor(w.w, dtype=torch.float32, device="cuda")
    dev = [t.cuda() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    _, saved = ops.fwd_train(*dev, lam, causal=causal, headnorm=1, norm_w=nw,
                             eps=float(np.float32(w.eps)), lambda_init=li)
    torch.cuda.synchronize()
    B, H, d, BH = w.B, w.H, w.d, w.B * w.H
    n_pad = -(-N // 128) * 128
    f = saved.view(torch.float32).cpu().numpy().astype(np.float64)
    o_all = f[:2 * BH * N * 2 * d].reshape(2, B, H, N, 2 * d)
    off = (2 * BH * N * 2 * d * 4 + 255) // 256 * 256 // 4
    lse = f[off:off + 2 * BH * n_pad].reshape(2, B, H, n_pad)[..., :N]
    q1, k1, q2, k2, v = (t.double().numpy() for t in (w.q1, w.k1, w.q2, w.k2, w.v))
    o_ref = oracle.fwd(q1, k1, q2, k2, v, lam_np.astype(np.float64), causal=causal,
                       headnorm=False)
    o2_ref = oracle.fwd(q2, k2, q1, k1, v, np.zeros(H), causal=causal, headnorm=False)
    for got, ref, name in ((o_all[0], o_ref, "o"), (o_all[1], o2_ref, "o2")):
        err = float(np.max(np.abs(got - ref)))
        assert err <= 2e-2 * float(np.max(np.abs(ref))), f"{name}: max-abs err {err:.3g}"
    for k, (q, kk) in enumerate(((q1, k1), (q2, k2))):
        s = np.einsum("bhid,bhjd->bhij", q, kk) / np.sqrt(d)
        if causal:
            s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
        m = s.max(axis=-1, keepdims=True)
        ref = (m[..., 0] + np.log(np.exp(s - m).sum(axis=-1))) / np.log(2.0)
        err = float(np.max(np.abs(lse[k] - ref)))
        assert err <= 2e-3, f"lse of map {k + 1}: max-abs err {err:.3g}"


def _full_size(name):
    if name == "needle_4k":  # the needle_4k_bwd bench configuration (d = 64)
        w = W.make("needle_4k")
        return w, float(np.float32(w.lambda_init_override))
    # the wide_4k_bwd bench configuration (d = 128)
    w = W.custom(3000, B=2, H=8, N=4096, d=128, causal=True, headnorm=True, random_w=True,
                 layer=12)
    return w, float(np.float32(ops.lambda_init(w.layer)))


@pytest.mark.parametrize("name", ["needle_4k", "wide_4k"])
@pytest.mark.parametrize("headnorm", [1, 0])
def test_bwd_full_size_invariants(name, headnorm):
    """The backward at the bench's full sizes, through properties that hold at any size.

    Each row of dS sums to zero (sum_j P (dW - D) = D - D), so for every head and map the
    sum of dK over all keys vanishes; without the norm (do = dy) the rows of P sum to one,
    so the sum of dV over all keys is (1 - lambda) sum_q dy_q.  Each sum's terms carry the
    bf16 rounding of P, dS and do (2^-8 of a term at most), so the residual is bounded by
    2^-8 of the sum of the terms' magnitudes even if every error had the same sign."""
    w, li = _full_size(name)
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device="cuda")
    nw = (torch.tensor(np.asarray(w.w, dtype=np.float32), device="cuda")
          if headnorm and w.w is not None else None)
    kw = dict(causal=True, headnorm=headnorm, norm_w=nw, eps=float(np.float32(w.eps)),
              lambda_init=li)
    dev = [t.cuda() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    dy = _dy(w, 77).cuda()
    _, saved = ops.fwd_train(*dev, lam, **kw)
    g = ops.bwd(*dev, lam, saved, dy, **kw)
    torch.cuda.synchronize()
    bound = 2.0 ** -8
    for k in ("dk1", "dk2"):
        t = g[k].double()
        resid = t.sum(dim=2).abs() / t.abs().sum(dim=2).clamp_min(1e-30)
        assert float(resid.max()) <= bound, f"{name} {k}: sum over keys {float(resid.max()):.3g}"
    if not headnorm:
        t = g["dv"].double()
        ref = (1.0 - lam.double())[None, :, None] * dy.double().sum(dim=2)
        resid = (t.sum(dim=2) - ref).abs() / t.abs().sum(dim=2).clamp_min(1e-30)
        assert float(resid.max()) <= bound, f"{name} dv: sum over keys {float(resid.max()):.3g}"
