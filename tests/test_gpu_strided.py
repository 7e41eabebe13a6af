"""diffattn_fwd_strided: the forward on views of other layouts ([B, N, H, d] storage
and mixtures), against the contiguous entry point (bitwise: same kernel, same math) and
the float64 oracle."""
import numpy as np
import pytest
import torch

from differential_attention_attn_gb300 import ops
from differential_attention_attn_gb300 import workloads as W
from tests import harness

pytestmark = pytest.mark.gpu


def _bnhd_view(t):
    """Copy a [B, H, N, c] tensor into [B, N, H, c] storage and return the [B, H, N, c] view."""
    return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)


def _args(w):
    li = harness.lambda_init_for(w, "gpu")
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device="cuda")
    nw = None if w.w is None else torch.tensor(w.w, dtype=torch.float32, device="cuda")
    kw = dict(causal=w.causal, headnorm=w.headnorm, norm_w=nw, eps=float(np.float32(w.eps)),
              lambda_init=li)
    return [t.cuda() for t in (w.q1, w.k1, w.q2, w.k2, w.v)], lam, kw


@pytest.mark.parametrize("N", [128, 200, 640])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("headnorm", [1, 2])
def test_bnhd_layout_matches_contiguous(N, causal, headnorm):
    w = W.custom(800 + N, B=2, H=3, N=N, d=64, causal=causal, headnorm=headnorm,
                 random_w=True, layer=5)
    dev, lam, kw = _args(w)
    ref = ops.fwd(*dev, lam, **kw)
    views = [_bnhd_view(t) for t in dev]
    assert not views[0].is_contiguous()
    out_store = torch.full((2, N, 3, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = out_store.permute(0, 2, 1, 3)
    ops.fwd_strided(*views, lam, out=out, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    err = float(np.max(np.abs(out.double().cpu().numpy() - harness.run_oracle(w))))
    assert err <= harness.bf16_tolerance(harness.run_oracle(w))


def test_mixed_layouts_and_padded_rows():
    """q contiguous, k/v in [B, N, H, c] storage, out with padded rows (row stride 136)."""
    w = W.custom(810, B=1, H=4, N=300, d=64, causal=True, headnorm=1, random_w=True, layer=2)
    dev, lam, kw = _args(w)
    ref = ops.fwd(*dev, lam, **kw)
    q1, k1, q2, k2, v = dev
    k1, k2, v = _bnhd_view(k1), _bnhd_view(k2), _bnhd_view(v)
    out_store = torch.zeros((1, 4, 300, 136), dtype=torch.bfloat16, device="cuda")
    out = out_store[..., :128]
    ops.fwd_strided(q1, k1, q2, k2, v, lam, out=out, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert float(out_store[..., 128:].abs().max()) == 0.0  # padding untouched


def test_strided_validation():
    w = W.custom(811, B=1, H=2, N=128, d=64, causal=True)
    dev, lam, kw = _args(w)
    q_bad = torch.empty((1, 2, 128, 68), dtype=torch.bfloat16, device="cuda")[..., :64]  # 68: not x8
    assert ops.fwd_strided(q_bad, *dev[1:], lam, raw_status=True, **kw) == ops.ERR_INVALID_ARG
    with pytest.raises(ValueError):
        ops.fwd_strided(dev[0].transpose(2, 3).contiguous().transpose(2, 3), *dev[1:], lam, **kw)


@pytest.mark.parametrize("N,causal,headnorm", [(128, True, 1), (300, True, 2), (256, False, 1),
                                               (200, False, 0)])
def test_d128_bnhd_layout_matches_contiguous(N, causal, headnorm):
    """The d = 128 kernel on [B, N, H, c] storage views (value width 256), with the
    output written into a [B, N, H, 256] view."""
    w = W.custom(820 + N, B=2, H=2, N=N, d=128, causal=causal, headnorm=headnorm,
                 random_w=True, layer=9)
    dev, lam, kw = _args(w)
    ref = ops.fwd(*dev, lam, **kw)
    views = [_bnhd_view(t) for t in dev]
    out_store = torch.full((2, N, 2, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = out_store.permute(0, 2, 1, 3)
    ops.fwd_strided(*views, lam, out=out, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    oracle_out = harness.run_oracle(w)
    err = float(np.max(np.abs(out.double().cpu().numpy() - oracle_out)))
    assert err <= harness.bf16_tolerance(oracle_out)


@pytest.mark.parametrize("Nq,Nkv,splits", [(1, 5000, 4), (16, 2000, 1), (200, 1000, 3)])
def test_kv_cache_in_bnhd_layout(Nq, Nkv, splits):
    """diffattn_fwd_kv_strided on a [B, Nkv, H, c] cache (and [B, Nq, H, c] queries and
    output) equals diffattn_fwd_kv on contiguous copies bitwise, single pass and split."""
    w = W.kv_cache(820 + Nq, B=2, H=3, Nq=Nq, Nkv=Nkv, causal=True)
    dev, lam, kw = _args(w)
    ref = ops.fwd_kv(*dev, lam, splits=splits, **kw)
    views = [_bnhd_view(t) for t in dev]
    out_store = torch.full((2, Nq, 3, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = out_store.permute(0, 2, 1, 3)
    ops.fwd_kv_strided(*views, lam, splits=splits, out=out, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    ref64 = harness.run_oracle_kv(w)
    assert float(np.max(np.abs(out.double().cpu().numpy() - ref64))) <= harness.bf16_tolerance(ref64)


def test_kv_strided_rejects_bad_strides():
    w = W.kv_cache(830, B=1, H=2, Nq=4, Nkv=300, causal=True)
    dev, lam, kw = _args(w)
    store = torch.zeros((1, 2, 300, 70), dtype=torch.bfloat16, device="cuda")
    k1 = store[..., :64]  # row stride 70: not a multiple of 8 elements
    st = ops.fwd_kv_strided(dev[0], k1, dev[2], dev[3], dev[4], lam, splits=1,
                            raw_status=True, **kw)
    assert st == ops.ERR_INVALID_ARG
