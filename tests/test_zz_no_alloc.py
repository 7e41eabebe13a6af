"""diffattn_fwd_kv_noalloc: the same results as diffattn_fwd_kv, with the split-KV
partial blocks on the library's own scratch area instead of a caller workspace.

Collected last on purpose (file name), and independent of the other tests: it
must pass alone and after them.
"""
import ctypes

import numpy as np
import pytest
import torch

from differential_attention_attn_gb300 import build as libbuild
from differential_attention_attn_gb300 import ops
from differential_attention_attn_gb300 import workloads as W
from tests import harness


def _args(w, device="cuda"):
    li = harness.lambda_init_for(w, "gpu")
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device=device)
    nw = None if w.w is None else torch.tensor(w.w, dtype=torch.float32, device=device)
    dev = [t.to(device) for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    kw = dict(causal=w.causal, headnorm=w.headnorm, norm_w=nw, eps=float(np.float32(w.eps)),
              lambda_init=li)
    return dev, lam, kw


@pytest.mark.gpu
def test_noalloc_matches_fwd_kv_on_two_calls_in_a_row():
    """Two consecutive calls (different shapes and split counts, so the second reads
    scratch left by the first) equal diffattn_fwd_kv with a fresh workspace bitwise."""
    cases = [W.kv_cache(900, B=1, H=32, Nq=1, Nkv=16384, causal=True, layer=24),
             W.kv_cache(901, B=2, H=3, Nq=200, Nkv=1000, causal=True)]
    got, want = [], []
    for w in cases:  # two no-alloc calls back to back on one stream
        dev, lam, kw = _args(w)
        got.append(ops.fwd_kv_noalloc(*dev, lam, splits=0, **kw))
    torch.cuda.synchronize()
    for w in cases:
        dev, lam, kw = _args(w)
        sp, _ = ops.fwd_kv_plan(w.B, w.H, w.N, w.n_kv, causal=w.causal, splits=0)
        want.append(ops.fwd_kv(*dev, lam, splits=sp, **kw))
    torch.cuda.synchronize()
    assert ops.fwd_kv_plan(1, 32, 1, 16384, causal=True, splits=0)[0] > 1
    for g, r in zip(got, want):
        assert torch.equal(g, r)


@pytest.mark.gpu
def test_noalloc_repeated_call_is_stable_and_matches_oracle():
    w = W.kv_cache(902, B=1, H=4, Nq=16, Nkv=3000, causal=True)
    dev, lam, kw = _args(w)
    a = ops.fwd_kv_noalloc(*dev, lam, splits=6, **kw).clone()
    b = ops.fwd_kv_noalloc(*dev, lam, splits=6, **kw)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    ref = harness.run_oracle_kv(w)
    err = float(np.max(np.abs(a.double().cpu().numpy() - ref)))
    assert err <= harness.bf16_tolerance(ref)


@pytest.mark.gpu
@pytest.mark.parametrize("causal,headnorm", [(True, 2), (False, 1), (False, 2)])
def test_noalloc_group_norm_and_non_causal_through_the_combine(causal, headnorm):
    """The mean-subtracting norm and the non-causal mask with splits > 1 (so the
    combine kernel runs), bitwise against diffattn_fwd_kv with a fresh workspace."""
    w = W.kv_cache(903 + headnorm, B=2, H=3, Nq=8, Nkv=2500, causal=causal, headnorm=headnorm)
    dev, lam, kw = _args(w)
    got = ops.fwd_kv_noalloc(*dev, lam, splits=5, **kw)
    torch.cuda.synchronize()
    want = ops.fwd_kv(*dev, lam, splits=5, **kw)
    torch.cuda.synchronize()
    assert torch.equal(got, want)


def test_noalloc_rejects_oversize_requests_before_launch():
    """A split count whose partial blocks exceed the 64 MiB scratch is refused on the host."""
    libbuild.build()
    lib = ops.load()
    d = ops.make_desc(8, 16, 4096, 64, ops.BF16, True, True, 1e-5, 0.2)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: refused before any launch
    st = lib.diffattn_fwd_kv_noalloc(ctypes.byref(d), 4096, fake, fake, fake, fake, fake, fake,
                                     None, fake, 2, None)
    assert st == ops.ERR_UNSUPPORTED
    assert ops.NOALLOC_SCRATCH_BYTES == 64 << 20
