"""The bounds-checked debug build (compiled with DIFFATTN_DEBUG): every kernel checks the
tensor-memory columns, shared-memory offsets and global indices it touches and reports
a failed check through the status word (DIFFATTN_ERR_BOUNDS | site << 8), skipping the
access.  With compute-sanitizer unavailable to these tests, this is how out-of-bounds
accesses are looked for: the tile-edge shapes of every path run through the debug
library, every status must stay clear, and every output must equal the release
library's bitwise (the checks change nothing else)."""
import ctypes

import numpy as np
import pytest
import torch

from differential_attention_attn_gb300 import build as libbuild
from differential_attention_attn_gb300 import ops
from differential_attention_attn_gb300 import workloads as W
from tests import harness

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    return ops.bind(ctypes.CDLL(libbuild.build(debug=True)))


def _both(dbg, fn):
    """fn(status) through the release and the debug library; returns both results and
    the debug call's status word."""
    ops.load()
    st_rel = torch.zeros(1, dtype=torch.int32, device="cuda")
    rel = fn(st_rel)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with ops.using(dbg):
        got = fn(st)
    torch.cuda.synchronize()
    assert int(st_rel.item()) == 0
    return rel, got, int(st.item())


def _check(rel, got, status, what):
    assert status == 0, f"{what}: bounds check failed, status {status:#x} (site {status >> 8})"
    if isinstance(rel, dict):
        for k in rel:
            assert torch.equal(rel[k], got[k]), f"{what}: {k} differs from the release build"
    else:
        assert torch.equal(rel, got), f"{what}: output differs from the release build"


@pytest.mark.parametrize("N", [1, 7, 128, 129, 200, 384])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("headnorm", [1, 2])
def test_forward_tile_edges(dbg, N, causal, headnorm):
    w = W.custom(1200 + N, B=2, H=3, N=N, d=64, causal=causal, headnorm=headnorm,
                 random_w=True, layer=4)
    rel, got, st = _both(dbg, lambda s: harness.run_gpu(w, status=s))
    _check(rel, got, st, f"fwd N={N}")


@pytest.mark.parametrize("Nq,Nkv,splits", [(1, 3000, 4), (16, 700, 3), (130, 130, 2)])
def test_kv_split_and_combine(dbg, Nq, Nkv, splits):
    w = W.kv_cache(1300 + Nq, B=1, H=3, Nq=Nq, Nkv=Nkv, causal=True)
    rel, got, st = _both(dbg, lambda s: harness.run_gpu_kv(w, splits=splits, status=s))
    _check(rel, got, st, f"kv {Nq}/{Nkv} splits {splits}")


@pytest.mark.parametrize("N,d", [(7, 64), (129, 64), (256, 64), (1, 128), (200, 128),
                                 (257, 128)])
def test_training_forward_and_backward(dbg, N, d):
    w = W.custom(1400 + N, B=1, H=2, N=N, d=d, causal=True, headnorm=True, random_w=True,
                 layer=3)
    dy = torch.from_numpy(np.random.default_rng(N).standard_normal((1, 2, N, 2 * d))).to(
        torch.bfloat16).cuda()
    li = harness.lambda_init_for(w, "gpu")
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device="cuda")
    nw = torch.tensor(w.w, dtype=torch.float32, device="cuda")
    dev = [t.cuda() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    kw = dict(causal=True, headnorm=True, norm_w=nw, eps=float(np.float32(w.eps)),
              lambda_init=li)

    def run(s):
        out, saved = ops.fwd_train(*dev, lam, status=s, **kw)
        g = ops.bwd(*dev, lam, saved, dy, status=s, **kw)
        # dk, dlambda, dnorm_w and the saved activations are deterministic; dq and dv
        # are summed with atomic adds (their last bits may differ run to run).
        return {"out": out, "saved": saved, "dk1": g["dk1"], "dk2": g["dk2"]}
    rel, got, st = _both(dbg, run)
    _check(rel, got, st, f"train N={N} d={d}")


@pytest.mark.parametrize("N", [1, 65, 200])
def test_d128(dbg, N):
    w = W.custom(1500 + N, B=1, H=2, N=N, d=128, causal=True, headnorm=True, random_w=True,
                 layer=2)
    rel, got, st = _both(dbg, lambda s: harness.run_gpu(w, status=s))
    _check(rel, got, st, f"d128 N={N}")
