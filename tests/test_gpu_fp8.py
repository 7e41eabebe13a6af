"""DIFFATTN_E4M3_QK: the d = 64 forward with fp8 (e4m3) query/key inputs, against the
float64 oracle fed the same e4m3 values (exactly representable, so the oracle sees what
the tensor cores see). Tolerance as for bf16: max-abs <= 2e-2 * max|oracle|."""
import numpy as np
import pytest
import torch

from differential_attention_attn_gb300 import ops
from differential_attention_attn_gb300 import workloads as W
from tests import harness

pytestmark = pytest.mark.gpu


def _e4m3(w):
    for name in ("q1", "k1", "q2", "k2"):
        setattr(w, name, getattr(w, name).float().to(torch.float8_e4m3fn))
    return w


def _run(w):
    li = harness.lambda_init_for(w, "gpu")
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device="cuda")
    nw = None if w.w is None else torch.tensor(w.w, dtype=torch.float32, device="cuda")
    dev = [t.cuda() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    out = ops.fwd_fp8(*dev, lam, causal=w.causal, headnorm=w.headnorm, norm_w=nw,
                      eps=float(np.float32(w.eps)), lambda_init=li)
    torch.cuda.synchronize()
    return out


def _cmp(gpu, ref, what):
    gpu = gpu.double().cpu().numpy()
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite"
    err = float(np.max(np.abs(gpu - ref)))
    tol = harness.bf16_tolerance(ref)
    assert err <= tol, f"{what}: max-abs err {err:.4g} > tol {tol:.4g}"


@pytest.mark.parametrize("N", [1, 128, 200, 384])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("headnorm", [1, 0])
def test_e4m3_matches_oracle(N, causal, headnorm):
    w = _e4m3(W.custom(950 + N, B=2, H=3, N=N, d=64, causal=causal, headnorm=headnorm,
                       random_w=True, layer=5))
    _cmp(_run(w), harness.run_oracle(w), f"e4m3 N={N} causal={causal} headnorm={headnorm}")


def test_e4m3_needle_rows():
    w = _e4m3(W.needle(9, B=1, H=4, N=1024, d=64))
    gpu = _run(w)
    ref = harness.run_oracle(w)
    q = w.meta["needle_query"]
    _cmp(gpu[:, :, q], ref[:, :, q], "e4m3 needle rows")
    _cmp(gpu, ref, "e4m3 needle all rows")


def test_e4m3_unsupported_modes():
    w = _e4m3(W.custom(960, B=1, H=2, N=128, d=64, causal=True, headnorm=2))
    li = 0.2
    lam = torch.ones(2, device="cuda")
    dev = [t.cuda() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    assert ops.fwd_fp8(*dev, lam, causal=True, headnorm=2, lambda_init=li,
                       raw_status=True) == ops.ERR_UNSUPPORTED


# diffattn_fwd_kv with e4m3 queries/keys: single pass and split-KV (partial
# kernel + combine), against the float64 oracle on the same e4m3 values.
@pytest.mark.parametrize("nq,nkv,splits,causal", [
    (1, 3000, 0, True), (1, 3000, 4, True), (16, 2000, 3, True), (16, 2000, 1, True),
    (200, 1000, 2, True), (200, 1000, 1, False), (7, 640, 5, False)])
@pytest.mark.parametrize("headnorm", [1, 0])
def test_e4m3_kv_matches_oracle(nq, nkv, splits, causal, headnorm):
    w = _e4m3(W.kv_cache(970 + nq + nkv, B=1, H=4, Nq=nq, Nkv=nkv, causal=causal, layer=7))
    w.headnorm = headnorm
    gpu = harness.run_gpu_kv(w, splits=splits)
    assert gpu.dtype == torch.bfloat16
    _cmp(gpu, harness.run_oracle_kv(w),
         f"e4m3 kv nq={nq} nkv={nkv} splits={splits} causal={causal} headnorm={headnorm}")


def test_e4m3_kv_noalloc_equals_workspace_call():
    w = _e4m3(W.kv_cache(985, B=1, H=8, Nq=1, Nkv=8192, causal=True, layer=12))
    a = harness.run_gpu_kv(w, splits=4)
    li = harness.lambda_init_for(w, "gpu")
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device="cuda")
    nw = torch.tensor(w.w, dtype=torch.float32, device="cuda")
    dev = [t.cuda() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    b = ops.fwd_kv_noalloc(*dev, lam, causal=True, headnorm=w.headnorm, norm_w=nw,
                           lambda_init=li, eps=float(np.float32(w.eps)), splits=4)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_e4m3_kv_group_norm_unsupported():
    w = _e4m3(W.kv_cache(986, B=1, H=2, Nq=4, Nkv=512, causal=True))
    w.headnorm = 2
    assert harness.run_gpu_kv(w, splits=2, raw_status=True) == ops.ERR_UNSUPPORTED
