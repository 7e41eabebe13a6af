"""The d = 128 forward (value width 256; two-pass kernel) against the float64 oracle.

Tolerance as for the d = 64 bf16 kernel: max-abs <= 2e-2 * max|oracle|.
"""
import numpy as np
import pytest
import torch

from differential_attention_attn_gb300 import workloads as W
from tests import harness

pytestmark = pytest.mark.gpu


def _cmp(gpu, ref, what):
    gpu = gpu.double().cpu().numpy() if isinstance(gpu, torch.Tensor) else gpu
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    err = float(np.max(np.abs(gpu - ref)))
    tol = harness.bf16_tolerance(ref)
    assert err <= tol, f"{what}: max-abs err {err:.4g} > tol {tol:.4g}"


@pytest.mark.parametrize("N", [1, 63, 64, 65, 128, 129, 200, 384])
@pytest.mark.parametrize("causal", [True, False])
def test_d128_tile_edges(N, causal):
    w = W.custom(900 + N, B=2, H=2, N=N, d=128, causal=causal, headnorm=True, random_w=True,
                 layer=6)
    _cmp(harness.run_gpu(w), harness.run_oracle(w), f"d128 N={N} causal={causal}")


@pytest.mark.parametrize("lam,headnorm", [(0.0, 1), (0.8, 1), (1.0, 0), (-0.5, 0), (0.5, 2)])
def test_d128_lambda_and_norm(lam, headnorm):
    w = W.custom(31, B=1, H=3, N=300, d=128, causal=True, headnorm=headnorm, random_w=True,
                 layer=3)
    w.lam_offset = np.full(w.H, lam)
    _cmp(harness.run_gpu(w), harness.run_oracle(w), f"lambda={lam} headnorm={headnorm}")


def test_d128_many_items():
    w = W.custom(32, B=2, H=8, N=512, d=128, causal=True, headnorm=True, random_w=True, layer=4)
    _cmp(harness.run_gpu(w), harness.run_oracle(w), "B2H8N512")


def test_d128_long_sampled():
    w = W.custom(33, B=1, H=4, N=4096, d=128, causal=True, headnorm=True, qk_scale=0.5,
                 random_w=True, layer=12)
    gpu = harness.run_gpu(w)
    bh, ri = harness.sample_rows(w, 48, full_heads=(1,))
    got = gpu.view(-1, w.N, 2 * w.d)[torch.from_numpy(bh).cuda(), torch.from_numpy(ri).cuda()]
    _cmp(got, harness.run_oracle_rows(w, bh, ri), "d128 N=4096 sampled")


@pytest.mark.parametrize("Nq,Nkv,causal", [(1, 4000, True), (16, 1000, True), (200, 700, True),
                                           (130, 130, True), (40, 300, False)])
@pytest.mark.parametrize("headnorm", [1, 2])
def test_d128_kv_cache(Nq, Nkv, causal, headnorm):
    """diffattn_fwd_kv with d = 128: queries at the last Nq of Nkv positions (single
    pass), against the oracle's key/value-cache form."""
    w = W.kv_cache(950 + Nq, B=2, H=2, Nq=Nq, Nkv=Nkv, d=128, causal=causal, headnorm=headnorm)
    _cmp(harness.run_gpu_kv(w, splits=0), harness.run_oracle_kv(w), f"d128 kv {Nq}/{Nkv}")


def test_d128_kv_square_is_the_plain_forward():
    w = W.kv_cache(960, B=1, H=3, Nq=300, Nkv=300, d=128, causal=True)
    a = harness.run_gpu_kv(w, splits=1)
    b = harness.run_gpu(w)
    assert torch.equal(a, b)


def test_d128_kv_refuses_splits():
    from differential_attention_attn_gb300 import ops
    w = W.kv_cache(961, B=1, H=2, Nq=4, Nkv=1000, d=128, causal=True)
    st = harness.run_gpu_kv(w, splits=2, raw_status=True)
    assert st == ops.ERR_UNSUPPORTED
    assert ops.fwd_kv_plan(1, 2, 4, 1000, causal=True, splits=0, d=128)[0] == 1
