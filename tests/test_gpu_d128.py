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
