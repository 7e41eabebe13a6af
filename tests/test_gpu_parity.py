"""CUDA path (through the C ABI) against the float64 oracle, element by element.

Tolerances: fp32 outputs max-abs <= 1e-5; bf16 outputs (fp32 accumulation)
max-abs <= 2e-2 * max|oracle|.  Inputs are the seeded workloads of
differential_attention_attn_gb300.workloads; the oracle receives exactly the
rounded values the kernel reads.
"""
import numpy as np
import pytest
import torch

import oracle
from differential_attention_attn_gb300 import ops
from differential_attention_attn_gb300 import workloads as W
from tests import harness

pytestmark = pytest.mark.gpu


def _cmp_bf16(gpu, ref, what=""):
    err = float(np.max(np.abs(gpu - ref)))
    tol = harness.bf16_tolerance(ref)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    assert err <= tol, f"{what}: max-abs err {err:.4g} > tol {tol:.4g}"
    return err, tol


# ----------------------------------------------------------------------------- fp32 path
def test_pages_example_f32():
    w = W.pages_example()
    out = harness.run_gpu(w).double().cpu().numpy()
    ref = harness.run_oracle(w)
    assert np.max(np.abs(out - ref)) <= 1e-5


@pytest.mark.parametrize("N,d,causal,headnorm", [
    (1, 8, True, True), (6, 8, False, False), (33, 16, True, False), (100, 64, False, True),
    (257, 128, True, True), (300, 32, False, False), (4096, 8, True, True)])
def test_f32_shapes(N, d, causal, headnorm):
    w = W.custom(31 + N, B=2, H=3, N=N, d=d, causal=causal, headnorm=headnorm,
                 dtype=torch.float32, random_w=True, layer=3)
    gpu = harness.run_gpu(w).double().cpu().numpy()
    if N > 1000:
        bh, ri = harness.sample_rows(w, 24)
        ref = harness.run_oracle_rows(w, bh, ri)
        gpu = gpu.reshape(-1, N, 2 * d)[bh, ri]
    else:
        ref = harness.run_oracle(w)
    assert np.max(np.abs(gpu - ref)) <= 1e-5


# ----------------------------------------------------------------------------- head norm
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dv", [16, 128, 256])
def test_headnorm_kernel(out_dtype, dv):
    rng = np.random.default_rng(dv)
    B, H, N = 2, 3, 77
    x = rng.standard_normal((B, H, N, dv)).astype(np.float32)
    wgt = (1 + 0.1 * rng.standard_normal((H, dv))).astype(np.float32)
    eps, li = np.float32(1e-5), np.float32(0.35)
    y = ops.headnorm(torch.from_numpy(x).cuda(), H=H, norm_w=torch.from_numpy(wgt).cuda(),
                     eps=float(eps), lambda_init=float(li), out_dtype=out_dtype)
    torch.cuda.synchronize()
    hidx = np.tile(np.repeat(np.arange(H), N), B)
    ref = oracle.headnorm(x.reshape(-1, dv).astype(np.float64), hidx, wgt.astype(np.float64),
                          H=H, eps=float(eps), lambda_init_value=float(li))
    got = y.double().cpu().numpy().reshape(-1, dv)
    if out_dtype == torch.float32:
        assert np.max(np.abs(got - ref)) <= 1e-5 * max(1.0, np.max(np.abs(ref)))
    else:  # one bf16 rounding of a value computed in fp32
        assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6)


# ----------------------------------------------------------------------------- bf16 fused kernel
@pytest.mark.parametrize("N", [1, 7, 128, 129, 200, 256, 384, 640])
@pytest.mark.parametrize("causal", [True, False])
def test_bf16_tile_edges(N, causal):
    w = W.custom(100 + N, B=2, H=3, N=N, d=64, causal=causal, headnorm=True, random_w=True,
                 layer=6)
    gpu = harness.run_gpu(w).double().cpu().numpy()
    ref = harness.run_oracle(w)
    _cmp_bf16(gpu, ref, f"N={N} causal={causal}")


@pytest.mark.parametrize("lam", [0.0, 0.8, 1.0])
@pytest.mark.parametrize("headnorm", [True, False])
def test_bf16_lambda_and_norm(lam, headnorm):
    w = W.custom(7, B=1, H=2, N=384, d=64, causal=True, headnorm=headnorm, layer=2)
    w.lam_offset = np.full(w.H, lam)
    gpu = harness.run_gpu(w).double().cpu().numpy()
    ref = harness.run_oracle(w)
    _cmp_bf16(gpu, ref, f"lambda={lam} headnorm={headnorm}")


def test_bf16_identical_maps_lambda_one_is_zero():
    """q2 = q1, k2 = k1, lambda = 1 cancels exactly: raw output is (close to) zero."""
    w = W.custom(8, B=1, H=2, N=256, d=64, causal=True, headnorm=False, layer=2)
    w.q2, w.k2 = w.q1.clone(), w.k1.clone()
    w.lam_offset = np.ones(w.H)
    gpu = harness.run_gpu(w).double().cpu().numpy()
    assert np.max(np.abs(gpu)) < 1e-6


def test_bf16_small_causal_full():
    w = W.make("small_causal")
    gpu = harness.run_gpu(w).double().cpu().numpy()
    _cmp_bf16(gpu, harness.run_oracle(w), "small_causal")


@pytest.mark.parametrize("name,per_head,full_heads", [
    ("mid_causal", 48, (0, 63)), ("needle_4k", 48, (0, 31)), ("long_16k", 16, (31,)),
    ("rising_4k", 48, (0, 31))])
def test_bf16_workload_sampled(name, per_head, full_heads):
    w = W.make(name)
    gpu = harness.run_gpu(w)
    bh, ri = harness.sample_rows(w, per_head, full_heads=full_heads)
    got = gpu.view(-1, w.N, 2 * w.d)[torch.from_numpy(bh).cuda(), torch.from_numpy(ri).cuda()]
    got = got.double().cpu().numpy()
    ref = harness.run_oracle_rows(w, bh, ri)
    _cmp_bf16(got, ref, name)


@pytest.mark.parametrize("slope,causal,headnorm", [
    (3.5, True, True), (1.0, True, False), (8.0, True, True), (3.5, False, True)])
def test_rising_logits_full(slope, causal, headnorm):
    """Logits that climb by a few base-2 units per key tile (both maps), every row
    compared: the running maximum moves on most tiles, exercising the exact path
    and the rescale of O."""
    w = W.rising(17, B=1, H=2, N=1000, d=64, slope=slope)
    w.causal, w.headnorm = causal, headnorm
    gpu = harness.run_gpu(w).double().cpu().numpy()
    _cmp_bf16(gpu, harness.run_oracle(w), f"rising slope {slope}")


def test_needle_rows_follow_the_needle():
    """In the needle workload, map1 of each question row is dominated by its needle key,
    so the raw output is close to (1-ish) * V[needle] - lambda * map2 V: check the GPU's
    needle rows against the oracle more tightly than the global bound."""
    w = W.needle(9, B=1, H=4, N=1024, d=64)
    gpu = harness.run_gpu(w).double().cpu().numpy()
    ref = harness.run_oracle(w)
    q = w.meta["needle_query"]
    _cmp_bf16(gpu[:, :, q], ref[:, :, q], "needle rows")
    _cmp_bf16(gpu, ref, "needle all rows")


def test_bf16_deterministic_and_status_clear():
    w = W.make("small_causal")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = harness.run_gpu(w, status=status)
    b = harness.run_gpu(w, status=status)
    assert torch.equal(a, b)
    assert int(status.item()) == 0


def test_bf16_writes_into_given_out_and_stream():
    w = W.custom(12, B=1, H=2, N=256, d=64, causal=True, layer=1)
    out = torch.full((1, 2, 256, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        harness.run_gpu(w, out=out)
    s.synchronize()
    assert torch.isfinite(out.float()).all()
    _cmp_bf16(out.double().cpu().numpy(), harness.run_oracle(w), "given out")


def test_bf16_rejects_misaligned():
    w = W.custom(13, B=1, H=1, N=128, d=64, causal=True)
    base = torch.empty(128 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    q1 = base[1:1 + 128 * 64].view(1, 1, 128, 64)  # 2-byte offset
    k = w.k1.cuda()
    st = ops.fwd(q1, k, k, k, w.v.cuda(), torch.ones(1, device="cuda"), causal=True,
                 raw_status=True)
    assert st == ops.ERR_INVALID_ARG


@pytest.mark.parametrize("causal", [True, False])
def test_bf16_many_items_per_cta(causal):
    """More (head, query-tile) work items than SMs (several waves of CTAs, causal and
    not, both query-tile extents); every output row is compared."""
    w = W.custom(77, B=8, H=12, N=384 if causal else 320, d=64, causal=causal, headnorm=True,
                 random_w=True, layer=9)
    gpu = harness.run_gpu(w).double().cpu().numpy()
    _cmp_bf16(gpu, harness.run_oracle(w), f"many items causal={causal}")


# ----------------------------------------------------------------------------- group-norm form
@pytest.mark.parametrize("N", [7, 128, 200, 640])
@pytest.mark.parametrize("causal", [True, False])
def test_bf16_group_norm(N, causal):
    """headnorm = 2 (mean-subtracting, the page's GroupNorm wording) in the fused epilogue."""
    w = W.custom(700 + N, B=2, H=3, N=N, d=64, causal=causal, headnorm=2, random_w=True,
                 layer=6)
    gpu = harness.run_gpu(w).double().cpu().numpy()
    _cmp_bf16(gpu, harness.run_oracle(w), f"group N={N} causal={causal}")


@pytest.mark.parametrize("N,d", [(6, 8), (100, 64), (257, 128)])
def test_f32_group_norm(N, d):
    w = W.custom(710 + N, B=2, H=2, N=N, d=d, causal=True, headnorm=2, dtype=torch.float32,
                 random_w=True, layer=3)
    gpu = harness.run_gpu(w).double().cpu().numpy()
    assert np.max(np.abs(gpu - harness.run_oracle(w))) <= 1e-5


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_group_norm_kernel(out_dtype):
    rng = np.random.default_rng(5)
    B, H, N, dv = 2, 3, 77, 128
    x = (rng.standard_normal((B, H, N, dv)) + 2.0).astype(np.float32)  # non-zero mean
    wgt = (1 + 0.1 * rng.standard_normal((H, dv))).astype(np.float32)
    eps, li = np.float32(1e-5), np.float32(0.35)
    y = ops.headnorm(torch.from_numpy(x).cuda(), H=H, norm_w=torch.from_numpy(wgt).cuda(),
                     eps=float(eps), lambda_init=float(li), out_dtype=out_dtype, mode=2)
    torch.cuda.synchronize()
    hidx = np.tile(np.repeat(np.arange(H), N), B)
    ref = oracle.groupnorm(x.reshape(-1, dv).astype(np.float64), hidx, wgt.astype(np.float64),
                           H=H, eps=float(eps), lambda_init_value=float(li))
    got = y.double().cpu().numpy().reshape(-1, dv)
    if out_dtype == torch.float32:
        assert np.max(np.abs(got - ref)) <= 1e-5 * max(1.0, np.max(np.abs(ref)))
    else:
        assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-5)
