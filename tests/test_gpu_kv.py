"""diffattn_fwd_kv on the GPU against the float64 oracle: split-KV, decoding
against a key/value cache and chunked prefill (fewer queries than keys,
bottom-right causal alignment).

Tolerance as for the single-pass bf16 kernel: max-abs <= 2e-2 * max|oracle|.
"""
import numpy as np
import pytest
import torch

from differential_attention_attn_gb300 import ops
from differential_attention_attn_gb300 import workloads as W
from tests import harness

pytestmark = pytest.mark.gpu


def _cmp(gpu, ref, what):
    gpu = gpu.double().cpu().numpy() if isinstance(gpu, torch.Tensor) else gpu
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    err = float(np.max(np.abs(gpu - ref)))
    tol = harness.bf16_tolerance(ref)
    assert err <= tol, f"{what}: max-abs err {err:.4g} > tol {tol:.4g}"


def _square(seed, B, H, N, causal):
    w = W.custom(seed, B=B, H=H, N=N, d=64, causal=causal, headnorm=True, random_w=True, layer=5)
    return w


@pytest.mark.parametrize("N", [128, 300, 512, 1000])
@pytest.mark.parametrize("splits", [2, 3, 0, 64])
@pytest.mark.parametrize("causal", [True, False])
def test_split_square_matches_oracle(N, splits, causal):
    w = _square(200 + N, 1, 3, N, causal)
    _cmp(harness.run_gpu_kv(w, splits=splits), harness.run_oracle(w),
         f"N={N} splits={splits} causal={causal}")


def test_single_split_is_the_single_pass_kernel():
    """splits = 1 runs the same kernel with the same configuration as diffattn_fwd:
    the outputs are bitwise equal."""
    w = _square(301, 2, 3, 700, True)
    a = harness.run_gpu(w)
    b = harness.run_gpu_kv(w, splits=1)
    assert torch.equal(a, b)


@pytest.mark.parametrize("Nq", [1, 7, 16, 128, 200])
@pytest.mark.parametrize("Nkv", [1000, 4097])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("splits", [1, 0, 5])
def test_kv_cache_matches_oracle(Nq, Nkv, causal, splits):
    w = W.kv_cache(400 + Nq + Nkv, B=2, H=3, Nq=Nq, Nkv=Nkv, causal=causal)
    _cmp(harness.run_gpu_kv(w, splits=splits), harness.run_oracle_kv(w),
         f"Nq={Nq} Nkv={Nkv} causal={causal} splits={splits}")


@pytest.mark.parametrize("Nkv", [1, 2, 127, 129])
def test_kv_tiny_cache(Nkv):
    """One query against a cache of one key (the output is (1 - lambda) v_0 before the
    norm) and around one key tile."""
    w = W.kv_cache(450 + Nkv, B=1, H=2, Nq=1, Nkv=Nkv, causal=True)
    _cmp(harness.run_gpu_kv(w, splits=0), harness.run_oracle_kv(w), f"Nkv={Nkv}")


def test_kv_rows_fully_masked_in_a_split():
    """Chunked prefill with a query offset that is not a multiple of the key tile:
    the top rows of a query tile see no key of the tile that holds its last row, so
    a split that starts there has rows whose first tile is fully masked."""
    w = W.kv_cache(470, B=1, H=2, Nq=256, Nkv=256 + 64, causal=True)
    for splits in (1, 2, 3):
        _cmp(harness.run_gpu_kv(w, splits=splits), harness.run_oracle_kv(w),
             f"offset 64 splits={splits}")


def test_decode_long_cache_sampled_heads():
    """Decoding step of 32 heads against a 16K-key cache (the long-sequence shape)."""
    w = W.kv_cache(480, B=1, H=32, Nq=1, Nkv=16384, causal=True, layer=24)
    sp, _ = ops.fwd_kv_plan(1, 32, 1, 16384, causal=True, splits=0)
    assert sp > 1
    _cmp(harness.run_gpu_kv(w, splits=0), harness.run_oracle_kv(w), "decode 16K")


def test_auto_split_prefill_sampled():
    """A prefill with fewer work items than SMs (4 heads x 32 query tiles): the planner
    splits the keys; sampled rows (all rows of one head) against the oracle."""
    w = W.custom(470, B=1, H=4, N=4096, d=64, causal=True, headnorm=True, random_w=True,
                 layer=7)
    sp, nbytes = ops.fwd_kv_plan(1, 4, 4096, 4096, causal=True, splits=0)
    assert sp > 1 and nbytes > 0
    gpu = harness.run_gpu_kv(w, splits=0)
    bh, ri = harness.sample_rows(w, 64, full_heads=(2,))
    got = gpu.view(-1, w.N, 2 * w.d)[torch.from_numpy(bh).cuda(), torch.from_numpy(ri).cuda()]
    _cmp(got, harness.run_oracle_rows(w, bh, ri), "4K prefill split")


def test_small_causal_through_fwd_kv():
    w = W.make("small_causal")
    for splits in (0, 4):
        _cmp(harness.run_gpu_kv(w, splits=splits), harness.run_oracle(w),
             f"small_causal splits={splits}")


def test_large_problems_do_not_split():
    """With more work items than SMs the planner keeps the single-pass kernel."""
    assert ops.fwd_kv_plan(2, 16, 4096, 4096, causal=True, splits=0) == (1, 0)


def test_workspace_reuse_and_stale_contents():
    """The workspace's previous contents do not matter, and one buffer serves
    consecutive calls on one stream."""
    w = W.kv_cache(490, B=1, H=4, Nq=16, Nkv=3000, causal=True)
    sp, nbytes = ops.fwd_kv_plan(1, 4, 16, 3000, causal=True, splits=6)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN bit patterns
    a = harness.run_gpu_kv(w, splits=6, workspace=ws)
    b = harness.run_gpu_kv(w, splits=6, workspace=ws)
    assert torch.equal(a, b)
    _cmp(a, harness.run_oracle_kv(w), "stale workspace")


def test_split_status_stays_clear():
    w = W.kv_cache(491, B=1, H=2, Nq=64, Nkv=2048, causal=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    harness.run_gpu_kv(w, splits=4, status=status)
    assert int(status.item()) == 0


def test_kv_rejects_short_workspace_on_device():
    w = W.kv_cache(492, B=1, H=2, Nq=64, Nkv=2048, causal=True)
    sp, nbytes = ops.fwd_kv_plan(1, 2, 64, 2048, causal=True, splits=4)
    ws = torch.empty(nbytes - 16, dtype=torch.uint8, device="cuda")
    assert harness.run_gpu_kv(w, splits=4, workspace=ws, raw_status=True) == ops.ERR_INVALID_ARG


@pytest.mark.parametrize("splits", [1, 3])
def test_kv_group_norm(splits):
    """headnorm = 2 through the split-KV combine kernel and the single-pass kernel."""
    w = W.kv_cache(495, B=1, H=3, Nq=40, Nkv=1500, causal=True)
    w.headnorm = 2
    _cmp(harness.run_gpu_kv(w, splits=splits), harness.run_oracle_kv(w), f"group splits={splits}")


def test_combine_reports_a_failed_partial_as_nan():
    """If the status word already holds an error when the partial kernel finishes (as it
    would after a CTA gave up on a wait), the combine writes NaN rather than merging
    scratch into a plausible output.  The error is planted on the host: no wait runs out
    and nothing faults."""
    w = W.kv_cache(940, B=1, H=4, Nq=16, Nkv=4096, causal=True)
    status = torch.full((1,), ops.ERR_TIMEOUT, dtype=torch.int32, device="cuda")
    out = harness.run_gpu_kv(w, splits=4, status=status)
    assert torch.isnan(out.float()).all()
    status.zero_()
    out = harness.run_gpu_kv(w, splits=4, status=status)
    assert int(status.item()) == 0 and torch.isfinite(out.float()).all()
