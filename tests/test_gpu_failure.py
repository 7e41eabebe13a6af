"""Failure detection without a GPU fault: a pipeline wait that nothing satisfies runs out
after its limit, raises the shared abort flag, the other waiting role leaves early, the
status reads DIFFATTN_ERR_TIMEOUT, and the context stays usable."""
import pytest
import torch

from differential_attention_attn_gb300 import ops
from differential_attention_attn_gb300 import workloads as W
from tests import harness

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_propagates():
    code, w0_us, w1_us = ops.selftest_wait(timeout_ns=50_000_000)  # 50 ms
    assert code == ops.ERR_TIMEOUT
    assert 45_000 <= w0_us < 1_000_000, w0_us         # ran to its own limit, not far beyond
    assert w1_us < 1_000_000, w1_us                   # left on the abort flag, not its 2 s limit
    # the context is still usable: a normal forward runs and matches the oracle
    w = W.custom(5, B=1, H=1, N=128, d=64, causal=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = harness.run_gpu(w, status=status)
    assert int(status.item()) == 0
    assert torch.isfinite(out.float()).all()


def test_selftest_rejects_bad_limits():
    st = torch.zeros(3, dtype=torch.int32, device="cuda")
    lib = ops.load()
    assert lib.diffattn_selftest_wait(ops._ptr(st), 0, None) == ops.ERR_INVALID_ARG
    assert lib.diffattn_selftest_wait(ops._ptr(st), 3_000_000_000, None) == ops.ERR_INVALID_ARG
