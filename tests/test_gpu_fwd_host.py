"""diffattn_fwd_host (inputs and output in host memory, copies on the call's
stream) gives the bytes diffattn_fwd gives on the same inputs, and matches the
float64 oracle through it."""
import numpy as np
import pytest
import torch

from differential_attention_attn_gb300 import ops
from differential_attention_attn_gb300 import workloads as W
from tests import harness

pytestmark = pytest.mark.gpu


def _both(w, *, pinned, dtype=torch.bfloat16, headnorm=None):
    li = harness.lambda_init_for(w, "gpu")
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device="cuda")
    nw = None if w.w is None else torch.tensor(w.w, dtype=torch.float32, device="cuda")
    host = [t.to(dtype).contiguous() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    if pinned:
        host = [t.pin_memory() for t in host]
    hn = w.headnorm if headnorm is None else headnorm
    kw = dict(causal=w.causal, headnorm=hn, norm_w=nw, eps=float(np.float32(w.eps)),
              lambda_init=li)
    ref = ops.fwd(*[t.cuda() for t in host], lam, **kw)
    out = ops.fwd_host(*host, lam, **kw)
    torch.cuda.synchronize()
    return ref.cpu(), out


@pytest.mark.parametrize("N,causal,headnorm,pinned", [
    (512, True, 1, True), (300, True, 2, False), (129, False, 0, True), (1, True, 1, False)])
def test_fwd_host_is_fwd_bitwise(N, causal, headnorm, pinned):
    w = W.custom(1200 + N, B=2, H=3, N=N, d=64, causal=causal, headnorm=headnorm,
                 random_w=True, layer=3)
    ref, out = _both(w, pinned=pinned)
    assert torch.equal(ref.view(torch.int16), out.view(torch.int16))


def test_fwd_host_d128_and_f32():
    w = W.custom(1301, B=1, H=2, N=256, d=128, causal=True, headnorm=True, random_w=True,
                 layer=2)
    ref, out = _both(w, pinned=True)
    assert torch.equal(ref.view(torch.int16), out.view(torch.int16))
    w = W.pages_example()
    ref, out = _both(w, pinned=False, dtype=torch.float32)
    assert torch.equal(ref, out)


def test_fwd_host_repeated_calls_two_streams():
    """Alternating two streams and two staging buffers (as bench.py's end-to-end leg
    does): every call's output equals diffattn_fwd's."""
    w = W.custom(1401, B=2, H=4, N=384, d=64, causal=True, headnorm=True, random_w=True,
                 layer=7)
    li = harness.lambda_init_for(w, "gpu")
    lam = torch.tensor(w.lambdas(li), dtype=torch.float32, device="cuda")
    kw = dict(causal=True, headnorm=1, eps=float(np.float32(w.eps)), lambda_init=li,
              norm_w=torch.tensor(w.w, dtype=torch.float32, device="cuda"))
    host = [t.contiguous().pin_memory() for t in (w.q1, w.k1, w.q2, w.k2, w.v)]
    ref = ops.fwd(*[t.cuda() for t in host], lam, **kw).cpu()
    need = ops.fwd_host_staging_bytes(w.B, w.H, w.N, w.d)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    staging = [torch.empty(need, dtype=torch.uint8, device="cuda") for _ in range(2)]
    outs = [torch.empty_like(ref).pin_memory() for _ in range(6)]
    for i, o in enumerate(outs):
        ops.fwd_host(*host, lam, out=o, staging=staging[i % 2], stream=streams[i % 2], **kw)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(ref.view(torch.int16), o.view(torch.int16))
