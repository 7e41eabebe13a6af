"""The float64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from differential_attention_attn_gb300 import workloads
from tests import pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("name", sorted(pins.PINS))
def test_pin(lib, name):
    ok, detail = pins.PINS[name](lib)
    assert ok, f"pin {name} failed: {detail}"


def test_pages_example_output_is_diff_map_times_v(lib):
    """The oracle's forward equals its own differential map times V on the page's example."""
    w = workloads.pages_example()
    f = w.f64
    wmap = oracle.diff_map(f(w.q1[0, 0]), f(w.k1[0, 0]), f(w.q2[0, 0]), f(w.k2[0, 0]), 0.8,
                           causal=False, lib=lib)
    out = oracle.fwd(f(w.q1), f(w.k1), f(w.q2), f(w.k2), f(w.v), [0.8], causal=False,
                     headnorm=False, lib=lib)
    assert np.max(np.abs(out[0, 0] - wmap @ f(w.v[0, 0]))) < 1e-14


def test_rejects_bad_rows(lib):
    z = np.zeros((1, 1, 4, 2))
    with pytest.raises(RuntimeError):
        oracle.fwd_rows(z, z, z, z, np.zeros((1, 1, 4, 4)), [0.5], [0], [4], causal=True,
                        headnorm=False, lib=lib)


def test_empty_inputs(lib):
    z = np.zeros((1, 2, 0, 8))
    out = oracle.fwd(z, z, z, z, np.zeros((1, 2, 0, 16)), [0.1, 0.2], causal=True,
                     headnorm=True, lib=lib)
    assert out.shape == (1, 2, 0, 16)
