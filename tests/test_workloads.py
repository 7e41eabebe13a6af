"""Seeded input generators: determinism, shapes and the needle structure."""
import numpy as np
import torch

from differential_attention_attn_gb300 import workloads as W


def test_pages_example_matches_page_recipe():
    torch.manual_seed(0)
    q1, k1, q2, k2 = torch.randn(4, 6, 8)
    v = torch.randn(6, 16)
    w = W.pages_example()
    for a, b in ((w.q1, q1), (w.k1, k1), (w.q2, q2), (w.k2, k2), (w.v, v)):
        assert torch.equal(a[0, 0], b)
    assert w.dtype == torch.float32 and not w.causal and not w.headnorm


def test_deterministic_and_bf16():
    a = W.make("small_causal")
    b = W.make("small_causal")
    assert torch.equal(a.q1, b.q1) and torch.equal(a.v, b.v)
    assert a.q1.dtype == torch.bfloat16 and a.v.shape == (1, 4, 512, 128)
    assert np.all((a.lam_offset >= 0.1) & (a.lam_offset <= 0.9))
    c = W.make("small_causal", seed_offset=1)
    assert not torch.equal(a.q1, c.q1)


def test_needle_structure():
    w = W.needle(7, B=2, H=3, N=256, d=64)
    pos, qry = w.meta["needle_pos"], w.meta["needle_query"]
    assert list(qry) == list(range(250, 256))
    for b in range(2):
        for h in range(3):
            assert len(set(pos[b, h])) == 6 and pos[b, h].max() < 250
            for k in range(6):
                assert torch.equal(w.k1[b, h, pos[b, h, k]].float(),
                                   4.0 * w.q1[b, h, qry[k]].float())
    assert np.all(w.lam_offset == 0.8) and w.lambda_init_override == 0.8


def test_mid_causal_weights_and_lambda_recipe():
    w = W.make("mid_causal")
    assert w.w.shape == (16, 128) and w.layer == 12 and w.lam_plus_lambda_init
    assert np.all(np.abs(w.lam_offset) <= 0.05)
    lam = w.lambdas(0.5)
    assert lam.dtype == np.float64 and np.all(np.abs(lam - 0.5) <= 0.05 + 1e-7)
