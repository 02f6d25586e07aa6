"""Pins of the oracle's LM head, log-softmax and top-k (CPU only).

LM head and distributions: "MFD drafter for Qwen3.5-4B" model table (the
target's LM head on the drafter's hidden states); project page "Multi-Future
Drafting", How it works, step 2 (one distribution per mode and position).
"""
import numpy as np
import pytest
import torch

import oracle
from tree_verified_speculative_gb300 import synth


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_lmhead_logits_match_float64_matmul():
    rng = np.random.default_rng(0)
    h = synth.bf16_round(rng.standard_normal((7, 96)).astype(np.float32))
    W = synth.bf16_round(rng.standard_normal((133, 96)).astype(np.float32))
    z = oracle.lmhead_logits(_bits(h), _bits(W))
    ref = h.double().numpy() @ W.double().numpy().T  # library matmul, fp64
    np.testing.assert_allclose(z, ref, rtol=0, atol=1e-12)
    # a vocab slice is the same columns
    zs = oracle.lmhead_logits(_bits(h), _bits(W), 40, 77)
    np.testing.assert_array_equal(zs, z[:, 40:77])


def test_logsoftmax_closed_forms():
    V = 50
    # equal logits: every log p is -log V exactly up to one fp32 rounding
    z = np.full((1, V), 3.25, np.float32)
    lp, tk, lse = oracle.logits_topk(z, V)
    assert np.all(lp == np.float32(-np.log(V)))
    assert list(tk[0]) == list(range(V))  # ties: token id ascending
    assert abs(lse[0] - (3.25 + np.log(V))) < 1e-12
    # one dominant logit: log p = -log(1 + (V-1) e^-D)
    D = 30.0
    z = np.zeros((1, V), np.float32)
    z[0, 17] = D
    lp, tk, lse = oracle.logits_topk(z, 3)
    assert tk[0, 0] == 17 and tk[0, 1] == 0 and tk[0, 2] == 1
    # z - LSE cancels in double: agreement to a few ulps of |z| = 30
    assert abs(float(lp[0, 0]) - (-np.log1p((V - 1) * np.exp(-D)))) < 1e-13
    assert lp[0, 1] == np.float32(-D - np.log1p((V - 1) * np.exp(-D)))


def test_logsoftmax_normalises():
    rng = np.random.default_rng(1)
    z = (3 * rng.standard_normal((5, 1000))).astype(np.float32)
    lp, tk, lse = oracle.logits_topk(z, 1000)
    for r in range(5):
        assert abs(np.exp(lp[r].astype(np.float64)).sum() - 1.0) < 1e-6
        # lse against scipy's logsumexp (an independent library routine)
        from scipy.special import logsumexp
        assert abs(lse[r] - logsumexp(z[r].astype(np.float64))) < 1e-12


@pytest.mark.parametrize("seed", range(6))
def test_topk_order_and_ties(seed):
    rng = np.random.default_rng(100 + seed)
    R, V, k = 4, 64, 9
    # values from a small set force many exact ties
    z = rng.choice(np.array([-1.5, 0.0, 0.5, 2.0], np.float32), size=(R, V)).astype(np.float32)
    lp, tk, _ = oracle.logits_topk(z, k)
    for r in range(R):
        from scipy.special import logsumexp
        full = (z[r].astype(np.float64) - logsumexp(z[r].astype(np.float64))).astype(np.float32)
        order = np.lexsort((np.arange(V), -full))  # log p desc, then token asc
        assert list(tk[r]) == list(order[:k])
        np.testing.assert_array_equal(lp[r], full[order[:k]])


def test_lmhead_topk_equals_logits_path():
    rng = np.random.default_rng(3)
    h = synth.bf16_round(rng.standard_normal((6, 64)).astype(np.float32))
    W = synth.bf16_round((rng.standard_normal((300, 64)) / 8).astype(np.float32))
    lp, tk, lse = oracle.lmhead_topk(_bits(h), _bits(W), 12, nthreads=2)
    z = h.double().numpy() @ W.double().numpy().T
    from scipy.special import logsumexp
    for r in range(6):
        full = (z[r] - logsumexp(z[r])).astype(np.float32)
        order = np.lexsort((np.arange(300), -full))
        assert list(tk[r]) == list(order[:12])
        np.testing.assert_allclose(lp[r], full[order[:12]], rtol=0, atol=2e-7)
        assert abs(lse[r] - logsumexp(z[r])) < 1e-9
