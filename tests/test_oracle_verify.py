"""Pins of the oracle's tree verification and its Philox/Gumbel draws (CPU only).

Model card "MFD drafter for Qwen3.5-4B", first paragraph, and project page
"Multi-Future Drafting", Figure 2 (c): the target verifies the tree in one
pass with the standard tree verification, so decoding is lossless.  Project
page, How it works, step 1 and the Abstract: under tree verification the
expected number of accepted tokens is the probability mass the tree covers.
Philox4x32-10: Salmon et al., "Parallel random numbers: as easy as 1, 2, 3".
"""
import numpy as np
import pytest

import oracle
from tree_verified_speculative_gb300 import synth

from bruteforce import node_sequences


def _hand_tree():
    # root 0 -> 1 (tok 5) -> 3 (tok 2);  root -> 2 (tok 7);  1 -> 4 (tok 8)
    parent = np.array([-1, 0, 0, 1, 1], np.int32)
    token = np.array([0, 5, 7, 2, 8], np.int32)
    return parent, token


def test_greedy_hand_case():
    parent, token = _hand_tree()
    V, L = 10, 3
    t = np.zeros((5, V), np.float32)
    t[0, 5] = 3.0
    t[1, 2] = 1.0
    t[3, 9] = 4.0
    acc, path, out, gap = oracle.verify(t, parent, token, 5, L)
    assert acc == 2
    assert list(path) == [0, 1, 3, -1]
    assert list(out) == [5, 2, 9, -1]
    assert gap[0] == 3.0 and gap[2] == 4.0


def test_greedy_ties_take_smallest_token():
    parent, token = _hand_tree()
    t = np.zeros((5, 10), np.float32)
    t[0, 7] = 2.0
    t[0, 5] = 2.0  # tie between 5 and 7: 5 wins
    acc, path, out, gap = oracle.verify(t, parent, token, 5, 3)
    assert out[0] == 5 and path[1] == 1 and gap[0] == 0.0
    # no matching child: accept 0, the argmax is the bonus
    t = np.zeros((5, 10), np.float32)
    t[0, 1] = 1.0
    acc, path, out, _ = oracle.verify(t, parent, token, 5, 3)
    assert acc == 0 and list(out[:1]) == [1] and out[1] == -1


def test_greedy_planted_closed_form():
    """Tiny case: +10 on mode 2's future makes the walk follow that future to
    the deepest tree node on it; the bonus is the future's next token."""
    c = synth.tiny(seed=1)
    lp, tk, _ = oracle.logits_topk(c.logits, c.topk)
    t = oracle.build_tree(lp.reshape(c.K, c.L, c.topk), tk.reshape(c.K, c.L, c.topk), c.B)
    n = int(t["n_nodes"])
    fut = c.fut[1]
    seqs = node_sequences(t["parent"], t["token"], n)
    deepest = max(len(q) for q in seqs if q == tuple(fut[:len(q)]))
    rng = np.random.default_rng(5)
    noise = synth.target_noise(c.B + 1, c.V, rng)
    rows, cols = synth.plant_sites(t["parent"], t["token"], t["depth"], n, fut)
    tl = synth.plant(noise, rows, cols)
    acc, path, out, _ = oracle.verify(tl, t["parent"], t["token"], n, c.L)
    assert acc == deepest
    assert list(out[:acc]) == list(fut[:acc])
    if acc < c.L:
        assert out[acc] == fut[acc]


def test_philox_against_independent_implementation():
    """Triton's Philox4x32 (run on the CPU by its interpreter) is an
    implementation written by another project."""
    import os
    os.environ.setdefault("TRITON_INTERPRET", "1")
    if os.environ.get("TRITON_INTERPRET") != "1":
        pytest.skip("triton interpreter not enabled")
    triton = pytest.importorskip("triton")
    import torch
    import triton.language as tl

    @triton.jit
    def _k(out_ptr, c1_ptr, seed, N: tl.constexpr):
        offs = tl.arange(0, N)
        c1 = tl.load(c1_ptr + offs)
        z = offs * 0
        a, b, c, d = tl.philox(seed, offs * 7919 + 3, c1, z, z, 10)
        tl.store(out_ptr + offs * 4 + 0, a)
        tl.store(out_ptr + offs * 4 + 1, b)
        tl.store(out_ptr + offs * 4 + 2, c)
        tl.store(out_ptr + offs * 4 + 3, d)

    N = 64
    for seed in (0, 12345, 0xDEADBEEFCAFEF00D & 0x7FFFFFFFFFFFFFFF):
        c1 = torch.arange(N, dtype=torch.int32) * 31 + 5
        out = torch.zeros(N * 4, dtype=torch.int32)
        _k[(1,)](out, c1, seed, N=N)
        got = out.numpy().view(np.uint32).reshape(N, 4)
        ctr = np.zeros((N, 4), np.uint32)
        ctr[:, 0] = np.arange(N, dtype=np.uint32) * 7919 + 3
        ctr[:, 1] = c1.numpy().astype(np.uint32)
        key = np.zeros((N, 2), np.uint32)
        key[:, 0] = seed & 0xFFFFFFFF
        key[:, 1] = seed >> 32
        np.testing.assert_array_equal(oracle.philox4x32_10(ctr, key), got)


def test_gumbel_layout_from_the_block_function():
    """G(seed, node, v) uses word v mod 4 of the Philox block at counter
    (v div 4, node, 0, 0), key (seed low, seed high): recomputed here from
    the block function (pinned to Triton's above) with numpy's logarithms."""
    V = 67
    for seed, node in ((0, 0), (987654321123, 5), (2 ** 63 + 11, 300)):
        g = oracle.gumbel(seed, node, V).astype(np.float64)
        v = np.arange(V)
        ctr = np.zeros((V, 4), np.uint32)
        ctr[:, 0] = v // 4
        ctr[:, 1] = node
        key = np.zeros((V, 2), np.uint32)
        key[:, 0] = seed & 0xFFFFFFFF
        key[:, 1] = (seed >> 32) & 0xFFFFFFFF
        x = oracle.philox4x32_10(ctr, key)[v, v % 4].astype(np.uint64)
        u = (2 * (x >> 9) + 1).astype(np.float64) * 2.0 ** -24
        np.testing.assert_allclose(g, -np.log(-np.log(u)), rtol=0, atol=2e-5)


def test_gumbel_moments():
    """G = -log(-log u) is standard Gumbel: mean = Euler-Mascheroni gamma,
    variance = pi^2 / 6."""
    g = np.concatenate([oracle.gumbel(s, 3, 50000) for s in range(8)]).astype(np.float64)
    n = g.size
    assert np.all(np.isfinite(g))
    assert abs(g.mean() - 0.5772156649) < 5 * np.sqrt(np.pi ** 2 / 6 / n)
    assert abs(g.var() - np.pi ** 2 / 6) < 0.03


def test_gumbel_max_frequencies_match_softmax():
    """Sampled verification at one node draws y ~ softmax(t / T)."""
    V, T = 6, 0.7
    t = np.array([[0.3, -1.0, 1.2, 0.0, 2.0, -0.4]], np.float32)
    parent = np.array([-1], np.int32)
    token = np.array([0], np.int32)
    n = 60000
    counts = np.zeros(V)
    for s in range(n):
        _, _, out, _ = oracle.verify(t, parent, token, 1, 1, temperature=T, seed=s * 2654435761 + 17)
        counts[out[0]] += 1
    p = np.exp(t[0].astype(np.float64) / T)
    p /= p.sum()
    chi2 = (((counts - n * p) ** 2) / (n * p)).sum()
    assert chi2 < 25.7  # 99.99th percentile of chi^2 with 5 dof


def test_coverage_identity():
    """Mean accepted length over seeds = covered target mass of the tree."""
    rng = np.random.default_rng(9)
    # a 9-node tree over V = 5, depth <= 3
    parent = np.array([-1, 0, 0, 1, 1, 2, 3, 3, 6], np.int32)
    token = np.array([0, 1, 3, 0, 2, 4, 1, 3, 2], np.int32)
    N, V, L, T = 9, 5, 3, 1.0
    t = rng.normal(0, 1.0, size=(N, V)).astype(np.float32)
    p = np.exp(t.astype(np.float64) / T)
    p /= p.sum(axis=1, keepdims=True)
    reach = np.zeros(N)
    reach[0] = 1.0
    for n in range(1, N):
        reach[n] = reach[parent[n]] * p[parent[n], token[n]]
    expect = reach[1:].sum()
    n_seeds = 40000
    acc = np.array([oracle.verify(t, parent, token, N, L, temperature=T, seed=s)[0] for s in range(n_seeds)])
    se = acc.std() / np.sqrt(n_seeds)
    assert abs(acc.mean() - expect) < 4 * se


def test_verify_rejects_bad_arguments():
    parent, token = _hand_tree()
    t = np.zeros((5, 10), np.float32)
    with pytest.raises(ValueError):
        oracle.verify(t, parent, token, 5, 3, temperature=-1.0)
