"""GPU parity: the mixture DDTree, bit-exact against the oracle given the same
fp32 top-k tables (node set and order, parents, tokens, depths, score bits,
modes, mask, positions).  Project page "Multi-Future Drafting", How it works,
step 3."""
import numpy as np
import pytest
import torch

import oracle
from tree_verified_speculative_gb300 import mfd, synth

from gpu_helpers import assert_tree_equal, gpu_tree

pytestmark = pytest.mark.gpu


def _random_tables(rng, n_req, K, L, k, V, values=None):
    lp = np.empty((n_req, K, L, k), np.float32)
    tk = np.empty((n_req, K, L, k), np.int32)
    for q in range(n_req):
        for m in range(K):
            for i in range(L):
                toks = rng.choice(V, size=k, replace=False)
                vals = (rng.choice(values, size=k) if values is not None
                        else -np.abs(rng.normal(3.0, 2.0, size=k))).astype(np.float32)
                order = np.lexsort((toks, -vals))
                lp[q, m, i] = vals[order]
                tk[q, m, i] = toks[order]
    return lp, tk


def _planted_tables(rng, n_req, K, L, k, V, n_shared):
    """Tables shaped like the drafter's: the planted future's token near
    -6.4, the rest of the top-k near -8 (not an LM head: fast to make)."""
    lp = np.empty((n_req, K, L, k), np.float32)
    tk = np.empty((n_req, K, L, k), np.int32)
    for q in range(n_req):
        fut = synth.futures(K, L, V, n_shared if np.isscalar(n_shared) else int(rng.integers(*n_shared)), rng)
        for m in range(K):
            for i in range(L):
                others = rng.choice(V, size=k + 4, replace=False)
                others = [t for t in others if t != fut[m, i]][: k - 1]
                toks = np.array([fut[m, i], *others])
                vals = np.concatenate([[-6.4 + rng.normal(0, 0.8)], -8.0 + rng.normal(0, 0.7, size=k - 1)])
                vals = vals.astype(np.float32)
                order = np.lexsort((toks, -vals))
                lp[q, m, i] = vals[order]
                tk[q, m, i] = toks[order]
    return lp, tk


def _compare(lp, tk, B, anchor=None, base_pos=None):
    g, st = gpu_tree(lp, tk, B, anchor, base_pos)
    assert st == 0
    o = oracle.build_tree(lp, tk, B, anchor, base_pos)
    for q in range(lp.shape[0]):
        assert_tree_equal(g, {k: v[q] for k, v in o.items()}, q)
    return g


def test_tiny_case():
    c = synth.tiny(seed=1)
    for topk in (8, 32):
        lp, tk, _ = oracle.logits_topk(c.logits, topk)
        for B in (1, 8, 40, 500):
            _compare(lp.reshape(1, c.K, c.L, topk), tk.reshape(1, c.K, c.L, topk), B)


@pytest.mark.parametrize("seed", range(24))
def test_random_tie_heavy(seed):
    rng = np.random.default_rng(seed)
    K = int(rng.integers(1, 6))
    L = int(rng.integers(1, 7))
    k = int(rng.integers(1, 9))
    V = 40
    vals = np.array([-0.25, -0.5, -1.0, -1.75], np.float32) if seed % 2 else \
        np.array([-0.1, -0.3, -0.7, -1.3], np.float32)
    lp, tk = _random_tables(rng, 2, K, L, k, V, vals)
    for B in (1, 5, 33, 128):
        _compare(lp, tk, B)


@pytest.mark.parametrize("B", [64, 256])
def test_pages_shape(B):
    rng = np.random.default_rng(B)
    lp, tk = _planted_tables(rng, 1, 8, 15, 16, 151936, 11)
    _compare(lp, tk, B, anchor=[42], base_pos=[977])


@pytest.mark.parametrize("seed", [33, 34, 35])
def test_wide_shape_topk32(seed):
    rng = np.random.default_rng(seed)
    lp, tk = _planted_tables(rng, 1, 8, 15, 32, 248320, 13)
    _compare(lp, tk, 256)


@pytest.mark.parametrize("V", [40, 64, 1000])
def test_wide_shape_topk32_shared_tokens_and_ties(V):
    """Top-32 rows whose pairs do not all fit the pool: depth 2 is counted,
    then made within a first bound.  Few distinct tokens (heavily shared
    between modes) and a coarse value grid (many equal scores)."""
    rng = np.random.default_rng(V)
    vals = np.array([-0.5, -1.0, -1.5, -2.0, -3.0], np.float32)
    lp, tk = _random_tables(rng, 2, 8, 15, 32, V, vals)
    for B in (64, 256):
        _compare(lp, tk, B)


def test_batched_32_requests():
    rng = np.random.default_rng(5)
    lp, tk = _planted_tables(rng, 32, 8, 15, 16, 151936, (8, 15))
    _compare(lp, tk, 128, anchor=np.arange(32) + 7, base_pos=np.arange(32) * 3)


def test_confident_deep_chains():
    """Confident modes (log p near 0 on the future): the tree reaches depth L."""
    rng = np.random.default_rng(8)
    lp, tk = _planted_tables(rng, 2, 8, 15, 16, 151936, 11)
    lp[..., 0] = -0.01 * (1 + rng.random(lp[..., 0].shape)).astype(np.float32)
    g = _compare(lp, tk, 256)
    assert g["depth"].max() == 15


def test_extreme_limits():
    rng = np.random.default_rng(9)
    lp, tk = _random_tables(rng, 1, 16, 16, 32, 100000)  # K*topk = 512 tokens per position
    _compare(lp, tk, 128)
    lp, tk = _random_tables(rng, 1, 4, 16, 32, 100000)
    _compare(lp, tk, 512)


def test_fewer_prefixes_than_budget_and_neg_inf():
    lp = np.array([[[[-0.5, -1.0]], [[-0.7, -np.inf]]]], np.float32)  # n_req=1, K=2, L=1, k=2
    tk = np.array([[[[3, 9]], [[9, 4]]]], np.int32)
    g = _compare(lp, tk, 10)
    assert g["n_nodes"][0] == 3


def test_deterministic_repeats():
    rng = np.random.default_rng(12)
    lp, tk = _planted_tables(rng, 4, 8, 15, 16, 151936, 11)
    first, _ = gpu_tree(lp, tk, 256)
    for _ in range(20):
        again, st = gpu_tree(lp, tk, 256)
        assert st == 0
        for k in first:
            np.testing.assert_array_equal(first[k], again[k])


def test_rejects_positive_or_unsorted_tables():
    lp = np.array([[[[0.5, -1.0]]]], np.float32)
    tk = np.array([[[[1, 2]]]], np.int32)
    _, st = gpu_tree(lp, tk, 4)
    assert st == mfd.MFD_ERR_INPUT
    lp = np.array([[[[-1.0, -0.5]]]], np.float32)
    _, st = gpu_tree(lp, tk, 4)
    assert st == mfd.MFD_ERR_INPUT
    lp = np.array([[[[-0.5, -1.0]]]], np.float32)
    tk = np.array([[[[2, 2]]]], np.int32)
    _, st = gpu_tree(lp, tk, 4)
    assert st == mfd.MFD_ERR_INPUT


@pytest.mark.parametrize("topk", [16, 5])
@pytest.mark.parametrize("kind", ["dup", "nan", "unsorted", "positive"])
@pytest.mark.parametrize("row", [0, 77, 119])
def test_rejects_bad_entries_anywhere(topk, kind, row):
    """The input checks cover every row of a full table, both rows a warp
    checks at once, the last entry of a row and rows narrower than their
    lane segment (top-5 in segments of 8): a repeated token, a NaN, an
    unsorted pair or a positive log p anywhere is MFD_ERR_INPUT, and the
    same tables without the fault build."""
    rng = np.random.default_rng(40 + row)
    lp, tk = _planted_tables(rng, 1, 8, 15, topk, 151936, 11)
    _, st = gpu_tree(lp, tk, 64)
    assert st == 0
    k, i = divmod(row, 15)
    j = topk - 1
    lp2, tk2 = lp.copy(), tk.copy()
    if kind == "dup":
        tk2[0, k, i, j] = tk2[0, k, i, 0]
    elif kind == "nan":
        lp2[0, k, i, j] = np.nan
    elif kind == "unsorted":
        lp2[0, k, i, j] = lp2[0, k, i, j - 1] + 0.5
        assert lp2[0, k, i, j] < 0
    else:
        lp2[0, k, i, j] = 0.25
    _, st = gpu_tree(lp2, tk2, 64)
    assert st == mfd.MFD_ERR_INPUT


def test_rejects_out_of_limits():
    rd = mfd.Round(1, 17, 2, 4, 8, 64)
    with pytest.raises(mfd.MfdError) as e:
        rd.build_tree()
    assert e.value.code == mfd.MFD_ERR_UNSUPPORTED


@pytest.mark.parametrize("value,shared", [(0.0, True), (0.0, False), (-1.0, True), (-1.0, False)])
def test_all_equal_log_probs_at_the_limits(value, shared):
    """Every log p equal, at the largest shape (K=16, L=16, top-32, B=128):
    every prefix of a depth ties with all others, so the token order decides
    everything (model card "MFD drafter for Qwen3.5-4B", first paragraph:
    ties to the lexicographically smaller ids).  At log p = 0 the first B
    prefixes in that order form a chain of depth L with siblings, the case
    where the pruning bound is weakest; with shared rows every prefix is
    held by all 16 modes.  The level search's pass count is bounded by
    2 + K*B*topk / (pool - K*B) = 39 here, below its limit of 64."""
    rng = np.random.default_rng(17 if shared else 18)
    K, L, k, B = 16, 16, 32, 128
    tk = np.empty((1, K, L, k), np.int32)
    for i in range(L):
        row = np.sort(rng.choice(1000, size=k, replace=False))
        for m in range(K):
            tk[0, m, i] = row if shared else np.sort(rng.choice(100000, size=k, replace=False))
    lp = np.full((1, K, L, k), value, np.float32)
    g = _compare(lp, tk, B)
    if value == 0.0:
        assert g["depth"].max() == L


def test_two_value_ties_deep_at_the_limits():
    """Log p drawn from {-0.001, -0.002} at K=16, L=16, top-32, B=128: deep
    trees where many prefixes tie at the cut-off."""
    rng = np.random.default_rng(19)
    lp, tk = _random_tables(rng, 2, 16, 16, 32, 5000, values=np.array([-0.001, -0.002], np.float32))
    _compare(lp, tk, 128)
