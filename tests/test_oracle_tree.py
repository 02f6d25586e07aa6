"""Pins of the oracle's mixture DDTree (CPU only).

Project page "Multi-Future Drafting", How it works, step 3: every prefix is
scored by its best mode, the B best prefixes over all modes form one tree,
exactly the union of the per-mode trees, found by merging the K best-first
searches into one heap.  Abstract / TL;DR: a product-ranked tree holding two
futures that disagree in m positions holds at least 2^(m-1) - 1 chimeras,
barring ties.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
from tree_verified_speculative_gb300 import synth

from bruteforce import brute_tree, node_sequences, product_brute, sort_prefixes

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden_chimeras():
    """m -> chimera count, from tests/golden/chimera_bound.txt (the pages' bound)."""
    with open(os.path.join(HERE, "golden", "chimera_bound.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    return {int(a): int(b) for a, b in rows}


CHIMERAS = _golden_chimeras()


def _oracle_nodes(t):
    n = int(t["n_nodes"])
    seqs = node_sequences(t["parent"], t["token"], n)
    return [(t["score"][i], seqs[i], int(t["mode"][i])) for i in range(1, n)]


def _assert_same(ora, ref):
    assert len(ora) == len(ref)
    for (s1, q1, m1), (s2, q2, m2) in zip(ora, ref):
        assert q1 == q2
        assert np.float32(s1).tobytes() == np.float32(s2).tobytes()
        assert m1 == m2


def _tiny_tables(topk):
    c = synth.tiny(seed=1)
    lp, tk, _ = oracle.logits_topk(c.logits, topk)
    return c, lp.reshape(c.K, c.L, topk), tk.reshape(c.K, c.L, topk)


@pytest.mark.parametrize("topk", [8, 32])
def test_tiny_case_matches_brute_force(topk):
    """Tiny case: K=2, L=4, V=32; every one of the 1,082,400 prefixes listed."""
    c, lp, tk = _tiny_tables(topk)
    for B in (1, 2, 8, 40):
        t = oracle.build_tree(lp, tk, B)
        _assert_same(_oracle_nodes(t), brute_tree(lp, tk, c.V, B))


def _random_tables(rng, K, L, k, V, values):
    lp = np.empty((K, L, k), np.float32)
    tk = np.empty((K, L, k), np.int32)
    for m in range(K):
        for i in range(L):
            toks = rng.choice(V, size=k, replace=False)
            vals = rng.choice(values, size=k).astype(np.float32)
            order = np.lexsort((toks, -vals))
            lp[m, i] = vals[order]
            tk[m, i] = toks[order]
    return lp, tk


@pytest.mark.parametrize("seed", range(40))
def test_random_ties_match_brute_force(seed):
    rng = np.random.default_rng(seed)
    K = int(rng.integers(1, 4))
    L = int(rng.integers(1, 5))
    k = int(rng.integers(1, 5))
    V = 8
    # a 4-value set forces exact score ties between prefixes and modes
    values = np.array([-0.25, -0.5, -1.0, -1.75], np.float32) if seed % 2 else \
        np.array([-0.1, -0.3, -0.7, -1.3], np.float32)  # inexact sums: rounding ties
    lp, tk = _random_tables(rng, K, L, k, V, values)
    for B in (1, 3, 10, 1000):
        t = oracle.build_tree(lp, tk, B)
        _assert_same(_oracle_nodes(t), brute_tree(lp, tk, V, B))


@pytest.mark.parametrize("seed", range(8))
def test_k1_is_product_ranked_tree(seed):
    """K = 1 reduces the mixture to DDTree's product ranking."""
    rng = np.random.default_rng(1000 + seed)
    L, k, V = 4, 4, 16
    lp, tk = _random_tables(rng, 1, L, k, V, np.array([-0.2, -0.6, -0.9, -2.0, -3.1], np.float32))
    for B in (5, 30, 400):
        t = oracle.build_tree(lp, tk, B)
        _assert_same(_oracle_nodes(t), product_brute(lp[0], tk[0], V, B))


def _structure_checks(t, B, L, n_finite=None, base_pos=0, anchor=0):
    n = int(t["n_nodes"])
    N = B + 1
    W32 = (N + 31) // 32
    assert t["mask"].shape == (N, W32)
    assert t["token"][0] == anchor and t["depth"][0] == 0 and t["parent"][0] == -1
    seqs = node_sequences(t["parent"], t["token"], n)
    assert len(set(seqs)) == n  # no duplicate sequences
    keys = [(-float(t["score"][i]), seqs[i]) for i in range(1, n)]
    assert keys == sorted(keys)  # node order = key order
    for i in range(1, n):
        p = int(t["parent"][i])
        assert 0 <= p < i
        assert t["depth"][i] == t["depth"][p] + 1 and 1 <= t["depth"][i] <= L
        assert t["score"][i] <= t["score"][p] or p == 0
        assert t["pos"][i] == base_pos + t["depth"][i]
        # mask row = ancestor-or-self set
        anc = set()
        a = i
        while a >= 0:
            anc.add(a)
            a = int(t["parent"][a])
        bits = {j for j in range(N) if (int(t["mask"][i, j // 32]) >> (j % 32)) & 1}
        assert bits == anc
    for i in range(n, N):
        assert t["parent"][i] == -1 and t["token"][i] == -1 and t["depth"][i] == -1
        assert not t["mask"][i].any() and t["score"][i] == -np.inf
    if n_finite is not None:
        assert n - 1 == min(B, n_finite)


def test_structure_on_pages_shape():
    """K=8, L=15, top-k 16, B=256 tables from planted futures (random, not an LM head)."""
    rng = np.random.default_rng(7)
    K, L, k, V = 8, 15, 16, 151936
    fut = synth.futures(K, L, V, 11, rng)
    lp = np.sort(-np.abs(rng.normal(8.0, 1.0, size=(K, L, k))).astype(np.float32), axis=2)[..., ::-1].copy()
    lp[..., 0] = -6.4 + rng.normal(0, 0.3, size=(K, L)).astype(np.float32)
    lp = np.sort(lp, axis=2)[..., ::-1].copy()
    tk = rng.integers(0, V, size=(K, L, k)).astype(np.int32)
    tk[..., 0] = fut
    for m in range(K):
        for i in range(L):  # distinct tokens within a row
            row = list(dict.fromkeys(tk[m, i].tolist()))
            while len(row) < k:
                row.append(int(rng.integers(0, V)))
                row = list(dict.fromkeys(row))
            tk[m, i] = row
    for B in (64, 256):
        t = oracle.build_tree(lp, tk, B, anchor=np.array([123]), base_pos=np.array([1000]))
        _structure_checks(t, B, L, base_pos=1000, anchor=123)
        assert int(t["n_nodes"]) == B + 1


def test_union_of_per_mode_trees():
    """The mixture tree equals the union of the per-mode trees cut at the
    common cut-off (the B-th best key)."""
    rng = np.random.default_rng(11)
    K, L, k, V, B = 4, 6, 5, 40, 60
    lp, tk = _random_tables(rng, K, L, k, V, np.array([-0.3, -0.8, -1.1, -1.9, -2.6], np.float32))
    t = oracle.build_tree(lp, tk, B)
    mix = _oracle_nodes(t)
    cut = (-float(mix[-1][0]), mix[-1][1])
    union = set()
    for m in range(K):
        tm = oracle.build_tree(lp[m:m + 1], tk[m:m + 1], B)
        for s, q, _ in _oracle_nodes(tm):
            if (-float(s), q) <= cut:
                union.add(q)
    assert union == {q for _, q, _ in mix}


def test_empty_and_degenerate():
    # fewer finite prefixes than B: the tree holds all of them
    lp = np.array([[[-0.5, -1.0]], [[-0.7, -np.inf]]], np.float32)  # K=2, L=1, k=2
    tk = np.array([[[3, 9]], [[9, 4]]], np.int32)
    t = oracle.build_tree(lp, tk, 10)
    assert int(t["n_nodes"]) == 3  # tokens 3 and 9; 9 takes its best mode, mode 1
    nodes = _oracle_nodes(t)
    assert [q for _, q, _ in nodes] == [(3,), (9,)]
    assert nodes[1][0] == np.float32(-0.7) and nodes[1][2] == 1
    # all -inf: only the root
    t = oracle.build_tree(np.full((1, 2, 2), -np.inf, np.float32), np.zeros((1, 2, 2), np.int32) + [[0, 1]], 4)
    assert int(t["n_nodes"]) == 1
    # B = 1: the single best depth-1 prefix
    t = oracle.build_tree(lp, tk, 1)
    assert _oracle_nodes(t)[0][1] == (3,)


# --------------------------------------------------------------------------
# chimera bound (abstract / TL;DR)

def _chimera_tables(m, L, rng):
    """K=1 tables: futures A and B share L-m positions and differ in m.
    Dyadic log-probs keep every fp32 sum exact; s(A) == s(B) by construction
    and no splice ties s(A)."""
    V = 64
    while True:
        A = rng.choice(V, size=L, replace=False).astype(np.int32)
        Bf = A.copy()
        diff = np.sort(rng.choice(L, size=m, replace=False))
        for j in diff:
            Bf[j] = (A[j] + 1 + int(rng.integers(0, V - 1))) % V
            while Bf[j] in A:
                Bf[j] = (Bf[j] + 1) % V
        a = -(1.0 + rng.integers(0, 32, size=m) / 16.0)
        b = -(1.0 + rng.integers(0, 32, size=m) / 16.0)
        b[-1] = a.sum() - b[:-1].sum()
        if not (-4.0 <= b[-1] < 0):
            continue
        splices = []
        for mask in itertools.product([0, 1], repeat=m):
            if all(x == 0 for x in mask) or all(x == 1 for x in mask):
                continue
            splices.append(sum(b[j] if mask[j] else a[j] for j in range(m)))
        if any(abs(sv - a.sum()) < 1e-12 for sv in splices):
            continue
        break
    k = 3
    lp = np.empty((1, L, k), np.float32)
    tk = np.empty((1, L, k), np.int32)
    di = {int(j): n for n, j in enumerate(diff)}
    for i in range(L):
        if i in di:
            vals = [a[di[i]], b[di[i]], -100.0]
            toks = [A[i], Bf[i], (max(A.max(), Bf.max()) + 1 + i) % V]
        else:
            vals = [-0.5, -100.0, -100.5]
            toks = [A[i], (max(A.max(), Bf.max()) + 1 + i) % V, (max(A.max(), Bf.max()) + 20 + i) % V]
        order = np.lexsort((np.asarray(toks), -np.asarray(vals)))
        lp[0, i] = np.asarray(vals, np.float32)[order]
        tk[0, i] = np.asarray(toks, np.int32)[order]
    return lp, tk, A, Bf


def _count_chimeras(nodes, A, Bf, L):
    full = [q for _, q, _ in nodes if len(q) == L]
    return sum(1 for q in full if q not in (tuple(A), tuple(Bf))
               and all(q[i] in (A[i], Bf[i]) for i in range(L)))


@pytest.mark.parametrize("m", [2, 3, 4, 5, 6])
def test_chimera_bound_exact(m):
    rng = np.random.default_rng(50 + m)
    L = 8
    lp, tk, A, Bf = _chimera_tables(m, L, rng)
    t = oracle.build_tree(lp, tk, 400)
    nodes = _oracle_nodes(t)
    seqs = [q for _, q, _ in nodes]
    iA, iB = seqs.index(tuple(A)), seqs.index(tuple(Bf))
    need = max(iA, iB) + 1  # smallest budget holding both futures
    assert _count_chimeras(nodes[:need], A, Bf, L) == CHIMERAS[m]
    # any larger budget holds at least as many
    for extra in (1, 10, 50):
        assert _count_chimeras(nodes[:need + extra], A, Bf, L) >= CHIMERAS[m]


def test_chimera_bound_on_tiny_case():
    """Tiny case, K=1 table = log of the mean of the two modes' probabilities:
    m = 2 differing positions, so at least one chimera once both futures are
    held.  The two-mode mixture tree is reported, not asserted."""
    c = synth.tiny(seed=1)
    z = c.logits.reshape(c.K, c.L, c.V).astype(np.float64)
    p = np.exp(z - z.max(axis=2, keepdims=True))
    p /= p.sum(axis=2, keepdims=True)
    mean_lp = np.log(p.mean(axis=0))  # [L, V]
    lp1, tk1, _ = oracle.logits_topk(mean_lp.astype(np.float32), c.V)
    lp1, tk1 = lp1.reshape(1, c.L, c.V), tk1.reshape(1, c.L, c.V)
    t = oracle.build_tree(lp1, tk1, 2000)
    nodes = _oracle_nodes(t)
    seqs = [q for _, q, _ in nodes]
    A, Bf = c.fut
    need = max(seqs.index(tuple(A)), seqs.index(tuple(Bf))) + 1
    assert _count_chimeras(nodes[:need], A, Bf, c.L) >= 1


def test_golden_chimera_counts_cover_m2_to_m6():
    assert sorted(CHIMERAS) == [2, 3, 4, 5, 6]
