"""Pins of the oracle's tree analytics (oracle/analytics.py): chimera
classes against a hand tree and the pages' chimera bound (project page
"Multi-Future Drafting", TL;DR and Abstract); covered mass against the
independent walk oracle (How it works, step 1: the expected accepted length
is the covered mass), exactly for greedy walks and in distribution for
sampled ones."""
import numpy as np
import pytest

import oracle
from oracle import analytics
from test_oracle_tree import CHIMERAS, _chimera_tables


def _tree_arrays(t, q=0):
    n = int(np.asarray(t["n_nodes"]).reshape(-1)[q])
    pick = lambda k: np.asarray(t[k]).reshape(-1, np.asarray(t[k]).shape[-1])[q]  # noqa: E731
    return pick("parent"), pick("token"), pick("depth"), n


def test_hand_tree_classes():
    # futures A = (1, 2, 3) and B = (1, 4, 5) share position 1
    futures = np.array([[1, 2, 3], [1, 4, 5]])
    # root; (1); (1,2); (1,4); (1,2,5); (1,4,3); (1,7); (2); (1,2,3)
    parent = np.array([-1, 0, 1, 1, 2, 3, 1, 0, 2])
    token = np.array([9, 1, 2, 4, 5, 3, 7, 2, 3])
    cls = analytics.node_classes(parent, token, 9, futures)
    F, C, O = analytics.ON_FUTURE, analytics.CHIMERA, analytics.OTHER
    assert list(cls) == [F, F, F, F, C, C, O, O, F]


def test_parents_must_come_first():
    with pytest.raises(ValueError):
        analytics.node_classes(np.array([-1, 2, 0]), np.array([0, 1, 2]), 3, np.array([[1, 2]]))


@pytest.mark.parametrize("m", [2, 3, 4, 5, 6])
def test_chimera_bound(m):
    """The smallest product-ranked (K = 1) tree holding two futures that
    differ in m positions holds exactly 2^(m-1) - 1 full-length chimeras when
    the futures score alike and no splice ties them (tests/golden)."""
    rng = np.random.default_rng(50 + m)
    L = 8
    lp, tk, A, Bf = _chimera_tables(m, L, rng)
    t = oracle.build_tree(lp, tk, 400)
    parent, token, depth, n = _tree_arrays(t)
    futures = np.stack([A, Bf])
    full = analytics.node_classes(parent, token, n, futures)
    # the smallest budget holding both futures: the later of their two nodes
    seqs = analytics._sequences(parent, token, n)
    need = max(seqs.index(tuple(int(x) for x in A)), seqs.index(tuple(int(x) for x in Bf))) + 1
    cls = full[:need]
    assert int(np.sum((cls == analytics.CHIMERA) & (depth[:need] == L))) == CHIMERAS[m]


def _random_tree(rng, K, L, k, V, B):
    lp = -np.abs(rng.normal(2.0, 1.0, size=(1, K, L, k))).astype(np.float32)
    tk = np.empty((1, K, L, k), np.int32)
    for m in range(K):
        for i in range(L):
            tk[0, m, i] = rng.choice(V, size=k, replace=False)
    order = np.argsort(-lp, axis=-1, kind="stable")
    lp = np.take_along_axis(lp, order, -1)
    tk = np.take_along_axis(tk, order, -1)
    return oracle.build_tree(lp, tk, B)


@pytest.mark.parametrize("seed", range(6))
def test_greedy_mass_is_the_walk(seed):
    """At T = 0 the covered mass is the greedy walk's accepted length, exactly."""
    rng = np.random.default_rng(seed)
    K, L, k, V, B = 3, 5, 4, 12, 40
    t = _random_tree(rng, K, L, k, V, B)
    parent, token, depth, n = _tree_arrays(t)
    tgt = rng.normal(0, 1, size=(n, V)).astype(np.float32)
    # lean the target toward the tree's tokens so that walks go deep
    for c in range(1, n):
        tgt[parent[c], token[c]] += np.float32(rng.uniform(0, 3))
    _, mass = analytics.covered_mass(parent, token, depth, n, tgt, 0.0, L)
    acc = oracle.verify(tgt, parent, token, n, L, 0.0, 0)[0]
    assert mass[0] == 1.0
    assert mass[1:].sum() == acc
    assert all(mass[d] == (1.0 if d <= acc else 0.0) for d in range(L + 1))


def test_sampled_mass_by_depth_matches_the_walks():
    """At T = 1, mass[d] = P(accepted >= d): the oracle walk over many seeds
    agrees depth by depth within four standard errors."""
    rng = np.random.default_rng(11)
    parent = np.array([-1, 0, 0, 1, 1, 2, 3, 3, 6], np.int32)
    token = np.array([0, 1, 3, 0, 2, 4, 1, 3, 2], np.int32)
    depth = np.array([0, 1, 1, 2, 2, 2, 3, 3, 4], np.int32)
    N, V, L, T = 9, 5, 4, 1.0
    tgt = rng.normal(0, 1.0, size=(N, V)).astype(np.float32)
    _, mass = analytics.covered_mass(parent, token, depth, N, tgt, T, L)
    n_seeds = 30000
    acc = np.array([oracle.verify(tgt, parent, token, N, L, T, s)[0] for s in range(n_seeds)])
    for d in range(1, L + 1):
        hit = (acc >= d).astype(np.float64)
        se = max(hit.std(), 1e-3) / np.sqrt(n_seeds)
        assert abs(hit.mean() - mass[d]) < 4 * se, (d, hit.mean(), mass[d])
    assert abs(acc.mean() - mass[1:].sum()) < 4 * acc.std() / np.sqrt(n_seeds)
