"""GPU parity of the tree analytics (mfd_tree_analytics) against the oracle's
(oracle/analytics.py): chimera classes exactly, reach and covered mass by
depth within 1e-6 (project page "Multi-Future Drafting", TL;DR and Abstract:
chimeras; How it works, step 1, and "What the modes are", Figure 3: covered
mass by depth)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import analytics
from tree_verified_speculative_gb300 import mfd, synth

from gpu_helpers import gpu_tree, np_, tree_outputs
from test_oracle_tree import CHIMERAS, _chimera_tables

pytestmark = pytest.mark.gpu

MASS_TOL = 1e-6


def _gpu(parent, token, depth, n_nodes, L, futures, t, temps):
    """Arrays [n_req, ...] on the host -> (classes, reach, mass) on the host."""
    d = lambda a, dt=torch.int32: torch.from_numpy(np.ascontiguousarray(a)).to(dt).cuda()  # noqa: E731
    cls, reach, mass, st = mfd.tree_analytics(d(parent), d(token), d(depth), d(n_nodes), L, d(futures),
                                             d(t, torch.float32), d(np.asarray(temps, np.float32), torch.float32))
    torch.cuda.synchronize()
    assert int(st.item()) == 0, mfd.status_string(int(st.item()))
    return np_(cls), np_(reach), np_(mass)


def _check(parent, token, depth, n_nodes, L, futures, t, temps):
    g_cls, g_reach, g_mass = _gpu(parent, token, depth, n_nodes, L, futures, t, temps)
    for q in range(parent.shape[0]):
        n = int(n_nodes[q])
        o_cls = analytics.node_classes(parent[q], token[q], n, futures[q])
        np.testing.assert_array_equal(g_cls[q, :n], o_cls)
        assert np.all(g_cls[q, n:] == -1)
        o_reach, o_mass = analytics.covered_mass(parent[q], token[q], depth[q], n, t[q], float(temps[q]), L)
        np.testing.assert_allclose(g_reach[q, :n], o_reach, rtol=0, atol=MASS_TOL)
        np.testing.assert_allclose(g_mass[q], o_mass, rtol=0, atol=MASS_TOL)
    return g_cls, g_mass


def test_hand_tree():
    futures = np.array([[[1, 2, 3], [1, 4, 5]]], np.int32)
    parent = np.array([[-1, 0, 1, 1, 2, 3, 1, 0, 2]], np.int32)
    token = np.array([[9, 1, 2, 4, 5, 3, 7, 2, 3]], np.int32)
    depth = np.array([[0, 1, 2, 2, 3, 3, 2, 1, 3]], np.int32)
    rng = np.random.default_rng(3)
    t = rng.normal(0, 1.5, size=(1, 9, 10)).astype(np.float32)
    for T in (0.0, 1.0, 0.5):
        cls, _ = _check(parent, token, depth, np.array([9]), 3, futures, t, [T])
    F, C, O = mfd.MFD_NODE_ON_FUTURE, mfd.MFD_NODE_CHIMERA, mfd.MFD_NODE_OTHER
    assert list(cls[0]) == [F, F, F, F, C, C, O, O, F]


@pytest.mark.parametrize("m", [2, 3, 4, 5, 6])
def test_chimera_bound_trees(m):
    """The product-ranked (K = 1) trees of the chimera bound: the classes the
    GPU gives count 2^(m-1) - 1 full-length chimeras at the smallest budget
    holding both futures (tests/golden/chimera_bound.txt)."""
    rng = np.random.default_rng(50 + m)
    L = 8
    lp, tk, A, Bf = _chimera_tables(m, L, rng)
    tr = oracle.build_tree(lp, tk, 400)
    n = int(tr["n_nodes"])
    futures = np.stack([A, Bf])[None].astype(np.int32)
    t = rng.normal(0, 1, size=(1, 401, 64)).astype(np.float32)  # the tables' tokens lie in [0, 64)
    cls, _ = _check(tr["parent"][None], tr["token"][None], tr["depth"][None], np.array([n]), L, futures, t, [1.0])
    seqs = analytics._sequences(tr["parent"], tr["token"], n)
    need = max(seqs.index(tuple(int(x) for x in A)), seqs.index(tuple(int(x) for x in Bf))) + 1
    full_len = tr["depth"][:need] == L
    assert int(np.sum((cls[0, :need] == mfd.MFD_NODE_CHIMERA) & full_len)) == CHIMERAS[m]


@pytest.fixture(scope="module")
def head():
    W = synth.lm_head(151936, 2560, seed=2024)
    return W, mfd.pack_lm_head(W.cuda())


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_pages_shape_rounds(head, T):
    """Four requests at the pages' shape (K=8, L=15, V=151,936, top-16,
    B=256) through the LM head and the tree, with target rows planted along a
    mode's future: classes against the K planted futures, reach and mass."""
    W, Wp = head
    n = 4
    rounds = [synth.round_inputs(W, 8, 15, 11, seed=4000 + q) for q in range(n)]
    rd = mfd.Round(n, 8, 15, 16, 256, 151936)
    rd.status.zero_()
    rd.lmhead_topk_packed(torch.cat([r.h for r in rounds], 0).cuda(), Wp)
    rd.build_tree()
    torch.cuda.synchronize()
    assert int(rd.status.item()) == 0
    g = tree_outputs(rd)
    t = np.empty((n, 257, 151936), np.float32)
    for q, r in enumerate(rounds):
        rows, cols = synth.plant_sites(g["parent"][q], g["token"][q], g["depth"][q], int(g["n_nodes"][q]),
                                       r.fut[r.target_mode])
        t[q] = synth.plant(synth.target_noise(257, 151936, np.random.default_rng(q)), rows, cols)
    futures = np.stack([r.fut for r in rounds]).astype(np.int32)
    cls, mass = _check(g["parent"], g["token"], g["depth"], g["n_nodes"], 15, futures, t, [T] * n)
    if T == 0.0:
        # greedy: the walk follows the planted future as far as the tree holds it
        assert all(mass[q, 1] == 1.0 for q in range(n))


def test_mixture_tree_holds_fewer_chimeras_than_the_product_tree(head):
    """The pages' claim on the synthetic generator (project page, TL;DR and
    Abstract: chimeras are 27-33% of a 64-node product tree; the mixture tree
    lets each mode keep its own future).  K = 8 modes with planted futures
    sharing 11 of 15 positions, drafted confidently (hidden scale 12: the
    planted token holds about 0.6 of its row, the pages' regime; at the
    benchmark's scale 6 it holds about 0.002 and 64-node trees stay too
    shallow to splice); the product tree is the K = 1 tree over the modes'
    mean marginals (the product of the modes' mean marginals, "What the modes
    are"), its table made by the oracle's LM head; both trees B = 64,
    classified on the GPU against the 8 futures.  Prints both shares."""
    W, Wp = head
    shares = {1: [], 8: []}
    for i in range(4):
        r = synth.round_inputs(W, 8, 15, 11, seed=5000 + i, scale=12.0)
        rd = mfd.Round(1, 8, 15, 16, 64, 151936)
        rd.status.zero_()
        rd.lmhead_topk_packed(r.h.cuda(), Wp)
        rd.build_tree()
        torch.cuda.synchronize()
        g8 = tree_outputs(rd)
        bits = r.h.contiguous().view(torch.int16).numpy().view(np.uint16)
        z = oracle.lmhead_logits(bits, W)  # [120, V] double
        z = z - z.max(axis=1, keepdims=True)
        p = np.exp(z)
        p /= p.sum(axis=1, keepdims=True)
        mean = p.reshape(8, 15, -1).mean(axis=0)  # [15, V]
        logm = np.log(mean).astype(np.float32)
        order = np.lexsort((np.broadcast_to(np.arange(logm.shape[1]), logm.shape), -logm), axis=1)[:, :16]
        lp1 = np.take_along_axis(logm, order, 1)[None, None]
        tk1 = order.astype(np.int32)[None, None]
        g1, st = gpu_tree(lp1, tk1, 64)
        assert st == 0
        t = np.zeros((2, 65, 151936), np.float32)
        fut = np.stack([r.fut, r.fut]).astype(np.int32)
        stack = lambda k: np.stack([g8[k][0], g1[k][0]])  # noqa: E731
        n_nodes = np.array([g8["n_nodes"][0], g1["n_nodes"][0]])
        cls, _, _ = _gpu(stack("parent"), stack("token"), stack("depth"), n_nodes, 15, fut, t, [0.0, 0.0])
        for j, K in enumerate((8, 1)):
            shares[K].append(float(np.mean(cls[j, 1:int(n_nodes[j])] == mfd.MFD_NODE_CHIMERA)))
    s8, s1 = float(np.mean(shares[8])), float(np.mean(shares[1]))
    print(f"chimera share of a 64-node tree: K=8 mixture {s8:.3f}, K=1 mean-marginal product {s1:.3f} "
          f"(per round {shares[8]} / {shares[1]})")
    assert s8 < s1
