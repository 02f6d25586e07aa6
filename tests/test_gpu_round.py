"""GPU parity of whole rounds on the five workloads (the three calls back to
back on one stream, as the benchmark runs them), against the oracle.

Stages are checked the way the method statement asks: top-k tables against
the oracle's LM head (sampled rows at full size); the tree bit-exact against
the oracle's tree built from the GPU's own tables; the walk against the
oracle's walk over the same tree and target logits."""
import numpy as np
import pytest
import torch

import oracle
from tree_verified_speculative_gb300 import mfd, synth

from gpu_helpers import assert_tree_equal, check_topk, check_walk, np_, tree_outputs

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_tiny_round():
    c = synth.tiny(seed=1)
    rd = mfd.Round(1, c.K, c.L, c.topk, c.B, c.V)
    rd.status.zero_()
    rd.logits_topk(torch.from_numpy(c.logits).cuda())
    rd.build_tree()
    torch.cuda.synchronize()
    lp, tk = np_(rd.tk_logp), np_(rd.tk_tok)
    o_lp, o_tk, _ = oracle.logits_topk(c.logits, c.topk)
    check_topk(lp, tk, o_lp, o_tk)
    g = tree_outputs(rd)
    o = oracle.build_tree(lp.reshape(c.K, c.L, c.topk), tk.reshape(c.K, c.L, c.topk), c.B)
    assert_tree_equal(g, o, 0)
    rng = np.random.default_rng(5)
    noise = synth.target_noise(c.B + 1, c.V, rng)
    rows, cols = synth.plant_sites(o["parent"], o["token"], o["depth"], int(o["n_nodes"]), c.fut[1])
    t = synth.plant(noise, rows, cols)
    rd.verify(torch.from_numpy(t[None]).cuda(), torch.zeros(1, device="cuda"),
              torch.zeros(1, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert int(rd.status.item()) == 0
    oa = oracle.verify(t, o["parent"], o["token"], int(o["n_nodes"]), c.L)
    check_walk(int(np_(rd.accept_len)[0]), np_(rd.path_nodes)[0], np_(rd.out_tokens)[0], *oa, sampled=False)


@pytest.fixture(scope="module")
def head():
    W = synth.lm_head(151936, 2560, seed=2024)
    return W, W.cuda()


def _round(W, Wd, rd, r: synth.Round, temperature: float, rows_checked, check_tables=True):
    """One round through the three calls; returns the numbers of exact walks."""
    rd.status.zero_()
    rd.lmhead_topk(r.h.cuda(), Wd)
    rd.build_tree()
    torch.cuda.synchronize()
    assert int(rd.status.item()) == 0
    K, L, k, B = rd.K, rd.L, rd.topk, rd.B
    lp, tk = np_(rd.tk_logp), np_(rd.tk_tok)
    if check_tables:
        o_lp, o_tk, _ = oracle.lmhead_topk(_bits(r.h[rows_checked]), _bits(W), k)
        check_topk(lp[rows_checked], tk[rows_checked], o_lp, o_tk)
    g = tree_outputs(rd)
    o = oracle.build_tree(lp.reshape(K, L, k), tk.reshape(K, L, k), B)
    assert_tree_equal(g, o, 0)
    rng = np.random.default_rng(r.seed % (2**32))
    noise = synth.target_noise(B + 1, W.shape[0], rng)
    rows, cols = synth.plant_sites(o["parent"], o["token"], o["depth"], int(o["n_nodes"]), r.fut[r.target_mode])
    t = synth.plant(noise, rows, cols)
    rd.verify(torch.from_numpy(t[None]).cuda(), torch.tensor([temperature], device="cuda"),
              torch.tensor([r.seed], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert int(rd.status.item()) == 0
    oa = oracle.verify(t, o["parent"], o["token"], int(o["n_nodes"]), L, temperature, r.seed)
    return check_walk(int(np_(rd.accept_len)[0]), np_(rd.path_nodes)[0], np_(rd.out_tokens)[0], *oa,
                      sampled=temperature > 0)


def test_pages_shape_greedy_b64(head):
    W, Wd = head
    rd = mfd.Round(1, 8, 15, 16, 64, 151936)
    r = synth.round_inputs(W, 8, 15, 11, seed=11)
    assert _round(W, Wd, rd, r, 0.0, np.arange(0, 120, 7))


def test_pages_shape_sampled_b256(head):
    """B=256, T=1 (the sampled budget case): 64 seeded rounds with W fixed and
    fresh futures, hidden states, target rows and seeds per round.  Every
    round's tree is bit-exact against the oracle built from the GPU's tables
    and its walk exact (up to the 1e-5 excuse); two rows a round are checked
    against the oracle's full-vocabulary LM head."""
    W, Wd = head
    rd = mfd.Round(1, 8, 15, 16, 256, 151936)
    n = 64
    exact = 0
    for i in range(n):
        r = synth.round_inputs(W, 8, 15, 11, seed=1000 + i)
        rows = np.array([(7 * i) % 120, (7 * i + 61) % 120])
        exact += _round(W, Wd, rd, r, 1.0, rows)
    assert exact >= n - 3


def test_batched_32_requests(head):
    W, Wd = head
    n = 32
    rng = np.random.default_rng(77)
    rounds = [synth.round_inputs(W, 8, 15, int(rng.integers(8, 15)), seed=500 + q) for q in range(n)]
    h = torch.cat([r.h for r in rounds], 0)
    rd = mfd.Round(n, 8, 15, 16, 128, 151936)
    rd.status.zero_()
    rd.lmhead_topk(h.cuda(), Wd)
    rd.build_tree()
    torch.cuda.synchronize()
    assert int(rd.status.item()) == 0
    lp, tk = np_(rd.tk_logp), np_(rd.tk_tok)
    rows = np.array([3, 500, 1800, 3839])
    o_lp, o_tk, _ = oracle.lmhead_topk(_bits(h[rows]), _bits(W), 16)
    check_topk(lp[rows], tk[rows], o_lp, o_tk)
    g = tree_outputs(rd)
    lp4, tk4 = lp.reshape(n, 8, 15, 16), tk.reshape(n, 8, 15, 16)
    o = oracle.build_tree(lp4, tk4, 128)
    for q in range(n):
        assert_tree_equal(g, {k: v[q] for k, v in o.items()}, q)
    t = np.empty((n, 129, 151936), np.float32)
    for q in range(n):
        noise = synth.target_noise(129, 151936, np.random.default_rng(q))
        rows_, cols_ = synth.plant_sites(o["parent"][q], o["token"][q], o["depth"][q], int(o["n_nodes"][q]),
                                         rounds[q].fut[rounds[q].target_mode])
        t[q] = synth.plant(noise, rows_, cols_)
    temps = np.array([0.0] * 16 + [1.0] * 16, np.float32)
    seeds = np.array([r.seed for r in rounds], np.uint64)
    rd.verify(torch.from_numpy(t).cuda(), torch.from_numpy(temps).cuda(),
              torch.from_numpy(seeds.view(np.int64)).cuda())
    torch.cuda.synchronize()
    assert int(rd.status.item()) == 0
    exact = 0
    for q in range(n):
        oa = oracle.verify(t[q], o["parent"][q], o["token"][q], int(o["n_nodes"][q]), 15, float(temps[q]),
                           int(seeds[q]))
        exact += check_walk(int(np_(rd.accept_len)[q]), np_(rd.path_nodes)[q], np_(rd.out_tokens)[q], *oa,
                            sampled=temps[q] > 0)
    assert exact >= 30


@pytest.mark.parametrize("temperature", [0.0, 1.0])
def test_subset_head_rounds(head, temperature):
    """Rounds with a 65,536-token draft vocabulary (project page "Multi-Future
    Drafting", In a serving engine): the drafter's head is the subset's rows
    of W, its futures lie in the subset, and the walk verifies against the
    target's full 151,936-token rows.  Tables against the oracle on the
    subset rows (ids looked up), the tree bit-exact, the walk exact."""
    W, _ = head
    ids = synth.vocab_subset(151936, 65536, seed=64)
    Wsub = W[torch.from_numpy(ids.astype(np.int64))].contiguous()
    Wp = mfd.pack_lm_head(Wsub.cuda())
    ids_d = torch.from_numpy(ids).cuda()
    rd = mfd.Round(1, 8, 15, 16, 256, 151936, V_draft=65536)
    exact = 0
    for i in range(3):
        r = synth.round_inputs(W, 8, 15, 11, seed=700 + i, vocab=ids)
        assert np.isin(r.fut, ids).all()
        rd.status.zero_()
        rd.lmhead_topk_subset(r.h.cuda(), Wp, ids_d)
        rd.build_tree()
        torch.cuda.synchronize()
        assert int(rd.status.item()) == 0
        lp, tk = np_(rd.tk_logp), np_(rd.tk_tok)
        rows = np.arange(i, 120, 17)
        o_lp, o_idx, _ = oracle.lmhead_topk(_bits(r.h[rows]), _bits(Wsub), 16)
        check_topk(lp[rows], tk[rows], o_lp, ids[o_idx])
        g = tree_outputs(rd)
        o = oracle.build_tree(lp.reshape(8, 15, 16), tk.reshape(8, 15, 16), 256)
        assert_tree_equal(g, o, 0)
        noise = synth.target_noise(257, 151936, np.random.default_rng(r.seed % (2**32)))
        prow, pcol = synth.plant_sites(o["parent"], o["token"], o["depth"], int(o["n_nodes"]), r.fut[r.target_mode])
        t = synth.plant(noise, prow, pcol)
        rd.verify(torch.from_numpy(t[None]).cuda(), torch.tensor([temperature], device="cuda"),
                  torch.tensor([r.seed], dtype=torch.int64, device="cuda"))
        torch.cuda.synchronize()
        assert int(rd.status.item()) == 0
        oa = oracle.verify(t, o["parent"], o["token"], int(o["n_nodes"]), 15, temperature, r.seed)
        exact += check_walk(int(np_(rd.accept_len)[0]), np_(rd.path_nodes)[0], np_(rd.out_tokens)[0], *oa,
                            sampled=temperature > 0)
    assert exact >= 2


@pytest.mark.slow
def test_wide_shape_greedy_round():
    """The wider shape as a whole round: K=8, L=15, H=5120, V=248,320, 13 of
    15 positions shared, top-32, B=256, greedy, through the packed weight
    (about 2.5 GB streamed) -- tables on sampled rows against the oracle's
    full-vocabulary LM head, the tree bit-exact, the walk over the full
    248,320-entry target rows exact."""
    V, H = 248320, 5120
    W = synth.lm_head(V, H, seed=4048)
    Wd = W.cuda()
    Wp = mfd.pack_lm_head(Wd)
    del Wd
    rd = mfd.Round(1, 8, 15, 32, 256, V)
    for i in range(2):
        r = synth.round_inputs(W, 8, 15, 13, seed=9 + i)
        rd.status.zero_()
        rd.lmhead_topk_packed(r.h.cuda(), Wp)
        rd.build_tree()
        torch.cuda.synchronize()
        assert int(rd.status.item()) == 0
        lp, tk = np_(rd.tk_logp), np_(rd.tk_tok)
        rows = np.array([0, 17, 59, 119]) if i == 0 else np.array([5, 64])
        o_lp, o_tk, _ = oracle.lmhead_topk(_bits(r.h[rows]), _bits(W), 32)
        check_topk(lp[rows], tk[rows], o_lp, o_tk)
        g = tree_outputs(rd)
        o = oracle.build_tree(lp.reshape(8, 15, 32), tk.reshape(8, 15, 32), 256)
        assert_tree_equal(g, o, 0)
        noise = synth.target_noise(257, V, np.random.default_rng(r.seed % (2**32)))
        prow, pcol = synth.plant_sites(o["parent"], o["token"], o["depth"], int(o["n_nodes"]),
                                       r.fut[r.target_mode])
        t = synth.plant(noise, prow, pcol)
        rd.verify(torch.from_numpy(t[None]).cuda(), torch.zeros(1, device="cuda"),
                  torch.tensor([r.seed], dtype=torch.int64, device="cuda"))
        torch.cuda.synchronize()
        assert int(rd.status.item()) == 0
        oa = oracle.verify(t, o["parent"], o["token"], int(o["n_nodes"]), 15)
        assert check_walk(int(np_(rd.accept_len)[0]), np_(rd.path_nodes)[0], np_(rd.out_tokens)[0], *oa,
                          sampled=False)
        # the target's future is planted along the tree: the walk follows it
        assert int(np_(rd.accept_len)[0]) >= 1


def test_single_mode_batch_round(head):
    """MFD-D's single-mode path at full size (project page "Multi-Future
    Drafting", In a serving engine): 8 requests in flight, so K = 1
    (mfd_mfdd_modes), L=15, H=2560, V=151,936, top-16, B=64, through the
    packed weight; requests alternate greedy and T=1.  Tables on sampled rows
    against the oracle's LM head, every tree bit-exact (the product-ranked
    tree), every walk exact."""
    W, Wd = head
    n = 8
    K = mfd.mfd_mfdd_modes(n, 8)
    assert K == 1
    rounds = [synth.round_inputs(W, K, 15, 15, seed=900 + q) for q in range(n)]
    h = torch.cat([r.h for r in rounds], 0)
    Wp = mfd.pack_lm_head(Wd)
    rd = mfd.Round(n, K, 15, 16, 64, 151936)
    rd.status.zero_()
    rd.lmhead_topk_packed(h.cuda(), Wp)
    rd.build_tree()
    torch.cuda.synchronize()
    assert int(rd.status.item()) == 0
    lp, tk = np_(rd.tk_logp), np_(rd.tk_tok)
    rows = np.array([0, 14, 15, 59, 100, 119])
    o_lp, o_tk, _ = oracle.lmhead_topk(_bits(h[rows]), _bits(W), 16)
    check_topk(lp[rows], tk[rows], o_lp, o_tk)
    g = tree_outputs(rd)
    o = oracle.build_tree(lp.reshape(n, K, 15, 16), tk.reshape(n, K, 15, 16), 64)
    for q in range(n):
        assert_tree_equal(g, {k: v[q] for k, v in o.items()}, q)
    t = np.empty((n, 65, 151936), np.float32)
    for q in range(n):
        noise = synth.target_noise(65, 151936, np.random.default_rng(50 + q))
        rows_, cols_ = synth.plant_sites(o["parent"][q], o["token"][q], o["depth"][q], int(o["n_nodes"][q]),
                                         rounds[q].fut[0])
        t[q] = synth.plant(noise, rows_, cols_)
    temps = np.array([0.0, 1.0] * (n // 2), np.float32)
    seeds = np.array([r.seed for r in rounds], np.uint64)
    rd.verify(torch.from_numpy(t).cuda(), torch.from_numpy(temps).cuda(),
              torch.from_numpy(seeds.view(np.int64)).cuda())
    torch.cuda.synchronize()
    assert int(rd.status.item()) == 0
    exact = 0
    for q in range(n):
        oa = oracle.verify(t[q], o["parent"][q], o["token"][q], int(o["n_nodes"][q]), 15, float(temps[q]),
                           int(seeds[q]))
        exact += check_walk(int(np_(rd.accept_len)[q]), np_(rd.path_nodes)[q], np_(rd.out_tokens)[q], *oa,
                            sampled=temps[q] > 0)
    assert exact >= n - 1
    # greedy walks follow the planted future as deep as the tree holds it
    assert all(int(np_(rd.accept_len)[q]) >= 1 for q in range(0, n, 2))
