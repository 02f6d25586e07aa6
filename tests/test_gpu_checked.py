"""The bounds-checked build (libmfd_checked.so, the sources compiled with
-DMFD_CHECKED): every shared-memory index the tree builder computes from data
is range-checked, clamped into its array if it is out of range, and reported
as MFD_ERR_CHECK.  It stands in for a memory checker on the GPU.  These tests
run the tiny, tie-heavy, deep and limit cases through it and require a clean
status and the oracle's trees, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from tree_verified_speculative_gb300 import mfd, synth

from gpu_helpers import assert_tree_equal, check_topk, check_walk, gpu_tree, np_
from test_gpu_tree import _planted_tables, _random_tables

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def checked_library():
    mfd.use_library(mfd.CHECKED_LIB_PATH)
    yield
    mfd.use_library(None)


def _compare(lp, tk, B):
    g, st = gpu_tree(lp, tk, B)
    assert st == 0, mfd.status_string(st)
    o = oracle.build_tree(lp, tk, B)
    for q in range(lp.shape[0]):
        assert_tree_equal(g, {k: v[q] for k, v in o.items()}, q)
    return g


def test_checked_library_is_the_one_called():
    assert mfd.load() is mfd.load(mfd.CHECKED_LIB_PATH)
    assert mfd.status_string(mfd.MFD_ERR_CHECK).startswith("bounds-checked build")


def test_checked_tiny_round():
    c = synth.tiny(seed=1)
    rd = mfd.Round(1, c.K, c.L, c.topk, c.B, c.V)
    rd.status.zero_()
    rd.logits_topk(torch.from_numpy(c.logits).cuda())
    rd.build_tree()
    torch.cuda.synchronize()
    assert int(rd.status.item()) == 0
    lp, tk = np_(rd.tk_logp), np_(rd.tk_tok)
    o_lp, o_tk, _ = oracle.logits_topk(c.logits, c.topk)
    check_topk(lp, tk, o_lp, o_tk)
    o = oracle.build_tree(lp.reshape(c.K, c.L, c.topk), tk.reshape(c.K, c.L, c.topk), c.B)
    from gpu_helpers import tree_outputs
    assert_tree_equal(tree_outputs(rd), o, 0)
    noise = synth.target_noise(c.B + 1, c.V, np.random.default_rng(5))
    rows, cols = synth.plant_sites(o["parent"], o["token"], o["depth"], int(o["n_nodes"]), c.fut[1])
    t = synth.plant(noise, rows, cols)
    rd.verify(torch.from_numpy(t[None]).cuda(), torch.zeros(1, device="cuda"),
              torch.zeros(1, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert int(rd.status.item()) == 0
    oa = oracle.verify(t, o["parent"], o["token"], int(o["n_nodes"]), c.L)
    assert check_walk(int(np_(rd.accept_len)[0]), np_(rd.path_nodes)[0], np_(rd.out_tokens)[0], *oa, sampled=False)


@pytest.mark.parametrize("seed", range(6))
def test_checked_tie_heavy(seed):
    rng = np.random.default_rng(300 + seed)
    K, L, k = int(rng.integers(1, 6)), int(rng.integers(1, 9)), int(rng.integers(2, 17))
    lp, tk = _random_tables(rng, 2, K, L, k, 40, values=np.array([-1.0, -2.0, -2.0, -3.5], np.float32))
    _compare(lp, tk, int(rng.integers(1, 80)))


def test_checked_pages_shape_and_deep():
    rng = np.random.default_rng(8)
    lp, tk = _planted_tables(rng, 2, 8, 15, 16, 151936, 11)
    _compare(lp, tk, 256)
    lp[..., 0] = -0.01 * (1 + rng.random(lp[..., 0].shape)).astype(np.float32)
    g = _compare(lp, tk, 256)
    assert g["depth"].max() == 15


def test_checked_limits():
    rng = np.random.default_rng(9)
    lp, tk = _random_tables(rng, 1, 16, 16, 32, 100000)
    _compare(lp, tk, 128)
    lp, tk = _random_tables(rng, 1, 4, 16, 32, 100000)
    _compare(lp, tk, 512)
    K, L, k = 16, 16, 32
    tk = np.empty((1, K, L, k), np.int32)
    for i in range(L):
        row = np.sort(rng.choice(1000, size=k, replace=False))
        tk[0, :, i] = row
    for value in (0.0, -1.0):
        g = _compare(np.full((1, K, L, k), value, np.float32), tk, 128)
        if value == 0.0:
            assert g["depth"].max() == L
