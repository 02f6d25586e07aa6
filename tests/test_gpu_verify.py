"""GPU parity: the tree verification walk against the oracle.  Greedy paths
are bit-exact; sampled paths are exact except from the first step whose
top-two perturbed scores (oracle) lie within 1e-5.  Model card "MFD drafter
for Qwen3.5-4B", first paragraph; project page, Figure 2 (c)."""
import numpy as np
import pytest
import torch

import oracle
from tree_verified_speculative_gb300 import mfd, synth

from gpu_helpers import check_walk, np_, status_of

pytestmark = pytest.mark.gpu


def _gpu_verify(t: np.ndarray, parent, token, n_nodes, L, temps, seeds):
    """t: [n_req, N, V]; parent/token [n_req, N]; n_nodes [n_req]."""
    n_req, N, V = t.shape
    rd = mfd.Round(n_req, 1, L, 1, N - 1, V)
    rd.parent.copy_(torch.from_numpy(np.asarray(parent, np.int32)))
    rd.token.copy_(torch.from_numpy(np.asarray(token, np.int32)))
    rd.n_nodes.copy_(torch.from_numpy(np.asarray(n_nodes, np.int32)))
    rd.status.zero_()
    temp = torch.tensor(np.asarray(temps, np.float32), device="cuda")
    seed = torch.tensor(np.asarray(seeds, np.uint64).view(np.int64), device="cuda")
    rd.verify(torch.from_numpy(t).cuda(), temp, seed)
    torch.cuda.synchronize()
    return np_(rd.accept_len), np_(rd.path_nodes), np_(rd.out_tokens), status_of(rd)


def _trees(rng, n_req, K, L, k, V, B):
    lp = np.empty((n_req, K, L, k), np.float32)
    tk = np.empty((n_req, K, L, k), np.int32)
    futs = []
    for q in range(n_req):
        fut = synth.futures(K, L, V, 11 if L >= 11 else 1, rng)
        futs.append(fut)
        for m in range(K):
            for i in range(L):
                others = [t for t in rng.choice(V, size=k + 4, replace=False) if t != fut[m, i]][: k - 1]
                toks = np.array([fut[m, i], *others])
                vals = np.concatenate([[-1.0], -3.0 + rng.normal(0, 0.5, size=k - 1)]).astype(np.float32)
                order = np.lexsort((toks, -vals))
                lp[q, m, i], tk[q, m, i] = vals[order], toks[order]
    return oracle.build_tree(lp, tk, B), futs


def _targets(rng, tree, futs, V, target_modes):
    n_req, N = tree["parent"].shape
    t = np.empty((n_req, N, V), np.float32)
    for q in range(n_req):
        noise = synth.target_noise(N, V, rng)
        rows, cols = synth.plant_sites(tree["parent"][q], tree["token"][q], tree["depth"][q],
                                       int(tree["n_nodes"][q]), futs[q][target_modes[q]])
        t[q] = synth.plant(noise, rows, cols)
    return t


def _compare(t, tree, L, temps, seeds):
    g_acc, g_path, g_out, st = _gpu_verify(t, tree["parent"], tree["token"], tree["n_nodes"], L, temps, seeds)
    assert st == 0
    exact = 0
    for q in range(t.shape[0]):
        o = oracle.verify(t[q], tree["parent"][q], tree["token"][q], int(tree["n_nodes"][q]), L, temps[q], seeds[q])
        exact += check_walk(int(g_acc[q]), g_path[q], g_out[q], *o, sampled=temps[q] > 0)
    return exact, g_acc


def test_hand_tree_greedy():
    parent = np.array([[-1, 0, 0, 1, 1]], np.int32)
    token = np.array([[0, 5, 7, 2, 8]], np.int32)
    t = np.zeros((1, 5, 40), np.float32)
    t[0, 0, 5] = 3.0
    t[0, 1, 2] = 1.0
    t[0, 3, 39] = 4.0
    acc, path, out, st = _gpu_verify(t, parent, token, [5], 3, [0.0], [0])
    assert st == 0 and acc[0] == 2
    assert list(path[0]) == [0, 1, 3, -1] and list(out[0]) == [5, 2, 39, -1]


@pytest.mark.parametrize("V", [50, 151936])
def test_greedy_planted(V):
    rng = np.random.default_rng(V)
    tree, futs = _trees(rng, 4, 8, 15, 16, 151936 if V > 1000 else V, 64)
    t = _targets(rng, tree, futs, V, [0, 3, 5, 7])
    exact, acc = _compare(t, tree, 15, [0.0] * 4, [0] * 4)
    assert exact == 4


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_sampled(T):
    rng = np.random.default_rng(int(T * 10))
    tree, futs = _trees(rng, 6, 8, 15, 16, 151936, 256)
    t = _targets(rng, tree, futs, 151936, [1, 2, 3, 4, 5, 6])
    seeds = [int(x) for x in rng.integers(0, 2**63 - 1, size=6)]
    exact, _ = _compare(t, tree, 15, [T] * 6, seeds)
    assert exact >= 5


def test_sampled_small_vocab_many_seeds():
    """V = 64: many draws per node; decisions agree with the oracle."""
    rng = np.random.default_rng(3)
    tree, futs = _trees(rng, 1, 4, 6, 8, 64, 40)
    t = _targets(rng, tree, futs, 64, [2])
    t = np.repeat(t, 64, axis=0)
    tree64 = {k: np.repeat(v, 64, axis=0) for k, v in tree.items()}
    seeds = list(range(1000, 1064))
    exact, _ = _compare(t, tree64, 6, [1.0] * 64, seeds)
    assert exact >= 60


def test_mixed_batch_32():
    rng = np.random.default_rng(32)
    tree, futs = _trees(rng, 32, 8, 15, 16, 151936, 128)
    modes = rng.integers(0, 8, size=32)
    t = _targets(rng, tree, futs, 151936, modes)
    temps = [0.0] * 16 + [1.0] * 16
    seeds = [int(x) for x in rng.integers(0, 2**63 - 1, size=32)]
    exact, _ = _compare(t, tree, 15, temps, seeds)
    assert exact >= 30


@pytest.mark.parametrize("V", [151936, 20000, 1000])
def test_cluster_walk_equals_grid_walk(V):
    """From 8 requests a round is walked by one thread-block cluster per
    request, below that by the cooperative grid.  Eight requests walked in one
    call (clusters) and each walked alone (grid) give the same walks, bit for
    bit, greedy and sampled (T = 1 and 0.7), and the oracle's on the greedy
    ones."""
    rng = np.random.default_rng(V)
    n = 8
    tree, futs = _trees(rng, n, 4, 15, 8, V, 96)
    t = _targets(rng, tree, futs, V, rng.integers(0, 4, size=n))
    temps = [0.0, 1.0, 0.7, 0.0, 1.0, 0.0, 0.7, 1.0]
    seeds = [int(x) for x in rng.integers(0, 2**63 - 1, size=n)]
    b_acc, b_path, b_out, st = _gpu_verify(t, tree["parent"], tree["token"], tree["n_nodes"], 15, temps, seeds)
    assert st == 0
    for q in range(n):
        a_acc, a_path, a_out, st = _gpu_verify(t[q:q + 1], tree["parent"][q:q + 1], tree["token"][q:q + 1],
                                               tree["n_nodes"][q:q + 1], 15, temps[q:q + 1], seeds[q:q + 1])
        assert st == 0
        assert int(a_acc[0]) == int(b_acc[q])
        np.testing.assert_array_equal(a_path[0], b_path[q])
        np.testing.assert_array_equal(a_out[0], b_out[q])
        if temps[q] == 0.0:
            o = oracle.verify(t[q], tree["parent"][q], tree["token"][q], int(tree["n_nodes"][q]), 15, 0.0, seeds[q])
            assert check_walk(int(b_acc[q]), b_path[q], b_out[q], *o, sampled=False)


def test_rejects_bad_temperature():
    parent = np.array([[-1, 0]], np.int32)
    token = np.array([[0, 1]], np.int32)
    t = np.zeros((1, 2, 16), np.float32)
    _, _, _, st = _gpu_verify(t, parent, token, [2], 2, [-1.0], [0])
    assert st == mfd.MFD_ERR_INPUT


def test_workspace_reuse_and_graph_replay():
    """The walk's exchange words need no zeroing between calls: the same
    workspace is reused after other writers (zeros, a byte pattern, random
    bytes, another call's scratch) and under CUDA-graph replay, with long
    greedy walks (many steps, so both parities of every word are reused)."""
    rng = np.random.default_rng(77)
    V = 151936
    tree, futs = _trees(rng, 2, 8, 15, 16, V, 128)
    t = _targets(rng, tree, futs, V, [4, 6])
    n_req, N = tree["parent"].shape
    ref = [oracle.verify(t[q], tree["parent"][q], tree["token"][q], int(tree["n_nodes"][q]), 15, 0.0, 0)
           for q in range(n_req)]
    assert max(int(r[0]) for r in ref) >= 3  # the walks are long
    rd = mfd.Round(n_req, 1, 15, 1, N - 1, V)
    rd.parent.copy_(torch.from_numpy(tree["parent"]))
    rd.token.copy_(torch.from_numpy(tree["token"]))
    rd.n_nodes.copy_(torch.from_numpy(tree["n_nodes"].astype(np.int32)))
    rd.status.zero_()
    td = torch.from_numpy(t).cuda()
    temp = torch.zeros(n_req, device="cuda")
    seed = torch.zeros(n_req, dtype=torch.int64, device="cuda")

    def check():
        torch.cuda.synchronize()
        assert status_of(rd) == 0
        acc, path, out = np_(rd.accept_len), np_(rd.path_nodes), np_(rd.out_tokens)
        for q in range(n_req):
            assert check_walk(int(acc[q]), path[q], out[q], *ref[q], sampled=False)
        rd.accept_len.fill_(-7)
        rd.path_nodes.fill_(-7)
        rd.out_tokens.fill_(-7)

    fills = [lambda: None, lambda: rd.ws.zero_(), lambda: rd.ws.fill_(1), lambda: rd.ws.fill_(0xFF),
             lambda: rd.ws.copy_(torch.randint(0, 256, rd.ws.shape, dtype=torch.uint8, device="cuda"))]
    for fill in fills:
        fill()
        rd.verify(td, temp, seed)
        check()
        rd.verify(td, temp, seed)  # right after a call: the previous call's words are in place
        check()
    # another op's scratch in between (top-k partials written into the same workspace)
    logits = torch.randn((4, 4096), device="cuda")
    tl = torch.empty((4, 8), device="cuda")
    tt = torch.empty((4, 8), dtype=torch.int32, device="cuda")
    mfd.mfd_logits_topk(logits, 8, tl, tt, None, rd.status, rd.ws)
    rd.verify(td, temp, seed)
    check()
    # graph capture and replay: identical launch parameters every replay
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        rd.verify(td, temp, seed)
    torch.cuda.current_stream().wait_stream(s)
    check()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rd.verify(td, temp, seed)
    for _ in range(4):
        g.replay()
        check()


def test_target_logits_in_pinned_host_memory():
    """Target logits left in page-locked host memory are read in place (only
    the rows on the walk cross the host link): the walks are the oracle's,
    bit for bit those of device-resident logits; pageable host memory is
    refused before any launch."""
    import ctypes

    rng = np.random.default_rng(77)
    tree, futs = _trees(rng, 4, 8, 15, 16, 151936, 64)
    t = _targets(rng, tree, futs, 151936, [0, 2, 4, 6])
    temps, seeds = [0.0, 0.0, 1.0, 1.0], [5, 6, 7, 8]
    n_req, N, V = t.shape
    rd = mfd.Round(n_req, 1, 15, 1, N - 1, V)
    rd.parent.copy_(torch.from_numpy(tree["parent"]))
    rd.token.copy_(torch.from_numpy(tree["token"]))
    rd.n_nodes.copy_(torch.from_numpy(tree["n_nodes"]))
    temp = torch.tensor(np.asarray(temps, np.float32), device="cuda")
    seed = torch.tensor(np.asarray(seeds, np.uint64).view(np.int64), device="cuda")
    outs = []
    for where in ("device", "pinned"):
        tt = torch.from_numpy(t).cuda() if where == "device" else torch.from_numpy(t).pin_memory()
        rd.status.zero_()
        rd.verify(tt, temp, seed)
        torch.cuda.synchronize()
        assert status_of(rd) == 0
        outs.append((np_(rd.accept_len), np_(rd.path_nodes), np_(rd.out_tokens)))
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)
    exact = 0
    for q in range(n_req):
        o = oracle.verify(t[q], tree["parent"][q], tree["token"][q], int(tree["n_nodes"][q]), 15, temps[q], seeds[q])
        exact += check_walk(int(outs[1][0][q]), outs[1][1][q], outs[1][2][q], *o, sampled=temps[q] > 0)
    assert exact >= 3
    pageable = np.ascontiguousarray(t)
    lib = mfd.load()
    rc = lib.mfd_verify(ctypes.c_void_p(pageable.ctypes.data), n_req, N - 1, V, 15, rd.parent.data_ptr(),
                        rd.token.data_ptr(), rd.n_nodes.data_ptr(), temp.data_ptr(), seed.data_ptr(),
                        rd.accept_len.data_ptr(), rd.path_nodes.data_ptr(), rd.out_tokens.data_ptr(),
                        rd.status.data_ptr(), rd.ws.data_ptr(), rd.ws.numel(), None)
    assert rc == mfd.MFD_ERR_INVALID_ARG


def test_sampled_coverage_identity():
    """Over many seeds the GPU's sampled walks accept, on average, the tree's
    covered target mass (project page, How it works, step 1: the accepted
    length is the probability mass the tree covers):
    E = sum over nodes of the product of softmax(t / T) along the path."""
    rng = np.random.default_rng(21)
    parent = np.array([-1, 0, 0, 1, 1, 2, 3, 3, 6], np.int32)
    token = np.array([0, 1, 3, 0, 2, 4, 1, 3, 2], np.int32)
    N, V, L, T, n_req = 9, 4096, 3, 1.0, 2048
    t = rng.normal(0, 1.0, size=(N, V)).astype(np.float32)
    for n in range(1, N):
        t[parent[n], token[n]] += 7.0  # the tree's tokens carry real mass
    p = np.exp(t.astype(np.float64) / T)
    p /= p.sum(axis=1, keepdims=True)
    reach = np.zeros(N)
    reach[0] = 1.0
    for n in range(1, N):
        reach[n] = reach[parent[n]] * p[parent[n], token[n]]
    expect = reach[1:].sum()
    acc, _, _, st = _gpu_verify(np.tile(t, (n_req, 1, 1)), np.tile(parent, (n_req, 1)), np.tile(token, (n_req, 1)),
                                [N] * n_req, L, [T] * n_req, [s * 7919 + 3 for s in range(n_req)])
    assert st == 0
    se = acc.std() / np.sqrt(n_req)
    assert 0.3 < expect < 2.5
    assert abs(acc.mean() - expect) < 4 * se, (acc.mean(), expect, se)


def test_bounded_wait_runs_out_and_workspace_recovers():
    """The walk's exchange waits are bounded: with the other CTAs' step
    results withheld (the library's fault-injection entry point) and a 200 us
    limit, every CTA gives up, the call ends with MFD_ERR_TIMEOUT instead of
    hanging, and the next ordinary call on the same workspace is exact."""
    rng = np.random.default_rng(23)
    V, L, B = 20000, 6, 15
    tree, futs = _trees(rng, 2, 2, L, 4, V, B)
    t = _targets(rng, tree, futs, V, [0, 1])
    rd = mfd.Round(2, 1, L, 1, B, V)
    rd.parent.copy_(torch.from_numpy(tree["parent"]))
    rd.token.copy_(torch.from_numpy(tree["token"]))
    rd.n_nodes.copy_(torch.from_numpy(tree["n_nodes"]))
    td = torch.from_numpy(t).cuda()
    temp = torch.zeros(2, device="cuda")
    seed = torch.zeros(2, dtype=torch.int64, device="cuda")
    for attempt in range(2):
        rd.status.zero_()
        mfd.mfd_verify_withheld_test(td, 2, B, V, L, rd.parent, rd.token, rd.n_nodes, temp, seed, rd.accept_len,
                                     rd.path_nodes, rd.out_tokens, rd.status, rd.ws, 200_000)
        torch.cuda.synchronize()
        assert status_of(rd) == mfd.MFD_ERR_TIMEOUT
        rd.status.zero_()
        rd.verify(td, temp, seed)
        torch.cuda.synchronize()
        assert status_of(rd) == 0
        for q in range(2):
            o = oracle.verify(t[q], tree["parent"][q], tree["token"][q], int(tree["n_nodes"][q]), L)
            assert check_walk(int(np_(rd.accept_len)[q]), np_(rd.path_nodes)[q], np_(rd.out_tokens)[q], *o,
                              sampled=False)
    with pytest.raises(mfd.MfdError) as e:
        mfd.mfd_verify_withheld_test(td, 2, B, V, L, rd.parent, rd.token, rd.n_nodes, temp, seed, rd.accept_len,
                                     rd.path_nodes, rd.out_tokens, rd.status, rd.ws, 10)
    assert e.value.code == mfd.MFD_ERR_INVALID_ARG
