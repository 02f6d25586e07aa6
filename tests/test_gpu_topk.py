"""GPU parity: LM head + log-softmax + top-k, and top-k of given logits,
against the CPU oracle (log-probs within 1e-4; top-k sets equal except at the
cut).  Model card "MFD drafter for Qwen3.5-4B", Model table; project page
"Multi-Future Drafting", How it works, step 2."""
import numpy as np
import pytest
import torch

import oracle
from tree_verified_speculative_gb300 import mfd, synth

from gpu_helpers import check_topk, np_, status_of

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _gpu_logits_topk(z: np.ndarray, topk: int):
    R, V = z.shape
    rd = mfd.Round(1, 1, R, topk, 1, V)
    rd.status.zero_()
    rd.logits_topk(torch.from_numpy(z).cuda())
    torch.cuda.synchronize()
    assert status_of(rd) == 0
    return np_(rd.tk_logp), np_(rd.tk_tok), np_(rd.lse)


def _gpu_lmhead(h: torch.Tensor, W: torch.Tensor, topk: int, Wd=None):
    R = h.shape[0]
    V = W.shape[0]
    rd = mfd.Round(1, 1, R, topk, 1, V)
    rd.status.zero_()
    rd.lmhead_topk(h.cuda(), W.cuda() if Wd is None else Wd)
    torch.cuda.synchronize()
    assert status_of(rd) == 0
    return np_(rd.tk_logp), np_(rd.tk_tok), np_(rd.lse)


def test_tiny_case_logits_topk():
    c = synth.tiny(seed=1)
    for topk in (8, 32):
        g = _gpu_logits_topk(c.logits, topk)
        o = oracle.logits_topk(c.logits, topk)
        check_topk(g[0], g[1], o[0], o[1])
        np.testing.assert_allclose(g[2], o[2], atol=1e-5)


@pytest.mark.parametrize("R,V,topk", [(1, 16, 1), (3, 1000, 8), (7, 5003, 16), (5, 70001, 32), (130, 2049, 16)])
def test_logits_topk_random(R, V, topk):
    rng = np.random.default_rng(R * 1000 + V)
    z = (2.0 * rng.standard_normal((R, V))).astype(np.float32)
    g = _gpu_logits_topk(z, topk)
    o = oracle.logits_topk(z, topk)
    check_topk(g[0], g[1], o[0], o[1])
    np.testing.assert_allclose(g[2], o[2], atol=1e-5)


def test_logits_topk_ties():
    rng = np.random.default_rng(4)
    z = rng.choice(np.array([-1.0, 0.5, 2.0, 2.0, 3.0], np.float32), size=(6, 3000)).astype(np.float32)
    g = _gpu_logits_topk(z, 16)
    o = oracle.logits_topk(z, 16)
    # ties resolve to the smaller token id on both sides
    np.testing.assert_array_equal(g[1], o[1])
    np.testing.assert_allclose(g[0], o[0], atol=1e-6)


@pytest.mark.parametrize("R,H,V,topk", [
    (1, 64, 16, 1), (5, 64, 300, 8), (120, 128, 1000, 16), (128, 256, 4099, 32), (130, 64, 2305, 16),
    (257, 192, 777, 8), (120, 2560, 20000, 16),
    # vocabularies that give every SM a 256-row tile, with one residue class
    # of the row bound (top-1), a top-k below its list width (5 of 8) and
    # the widest list (32)
    (64, 128, 40000, 1), (7, 256, 39000, 5), (128, 128, 50001, 32)])
def test_lmhead_topk_small(R, H, V, topk):
    rng = np.random.default_rng(R + H + V)
    h = synth.bf16_round(rng.standard_normal((R, H)).astype(np.float32))
    W = synth.bf16_round((rng.standard_normal((V, H)) / np.sqrt(H)).astype(np.float32))
    g = _gpu_lmhead(h, W, topk)
    o = oracle.lmhead_topk(_bits(h), _bits(W), topk)
    check_topk(g[0], g[1], o[0], o[1])
    np.testing.assert_allclose(g[2], o[2], atol=5e-5)


@pytest.fixture(scope="module")
def head_2560():
    W = synth.lm_head(151936, 2560, seed=2024)
    return W, W.cuda()


@pytest.mark.parametrize("R", [1, 15, 25])
def test_staged_hidden_rows_match_unstaged(head_2560, R):
    """Hidden rows that span 144 KB or less (here 1, 15 and 25 rows of 5 KB)
    are read from a zero-padded copy in the workspace; 40 rows (200 KB) are
    read in place.  The same rows give bit-identical tables either way, on
    the row-major and the packed weight: each MMA row is independent."""
    W, Wd = head_2560
    h = synth.round_inputs(W, 8, 15, 11, seed=70).h[:40]
    Wp = mfd.pack_lm_head(Wd)
    for packed in (False, True):
        out = []
        for rows in (R, 40):
            rd = mfd.Round(1, 1, rows, 16, 1, 151936)
            rd.status.zero_()
            hd = h[:rows].contiguous().cuda()
            if packed:
                rd.lmhead_topk_packed(hd, Wp)
            else:
                rd.lmhead_topk(hd, Wd)
            torch.cuda.synchronize()
            assert status_of(rd) == 0
            out.append((np_(rd.tk_tok)[:R], np_(rd.tk_logp)[:R].view(np.uint32), np_(rd.lse)[:R].view(np.uint32)))
        for a, b in zip(*out):
            np.testing.assert_array_equal(a, b)


def test_lmhead_bounded_wait_runs_out_and_next_call_is_exact(head_2560):
    """The LM head's pipeline waits are bounded: with the producers stopped
    after each CTA's first tile (the library's fault-injection entry point),
    the MMA warp's wait runs out, the call ends with MFD_ERR_TIMEOUT instead
    of hanging, every CTA returns (the stream synchronises), and the next
    ordinary call on the same buffers gives the earlier results bit for bit."""
    W, Wd = head_2560
    Wp = mfd.pack_lm_head(Wd)
    h = synth.round_inputs(W, 8, 15, 11, seed=72).h.cuda()
    rd = mfd.Round(1, 8, 15, 16, 1, 151936)
    rd.status.zero_()
    rd.lmhead_topk_packed(h, Wp)
    torch.cuda.synchronize()
    assert status_of(rd) == 0
    ref = (np_(rd.tk_tok).copy(), np_(rd.tk_logp).view(np.uint32).copy(), np_(rd.lse).view(np.uint32).copy())
    for attempt in range(2):
        rd.status.zero_()
        mfd.mfd_lmhead_withheld_test(h, Wp, 151936, 16, rd.tk_logp, rd.tk_tok, rd.lse, rd.status, rd.ws)
        torch.cuda.synchronize()
        assert status_of(rd) == mfd.MFD_ERR_TIMEOUT
        rd.status.zero_()
        rd.lmhead_topk_packed(h, Wp)
        torch.cuda.synchronize()
        assert status_of(rd) == 0
        np.testing.assert_array_equal(np_(rd.tk_tok), ref[0])
        np.testing.assert_array_equal(np_(rd.tk_logp).view(np.uint32), ref[1])
        np.testing.assert_array_equal(np_(rd.lse).view(np.uint32), ref[2])


def test_lmhead_pages_shape_sampled_rows(head_2560):
    """K=8, L=15, H=2560, V=151936, top-k 16, planted futures (11 of 15
    shared): all 120 rows through the kernel, 24 of them checked against the
    oracle's full-vocabulary row."""
    W, Wd = head_2560
    r = synth.round_inputs(W, 8, 15, 11, seed=7)
    g = _gpu_lmhead(r.h, W, 16, Wd)
    rows = np.random.default_rng(0).choice(120, size=24, replace=False)
    o = oracle.lmhead_topk(_bits(r.h[rows]), _bits(W), 16)
    check_topk(g[0][rows], g[1][rows], o[0], o[1])
    np.testing.assert_allclose(g[2][rows], o[2], atol=5e-5)
    # every row is a distribution: the planted token is the usual argmax
    assert np.mean(g[1][:, 0] == r.fut.reshape(-1)) > 0.5


def test_lmhead_batched_3840_rows_sampled(head_2560):
    """32 requests x 8 modes x 15 positions = 3840 rows (30 M tiles)."""
    W, Wd = head_2560
    hs = [synth.round_inputs(W, 8, 15, 8 + (q % 7), seed=100 + q).h for q in range(32)]
    h = torch.cat(hs, 0)
    g = _gpu_lmhead(h, W, 16, Wd)
    rows = np.array([0, 127, 128, 1000, 1919, 2047, 3000, 3839])
    o = oracle.lmhead_topk(_bits(h[rows]), _bits(W), 16)
    check_topk(g[0][rows], g[1][rows], o[0], o[1])


def test_lmhead_rejects_bad_arguments():
    h = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda")  # H not a multiple of 64
    W = torch.zeros((64, 100), dtype=torch.bfloat16, device="cuda")
    rd = mfd.Round(1, 1, 4, 8, 1, 64)
    with pytest.raises(mfd.MfdError) as e:
        rd.lmhead_topk(h, W)
    assert e.value.code == mfd.MFD_ERR_UNSUPPORTED


def _expected_packed(W: np.ndarray) -> np.ndarray:
    """The packed layout written out plainly (uint16 view of bf16): per
    256-row tile and 64-element K slice a block of 256 rows x 64 elements,
    row r's 16-byte chunk j stored at chunk position j ^ (r % 8); rows past V
    zero."""
    V, H = W.shape
    nt, nk = -(-V // 256), H // 64
    Wpad = np.zeros((nt * 256, H), np.uint16)
    Wpad[:V] = W
    out = np.empty((nt, nk, 256, 8, 8), np.uint16)  # tile, slice, row, chunk position, element
    for r in range(256):
        for pos in range(8):
            j = pos ^ (r % 8)
            out[:, :, r, pos, :] = Wpad.reshape(nt, 256, nk, 8, 8)[:, r, :, j, :]
    return out.reshape(-1)


def test_pack_layout():
    rng = np.random.default_rng(5)
    V, H = 300, 128
    W = torch.from_numpy(rng.standard_normal((V, H)).astype(np.float32)).to(torch.bfloat16)
    Wp = mfd.pack_lm_head(W.cuda())
    torch.cuda.synchronize()
    assert Wp.numel() == mfd.mfd_lmhead_packed_bytes(V, H) == 2 * 256 * H * 2
    got = Wp.cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(got, _expected_packed(_bits(W).reshape(V, H)))


@pytest.mark.parametrize("R,H,V,topk", [(120, 2560, 151936, 16), (37, 128, 1000, 8), (200, 256, 4099, 32),
                                        (1, 64, 16, 1), (300, 128, 5000, 16), (3840, 2560, 151936, 16)])
def test_packed_weight_bit_identical(R, H, V, topk):
    """mfd_lmhead_topk_packed gives exactly mfd_lmhead_topk's results, at one
    M tile and at several (300 rows: three M tiles, the last one ragged;
    3840: 32 requests of 120 rows)."""
    rng = np.random.default_rng(R + H + V)
    if V == 151936:
        W = synth.lm_head(V, H, seed=2024)
        h = torch.cat([synth.round_inputs(W, 8, 15, 11, seed=3 + q).h for q in range(R // 120)], 0)
    else:
        W = torch.from_numpy((rng.standard_normal((V, H)) / np.sqrt(H)).astype(np.float32)).to(torch.bfloat16)
        h = torch.from_numpy(rng.standard_normal((R, H)).astype(np.float32)).to(torch.bfloat16)
    Wd, hd = W.cuda(), h.cuda()
    a = mfd.Round(1, 1, R, topk, 1, V)
    b = mfd.Round(1, 1, R, topk, 1, V)
    a.status.zero_()
    b.status.zero_()
    a.lmhead_topk(hd, Wd)
    Wp = mfd.pack_lm_head(Wd)
    b.lmhead_topk_packed(hd, Wp)
    torch.cuda.synchronize()
    assert status_of(a) == 0 and status_of(b) == 0
    np.testing.assert_array_equal(np_(a.tk_tok), np_(b.tk_tok))
    np.testing.assert_array_equal(np_(a.tk_logp).view(np.uint32), np_(b.tk_logp).view(np.uint32))
    np.testing.assert_array_equal(np_(a.lse).view(np.uint32), np_(b.lse).view(np.uint32))


@pytest.mark.parametrize("R", [120, 300])
def test_subset_head(R):
    """Draft-vocabulary subset head (project page "Multi-Future Drafting", In
    a serving engine): the LM head, log-softmax and top-k over the subset's
    rows, with tokens written as vocabulary ids.  Exactly the packed head on
    the subset rows with the ids looked up, and the oracle's top-k on sampled
    rows.  300 rows span three M tiles."""
    rng = np.random.default_rng(R + 7)
    V_full, H, n_sub, topk = 20000, 256, 4096, 16
    ids = synth.vocab_subset(V_full, n_sub, seed=R)
    assert np.all(np.diff(ids) > 0)
    W = torch.from_numpy((rng.standard_normal((V_full, H)) / np.sqrt(H)).astype(np.float32)).to(torch.bfloat16)
    Wsub = W[torch.from_numpy(ids.astype(np.int64))].contiguous()
    h = torch.from_numpy(rng.standard_normal((R, H)).astype(np.float32)).to(torch.bfloat16)
    Wp = mfd.pack_lm_head(Wsub.cuda())
    a = mfd.Round(1, 1, R, topk, 1, V_full, V_draft=n_sub)
    b = mfd.Round(1, 1, R, topk, 1, n_sub)
    a.status.zero_()
    b.status.zero_()
    a.lmhead_topk_subset(h.cuda(), Wp, torch.from_numpy(ids).cuda())
    b.lmhead_topk_packed(h.cuda(), Wp)
    torch.cuda.synchronize()
    assert status_of(a) == 0 and status_of(b) == 0
    np.testing.assert_array_equal(np_(a.tk_tok), ids[np_(b.tk_tok)])
    np.testing.assert_array_equal(np_(a.tk_logp).view(np.uint32), np_(b.tk_logp).view(np.uint32))
    np.testing.assert_array_equal(np_(a.lse).view(np.uint32), np_(b.lse).view(np.uint32))
    rows = np.array([0, 1, R // 2, R - 1])
    o_lp, o_idx, _ = oracle.lmhead_topk(_bits(h[rows]), _bits(Wsub), topk)
    check_topk(np_(a.tk_logp)[rows], np_(a.tk_tok)[rows], o_lp, ids[o_idx])


def test_subset_head_rejects_ids_out_of_range():
    """A vocabulary id at or past V_full sets MFD_ERR_INPUT and is written as -1."""
    rng = np.random.default_rng(3)
    V_full, H, n_sub, topk = 5000, 128, 1024, 8
    ids = synth.vocab_subset(V_full, n_sub, seed=4) + V_full  # every id out of range
    W = torch.from_numpy((rng.standard_normal((n_sub, H)) / np.sqrt(H)).astype(np.float32)).to(torch.bfloat16)
    h = torch.from_numpy(rng.standard_normal((16, H)).astype(np.float32)).to(torch.bfloat16)
    a = mfd.Round(1, 1, 16, topk, 1, V_full, V_draft=n_sub)
    a.status.zero_()
    a.lmhead_topk_subset(h.cuda(), mfd.pack_lm_head(W.cuda()), torch.from_numpy(ids.astype(np.int32)).cuda())
    torch.cuda.synchronize()
    assert status_of(a) == mfd.MFD_ERR_INPUT
    assert np.all(np_(a.tk_tok) == -1)


def _tile(V: int) -> int:
    """Vocabulary rows of one LM-head tile at one M tile: 256, or 128 when
    256-row tiles would leave SMs without one (the library's rule)."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    return 256 if -(-V // 256) >= n_sm else 128


def _ranges(V: int, tile: int) -> list[tuple[int, int]]:
    """The LM head's vocabulary ranges at one M tile, as spans [t0, t1) of
    tiles: min(tiles, SMs) contiguous ranges, or, when at most three quarters
    of those would hold the largest share, the fewest ranges with the same
    largest share (the split the library's host code plans for R <= 128
    rows)."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    n_vt = -(-V // tile)
    P = min(n_vt, n_sm, 256)
    most = -(-n_vt // P)
    if 4 * (n_vt - (most - 1) * P) <= 3 * P:
        P = -(-n_vt // most)  # the fewest ranges with the same largest range
    return [(r * n_vt // P, (r + 1) * n_vt // P) for r in range(P)]


@pytest.mark.parametrize("packed", [False, True])
def test_lmhead_ties_duplicate_rows(packed):
    """Equal logits must come out in increasing token-id order, and a tie
    across the cut must keep the smallest ids (model card "MFD drafter for
    Qwen3.5-4B", first paragraph: the B best prefixes, ties to the smaller
    ids; project page, How it works, step 3).  Groups of identical weight
    rows give exactly equal logits on both sides: (i) inside one range's
    first 32 columns (the sorted first chunk), (ii) in different tiles of
    one range, (iii) in different vocabulary ranges, and (iv) six
    copies across ranges with top-4, so the cut falls inside the tie.  Each
    hidden row points at one group, whose members are then its best
    logits."""
    V, H, topk = 51200, 128, 4
    rng = np.random.default_rng(31)
    TILE = _tile(V)
    ranges = _ranges(V, TILE)
    rg = lambda i: ranges[i * len(ranges) // 152]  # noqa: E731  (a range by its place among 152)
    two = [r_ for r_ in ranges if r_[1] - r_[0] >= 2]
    assert two, "expected a range with two tiles"
    t2 = two[len(two) // 2]
    groups = [
        [rg(5)[0] * TILE + 3, rg(5)[0] * TILE + 17, rg(5)[0] * TILE + 30],
        [t2[0] * TILE + 100, (t2[0] + 1) * TILE + 7],
        [ranges[0][0] * TILE + 120, rg(40)[0] * TILE + 5, rg(100)[0] * TILE + 127, ranges[-1][0] * TILE + 1],
        [rg(i)[0] * TILE + 11 * i % TILE for i in (2, 30, 31, 77, 120, 151)],
    ]
    members = [v for g in groups for v in g]
    assert len(set(members)) == len(members) and max(members) < V
    Wf = (rng.standard_normal((V, H)) / np.sqrt(H)).astype(np.float32)
    for g in groups:
        for v in g[1:]:
            Wf[v] = Wf[g[0]]
    W = synth.bf16_round(Wf)
    Wr = W.float().numpy()
    hrows = []
    for g in groups:
        for rep in range(2):  # two hidden rows per group
            u = Wr[g[0]] / np.linalg.norm(Wr[g[0]])
            hrows.append(8.0 * u + 0.3 * rng.standard_normal(H))
    h = synth.bf16_round(np.asarray(hrows, np.float32))
    R = h.shape[0]
    rd = mfd.Round(1, 1, R, topk, 1, V)
    rd.status.zero_()
    if packed:
        rd.lmhead_topk_packed(h.cuda(), mfd.pack_lm_head(W.cuda()))
    else:
        rd.lmhead_topk(h.cuda(), W.cuda())
    torch.cuda.synchronize()
    assert status_of(rd) == 0
    g_lp, g_tok = np_(rd.tk_logp), np_(rd.tk_tok)
    o_lp, o_tok, _ = oracle.lmhead_topk(_bits(h), _bits(W), topk)
    check_topk(g_lp, g_tok, o_lp, o_tok)
    for gi, g in enumerate(groups):
        want = sorted(g)[:topk]
        for r in (2 * gi, 2 * gi + 1):
            # the group members are the row's best logits, tied exactly
            assert list(o_tok[r, :len(want)]) == want, (gi, r, o_tok[r])
            assert list(g_tok[r, :len(want)]) == want, (gi, r, g_tok[r])
            assert len(set(g_lp[r, :len(want)].view(np.uint32).tolist())) == 1


def _splitmix64_finalizer(z: int) -> int:
    """The published splitmix64 finalizer (Steele, Lea, Flood, OOPSLA'14)."""
    m = (1 << 64) - 1
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def test_row_bound_stale_and_foreign_scratch(head_2560):
    """At one M tile the ranges share a per-row bound on the row's k-th best
    logit through the workspace (a column below it cannot reach the top-k).
    The bound must never outlive its call: scratch filled with a large
    pattern before the first call, and a call with logits 16x larger before
    an ordinary one on the same scratch, leave the ordinary call's tables
    bit-identical to those of a fresh workspace.  Each call advances the
    generation word at the start of the scratch by one and leaves the ready
    word at the splitmix64 finalizer of the new generation."""
    W, Wd = head_2560
    Wp = mfd.pack_lm_head(Wd)
    h = synth.round_inputs(W, 8, 15, 11, seed=73).h.cuda()

    def run(rd, x):
        rd.status.zero_()
        rd.lmhead_topk_packed(x, Wp)
        torch.cuda.synchronize()
        assert status_of(rd) == 0
        return np_(rd.tk_tok).copy(), np_(rd.tk_logp).view(np.uint32).copy(), np_(rd.lse).view(np.uint32).copy()

    fresh = mfd.Round(1, 8, 15, 16, 1, 151936)
    fresh.ws.zero_()
    ref = run(fresh, h)
    rd = mfd.Round(1, 8, 15, 16, 1, 151936)
    rd.ws.view(torch.uint8).fill_(0x7F)
    for got in (run(rd, h), (run(rd, (h.float() * 16).to(torch.bfloat16)), run(rd, h))[1]):
        for a, b in zip(got, ref):
            np.testing.assert_array_equal(a, b)
    words = rd.ws.view(torch.uint8)[:16].cpu().numpy().view(np.uint64)
    gen, ready = int(words[0]), int(words[1])
    run(rd, h)
    words = rd.ws.view(torch.uint8)[:16].cpu().numpy().view(np.uint64)
    assert int(words[0]) == (gen + 1) % (1 << 64)
    assert int(words[1]) == _splitmix64_finalizer(int(words[0]))
    assert ready == _splitmix64_finalizer(gen)


@pytest.mark.parametrize("packed,topk", [(False, 2), (True, 2), (True, 8)])
def test_row_bound_every_logit_tied(packed, topk):
    """A weight of one repeated row gives every column of a hidden row the
    same logit.  Range heads never change then (a later column never beats
    an equal one), so with top-2 both residue classes of the row bound get
    that value and the bound equals every value it gates; with top-8 classes
    stay empty and the bound stays -inf.  Either way the top-k must be token
    ids 0..k-1 in order, each with log p = -log V."""
    V, H = 20000, 128
    rng = np.random.default_rng(5)
    row = (rng.standard_normal(H) / np.sqrt(H)).astype(np.float32)
    W = synth.bf16_round(np.tile(row, (V, 1)))
    h = synth.bf16_round(rng.standard_normal((37, H)).astype(np.float32))
    rd = mfd.Round(1, 1, 37, topk, 1, V)
    rd.status.zero_()
    if packed:
        rd.lmhead_topk_packed(h.cuda(), mfd.pack_lm_head(W.cuda()))
    else:
        rd.lmhead_topk(h.cuda(), W.cuda())
    torch.cuda.synchronize()
    assert status_of(rd) == 0
    tok, lp = np_(rd.tk_tok), np_(rd.tk_logp)
    assert (tok == np.arange(topk)[None, :]).all()
    np.testing.assert_allclose(lp, -np.log(V), atol=1e-4)
    o_lp, o_tok, _ = oracle.lmhead_topk(_bits(h), _bits(W), topk)
    assert (o_tok == np.arange(topk)[None, :]).all()


def test_row_bound_under_graph_replay(head_2560):
    """The LM head captured once in a CUDA graph and replayed with new hidden
    rows each time: every replay clears the row bound behind a generation
    that the replay itself advances on the device, so each gives the tables
    of a direct call on those rows, bit for bit."""
    W, Wd = head_2560
    Wp = mfd.pack_lm_head(Wd)
    hs = [synth.round_inputs(W, 8, 15, 11, seed=80 + i).h.cuda() for i in range(4)]
    rd = mfd.Round(1, 8, 15, 16, 1, 151936)
    h_static = torch.empty_like(hs[0])
    h_static.copy_(hs[0])
    rd.status.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        rd.lmhead_topk_packed(h_static, Wp)  # warm-up on a side stream, as before a capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rd.lmhead_topk_packed(h_static, Wp)
    ref = mfd.Round(1, 8, 15, 16, 1, 151936)
    for i in (1, 2, 0, 3, 1):
        h_static.copy_(hs[i])
        rd.status.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert status_of(rd) == 0
        ref.status.zero_()
        ref.lmhead_topk_packed(hs[i], Wp)
        torch.cuda.synchronize()
        assert status_of(ref) == 0
        np.testing.assert_array_equal(np_(rd.tk_tok), np_(ref.tk_tok))
        np.testing.assert_array_equal(np_(rd.tk_logp).view(np.uint32), np_(ref.tk_logp).view(np.uint32))
        np.testing.assert_array_equal(np_(rd.lse).view(np.uint32), np_(ref.lse).view(np.uint32))
