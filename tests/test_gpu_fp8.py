"""GPU parity of the FP8 drafter head (project page "Multi-Future Drafting",
In a serving engine, Figure 5 caption: the drafter's linear layers in FP8,
quantized online, acceptance unchanged).  The quantized weight and hidden rows
are bit-exact against the oracle's E4M3 encoding; the head's log-probs are
within 1e-4 of the oracle's FP8 head (exact E4M3 products accumulated in fp32
on the GPU, in double in the oracle); whole rounds keep the tree bit-exact
and the walk exact over the full vocabulary."""
import numpy as np
import pytest
import torch

import oracle
from tree_verified_speculative_gb300 import mfd, synth

from gpu_helpers import assert_tree_equal, check_topk, check_walk, np_, status_of, tree_outputs

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _expected_fp8_packed(q: np.ndarray) -> np.ndarray:
    """E4M3 bytes [V][H] in the packed order: per 256-row tile and 128-value
    K slice, rows of 128 bytes whose 16-byte chunk j sits at j ^ (row % 8);
    rows past V zero."""
    V, H = q.shape
    nt, nk = -(-V // 256), H // 128
    pad = np.zeros((nt * 256, H), np.uint8)
    pad[:V] = q
    out = np.empty((nt, nk, 256, 8, 16), np.uint8)
    src = pad.reshape(nt, 256, nk, 8, 16)
    for r in range(256):
        for pos in range(8):
            out[:, :, r, pos, :] = src[:, r, :, pos ^ (r % 8), :]
    return out.reshape(-1)


def test_fp8_pack_layout():
    rng = np.random.default_rng(5)
    V, H = 300, 256
    W = synth.bf16_round((rng.standard_normal((V, H)) * 0.05).astype(np.float32))
    Wp = mfd.pack_lm_head_fp8(W.cuda())
    torch.cuda.synchronize()
    n = mfd.mfd_lmhead_packed_fp8_bytes(V, H)
    assert Wp.numel() == n == 2 * 256 * H + 256
    got = Wp.cpu().numpy()
    q, scale = oracle.fp8_quantize(W)
    np.testing.assert_array_equal(got[:n - 256], _expected_fp8_packed(q))
    amax = got[n - 256:n - 252].view(np.float32)[0]
    assert amax == np.abs(W.float().numpy()).max()
    assert np.float32(amax) / np.float32(448.0) == np.float32(scale)


def test_fp8_quantize_rows():
    rng = np.random.default_rng(6)
    R, H = 37, 2560
    x = rng.standard_normal((R, H)).astype(np.float32) * np.exp2(rng.uniform(-8, 8, size=(R, 1))).astype(np.float32)
    x[3] = 0.0
    xb = synth.bf16_round(x)
    q = torch.empty((R, H), dtype=torch.uint8, device="cuda")
    sc = torch.empty((R,), dtype=torch.float32, device="cuda")
    mfd.mfd_fp8_quantize_rows(xb.cuda(), q, sc)
    torch.cuda.synchronize()
    gq, gs = np_(q), np_(sc)
    for r in range(R):
        oq, os_ = oracle.fp8_quantize(xb[r:r + 1])
        np.testing.assert_array_equal(gq[r], oq[0], err_msg=f"row {r}")
        assert gs[r] == np.float32(os_), r
    assert gs[3] == 0.0 and not gq[3].any()


def _gpu_fp8(h, W, topk, Wp=None):
    R, H = h.shape
    V = W.shape[0]
    rd = mfd.Round(1, 1, R, topk, 1, V, H=H)
    rd.status.zero_()
    rd.lmhead_topk_fp8(h.cuda(), mfd.pack_lm_head_fp8(W.cuda()) if Wp is None else Wp)
    torch.cuda.synchronize()
    assert status_of(rd) == 0
    return np_(rd.tk_logp), np_(rd.tk_tok), np_(rd.lse)


@pytest.mark.parametrize("R,H,V,topk", [
    (1, 128, 16, 1), (5, 128, 300, 8), (120, 256, 4099, 16), (130, 128, 2305, 16), (257, 384, 777, 8),
    (120, 2560, 20000, 16), (40, 5120, 3000, 32)])
def test_lmhead_fp8_small(R, H, V, topk):
    rng = np.random.default_rng(R + H + V)
    h = synth.bf16_round(rng.standard_normal((R, H)).astype(np.float32))
    W = synth.bf16_round((rng.standard_normal((V, H)) / np.sqrt(H)).astype(np.float32))
    g = _gpu_fp8(h, W, topk)
    o_lp, o_tk, o_lse, _, _ = oracle.lmhead_fp8_topk(h, W, topk)
    check_topk(g[0], g[1], o_lp, o_tk)
    np.testing.assert_allclose(g[2], o_lse, atol=5e-5)


def test_lmhead_fp8_rejects_h_not_multiple_of_128():
    h = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    rd = mfd.Round(1, 1, 4, 8, 1, 64, H=128)
    with pytest.raises(mfd.MfdError) as e:
        mfd.mfd_lmhead_topk_fp8(h, torch.zeros(1 << 16, dtype=torch.uint8, device="cuda"), 64, 8, rd.tk_logp,
                                rd.tk_tok, rd.lse, rd.status, rd.ws)
    assert e.value.code == mfd.MFD_ERR_UNSUPPORTED
    assert mfd.mfd_lmhead_packed_fp8_bytes(1000, 64) == 0


@pytest.fixture(scope="module")
def head():
    W = synth.lm_head(151936, 2560, seed=2024)
    return W, mfd.pack_lm_head_fp8(W.cuda())


@pytest.mark.parametrize("R", [1, 15])
def test_fp8_staged_hidden_rows_match_unstaged(head, R):
    """E4M3 hidden rows that span 144 KB or less are quantized into a
    zero-padded copy; 60 rows (150 KB) are not padded.  The same rows give
    bit-identical tables either way."""
    W, Wp = head
    h = synth.round_inputs(W, 8, 15, 11, seed=71).h[:60]
    out = []
    for rows in (R, 60):
        rd = mfd.Round(1, 1, rows, 16, 1, 151936, H=2560)
        rd.status.zero_()
        rd.lmhead_topk_fp8(h[:rows].contiguous().cuda(), Wp)
        torch.cuda.synchronize()
        assert status_of(rd) == 0
        out.append((np_(rd.tk_tok)[:R], np_(rd.tk_logp)[:R].view(np.uint32), np_(rd.lse)[:R].view(np.uint32)))
    for a, b in zip(*out):
        np.testing.assert_array_equal(a, b)


def test_lmhead_fp8_pages_shape_sampled_rows(head):
    """K=8, L=15, H=2560, V=151,936, top-16: all 120 rows through the FP8
    head, 12 of them against the oracle's FP8 head over the full vocabulary;
    the planted token stays the usual argmax."""
    W, Wp = head
    r = synth.round_inputs(W, 8, 15, 11, seed=7)
    g = _gpu_fp8(r.h, W, 16, Wp)
    rows = np.random.default_rng(1).choice(120, size=12, replace=False)
    o_lp, o_tk, o_lse, _, _ = oracle.lmhead_fp8_topk(r.h[rows], W, 16)
    check_topk(g[0][rows], g[1][rows], o_lp, o_tk)
    np.testing.assert_allclose(g[2][rows], o_lse, atol=5e-5)
    assert np.mean(g[1][:, 0] == r.fut.reshape(-1)) > 0.5


@pytest.mark.parametrize("temperature", [0.0, 1.0])
def test_fp8_head_rounds(head, temperature):
    """Rounds through the FP8 head: tables on sampled rows against the oracle's
    FP8 head, the tree bit-exact from the GPU's tables, the walk exact over the
    target's full rows (FP8 changes the draft only: verification is the
    target's)."""
    W, Wp = head
    rd = mfd.Round(1, 8, 15, 16, 256, 151936, H=2560)
    exact = 0
    for i in range(2):
        r = synth.round_inputs(W, 8, 15, 11, seed=800 + i)
        rd.status.zero_()
        rd.lmhead_topk_fp8(r.h.cuda(), Wp)
        rd.build_tree()
        torch.cuda.synchronize()
        assert status_of(rd) == 0
        lp, tk = np_(rd.tk_logp), np_(rd.tk_tok)
        rows = np.array([i, 60 + i, 119 - i])
        o_lp, o_tk, _, _, _ = oracle.lmhead_fp8_topk(r.h[rows], W, 16)
        check_topk(lp[rows], tk[rows], o_lp, o_tk)
        o = oracle.build_tree(lp.reshape(8, 15, 16), tk.reshape(8, 15, 16), 256)
        assert_tree_equal(tree_outputs(rd), o, 0)
        noise = synth.target_noise(257, 151936, np.random.default_rng(r.seed % (2**32)))
        prow, pcol = synth.plant_sites(o["parent"], o["token"], o["depth"], int(o["n_nodes"]), r.fut[r.target_mode])
        t = synth.plant(noise, prow, pcol)
        rd.verify(torch.from_numpy(t[None]).cuda(), torch.tensor([temperature], device="cuda"),
                  torch.tensor([r.seed], dtype=torch.int64, device="cuda"))
        torch.cuda.synchronize()
        assert status_of(rd) == 0
        oa = oracle.verify(t, o["parent"], o["token"], int(o["n_nodes"]), 15, temperature, r.seed)
        exact += check_walk(int(np_(rd.accept_len)[0]), np_(rd.path_nodes)[0], np_(rd.out_tokens)[0], *oa,
                            sampled=temperature > 0)
    assert exact >= 1
