"""Pins of the oracle's FP8 drafter head (project page "Multi-Future Drafting",
In a serving engine, Figure 5 caption: the drafter's linear layers in FP8,
the serving engine's online option).  The E4M3 encoding is checked against
torch's own float8_e4m3fn conversion, an implementation written by another
project, on every code, on random values across the range, on every midpoint
between neighbours (ties to even) and on the saturating edge; the FP8 LM head
against a plain numpy restatement that quantizes through torch's conversion."""
import numpy as np
import pytest
import torch

import oracle
from tree_verified_speculative_gb300 import synth


def _torch_e4m3(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_value(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(b, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_every_code_decodes_like_torch():
    codes = np.arange(256, dtype=np.uint8)
    a, b = oracle.e4m3_value(codes), _torch_value(codes)
    nan = np.isnan(b)
    assert list(np.flatnonzero(nan)) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(a), nan)
    np.testing.assert_array_equal(a[~nan], b[~nan])
    assert a[0x7E] == 448.0 and a[0x01] == 2.0 ** -9


def test_encoding_matches_torch_on_random_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.uniform(-448, 448, 4000),
        np.sign(rng.standard_normal(4000)) * np.exp2(rng.uniform(-12, 8.8, 4000)),  # every binade, subnormals
        rng.standard_normal(2000) * 0.01,
    ]).astype(np.float32)
    x = np.clip(x, -448, 448)
    np.testing.assert_array_equal(oracle.e4m3(x), _torch_e4m3(x))


def test_midpoints_round_to_even():
    vals = np.sort(np.unique(_torch_value(np.arange(0, 0x7F, dtype=np.uint8))))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (vals[:-1] + vals[1:]) / 2)  # midpoints exact in fp32
    got = oracle.e4m3(mids)
    np.testing.assert_array_equal(got, _torch_e4m3(mids))
    # ties go to the code with an even mantissa
    assert np.all(got & 1 == 0)
    np.testing.assert_array_equal(oracle.e4m3(-mids), _torch_e4m3(-mids))


def test_saturation_and_nan():
    big = np.array([448.0, 449.0, 464.0, 480.0, 1e6, 3e38, np.inf], np.float32)
    assert list(oracle.e4m3(big)) == [0x7E] * len(big)
    assert list(oracle.e4m3(-big)) == [0xFE] * len(big)
    assert oracle.e4m3(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F
    assert list(oracle.e4m3(np.array([0.0, -0.0], np.float32))) == [0x00, 0x80]


def _numpy_fp8_head(h, W, topk):
    """The FP8 head restated in numpy, quantizing through torch's conversion."""
    hf, Wf = h.float().numpy(), W.float().numpy()
    aW = np.float32(np.abs(Wf).max())
    qW = _torch_value(_torch_e4m3(Wf * (np.float32(448.0) / aW)))
    sW = aW / np.float32(448.0)
    z = np.empty((hf.shape[0], Wf.shape[0]))
    for r in range(hf.shape[0]):
        a = np.float32(np.abs(hf[r]).max())
        q = _torch_value(_torch_e4m3(hf[r] * (np.float32(448.0) / a)))
        f = np.float32(a / np.float32(448.0)) * sW
        z[r] = np.float64(f) * (qW @ q)
    m = z.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(z - m).sum(axis=1))
    lp = (z - lse[:, None]).astype(np.float32)
    tok = np.stack([np.lexsort((np.arange(z.shape[1]), -row))[:topk] for row in lp])
    return np.take_along_axis(lp, tok, 1), tok, lse, sW


def test_fp8_head_matches_numpy_restatement():
    rng = np.random.default_rng(3)
    R, H, V = 6, 256, 3000
    W = synth.bf16_round((rng.standard_normal((V, H)) / np.sqrt(H)).astype(np.float32))
    h = synth.bf16_round(rng.standard_normal((R, H)).astype(np.float32))
    lp, tk, lse, sW, t = oracle.lmhead_fp8_topk(h, W, 16)
    n_lp, n_tk, n_lse, n_sW = _numpy_fp8_head(h, W, 16)
    assert sW == n_sW
    np.testing.assert_array_equal(t, np.abs(h.float().numpy()).max(axis=1) / np.float32(448.0))
    np.testing.assert_array_equal(tk, n_tk)
    np.testing.assert_allclose(lp, n_lp, rtol=0, atol=2e-6)
    np.testing.assert_allclose(lse, n_lse, rtol=0, atol=1e-9)


def test_fp8_head_stays_close_to_bf16_head():
    """FP8 changes the draft distribution only slightly: on the planted
    hidden states the best token is the same and the log-probs move by well
    under 0.1 (3 mantissa bits: a relative step of at most 2^-4 per value,
    averaging out over the 2560-term sums)."""
    V, H = 20000, 2560
    W = synth.lm_head(V, H, seed=5)
    r = synth.round_inputs(W, 2, 4, 2, seed=6)
    a = oracle.lmhead_topk(r.h, W, 8)
    b = oracle.lmhead_fp8_topk(r.h, W, 8)
    assert np.array_equal(a[1][:, 0], b[1][:, 0])
    assert np.max(np.abs(a[0][:, 0] - b[0][:, 0])) < 0.1


def test_zero_rows_quantize_to_zero():
    x = torch.zeros((3, 64), dtype=torch.bfloat16)
    q, sc = oracle.fp8_quantize(x)
    assert sc == 0.0 and not q.any()
