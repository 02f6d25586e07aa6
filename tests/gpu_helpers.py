"""Helpers shared by the GPU parity tests: run the CUDA path through the
C ABI (the ctypes binding) and compare with the oracle at the tolerances the
method statement fixes."""
from __future__ import annotations

import numpy as np
import torch

from tree_verified_speculative_gb300 import mfd

LOGP_TOL = 1e-4  # log-probabilities, absolute
GAP_TOL = 1e-5  # sampled verification: decisions closer than this are excused


def np_(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def status_of(rd: mfd.Round) -> int:
    return int(rd.status.item())


def check_topk(g_lp, g_tok, o_lp, o_tok, tol=LOGP_TOL):
    """Top-k tables agree.

    - Values, position by position, within tol.
    - Each GPU row is sorted by (log p desc, token id asc) exactly: equal
      values come in increasing id order.
    - Tokens, position by position: equal to the oracle's, except where the
      oracle's value at that position lies within tol of another of the
      row's values (a near tie the two precisions may order differently),
      where the token must be one of that near-tied group; tokens in the set
      difference must lie within tol of the k-th value (the cut)."""
    g_lp, g_tok, o_lp, o_tok = map(np.asarray, (g_lp, g_tok, o_lp, o_tok))
    assert g_lp.shape == o_lp.shape
    np.testing.assert_allclose(g_lp, o_lp, rtol=0, atol=tol)
    k = o_lp.shape[1]
    for r in range(o_lp.shape[0]):
        for j in range(k - 1):
            a, b = float(g_lp[r, j]), float(g_lp[r, j + 1])
            assert a > b or (a == b and int(g_tok[r, j]) < int(g_tok[r, j + 1])), \
                f"row {r}: GPU entries {j}, {j + 1} out of (log p desc, id asc) order"
        cut = float(o_lp[r, -1])
        gs, os_ = set(g_tok[r].tolist()), set(o_tok[r].tolist())
        for t in gs ^ os_:
            if t in gs:
                v = float(g_lp[r][list(g_tok[r]).index(t)])
            else:
                v = float(o_lp[r][list(o_tok[r]).index(t)])
            assert abs(v - cut) <= tol, f"row {r}: token {t} (logp {v}) differs and is not at the cut {cut}"
        for j in range(k):
            if int(g_tok[r, j]) == int(o_tok[r, j]):
                continue
            v = float(o_lp[r, j])
            group = {int(o_tok[r, i]) for i in range(k) if abs(float(o_lp[r, i]) - v) <= tol}
            near_cut = abs(v - cut) <= tol
            assert len(group) > 1 or near_cut, \
                f"row {r} position {j}: token {int(g_tok[r, j])} where the oracle has {int(o_tok[r, j])}"
            assert int(g_tok[r, j]) in group or near_cut, \
                f"row {r} position {j}: token {int(g_tok[r, j])} outside the near-tied group {sorted(group)}"


def tree_outputs(rd: mfd.Round) -> dict:
    return {
        "parent": np_(rd.parent), "token": np_(rd.token), "depth": np_(rd.depth), "score": np_(rd.score),
        "mode": np_(rd.mode), "mask": np_(rd.mask).view(np.uint32), "pos": np_(rd.pos), "n_nodes": np_(rd.n_nodes),
    }


def assert_tree_equal(g: dict, o: dict, q: int | None = None):
    """Bit-exact tree: node set and order, parents, tokens, depths, score
    bits, modes, mask and positions."""
    for k in ("n_nodes", "parent", "token", "depth", "mode", "pos"):
        a = g[k] if q is None else g[k][q]
        b = o[k]
        np.testing.assert_array_equal(a, b, err_msg=k)
    a = g["score"] if q is None else g["score"][q]
    np.testing.assert_array_equal(a.view(np.uint32), o["score"].view(np.uint32), err_msg="score bits")
    a = g["mask"] if q is None else g["mask"][q]
    np.testing.assert_array_equal(a, o["mask"], err_msg="mask")


def gpu_tree(lp: np.ndarray, tk: np.ndarray, B: int, anchor=None, base_pos=None) -> tuple[dict, int]:
    """Build trees on the GPU from given tables [n_req, K, L, topk]."""
    n_req, K, L, topk = lp.shape
    rd = mfd.Round(n_req, K, L, topk, B, V=max(16, topk))
    rd.tk_logp.copy_(torch.from_numpy(np.ascontiguousarray(lp.reshape(-1, topk))))
    rd.tk_tok.copy_(torch.from_numpy(np.ascontiguousarray(tk.reshape(-1, topk))))
    if anchor is not None:
        rd.anchor.copy_(torch.from_numpy(np.asarray(anchor, np.int32)))
    if base_pos is not None:
        rd.base_pos.copy_(torch.from_numpy(np.asarray(base_pos, np.int32)))
    rd.status.zero_()
    rd.build_tree()
    torch.cuda.synchronize()
    return tree_outputs(rd), status_of(rd)


def check_walk(g_acc, g_path, g_out, o_acc, o_path, o_out, o_gap, sampled: bool):
    """Greedy: exact.  Sampled: exact up to the first step whose top-two
    perturbed scores (oracle) lie within GAP_TOL; from there on excused."""
    L1 = len(o_path)
    if not sampled:
        assert g_acc == o_acc
        np.testing.assert_array_equal(g_path, o_path)
        np.testing.assert_array_equal(g_out, o_out)
        return True
    for j in range(L1):
        if o_path[j] < 0:
            break
        if o_gap[j] < GAP_TOL:
            return False  # excused from here on
        assert g_path[j] == o_path[j], f"step {j}"
        assert g_out[j] == o_out[j], f"step {j}"
    assert g_acc == o_acc
    np.testing.assert_array_equal(g_path, o_path)
    np.testing.assert_array_equal(g_out, o_out)
    return True
