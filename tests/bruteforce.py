"""Brute-force references used to pin the oracle (tests only).

Written independently of ``oracle/``: every prefix up to depth L is listed,
scored by every mode, and the whole list is sorted.  Nothing here is a heap
or a best-first search.
"""
from __future__ import annotations

import itertools

import numpy as np


def mode_score_tables(tk_logp: np.ndarray, tk_tok: np.ndarray, V: int) -> np.ndarray:
    """Dense per-mode log-prob tables [K, L, V]; tokens outside a row's top-k
    get -inf (the mode cannot reach them)."""
    K, L, k = tk_logp.shape
    dense = np.full((K, L, V), -np.inf, dtype=np.float32)
    for m in range(K):
        for i in range(L):
            dense[m, i, tk_tok[m, i]] = tk_logp[m, i]
    return dense


def all_prefixes(tk_logp: np.ndarray, tk_tok: np.ndarray, V: int, alphabet=None):
    """Every token sequence of depth 1..L over `alphabet` (default range(V)),
    with s = max over modes of the fp32 left fold, and the smallest mode
    attaining it.  Returns a list of (s, seq tuple, mode) with s > -inf."""
    K, L, _ = tk_logp.shape
    dense = mode_score_tables(tk_logp, tk_tok, V)
    alphabet = list(range(V)) if alphabet is None else list(alphabet)
    out = []
    # per mode, score[d] arrays over the product alphabet^d built one depth at a time
    A = np.asarray(alphabet, dtype=np.int64)
    prev = None  # [K, n_seq] scores at depth d-1
    prev_seqs = None
    for d in range(1, L + 1):
        if d == 1:
            seqs = A[:, None]
            sc = dense[:, 0, A]  # [K, |A|]
        else:
            n_prev = prev_seqs.shape[0]
            seqs = np.concatenate([np.repeat(prev_seqs, len(A), axis=0),
                                   np.tile(A, n_prev)[:, None]], axis=1)
            add = dense[:, d - 1, A]  # [K, |A|]
            sc = (np.repeat(prev, len(A), axis=1) + np.tile(add, (1, n_prev))).astype(np.float32)
        s = sc.max(axis=0)
        mode = np.argmax(sc == s[None, :], axis=0)
        keep = s > -np.inf
        for i in np.nonzero(keep)[0]:
            out.append((np.float32(s[i]), tuple(int(t) for t in seqs[i]), int(mode[i])))
        prev, prev_seqs = sc, seqs
    return out


def sort_prefixes(items):
    """Sort by (s descending, token ids lexicographically ascending, a proper
    prefix first)."""
    return sorted(items, key=lambda e: (-float(e[0]), e[1]))


def brute_tree(tk_logp, tk_tok, V, B, alphabet=None):
    return sort_prefixes(all_prefixes(tk_logp, tk_tok, V, alphabet))[:B]


def node_sequences(parent, token, n_nodes):
    """Token sequence of every node (root = empty) from the parent links."""
    seqs = [()]
    for n in range(1, n_nodes):
        p = int(parent[n])
        assert 0 <= p < n
        seqs.append(seqs[p] + (int(token[n]),))
    return seqs


def product_brute(tk_logp1, tk_tok1, V, B):
    """K = 1 product-ranked tree (DDTree) by listing every rank tuple."""
    L, k = tk_logp1.shape
    items = []
    for d in range(1, L + 1):
        for ranks in itertools.product(range(k), repeat=d):
            s = np.float32(tk_logp1[0, ranks[0]])
            for i in range(1, d):
                s = np.float32(s + tk_logp1[i, ranks[i]])
            if s == -np.inf:
                continue
            items.append((s, tuple(int(tk_tok1[i, ranks[i]]) for i in range(d)), 0))
    return sort_prefixes(items)[:B]
