"""Seeded synthetic inputs for the MFD round (no method arithmetic here).

This module only draws inputs: LM-head weights, drafter hidden states with
planted per-mode futures, raw logits for the tiny case, and target logits
with a planted future.  It computes no log-softmax, no score, no tree and no
verification; both the CUDA path and the CPU oracle receive the arrays it
returns.

The shapes follow the pages' setting (project page "Multi-Future Drafting",
How it works, and the "MFD drafter for Qwen3.5-4B" model table): K = 8 modes,
a block of 16 with L = 15 drafted positions, width 2560, budgets 64-256.

Recipe (all numpy ``Generator(PCG64(seed))``):

* LM head ``W [V, H]``: N(0, sigma^2) with sigma = 1/sqrt(H), rounded to bf16.
* Futures ``t [K, L]``: ``n_shared`` positions (chosen at random) carry one
  token common to all modes; the other positions draw a token per mode;
  tokens uniform on [0, V).
* Hidden states ``h[k, i] = scale * W[t_ki] / ||W[t_ki]|| + N(0, 1)^H``,
  rounded to bf16; row r = k * L + i.
* Target logits ``[N, V]``: N(0, 1) per entry; then for every tree node whose
  token sequence is a prefix of the chosen mode's future at depth d < L, the
  entry of that future's token at depth d + 1 gets +plant (10).  The plant
  depends on the tree, so it is applied after the tree exists.
"""
from __future__ import annotations

import concurrent.futures as _cf
from dataclasses import dataclass

import numpy as np
import torch


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def bf16_round(x: np.ndarray) -> torch.Tensor:
    """fp32 numpy -> torch bf16 CPU tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def lm_head(V: int, H: int, seed: int, sigma: float | None = None, chunk_rows: int = 8192) -> torch.Tensor:
    """bf16 LM head W [V, H] ~ N(0, sigma^2), sigma = 1/sqrt(H) by default.

    Drawn in row chunks with independent child seeds so that it can run on a
    thread pool; the result depends only on (V, H, seed, sigma, chunk_rows)."""
    sigma = 1.0 / np.sqrt(H) if sigma is None else sigma
    W = torch.empty((V, H), dtype=torch.bfloat16)
    starts = list(range(0, V, chunk_rows))
    seeds = np.random.SeedSequence(seed).spawn(len(starts))

    def fill(i: int) -> None:
        s = starts[i]
        e = min(V, s + chunk_rows)
        g = np.random.Generator(np.random.PCG64(seeds[i]))
        x = g.standard_normal((e - s, H), dtype=np.float32)
        x *= np.float32(sigma)
        W[s:e] = torch.from_numpy(x).to(torch.bfloat16)

    with _cf.ThreadPoolExecutor(max_workers=min(16, max(1, len(starts)))) as ex:
        list(ex.map(fill, range(len(starts))))
    return W


def futures(K: int, L: int, V: int, n_shared: int, rng: np.random.Generator,
            vocab: np.ndarray | None = None) -> np.ndarray:
    """Per-mode planted futures int32 [K, L] sharing n_shared positions;
    tokens uniform on [0, V), or on the ids of `vocab` (a draft vocabulary)."""
    hi = V if vocab is None else len(vocab)
    t = rng.integers(0, hi, size=(K, L), dtype=np.int64)
    shared = rng.choice(L, size=n_shared, replace=False)
    common = rng.integers(0, hi, size=(n_shared,), dtype=np.int64)
    t[:, shared] = common[None, :]
    if vocab is not None:
        t = np.asarray(vocab, np.int64)[t]
    return t.astype(np.int32)


def vocab_subset(V: int, n: int, seed: int) -> np.ndarray:
    """A draft vocabulary: n distinct ids of [0, V), increasing -- the
    stand-in for the target's most frequent tokens."""
    rng = _rng(seed)
    return np.sort(rng.choice(V, size=n, replace=False)).astype(np.int32)


def hidden(W: torch.Tensor, fut: np.ndarray, rng: np.random.Generator, scale: float = 6.0) -> torch.Tensor:
    """bf16 hidden states [K*L, H]: scale * W[t]/||W[t]|| + N(0, 1)."""
    K, L = fut.shape
    H = W.shape[1]
    rows = W[torch.from_numpy(fut.reshape(-1).astype(np.int64))].float().numpy().astype(np.float64)
    unit = rows / np.linalg.norm(rows, axis=1, keepdims=True)
    noise = rng.standard_normal((K * L, H), dtype=np.float32).astype(np.float64)
    return bf16_round((scale * unit + noise).astype(np.float32))


def target_noise(N: int, V: int, rng: np.random.Generator) -> np.ndarray:
    """fp32 N(0, 1) target logits [N, V] before the plant."""
    return rng.standard_normal((N, V), dtype=np.float32)


def plant_sites(parent: np.ndarray, token: np.ndarray, depth: np.ndarray, n_nodes: int,
                future: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(rows, cols) that get the plant: node n whose token sequence equals
    future[:d] (d = depth[n] < L) gets +plant at column future[d]."""
    L = future.shape[0]
    on = np.zeros(n_nodes, dtype=bool)
    on[0] = True
    rows, cols = [], []
    for n in range(n_nodes):
        d = int(depth[n])
        if n > 0:
            p = int(parent[n])
            on[n] = on[p] and int(token[n]) == int(future[d - 1])
        if on[n] and d < L:
            rows.append(n)
            cols.append(int(future[d]))
    return np.asarray(rows, np.int64), np.asarray(cols, np.int64)


def plant(noise: np.ndarray, rows: np.ndarray, cols: np.ndarray, amount: float = 10.0) -> np.ndarray:
    """Copy of noise with +amount at (rows, cols)."""
    t = noise.copy()
    t[rows, cols] += np.float32(amount)
    return t


# ---------------------------------------------------------------------------
@dataclass
class Tiny:
    """Tiny exact case: K=2, L=4, V=32, fp32 logits N(0, 2^2) with +8 on two
    planted futures (one per mode) sharing positions 1 and 3, differing at 2
    and 4; top-k 8, B = 8; target rows N(0, 1) with +10 on mode 2's future."""
    logits: np.ndarray  # [K*L, V] fp32, row k*L + i
    fut: np.ndarray  # [K, L]
    K: int = 2
    L: int = 4
    V: int = 32
    topk: int = 8
    B: int = 8


def tiny(seed: int = 1) -> Tiny:
    rng = _rng(seed)
    K, L, V = 2, 4, 32
    a = rng.choice(V, size=L, replace=False).astype(np.int32)
    b = a.copy()
    for pos in (1, 3):
        choices = [v for v in range(V) if v != a[pos]]
        b[pos] = choices[int(rng.integers(0, len(choices)))]
    fut = np.stack([a, b])
    z = (2.0 * rng.standard_normal((K, L, V))).astype(np.float32)
    for k in range(K):
        for i in range(L):
            z[k, i, fut[k, i]] += np.float32(8.0)
    return Tiny(logits=z.reshape(K * L, V), fut=fut)


@dataclass
class Round:
    """One request's drafting inputs for one round."""
    h: torch.Tensor  # bf16 [K*L, H]
    fut: np.ndarray  # int32 [K, L]
    target_mode: int  # the mode whose future the target plant follows
    seed: int  # Philox seed for sampled verification


def round_inputs(W: torch.Tensor, K: int, L: int, n_shared: int, seed: int,
                 vocab: np.ndarray | None = None, scale: float = 6.0) -> Round:
    """W is the full-vocabulary head; with `vocab`, the futures are drawn from
    that draft vocabulary.  `scale` sets how confident the drafter is in its
    futures (the planted token's logit is about `scale`)."""
    rng = _rng(seed)
    fut = futures(K, L, W.shape[0], n_shared, rng, vocab)
    h = hidden(W, fut, rng, scale)
    m = int(rng.integers(0, K))
    s = int(rng.integers(0, 2**63 - 1))
    return Round(h=h, fut=fut, target_mode=m, seed=s)
