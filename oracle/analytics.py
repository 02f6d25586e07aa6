"""Tree analytics, plain numpy -- TEST INFRASTRUCTURE of the oracle: only
tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may use it.

Two measures the project page "Multi-Future Drafting" reasons with:

- Chimeras (TL;DR, and "The problem: a product splices futures"): a
  prefix stitched together from different futures -- at every position its
  token is some future's token there -- that is a prefix of none of them, so
  the target never says it.
- Covered mass by depth (How it works, step 1: the expected number of
  accepted tokens is the probability mass the tree covers): the mass of a
  node is the probability that the walk reaches it, the product along its
  path of the target's probability of each next token; summed per depth it
  is P(accepted >= d), and over all depths the expected accepted length.
"""
from __future__ import annotations

import numpy as np

ON_FUTURE, CHIMERA, OTHER = 0, 1, 2


def _sequences(parent: np.ndarray, token: np.ndarray, n_nodes: int) -> list[tuple[int, ...]]:
    """Token sequence of every node (the root's is empty; parents come first)."""
    seqs: list[tuple[int, ...]] = [()]
    for n in range(1, n_nodes):
        p = int(parent[n])
        if not 0 <= p < n:
            raise ValueError("parent must precede its child")
        seqs.append(seqs[p] + (int(token[n]),))
    return seqs


def node_classes(parent: np.ndarray, token: np.ndarray, n_nodes: int, futures: np.ndarray) -> np.ndarray:
    """int32 [n_nodes]: ON_FUTURE for the root and every prefix of a future,
    CHIMERA for a splice of the futures that is a prefix of none of them,
    OTHER for a prefix with a token that no future has at that position.
    futures: int [F][L], one row per future."""
    fut = np.asarray(futures)
    seqs = _sequences(parent, token, n_nodes)
    out = np.empty(n_nodes, np.int32)
    for n, s in enumerate(seqs):
        d = len(s)
        if d == 0:
            out[n] = ON_FUTURE
            continue
        if d > fut.shape[1]:
            out[n] = OTHER
            continue
        prefix_of = any(tuple(int(x) for x in fut[f, :d]) == s for f in range(fut.shape[0]))
        splice = all(any(int(fut[f, i]) == s[i] for f in range(fut.shape[0])) for i in range(d))
        out[n] = ON_FUTURE if prefix_of else (CHIMERA if splice else OTHER)
    return out


def _step_probs(row: np.ndarray, temperature: float) -> np.ndarray:
    """The target's distribution over the next token at a node: softmax(t / T)
    in double for T > 0; for T = 0 the greedy choice (smallest id on ties)."""
    row = np.asarray(row, np.float64)
    if temperature > 0:
        z = row / temperature
        z = z - z.max()
        p = np.exp(z)
        return p / p.sum()
    p = np.zeros_like(row)
    p[int(np.argmax(row))] = 1.0  # argmax returns the first maximum: the smallest id
    return p


def covered_mass(parent: np.ndarray, token: np.ndarray, depth: np.ndarray, n_nodes: int, t: np.ndarray,
                 temperature: float, L: int) -> tuple[np.ndarray, np.ndarray]:
    """(reach [n_nodes], mass [L + 1]): reach[n] is the probability that the
    walk arrives at node n (1 at the root); mass[d] sums reach over the nodes
    at depth d (mass[0] = 1)."""
    reach = np.zeros(n_nodes)
    reach[0] = 1.0
    probs: dict[int, np.ndarray] = {}
    for n in range(1, n_nodes):
        p = int(parent[n])
        if p not in probs:
            probs[p] = _step_probs(t[p], temperature)
        reach[n] = reach[p] * probs[p][int(token[n])]
    mass = np.zeros(L + 1)
    for n in range(n_nodes):
        mass[int(depth[n])] += reach[n]
    return reach, mass
