"""CPU oracle for the Multi-Future Drafting round -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and the two share no
code.

The arithmetic lives in ``mfd_oracle.c`` (plain C, compiled here with gcc
``-O2 -fno-fast-math -ffp-contract=off -fopenmp``); this module only marshals
numpy arrays.  Each function cites the passage of the pages it follows:

* ``lmhead_logits`` / ``lmhead_topk`` -- "MFD drafter for Qwen3.5-4B" model
  card, Model table: the target's LM head applied to the drafter's hidden
  states; project page "Multi-Future Drafting", How it works, step 2: one
  distribution per (mode, position).
* ``logits_topk`` -- the same log-softmax and top-k from given fp32 logits.
* ``e4m3`` / ``e4m3_value`` / ``fp8_quantize`` / ``lmhead_fp8_topk`` -- the
  FP8 drafter head: project page, In a serving engine, Figure 5 caption (the
  drafter's linear layers in FP8, quantized online; acceptance unchanged).
* ``build_tree`` -- project page, How it works, step 3: prefixes scored by
  their best mode, the B best kept as one tree, found by merging the K
  per-mode best-first searches into one heap.
* ``verify`` -- model card, first paragraph, and project page Figure 2 (c):
  standard (lossless) tree verification, greedy or sampled.
* ``philox4x32_10`` / ``gumbel`` -- Salmon et al., "Parallel random numbers:
  as easy as 1, 2, 3" (SC'11), Philox4x32 with 10 rounds.

Parity pins: every function here is checked by ``tests/test_oracle_*.py``
against brute force, closed forms, an independent Philox implementation and
the pages' invariants.  The only part without a pin is the pages' own worked
example (Figure 1/2), whose probabilities are not printed in the text:
parity unpinned for that example.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mfd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc) and return its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, u64, f32 = ctypes.c_int, ctypes.c_uint64, ctypes.c_float
            lib.oracle_lmhead_logits.argtypes = [P, i32, i32, P, i32, i32, P, i32]
            lib.oracle_lmhead_logits.restype = None
            lib.oracle_lmhead_topk.argtypes = [P, i32, i32, P, i32, i32, P, P, P, i32]
            lib.oracle_lmhead_topk.restype = i32
            lib.oracle_e4m3.argtypes = [f32]
            lib.oracle_e4m3.restype = ctypes.c_uint8
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_fp8_quantize.argtypes = [P, ctypes.c_size_t, P, P]
            lib.oracle_fp8_quantize.restype = None
            lib.oracle_lmhead_fp8_topk.argtypes = [P, i32, i32, P, i32, i32, P, P, P, P, P, i32]
            lib.oracle_lmhead_fp8_topk.restype = i32
            lib.oracle_logits_topk.argtypes = [P, i32, i32, i32, P, P, P]
            lib.oracle_logits_topk.restype = i32
            lib.oracle_build_tree.argtypes = [P, P, i32, i32, i32, i32, ctypes.c_int32,
                                              ctypes.c_int32] + [P] * 8
            lib.oracle_build_tree.restype = i32
            lib.oracle_philox_batch.argtypes = [P, P, i32, P]
            lib.oracle_philox_batch.restype = None
            lib.oracle_gumbel.argtypes = [u64, ctypes.c_int32, ctypes.c_int32]
            lib.oracle_gumbel.restype = f32
            lib.oracle_gumbel_batch.argtypes = [u64, ctypes.c_int32, i32, P]
            lib.oracle_gumbel_batch.restype = None
            lib.oracle_verify.argtypes = [P, i32, i32, i32, P, P, f32, u64, P, P, P, P]
            lib.oracle_verify.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(a) -> np.ndarray:
    """Accept bf16 as uint16 bit patterns (numpy) or a torch bf16 CPU tensor."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16
        return np.ascontiguousarray(a)
    import torch  # only for converting a torch bf16 tensor's bits

    assert a.dtype == torch.bfloat16
    return np.ascontiguousarray(a.contiguous().view(torch.int16).numpy().view(np.uint16))


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


def lmhead_logits(h, W, v0: int = 0, v1: int | None = None, nthreads: int = 0) -> np.ndarray:
    """z[r, v] = sum_h h[r, h] W[v, h] in double, for v in [v0, v1)."""
    hb, wb = _bf16_bits(h), _bf16_bits(W)
    R, H = hb.shape
    V = wb.shape[0]
    v1 = V if v1 is None else v1
    z = np.empty((R, v1 - v0), dtype=np.float64)
    _load().oracle_lmhead_logits(_ptr(hb), R, H, _ptr(wb), v0, v1, _ptr(z), nthreads)
    return z


def lmhead_topk(h, W, topk: int, nthreads: int = 0):
    """Per row: log-softmax over the vocabulary of h W^T, then the top-k.

    Returns (tk_logp f32 [R, topk], tk_tok i32 [R, topk], lse f64 [R]); each
    row sorted by (log p descending, token id ascending)."""
    hb, wb = _bf16_bits(h), _bf16_bits(W)
    R, H = hb.shape
    V = wb.shape[0]
    lp = np.empty((R, topk), np.float32)
    tk = np.empty((R, topk), np.int32)
    lse = np.empty((R,), np.float64)
    rc = _load().oracle_lmhead_topk(_ptr(hb), R, H, _ptr(wb), V, topk, _ptr(lp), _ptr(tk),
                                   _ptr(lse), nthreads)
    if rc:
        raise ValueError(f"oracle_lmhead_topk failed ({rc})")
    return lp, tk, lse


def e4m3(x) -> np.ndarray:
    """FP8 E4M3 bytes of fp32 values: round to nearest even, saturating at
    +-448 (project page "Multi-Future Drafting", Figure 5 caption: the
    drafter's linears in FP8; the format reading is in mfd_oracle.c)."""
    a = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    lib = _load()
    return np.array([lib.oracle_e4m3(float(v)) for v in a], np.uint8).reshape(np.shape(x))


def e4m3_value(b) -> np.ndarray:
    """Exact values of E4M3 bytes (NaN for 0x7F / 0xFF)."""
    a = np.ascontiguousarray(b, dtype=np.uint8).reshape(-1)
    lib = _load()
    return np.array([lib.oracle_e4m3_value(int(v)) for v in a], np.float64).reshape(np.shape(b))


def fp8_quantize(x) -> tuple[np.ndarray, float]:
    """One scale for all of x (bf16): (E4M3 bytes, scale = max|x| / 448)."""
    xb = _bf16_bits(x)
    q = np.empty(xb.shape, np.uint8)
    sc = ctypes.c_float()
    _load().oracle_fp8_quantize(_ptr(xb), xb.size, _ptr(q), ctypes.byref(sc))
    return q, float(sc.value)


def lmhead_fp8_topk(h, W, topk: int, nthreads: int = 0):
    """The FP8 LM head (weight one scale, each hidden row its own), then the
    log-softmax and top-k as lmhead_topk.  Returns (tk_logp, tk_tok, lse,
    weight scale, row scales [R])."""
    hb, wb = _bf16_bits(h), _bf16_bits(W)
    R, H = hb.shape
    V = wb.shape[0]
    lp = np.empty((R, topk), np.float32)
    tk = np.empty((R, topk), np.int32)
    lse = np.empty((R,), np.float64)
    t = np.empty((R,), np.float32)
    sW = ctypes.c_float()
    rc = _load().oracle_lmhead_fp8_topk(_ptr(hb), R, H, _ptr(wb), V, topk, _ptr(lp), _ptr(tk), _ptr(lse),
                                       ctypes.byref(sW), _ptr(t), nthreads)
    if rc:
        raise ValueError(f"oracle_lmhead_fp8_topk failed ({rc})")
    return lp, tk, lse, float(sW.value), t


def logits_topk(logits: np.ndarray, topk: int):
    """Log-softmax (double) and top-k of fp32 logits [R, V]."""
    z = np.ascontiguousarray(logits, dtype=np.float32)
    R, V = z.shape
    lp = np.empty((R, topk), np.float32)
    tk = np.empty((R, topk), np.int32)
    lse = np.empty((R,), np.float64)
    rc = _load().oracle_logits_topk(_ptr(z), R, V, topk, _ptr(lp), _ptr(tk), _ptr(lse))
    if rc:
        raise ValueError(f"oracle_logits_topk failed ({rc})")
    return lp, tk, lse


def build_tree(tk_logp: np.ndarray, tk_tok: np.ndarray, B: int, anchor=None, base_pos=None):
    """Mixture DDTree for n_req requests.

    tk_logp / tk_tok: [n_req, K, L, topk] (or [K, L, topk] for one request).
    Returns a dict of arrays with a leading n_req axis: parent, token, depth,
    score, mode, pos [n_req, B+1], mask uint32 [n_req, B+1, ceil((B+1)/32)],
    n_nodes [n_req]."""
    lp = np.ascontiguousarray(tk_logp, dtype=np.float32)
    tk = np.ascontiguousarray(tk_tok, dtype=np.int32)
    single = lp.ndim == 3
    if single:
        lp, tk = lp[None], tk[None]
    n_req, K, L, topk = lp.shape
    N = B + 1
    W32 = (N + 31) // 32
    anchor = np.zeros(n_req, np.int32) if anchor is None else np.asarray(anchor, np.int32).reshape(n_req)
    base_pos = np.zeros(n_req, np.int32) if base_pos is None else np.asarray(base_pos, np.int32).reshape(n_req)
    out = {
        "parent": np.empty((n_req, N), np.int32),
        "token": np.empty((n_req, N), np.int32),
        "depth": np.empty((n_req, N), np.int32),
        "score": np.empty((n_req, N), np.float32),
        "mode": np.empty((n_req, N), np.int32),
        "mask": np.empty((n_req, N, W32), np.uint32),
        "pos": np.empty((n_req, N), np.int32),
        "n_nodes": np.empty((n_req,), np.int32),
    }
    lib = _load()
    for q in range(n_req):
        nn = np.zeros(1, np.int32)
        views = [np.ascontiguousarray(out[k][q]) for k in ("parent", "token", "depth", "score", "mode", "mask", "pos")]
        rc = lib.oracle_build_tree(_ptr(np.ascontiguousarray(lp[q])), _ptr(np.ascontiguousarray(tk[q])), K, L, topk, B,
                                   int(anchor[q]), int(base_pos[q]), *[_ptr(v) for v in views], _ptr(nn))
        if rc:
            raise ValueError(f"oracle_build_tree failed ({rc})")
        for k, v in zip(("parent", "token", "depth", "score", "mode", "mask", "pos"), views):
            out[k][q] = v
        out["n_nodes"][q] = nn[0]
    if single:
        out = {k: v[0] for k, v in out.items()}
    return out


def verify(target_logits: np.ndarray, parent: np.ndarray, token: np.ndarray, n_nodes: int, L: int,
           temperature: float = 0.0, seed: int = 0):
    """Tree verification walk for one request.

    target_logits: fp32 [N, V] (row n = the target's logits after node n).
    Returns (accept_len, path_nodes [L+1], out_tokens [L+1], gap [L+1])."""
    t = np.ascontiguousarray(target_logits, dtype=np.float32)
    N, V = t.shape
    par = np.ascontiguousarray(parent, dtype=np.int32)
    tok = np.ascontiguousarray(token, dtype=np.int32)
    acc = np.zeros(1, np.int32)
    path = np.empty(L + 1, np.int32)
    outt = np.empty(L + 1, np.int32)
    gap = np.empty(L + 1, np.float32)
    rc = _load().oracle_verify(_ptr(t), int(n_nodes), V, L, _ptr(par), _ptr(tok), float(temperature),
                               int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(acc), _ptr(path), _ptr(outt), _ptr(gap))
    if rc:
        raise ValueError(f"oracle_verify failed ({rc})")
    return int(acc[0]), path, outt, gap


def philox4x32_10(ctr: np.ndarray, key: np.ndarray) -> np.ndarray:
    """Philox4x32-10 block function: ctr uint32 [n, 4], key uint32 [n, 2] -> uint32 [n, 4]."""
    c = np.ascontiguousarray(ctr, dtype=np.uint32).reshape(-1, 4)
    k = np.ascontiguousarray(key, dtype=np.uint32).reshape(-1, 2)
    assert c.shape[0] == k.shape[0]
    out = np.empty_like(c)
    _load().oracle_philox_batch(_ptr(c), _ptr(k), c.shape[0], _ptr(out))
    return out


def gumbel(seed: int, node: int, V: int) -> np.ndarray:
    """fp32 Gumbel noise G(seed, node, v) for v in [0, V)."""
    g = np.empty(V, np.float32)
    _load().oracle_gumbel_batch(int(seed) & 0xFFFFFFFFFFFFFFFF, int(node), V, _ptr(g))
    return g
