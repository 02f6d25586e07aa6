"""Thin ctypes binding of libmfd (include/mfd.h).

Each ``mfd_*`` function has the C entry point's name and arguments; torch
tensors stand in for device pointers, and the current torch CUDA stream is
used unless one is given.  The binding only marshals arguments: every step of
the round runs in the library's CUDA kernels.  There is no fallback: if the
library has not been built, or the device is not an sm_103a GPU, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmfd.so")
CHECKED_LIB_PATH = os.path.join(_HERE, "_build", "libmfd_checked.so")

MFD_OK = 0
MFD_ERR_INVALID_ARG = 1
MFD_ERR_UNSUPPORTED = 2
MFD_ERR_WORKSPACE = 3
MFD_ERR_CUDA = 4
MFD_ERR_TIMEOUT = 5
MFD_ERR_INPUT = 6
MFD_ERR_CHECK = 7

MFD_OP_LMHEAD_TOPK = 0
MFD_OP_LOGITS_TOPK = 1
MFD_OP_BUILD_TREE = 2
MFD_OP_VERIFY = 3
MFD_OP_TREE_ANALYTICS = 4
MFD_NODE_ON_FUTURE, MFD_NODE_CHIMERA, MFD_NODE_OTHER = 0, 1, 2

EXPORTS = ("mfd_status_string", "mfd_workspace_size", "mfd_lmhead_topk", "mfd_lmhead_packed_bytes",
           "mfd_lmhead_pack", "mfd_lmhead_topk_packed", "mfd_lmhead_topk_subset", "mfd_logits_topk",
           "mfd_logits_topk_noalloc",
           "mfd_build_tree", "mfd_verify", "mfd_verify_withheld_test", "mfd_lmhead_withheld_test", "mfd_mfdd_modes",
           "mfd_lmhead_packed_fp8_bytes", "mfd_lmhead_pack_fp8", "mfd_fp8_quantize_rows",
           "mfd_lmhead_fp8_workspace_bytes", "mfd_lmhead_topk_fp8", "mfd_tree_analytics")
NOALLOC_SCRATCH_BYTES = 4 << 20

_lock = threading.Lock()
_lib = None
_libs: dict[str, ctypes.CDLL] = {}


class MfdError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (code {code})")
        self.code = code


def use_library(path: str | None) -> None:
    """Route every call of this module through the library at `path` (for
    instance CHECKED_LIB_PATH, the bounds-checked build), or back to
    libmfd.so with None."""
    global _lib
    lib = load(path or LIB_PATH)
    with _lock:
        _lib = lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libmfd.so (or the library at `path`); raises if it is missing (no
    fallback)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if p in _libs:
            if path is None:
                _lib = _libs[p]
            return _libs[p]
        if not os.path.exists(p):
            raise RuntimeError(f"libmfd.so not built ({p}); run `python -m tree_verified_speculative_gb300.build`")
        lib = ctypes.CDLL(p)
        P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.mfd_status_string.argtypes = [I]
        lib.mfd_status_string.restype = ctypes.c_char_p
        lib.mfd_workspace_size.argtypes = [I] * 8
        lib.mfd_workspace_size.restype = SZ
        lib.mfd_lmhead_topk.argtypes = [P, I, I, P, I, I, P, P, P, P, P, SZ, P]
        lib.mfd_lmhead_topk.restype = I
        lib.mfd_lmhead_packed_bytes.argtypes = [I, I]
        lib.mfd_lmhead_packed_bytes.restype = SZ
        lib.mfd_lmhead_pack.argtypes = [P, I, I, P, SZ, P]
        lib.mfd_lmhead_pack.restype = I
        lib.mfd_lmhead_topk_packed.argtypes = [P, I, I, P, I, I, P, P, P, P, P, SZ, P]
        lib.mfd_lmhead_topk_packed.restype = I
        lib.mfd_lmhead_withheld_test.argtypes = [P, I, I, P, I, I, P, P, P, P, P, SZ, P]
        lib.mfd_lmhead_withheld_test.restype = I
        lib.mfd_lmhead_topk_subset.argtypes = [P, I, I, P, I, P, I, I, P, P, P, P, P, SZ, P]
        lib.mfd_lmhead_topk_subset.restype = I
        lib.mfd_logits_topk.argtypes = [P, I, I, I, P, P, P, P, P, SZ, P]
        lib.mfd_logits_topk.restype = I
        lib.mfd_logits_topk_noalloc.argtypes = [P, I, I, I, P, P, P, P, P]
        lib.mfd_logits_topk_noalloc.restype = I
        lib.mfd_build_tree.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]
        lib.mfd_build_tree.restype = I
        lib.mfd_verify.argtypes = [P, I, I, I, I, P, P, P, P, P, P, P, P, P, P, SZ, P]
        lib.mfd_verify.restype = I
        lib.mfd_verify_withheld_test.argtypes = [P, I, I, I, I, P, P, P, P, P, P, P, P, P, P, SZ,
                                                 ctypes.c_uint64, P]
        lib.mfd_verify_withheld_test.restype = I
        lib.mfd_mfdd_modes.argtypes = [I, I]
        lib.mfd_mfdd_modes.restype = I
        lib.mfd_lmhead_packed_fp8_bytes.argtypes = [I, I]
        lib.mfd_lmhead_packed_fp8_bytes.restype = SZ
        lib.mfd_lmhead_pack_fp8.argtypes = [P, I, I, P, SZ, P]
        lib.mfd_lmhead_pack_fp8.restype = I
        lib.mfd_fp8_quantize_rows.argtypes = [P, I, I, P, P, P]
        lib.mfd_fp8_quantize_rows.restype = I
        lib.mfd_lmhead_fp8_workspace_bytes.argtypes = [I, I, I, I]
        lib.mfd_lmhead_fp8_workspace_bytes.restype = SZ
        lib.mfd_lmhead_topk_fp8.argtypes = [P, I, I, P, I, I, P, P, P, P, P, SZ, P]
        lib.mfd_lmhead_topk_fp8.restype = I
        lib.mfd_tree_analytics.argtypes = [P, P, P, P, I, I, I, P, I, P, I, P, P, P, P, P, P, SZ, P]
        lib.mfd_tree_analytics.restype = I
        _libs[p] = lib
        if path is None:
            _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().mfd_status_string(int(code)).decode()


def _p(t) -> int | None:
    if t is None:
        return None
    assert isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous(), "device tensors, contiguous"
    return t.data_ptr()


def _p_dev_or_pinned(t) -> int:
    """A device tensor, or a page-locked host tensor (read in place by the
    kernel through its mapped address)."""
    assert isinstance(t, torch.Tensor) and t.is_contiguous() and (t.is_cuda or t.is_pinned()), \
        "device or pinned host tensor, contiguous"
    return t.data_ptr()


def _s(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(rc: int, where: str) -> None:
    if rc != MFD_OK:
        raise MfdError(rc, where)


def mfd_tree_analytics(parent, token, depth, n_nodes, L, futures, target_logits, temperature, node_class, reach,
                       mass, status, ws, stream=None) -> None:
    """Chimera classes and covered mass of trees (see include/mfd.h):
    futures int32 [n_req][F][L], target_logits fp32 [n_req][B+1][V]."""
    n_req, N = parent.shape
    F = futures.shape[1]
    V = target_logits.shape[-1]
    rc = load().mfd_tree_analytics(_p(parent), _p(token), _p(depth), _p(n_nodes), n_req, N - 1, L, _p(futures), F,
                                   _p(target_logits), V, _p(temperature), _p(node_class), _p(reach), _p(mass),
                                   _p(status), _p(ws), ws.numel() * ws.element_size(), _s(stream))
    _check(rc, "mfd_tree_analytics")


def tree_analytics(parent, token, depth, n_nodes, L, futures, target_logits, temperature, stream=None):
    """mfd_tree_analytics with its outputs and scratch allocated here:
    returns (node_class, reach, mass, status) device tensors."""
    n_req, N = parent.shape
    dev = parent.device
    cls = torch.empty((n_req, N), dtype=torch.int32, device=dev)
    reach = torch.empty((n_req, N), dtype=torch.float64, device=dev)
    mass = torch.empty((n_req, L + 1), dtype=torch.float64, device=dev)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    ws = torch.empty((mfd_workspace_size(MFD_OP_TREE_ANALYTICS, n_req, 1, 1, 1, N - 1),), dtype=torch.uint8,
                     device=dev)
    mfd_tree_analytics(parent, token, depth, n_nodes, L, futures, target_logits, temperature, cls, reach, mass,
                       status, ws, stream)
    return cls, reach, mass, status


def mfd_mfdd_modes(n_req: int, K: int) -> int:
    """Modes an MFD-D round drafts with: K below three requests, else 1."""
    return int(load().mfd_mfdd_modes(int(n_req), int(K)))


def mfd_workspace_size(op: int, n_req: int = 1, K: int = 1, L: int = 1, topk: int = 1, B: int = 1,
                       R: int = 1, V: int = 16) -> int:
    return int(load().mfd_workspace_size(op, n_req, K, L, topk, B, R, V))


def mfd_lmhead_topk(h, W, topk, tk_logp, tk_tok, lse, status, ws, stream=None) -> None:
    R, H = h.shape
    V = W.shape[0]
    assert h.dtype == torch.bfloat16 and W.dtype == torch.bfloat16 and W.shape[1] == H
    rc = load().mfd_lmhead_topk(_p(h), R, H, _p(W), V, topk, _p(tk_logp), _p(tk_tok), _p(lse), _p(status),
                                _p(ws), ws.numel() * ws.element_size(), _s(stream))
    _check(rc, "mfd_lmhead_topk")


def mfd_lmhead_packed_bytes(V: int, H: int) -> int:
    return int(load().mfd_lmhead_packed_bytes(V, H))


def mfd_lmhead_pack(W, W_packed, stream=None) -> None:
    V, H = W.shape
    assert W.dtype == torch.bfloat16
    rc = load().mfd_lmhead_pack(_p(W), V, H, _p(W_packed), W_packed.numel() * W_packed.element_size(), _s(stream))
    _check(rc, "mfd_lmhead_pack")


def pack_lm_head(W, stream=None):
    """The packed copy of W (a new device buffer, allocated here, once)."""
    V, H = W.shape
    n = mfd_lmhead_packed_bytes(V, H)
    if n == 0:
        raise MfdError(MFD_ERR_UNSUPPORTED, "mfd_lmhead_packed_bytes")
    Wp = torch.empty((n,), dtype=torch.uint8, device=W.device)
    mfd_lmhead_pack(W, Wp, stream)
    return Wp


def mfd_lmhead_topk_packed(h, W_packed, V, topk, tk_logp, tk_tok, lse, status, ws, stream=None) -> None:
    R, H = h.shape
    assert h.dtype == torch.bfloat16
    rc = load().mfd_lmhead_topk_packed(_p(h), R, H, _p(W_packed), V, topk, _p(tk_logp), _p(tk_tok), _p(lse),
                                       _p(status), _p(ws), ws.numel() * ws.element_size(), _s(stream))
    _check(rc, "mfd_lmhead_topk_packed")


def mfd_lmhead_withheld_test(h, W_packed, V, topk, tk_logp, tk_tok, lse, status, ws, stream=None) -> None:
    """mfd_lmhead_topk_packed with the fault injection of its C entry point:
    the producers stop after the first tile, so the kernel's bounded wait
    runs out (*status = MFD_ERR_TIMEOUT after about a second)."""
    R, H = h.shape
    assert h.dtype == torch.bfloat16
    rc = load().mfd_lmhead_withheld_test(_p(h), R, H, _p(W_packed), V, topk, _p(tk_logp), _p(tk_tok), _p(lse),
                                         _p(status), _p(ws), ws.numel() * ws.element_size(), _s(stream))
    _check(rc, "mfd_lmhead_withheld_test")


def mfd_lmhead_packed_fp8_bytes(V: int, H: int) -> int:
    return int(load().mfd_lmhead_packed_fp8_bytes(V, H))


def mfd_lmhead_pack_fp8(W, W_packed, stream=None) -> None:
    V, H = W.shape
    assert W.dtype == torch.bfloat16
    rc = load().mfd_lmhead_pack_fp8(_p(W), V, H, _p(W_packed), W_packed.numel() * W_packed.element_size(),
                                    _s(stream))
    _check(rc, "mfd_lmhead_pack_fp8")


def pack_lm_head_fp8(W, stream=None):
    """The E4M3 packed copy of W with its scale trailer (a new device buffer,
    allocated here, once)."""
    V, H = W.shape
    n = mfd_lmhead_packed_fp8_bytes(V, H)
    if n == 0:
        raise MfdError(MFD_ERR_UNSUPPORTED, "mfd_lmhead_packed_fp8_bytes")
    Wp = torch.empty((n,), dtype=torch.uint8, device=W.device)
    mfd_lmhead_pack_fp8(W, Wp, stream)
    return Wp


def mfd_fp8_quantize_rows(x, q, scale, stream=None) -> None:
    R, H = x.shape
    assert x.dtype == torch.bfloat16 and q.dtype == torch.uint8 and scale.dtype == torch.float32
    rc = load().mfd_fp8_quantize_rows(_p(x), R, H, _p(q), _p(scale), _s(stream))
    _check(rc, "mfd_fp8_quantize_rows")


def mfd_lmhead_fp8_workspace_bytes(R: int, H: int, V: int, topk: int) -> int:
    return int(load().mfd_lmhead_fp8_workspace_bytes(R, H, V, topk))


def mfd_lmhead_topk_fp8(h, W_packed_fp8, V, topk, tk_logp, tk_tok, lse, status, ws, stream=None) -> None:
    R, H = h.shape
    assert h.dtype == torch.bfloat16
    rc = load().mfd_lmhead_topk_fp8(_p(h), R, H, _p(W_packed_fp8), V, topk, _p(tk_logp), _p(tk_tok), _p(lse),
                                    _p(status), _p(ws), ws.numel() * ws.element_size(), _s(stream))
    _check(rc, "mfd_lmhead_topk_fp8")


def mfd_lmhead_topk_subset(h, W_packed, vocab_ids, V_full, topk, tk_logp, tk_tok, lse, status, ws,
                           stream=None) -> None:
    """The LM head over a draft-vocabulary subset: W_packed holds the packed
    rows of the subset, vocab_ids (int32, increasing) their vocabulary ids;
    tk_tok receives vocabulary ids."""
    assert vocab_ids.dtype == torch.int32
    rc = load().mfd_lmhead_topk_subset(_p(h), h.shape[0], h.shape[1], _p(W_packed), vocab_ids.numel(),
                                       _p(vocab_ids), V_full, topk, _p(tk_logp), _p(tk_tok), _p(lse), _p(status),
                                       _p(ws), ws.numel() * ws.element_size(), _s(stream))
    _check(rc, "mfd_lmhead_topk_subset")


def mfd_logits_topk(logits, topk, tk_logp, tk_tok, lse, status, ws, stream=None) -> None:
    R, V = logits.shape
    assert logits.dtype == torch.float32
    rc = load().mfd_logits_topk(_p(logits), R, V, topk, _p(tk_logp), _p(tk_tok), _p(lse), _p(status), _p(ws),
                                ws.numel() * ws.element_size(), _s(stream))
    _check(rc, "mfd_logits_topk")


def mfd_logits_topk_noalloc(logits, topk, tk_logp, tk_tok, lse, status, stream=None) -> None:
    """mfd_logits_topk without a workspace argument, for callers that cannot
    allocate device memory where they call it; it uses the library's fixed
    per-device scratch, so calls must not overlap on the GPU."""
    R, V = logits.shape
    assert logits.dtype == torch.float32
    rc = load().mfd_logits_topk_noalloc(_p(logits), R, V, topk, _p(tk_logp), _p(tk_tok), _p(lse), _p(status),
                                        _s(stream))
    _check(rc, "mfd_logits_topk_noalloc")


def mfd_build_tree(tk_logp, tk_tok, n_req, K, L, topk, B, anchor_tok, base_pos, parent, token, depth, score,
                   mode, mask, pos, n_nodes, status, ws, stream=None) -> None:
    rc = load().mfd_build_tree(_p(tk_logp), _p(tk_tok), n_req, K, L, topk, B, _p(anchor_tok), _p(base_pos),
                               _p(parent), _p(token), _p(depth), _p(score), _p(mode), _p(mask), _p(pos),
                               _p(n_nodes), _p(status), _p(ws), ws.numel() * ws.element_size(), _s(stream))
    _check(rc, "mfd_build_tree")


def mfd_verify(target_logits, n_req, B, V, L, parent, token, n_nodes, temperature, seed, accept_len,
               path_nodes, out_tokens, status, ws, stream=None) -> None:
    rc = load().mfd_verify(_p_dev_or_pinned(target_logits), n_req, B, V, L, _p(parent), _p(token), _p(n_nodes),
                           _p(temperature), _p(seed), _p(accept_len), _p(path_nodes), _p(out_tokens),
                           _p(status), _p(ws), ws.numel() * ws.element_size(), _s(stream))
    _check(rc, "mfd_verify")


def mfd_verify_withheld_test(target_logits, n_req, B, V, L, parent, token, n_nodes, temperature, seed,
                             accept_len, path_nodes, out_tokens, status, ws, wait_limit_ns, stream=None) -> None:
    """mfd_verify with the fault injection of its C entry point: the step
    results of all but each group's first CTA are withheld and every wait is
    limited to wait_limit_ns, so *status ends as MFD_ERR_TIMEOUT."""
    rc = load().mfd_verify_withheld_test(_p_dev_or_pinned(target_logits), n_req, B, V, L, _p(parent), _p(token),
                                         _p(n_nodes), _p(temperature), _p(seed), _p(accept_len), _p(path_nodes),
                                         _p(out_tokens), _p(status), _p(ws), ws.numel() * ws.element_size(),
                                         int(wait_limit_ns), _s(stream))
    _check(rc, "mfd_verify_withheld_test")


# ---------------------------------------------------------------------------
class Round:
    """Device buffers for one drafting round of n_req requests, reused from
    call to call (allocation happens here, once, never inside the calls)."""

    def __init__(self, n_req: int, K: int, L: int, topk: int, B: int, V: int, device="cuda", V_draft: int | None = None,
                 H: int | None = None):
        """V: the target vocabulary (verification); V_draft: the draft
        vocabulary of a subset head (lmhead_topk_subset), if any; H: the
        hidden width, needed only to size the FP8 head's scratch."""
        self.n_req, self.K, self.L, self.topk, self.B, self.V = n_req, K, L, topk, B, V
        R = n_req * K * L
        N = B + 1
        W32 = (N + 31) // 32
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.R = R
        self.tk_logp = torch.empty((R, topk), dtype=torch.float32, device=dev)
        self.tk_tok = torch.empty((R, topk), **i32)
        self.lse = torch.empty((R,), dtype=torch.float32, device=dev)
        self.parent = torch.empty((n_req, N), **i32)
        self.token = torch.empty((n_req, N), **i32)
        self.depth = torch.empty((n_req, N), **i32)
        self.score = torch.empty((n_req, N), dtype=torch.float32, device=dev)
        self.mode = torch.empty((n_req, N), **i32)
        self.mask = torch.empty((n_req, N, W32), **i32)
        self.pos = torch.empty((n_req, N), **i32)
        self.n_nodes = torch.empty((n_req,), **i32)
        self.accept_len = torch.empty((n_req,), **i32)
        self.path_nodes = torch.empty((n_req, L + 1), **i32)
        self.out_tokens = torch.empty((n_req, L + 1), **i32)
        self.status = torch.zeros((1,), **i32)
        self.anchor = torch.zeros((n_req,), **i32)
        self.base_pos = torch.zeros((n_req,), **i32)
        ws = max(mfd_workspace_size(MFD_OP_LMHEAD_TOPK, n_req, K, L, topk, B, R, V),
                 mfd_workspace_size(MFD_OP_LMHEAD_TOPK, n_req, K, L, topk, B, R, V_draft or V),
                 mfd_workspace_size(MFD_OP_LOGITS_TOPK, n_req, K, L, topk, B, R, V),
                 mfd_workspace_size(MFD_OP_BUILD_TREE, n_req, K, L, topk, B, R, V),
                 mfd_workspace_size(MFD_OP_VERIFY, n_req, K, L, topk, B, R, V),
                 mfd_lmhead_fp8_workspace_bytes(R, H, V, topk) if H else 0)
        self.ws = torch.empty((ws + 255) // 256 * 256, dtype=torch.uint8, device=dev)

    def lmhead_topk(self, h, W, stream=None):
        mfd_lmhead_topk(h, W, self.topk, self.tk_logp, self.tk_tok, self.lse, self.status, self.ws, stream)

    def lmhead_topk_packed(self, h, W_packed, stream=None):
        mfd_lmhead_topk_packed(h, W_packed, self.V, self.topk, self.tk_logp, self.tk_tok, self.lse, self.status,
                               self.ws, stream)

    def lmhead_topk_fp8(self, h, W_packed_fp8, stream=None):
        """The FP8 drafter head (E4M3 packed weight); the Round must have
        been made with H."""
        mfd_lmhead_topk_fp8(h, W_packed_fp8, self.V, self.topk, self.tk_logp, self.tk_tok, self.lse, self.status,
                            self.ws, stream)

    def lmhead_topk_subset(self, h, W_packed, vocab_ids, stream=None):
        """Draft over the subset whose packed rows are W_packed; tk_tok gets
        vocabulary ids (< self.V)."""
        mfd_lmhead_topk_subset(h, W_packed, vocab_ids, self.V, self.topk, self.tk_logp, self.tk_tok, self.lse,
                               self.status, self.ws, stream)

    def logits_topk(self, logits, stream=None):
        mfd_logits_topk(logits, self.topk, self.tk_logp, self.tk_tok, self.lse, self.status, self.ws, stream)

    def build_tree(self, stream=None):
        mfd_build_tree(self.tk_logp, self.tk_tok, self.n_req, self.K, self.L, self.topk, self.B, self.anchor,
                       self.base_pos, self.parent, self.token, self.depth, self.score, self.mode, self.mask,
                       self.pos, self.n_nodes, self.status, self.ws, stream)

    def verify(self, target_logits, temperature, seed, stream=None):
        mfd_verify(target_logits, self.n_req, self.B, self.V, self.L, self.parent, self.token, self.n_nodes,
                   temperature, seed, self.accept_len, self.path_nodes, self.out_tokens, self.status, self.ws,
                   stream)
