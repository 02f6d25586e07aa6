"""The workspace-free entry point, mfd_logits_topk_noalloc, against
mfd_logits_topk.

Some callers cannot allocate device memory where they call the library --
code that runs after its memory budget is fixed, or that must not pay the
implicit device synchronisation of an allocation.  For them the library keeps
one fixed scratch array per GPU and this entry point uses it instead of a
caller workspace.  This file is collected last on purpose, and it must pass
both on its own in a fresh process and after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from tree_verified_speculative_gb300 import mfd

from gpu_helpers import check_topk, np_

pytestmark = pytest.mark.gpu


def _with_workspace(z: torch.Tensor, topk: int):
    R, V = z.shape
    lp = torch.empty((R, topk), dtype=torch.float32, device="cuda")
    tk = torch.empty((R, topk), dtype=torch.int32, device="cuda")
    lse = torch.empty((R,), dtype=torch.float32, device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ws = torch.empty(mfd.mfd_workspace_size(mfd.MFD_OP_LOGITS_TOPK, R=R, V=V, topk=topk), dtype=torch.uint8,
                     device="cuda")
    mfd.mfd_logits_topk(z, topk, lp, tk, lse, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return np_(lp), np_(tk), np_(lse)


def _no_alloc(z: torch.Tensor, topk: int):
    """Through the C ABI directly: no workspace argument exists."""
    R, V = z.shape
    lp = torch.empty((R, topk), dtype=torch.float32, device="cuda")
    tk = torch.empty((R, topk), dtype=torch.int32, device="cuda")
    lse = torch.empty((R,), dtype=torch.float32, device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    lib = mfd.load()
    rc = lib.mfd_logits_topk_noalloc(ctypes.c_void_p(z.data_ptr()), R, V, topk, ctypes.c_void_p(lp.data_ptr()),
                                     ctypes.c_void_p(tk.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
                                     ctypes.c_void_p(st.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == mfd.MFD_OK, mfd.status_string(rc)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return np_(lp), np_(tk), np_(lse)


def test_no_alloc_matches_workspace_path_on_two_calls_in_a_row():
    rng = np.random.default_rng(2027)
    # two different problems back to back: the second call finds the first
    # call's data still in the shared scratch and must not depend on it
    cases = [((120, 151936), 16), ((7, 5003), 32)]
    for (R, V), topk in cases:
        z = torch.from_numpy((2.0 * rng.standard_normal((R, V))).astype(np.float32)).cuda()
        ref = _with_workspace(z, topk)
        got = _no_alloc(z, topk)
        check_topk(got[0], got[1], ref[0], ref[1])
        np.testing.assert_allclose(got[2], ref[2], rtol=0, atol=1e-5)


def test_no_alloc_rejects_problems_larger_than_its_scratch():
    R, V, topk = 4096, 151936, 32
    need = mfd.mfd_workspace_size(mfd.MFD_OP_LOGITS_TOPK, R=R, V=V, topk=topk)
    assert need > mfd.NOALLOC_SCRATCH_BYTES
    z = torch.empty((1,), dtype=torch.float32, device="cuda")
    out = torch.empty((1,), dtype=torch.int32, device="cuda")
    rc = mfd.load().mfd_logits_topk_noalloc(ctypes.c_void_p(z.data_ptr()), R, V, topk, ctypes.c_void_p(z.data_ptr()),
                                            ctypes.c_void_p(out.data_ptr()), None, ctypes.c_void_p(out.data_ptr()),
                                            None)
    assert rc == mfd.MFD_ERR_WORKSPACE
