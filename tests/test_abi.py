"""CPU checks of the C ABI: the library builds, loads and exports every
function include/mfd.h declares; argument checks that return before any
CUDA call behave as documented.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

from tree_verified_speculative_gb300 import build as mfd_build
from tree_verified_speculative_gb300 import mfd

HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(HERE, "..", "include", "mfd.h")


@pytest.fixture(scope="module")
def lib():
    mfd_build.build()
    return mfd.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mfd_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert set(names) >= {"mfd_lmhead_topk", "mfd_build_tree", "mfd_verify"}
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(mfd.EXPORTS)


def test_status_strings(lib):
    for code in range(7):
        assert lib.mfd_status_string(code)
    assert b"unknown" in lib.mfd_status_string(99)


def test_workspace_size_host_only_ops(lib):
    assert mfd.mfd_workspace_size(mfd.MFD_OP_BUILD_TREE, n_req=3) > 0
    assert mfd.mfd_workspace_size(mfd.MFD_OP_LOGITS_TOPK, R=4, V=32, topk=8) > 0
    assert mfd.mfd_workspace_size(mfd.MFD_OP_LOGITS_TOPK, R=4, V=32, topk=33) == 0
    assert mfd.mfd_workspace_size(99) == 0


def test_argument_errors_before_any_cuda_call(lib):
    fake = ctypes.c_void_p(0x100000)
    # NULL inputs
    rc = lib.mfd_build_tree(None, None, 1, 8, 15, 16, 64, None, None, *([None] * 9), None, 0, None)
    assert rc == mfd.MFD_ERR_INVALID_ARG
    args = [fake] * 2 + [1, 17, 15, 16, 64] + [fake, None] + [fake] * 9 + [fake, 1 << 20, None]
    assert lib.mfd_build_tree(*args) == mfd.MFD_ERR_UNSUPPORTED  # K > 16
    args = [fake] * 2 + [1, 8, 15, 16, 512] + [fake, None] + [fake] * 9 + [fake, 1 << 20, None]
    assert lib.mfd_build_tree(*args) == mfd.MFD_ERR_UNSUPPORTED  # K * B > 2048
    args = [fake] * 2 + [1, 8, 15, 16, 64] + [fake, None] + [fake] * 9 + [fake, 16, None]
    assert lib.mfd_build_tree(*args) == mfd.MFD_ERR_WORKSPACE
    rc = lib.mfd_logits_topk(fake, 4, 32, 40, fake, fake, None, fake, fake, 1 << 20, None)
    assert rc == mfd.MFD_ERR_UNSUPPORTED  # topk > 32
    rc = lib.mfd_lmhead_topk(ctypes.c_void_p(0x100004), 4, 64, fake, 1000, 8, fake, fake, None, fake, fake,
                             1 << 20, None)
    assert rc == mfd.MFD_ERR_INVALID_ARG  # h not 16-byte aligned


@pytest.mark.parametrize("K,L,topk,B", [(16, 16, 32, 128), (4, 16, 32, 512), (8, 15, 16, 256), (8, 15, 32, 256),
                                        (1, 16, 32, 512), (16, 1, 1, 1)])
def test_tree_limits_fit_shared_memory(lib, K, L, topk, B):
    """Every shape inside the documented limits passes the tree's shared-memory
    budget check (the call then stops at the deliberately tiny workspace)."""
    fake = ctypes.c_void_p(0x100000)
    args = [fake] * 2 + [1, K, L, topk, B] + [fake, None] + [fake] * 9 + [fake, 16, None]
    assert lib.mfd_build_tree(*args) == mfd.MFD_ERR_WORKSPACE


def test_packed_weight_entry_points_arguments(lib):
    """mfd_lmhead_packed_bytes, mfd_lmhead_pack and mfd_lmhead_topk_packed:
    sizes and the argument errors returned before any CUDA call."""
    assert mfd.mfd_lmhead_packed_bytes(151936, 2560) == 594 * 256 * 2560 * 2
    assert mfd.mfd_lmhead_packed_bytes(256, 64) == 256 * 64 * 2
    assert mfd.mfd_lmhead_packed_bytes(257, 64) == 512 * 64 * 2  # the last tile is padded
    assert mfd.mfd_lmhead_packed_bytes(1000, 100) == 0  # H not a multiple of 64
    assert mfd.mfd_lmhead_packed_bytes(8, 64) == 0  # V < 16
    fake = ctypes.c_void_p(0x100000)
    assert lib.mfd_lmhead_pack(None, 1000, 128, fake, 1 << 30, None) == mfd.MFD_ERR_INVALID_ARG
    assert lib.mfd_lmhead_pack(fake, 1000, 128, ctypes.c_void_p(0x100010), 1 << 30, None) == mfd.MFD_ERR_INVALID_ARG
    assert lib.mfd_lmhead_pack(fake, 1000, 100, fake, 1 << 30, None) == mfd.MFD_ERR_UNSUPPORTED
    assert lib.mfd_lmhead_pack(fake, 1000, 128, fake, 1024, None) == mfd.MFD_ERR_WORKSPACE
    args = [fake, 4, 64, None, 1000, 8, fake, fake, None, fake, fake, 1 << 20, None]
    assert lib.mfd_lmhead_topk_packed(*args) == mfd.MFD_ERR_INVALID_ARG  # no packed weight
    args[3] = ctypes.c_void_p(0x100080)
    assert lib.mfd_lmhead_topk_packed(*args) == mfd.MFD_ERR_INVALID_ARG  # not 256-byte aligned
    args[3] = fake
    args[5] = 40
    assert lib.mfd_lmhead_topk_packed(*args) == mfd.MFD_ERR_UNSUPPORTED  # topk > 32


def test_subset_head_entry_point_arguments(lib):
    """mfd_lmhead_topk_subset: argument errors returned before any CUDA call."""
    fake = ctypes.c_void_p(0x100000)
    def call(Wp=fake, V_sub=1000, ids=fake, V_full=5000, topk=8):
        return lib.mfd_lmhead_topk_subset(fake, 4, 64, Wp, V_sub, ids, V_full, topk, fake, fake, None, fake, fake,
                                          1 << 20, None)
    assert call(Wp=None) == mfd.MFD_ERR_INVALID_ARG  # no packed weight
    assert call(ids=None) == mfd.MFD_ERR_INVALID_ARG  # no id table
    assert call(ids=ctypes.c_void_p(0x100002)) == mfd.MFD_ERR_INVALID_ARG  # id table not 4-byte aligned
    assert call(V_full=999) == mfd.MFD_ERR_INVALID_ARG  # the full vocabulary is smaller than the subset
    assert call(V_full=1 << 30) == mfd.MFD_ERR_INVALID_ARG
    assert call(Wp=ctypes.c_void_p(0x100080)) == mfd.MFD_ERR_INVALID_ARG  # packed weight not 256-byte aligned
    assert call(topk=40) == mfd.MFD_ERR_UNSUPPORTED


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++17")])
def test_header_compiles_standalone(lang, std, tmp_path):
    """include/mfd.h is plain C: it compiles on its own as C99 and as C++17,
    with no CUDA or torch headers."""
    import shutil
    import subprocess

    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("use.c" if lang == "c" else "use.cpp")
    src.write_text('#include "mfd.h"\nint main(void) { return (int)mfd_workspace_size(MFD_OP_BUILD_TREE, 1, 8, 15, 16,'
                   ' 256, 120, 151936) == 0; }\n')
    r = subprocess.run([cc, "-x", lang, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(HERE, "..", "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_mfdd_switch_rule(lib):
    """MFD-D (project page "Multi-Future Drafting", In a serving engine): all
    K modes below three requests in flight, the single-mode path from three
    on; invalid arguments give 0."""
    assert [mfd.mfd_mfdd_modes(n, 8) for n in (1, 2, 3, 4, 32)] == [8, 8, 1, 1, 1]
    assert mfd.mfd_mfdd_modes(2, 1) == 1
    assert mfd.mfd_mfdd_modes(0, 8) == 0 and mfd.mfd_mfdd_modes(1, 0) == 0 and mfd.mfd_mfdd_modes(1, 17) == 0
