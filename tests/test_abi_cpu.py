"""The C-ABI library loads and exports every symbol include/gdn.h declares,
and its host-side argument checks reject bad calls before any CUDA work.
No test here launches a kernel (they run without a GPU)."""
import ctypes
import os
import re

import pytest

from chunked_linear_recurrence_gated_gb300 import build, gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gdn.load()


def header_functions(name="gdn.h"):
    text = open(os.path.join(ROOT, "include", name)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert header_functions() == sorted(gdn.EXPORTS)
    assert header_functions("gdn_conv.h") == sorted(gdn.CONV_EXPORTS)


def test_library_exports_every_header_symbol(lib):
    for name in (header_functions() + header_functions("gdn_conv.h")
                 + header_functions("gdn_profile.h")):
        assert hasattr(lib, name), name


def test_diag_checks_workspace(lib):
    assert lib.gdn_diag_wait_timeout(None, 20, None) == 3
    assert lib.gdn_diag_wait_timeout(ctypes.c_void_p(FAKE + 16), 20, None) == 3


def test_version_and_status_strings(lib):
    assert lib.gdn_version() >= 100
    assert gdn.gdn_status_str(0) == "GDN_OK"
    assert gdn.gdn_status_str(3) == "GDN_ERR_WORKSPACE"


def shape(B=1, T=128, H=2, dk=128, dv=128, dtype=1):
    return gdn.gdn_shape(B, T, H, dk, dv, dtype)


def test_workspace_bytes(lib):
    s = shape()
    f = lib.gdn_chunk_workspace_bytes(ctypes.byref(s), 0)
    b = lib.gdn_chunk_workspace_bytes(ctypes.byref(s), 1)
    assert 0 < f < b
    assert f % 256 == 0
    bad = shape(dk=96)
    assert lib.gdn_chunk_workspace_bytes(ctypes.byref(bad), 0) == 0
    assert lib.gdn_varlen_workspace_bytes(ctypes.byref(shape()), 3, 1) > 0
    assert lib.gdn_varlen_workspace_bytes(ctypes.byref(shape(B=2)), 3, 1) == 0


def test_path_selection_independent_of_T(lib):
    for dtype in (0, 1):
        for dk in (64, 128):
            for dv in (64, 128, 256):
                paths = {lib.gdn_path(ctypes.byref(shape(T=T, dk=dk, dv=dv, dtype=dtype)))
                         for T in (1, 64, 1000, 262144)}
                assert len(paths) == 1 and paths.pop() in (1, 2)
    assert lib.gdn_path(ctypes.byref(shape(dv=96))) == 0


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: every call below fails its checks


def call_fwd(lib, s, ptrs=None, ws=FAKE, wsb=1 << 40):
    p = ptrs or [FAKE] * 5 + [None, FAKE, None]
    return lib.gdn_chunk_fwd(ctypes.byref(s), *[ctypes.c_void_p(x) if x else None for x in p],
                             ctypes.c_void_p(ws) if ws else None, wsb, None)


def test_invalid_shapes(lib):
    assert call_fwd(lib, shape(B=0)) == 1
    assert call_fwd(lib, shape(T=-1)) == 1
    assert call_fwd(lib, shape(H=0)) == 1
    assert call_fwd(lib, shape(dk=96)) == 2
    assert call_fwd(lib, shape(dv=32)) == 2
    assert call_fwd(lib, shape(dtype=7)) == 2
    assert lib.gdn_chunk_fwd(None, *([None] * 8), None, 0, None) == 1


def test_null_and_misaligned_pointers(lib):
    s = shape()
    assert call_fwd(lib, s, [None] + [FAKE] * 4 + [None, FAKE, None]) == 1
    assert call_fwd(lib, s, [FAKE + 2] + [FAKE] * 4 + [None, FAKE, None]) == 1
    assert call_fwd(lib, s, [FAKE] * 5 + [FAKE + 4, FAKE, None]) == 1  # S_in misaligned
    assert call_fwd(lib, s, [FAKE] * 5 + [None, FAKE + 8, None]) == 1  # o misaligned


def test_workspace_checks(lib):
    s = shape()
    assert call_fwd(lib, s, ws=None) == 3
    assert call_fwd(lib, s, ws=FAKE + 16) == 3
    need = lib.gdn_chunk_workspace_bytes(ctypes.byref(s), 0)
    assert call_fwd(lib, s, wsb=need - 1) == 3
    sb = shape()
    need_b = lib.gdn_chunk_workspace_bytes(ctypes.byref(sb), 1)
    rc = lib.gdn_chunk_bwd(ctypes.byref(sb), *[ctypes.c_void_p(FAKE)] * 5, None,
                           ctypes.c_void_p(FAKE), None, *[ctypes.c_void_p(FAKE)] * 5, None,
                           ctypes.c_void_p(FAKE), need_b - 256, None)
    assert rc == 3


def test_varlen_host_checks(lib):
    s = shape(B=1, T=300)
    args = [ctypes.c_void_p(FAKE)] * 5 + [None, ctypes.c_void_p(FAKE), None,
                                          ctypes.c_void_p(FAKE), ctypes.c_size_t(1 << 40), None]
    assert lib.gdn_varlen_fwd(ctypes.byref(s), None, 3, *args) == 1        # no cu_seqlens
    assert lib.gdn_varlen_fwd(ctypes.byref(s), ctypes.c_void_p(FAKE), 0, *args) == 1  # nseq 0
    s2 = shape(B=2, T=300)
    assert lib.gdn_varlen_fwd(ctypes.byref(s2), ctypes.c_void_p(FAKE), 3, *args) == 1  # B != 1


def test_saved_products_sizes_and_checks(lib):
    s = shape()
    saved = lib.gdn_chunk_saved_bytes(ctypes.byref(s))
    ws_saved = lib.gdn_chunk_workspace_bytes(ctypes.byref(s), gdn.GDN_WS_SAVED)
    ws_bwd = lib.gdn_chunk_workspace_bytes(ctypes.byref(s), 1)
    assert saved > 0 and saved % 256 == 0
    assert 0 < ws_saved < ws_bwd
    assert lib.gdn_chunk_saved_bytes(ctypes.byref(shape(dk=64, dv=64, dtype=0))) == 256
    assert lib.gdn_chunk_saved_bytes(ctypes.byref(shape(dk=96))) == 0
    P = ctypes.c_void_p
    fwd_args = [P(FAKE)] * 5 + [None, P(FAKE), None]

    def fwd_save(sv, svb):
        return lib.gdn_chunk_fwd_save(ctypes.byref(s), *fwd_args, sv, svb, P(FAKE),
                                      ctypes.c_size_t(1 << 40), None)

    assert fwd_save(None, 1 << 40) == 3                 # no saved buffer
    assert fwd_save(P(FAKE + 16), 1 << 40) == 3         # misaligned
    assert fwd_save(P(FAKE), saved - 256) == 3          # too small
    bwd_args = [P(FAKE)] * 5 + [None, P(FAKE), None] + [P(FAKE)] * 5 + [None]
    rc = lib.gdn_chunk_bwd_saved(ctypes.byref(s), *bwd_args, P(FAKE), saved, P(FAKE),
                                 ws_saved - 256, None)
    assert rc == 3                                      # workspace too small
    rc = lib.gdn_chunk_bwd_saved(ctypes.byref(s), *bwd_args, None, saved, P(FAKE), ws_saved, None)
    assert rc == 3


def conv_shape(B=2, T=100, C=64, W=4, dtype=1, act=1):
    return gdn.gdn_conv_shape(B, T, C, W, dtype, act)


def test_conv_host_checks(lib):
    P = ctypes.c_void_p
    ws = lib.gdn_conv_workspace_bytes(ctypes.byref(conv_shape()))
    assert ws > 0 and ws % 256 == 0
    assert lib.gdn_conv_workspace_bytes(ctypes.byref(conv_shape(W=9))) == 0
    assert lib.gdn_conv_workspace_bytes(ctypes.byref(conv_shape(C=66))) == 0

    def fwd(s, x=FAKE, w=FAKE, b=None, si=None, y=FAKE, so=FAKE):
        return lib.gdn_conv_fwd(ctypes.byref(s), *[P(v) if v else None for v in (x, w, b, si, y, so)],
                                None)

    assert fwd(conv_shape(B=0)) == 1
    assert fwd(conv_shape(act=3)) == 1
    assert fwd(conv_shape(W=1)) == 2
    assert fwd(conv_shape(C=6)) == 2
    assert fwd(conv_shape(dtype=5)) == 2
    assert fwd(conv_shape(), x=FAKE + 8) == 1          # misaligned input
    assert fwd(conv_shape(), w=None) == 1              # weights required
    assert fwd(conv_shape(), si=FAKE, so=FAKE) == 1    # state_out aliases state_in
    s = conv_shape()
    args = [P(FAKE)] * 2 + [None, None, P(FAKE), None, P(FAKE), P(FAKE), None, None]
    assert lib.gdn_conv_bwd(ctypes.byref(s), *args, None, ws, None) == 3
    assert lib.gdn_conv_bwd(ctypes.byref(s), *args, P(FAKE), ws - 256, None) == 3
    assert lib.gdn_conv_bwd(ctypes.byref(s), *args, P(FAKE + 16), ws, None) == 3


def test_noalloc_limit_matches_its_documentation(lib):
    """The no-allocation forward accepts exactly the shapes whose forward
    workspace fits GDN_NOALLOC_SCRATCH_BYTES (documented as 849 block-heads
    for one sequence and head, 816 for 16 heads, at dk = dv = 128 bf16)."""
    lim = 64 << 20
    fits = lambda nb, H: lib.gdn_chunk_workspace_bytes(
        ctypes.byref(shape(B=1, T=64 * nb, H=H)), 0) <= lim
    assert fits(849, 1) and not fits(850, 1)
    assert fits(816 // 16, 16) and not fits(816 // 16 + 1, 16)
