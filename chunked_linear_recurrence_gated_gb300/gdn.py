"""Thin ctypes binding of libgdn.so (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module
only turns torch tensors into pointers, allocates outputs and the workspace on
the caller's behalf (torch owns that memory), and raises on a non-OK status.
The library must have been built (``build.py``); there is no fallback.

The function names follow the C ABI in include/gdn.h.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

GDN_OK = 0
GDN_DTYPE_F32 = 0
GDN_DTYPE_BF16 = 1

_STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED",
           3: "GDN_ERR_WORKSPACE", 4: "GDN_ERR_CUDA", 5: "GDN_ERR_TIMEOUT"}

EXPORTS = ["gdn_chunk_workspace_bytes", "gdn_chunk_fwd", "gdn_chunk_bwd",
           "gdn_varlen_workspace_bytes", "gdn_varlen_fwd", "gdn_varlen_bwd",
           "gdn_status_str", "gdn_workspace_status", "gdn_path", "gdn_version",
           "gdn_chunk_fwd_noalloc", "gdn_chunk_saved_bytes", "gdn_chunk_fwd_save",
           "gdn_chunk_bwd_saved", "gdn_noalloc_status"]
GDN_WS_SAVED = 2
# include/gdn_conv.h
CONV_EXPORTS = ["gdn_conv_workspace_bytes", "gdn_conv_fwd", "gdn_conv_bwd"]
CONV_ACT = {"none": 0, "silu": 1}


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {_STATUS.get(status, status)}")
        self.status = status


class gdn_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("dtype", ctypes.c_int)]


class gdn_conv_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("C", ctypes.c_int),
                ("W", ctypes.c_int), ("dtype", ctypes.c_int), ("act", ctypes.c_int)]


_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libgdn.so. Raises if it is missing (no CPU fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libgdn.so not built ({path}); run "
                               "`python -m chunked_linear_recurrence_gated_gb300.build`")
        _build.build()
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    SP = ctypes.POINTER(gdn_shape)
    lib.gdn_chunk_workspace_bytes.argtypes = [SP, I]
    lib.gdn_chunk_workspace_bytes.restype = Z
    lib.gdn_varlen_workspace_bytes.argtypes = [SP, I, I]
    lib.gdn_varlen_workspace_bytes.restype = Z
    lib.gdn_chunk_fwd.argtypes = [SP] + [P] * 8 + [P, Z, P]
    lib.gdn_chunk_bwd.argtypes = [SP] + [P] * 14 + [P, Z, P]
    lib.gdn_varlen_fwd.argtypes = [SP, P, I] + [P] * 8 + [P, Z, P]
    lib.gdn_varlen_bwd.argtypes = [SP, P, I] + [P] * 14 + [P, Z, P]
    for f in (lib.gdn_chunk_fwd, lib.gdn_chunk_bwd, lib.gdn_varlen_fwd, lib.gdn_varlen_bwd):
        f.restype = I
    lib.gdn_status_str.argtypes = [I]
    lib.gdn_status_str.restype = ctypes.c_char_p
    lib.gdn_workspace_status.argtypes = [P, P]
    lib.gdn_workspace_status.restype = I
    lib.gdn_path.argtypes = [SP]
    lib.gdn_path.restype = I
    lib.gdn_version.argtypes = []
    lib.gdn_version.restype = I
    lib.gdn_chunk_fwd_noalloc.argtypes = [SP] + [P] * 8 + [P]
    lib.gdn_chunk_fwd_noalloc.restype = I
    lib.gdn_noalloc_status.argtypes = [P]
    lib.gdn_noalloc_status.restype = I
    lib.gdn_diag_wait_timeout_noalloc.argtypes = [I, P]
    lib.gdn_diag_wait_timeout_noalloc.restype = I
    lib.gdn_diag_set_fwd_split.argtypes = [I, I, I]
    lib.gdn_diag_set_fwd_split.restype = None
    lib.gdn_chunk_saved_bytes.argtypes = [SP]
    lib.gdn_chunk_saved_bytes.restype = Z
    lib.gdn_chunk_fwd_save.argtypes = [SP] + [P] * 8 + [P, Z, P, Z, P]
    lib.gdn_chunk_fwd_save.restype = I
    lib.gdn_chunk_bwd_saved.argtypes = [SP] + [P] * 14 + [P, Z, P, Z, P]
    lib.gdn_chunk_bwd_saved.restype = I
    CP = ctypes.POINTER(gdn_conv_shape)
    lib.gdn_conv_workspace_bytes.argtypes = [CP]
    lib.gdn_conv_workspace_bytes.restype = Z
    lib.gdn_conv_fwd.argtypes = [CP] + [P] * 6 + [P]
    lib.gdn_conv_fwd.restype = I
    lib.gdn_conv_bwd.argtypes = [CP] + [P] * 10 + [P, Z, P]
    lib.gdn_conv_bwd.restype = I
    lib.gdn_profile_arm.argtypes = [P, I]
    lib.gdn_profile_arm.restype = None
    lib.gdn_profile_count.argtypes = []
    lib.gdn_profile_count.restype = I
    lib.gdn_diag_wait_timeout.argtypes = [P, I, P]
    lib.gdn_diag_wait_timeout.restype = I
    lib.gdn_profile_name.argtypes = [I]
    lib.gdn_profile_name.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GDN_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return GDN_DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _p(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def shape_of(q: torch.Tensor, v: torch.Tensor) -> gdn_shape:
    B, T, H, dk = q.shape
    return gdn_shape(B, T, H, dk, v.shape[-1], _dtype_code(q))


def path(q, v) -> int:
    s = shape_of(q, v)
    return load().gdn_path(ctypes.byref(s))


def chunk_workspace_bytes(shape: gdn_shape, is_bwd: bool) -> int:
    return load().gdn_chunk_workspace_bytes(ctypes.byref(shape), int(is_bwd))


def varlen_workspace_bytes(shape: gdn_shape, nseq: int, is_bwd: bool) -> int:
    return load().gdn_varlen_workspace_bytes(ctypes.byref(shape), nseq, int(is_bwd))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _check(rc: int, where: str):
    if rc != GDN_OK:
        raise GdnError(rc, where)


def gdn_chunk_fwd(q, k, v, g, beta, S_in=None, o=None, S_out=None, workspace=None,
                  stream=None, want_state=True):
    """Forward of one chunk. Returns (o, S_out)."""
    lib = load()
    s = shape_of(q, v)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if o is None:
        o = torch.empty(B, T, H, dv, dtype=q.dtype, device=q.device)
    if S_out is None and want_state:
        S_out = torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
    need = lib.gdn_chunk_workspace_bytes(ctypes.byref(s), 0)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    rc = lib.gdn_chunk_fwd(ctypes.byref(s), _p(q), _p(k), _p(v), _p(g), _p(beta), _p(S_in),
                           _p(o), _p(S_out), _p(workspace), workspace.numel(), _stream(stream))
    _check(rc, "gdn_chunk_fwd")
    return o, S_out


def gdn_chunk_bwd(q, k, v, g, beta, S_in, dout, dS_out=None, grads=None, dS_in=None,
                  workspace=None, stream=None, want_state=True):
    """Backward of one chunk. Returns (dq, dk, dv, dg, dbeta, dS_in)."""
    lib = load()
    s = shape_of(q, v)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                 torch.empty_like(g), torch.empty_like(beta))
    if dS_in is None and want_state:
        dS_in = torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
    need = lib.gdn_chunk_workspace_bytes(ctypes.byref(s), 1)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    rc = lib.gdn_chunk_bwd(ctypes.byref(s), _p(q), _p(k), _p(v), _p(g), _p(beta), _p(S_in),
                           _p(dout), _p(dS_out), *[_p(t) for t in grads], _p(dS_in),
                           _p(workspace), workspace.numel(), _stream(stream))
    _check(rc, "gdn_chunk_bwd")
    return (*grads, dS_in)


def chunk_saved_bytes(shape: gdn_shape) -> int:
    return load().gdn_chunk_saved_bytes(ctypes.byref(shape))


def gdn_chunk_fwd_save(q, k, v, g, beta, S_in=None, saved=None, o=None, S_out=None,
                       workspace=None, stream=None, want_state=True):
    """Forward of one chunk that keeps its per-block products for
    gdn_chunk_bwd_saved. Returns (o, S_out, saved)."""
    lib = load()
    s = shape_of(q, v)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if o is None:
        o = torch.empty(B, T, H, dv, dtype=q.dtype, device=q.device)
    if S_out is None and want_state:
        S_out = torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
    if saved is None:
        saved = alloc_workspace(lib.gdn_chunk_saved_bytes(ctypes.byref(s)), q.device)
    if workspace is None:
        workspace = alloc_workspace(lib.gdn_chunk_workspace_bytes(ctypes.byref(s), GDN_WS_SAVED),
                                    q.device)
    rc = lib.gdn_chunk_fwd_save(ctypes.byref(s), _p(q), _p(k), _p(v), _p(g), _p(beta), _p(S_in),
                                _p(o), _p(S_out), _p(saved), saved.numel(), _p(workspace),
                                workspace.numel(), _stream(stream))
    _check(rc, "gdn_chunk_fwd_save")
    return o, S_out, saved


def gdn_chunk_bwd_saved(q, k, v, g, beta, S_in, dout, saved, dS_out=None, grads=None,
                        dS_in=None, workspace=None, stream=None, want_state=True):
    """Backward of one chunk from the products gdn_chunk_fwd_save kept.
    Returns (dq, dk, dv, dg, dbeta, dS_in)."""
    lib = load()
    s = shape_of(q, v)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                 torch.empty_like(g), torch.empty_like(beta))
    if dS_in is None and want_state:
        dS_in = torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(lib.gdn_chunk_workspace_bytes(ctypes.byref(s), GDN_WS_SAVED),
                                    q.device)
    rc = lib.gdn_chunk_bwd_saved(ctypes.byref(s), _p(q), _p(k), _p(v), _p(g), _p(beta),
                                 _p(S_in), _p(dout), _p(dS_out), *[_p(t) for t in grads],
                                 _p(dS_in), _p(saved), saved.numel(), _p(workspace),
                                 workspace.numel(), _stream(stream))
    _check(rc, "gdn_chunk_bwd_saved")
    return (*grads, dS_in)


def gdn_varlen_fwd(cu_seqlens, q, k, v, g, beta, S0=None, o=None, S_final=None,
                   workspace=None, stream=None):
    """Packed varlen forward (q: [1, T, H, dk]). Returns (o, S_final [nseq, H, dk, dv])."""
    lib = load()
    s = shape_of(q, v)
    _, T, H, dk = q.shape
    dv = v.shape[-1]
    nseq = cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty(1, T, H, dv, dtype=q.dtype, device=q.device)
    if S_final is None:
        S_final = torch.empty(nseq, H, dk, dv, dtype=torch.float32, device=q.device)
    need = lib.gdn_varlen_workspace_bytes(ctypes.byref(s), nseq, 0)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    rc = lib.gdn_varlen_fwd(ctypes.byref(s), _p(cu_seqlens), nseq, _p(q), _p(k), _p(v), _p(g),
                            _p(beta), _p(S0), _p(o), _p(S_final), _p(workspace),
                            workspace.numel(), _stream(stream))
    _check(rc, "gdn_varlen_fwd")
    return o, S_final


def gdn_varlen_bwd(cu_seqlens, q, k, v, g, beta, S0, dout, dS_final=None, grads=None,
                   dS0=None, workspace=None, stream=None):
    """Packed varlen backward. Returns (dq, dk, dv, dg, dbeta, dS0)."""
    lib = load()
    s = shape_of(q, v)
    _, T, H, dk = q.shape
    dv = v.shape[-1]
    nseq = cu_seqlens.numel() - 1
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                 torch.empty_like(g), torch.empty_like(beta))
    if dS0 is None:
        dS0 = torch.empty(nseq, H, dk, dv, dtype=torch.float32, device=q.device)
    need = lib.gdn_varlen_workspace_bytes(ctypes.byref(s), nseq, 1)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    rc = lib.gdn_varlen_bwd(ctypes.byref(s), _p(cu_seqlens), nseq, _p(q), _p(k), _p(v), _p(g),
                            _p(beta), _p(S0), _p(dout), _p(dS_final), *[_p(t) for t in grads],
                            _p(dS0), _p(workspace), workspace.numel(), _stream(stream))
    _check(rc, "gdn_varlen_bwd")
    return (*grads, dS0)


def conv_shape_of(x: torch.Tensor, w: torch.Tensor, act: str) -> gdn_conv_shape:
    B, T, C = x.shape
    return gdn_conv_shape(B, T, C, w.shape[1], _dtype_code(x), CONV_ACT[act])


def gdn_conv_fwd(x, w, b=None, state_in=None, act="silu", y=None, state_out=None,
                 want_state=True, stream=None):
    """Causal short convolution of one chunk, x [B, T, C]. Returns (y, state_out [B, W-1, C])."""
    lib = load()
    s = conv_shape_of(x, w, act)
    B, T, C = x.shape
    if y is None:
        y = torch.empty_like(x)
    if state_out is None and want_state:
        state_out = torch.empty(B, w.shape[1] - 1, C, dtype=x.dtype, device=x.device)
    rc = lib.gdn_conv_fwd(ctypes.byref(s), _p(x), _p(w), _p(b), _p(state_in), _p(y),
                          _p(state_out), _stream(stream))
    _check(rc, "gdn_conv_fwd")
    return y, state_out


def gdn_conv_bwd(x, w, b, state_in, dy, dstate_out=None, act="silu", dx=None, dw=None,
                 db=None, dstate_in=None, workspace=None, stream=None, want_state=True):
    """Backward of one chunk. Returns (dx, dw, db, dstate_in)."""
    lib = load()
    s = conv_shape_of(x, w, act)
    B, T, C = x.shape
    if dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        dw = torch.empty_like(w)
    if db is None and b is not None:
        db = torch.empty_like(b)
    if dstate_in is None and want_state:
        dstate_in = torch.empty(B, w.shape[1] - 1, C, dtype=x.dtype, device=x.device)
    if workspace is None:
        workspace = alloc_workspace(lib.gdn_conv_workspace_bytes(ctypes.byref(s)), x.device)
    rc = lib.gdn_conv_bwd(ctypes.byref(s), _p(x), _p(w), _p(b), _p(state_in), _p(dy),
                          _p(dstate_out), _p(dx), _p(dw), _p(db), _p(dstate_in), _p(workspace),
                          workspace.numel(), _stream(stream))
    _check(rc, "gdn_conv_bwd")
    return dx, dw, db, dstate_in


def gdn_workspace_status(workspace, stream=None) -> int:
    return load().gdn_workspace_status(_p(workspace), _stream(stream))


def diag_wait_timeout(workspace, limit_log2=20, stream=None) -> int:
    """Runs the bounded-wait self-check (include/gdn_profile.h); read the
    outcome with gdn_workspace_status."""
    return load().gdn_diag_wait_timeout(_p(workspace), limit_log2, _stream(stream))


def gdn_noalloc_status(stream=None) -> int:
    return load().gdn_noalloc_status(_stream(stream))


def diag_wait_timeout_noalloc(limit_log2=20, stream=None) -> int:
    """The bounded-wait self-check on the no-allocation forward's scratch;
    read the outcome with gdn_noalloc_status."""
    return load().gdn_diag_wait_timeout_noalloc(limit_log2, _stream(stream))


def set_fwd_split(segments=0, first_permille=0, chain_rg=0):
    """Measurement override of the split forward (include/gdn_profile.h):
    segments 1 = no split, 0 = the library's default."""
    load().gdn_diag_set_fwd_split(segments, first_permille, chain_rg)


def gdn_status_str(code: int) -> str:
    return load().gdn_status_str(code).decode()


class KernelTimer:
    """Per-kernel CUDA-event timing through the library's diagnostic hook
    (include/gdn_profile.h). Events are recorded on the stream each kernel is
    launched on, around every launch of the calls made while armed."""

    def __init__(self, capacity: int = 4096):
        self.capacity = capacity
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        self.n = 0
        self.names = []

    def __enter__(self):
        for e in self.events:  # materialise the lazily-created events
            e.record()
        torch.cuda.synchronize()
        self._handles = (ctypes.c_void_p * self.capacity)(
            *[e.cuda_event for e in self.events])
        load().gdn_profile_arm(ctypes.cast(self._handles, ctypes.c_void_p), self.capacity)
        return self

    def __exit__(self, *exc):
        lib = load()
        self.n = lib.gdn_profile_count()
        self.names = [lib.gdn_profile_name(i) for i in range(self.n)]
        lib.gdn_profile_arm(None, 0)
        return False

    def per_kernel(self):
        """{kernel name: [durations in ms]} (call after synchronising)."""
        out = {}
        for i in range(self.n - 1):
            name = self.names[i]
            if name is None:
                continue
            out.setdefault(name.decode(), []).append(self.events[i].elapsed_time(self.events[i + 1]))
        return out
