"""Thin ctypes binding of libhypic.so (include/hypic.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  Tensors are passed as device pointers (``tensor.data_ptr()``);
PyTorch provides the device memory and the stream.  There is no fallback: if
the library is not built, or a call fails, this module raises.
"""
import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhypic.so")

GATED_DELTA, SCALAR_DECAY, DIAG_GATE, KDA = 0, 1, 2, 3
F32, BF16 = 0, 1
ACT_NONE, ACT_SILU = 0, 1
MAX_SEGMENTS = 2048

STATUS = {0: "HYPIC_OK", 1: "HYPIC_ERR_INVALID_ARG", 2: "HYPIC_ERR_SHAPE", 3: "HYPIC_ERR_DTYPE",
          4: "HYPIC_ERR_UNSUPPORTED", 5: "HYPIC_ERR_WORKSPACE", 6: "HYPIC_ERR_CUDA",
          7: "HYPIC_ERR_TIMEOUT"}

# Every symbol include/hypic.h declares.
EXPORTS = ("hypic_version", "hypic_last_error", "hypic_workspace_size",
           "hypic_workspace_status", "hypic_async_status", "hypic_segment_build",
           "hypic_segment_build_noalloc", "hypic_noalloc_status", "hypic_compose",
           "hypic_seam_advance", "hypic_selftest_bounded_wait", "hypic_segment_forward")


class HypicError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s: %s" % (STATUS.get(status, status), msg))
        self.status = status


class Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n_layers", "n_heads", "d_k", "d_v", "seam_w", "conv_k", "mode", "in_dtype", "conv_act")]


class Tokens(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("alpha", ctypes.c_void_p), ("beta", ctypes.c_void_p),
                ("conv_w", ctypes.c_void_p), ("n_tokens", ctypes.c_int64)]


_lib = None


def lib():
    """Load libhypic.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libhypic.so is not built (run linear_attn_state_chunked_gb300."
                               "build_ext.build() or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64p, i32p, fp = (ctypes.c_void_p, ctypes.c_int32,
                                   ctypes.POINTER(ctypes.c_int64),
                                   ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p)
        L.hypic_version.restype = ctypes.c_int
        L.hypic_last_error.restype = ctypes.c_char_p
        L.hypic_workspace_size.restype = ctypes.c_size_t
        L.hypic_workspace_size.argtypes = [ctypes.POINTER(Desc)]
        L.hypic_workspace_status.restype = ctypes.c_int
        L.hypic_workspace_status.argtypes = [vp, vp]
        L.hypic_async_status.restype = ctypes.c_int
        L.hypic_async_status.argtypes = [vp]
        L.hypic_noalloc_status.restype = ctypes.c_int
        L.hypic_noalloc_status.argtypes = [vp]
        L.hypic_selftest_bounded_wait.restype = ctypes.c_int
        L.hypic_selftest_bounded_wait.argtypes = [vp, ctypes.c_int64, vp]
        L.hypic_segment_build.restype = ctypes.c_int
        L.hypic_segment_build.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(Tokens), i64p, i32,
                                          fp, fp, vp, ctypes.c_size_t, vp]
        L.hypic_segment_forward.restype = ctypes.c_int
        L.hypic_segment_forward.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(Tokens), i64p, i32,
                                            fp, fp, fp, vp]
        L.hypic_segment_build_noalloc.restype = ctypes.c_int
        L.hypic_segment_build_noalloc.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(Tokens), i64p,
                                                  i32, fp, fp, vp]
        L.hypic_compose.restype = ctypes.c_int
        L.hypic_compose.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(Tokens), i64p, i32,
                                    i32p, i32, fp, fp, fp, fp, fp, fp, vp]
        L.hypic_seam_advance.restype = ctypes.c_int
        L.hypic_seam_advance.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(Tokens), i64p, i32,
                                         i32p, i32, fp, fp, fp, vp]
        _lib = L
    return _lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def make_desc(d):
    return Desc(*(int(d.get(n, 0)) for n in ("n_layers", "n_heads", "d_k", "d_v", "seam_w", "conv_k",
                                             "mode", "in_dtype", "conv_act")))


def make_tokens(tok, n_tokens):
    if tok is None:
        return None
    return Tokens(_p(tok.get("q")), _p(tok.get("k")), _p(tok.get("v")), _p(tok.get("alpha")),
                  _p(tok.get("beta")), _p(tok.get("conv_w")), int(n_tokens))


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc):
    if rc != 0:
        raise HypicError(rc, lib().hypic_last_error().decode())


def _i64(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int64))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _i32(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _tok_n(tok, n_tokens):
    if n_tokens is not None:
        return n_tokens
    return tok["k"].shape[1]


def workspace_size(desc):
    d = make_desc(desc)
    return int(lib().hypic_workspace_size(ctypes.byref(d)))


def workspace_status(workspace, stream=None):
    """Raise HypicError(HYPIC_ERR_TIMEOUT) if a device-side wait of a build on
    this workspace gave up; waits for the stream."""
    _check(lib().hypic_workspace_status(_p(workspace), _stream(stream)))


def async_status(stream=None):
    """Raise HypicError(HYPIC_ERR_TIMEOUT) if a device-side wait of a compose or
    seam-advance call on the current device gave up since the last query
    (clears the report); waits for the stream."""
    _check(lib().hypic_async_status(_stream(stream)))


def noalloc_status(stream=None):
    """Raise HypicError(HYPIC_ERR_TIMEOUT) if a device-side wait of the last
    segment_build_noalloc on the current device gave up; waits for the stream."""
    _check(lib().hypic_noalloc_status(_stream(stream)))


def selftest_bounded_wait(workspace, max_cycles, stream=None):
    """Run the bounded-wait self-test into the workspace status word (read it
    back with workspace_status, which then raises HYPIC_ERR_TIMEOUT); with
    workspace=None into the device status word that async_status reads."""
    _check(lib().hypic_selftest_bounded_wait(_p(workspace), int(max_cycles), _stream(stream)))


def pair_shapes(desc, n_seg):
    """Shapes of the T and S cache tensors for n_seg segments."""
    L, H, D = desc["n_layers"], desc["n_heads"], desc["d_k"]
    if desc["mode"] in (GATED_DELTA, KDA):
        tshape = (L, n_seg, H, D, D)
    elif desc["mode"] == DIAG_GATE:
        tshape = (L, n_seg, H, D)
    else:
        tshape = (L, n_seg, H)
    return tshape, (L, n_seg, H, D, desc["d_v"])


def segment_build(desc, tok, seg_off, T_out, S_out, workspace, stream=None, n_tokens=None):
    d = make_desc(desc)
    t = make_tokens(tok, _tok_n(tok, n_tokens))
    off, offp = _i64(seg_off)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().hypic_segment_build(ctypes.byref(d), ctypes.byref(t), offp, len(off) - 1,
                                     _p(T_out), _p(S_out), _p(workspace), ws_bytes,
                                     _stream(stream)))


def segment_forward(desc, tok, seg_off, o_out, T_out=None, S_out=None, stream=None, n_tokens=None):
    """Per-token outputs of every segment body from a zero state (fp32
    [L][N][H][d_v]; seam-token rows untouched), plus the pair when T_out /
    S_out are given."""
    d = make_desc(desc)
    t = make_tokens(tok, _tok_n(tok, n_tokens))
    off, offp = _i64(seg_off)
    _check(lib().hypic_segment_forward(ctypes.byref(d), ctypes.byref(t), offp, len(off) - 1, _p(o_out),
                                       _p(T_out), _p(S_out), _stream(stream)))


def segment_build_noalloc(desc, tok, seg_off, T_out, S_out, stream=None, n_tokens=None):
    """segment_build for callers that cannot allocate device memory: uses the
    library's own static scratch instead of a workspace (see include/hypic.h)."""
    d = make_desc(desc)
    t = make_tokens(tok, _tok_n(tok, n_tokens))
    off, offp = _i64(seg_off)
    _check(lib().hypic_segment_build_noalloc(ctypes.byref(d), ctypes.byref(t), offp, len(off) - 1,
                                             _p(T_out), _p(S_out), _stream(stream)))


def compose(desc, tok, seg_off, order, T, S, S_final, S_init=None, S_prefix_out=None,
            o_out=None, stream=None, n_tokens=None):
    d = make_desc(desc)
    t = make_tokens(tok, _tok_n(tok, n_tokens)) if tok is not None else None
    off, offp = _i64(seg_off)
    ordr, ordp = _i32(order)
    _check(lib().hypic_compose(ctypes.byref(d), ctypes.byref(t) if t is not None else None,
                               offp, len(off) - 1, ordp, len(ordr), _p(T), _p(S), _p(S_init),
                               _p(S_prefix_out), _p(S_final), _p(o_out), _stream(stream)))


def seam_advance(desc, tok, seg_off, order, S_in, o_out, S_out=None, stream=None, n_tokens=None):
    d = make_desc(desc)
    t = make_tokens(tok, _tok_n(tok, n_tokens))
    off, offp = _i64(seg_off)
    ordr, ordp = _i32(order)
    _check(lib().hypic_seam_advance(ctypes.byref(d), ctypes.byref(t), offp, len(off) - 1, ordp,
                                    len(ordr), _p(S_in), _p(o_out), _p(S_out), _stream(stream)))
