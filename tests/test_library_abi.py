"""The C-ABI library loads, exports every symbol include/hypic.h declares, and
rejects bad arguments on the host before launching anything (CPU only: every
call here fails validation, so no kernel is ever launched)."""
import ctypes
import os
import re

import numpy as np
import pytest

from linear_attn_state_chunked_gb300 import hypic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hypic.h")

FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(hypic.LIB_PATH):
        from linear_attn_state_chunked_gb300 import build_ext
        build_ext.build()
    return hypic.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hypic_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    syms = declared_symbols()
    assert set(syms) == set(hypic.EXPORTS)
    for s in syms:
        assert hasattr(L, s), s
    assert L.hypic_version() == 4
    assert b"" == L.hypic_last_error()


def _desc(**over):
    d = dict(n_layers=2, n_heads=4, d_k=64, d_v=64, seam_w=8, conv_k=0, mode=0, in_dtype=1)
    d.update(over)
    return d


def _tok(**over):
    t = dict(q=FAKE, k=FAKE, v=FAKE, alpha=FAKE, beta=FAKE, conv_w=None)
    t.update(over)
    return t


def _build(desc, tok=None, seg_off=(0, 10, 20), n_tokens=20, T=FAKE, S=FAKE, ws=FAKE,
           ws_bytes=256):
    d = hypic.make_desc(desc)
    t = hypic.make_tokens(tok if tok is not None else _tok(), n_tokens)
    off = np.asarray(seg_off, dtype=np.int64)
    return hypic.lib().hypic_segment_build(
        ctypes.byref(d), ctypes.byref(t), off.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        len(off) - 1, T, S, ws, ws_bytes, None)


def _compose(desc, order=(0, 1), seg_off=(0, 10, 20), tok=None, T=FAKE, S=FAKE, S_final=FAKE,
             o=FAKE, S_init=None, n_tokens=20, n_seg=None):
    d = hypic.make_desc(desc)
    t = hypic.make_tokens(tok if tok is not None else _tok(), n_tokens)
    off = np.asarray(seg_off, dtype=np.int64)
    ordr = np.asarray(order, dtype=np.int32)
    return hypic.lib().hypic_compose(
        ctypes.byref(d), ctypes.byref(t), off.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        len(off) - 1 if n_seg is None else n_seg,
        ordr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(ordr),
        T, S, S_init, None, S_final, o, None)


def _seam(desc, order=(0, 1), seg_off=(0, 10, 20), tok=None, S_in=FAKE, o=FAKE, n_tokens=20):
    d = hypic.make_desc(desc)
    t = hypic.make_tokens(tok if tok is not None else _tok(), n_tokens)
    off = np.asarray(seg_off, dtype=np.int64)
    ordr = np.asarray(order, dtype=np.int32)
    return hypic.lib().hypic_seam_advance(
        ctypes.byref(d), ctypes.byref(t), off.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        len(off) - 1, ordr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(ordr),
        S_in, o, None, None)


BAD_BUILD = [
    ("mode", dict(desc=_desc(mode=4)), 1),
    ("dtype", dict(desc=_desc(in_dtype=7)), 3),
    ("d_k != d_v", dict(desc=_desc(d_v=32)), 4),
    ("d unsupported", dict(desc=_desc(d_k=48, d_v=48)), 4),
    ("layers", dict(desc=_desc(n_layers=0)), 2),
    ("seam_w", dict(desc=_desc(seam_w=65)), 2),
    ("conv_k", dict(desc=_desc(conv_k=5)), 4),
    ("conv without seam", dict(desc=_desc(conv_k=4, seam_w=2)), 4),
    ("conv_w missing", dict(desc=_desc(conv_k=4)), 1),
    ("conv_act unknown", dict(desc=_desc(conv_k=4, conv_act=2)), 1),
    ("conv_act without conv", dict(desc=_desc(conv_act=1)), 1),
    ("k null", dict(desc=_desc(), tok=_tok(k=None)), 1),
    ("beta null", dict(desc=_desc(), tok=_tok(beta=None)), 1),
    ("v misaligned", dict(desc=_desc(), tok=_tok(v=FAKE + 4)), 1),
    ("offsets decrease", dict(desc=_desc(), seg_off=(0, 12, 11)), 2),
    ("offset negative", dict(desc=_desc(), seg_off=(-1, 10)), 2),
    ("offsets past N", dict(desc=_desc(), seg_off=(0, 10, 21)), 2),
    ("too many tokens", dict(desc=_desc(), n_tokens=1 << 31), 2),
    ("T null", dict(desc=_desc(), T=None), 1),
    ("S misaligned", dict(desc=_desc(), S=FAKE + 8), 1),
    ("no workspace", dict(desc=_desc(), ws=None), 5),
    ("workspace small", dict(desc=_desc(), ws_bytes=16), 5),
    ("workspace misaligned", dict(desc=_desc(), ws=FAKE + 16), 5),
]


@pytest.mark.parametrize("what,kw,code", BAD_BUILD, ids=[b[0] for b in BAD_BUILD])
def test_build_rejects(L, what, kw, code):
    rc = _build(**kw)
    assert rc == code, (what, rc, L.hypic_last_error())
    assert L.hypic_last_error() != b""


def test_build_rejects_too_many_segments(L):
    off = np.arange(hypic.MAX_SEGMENTS + 2, dtype=np.int64)
    assert _build(_desc(), seg_off=off, n_tokens=len(off)) == 2


BAD_COMPOSE = [
    ("order out of range", dict(order=(0, 2)), 2),
    ("order negative", dict(order=(-1,)), 2),
    ("no o_out with seams", dict(o=None), 1),
    ("no S_final", dict(S_final=None), 1),
    ("T null", dict(T=None), 1),
    ("tokens q null", dict(tok=_tok(q=None)), 1),
    ("S_init misaligned", dict(S_init=FAKE + 4), 1),
    ("n_seg too large", dict(n_seg=hypic.MAX_SEGMENTS + 1), 2),
]


@pytest.mark.parametrize("what,kw,code", BAD_COMPOSE, ids=[b[0] for b in BAD_COMPOSE])
def test_compose_rejects(L, what, kw, code):
    rc = _compose(_desc(), **kw)
    assert rc == code, (what, rc, L.hypic_last_error())


BAD_SEAM = [
    ("order out of range", dict(order=(3,)), 2),
    ("S_in null", dict(S_in=None), 1),
    ("o null", dict(o=None), 1),
    ("offsets past N", dict(seg_off=(0, 30)), 2),
]


@pytest.mark.parametrize("what,kw,code", BAD_SEAM, ids=[b[0] for b in BAD_SEAM])
def test_seam_rejects(L, what, kw, code):
    rc = _seam(_desc(), **kw)
    assert rc == code, (what, rc, L.hypic_last_error())


def test_workspace_size(L):
    n = hypic.workspace_size(_desc())
    assert n > 0 and n % 256 == 0


def test_binding_raises_with_message(L):
    with pytest.raises(hypic.HypicError) as ei:
        hypic._check(_build(_desc(mode=9)))
    assert "HYPIC_ERR_INVALID_ARG" in str(ei.value) and "mode" in str(ei.value)


def test_selftest_rejects_bad_arguments(L):
    """Argument checks of the bounded-wait self-test happen on the host,
    before anything is launched (no GPU needed)."""
    assert L.hypic_selftest_bounded_wait(FAKE + 16, 1000, None) == 5
    assert L.hypic_selftest_bounded_wait(None, 0, None) == 2  # NULL: the device status word
    assert L.hypic_selftest_bounded_wait(FAKE, 0, None) == 2
    assert L.hypic_selftest_bounded_wait(FAKE, (1 << 34) + 1, None) == 2
    assert b"max_cycles" in L.hypic_last_error()


def _forward(desc, tok=None, seg_off=(0, 10, 20), n_tokens=20, o=FAKE, T=None, S=None):
    d = hypic.make_desc(desc)
    t = hypic.make_tokens(tok if tok is not None else _tok(), n_tokens)
    off = np.asarray(seg_off, dtype=np.int64)
    return hypic.lib().hypic_segment_forward(
        ctypes.byref(d), ctypes.byref(t), off.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        len(off) - 1, o, T, S, None)


BAD_FORWARD = [
    ("o_out null", dict(desc=_desc(), o=None), 1),
    ("o_out misaligned", dict(desc=_desc(), o=FAKE + 4), 1),
    ("q null", dict(desc=_desc(), tok=_tok(q=None)), 1),
    ("T misaligned", dict(desc=_desc(), T=FAKE + 8), 1),
    ("S misaligned", dict(desc=_desc(), S=FAKE + 8), 1),
    ("mode", dict(desc=_desc(mode=4)), 1),
    ("offsets past N", dict(desc=_desc(), seg_off=(0, 10, 21)), 2),
]


@pytest.mark.parametrize("what,kw,code", BAD_FORWARD, ids=[b[0] for b in BAD_FORWARD])
def test_forward_rejects(L, what, kw, code):
    """The segment forward validates on the host like the build (q and the
    output are required, T and S optional but aligned) and launches nothing
    on error."""
    assert _forward(**kw) == code
    assert L.hypic_last_error() != b""


def test_forward_empty_request_is_ok(L):
    assert _forward(desc=_desc(), seg_off=(0,), n_tokens=0) == 0
