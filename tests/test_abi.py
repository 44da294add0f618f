"""The C-ABI library loads, exports every entry point include/attn_fwd.h
declares, and rejects invalid arguments before touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_fwd.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_contract():
    names = _declared()
    for n in ("attn_fwd", "attn_fwd_varlen", "attn_fwd_paged", "attn_splitkv_combine"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = A.library()
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (attn_\w+)", out))
    for name in _declared():
        assert name in exported, name
        assert getattr(lib, name) is not None
    assert set(_lib.EXPORTS) == set(_declared())


def test_status_strings():
    lib = A.library()
    assert lib.attn_status_string(0) == b"ok"
    assert lib.attn_status_string(2) == b"unsupported configuration"
    assert lib.attn_status_string(4) == b"kernel wait timed out"


S = _lib.attn_strides


def _fwd(**kw):
    a = dict(q=1 << 12, k=1 << 12, v=1 << 12, o=1 << 12, lse=None, B=1, Hq=2, Hkv=2, Lq=8, Lk=8,
             d=64, dtype=1, s=S(1024, 512, 64))
    a.update(kw)
    st = a["s"]
    opts = _lib.attn_opts(0.0, 0, 0.0, None)
    return A.library().attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"],
                                a["Hkv"], a["Lq"], a["Lk"], a["d"], a["dtype"], st, st, st, st,
                                ctypes.byref(opts), None)


def test_validation_rejects_before_launch():
    assert _fwd(d=96) == 2                 # unsupported head dim
    assert _fwd(Hq=3, Hkv=2) == 1          # Hq % Hkv
    assert _fwd(q=None) == 1               # null pointer
    assert _fwd(q=(1 << 12) + 2) == 1      # misaligned base
    assert _fwd(s=S(1024, 512, 60)) == 1   # row stride not a multiple of 16 bytes
    assert _fwd(dtype=7) == 1
    assert _fwd(B=0) == 0                  # empty problem: no-op
    assert _fwd(Lq=0) == 0


def test_option_combinations_rejected_before_launch():
    """Soft-cap with ALiBi or bias, ALiBi with bias, bias outside the dense
    entry point: ATTN_ERR_UNSUPPORTED; misaligned ALiBi/bias: ATTN_ERR_INVALID."""
    lib = A.library()
    p = 1 << 12
    st = S(1024, 512, 64)

    def dense(**kw):
        o = _lib.attn_opts()
        for key, val in kw.items():
            setattr(o, key, val)
        return lib.attn_fwd(p, p, p, p, None, 1, 2, 2, 8, 8, 64, 1, st, st, st, st,
                            ctypes.byref(o), None)

    assert dense(softcap=30.0, alibi_slopes=p) == 2
    assert dense(softcap=30.0, bias=p, bias_strides=S(0, 0, 8)) == 2
    assert dense(alibi_slopes=p, bias=p, bias_strides=S(0, 0, 8)) == 2
    assert dense(alibi_slopes=p + 2) == 1              # misaligned slopes
    assert dense(alibi_slopes=p, alibi_stride=1) == 1  # stride < Hq
    assert dense(bias=p + 8, bias_strides=S(0, 0, 8)) == 1  # base not 16-byte aligned
    assert dense(bias=p, bias_strides=S(0, 0, 12)) == 1     # row stride not a multiple of 8
    o = _lib.attn_opts()
    o.bias, o.bias_strides = p, S(0, 0, 8)
    cu = p
    assert lib.attn_fwd_varlen(p, p, p, p, None, cu, cu, 1, 8, 8, 8, 2, 2, 64, 1, st, st, st, st,
                               ctypes.byref(o), None) == 2
    assert lib.attn_fwd_paged(p, p, p, p, p, p, None, 1, 1, 8, 2, 128, 1, 64, 4, 2, 1, None, None,
                              ctypes.byref(o), None) == 2


def test_paged_validation():
    lib = A.library()
    opts = _lib.attn_opts(0.0, 0, 0.0, None)
    p = 1 << 12

    def call(**kw):
        a = dict(B=2, Lq=1, Hq=8, Hkv=2, d=128, page=64, num_pages=4, max_pages=2, splits=1)
        a.update(kw)
        return lib.attn_fwd_paged(p, p, p, p, p, p, None, a["B"], a["Lq"], a["Hq"], a["Hkv"],
                                  a["d"], 1, a["page"], a["num_pages"], a["max_pages"],
                                  a["splits"], None, None, ctypes.byref(opts), None)

    assert call(page=48) == 2       # page size must be a power of two in [16, 256]
    assert call(Lq=5, d=96) == 2    # head dim (Lq * g > 16 routes to the prefill kernel)
    assert call(splits=65) == 1
    assert call(splits=3) == 1      # splits > 1 needs the scratch buffers
    assert call(num_pages=0) == 1
    assert call(B=0) == 0


def test_workspace_and_auto_splits():
    assert A.attn_paged_workspace_bytes(64, 1, 32, 128, 1) == 0
    assert A.attn_paged_workspace_bytes(64, 1, 32, 128, 4) == 4 * 64 * 32 * 129 * 4
    s = A.attn_paged_auto_splits(64, 8, 128)
    assert 1 <= s <= 64
    assert A.attn_paged_auto_splits(1, 1, 1) == 1


def test_paged_window_pages():
    """W of the paged split layout: every page without a left window, else the
    pages the band [L - Lq - left, L) can touch (its length over the page size,
    plus one for a band that starts inside a page), capped by the table."""
    W = A.attn_paged_window_pages
    assert W(1, 64, 100) == 100                                  # no window
    assert W(1, 64, 100, window=(-1, 5)) == 100                  # right bound only
    assert W(1, 64, 100, causal=True) == 100
    assert W(1, 64, 100, window=(255, -1)) == 4 + 1              # 256 keys: 4 pages + 1
    assert W(1, 64, 100, window=(256, -1)) == 5 + 1
    assert W(4, 16, 100, window=(0, 0)) == 1 + 1
    assert W(1, 64, 3, window=(1000, -1)) == 3                   # capped by the table
    # The band [L - Lq - left, L) never spans more pages than W, wherever it starts.
    for Lq, page, left in ((1, 64, 300), (4, 32, 40), (2, 16, 0)):
        w = W(Lq, page, 1000, window=(left, -1))
        for L in range(Lq + left, Lq + left + 3 * page):
            lo = L - Lq - left
            assert (L + page - 1) // page - lo // page <= w


def test_combine_validation():
    lib = A.library()
    p = 1 << 12
    assert lib.attn_splitkv_combine(p, p, 0, 1, 1, 1, 128, None, p, 1, None, None) == 1
    assert lib.attn_splitkv_combine(p, p, 2, 1, 1, 1, 80, None, p, 1, None, None) == 2
    assert lib.attn_splitkv_combine(p, p, 2, 0, 1, 1, 128, None, p, 1, None, None) == 0
