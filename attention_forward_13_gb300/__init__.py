"""GB300 (sm_103a) fused attention forward: thin Python binding of the C ABI.

Every function here only marshals torch tensors (device pointers, sizes,
strides, the current CUDA stream) into the C library ``libattn_fwd.so``; all
arithmetic runs in the library's CUDA kernels.  There is no fallback: if the
library is missing and cannot be built, or a call fails, an exception is
raised.  Output tensors are allocated with torch when not given.

    o, lse = attn_fwd(q, k, v, causal=True)                 # [B,H,L,d]
    o, lse = attn_fwd_varlen(q, k, v, cu_q, cu_k, max_q)    # [total,H,d]
    o, lse = attn_fwd_paged(q, k_pool, v_pool, block_table, seqlens_k)
    o, lse = attn_splitkv_combine(o_part, lse_part)
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

__all__ = ["attn_fwd", "attn_fwd_varlen", "attn_fwd_paged", "attn_splitkv_combine",
           "attn_paged_workspace_bytes", "attn_paged_auto_splits", "attn_device_error",
           "attn_selftest_timeout", "attn_last_kernel_name", "attn_paged_window_pages",
           "attn_fwd_paged_noalloc", "attn_dense_schedule", "gqa_pack", "AttnError", "library"]


class AttnError(RuntimeError):
    def __init__(self, status: int, fn: str):
        self.status = status
        super().__init__(f"{fn}: {_lib.STATUS.get(status, status)}")


def library() -> ctypes.CDLL:
    return _lib.load()


def _check(status: int, fn: str):
    if status != 0:
        raise AttnError(status, fn)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _lib.ATTN_BF16
    if t.dtype == torch.float16:
        return _lib.ATTN_F16
    if t.dtype == torch.float8_e4m3fn:
        return _lib.ATTN_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _opts(scale, causal, softcap, sink, window=None, top_left=False, alibi=None, bias=None,
          scale_p=None, scale_o=None):
    o = _lib.attn_opts()
    o.scale = float(scale) if scale is not None else 0.0
    o.causal = 1 if causal else 0
    o.softcap = float(softcap) if softcap else 0.0
    o.sink = sink.data_ptr() if sink is not None else None
    if window is not None:
        o.use_window = 1
        o.window_left, o.window_right = int(window[0]), int(window[1])
    o.top_left = 1 if top_left else 0
    if alibi is not None:
        o.alibi_slopes = alibi.data_ptr()
        o.alibi_stride = 0 if alibi.dim() == 1 else int(alibi.stride(0))
    if bias is not None:
        o.bias = bias.data_ptr()
        o.bias_strides = _lib.attn_strides(*_bias_strides(bias))
    o.scale_p = float(scale_p) if scale_p else 0.0
    o.scale_o = float(scale_o) if scale_o else 0.0
    return o


def _check_alibi(alibi, B, Hq, device):
    """ALiBi slopes: fp32 [Hq] (shared by every batch) or [B, Hq] (row-contiguous)."""
    if alibi is None:
        return None
    if alibi.dtype != torch.float32 or alibi.device != device or alibi.stride(-1) != 1 or \
            alibi.shape[-1] != Hq or alibi.dim() not in (1, 2) or \
            (alibi.dim() == 2 and alibi.shape[0] != B):
        raise ValueError("alibi_slopes must be fp32 [Hq] or [B, Hq] on the same device")
    return alibi


def _bias_strides(bias):
    """(batch, head, row) element strides of a bias viewed as [B, Hq, Lq, Lk]
    (size-1 broadcast dimensions get stride 0)."""
    if bias.dim() != 4 or bias.stride(3) != 1:
        raise ValueError("bias must be 4-D [B|1, Hq|1, Lq, Lk] with a unit key stride")
    return tuple(0 if bias.shape[i] == 1 else bias.stride(i) for i in range(3))


def _strides_bhld(t):
    s = t.stride()
    if s[3] != 1:
        raise ValueError("innermost (head-dim) stride must be 1")
    return _lib.attn_strides(s[0], s[1], s[2])


def _strides_thd(t):
    s = t.stride()
    if s[2] != 1:
        raise ValueError("innermost (head-dim) stride must be 1")
    return _lib.attn_strides(0, s[1], s[0])


def _check_sink(sink, Hq, device):
    if sink is None:
        return None
    if sink.dtype != torch.float32 or sink.numel() != Hq or sink.device != device:
        raise ValueError("sink must be fp32 [Hq] on the same device")
    return sink.contiguous()


def attn_fwd(q, k, v, o=None, lse=True, causal=False, scale=None, softcap=0.0, sink=None,
             stream=None, window=None, top_left=False, alibi_slopes=None, bias=None,
             scale_p=None, scale_o=None):
    """Dense attention.  q [B,Hq,Lq,d], k/v [B,Hkv,Lk,d] (any strides with d-stride 1).
    ``window`` = (left, right) keeps keys i+Lk-Lq-left <= j <= i+Lk-Lq+right (a
    negative side is unbounded); ``top_left`` drops the Lk-Lq shift.
    ``alibi_slopes``: fp32 [Hq] or [B,Hq]; ``bias``: [B|1,Hq|1,Lq,Lk] in the input
    dtype, added to the scaled score.  float8_e4m3fn inputs (d = 128) run the FP8 path: O is
    e4m3, scale_o * scale_p * softmax(S) V saturated.  Returns (o [B,Hq,Lq,d], lse fp32
    [B,Hq,Lq] or None)."""
    B, Hq, Lq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    if o is None:
        o = torch.empty((B, Hq, Lq, d), dtype=q.dtype, device=q.device)
    lse_t = None
    if lse is True:
        lse_t = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    elif isinstance(lse, torch.Tensor):
        lse_t = lse
    sink = _check_sink(sink, Hq, q.device)
    alibi_slopes = _check_alibi(alibi_slopes, B, Hq, q.device)
    if bias is not None and (bias.dtype != q.dtype or bias.device != q.device):
        raise ValueError("bias must have the input dtype and device")
    opts = _opts(scale, causal, softcap, sink, window, top_left, alibi_slopes, bias, scale_p,
                 scale_o)
    st = library().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse_t), B, Hq, Hkv, Lq, Lk,
                            d, _dtype_code(q), _strides_bhld(q), _strides_bhld(k),
                            _strides_bhld(v), _strides_bhld(o), ctypes.byref(opts),
                            _stream(stream))
    _check(st, "attn_fwd")
    return o, lse_t


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, o=None, lse=True,
                    causal=False, scale=None, softcap=0.0, sink=None, stream=None, window=None,
                    top_left=False, alibi_slopes=None, scale_p=None, scale_o=None):
    """Group mode.  q [total_q,Hq,d], k/v [total_k,Hkv,d], cu_seqlens int32 [B+1] on the
    device.  Returns (o [total_q,Hq,d], lse fp32 [Hq,total_q] or None)."""
    total_q, Hq, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    B = cu_seqlens_q.numel() - 1
    for cu in (cu_seqlens_q, cu_seqlens_k):
        if cu.dtype != torch.int32 or cu.device != q.device or not cu.is_contiguous():
            raise ValueError("cu_seqlens must be contiguous int32 on the device")
    if o is None:
        o = torch.empty((total_q, Hq, d), dtype=q.dtype, device=q.device)
    lse_t = None
    if lse is True:
        lse_t = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    elif isinstance(lse, torch.Tensor):
        lse_t = lse
    sink = _check_sink(sink, Hq, q.device)
    alibi_slopes = _check_alibi(alibi_slopes, B, Hq, q.device)
    opts = _opts(scale, causal, softcap, sink, window, top_left, alibi_slopes, None, scale_p,
                 scale_o)
    st = library().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse_t),
                                   _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, total_q, total_k,
                                   int(max_seqlen_q), Hq, Hkv, d, _dtype_code(q),
                                   _strides_thd(q), _strides_thd(k), _strides_thd(v),
                                   _strides_thd(o), ctypes.byref(opts), _stream(stream))
    _check(st, "attn_fwd_varlen")
    return o, lse_t


def attn_paged_workspace_bytes(B, Lq, Hq, d, num_splits) -> int:
    return int(library().attn_paged_workspace_bytes(B, Lq, Hq, d, num_splits))


def attn_paged_auto_splits(B, Hkv, max_pages_per_seq) -> int:
    return int(library().attn_paged_auto_splits(B, Hkv, max_pages_per_seq))


def attn_paged_window_pages(Lq, page_size, max_pages_per_seq, window=None, causal=False,
                            top_left=False) -> int:
    """Pages of one sequence the paged split layout tiles (W of attn_fwd_paged)."""
    opts = _opts(None, causal, 0.0, None, window, top_left)
    return int(library().attn_paged_window_pages(Lq, page_size, max_pages_per_seq,
                                                 ctypes.byref(opts)))


def gqa_pack(Hq, Hkv) -> int:
    """Query heads per tile the library packs for Hq / Hkv (PackGQA): g when
    g = Hq / Hkv is 2, 4, 8 or 16, else 1."""
    g = Hq // Hkv if Hkv > 0 and Hq % Hkv == 0 else 1
    return g if g in (2, 4, 8, 16) else 1


def attn_dense_schedule(B, Hq, Lq, Lk, grid, causal=False, window=None, top_left=False, Hkv=None):
    """The static schedule attn_fwd runs on `grid` CTAs for a dense masked
    problem: a list of `grid` lists of work items (CTA by CTA, in run order),
    or None where the problem keeps the plain snake order.  Hkv defaults to
    Hq (no head packing)."""
    Hkv = Hq if Hkv is None else Hkv
    opts = _opts(None, causal, 0.0, None, window, top_left)
    pack = gqa_pack(Hq, Hkv)
    per = 256 // pack
    n = B * (Hq // pack) * ((Lq + per - 1) // per) if Lq > 0 else 0
    off = (ctypes.c_int32 * (max(grid, 0) + 1))()
    item = (ctypes.c_int32 * max(n, 1))()
    st = library().attn_dense_schedule(B, Hq, Hkv, Lq, Lk, ctypes.byref(opts), grid, off, item)
    if st == 2:
        return None
    _check(st, "attn_dense_schedule")
    return [list(item[off[c]:off[c + 1]]) for c in range(grid)]


def attn_fwd_paged(q, k_pool, v_pool, block_table, seqlens_k, num_splits=0, o=None, lse=True,
                   causal=False, scale=None, softcap=0.0, sink=None, workspace=None,
                   stream=None, window=None, top_left=False, alibi_slopes=None):
    """Paged KV.  q [B,Lq,Hq,d], pools [num_pages,page,Hkv,d], block_table int32
    [B,max_pages], seqlens_k int32 [B] (all on the device, contiguous).
    Returns (o [B,Lq,Hq,d], lse fp32 [B,Hq,Lq] or None)."""
    B, Lq, Hq, d = q.shape
    num_pages, page, Hkv, _ = k_pool.shape
    max_pages = block_table.shape[1]
    for t in (q, k_pool, v_pool, block_table, seqlens_k):
        if not t.is_contiguous():
            raise ValueError("paged inputs must be contiguous")
    if Lq * (Hq // Hkv) > 16:
        num_splits = 1  # chunked prefill: the prefill kernel, no split-KV scratch
    elif num_splits == 0:
        num_splits = attn_paged_auto_splits(
            B, Hkv, attn_paged_window_pages(Lq, page, max_pages, window, causal, top_left))
    if o is None:
        o = torch.empty((B, Lq, Hq, d), dtype=q.dtype, device=q.device)
    lse_t = None
    if lse is True:
        lse_t = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    elif isinstance(lse, torch.Tensor):
        lse_t = lse
    o_part = lse_part = None
    if num_splits > 1:
        rows = B * Hq * Lq
        need = num_splits * rows * (d + 1)
        if workspace is None or workspace.numel() < need:
            workspace = torch.empty(need, dtype=torch.float32, device=q.device)
        o_part = workspace[: num_splits * rows * d]
        lse_part = workspace[num_splits * rows * d: need]
    sink = _check_sink(sink, Hq, q.device)
    alibi_slopes = _check_alibi(alibi_slopes, B, Hq, q.device)
    opts = _opts(scale, causal, softcap, sink, window, top_left, alibi_slopes)
    st = library().attn_fwd_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                  _ptr(seqlens_k), _ptr(o), _ptr(lse_t), B, Lq, Hq, Hkv, d,
                                  _dtype_code(q), page, num_pages, max_pages, num_splits,
                                  _ptr(o_part), _ptr(lse_part), ctypes.byref(opts),
                                  _stream(stream))
    _check(st, "attn_fwd_paged")
    return o, lse_t


def attn_fwd_paged_noalloc(q, k_pool, v_pool, block_table, seqlens_k, num_splits=0, o=None,
                           lse=True, causal=False, scale=None, softcap=0.0, sink=None,
                           stream=None, window=None, top_left=False, alibi_slopes=None):
    """attn_fwd_paged for callers that cannot allocate device scratch: the split
    partials live in a fixed 16 MiB array inside the library (shared by all
    calls on a GPU; calls overlapping on the GPU race).  Outputs are allocated
    here only when not given."""
    B, Lq, Hq, d = q.shape
    num_pages, page, Hkv, _ = k_pool.shape
    if o is None:
        o = torch.empty((B, Lq, Hq, d), dtype=q.dtype, device=q.device)
    lse_t = None
    if lse is True:
        lse_t = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    elif isinstance(lse, torch.Tensor):
        lse_t = lse
    sink = _check_sink(sink, Hq, q.device)
    alibi_slopes = _check_alibi(alibi_slopes, B, Hq, q.device)
    opts = _opts(scale, causal, softcap, sink, window, top_left, alibi_slopes)
    st = library().attn_fwd_paged_noalloc(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                          _ptr(seqlens_k), _ptr(o), _ptr(lse_t), B, Lq, Hq, Hkv,
                                          d, _dtype_code(q), page, num_pages,
                                          block_table.shape[1], num_splits, ctypes.byref(opts),
                                          _stream(stream))
    _check(st, "attn_fwd_paged_noalloc")
    return o, lse_t


def attn_splitkv_combine(o_partial, lse_partial, sink=None, dtype=torch.bfloat16, o=None,
                         lse=True, stream=None):
    """Merge split partials.  o_partial fp32 [S,B,Hq,Lq,d], lse_partial fp32 [S,B,Hq,Lq].
    Returns (o [B,Lq,Hq,d] in ``dtype``, lse fp32 [B,Hq,Lq] or None)."""
    S, B, Hq, Lq, d = o_partial.shape
    if o is None:
        o = torch.empty((B, Lq, Hq, d), dtype=dtype, device=o_partial.device)
    lse_t = None
    if lse is True:
        lse_t = torch.empty((B, Hq, Lq), dtype=torch.float32, device=o_partial.device)
    elif isinstance(lse, torch.Tensor):
        lse_t = lse
    sink = _check_sink(sink, Hq, o_partial.device)
    st = library().attn_splitkv_combine(_ptr(o_partial.contiguous()),
                                        _ptr(lse_partial.contiguous()), S, B, Hq, Lq, d,
                                        _ptr(sink), _ptr(o), _dtype_code(o), _ptr(lse_t),
                                        _stream(stream))
    _check(st, "attn_splitkv_combine")
    return o, lse_t


def attn_device_error() -> int:
    """Synchronises, reads and clears the device error word; returns its bits."""
    bits = ctypes.c_uint(0)
    st = library().attn_device_error(ctypes.byref(bits))
    if st not in (0, 4):
        raise AttnError(st, "attn_device_error")
    return int(bits.value)


def attn_selftest_timeout(timeout_ns: int, stream=None) -> None:
    _check(library().attn_selftest_timeout(int(timeout_ns), _stream(stream)),
           "attn_selftest_timeout")


def attn_last_kernel_name() -> str:
    return library().attn_last_kernel_name().decode()
