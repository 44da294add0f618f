"""attn_fwd_paged_noalloc through the C ABI, against the fp64 oracle and
against attn_fwd_paged with caller-provided scratch.

The no-allocation entry point serves callers that cannot allocate device
memory at call time (a plugin whose host engine owns every allocation, a
serving loop that must not call cudaMalloc because it can synchronise the
device).  It takes its split-KV scratch from a fixed array inside the
library instead of caller buffers.  Calls in a row, with different shapes
and split counts, must each match the oracle within the parity tolerance of
the other tests and equal attn_fwd_paged bit for bit at the same split
count; the later calls check that what an earlier call left in the shared
array does not leak into them.  Also covered: an automatic split count that
is lowered to fit the array, and a chunked prefill (more than 16 query rows
per kv head) with an explicit split count, which needs no scratch and must
not be rejected.  This file is collected last so a run stopping at the first
failure has already run every other test.
"""
import ctypes
import math

import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import _lib, inputs
from tests._parity import check, f64, no_device_error

pytestmark = pytest.mark.gpu


def _noalloc_via_abi(inp, splits):
    lib = A.library()
    q, kp, vp = inp.q.cuda(), inp.k_pool.cuda(), inp.v_pool.cuda()
    bt, sl = inp.block_table.cuda(), inp.seqlens_k.cuda()
    B, Lq, Hq, d = q.shape
    num_pages, page, Hkv, _ = kp.shape
    o = torch.full((B, Lq, Hq, d), float("nan"), dtype=q.dtype, device="cuda")
    lse = torch.full((B, Hq, Lq), float("nan"), dtype=torch.float32, device="cuda")
    sink = inp.sink.cuda() if inp.sink is not None else None
    opts = _lib.attn_opts(0.0, 1 if inp.causal else 0, float(inp.softcap),
                          sink.data_ptr() if sink is not None else None)
    keep = (q, kp, vp, bt, sl, sink)  # alive until the stream is synchronised
    st = lib.attn_fwd_paged_noalloc(q.data_ptr(), kp.data_ptr(), vp.data_ptr(), bt.data_ptr(),
                                    sl.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Lq, Hq, Hkv,
                                    d, 1 if q.dtype == torch.bfloat16 else 0, page, num_pages,
                                    bt.shape[1], splits, ctypes.byref(opts),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, _lib.STATUS.get(st, st)
    torch.cuda.synchronize()
    del keep
    return o, lse


def _with_scratch(inp, splits):
    o, lse = A.attn_fwd_paged(inp.q.cuda(), inp.k_pool.cuda(), inp.v_pool.cuda(),
                              inp.block_table.cuda(), inp.seqlens_k.cuda(), num_splits=splits,
                              causal=inp.causal, softcap=inp.softcap,
                              sink=inp.sink.cuda() if inp.sink is not None else None)
    torch.cuda.synchronize()
    return o, lse


def _oracle(inp):
    d = inp.q.shape[-1]
    return oracle.attn_paged(f64(inp.q), f64(inp.k_pool), f64(inp.v_pool),
                             inp.block_table.numpy(), inp.seqlens_k.numpy(), 1 / math.sqrt(d),
                             inp.causal, inp.softcap,
                             None if inp.sink is None else f64(inp.sink))


def _case(inp, splits, scratch_splits, what):
    o, lse = _noalloc_via_abi(inp, splits)
    ro, rl = _oracle(inp)
    check(o, lse, ro, rl, f"noalloc {what} vs oracle")
    o_ref, l_ref = _with_scratch(inp, scratch_splits)
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), f"noalloc {what} vs scratch path"


def test_noalloc_calls_in_a_row():
    first = inputs.paged([700, 64, 1, 2000], 1, 32, 8, 128, 64, 60, seed=314, with_sink=True)
    second = inputs.paged([90, 400, 33], 2, 8, 2, 128, 16, 40, seed=2718, causal=True,
                          softcap=30.0)
    for inp, splits in ((first, 4), (second, 3), (first, 2)):
        _case(inp, splits, splits, f"splits={splits}")
    no_device_error()


def test_noalloc_lowers_the_automatic_split_count():
    """B64 Hq32 Hkv8 Lq4 d128 with a 128-column block table: the automatic
    count (4) needs more scratch than the array holds, so the call runs with
    the largest count that fits (3)."""
    B, Lq, Hq, Hkv, d, page, max_pages = 64, 4, 32, 8, 128, 64, 128
    auto = A.attn_paged_auto_splits(B, Hkv, max_pages)
    assert A.attn_paged_workspace_bytes(B, Lq, Hq, d, auto) > _lib.NOALLOC_SCRATCH_BYTES
    fit = auto
    while fit > 1 and A.attn_paged_workspace_bytes(B, Lq, Hq, d, fit) > _lib.NOALLOC_SCRATCH_BYTES:
        fit -= 1
    assert 1 < fit < auto
    lens = inputs.random_lengths(B, 4, 3000, seed=55)
    npages = sum((L + page - 1) // page for L in lens) + 8
    inp = inputs.paged(lens, Lq, Hq, Hkv, d, page, npages, max_pages=max_pages, seed=56,
                       causal=True)
    _case(inp, 0, fit, f"auto splits lowered {auto}->{fit}")
    no_device_error()


def test_noalloc_chunked_prefill_ignores_num_splits():
    """Lq * Hq / Hkv > 16 runs the prefill kernel, which uses no scratch; an
    explicit split count whose nominal scratch would not fit is not rejected."""
    lens, Lq, Hq, Hkv, d, page = [600, 1100, 300], 256, 16, 4, 128, 32
    assert A.attn_paged_workspace_bytes(len(lens), Lq, Hq, d, 64) > _lib.NOALLOC_SCRATCH_BYTES
    npages = sum((L + page - 1) // page for L in lens) + 4
    inp = inputs.paged(lens, Lq, Hq, Hkv, d, page, npages, seed=57, causal=True,
                       with_sink=True)
    _case(inp, 64, 0, "chunked prefill, num_splits=64")
    no_device_error()


def test_noalloc_rejects_scratch_beyond_limit():
    lib = A.library()
    B, Lq, Hq, d, splits = 64, 1, 32, 128, 64
    assert lib.attn_paged_workspace_bytes(B, Lq, Hq, d, splits) > _lib.NOALLOC_SCRATCH_BYTES
    opts = _lib.attn_opts(0.0, 0, 0.0, None)
    p = 1 << 12
    st = lib.attn_fwd_paged_noalloc(p, p, p, p, p, p, None, B, Lq, Hq, 8, d, 1, 64, 10240, 128,
                                    splits, ctypes.byref(opts), None)
    assert st == 1  # ATTN_ERR_INVALID, nothing launched
