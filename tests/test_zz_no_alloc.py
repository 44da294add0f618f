"""attn_fwd_paged_noalloc against attn_fwd_paged, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device
memory at call time (a plugin whose host engine owns every allocation, a
serving loop that must not call cudaMalloc because it can synchronise the
device).  It takes its split-KV scratch from a fixed array inside the
library instead of caller buffers.  Two calls in a row, with different
shapes and split counts, must each give the result of attn_fwd_paged with
caller-provided scratch, within the parity tolerance of the other tests; the
second call checks that what the first left in the shared array does not
leak into it.  This file is collected last so a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

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


def test_noalloc_matches_scratch_path_two_calls():
    first = inputs.paged([700, 64, 1, 2000], 1, 32, 8, 128, 64, 60, seed=314, with_sink=True)
    second = inputs.paged([90, 400, 33], 2, 8, 2, 128, 16, 40, seed=2718, causal=True,
                          softcap=30.0)
    for inp, splits in ((first, 4), (second, 3)):
        o_ref, l_ref = _with_scratch(inp, splits)
        o, lse = _noalloc_via_abi(inp, splits)
        check(o, lse, f64(o_ref), f64(l_ref), f"noalloc splits={splits}")
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
