"""GPU parity of the additive score terms and the top-left mask alignment
against the fp64 oracle: ALiBi (one slope per (batch, query head), aligned
like the mask) on the dense, group-mode and paged paths; the elementwise bias
on the dense path, full and broadcast, with ragged key counts; top-left causal
and window masks.

The terms follow the Composable Kernel FMHA forward page: the bias kargs
(S'' = S' + Bias), the ALiBi position encoding built from the left/right
window, and MASK_FROM_TOP_LEFT."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import inputs
from tests._parity import check, cuda, f64, no_device_error

pytestmark = pytest.mark.gpu


def _slopes(B, Hq, per_batch, seed):
    g = torch.Generator().manual_seed(seed)
    base = torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=torch.float32)
    if per_batch:
        return base[None, :] * (0.5 + torch.rand((B, Hq), generator=g))
    return base


ALIBI_CASES = [
    # B, Hq, Hkv, Lq, Lk, d, dtype, causal, window, top_left, per_batch
    (2, 4, 2, 300, 300, 128, "bf16", True, None, False, False),
    (1, 4, 4, 200, 700, 64, "f16", False, None, False, True),
    (2, 2, 1, 513, 260, 128, "bf16", True, None, True, True),      # top-left causal, Lq > Lk
    (1, 2, 2, 384, 900, 64, "bf16", False, (100, 40), True, False),  # top-left band
    (1, 2, 2, 640, 640, 128, "bf16", True, (256, -1), False, True),
]


@pytest.mark.parametrize("case", ALIBI_CASES, ids=[str(i) for i in range(len(ALIBI_CASES))])
def test_dense_alibi_parity(case):
    B, Hq, Hkv, Lq, Lk, d, dt, causal, win, tl, per_batch = case
    inp = inputs.dense(B, Hq, Hkv, Lq, Lk, d, dt, seed=51 + Lq + Lk, causal=causal)
    sl = _slopes(B, Hq, per_batch, Lq)
    o, lse = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), causal=causal, window=win,
                        top_left=tl, alibi_slopes=cuda(sl))
    torch.cuda.synchronize()
    assert "_alibi_" in A.attn_last_kernel_name()
    ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), 1 / math.sqrt(d), causal,
                               window=win if win else (-1, -1), top_left=tl, alibi=sl.numpy())
    check(o, lse, ro, rl, f"dense alibi {case}")
    no_device_error()


BIAS_CASES = [
    # B, Hq, Hkv, Lq, Lk, d, dtype, causal, bias shape (B|1, H|1), sink
    (2, 4, 2, 300, 300, 128, "bf16", True, (2, 4), False),
    (1, 2, 2, 200, 333, 64, "f16", False, (1, 2), True),      # ragged keys, per-head broadcast
    (2, 2, 2, 129, 517, 128, "bf16", False, (1, 1), False),   # one bias for all heads
    (1, 4, 4, 640, 640, 64, "bf16", True, (1, 4), False),
]


@pytest.mark.parametrize("case", BIAS_CASES, ids=[str(i) for i in range(len(BIAS_CASES))])
def test_dense_bias_parity(case):
    B, Hq, Hkv, Lq, Lk, d, dt, causal, (bb, bh), sink = case
    inp = inputs.dense(B, Hq, Hkv, Lq, Lk, d, dt, seed=71 + Lq + Lk, causal=causal,
                       with_sink=sink)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    g = torch.Generator().manual_seed(Lk)
    lk_pad = (Lk + 7) // 8 * 8 + 8  # row stride a multiple of 8, with slack past Lk
    store = (torch.randn((bb, bh, Lq, lk_pad), generator=g) * 1.5).to(tdt)
    bias = store[..., :Lk]
    o, lse = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), causal=causal,
                        sink=cuda(inp.sink), bias=cuda(store)[..., :Lk])
    torch.cuda.synchronize()
    assert "_bias_" in A.attn_last_kernel_name()
    ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), 1 / math.sqrt(d), causal,
                               sink=None if inp.sink is None else f64(inp.sink),
                               bias=f64(bias))
    check(o, lse, ro, rl, f"dense bias {case}")
    no_device_error()


def test_bias_of_minus_inf_above_diagonal_is_causal():
    """A bias holding -inf above the bottom-right diagonal reproduces the
    causal kernel's output (same rows kept; the remaining bias is zero)."""
    B, H, L, d = 1, 2, 300, 128
    inp = inputs.dense(B, H, H, L, L, d, "bf16", seed=5)
    i = torch.arange(L)[:, None]
    j = torch.arange(L)[None, :]
    neg = torch.where(j > i, float("-inf"), 0.0).to(torch.bfloat16)
    store = torch.zeros((1, 1, L, 304), dtype=torch.bfloat16)
    store[..., :L] = neg
    o1, l1 = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), bias=cuda(store)[..., :L])
    o2, l2 = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), 1 / math.sqrt(d), True)
    check(o1, l1, ro, rl, "bias -inf causal")
    check(o2, l2, ro, rl, "causal")
    no_device_error()


def test_top_left_causal_dense_and_varlen():
    inp = inputs.dense(1, 4, 2, 700, 300, 128, "bf16", seed=9, causal=True)
    o, lse = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), causal=True, top_left=True)
    torch.cuda.synchronize()
    assert "_topleft_" in A.attn_last_kernel_name()
    ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), 1 / math.sqrt(128), True,
                               top_left=True)
    check(o, lse, ro, rl, "top-left causal Lq > Lk")
    lq, lk = [5, 300, 129, 1], [700, 100, 129, 40]
    vin = inputs.varlen(lq, lk, 4, 2, 64, "bf16", seed=13, causal=True)
    sl = _slopes(4, 4, True, 3)
    o, lse = A.attn_fwd_varlen(cuda(vin.q), cuda(vin.k), cuda(vin.v), cuda(vin.cu_seqlens_q),
                               cuda(vin.cu_seqlens_k), vin.max_seqlen_q, causal=True,
                               top_left=True, alibi_slopes=cuda(sl))
    torch.cuda.synchronize()
    ro, rl = oracle.attn_varlen(f64(vin.q), f64(vin.k), f64(vin.v), vin.cu_seqlens_q.numpy(),
                                vin.cu_seqlens_k.numpy(), 1 / math.sqrt(64), True, top_left=True,
                                alibi=sl.numpy())
    check(o, lse, ro, rl, "varlen top-left causal alibi")
    no_device_error()


PAGED_CASES = [
    # lens, Lq, Hq, Hkv, d, page, splits, causal, window, top_left
    ([1, 64, 700], 1, 8, 2, 128, 64, 3, False, None, False),
    ([50, 1290], 4, 8, 2, 128, 32, 2, True, None, False),
    ([90, 911], 2, 4, 4, 64, 128, 4, True, (100, -1), True),
    ([4096], 1, 16, 1, 128, 64, 0, False, (1000, -1), False),
]


@pytest.mark.parametrize("case", PAGED_CASES, ids=[str(i) for i in range(len(PAGED_CASES))])
def test_paged_alibi_parity(case):
    lens, Lq, Hq, Hkv, d, page, splits, causal, win, tl = case
    npages = sum((L + page - 1) // page for L in lens) + 5
    inp = inputs.paged(lens, Lq, Hq, Hkv, d, page, npages, seed=len(lens) + page + 11,
                       causal=causal)
    sl = _slopes(len(lens), Hq, True, page)
    o, lse = A.attn_fwd_paged(cuda(inp.q), cuda(inp.k_pool), cuda(inp.v_pool),
                              cuda(inp.block_table), cuda(inp.seqlens_k), num_splits=splits,
                              causal=causal, window=win, top_left=tl, alibi_slopes=cuda(sl))
    torch.cuda.synchronize()
    ro, rl = oracle.attn_paged(f64(inp.q), f64(inp.k_pool), f64(inp.v_pool),
                               inp.block_table.numpy(), inp.seqlens_k.numpy(), 1 / math.sqrt(d),
                               causal, window=win if win else (-1, -1), top_left=tl,
                               alibi=sl.numpy())
    check(o, lse, ro, rl, f"paged alibi {case}")
    no_device_error()
