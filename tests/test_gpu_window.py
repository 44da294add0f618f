"""GPU parity of the sliding-window (local attention band) mask against the
fp64 oracle: dense, group-mode and paged problems, windows that cut tile
boundaries, one-sided and two-sided bands, a band combined with causal, rows
the band leaves without keys, and the paged split layout over the band.

The mask is the Composable Kernel FMHA forward kernel's mask built from
window_size_left / window_size_right (fmha_fwd_pagedkv_kernel.hpp, the mask
kernel arguments and the mask set-up of operator()), bottom-right aligned like
the causal mask."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import inputs
from tests._parity import check, cuda, f64, no_device_error

pytestmark = pytest.mark.gpu

DENSE_WINDOW_CASES = [
    # B, Hq, Hkv, Lq, Lk, d, dtype, causal, window, softcap, sink
    (1, 2, 2, 700, 700, 128, "bf16", False, (100, 50), 0.0, False),   # two-sided band
    (1, 2, 2, 600, 600, 64, "f16", True, (128, -1), 0.0, False),      # causal sliding window
    (1, 4, 2, 300, 900, 128, "bf16", False, (0, 0), 0.0, False),      # diagonal only, Lq < Lk
    (1, 2, 2, 900, 300, 128, "bf16", True, (64, -1), 0.0, False),     # Lq > Lk: keyless rows
    (1, 2, 2, 1024, 1024, 128, "bf16", False, (-1, 10), 0.0, False),  # right bound only
    (1, 4, 4, 520, 520, 64, "bf16", True, (300, -1), 30.0, True),     # softcap + sink
    (2, 4, 4, 1000, 1000, 128, "bf16", False, (5, 5), 0.0, False),    # narrow band
    (1, 2, 2, 385, 385, 128, "f16", False, (127, 128), 0.0, True),    # band of exactly one tile
    (1, 2, 1, 260, 1300, 64, "bf16", True, (2000, -1), 0.0, False),   # band wider than keys
]


@pytest.mark.parametrize("case", DENSE_WINDOW_CASES,
                         ids=[str(i) for i in range(len(DENSE_WINDOW_CASES))])
def test_dense_window_parity(case):
    B, Hq, Hkv, Lq, Lk, d, dt, causal, win, cap, sink = case
    inp = inputs.dense(B, Hq, Hkv, Lq, Lk, d, dt, seed=31 + Lq + Lk, value_scale=2.0 if cap else 1.0,
                       causal=causal, softcap=cap, with_sink=sink)
    o, lse = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), causal=causal, softcap=cap,
                        sink=cuda(inp.sink), window=win)
    torch.cuda.synchronize()
    assert "_window_" in A.attn_last_kernel_name() or (causal and win[1] < 0 and win[0] < 0)
    ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), 1 / math.sqrt(d), causal, cap,
                               None if inp.sink is None else f64(inp.sink), window=win)
    check(o, lse, ro, rl, f"dense window {win}")
    no_device_error()


def test_unbounded_window_is_the_unmasked_kernel():
    """A window with both sides negative selects the unmasked kernel; a band
    wider than every sequence runs the masked kernel but masks nothing, and the
    result is bit-identical (the per-tile arithmetic does not depend on the
    order the tiles are visited in)."""
    inp = inputs.dense(1, 4, 4, 700, 700, 128, "bf16", seed=8)
    q, k, v = cuda(inp.q), cuda(inp.k), cuda(inp.v)
    o0, l0 = A.attn_fwd(q, k, v)
    n0 = A.attn_last_kernel_name()
    o1, l1 = A.attn_fwd(q, k, v, window=(-1, -1))
    n1 = A.attn_last_kernel_name()
    o2, l2 = A.attn_fwd(q, k, v, window=(5000, 5000))
    n2 = A.attn_last_kernel_name()
    torch.cuda.synchronize()
    assert "_nomask_" in n0 and n1 == n0 and "_window_" in n2
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    assert torch.equal(o0, o2) and torch.equal(l0, l2)
    no_device_error()


VARLEN_WINDOW_CASES = [
    # lens_q, lens_k, Hq, Hkv, d, dtype, causal, window
    ([1, 0, 130, 257, 500], None, 4, 2, 128, "bf16", True, (64, -1)),
    ([5, 100, 64], [300, 100, 1], 2, 2, 64, "f16", False, (32, 16)),
    ([513, 1, 129], [513, 1000, 0], 8, 2, 128, "bf16", False, (200, 0)),
]


@pytest.mark.parametrize("case", VARLEN_WINDOW_CASES,
                         ids=[str(i) for i in range(len(VARLEN_WINDOW_CASES))])
def test_varlen_window_parity(case):
    lq, lk, Hq, Hkv, d, dt, causal, win = case
    lk = lk if lk is not None else lq
    inp = inputs.varlen(lq, lk, Hq, Hkv, d, dt, seed=sum(lq) + 17, causal=causal)
    o, lse = A.attn_fwd_varlen(cuda(inp.q), cuda(inp.k), cuda(inp.v), cuda(inp.cu_seqlens_q),
                               cuda(inp.cu_seqlens_k), inp.max_seqlen_q, causal=causal,
                               window=win)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_varlen(f64(inp.q), f64(inp.k), f64(inp.v), inp.cu_seqlens_q.numpy(),
                                inp.cu_seqlens_k.numpy(), 1 / math.sqrt(d), causal, window=win)
    check(o, lse, ro, rl, f"varlen window {win}")
    no_device_error()


PAGED_WINDOW_CASES = [
    # lens, Lq, Hq, Hkv, d, page, splits, causal, window
    ([1, 64, 700], 1, 8, 2, 128, 64, 1, True, (100, -1)),
    ([1, 64, 700], 1, 8, 2, 128, 64, 3, True, (100, -1)),     # splits tile the band
    ([0, 17, 3000], 1, 8, 2, 128, 16, 0, False, (500, 0)),    # auto splits over W
    ([50, 1290], 4, 8, 2, 128, 32, 2, True, (40, -1)),        # Lq * g = 16
    ([90, 911], 2, 4, 4, 64, 128, 4, False, (0, 0)),          # diagonal only
    ([4096], 1, 16, 1, 128, 64, 5, False, (1000, -1)),        # MQA
]


@pytest.mark.parametrize("case", PAGED_WINDOW_CASES,
                         ids=[str(i) for i in range(len(PAGED_WINDOW_CASES))])
def test_paged_window_parity(case):
    lens, Lq, Hq, Hkv, d, page, splits, causal, win = case
    npages = sum((L + page - 1) // page for L in lens) + 5
    inp = inputs.paged(lens, Lq, Hq, Hkv, d, page, npages, seed=len(lens) + page + d + 3,
                       causal=causal)
    o, lse = A.attn_fwd_paged(cuda(inp.q), cuda(inp.k_pool), cuda(inp.v_pool),
                              cuda(inp.block_table), cuda(inp.seqlens_k), num_splits=splits,
                              causal=causal, window=win)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_paged(f64(inp.q), f64(inp.k_pool), f64(inp.v_pool),
                               inp.block_table.numpy(), inp.seqlens_k.numpy(), 1 / math.sqrt(d),
                               causal, window=win)
    check(o, lse, ro, rl, f"paged window {win}")
    no_device_error()


def test_paged_window_partials_follow_the_band_layout():
    """With a left window the splits tile the pages from the first kept key on
    (W = attn_paged_window_pages); each split's partial O/LSE equals the
    oracle's partial over the same pages."""
    lens, Lq, Hq, Hkv, d, page, S, win = [1, 130, 2000, 0, 777], 1, 8, 2, 128, 64, 3, (300, -1)
    inp = inputs.paged(lens, Lq, Hq, Hkv, d, page, 60, seed=123)
    B = len(lens)
    rows = B * Hq * Lq
    ws = torch.full((S * rows * (d + 1),), float("nan"), dtype=torch.float32, device="cuda")
    A.attn_fwd_paged(cuda(inp.q), cuda(inp.k_pool), cuda(inp.v_pool), cuda(inp.block_table),
                     cuda(inp.seqlens_k), num_splits=S, workspace=ws, window=win)
    torch.cuda.synchronize()
    op = ws[: S * rows * d].view(S, B, Hq, Lq, d)
    lp = ws[S * rows * d:].view(S, B, Hq, Lq)
    W = A.attn_paged_window_pages(Lq, page, inp.block_table.shape[1], window=win)
    assert W == min(inp.block_table.shape[1], (Lq + win[0] + page - 1) // page + 1)
    chunk = (W + S - 1) // S
    ro, rl = oracle.attn_paged_partials(f64(inp.q), f64(inp.k_pool), f64(inp.v_pool),
                                        inp.block_table.numpy(), inp.seqlens_k.numpy(), S, chunk,
                                        1 / math.sqrt(d), window=win)
    lg = f64(lp)
    assert np.array_equal(np.isneginf(lg), np.isneginf(rl))
    live = ~np.isneginf(rl)
    assert np.abs(lg[live] - rl[live]).max() <= 1e-3
    og = f64(op)
    err = np.abs(og - ro)[np.broadcast_to(live[..., None], og.shape)]
    assert err.max() <= 2e-2
    no_device_error()


def test_sliding_window_full_size_sampled():
    """Causal sliding window of 512 keys on the dense B4 H16 L2048 d128 shape:
    sampled (batch, head, row-range) blocks against the oracle on those rows
    (the key range is cut at the last sampled row's diagonal, which keeps
    every row's band identical to the full problem)."""
    B, H, L, d, win = 4, 16, 2048, 128, (512, -1)
    inp = inputs.dense(B, H, H, L, L, d, "bf16", seed=2024, device="cuda", causal=True)
    o, lse = A.attn_fwd(inp.q, inp.k, inp.v, causal=True, window=win)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    for _ in range(6):
        b, h = int(rng.integers(B)), int(rng.integers(H))
        r0 = int(rng.integers(0, L - 64))
        r1 = r0 + 64
        qs = f64(inp.q[b:b + 1, h:h + 1, r0:r1])
        ks = f64(inp.k[b:b + 1, h:h + 1, :r1])
        vs = f64(inp.v[b:b + 1, h:h + 1, :r1])
        ro, rl = oracle.attn_dense(qs, ks, vs, 1 / math.sqrt(d), True, window=win)
        check(o[b:b + 1, h:h + 1, r0:r1], lse[b:b + 1, h:h + 1, r0:r1], ro, rl,
              f"sampled b{b} h{h} rows {r0}:{r1}")
    no_device_error()
