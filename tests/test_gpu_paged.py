"""GPU parity of the paged-KV split-KV kernel and the split combine against the
fp64 oracle, including empty sequences, partial last pages, empty splits,
causal chunks; the full-size decode workload is compared whole in
test_gpu_full_size.py."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import inputs
from tests._parity import check, cuda, f64, no_device_error

pytestmark = pytest.mark.gpu

PAGED_CASES = [
    # lens, Lq, Hq, Hkv, d, page, splits, dtype, causal, softcap, sink
    ([1, 64, 200], 1, 8, 2, 128, 64, 1, "bf16", False, 0.0, False),
    ([1, 64, 200], 1, 8, 2, 128, 64, 3, "bf16", False, 0.0, False),   # empty splits
    ([0, 17, 300], 1, 8, 2, 128, 16, 0, "bf16", False, 0.0, True),    # L = 0, auto splits
    ([700, 5], 1, 4, 4, 64, 256, 2, "f16", False, 0.0, False),        # big pages, d = 64
    ([50, 129], 4, 8, 2, 128, 32, 2, "bf16", True, 0.0, False),       # Lq*g = 16, causal
    ([333, 1000, 64], 1, 32, 8, 128, 64, 4, "bf16", False, 30.0, True),
    ([90, 91], 2, 4, 4, 128, 128, 1, "f16", True, 0.0, True),         # g = 1, Lq = 2
    ([4096], 1, 16, 1, 128, 64, 5, "bf16", False, 0.0, False),        # MQA g = 16
]


def _run_paged(inp, splits):
    q, kp, vp = cuda(inp.q), cuda(inp.k_pool), cuda(inp.v_pool)
    bt, sl = cuda(inp.block_table), cuda(inp.seqlens_k)
    return A.attn_fwd_paged(q, kp, vp, bt, sl, num_splits=splits, causal=inp.causal,
                            softcap=inp.softcap, sink=cuda(inp.sink))


@pytest.mark.parametrize("case", PAGED_CASES, ids=[str(i) for i in range(len(PAGED_CASES))])
def test_paged_parity(case):
    lens, Lq, Hq, Hkv, d, page, splits, dt, causal, cap, sink = case
    npages = sum((L + page - 1) // page for L in lens) + 5
    inp = inputs.paged(lens, Lq, Hq, Hkv, d, page, npages, dtype=dt, seed=len(lens) + page + d,
                       causal=causal, softcap=cap, with_sink=sink)
    o, lse = _run_paged(inp, splits)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_paged(f64(inp.q), f64(inp.k_pool), f64(inp.v_pool),
                               inp.block_table.numpy(), inp.seqlens_k.numpy(), 1 / math.sqrt(d),
                               causal, cap, None if inp.sink is None else f64(inp.sink))
    check(o, lse, ro, rl, "paged")
    no_device_error()


def test_paged_partials_match_oracle_splits():
    """The per-split partial O/LSE the kernel writes equal the oracle's split
    partials (same split convention), before the combine."""
    lens, Lq, Hq, Hkv, d, page, S = [1, 130, 640, 0], 1, 8, 2, 128, 64, 4
    inp = inputs.paged(lens, Lq, Hq, Hkv, d, page, 30, seed=99)
    B = len(lens)
    rows = B * Hq * Lq
    ws = torch.full((S * rows * (d + 1),), float("nan"), dtype=torch.float32, device="cuda")
    A.attn_fwd_paged(cuda(inp.q), cuda(inp.k_pool), cuda(inp.v_pool), cuda(inp.block_table),
                     cuda(inp.seqlens_k), num_splits=S, workspace=ws)
    torch.cuda.synchronize()
    op = ws[: S * rows * d].view(S, B, Hq, Lq, d)
    lp = ws[S * rows * d:].view(S, B, Hq, Lq)
    max_pages = inp.block_table.shape[1]
    chunk = (max_pages + S - 1) // S
    ro, rl = oracle.attn_paged_partials(f64(inp.q), f64(inp.k_pool), f64(inp.v_pool),
                                        inp.block_table.numpy(), inp.seqlens_k.numpy(), S, chunk,
                                        1 / math.sqrt(d))
    lg = f64(lp)
    assert np.array_equal(np.isneginf(lg), np.isneginf(rl))
    live = ~np.isneginf(rl)
    assert np.abs(lg[live] - rl[live]).max() <= 1e-3
    og = f64(op)
    err = np.abs(og - ro)[np.broadcast_to(live[..., None], og.shape)]
    assert err.max() <= 2e-2
    no_device_error()


def test_combine_parity():
    g = torch.Generator().manual_seed(5)
    for S, B, Hq, Lq, d, sink in ((1, 2, 4, 1, 128, False), (5, 3, 8, 2, 128, True),
                                  (7, 2, 2, 3, 64, False), (64, 1, 2, 1, 128, True)):
        op = torch.randn((S, B, Hq, Lq, d), generator=g)
        lp = 3 * torch.randn((S, B, Hq, Lq), generator=g)
        drop = torch.rand((S, B, Hq, Lq), generator=g) < 0.3
        lp[drop] = float("-inf")
        lp[:, 0, 0, 0] = float("-inf")  # a row with every split empty
        sk = torch.randn(Hq, generator=g) if sink else None
        o, lse = A.attn_splitkv_combine(op.cuda(), lp.cuda(), sink=cuda(sk))
        torch.cuda.synchronize()
        rows = B * Hq * Lq
        sink_rows = None
        if sk is not None:
            sink_rows = np.broadcast_to(f64(sk)[None, :, None], (B, Hq, Lq)).reshape(-1)
        ro, rl = oracle.combine(f64(op).reshape(S, rows, d), f64(lp).reshape(S, rows), sink_rows)
        check(o, lse, ro.reshape(B, Hq, Lq, d).transpose(0, 2, 1, 3), rl.reshape(B, Hq, Lq),
              f"combine S={S}")
    no_device_error()


def test_split_results_are_repeatable_and_match_one_split():
    """The split-KV path is deterministic (fixed reduction orders), so three
    runs agree bit for bit, and with 4 or 8 splits it agrees with the single
    split within two bf16 steps at |O| < 1 (0.01): a lost or duplicated P.V
    contribution, as from a partial O read before its last P.V completes,
    shows up far above that."""
    inp = inputs.workload(4, device="cuda")
    bt, sl = inp.block_table.cuda(), inp.seqlens_k.cuda()
    o1, l1 = A.attn_fwd_paged(inp.q, inp.k_pool, inp.v_pool, bt, sl, num_splits=1)
    outs = []
    for splits in (4, 4, 4, 8):
        o, lse = A.attn_fwd_paged(inp.q, inp.k_pool, inp.v_pool, bt, sl, num_splits=splits)
        torch.cuda.synchronize()
        outs.append((splits, o.clone(), lse.clone()))
    for _, o, lse in outs[1:3]:
        assert torch.equal(o, outs[0][1]) and torch.equal(lse, outs[0][2])
    for splits, o, lse in outs:
        err = (o.float() - o1.float()).abs().max().item()
        assert err <= 0.01, (splits, err)
        assert (lse - l1).abs().max().item() <= 1e-4
    no_device_error()


def test_timeout_path_reports_and_recovers():
    """A kernel whose wait can never complete gives up after its limit, sets
    the error word and returns; the context stays usable."""
    A.attn_selftest_timeout(20_000_000)  # 20 ms
    bits = A.attn_device_error()
    assert bits & (1 << 20)
    assert A.attn_device_error() == 0  # read-and-clear
    inp = inputs.dense(1, 2, 2, 64, 64, 64, "bf16", seed=1)
    o, lse = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v))
    torch.cuda.synchronize()
    ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), 1 / 8.0)
    check(o, lse, ro, rl, "after timeout")
    no_device_error()
