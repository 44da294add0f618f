"""GPU parity of chunked prefill over a paged KV cache (attn_fwd_paged with
Lq * g > 16: the prefill kernel with its K/V tiles gathered through the
block table) against the fp64 oracle.

Composable Kernel paged-KV kernel (page block navigator: key j of sequence b
is row j mod page of physical page block_table[b][j / page]); the chunk's
queries are the last Lq positions of each sequence (bottom-right masks)."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import inputs
from tests._parity import check, cuda, f64, no_device_error

pytestmark = pytest.mark.gpu

CASES = [
    # lens, Lq, Hq, Hkv, d, page, dtype, causal, softcap, sink, window, top_left, alibi
    ([300, 1000, 64], 64, 8, 2, 128, 64, "bf16", True, 0.0, False, None, False, False),
    ([2000, 513], 300, 4, 4, 64, 16, "bf16", True, 30.0, True, None, False, False),
    ([777], 129, 16, 1, 128, 256, "f16", False, 0.0, False, None, False, False),
    ([1500, 40], 200, 8, 2, 128, 32, "bf16", True, 0.0, False, (256, -1), False, False),
    ([900, 300], 100, 4, 2, 64, 128, "bf16", True, 0.0, False, None, True, True),
    ([50, 600, 0], 100, 8, 8, 128, 64, "bf16", True, 0.0, True, None, False, False),  # L < Lq, L = 0
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_paged_prefill_parity(case):
    lens, Lq, Hq, Hkv, d, page, dt, causal, cap, sink, win, tl, alibi = case
    npages = sum((L + page - 1) // page for L in lens) + 7
    inp = inputs.paged(lens, Lq, Hq, Hkv, d, page, npages, dtype=dt, seed=sum(lens) + Lq,
                       causal=causal, softcap=cap, with_sink=sink)
    sl = None
    if alibi:
        sl = torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=torch.float32)
    o, lse = A.attn_fwd_paged(cuda(inp.q), cuda(inp.k_pool), cuda(inp.v_pool),
                              cuda(inp.block_table), cuda(inp.seqlens_k), causal=causal,
                              softcap=cap, sink=cuda(inp.sink), window=win, top_left=tl,
                              alibi_slopes=cuda(sl))
    torch.cuda.synchronize()
    assert A.attn_last_kernel_name().startswith("attn_prefill_tcgen05")
    ro, rl = oracle.attn_paged(f64(inp.q), f64(inp.k_pool), f64(inp.v_pool),
                               inp.block_table.numpy(), inp.seqlens_k.numpy(), 1 / math.sqrt(d),
                               causal, cap, None if inp.sink is None else f64(inp.sink),
                               window=win if win else (-1, -1), top_left=tl,
                               alibi=None if sl is None else sl.numpy())
    check(o, lse, ro, rl, f"paged prefill {case}")
    no_device_error()


def test_paged_prefill_matches_dense_on_a_gathered_cache():
    """The same chunk through the paged path and through attn_fwd on the
    gathered contiguous K/V gives the same rows (both kernels are the same
    prefill kernel; only the K/V addressing differs)."""
    lens, Lq, H, d, page = [1000, 700], 256, 8, 128, 32
    inp = inputs.paged(lens, Lq, H, H, d, page, sum((L + page - 1) // page for L in lens) + 3,
                       seed=77, causal=True)
    o, lse = A.attn_fwd_paged(cuda(inp.q), cuda(inp.k_pool), cuda(inp.v_pool),
                              cuda(inp.block_table), cuda(inp.seqlens_k), causal=True)
    torch.cuda.synchronize()
    for b, L in enumerate(lens):
        pages = inp.block_table[b, : (L + page - 1) // page].long()
        kc = inp.k_pool[pages].reshape(-1, H, d)[:L].transpose(0, 1)[None].contiguous()
        vc = inp.v_pool[pages].reshape(-1, H, d)[:L].transpose(0, 1)[None].contiguous()
        qd = inp.q[b:b + 1].transpose(1, 2).contiguous()
        od, ld = A.attn_fwd(cuda(qd), cuda(kc), cuda(vc), causal=True)
        torch.cuda.synchronize()
        assert torch.equal(od[0].transpose(0, 1), o[b]), f"sequence {b}"
        assert torch.equal(ld[0], lse[b])
    no_device_error()


def test_chunked_prefill_workload_sampled():
    """The chunked-prefill workload (8 sequences of U[2048, 8192] cached keys,
    chunk of 512 queries, Hq 32 / Hkv 8, d 128, page 64, causal): sampled
    (sequence, head) pairs against the oracle on those rows."""
    lens = inputs.random_lengths(8, 2048, 8192, seed=1010)
    Lq, Hq, Hkv, d, page = 512, 32, 8, 128, 64
    npages = sum((L + page - 1) // page for L in lens) + 16
    inp = inputs.paged(lens, Lq, Hq, Hkv, d, page, npages, seed=1010, device="cuda", causal=True)
    o, lse = A.attn_fwd_paged(inp.q, inp.k_pool, inp.v_pool, inp.block_table.cuda(),
                              inp.seqlens_k.cuda(), causal=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    for _ in range(4):
        b = int(rng.integers(len(lens)))
        h = int(rng.integers(Hq))
        L = lens[b]
        pages = inp.block_table[b, : (L + page - 1) // page].long().cuda()
        hk = h // (Hq // Hkv)
        kc = inp.k_pool[pages].reshape(-1, Hkv, d)[:L, hk]
        vc = inp.v_pool[pages].reshape(-1, Hkv, d)[:L, hk]
        ro, rl = oracle.attn_dense(f64(inp.q[b, :, h])[None, None], f64(kc)[None, None],
                                   f64(vc)[None, None], 1 / math.sqrt(d), True)
        check(o[b, :, h][None, None], lse[b, h][None, None], ro, rl, f"sampled b{b} h{h}")
    no_device_error()
