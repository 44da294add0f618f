"""The prefill kernel's work order in group mode, over a paged cache, and
on the host-packed static schedule of dense masked problems.

In group mode and over a paged cache the (query block, sequence) slots are
sorted by their K/V step count in every CTA before any work starts; more than 2048 slots fall back to the plain
order, and step counts above 254 share the top cost.  The order decides only
which CTA computes an item, never how, so every case here must match the
oracle and the per-sequence dense results exactly as any other order would.
Dense problems with a causal or window mask run each CTA's list from a
schedule packed on the host (longest processing time first); a lone
(batch, head) has fewer blocks than CTAs and keeps the plain order.

Composable Kernel FMHA forward page: group mode (seqstart_q / seqstart_k)
and the paged-KV block table; the sort is this implementation's schedule."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import inputs
from tests._parity import check, cuda, f64, no_device_error

pytestmark = pytest.mark.gpu


def test_varlen_more_slots_than_the_sort_takes():
    """520 sequences with max_seqlen_q 1024 give 4 x 520 = 2080 slots, past
    the sort's 2048: the plain order runs and every row still matches."""
    g = torch.Generator().manual_seed(520)
    lens = [1024] + [int(x) for x in torch.randint(1, 41, (519,), generator=g)]
    inp = inputs.varlen(lens, lens, 2, 1, 64, "bf16", seed=520, causal=True)
    assert inp.max_seqlen_q == 1024 and 4 * len(lens) > 2048
    o, lse = A.attn_fwd_varlen(cuda(inp.q), cuda(inp.k), cuda(inp.v), cuda(inp.cu_seqlens_q),
                               cuda(inp.cu_seqlens_k), inp.max_seqlen_q, causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_varlen(f64(inp.q), f64(inp.k), f64(inp.v), inp.cu_seqlens_q.numpy(),
                                inp.cu_seqlens_k.numpy(), 1 / math.sqrt(64), True)
    check(o, lse, ro, rl, "varlen, plain order")
    no_device_error()


@pytest.mark.parametrize("causal", [True, False])
def test_varlen_sorted_order_equals_per_sequence_dense(causal):
    """Sequences of very different lengths (their slots sort far from the
    plain order): each sequence's rows are bit-identical to the dense kernel
    run on that sequence alone."""
    lens = [1500, 3, 700, 0, 129, 2049, 256]
    H, Hkv, d = 4, 2, 128
    inp = inputs.varlen(lens, lens, H, Hkv, d, "bf16", seed=77, causal=causal)
    o, lse = A.attn_fwd_varlen(cuda(inp.q), cuda(inp.k), cuda(inp.v), cuda(inp.cu_seqlens_q),
                               cuda(inp.cu_seqlens_k), inp.max_seqlen_q, causal=causal)
    torch.cuda.synchronize()
    cu = inp.cu_seqlens_q.tolist()
    for b, L in enumerate(lens):
        if L == 0:
            continue
        s0, s1 = cu[b], cu[b + 1]
        q = cuda(inp.q[s0:s1].transpose(0, 1)[None].contiguous())
        k = cuda(inp.k[s0:s1].transpose(0, 1)[None].contiguous())
        v = cuda(inp.v[s0:s1].transpose(0, 1)[None].contiguous())
        od, ld = A.attn_fwd(q, k, v, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(od[0].transpose(0, 1), o[s0:s1]), f"sequence {b}"
        assert torch.equal(ld[0], lse[:, s0:s1]), f"sequence {b} LSE"
    no_device_error()


def test_paged_chunk_over_a_cache_past_the_top_cost():
    """A chunk of 256 queries over a 40000-key cache (313 K/V steps, past the
    top cost of 254) beside short caches: sampled rows of the long sequence
    and the short sequences in full match the oracle."""
    lens = [40000, 300, 2000, 256]
    Lq, Hq, Hkv, d, page = 256, 4, 2, 128, 64
    npages = sum((L + page - 1) // page for L in lens) + 4
    inp = inputs.paged(lens, Lq, Hq, Hkv, d, page, npages, seed=313, causal=True)
    o, lse = A.attn_fwd_paged(cuda(inp.q), cuda(inp.k_pool), cuda(inp.v_pool),
                              cuda(inp.block_table), cuda(inp.seqlens_k), causal=True)
    torch.cuda.synchronize()
    assert A.attn_last_kernel_name().startswith("attn_prefill_tcgen05")
    short = [1, 2, 3]
    ro, rl = oracle.attn_paged(f64(inp.q[short]), f64(inp.k_pool), f64(inp.v_pool),
                               inp.block_table[short].numpy(), inp.seqlens_k[short].numpy(),
                               1 / math.sqrt(d), True)
    check(o[short], lse[short], ro, rl, "short caches")
    # the long sequence, two heads, rows [192, 256): gather its cache
    L = lens[0]
    pages = inp.block_table[0, : (L + page - 1) // page].long()
    for h in (0, 3):
        hk = h // (Hq // Hkv)
        kc = inp.k_pool[pages].reshape(-1, Hkv, d)[:L, hk]
        vc = inp.v_pool[pages].reshape(-1, Hkv, d)[:L, hk]
        r0, r1 = 192, 256
        # rows r0..r1 of the chunk: bottom-right alignment keeps keys < L - Lq + row + 1
        keep = L - Lq + r1
        ro, rl = oracle.attn_dense(f64(inp.q[0, r0:r1, h])[None, None], f64(kc[:keep])[None, None],
                                   f64(vc[:keep])[None, None], 1 / math.sqrt(d), True)
        check(o[0, r0:r1, h][None, None], lse[0, h, r0:r1][None, None], ro, rl, f"long seq h{h}")
    no_device_error()


@pytest.mark.parametrize("window,top_left", [(None, False), ((700, 0), False), ((300, 200), True)])
def test_dense_static_schedule_equals_single_head(window, top_left):
    """A dense masked problem with more query blocks than CTAs runs on the
    host-packed static schedule; a single (batch, head) has fewer blocks than
    CTAs and runs one block per CTA.  Both compute every block the same way,
    so sampled heads are bit-identical between the two launches."""
    B, H, L, d = 2, 16, 4096, 128
    causal = window is None
    inp = inputs.dense(B, H, H, L, L, d, "bf16", seed=4096, device="cuda", causal=True)
    o, lse = A.attn_fwd(inp.q, inp.k, inp.v, causal=causal, window=window, top_left=top_left)
    torch.cuda.synchronize()
    for b, h in [(0, 0), (1, 7), (1, 15)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        o1, l1 = A.attn_fwd(inp.q[sl].contiguous(), inp.k[sl].contiguous(), inp.v[sl].contiguous(),
                            causal=causal, window=window, top_left=top_left)
        torch.cuda.synchronize()
        assert torch.equal(o1, o[sl]), f"b{b} h{h}"
        assert torch.equal(l1, lse[sl]), f"b{b} h{h} LSE"
    no_device_error()


def test_dense_schedule_with_keyless_blocks():
    """Lq 3000 > Lk 1000, causal (bottom-right): rows below 2000 keep no key,
    so most query blocks cost only their fixed share; the 768 blocks of
    4 x 16 heads run on the static schedule.  Keyless rows give O = 0 and
    LSE = -inf; the other rows of sampled heads match the oracle."""
    B, H, Lq, Lk, d = 4, 16, 3000, 1000, 128
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert A.attn_dense_schedule(B, H, Lq, Lk, min(sms, 768), causal=True) is not None
    inp = inputs.dense(B, H, H, Lq, Lk, d, "bf16", seed=3000, device="cuda", causal=True)
    o, lse = A.attn_fwd(inp.q, inp.k, inp.v, causal=True)
    torch.cuda.synchronize()
    cut = Lq - Lk
    assert torch.all(o[:, :, :cut] == 0)
    assert torch.all(torch.isneginf(lse[:, :, :cut]))
    for b, h in [(0, 0), (1, 7), (3, 15)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ro, rl = oracle.attn_dense(f64(inp.q[sl][:, :, cut:]), f64(inp.k[sl]), f64(inp.v[sl]),
                                   1 / math.sqrt(d), True)
        check(o[sl][:, :, cut:], lse[sl][:, :, cut:], ro, rl, f"keyless blocks b{b} h{h}")
    no_device_error()
