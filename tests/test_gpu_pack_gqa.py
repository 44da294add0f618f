"""PackGQA in the prefill kernel (FlashAttention-3 epilogue, the PackGQA row
<-> (head, query) mapping): when g = Hq / Hkv is 2, 4, 8 or 16, the g query
heads of a kv head share every 128-row tile (128 / g queries of each), so
each K/V tile in shared memory serves the whole group.

Checked against the fp64 oracle for every packing factor on the dense,
group-mode and paged (chunked prefill) entry points, with ragged query
counts, masks, sinks, soft-cap and ALiBi (per-head slopes and sinks are
where a wrong row -> head mapping would show); and bit for bit against the
same heads run one at a time without packing (Hq = Hkv = 1): a row's
arithmetic does not depend on which rows share its tile."""
import math

import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import inputs
from tests._parity import check, cuda, f64, no_device_error

pytestmark = pytest.mark.gpu

DENSE = [
    # B, Hq, Hkv, Lq, Lk, d, dtype, causal, softcap, sink, window, alibi
    (2, 4, 2, 300, 300, 128, "bf16", True, 0.0, True, None, False),        # g = 2
    (1, 32, 8, 200, 777, 128, "bf16", True, 0.0, False, None, True),       # g = 4, Lq < Lk, ALiBi
    (1, 16, 2, 77, 77, 64, "f16", False, 30.0, True, None, False),         # g = 8, soft-cap
    (2, 16, 1, 45, 300, 128, "bf16", True, 0.0, True, (64, 0), False),     # g = 16 (MQA), window
    (1, 8, 2, 1, 513, 128, "bf16", True, 0.0, False, None, False),         # one query row
    (1, 12, 4, 130, 130, 64, "bf16", True, 0.0, True, None, False),        # g = 3: not packed
]


def _slopes(Hq):
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=torch.float32)


@pytest.mark.parametrize("case", DENSE, ids=[str(i) for i in range(len(DENSE))])
def test_pack_dense_parity(case):
    B, Hq, Hkv, Lq, Lk, d, dt, causal, cap, sink, win, alibi = case
    inp = inputs.dense(B, Hq, Hkv, Lq, Lk, d, dt, seed=Hq * 100 + Lq, causal=causal,
                       softcap=cap, with_sink=sink)
    sl = _slopes(Hq) if alibi else None
    o, lse = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), causal=causal, softcap=cap,
                        sink=cuda(inp.sink), window=win, alibi_slopes=cuda(sl))
    torch.cuda.synchronize()
    ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), 1 / math.sqrt(d), causal, cap,
                               None if inp.sink is None else f64(inp.sink),
                               window=win if win else (-1, -1),
                               alibi=None if sl is None else sl.numpy())
    check(o, lse, ro, rl, f"packed dense {case}")
    no_device_error()


@pytest.mark.parametrize("g", [2, 4, 8, 16])
def test_pack_varlen_parity(g):
    lens = [1, 0, 37, 300, 129]
    Hkv = 2
    inp = inputs.varlen(lens, lens, Hkv * g, Hkv, 128, "bf16", seed=g, causal=True,
                        with_sink=True)
    o, lse = A.attn_fwd_varlen(cuda(inp.q), cuda(inp.k), cuda(inp.v), cuda(inp.cu_seqlens_q),
                               cuda(inp.cu_seqlens_k), inp.max_seqlen_q, causal=True,
                               sink=cuda(inp.sink))
    torch.cuda.synchronize()
    ro, rl = oracle.attn_varlen(f64(inp.q), f64(inp.k), f64(inp.v), inp.cu_seqlens_q.numpy(),
                                inp.cu_seqlens_k.numpy(), 1 / math.sqrt(128), True, 0.0,
                                f64(inp.sink))
    check(o, lse, ro, rl, f"packed varlen g={g}")
    no_device_error()


@pytest.mark.parametrize("Lq,g", [(8, 4), (24, 8), (100, 4), (5, 16)])
def test_pack_chunked_prefill_parity(Lq, g):
    """Short chunks over a paged cache (Lq * g > 16 goes to the prefill
    kernel): the packed tile holds all g heads of the chunk's rows."""
    lens, Hkv, d, page = [400, 64, 1000], 2, 128, 32
    npages = sum((L + page - 1) // page for L in lens) + 3
    inp = inputs.paged(lens, Lq, Hkv * g, Hkv, d, page, npages, seed=Lq * g, causal=True,
                       with_sink=True)
    o, lse = A.attn_fwd_paged(cuda(inp.q), cuda(inp.k_pool), cuda(inp.v_pool),
                              cuda(inp.block_table), cuda(inp.seqlens_k), causal=True,
                              sink=cuda(inp.sink))
    torch.cuda.synchronize()
    assert A.attn_last_kernel_name().startswith("attn_prefill_tcgen05")
    ro, rl = oracle.attn_paged(f64(inp.q), f64(inp.k_pool), f64(inp.v_pool),
                               inp.block_table.numpy(), inp.seqlens_k.numpy(), 1 / math.sqrt(d),
                               True, 0.0, f64(inp.sink))
    check(o, lse, ro, rl, f"packed chunked prefill Lq={Lq} g={g}")
    no_device_error()


@pytest.mark.parametrize("Hq,Hkv,L", [(32, 8, 1024), (16, 1, 700), (8, 4, 333)])
def test_pack_equals_unpacked_heads(Hq, Hkv, L):
    """Packed GQA result, head by head, equals the same head run alone as
    one-head attention (no packing), bit for bit."""
    inp = inputs.dense(1, Hq, Hkv, L, L, 128, "bf16", seed=L, device="cuda", causal=True)
    o, lse = A.attn_fwd(inp.q, inp.k, inp.v, causal=True)
    torch.cuda.synchronize()
    g = Hq // Hkv
    for h in sorted({0, g - 1, Hq // 2, Hq - 1}):
        hk = h // g
        o1, l1 = A.attn_fwd(inp.q[:, h:h + 1].contiguous(), inp.k[:, hk:hk + 1].contiguous(),
                            inp.v[:, hk:hk + 1].contiguous(), causal=True)
        torch.cuda.synchronize()
        assert torch.equal(o1, o[:, h:h + 1]), f"head {h}"
        assert torch.equal(l1, lse[:, h:h + 1]), f"head {h} LSE"
    no_device_error()
