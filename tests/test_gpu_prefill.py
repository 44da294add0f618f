"""GPU parity of the dense and varlen (group-mode) prefill kernel against the
fp64 oracle, element by element, on seeded inputs; plus sampled rows of the
full-size dense workloads."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import inputs
from tests._parity import check, cuda, dense_case, dense_rows_reference, f64, no_device_error

pytestmark = pytest.mark.gpu

DENSE_CASES = [
    # B, Hq, Hkv, Lq, Lk, d, dtype, causal, softcap, sink, value_scale
    (1, 2, 2, 128, 128, 64, "f16", False, 0.0, False, 1.0),      # workload 1 shape
    (2, 4, 4, 300, 300, 128, "bf16", True, 0.0, False, 1.0),     # ragged tail, 2 query blocks
    (1, 2, 2, 100, 700, 64, "f16", False, 0.0, False, 1.0),      # Lq < Lk, ragged keys
    (1, 2, 2, 400, 150, 128, "bf16", True, 0.0, False, 1.0),     # Lq > Lk: empty rows
    (1, 2, 1, 130, 1000, 128, "bf16", True, 0.0, False, 1.0),    # Lq < Lk causal, MQA
    (1, 8, 2, 513, 513, 128, "bf16", True, 0.0, False, 1.0),     # GQA g = 4
    (1, 4, 4, 257, 257, 64, "bf16", True, 30.0, True, 2.0),      # softcap + sink
    (2, 2, 2, 190, 77, 128, "f16", False, 0.0, True, 1.0),       # sink only
    (1, 2, 2, 1, 77, 128, "bf16", False, 0.0, False, 1.0),       # single query
    (1, 2, 2, 1, 1, 64, "bf16", True, 0.0, False, 1.0),          # single token
    (1, 2, 2, 1024, 1024, 128, "bf16", True, 0.0, False, 1.0),   # full tiles, 4 blocks
    (1, 2, 2, 640, 640, 64, "f16", True, 5.0, False, 3.0),       # fp16 softcap
]


@pytest.mark.parametrize("case", DENSE_CASES, ids=[str(i) for i in range(len(DENSE_CASES))])
def test_dense_parity(case):
    B, Hq, Hkv, Lq, Lk, d, dt, causal, cap, sink, vs = case
    inp = inputs.dense(B, Hq, Hkv, Lq, Lk, d, dt, seed=7 + Lq + Lk, value_scale=vs,
                       causal=causal, softcap=cap, with_sink=sink)
    dense_case(inp)
    no_device_error()


def test_workload1_tiny_full():
    inp = inputs.workload(1)
    dense_case(inp)
    no_device_error()


def test_default_scale_and_lse_optional():
    inp = inputs.dense(1, 2, 2, 200, 200, 128, "bf16", seed=3, causal=True)
    o1, l1 = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), causal=True)  # scale <= 0 -> 1/sqrt(d)
    o2, l2 = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), causal=True, lse=False)
    torch.cuda.synchronize()
    assert l2 is None
    ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), 1 / math.sqrt(128), True)
    check(o1, l1, ro, rl, "default scale")
    assert torch.equal(o1, o2)
    no_device_error()


def test_lk_zero_gives_empty_rows():
    inp = inputs.dense(1, 2, 2, 50, 0, 64, "bf16", seed=4, with_sink=True)
    o, l = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v))
    o2, l2 = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), sink=cuda(inp.sink))
    torch.cuda.synchronize()
    assert torch.count_nonzero(o) == 0 and torch.all(torch.isneginf(l))
    assert torch.count_nonzero(o2) == 0
    assert torch.allclose(l2.cpu(), inp.sink.view(1, 2, 1).expand(1, 2, 50))
    no_device_error()


def test_strided_bshd_layout():
    """Q/K/V/O as [B,L,H,d] memory viewed as [B,H,L,d] (row stride H*d)."""
    B, L, H, d = 2, 333, 4, 128
    base = inputs.dense(B, H, H, L, L, d, "bf16", seed=11, causal=True)
    qs = base.q.transpose(1, 2).contiguous().cuda()  # [B,L,H,d] storage
    ks = base.k.transpose(1, 2).contiguous().cuda()
    vs = base.v.transpose(1, 2).contiguous().cuda()
    q, k, v = qs.transpose(1, 2), ks.transpose(1, 2), vs.transpose(1, 2)
    o_store = torch.empty((B, L, H, d), dtype=torch.bfloat16, device="cuda")
    o, lse = A.attn_fwd(q, k, v, o=o_store.transpose(1, 2), causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_dense(f64(base.q), f64(base.k), f64(base.v), 1 / math.sqrt(d), True)
    check(o, lse, ro, rl, "BSHD strides")
    no_device_error()


VARLEN_CASES = [
    # lens_q, lens_k, Hq, Hkv, d, dtype, causal, softcap, sink, value_scale
    ([1, 0, 130, 257, 500], None, 4, 2, 128, "bf16", True, 30.0, True, 2.0),
    ([5, 100, 64], [300, 100, 1], 2, 2, 64, "f16", True, 0.0, False, 1.0),
    ([77, 256, 300], None, 4, 4, 64, "bf16", False, 0.0, True, 1.0),
    ([513, 1, 129], [513, 1000, 0], 8, 2, 128, "bf16", False, 0.0, False, 1.0),
]


@pytest.mark.parametrize("case", VARLEN_CASES, ids=[str(i) for i in range(len(VARLEN_CASES))])
def test_varlen_parity(case):
    lq, lk, Hq, Hkv, d, dt, causal, cap, sink, vs = case
    lk = lk if lk is not None else lq
    inp = inputs.varlen(lq, lk, Hq, Hkv, d, dt, seed=sum(lq) + 5, value_scale=vs, causal=causal,
                        softcap=cap, with_sink=sink)
    o, lse = A.attn_fwd_varlen(cuda(inp.q), cuda(inp.k), cuda(inp.v), cuda(inp.cu_seqlens_q),
                               cuda(inp.cu_seqlens_k), inp.max_seqlen_q, causal=causal,
                               softcap=cap, sink=cuda(inp.sink))
    torch.cuda.synchronize()
    ro, rl = oracle.attn_varlen(f64(inp.q), f64(inp.k), f64(inp.v), inp.cu_seqlens_q.numpy(),
                                inp.cu_seqlens_k.numpy(), 1 / math.sqrt(d), causal, cap,
                                None if inp.sink is None else f64(inp.sink))
    check(o, lse, ro, rl, "varlen")
    no_device_error()


def _sampled_dense(inp, picks, g):
    d = inp.q.shape[-1]
    sc = 1 / math.sqrt(d)
    o, lse = A.attn_fwd(inp.q, inp.k, inp.v, causal=inp.causal)
    torch.cuda.synchronize()
    worst = 0.0
    for b, h, r0, r1 in picks:
        ro, rl = dense_rows_reference(inp.q, inp.k, inp.v, b, h, (r0, r1), g, inp.causal, sc)
        worst = max(worst, check(o[b:b + 1, h:h + 1, r0:r1], lse[b:b + 1, h:h + 1, r0:r1], ro,
                                 rl, f"rows b{b} h{h} {r0}:{r1}"))
    no_device_error()
    return worst


def test_workload2_full_size_sampled():
    """Dense causal prefill B4 H16 L2048 d128 at full size, sampled rows."""
    inp = inputs.workload(2, device="cuda")
    picks = [(0, 0, 0, 64), (1, 7, 1000, 1064), (3, 15, 1984, 2048), (2, 3, 255, 257)]
    _sampled_dense(inp, picks, 1)


def test_workload3_full_size_sampled():
    """GQA causal prefill B2 Hq32 Hkv8 L8192 d128 at full size, sampled rows."""
    inp = inputs.workload(3, device="cuda")
    picks = [(0, 0, 0, 32), (0, 5, 4095, 4127), (1, 31, 8160, 8192), (1, 12, 8000, 8032)]
    _sampled_dense(inp, picks, 4)


def test_workload5_full_size_sampled():
    """Varlen causal prefill with softcap 30 and sinks: 16 sequences in
    [128, 4096], sampled sequences compared in full."""
    inp = inputs.workload(5, device="cuda")
    cu = inp.cu_seqlens_q
    o, lse = A.attn_fwd_varlen(inp.q, inp.k, inp.v, cu.cuda(), inp.cu_seqlens_k.cuda(),
                               inp.max_seqlen_q, causal=True, softcap=30.0, sink=inp.sink)
    torch.cuda.synchronize()
    lens = (cu[1:] - cu[:-1]).tolist()
    order = np.argsort(lens)
    for bsel in (int(order[0]), int(order[len(order) // 2]), int(order[-1])):
        s0, s1 = int(cu[bsel]), int(cu[bsel + 1])
        # the sequence alone, rows [max(0, L-192), L): the last rows see every key
        r0 = max(0, (s1 - s0) - 192)
        q = f64(inp.q[s0 + r0:s1])
        k = f64(inp.k[s0:s1])
        v = f64(inp.v[s0:s1])
        cq = np.array([0, s1 - s0 - r0], dtype=np.int32)
        # the cut keeps bottom-right alignment: Lk - Lq' = r0
        ro, rl = oracle.attn_varlen(q, k, v, cq, np.array([0, s1 - s0], dtype=np.int32),
                                    1 / math.sqrt(64), True, 30.0, f64(inp.sink))
        check(o[s0 + r0:s1], lse[:, s0 + r0:s1], ro, rl, f"seq {bsel}")
    no_device_error()
