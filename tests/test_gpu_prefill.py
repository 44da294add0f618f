"""GPU parity of the dense and varlen (group-mode) prefill kernel against the
fp64 oracle, element by element, on seeded inputs (the full-size workloads
are compared whole in test_gpu_full_size.py)."""
import math

import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import inputs
from tests._parity import check, cuda, dense_case, f64, no_device_error

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


@pytest.mark.parametrize("d", [64, 128])
def test_softcap_logits_far_past_the_cap(d):
    """Soft-cap 30 with rows 200-259 scaled so their logits run far past the
    cap (Q x 40: tanh saturates, the kernel's r = 1 / (2^(2y log2 e) + 1)
    reaches 0 and 1) next to rows with small logits, in one launch; every
    row must match the oracle."""
    inp = inputs.dense(1, 4, 2, 700, 700, d, "bf16", seed=70 + d, causal=True, softcap=30.0,
                       with_sink=True)
    q = inp.q.clone()
    q[:, :, 200:260] = (q[:, :, 200:260].float() * 40.0).to(q.dtype)
    o, lse = A.attn_fwd(cuda(q), cuda(inp.k), cuda(inp.v), causal=True, softcap=30.0,
                        sink=cuda(inp.sink))
    torch.cuda.synchronize()
    ro, rl = oracle.attn_dense(f64(q), f64(inp.k), f64(inp.v), 1 / math.sqrt(d), True, 30.0,
                               f64(inp.sink))
    check(o, lse, ro, rl, f"soft-cap far past the cap d={d}")
    no_device_error()
