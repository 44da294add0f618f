"""Whole-output parity of the four full-size workloads against the fp64
oracle: every element of O and of LSE, on the same seeded inputs, in the
launch configuration the benchmark times (default scale, automatic split
count for decode).

* dense causal prefill B4 H16 L2048 d128 bf16;
* GQA causal prefill B2 Hq32 Hkv8 L8192 d128 bf16 (4 query heads per kv head);
* paged-KV decode B64 Hq32 Hkv8 d128, page 64, L_b ~ U[512, 8192] over a
  10240-page pool (the oracle runs on 8 sequences at a time, each chunk with
  only its own pages, to bound host memory);
* varlen causal prefill, 16 sequences L_b ~ U[128, 4096], H16 d64, values x2,
  soft-cap 30 and one sink logit per head.

Bounds (tests/_parity.py): |O_gpu - O_exact| <= 2e-2 + 1/2 ulp(O_exact),
mean |O_gpu - O_exact| <= 2e-3, |LSE_gpu - LSE_exact| <= 1e-3.  Each test
prints one line with its maximum and mean error and the number of elements
above 2e-2 (run with -s to see them)."""
import math

import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import inputs
from tests._parity import check, compact_paged, f64, merge_stats, no_device_error, report

pytestmark = pytest.mark.gpu


def _dense_full(n, name):
    inp = inputs.workload(n, device="cuda")
    d = inp.q.shape[-1]
    o, lse = A.attn_fwd(inp.q, inp.k, inp.v, causal=True)
    torch.cuda.synchronize()
    no_device_error()
    og, lg = f64(o), f64(lse)
    q, k, v = f64(inp.q), f64(inp.k), f64(inp.v)
    del inp, o, lse
    ro, rl = oracle.attn_dense(q, k, v, 1 / math.sqrt(d), True)
    st = {}
    check(og, lg, ro, rl, name, stats=st)
    report(name, st)


def test_workload2_full():
    """Dense causal prefill B4 H16 L2048 d128 bf16, every element."""
    _dense_full(2, "workload 2 dense causal B4 H16 L2048 d128")


def test_workload3_full():
    """GQA causal prefill B2 Hq32 Hkv8 L8192 d128 bf16, every element."""
    _dense_full(3, "workload 3 GQA causal B2 Hq32 Hkv8 L8192 d128")


def test_workload4_full():
    """Paged decode B64 Hq32 Hkv8 d128 page 64 (auto splits + combine), all 64
    sequences."""
    inp = inputs.workload(4, device="cuda")
    o, lse = A.attn_fwd_paged(inp.q, inp.k_pool, inp.v_pool, inp.block_table.cuda(),
                              inp.seqlens_k.cuda())
    torch.cuda.synchronize()
    no_device_error()
    og, lg = f64(o), f64(lse)
    total = {}
    B = inp.q.shape[0]
    for c0 in range(0, B, 8):
        bsel = list(range(c0, min(B, c0 + 8)))
        kp, vp, nbt, sl = compact_paged(inp, bsel)
        ro, rl = oracle.attn_paged(f64(inp.q[bsel]), kp, vp, nbt, sl, 1 / math.sqrt(128))
        st = {}
        check(og[bsel], lg[bsel], ro, rl, f"workload 4 sequences {bsel[0]}..{bsel[-1]}", stats=st)
        merge_stats(total, st)
    report("workload 4 paged decode B64 Hq32 Hkv8 d128 page 64", total)


def test_workload5_full():
    """Varlen causal prefill, soft-cap 30 and sinks, 16 sequences, every element."""
    inp = inputs.workload(5, device="cuda")
    o, lse = A.attn_fwd_varlen(inp.q, inp.k, inp.v, inp.cu_seqlens_q.cuda(),
                               inp.cu_seqlens_k.cuda(), inp.max_seqlen_q, causal=True,
                               softcap=30.0, sink=inp.sink)
    torch.cuda.synchronize()
    no_device_error()
    ro, rl = oracle.attn_varlen(f64(inp.q), f64(inp.k), f64(inp.v), inp.cu_seqlens_q.numpy(),
                                inp.cu_seqlens_k.numpy(), 1 / math.sqrt(64), True, 30.0,
                                f64(inp.sink))
    st = {}
    check(o, lse, ro, rl, "workload 5", stats=st)
    report("workload 5 varlen causal soft-cap 30 + sink, 16 seqs H16 d64", st)
