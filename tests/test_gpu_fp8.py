"""GPU parity of the FP8 (e4m3) static-quantisation path against the fp64
oracle: e4m3 Q, K, V (d = 128), S = Q K^T on the kind::f8f6f4 tensor path,
V widened to fp16 on chip, O = saturate_e4m3(scale_o * scale_p * softmax(S) V).

Composable Kernel FMHA forward: FmhaFwdFp8StaticQuantKargs (scale_p,
scale_o) and the pipeline's P / O element functions.  The oracle takes the
e4m3 input values exactly and returns O * scale_p * scale_o in fp64; the test
rounds it to e4m3 as the kernel's epilogue does."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import inputs
from tests._parity import check_e4m3, cuda, f64, no_device_error

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, Lq, Lk, causal, window, sink, scale_p, scale_o
    (1, 2, 2, 300, 300, True, None, False, 448.0, 2.0 / 448.0),
    (2, 4, 2, 257, 700, False, None, True, 1.0, 1.0),
    (1, 8, 2, 513, 513, True, None, False, 448.0, 4.0 / 448.0),
    (1, 2, 2, 640, 900, False, (128, 64), False, 1.0, 1.5),
    (1, 2, 1, 100, 40, True, None, False, 1.0, 1.0),     # Lq > Lk: keyless rows
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_fp8_dense_parity(case):
    B, Hq, Hkv, Lq, Lk, causal, win, sink, sp, so = case
    inp = inputs.dense(B, Hq, Hkv, Lq, Lk, 128, "e4m3", seed=91 + Lq + Lk, causal=causal,
                       with_sink=sink)
    assert inp.q.dtype == torch.float8_e4m3fn
    o, lse = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), causal=causal, window=win,
                        sink=cuda(inp.sink), scale_p=sp, scale_o=so)
    torch.cuda.synchronize()
    assert o.dtype == torch.float8_e4m3fn
    assert "_e4m3_" in A.attn_last_kernel_name()
    ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), 1 / math.sqrt(128), causal,
                               sink=None if inp.sink is None else f64(inp.sink),
                               window=win if win else (-1, -1), o_scale=sp * so)
    check_e4m3(o, lse, ro, rl, f"fp8 dense {case}", o_scale=sp * so,
               vmax=float(np.abs(f64(inp.v)).max()))
    no_device_error()


def test_fp8_varlen_parity():
    lq, lk = [5, 300, 129, 1], [700, 100, 129, 40]
    inp = inputs.varlen(lq, lk, 4, 2, 128, "e4m3", seed=23, causal=True)
    o, lse = A.attn_fwd_varlen(cuda(inp.q), cuda(inp.k), cuda(inp.v), cuda(inp.cu_seqlens_q),
                               cuda(inp.cu_seqlens_k), inp.max_seqlen_q, causal=True,
                               scale_p=448.0, scale_o=1.0 / 448.0)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_varlen(f64(inp.q), f64(inp.k), f64(inp.v), inp.cu_seqlens_q.numpy(),
                                inp.cu_seqlens_k.numpy(), 1 / math.sqrt(128), True, o_scale=1.0)
    check_e4m3(o, lse, ro, rl, "fp8 varlen", vmax=float(np.abs(f64(inp.v)).max()))
    no_device_error()


def test_fp8_saturates_large_outputs():
    """scale_o large enough to push |O| past 448: the output saturates to
    +-448 (satfinite), never inf or NaN."""
    inp = inputs.dense(1, 2, 2, 200, 200, 128, "e4m3", seed=5)
    o, lse = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), scale_o=4000.0)
    torch.cuda.synchronize()
    of = f64(o)
    ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), 1 / math.sqrt(128),
                               o_scale=4000.0)
    assert np.all(np.isfinite(of)) and np.abs(of).max() == 448.0
    check_e4m3(o, lse, ro, rl, "fp8 saturation", o_scale=4000.0,
               vmax=float(np.abs(f64(inp.v)).max()))
    no_device_error()


def test_fp8_causal_workload_sampled():
    """The headline shape in e4m3 (B4 H16 L2048 d128, causal): sampled rows."""
    B, H, L = 4, 16, 2048
    inp = inputs.dense(B, H, H, L, L, 128, "e4m3", seed=1002, device="cuda", causal=True)
    o, lse = A.attn_fwd(inp.q, inp.k, inp.v, causal=True, scale_p=448.0, scale_o=1.0 / 448.0)
    torch.cuda.synchronize()
    rng = np.random.default_rng(8)
    for _ in range(4):
        b, h = int(rng.integers(B)), int(rng.integers(H))
        r0 = int(rng.integers(0, L - 64))
        r1 = r0 + 64
        ro, rl = oracle.attn_dense(f64(inp.q[b:b + 1, h:h + 1, r0:r1]),
                                   f64(inp.k[b:b + 1, h:h + 1, :r1]),
                                   f64(inp.v[b:b + 1, h:h + 1, :r1]), 1 / math.sqrt(128), True)
        check_e4m3(o[b:b + 1, h:h + 1, r0:r1], lse[b:b + 1, h:h + 1, r0:r1], ro, rl,
                   f"fp8 sampled b{b} h{h}", vmax=float(np.abs(f64(inp.v[b, h])).max()))
    no_device_error()
