"""Masked keys that carry huge scores must not change any output row.

The prefill kernel takes a tile's row maximum from the tensor-memory load
itself where no key of the tile is masked, and from the kept keys only where
some are (the causal / window band, the tail past Lk).  These cases plant keys
whose scores run ~30x past the others exactly where the mask drops them for
some rows and keeps them for others: a maximum taken over masked keys would
push every kept weight of those rows below the fp32 range and leave O = 0 / 0.
Each case is compared element by element with the fp64 oracle, which applies
the mask by definition."""
import math

import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import inputs
from tests._parity import check, cuda, f64, no_device_error

pytestmark = pytest.mark.gpu


def _plant(k, rows, factor=30.0):
    """K rows `rows` (a slice of the key axis, dim -2) scaled by `factor`."""
    k = k.clone()
    k[..., rows, :] = (k[..., rows, :].float() * factor).to(k.dtype)
    return k


@pytest.mark.parametrize("d,dt", [(128, "bf16"), (64, "bf16"), (128, "f16")])
def test_causal_future_keys_with_huge_scores(d, dt):
    """Keys 401-639 scaled x30: rows 0-400 mask all of them (several of those
    rows share tiles with rows that keep them), rows past 400 keep some."""
    inp = inputs.dense(1, 4, 2, 640, 640, d, dt, seed=900 + d, causal=True)
    k = _plant(inp.k, slice(401, 640))
    o, lse = A.attn_fwd(cuda(inp.q), cuda(k), cuda(inp.v), causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_dense(f64(inp.q), f64(k), f64(inp.v), 1 / math.sqrt(d), True)
    check(o, lse, ro, rl, f"causal, masked future keys x30, d={d} {dt}")
    no_device_error()


def test_window_left_keys_with_huge_scores():
    """Causal window of 200 keys to the left: keys 0-99 scaled x30 are kept by
    rows 0-299 and dropped by every later row (the band's left edge crosses
    the tiles that hold them)."""
    inp = inputs.dense(1, 2, 2, 800, 800, 128, "bf16", seed=911, causal=True)
    k = _plant(inp.k, slice(0, 100))
    o, lse = A.attn_fwd(cuda(inp.q), cuda(k), cuda(inp.v), causal=True, window=(200, -1))
    torch.cuda.synchronize()
    ro, rl = oracle.attn_dense(f64(inp.q), f64(k), f64(inp.v), 1 / math.sqrt(128), True,
                               window=(200, -1))
    check(o, lse, ro, rl, "window (200, causal), masked left keys x30")
    no_device_error()


def test_varlen_future_keys_with_huge_scores():
    """Group mode: in each sequence the last third of the keys is scaled x30,
    so the causal band masks them for the earlier rows of the same tiles."""
    lens = [300, 517, 130]
    inp = inputs.varlen(lens, lens, 4, 4, 128, "bf16", seed=921, causal=True)
    k = inp.k.clone()
    cu = inp.cu_seqlens_k.tolist()
    for b, L in enumerate(lens):
        s0 = cu[b] + (2 * L) // 3
        k[s0:cu[b + 1]] = (k[s0:cu[b + 1]].float() * 30.0).to(k.dtype)
    o, lse = A.attn_fwd_varlen(cuda(inp.q), cuda(k), cuda(inp.v), cuda(inp.cu_seqlens_q),
                               cuda(inp.cu_seqlens_k), inp.max_seqlen_q, causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_varlen(f64(inp.q), f64(k), f64(inp.v), inp.cu_seqlens_q.numpy(),
                                inp.cu_seqlens_k.numpy(), 1 / math.sqrt(128), True)
    check(o, lse, ro, rl, "varlen causal, masked future keys x30")
    no_device_error()
