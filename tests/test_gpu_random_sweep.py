"""A seeded random sweep of the three entry points against the fp64 oracle.

Each case draws its shape and options at random within what the entry point
accepts: batch, query and kv heads (GQA group 1-16, so every PackGQA factor
and both epilogue store paths are drawn), lengths (0 to a few
hundred, ragged, Lq != Lk), head dimension 64/128, fp16/bf16, causal, sliding
window in either alignment, soft-cap, sink and ALiBi (the score transforms
exclusive of one another), page size and split count for the paged cache.
The draws are fixed by the seed, so a failure names a reproducible case.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_13_gb300 as A
from attention_forward_13_gb300 import inputs
from tests._parity import check, cuda, f64, no_device_error

pytestmark = pytest.mark.gpu

SEED = 20261203


def _options(rng):
    causal = bool(rng.integers(2))
    win = None
    if rng.random() < 0.4:
        win = (int(rng.choice([-1, 0, int(rng.integers(1, 300))])),
               int(rng.choice([-1, 0, int(rng.integers(1, 300))])))
        if win == (-1, -1):
            win = None
    top_left = bool(rng.integers(2)) if (causal or win is not None) else False
    xf = ["none", "softcap", "alibi"][int(rng.integers(3))]
    sink = bool(rng.integers(2))
    return causal, win, top_left, xf, sink


def _slopes(rng, B, Hq):
    base = np.array([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)])
    if rng.random() < 0.5:
        return torch.tensor(base, dtype=torch.float32)
    return torch.tensor(base[None, :] * (0.5 + rng.random((B, Hq))), dtype=torch.float32)


def _dense_cases(n):
    rng = np.random.default_rng(SEED)
    out = []
    for _ in range(n):
        B = int(rng.integers(1, 3))
        Hkv = int(rng.choice([1, 2, 4]))
        g = int(rng.choice([1, 2, 4, 8, 16]))
        Lq = int(rng.integers(1, 513))
        Lk = Lq if rng.random() < 0.5 else int(rng.integers(1, 513))
        d = int(rng.choice([64, 128]))
        dt = str(rng.choice(["bf16", "f16"]))
        out.append((B, Hkv * g, Hkv, Lq, Lk, d, dt) + _options(rng) + (int(rng.integers(1 << 30)),))
    return out


def _varlen_cases(n):
    rng = np.random.default_rng(SEED + 1)
    out = []
    for _ in range(n):
        B = int(rng.integers(1, 7))
        lq = [int(x) for x in rng.integers(0, 400, B)]
        lk = lq if rng.random() < 0.5 else [int(x) for x in rng.integers(0, 400, B)]
        Hkv = int(rng.choice([1, 2]))
        g = int(rng.choice([1, 2, 4, 8, 16]))
        d = int(rng.choice([64, 128]))
        dt = str(rng.choice(["bf16", "f16"]))
        out.append((lq, lk, Hkv * g, Hkv, d, dt) + _options(rng) + (int(rng.integers(1 << 30)),))
    return out


def _paged_cases(n):
    rng = np.random.default_rng(SEED + 2)
    out = []
    for _ in range(n):
        B = int(rng.integers(1, 5))
        lens = [int(x) for x in rng.integers(0, 900, B)]
        Lq = int(rng.choice([1, 2, 4, 64, 200]))
        Hkv = int(rng.choice([1, 2]))
        g = int(rng.choice([1, 4, 8]))
        d = int(rng.choice([64, 128]))
        page = int(rng.choice([16, 32, 64, 128]))
        splits = int(rng.choice([0, 1, 3]))
        out.append((lens, Lq, Hkv * g, Hkv, d, page, splits) + _options(rng) +
                   (int(rng.integers(1 << 30)),))
    return out


DENSE = _dense_cases(16)
VARLEN = _varlen_cases(10)
PAGED = _paged_cases(10)


@pytest.mark.parametrize("case", DENSE, ids=[f"dense{i}" for i in range(len(DENSE))])
def test_random_dense(case):
    B, Hq, Hkv, Lq, Lk, d, dt, causal, win, tl, xf, sink, seed = case
    cap = 30.0 if xf == "softcap" else 0.0
    inp = inputs.dense(B, Hq, Hkv, Lq, Lk, d, dt, seed=seed, value_scale=2.0 if cap else 1.0,
                       causal=causal, softcap=cap, with_sink=sink)
    sl = _slopes(np.random.default_rng(seed), B, Hq) if xf == "alibi" else None
    o, lse = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), causal=causal, softcap=cap,
                        sink=cuda(inp.sink), window=win, top_left=tl, alibi_slopes=cuda(sl))
    torch.cuda.synchronize()
    ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), 1 / math.sqrt(d), causal, cap,
                               None if inp.sink is None else f64(inp.sink),
                               window=win if win else (-1, -1), top_left=tl,
                               alibi=None if sl is None else sl.numpy())
    check(o, lse, ro, rl, f"dense {case}")
    no_device_error()


@pytest.mark.parametrize("case", VARLEN, ids=[f"varlen{i}" for i in range(len(VARLEN))])
def test_random_varlen(case):
    lq, lk, Hq, Hkv, d, dt, causal, win, tl, xf, sink, seed = case
    cap = 30.0 if xf == "softcap" else 0.0
    inp = inputs.varlen(lq, lk, Hq, Hkv, d, dt, seed=seed, value_scale=2.0 if cap else 1.0,
                        causal=causal, softcap=cap, with_sink=sink)
    sl = _slopes(np.random.default_rng(seed), len(lq), Hq) if xf == "alibi" else None
    o, lse = A.attn_fwd_varlen(cuda(inp.q), cuda(inp.k), cuda(inp.v), cuda(inp.cu_seqlens_q),
                               cuda(inp.cu_seqlens_k), inp.max_seqlen_q, causal=causal,
                               softcap=cap, sink=cuda(inp.sink), window=win, top_left=tl,
                               alibi_slopes=cuda(sl))
    torch.cuda.synchronize()
    ro, rl = oracle.attn_varlen(f64(inp.q), f64(inp.k), f64(inp.v), inp.cu_seqlens_q.numpy(),
                                inp.cu_seqlens_k.numpy(), 1 / math.sqrt(d), causal, cap,
                                None if inp.sink is None else f64(inp.sink),
                                window=win if win else (-1, -1), top_left=tl,
                                alibi=None if sl is None else sl.numpy())
    check(o, lse, ro, rl, f"varlen {case}")
    no_device_error()


@pytest.mark.parametrize("case", PAGED, ids=[f"paged{i}" for i in range(len(PAGED))])
def test_random_paged(case):
    lens, Lq, Hq, Hkv, d, page, splits, causal, win, tl, xf, sink, seed = case
    cap = 30.0 if xf == "softcap" else 0.0
    npages = sum((L + page - 1) // page for L in lens) + 3
    inp = inputs.paged(lens, Lq, Hq, Hkv, d, page, npages, seed=seed,
                       value_scale=2.0 if cap else 1.0, causal=causal, softcap=cap,
                       with_sink=sink)
    sl = _slopes(np.random.default_rng(seed), len(lens), Hq) if xf == "alibi" else None
    o, lse = A.attn_fwd_paged(cuda(inp.q), cuda(inp.k_pool), cuda(inp.v_pool),
                              cuda(inp.block_table), cuda(inp.seqlens_k), num_splits=splits,
                              causal=causal, softcap=cap, sink=cuda(inp.sink), window=win,
                              top_left=tl, alibi_slopes=cuda(sl))
    torch.cuda.synchronize()
    ro, rl = oracle.attn_paged(f64(inp.q), f64(inp.k_pool), f64(inp.v_pool),
                               inp.block_table.numpy(), inp.seqlens_k.numpy(), 1 / math.sqrt(d),
                               causal, cap, None if inp.sink is None else f64(inp.sink),
                               window=win if win else (-1, -1), top_left=tl,
                               alibi=None if sl is None else sl.numpy())
    check(o, lse, ro, rl, f"paged {case}")
    no_device_error()


def _fp8_cases(n):
    rng = np.random.default_rng(SEED + 3)
    out = []
    for _ in range(n):
        varlen = bool(rng.integers(2))
        Hkv = int(rng.choice([1, 2]))
        g = int(rng.choice([1, 2, 4]))
        causal = bool(rng.integers(2))
        win = None
        if rng.random() < 0.3:
            win = (int(rng.integers(0, 300)), int(rng.choice([-1, 0])))
        sp = float(rng.choice([1.0, 448.0]))
        so = float(rng.choice([1.0, 2.0])) / sp
        if varlen:
            B = int(rng.integers(1, 5))
            shape = ([int(x) for x in rng.integers(0, 400, B)],)
        else:
            Lq = int(rng.integers(1, 513))
            shape = (int(rng.integers(1, 3)), Lq, Lq if rng.random() < 0.5 else int(rng.integers(1, 513)))
        out.append((varlen, shape, Hkv * g, Hkv, causal, win, sp, so, int(rng.integers(1 << 30))))
    return out


FP8 = _fp8_cases(8)


@pytest.mark.parametrize("case", FP8, ids=[f"fp8_{i}" for i in range(len(FP8))])
def test_random_fp8(case):
    """FP8 e4m3 static quantisation (d = 128), dense or group mode: O within
    one e4m3 step of the rounded oracle (scale_p * scale_o applied)."""
    from tests._parity import check_e4m3
    varlen, shape, Hq, Hkv, causal, win, sp, so, seed = case
    if varlen:
        (lens,) = shape
        inp = inputs.varlen(lens, lens, Hq, Hkv, 128, "e4m3", seed=seed, causal=causal)
        o, lse = A.attn_fwd_varlen(cuda(inp.q), cuda(inp.k), cuda(inp.v), cuda(inp.cu_seqlens_q),
                                   cuda(inp.cu_seqlens_k), inp.max_seqlen_q, causal=causal,
                                   window=win, scale_p=sp, scale_o=so)
        torch.cuda.synchronize()
        ro, rl = oracle.attn_varlen(f64(inp.q), f64(inp.k), f64(inp.v), inp.cu_seqlens_q.numpy(),
                                    inp.cu_seqlens_k.numpy(), 1 / math.sqrt(128), causal,
                                    window=win if win else (-1, -1), o_scale=sp * so)
    else:
        B, Lq, Lk = shape
        inp = inputs.dense(B, Hq, Hkv, Lq, Lk, 128, "e4m3", seed=seed, causal=causal)
        o, lse = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), causal=causal, window=win,
                            scale_p=sp, scale_o=so)
        torch.cuda.synchronize()
        ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), 1 / math.sqrt(128), causal,
                                   window=win if win else (-1, -1), o_scale=sp * so)
    check_e4m3(o, lse, ro, rl, f"fp8 {case}", o_scale=sp * so,
               vmax=float(np.abs(f64(inp.v)).max()) if f64(inp.v).size else 0.0)
    no_device_error()
