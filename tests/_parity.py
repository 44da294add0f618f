"""Helpers for the GPU-vs-oracle parity tests.

Tolerances (fp16/bf16 outputs).  The oracle's O is rounded once to the output
type (round to nearest even), as the oracle definition states; then per
element |O_gpu - O_ref| <= max(2e-2, one ulp of the output type at |O_ref|)
and the mean of |O_gpu - O_ref| <= 2e-3.  The ulp term only matters where
|O| >= 4 in bf16 (|O| >= 32 in fp16): there one ulp exceeds 2e-2, so two
correctly rounded results of fp32 values a hair apart can differ by it.
LSE: abs <= 1e-3; an LSE of -inf must match exactly.
"""
import math

import numpy as np
import torch

import oracle
import attention_forward_13_gb300 as A

O_MAX, O_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3
MANT_BITS = {torch.bfloat16: 7, torch.float16: 10, torch.float32: 23}


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def round_to(x: np.ndarray, dtype) -> np.ndarray:
    """fp64 -> dtype (RNE) -> fp64."""
    if dtype == torch.float32:
        return x.astype(np.float32).astype(np.float64)
    t = torch.from_numpy(np.ascontiguousarray(x))
    # fp64 -> fp32 is exact enough here (fp32 has 16 more bits than bf16/fp16
    # to the first rounding), then one rounding to the 16-bit type.
    return t.to(torch.float32).to(dtype).to(torch.float64).numpy()


def ulp(x: np.ndarray, dtype) -> np.ndarray:
    m = MANT_BITS[dtype]
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    return np.exp2(np.floor(np.log2(ax)) - m)


def check(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    dtype = o_gpu.dtype if isinstance(o_gpu, torch.Tensor) else torch.float32
    o = f64(o_gpu) if isinstance(o_gpu, torch.Tensor) else o_gpu
    assert o.shape == o_ref.shape, (what, o.shape, o_ref.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    ref = round_to(o_ref, dtype)
    err = np.abs(o - ref)
    bound = np.maximum(O_MAX, ulp(ref, dtype))
    if err.size:
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        assert np.all(err <= bound), (f"{what}: O err {err[i]} at |O|={abs(ref[i])} "
                                      f"(bound {bound[i]}), max err {err.max()}")
    assert (err.mean() if err.size else 0.0) <= O_MEAN, f"{what}: O mean err {err.mean()}"
    if lse_gpu is not None:
        lg = f64(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
        assert lg.shape == lse_ref.shape, (what, lg.shape, lse_ref.shape)
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lg), inf_ref), f"{what}: -inf LSE pattern differs"
        fin = ~inf_ref
        if fin.any():
            e = np.abs(lg[fin] - lse_ref[fin])
            assert e.max() <= LSE_TOL, f"{what}: LSE max err {e.max()}"
    return float(err.max(initial=0.0))


def no_device_error():
    bits = A.attn_device_error()
    assert bits == 0, f"device error word {bits:#x}"


def cuda(t):
    return None if t is None else t.to("cuda")


def dense_case(inp, scale=None):
    """Run attn_fwd on the inputs and compare every element with the oracle."""
    d = inp.q.shape[-1]
    sc = scale if scale is not None else 1.0 / math.sqrt(d)
    sink = cuda(inp.sink)
    o, lse = A.attn_fwd(cuda(inp.q), cuda(inp.k), cuda(inp.v), causal=inp.causal,
                        scale=scale, softcap=inp.softcap, sink=sink)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_dense(f64(inp.q), f64(inp.k), f64(inp.v), sc, inp.causal, inp.softcap,
                               None if inp.sink is None else f64(inp.sink))
    return check(o, lse, ro, rl, "dense")


def dense_rows_reference(q, k, v, b, h, rows, g, causal, scale, softcap=0.0, sink=None):
    """Oracle on query rows [r0, r1) of head (b, h) only.  For bottom-right
    causal masking the key range is cut to what row r1-1 can see, which keeps
    every row's mask identical to the full problem."""
    r0, r1 = rows
    Lq, Lk = q.shape[2], k.shape[2]
    hk = h // g
    kend = min(Lk, r1 + (Lk - Lq)) if causal else Lk
    kend = max(kend, 0)
    qs = f64(q[b:b + 1, h:h + 1, r0:r1])
    ks = f64(k[b:b + 1, hk:hk + 1, :kend])
    vs = f64(v[b:b + 1, hk:hk + 1, :kend])
    # With kend = r1 + Lk - Lq, row i' of the cut problem keeps
    # j <= i' + kend - (r1 - r0) = (r0 + i') + (Lk - Lq): the full problem's mask.
    sk = None if sink is None else f64(sink[h:h + 1])
    return oracle.attn_dense(qs, ks, vs, scale, causal, softcap, sk)
