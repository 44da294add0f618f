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


# ---------------------------------------------------------------------------
# OCP FP8 e4m3 ("fn" variant): sign, 4 exponent bits (bias 7), 3 mantissa bits,
# no infinities; largest finite 448 = 1.75 * 2^8; normals from 2^-6;
# subnormals are multiples of 2^-9.  Written from that definition.
E4M3_MAX = 448.0


def ulp_e4m3(x: np.ndarray) -> np.ndarray:
    """Spacing of e4m3 values at |x| (2^-9 in the subnormal range)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -6)))
    return np.exp2(np.maximum(e, -6.0) - 3.0)


def round_e4m3(x: np.ndarray) -> np.ndarray:
    """fp64 -> nearest e4m3 value (ties to even mantissa), saturated to +-448
    (the conversion the kernel's epilogue performs, taken here in fp64)."""
    x = np.asarray(x, dtype=np.float64)
    q = ulp_e4m3(x)
    r = np.round(np.abs(x) / q) * q  # numpy rounds half to even
    return np.sign(x) * np.minimum(r, E4M3_MAX)


def check_e4m3(o_gpu, lse_gpu, o_ref, lse_ref, what="", min_exact=0.95, o_scale=1.0, vmax=None):
    """e4m3 output.  Before its final rounding the kernel's O differs from the
    exact one by at most o_scale * 2^-11 * max|V| (P is rounded to fp16, a
    relative 2^-11, before P.V; the fp32 sums add far less); the allowance
    doubles that.  So each element must lie within one e4m3 step (at the
    larger of the two magnitudes) plus that absolute term of the oracle
    rounded to e4m3, and at least min_exact of them must be equal (only
    values near a rounding boundary may differ).  LSE as for the 16-bit types."""
    o = f64(o_gpu)
    ref = round_e4m3(o_ref)
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    err = np.abs(o - ref)
    step = ulp_e4m3(np.maximum(np.abs(ref), np.abs(o)))
    floor = 0.0 if vmax is None else o_scale * 2.0 ** -10 * vmax
    bad = err > step * 1.0000001 + floor
    assert not bad.any(), (f"{what}: O off by more than one e4m3 step + {floor} "
                           f"(max {err.max()}, {int(bad.sum())} elements)")
    exact = float(np.mean(err == 0.0)) if err.size else 1.0
    assert exact >= min_exact, f"{what}: only {exact:.3f} of O equal the rounded oracle"
    if lse_gpu is not None:
        lg = f64(lse_gpu)
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lg), inf_ref), f"{what}: -inf LSE pattern differs"
        fin = ~inf_ref
        if fin.any():
            assert np.abs(lg[fin] - lse_ref[fin]).max() <= LSE_TOL, f"{what}: LSE"
    return exact


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
