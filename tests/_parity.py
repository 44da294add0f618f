"""Helpers for the GPU-vs-oracle parity tests.

Tolerances (fp16/bf16 outputs).  The GPU's O is compared with the oracle's
UNROUNDED fp64 O.  Per element
    |O_gpu - O_exact| <= 2e-2 + 1/2 ulp(O_exact)
where the half ulp (of the output type, at |O_exact|) is the rounding every
correct fp16/bf16 output carries and 2e-2 is the budget for the kernel's own
arithmetic.  The half ulp is 2^-9 |O| or less in bf16 (2^-12 |O| in fp16):
below 2e-2 while |O| < 8 in bf16, the larger term from |O| >= 8 on.  The
mean bound, 2e-3, applies to |O_gpu - O_ref| with O_ref the oracle's output
as the oracle defines it: O rounded once to the output type (RNE).  Against
the unrounded value the mean would include the output rounding itself, about
ulp/4 on average, which is 0.002 already at |O| in [1, 2) in bf16; check()
reports that mean as well.  It also counts the elements whose error exceeds
2e-2 (those that needed the half-ulp term) and returns them in its
statistics.
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


def check(o_gpu, lse_gpu, o_ref, lse_ref, what="", stats=None):
    """Compare GPU O/LSE with the fp64 oracle (o_ref unrounded); returns the max O error.
    If ``stats`` is a dict it receives the max error, the mean error, the count
    of elements above 2e-2 and the largest |O_exact| among them, and the max
    LSE error."""
    dtype = o_gpu.dtype if isinstance(o_gpu, torch.Tensor) else torch.float32
    o = f64(o_gpu) if isinstance(o_gpu, torch.Tensor) else o_gpu
    assert o.shape == o_ref.shape, (what, o.shape, o_ref.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    err = np.abs(o - o_ref)
    bound = O_MAX + 0.5 * ulp(o_ref, dtype)
    if err.size:
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        assert np.all(err <= bound), (f"{what}: O err {err[i]} at |O|={abs(o_ref[i])} "
                                      f"(bound {bound[i]}), max err {err.max()}")
    mean_exact = float(err.mean()) if err.size else 0.0
    err_r = np.abs(o - round_to(o_ref, dtype))
    mean = float(err_r.mean()) if err.size else 0.0
    assert mean <= O_MEAN, f"{what}: O mean err {mean} (against the oracle rounded to {dtype})"
    over = err > O_MAX
    lse_err = 0.0
    if lse_gpu is not None:
        lg = f64(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
        assert lg.shape == lse_ref.shape, (what, lg.shape, lse_ref.shape)
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lg), inf_ref), f"{what}: -inf LSE pattern differs"
        fin = ~inf_ref
        if fin.any():
            e = np.abs(lg[fin] - lse_ref[fin])
            lse_err = float(e.max())
            assert lse_err <= LSE_TOL, f"{what}: LSE max err {lse_err}"
    if stats is not None:
        stats.update(max_err=float(err.max(initial=0.0)), mean_err=mean, mean_exact=mean_exact,
                     n=int(err.size), n_over_2e2=int(over.sum()),
                     max_abs_o_over=float(np.abs(o_ref[over]).max(initial=0.0)),
                     lse_max_err=lse_err)
    return float(err.max(initial=0.0))


def merge_stats(total, part):
    """Accumulate check() statistics over pieces of one output."""
    if not total:
        total.update(part)
        total["_sum"] = part["mean_err"] * part["n"]
        total["_sum_x"] = part["mean_exact"] * part["n"]
        return total
    total["_sum"] += part["mean_err"] * part["n"]
    total["_sum_x"] += part["mean_exact"] * part["n"]
    total["n"] += part["n"]
    total["mean_err"] = total["_sum"] / max(total["n"], 1)
    total["mean_exact"] = total["_sum_x"] / max(total["n"], 1)
    for k in ("max_err", "max_abs_o_over", "lse_max_err"):
        total[k] = max(total[k], part[k])
    total["n_over_2e2"] += part["n_over_2e2"]
    return total


def report(what, stats):
    """One line per full-size comparison (shown with pytest -s or -rP)."""
    print(f"PARITY {what}: {stats['n']} O elements, max |dO| {stats['max_err']:.4g}, "
          f"mean |dO| {stats['mean_err']:.3g} (vs rounded oracle; {stats['mean_exact']:.3g} vs "
          f"exact), above 2e-2: {stats['n_over_2e2']} "
          f"(largest |O| there {stats['max_abs_o_over']:.3g}), max |dLSE| "
          f"{stats['lse_max_err']:.3g}")


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


def compact_paged(inp, bsel):
    """The chosen sequences of a paged problem with only their own pages, in
    fp64, and a renumbered block table (bounds the oracle's host memory on a
    large pool)."""
    page = inp.page_size
    bt = inp.block_table
    lens = inp.seqlens_k
    pages, rows = [], []
    for b in bsel:
        n = (int(lens[b]) + page - 1) // page
        ids = bt[b, :n].tolist()
        rows.append(list(range(len(pages), len(pages) + n)))
        pages.extend(ids)
    idx = torch.tensor(pages, dtype=torch.long, device=inp.k_pool.device)
    kp = f64(inp.k_pool.index_select(0, idx))
    vp = f64(inp.v_pool.index_select(0, idx))
    maxn = max(max(len(r) for r in rows), 1)
    nbt = np.zeros((len(bsel), maxn), dtype=np.int32)
    for i, r in enumerate(rows):
        nbt[i, :len(r)] = r
    return kp, vp, nbt, lens[list(bsel)].numpy()

