"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, never against the oracle itself or the CUDA path.

Each ``pin_*`` function raises AssertionError on a mismatch and takes the
oracle variant to check (0 = the real oracle, n > 0 = a build with planted
mistake n).  ``test_mutants_are_caught`` proves the pins have teeth: every
planted mistake (see oracle.MUTANTS and the MUTANT() sites of attn_oracle.c:
wrong index, dropped scale, dropped cap, top-left causal, dropped sink,
dropped max term, transposed V, interleaved GQA grouping, a left-window bound
off by one, a flipped ALiBi sign, a shifted bias row, the output scale applied
to LSE, the output scale dropped in group mode) fails at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from tests import _brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")
EV = {"math": math}


def _ev(x):
    return float(eval(x, EV)) if isinstance(x, str) else float(x)


def _evtree(t):
    return np.vectorize(_ev, otypes=[float])(np.array(t, dtype=object))


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(a - b))
    err = np.nan_to_num(err, nan=np.inf)
    assert float(err.max(initial=0.0)) <= tol, f"{what}: max err {err.max()} > {tol}"


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_golden(mutant=0):
    """Hand-derived closed forms (tests/golden/closed_forms.json)."""
    cases = json.load(open(GOLDEN))
    for c in cases["dense"]:
        q, k, v = (np.array(c[x], dtype=np.float64) for x in ("q", "k", "v"))
        o, lse = oracle.attn_dense(q, k, v, c["scale"], c["causal"], c["softcap"],
                                   c["sink"], mutant=mutant, o_scale=c.get("o_scale", 1.0))
        _close(o, _evtree(c["expect_o"]), 1e-13, c["name"] + " O")
        _close(lse, _evtree(c["expect_lse"]), 1e-13, c["name"] + " LSE")
    for c in cases["combine"]:
        o, lse = oracle.combine(np.array(c["o_part"]), _evtree(c["lse_part"]), mutant=mutant)
        _close(o, _evtree(c["expect_o"]), 1e-13, c["name"] + " O")
        _close(lse, _evtree(c["expect_lse"]), 1e-13, c["name"] + " LSE")


def pin_rows_sum_to_one(mutant=0):
    """Every materialised softmax row (plus the sink mass) sums to 1."""
    r = _rng(1)
    for causal, sink in ((False, None), (True, None), (True, r.standard_normal(4))):
        q = r.standard_normal((2, 4, 9, 8))
        k = r.standard_normal((2, 2, 13, 8))
        v = r.standard_normal((2, 2, 13, 8))
        o, lse, s, p = oracle.attn_dense(q, k, v, 0.35, causal, 0.0, sink, want_sp=True,
                                         mutant=mutant)
        tot = p.sum(-1)
        if sink is not None:
            tot = tot + np.exp(np.asarray(sink)[None, :, None] - lse)
        _close(tot, np.ones_like(tot), 1e-12, "row sums")


def pin_identical_keys(mutant=0):
    """All keys equal: O_i = mean_j v_j and LSE_i = s_i + ln Lk (closed form)."""
    r = _rng(2)
    d, Lk = 16, 37
    q = r.standard_normal((1, 3, 5, d))
    k1 = r.standard_normal(d)
    k = np.broadcast_to(k1, (1, 3, Lk, d)).copy()
    v = r.standard_normal((1, 3, Lk, d))
    scale = 0.21
    o, lse = oracle.attn_dense(q, k, v, scale, mutant=mutant)
    _close(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), 1e-12, "mean of V")
    s = scale * np.einsum("bhid,d->bhi", q, k1)
    _close(lse, s + math.log(Lk), 1e-12, "LSE identical keys")


def pin_one_hot(mutant=0):
    """One dominant score selects its V row, up to exp(-gap)."""
    r = _rng(3)
    d, Lk = 8, 11
    k = 0.01 * r.standard_normal((1, 1, Lk, d))
    jstar = 7
    k[0, 0, jstar] = 0.0
    k[0, 0, jstar, 0] = 50.0
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 1.0
    v = r.standard_normal((1, 1, Lk, d))
    o, lse = oracle.attn_dense(q, k, v, 1.0, mutant=mutant)
    gap = 50.0 - 0.5
    tol = Lk * math.exp(-gap) * np.abs(v).max() * 2
    _close(o[0, 0, 0], v[0, 0, jstar], tol, "one-hot row")


def pin_lse_fsum(mutant=0):
    """LSE equals log sum exp of the scores, summed independently with fsum."""
    r = _rng(4)
    q = r.standard_normal((1, 2, 4, 5))
    k = r.standard_normal((1, 2, 6, 5))
    v = r.standard_normal((1, 2, 6, 5))
    scale = 0.7
    o, lse = oracle.attn_dense(q, k, v, scale, mutant=mutant)
    for h in range(2):
        for i in range(4):
            sc = [scale * math.fsum(q[0, h, i, t] * k[0, h, j, t] for t in range(5))
                  for j in range(6)]
            m = max(sc)
            ref = m + math.log(math.fsum(math.exp(x - m) for x in sc))
            assert abs(lse[0, h, i] - ref) <= 1e-13, (h, i, lse[0, h, i], ref)


def pin_causal_row0(mutant=0):
    """Causal with Lq = Lk: row 0 sees key 0 only, so O_0 = V[0] exactly."""
    r = _rng(5)
    q = r.standard_normal((2, 3, 10, 8))
    k = r.standard_normal((2, 3, 10, 8))
    v = r.standard_normal((2, 3, 10, 8))
    o, lse = oracle.attn_dense(q, k, v, 0.4, causal=True, mutant=mutant)
    _close(o[:, :, 0], v[:, :, 0], 0.0, "causal row 0")
    _close(lse[:, :, 0], 0.4 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]), 1e-14,
           "causal row 0 LSE")


def pin_empty_rows(mutant=0):
    """Bottom-right causal with Lq > Lk leaves the first Lq - Lk rows empty:
    O = 0 and LSE = -inf, or LSE = sigma with a sink (store_zero)."""
    r = _rng(6)
    q = r.standard_normal((1, 2, 7, 4))
    k = r.standard_normal((1, 2, 3, 4))
    v = r.standard_normal((1, 2, 3, 4))
    o, lse = oracle.attn_dense(q, k, v, 0.5, causal=True, mutant=mutant)
    assert np.all(o[:, :, :4] == 0.0)
    assert np.all(np.isneginf(lse[:, :, :4]))
    assert np.all(np.isfinite(lse[:, :, 4:]))
    sink = np.array([0.3, -1.2])
    o, lse = oracle.attn_dense(q, k, v, 0.5, causal=True, sink=sink, mutant=mutant)
    assert np.all(o[:, :, :4] == 0.0)
    _close(lse[0, :, :4], np.broadcast_to(sink[:, None], (2, 4)), 0.0, "sink-only rows")


def pin_brute_force(mutant=0):
    """A second implementation in plain Python floats agrees to 1e-12."""
    r = _rng(7)
    cases = [
        dict(B=1, Hq=2, Hkv=2, Lq=3, Lk=5, d=4, causal=False, cap=0.0, sink=False),
        dict(B=2, Hq=4, Hkv=2, Lq=5, Lk=3, d=3, causal=True, cap=0.0, sink=False),
        dict(B=1, Hq=3, Hkv=1, Lq=4, Lk=6, d=5, causal=True, cap=0.8, sink=True),
        dict(B=1, Hq=2, Hkv=1, Lq=6, Lk=6, d=2, causal=True, cap=0.0, sink=True),
        dict(B=1, Hq=1, Hkv=1, Lq=1, Lk=8, d=8, causal=False, cap=2.0, sink=False),
    ]
    for c in cases:
        q = r.standard_normal((c["B"], c["Hq"], c["Lq"], c["d"]))
        k = r.standard_normal((c["B"], c["Hkv"], c["Lk"], c["d"]))
        v = r.standard_normal((c["B"], c["Hkv"], c["Lk"], c["d"]))
        sink = r.standard_normal(c["Hq"]) if c["sink"] else None
        scale = 1.0 / math.sqrt(c["d"])
        o, lse = oracle.attn_dense(q, k, v, scale, c["causal"], c["cap"], sink, mutant=mutant)
        bo, bl = _brute.dense(q.tolist(), k.tolist(), v.tolist(), scale, c["causal"], c["cap"],
                              None if sink is None else sink.tolist())
        _close(o, np.array(bo), 1e-12, f"brute O {c}")
        _close(lse, np.array(bl), 1e-12, f"brute LSE {c}")


def pin_softcap_limits(mutant=0):
    """Cap -> infinity reproduces the uncapped result; every capped score obeys |s| <= cap."""
    r = _rng(8)
    q = 3 * r.standard_normal((1, 2, 6, 8))
    k = 3 * r.standard_normal((1, 2, 9, 8))
    v = r.standard_normal((1, 2, 9, 8))
    o0, l0 = oracle.attn_dense(q, k, v, 0.3, mutant=mutant)
    o1, l1 = oracle.attn_dense(q, k, v, 0.3, softcap=1e9, mutant=mutant)
    _close(o1, o0, 1e-9, "cap->inf O")
    _close(l1, l0, 1e-9, "cap->inf LSE")
    cap = 0.5
    _, _, s, _ = oracle.attn_dense(q, k, v, 0.3, softcap=cap, want_sp=True, mutant=mutant)
    assert np.all(np.abs(s) <= cap)
    # and the capped scores are cap*tanh(raw/cap)
    raw = 0.3 * np.einsum("bhid,bhjd->bhij", q, k)
    _close(s, cap * np.tanh(raw / cap), 1e-14, "capped scores")


def pin_sink_limits(mutant=0):
    """sigma = -inf is no sink; sigma -> +inf drives O to 0 and LSE to sigma."""
    r = _rng(9)
    q = r.standard_normal((1, 2, 5, 4))
    k = r.standard_normal((1, 2, 7, 4))
    v = r.standard_normal((1, 2, 7, 4))
    o0, l0 = oracle.attn_dense(q, k, v, 0.5, mutant=mutant)
    o1, l1 = oracle.attn_dense(q, k, v, 0.5, sink=np.array([-np.inf, -np.inf]), mutant=mutant)
    _close(o1, o0, 0.0, "sink -inf O")
    _close(l1, l0, 0.0, "sink -inf LSE")
    big = 60.0
    o2, l2 = oracle.attn_dense(q, k, v, 0.5, sink=np.array([big, big]), mutant=mutant)
    _close(o2, np.zeros_like(o2), 1e-20, "sink +inf O")
    _close(l2, np.full_like(l2, big), 1e-12, "sink +inf LSE")


def pin_gqa_equals_repeated_mha(mutant=0):
    """GQA with g = 4, Hkv = 8 equals MHA on K/V with each kv head repeated for
    its 4 consecutive query heads (Composable Kernel: kv head = h / ratio)."""
    r = _rng(10)
    q = r.standard_normal((1, 32, 3, 4))
    k = r.standard_normal((1, 8, 5, 4))
    v = r.standard_normal((1, 8, 5, 4))
    og, lg = oracle.attn_dense(q, k, v, 0.5, causal=True, mutant=mutant)
    om, lm = oracle.attn_dense(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), 0.5,
                               causal=True, mutant=mutant)
    _close(og, om, 0.0, "GQA O")
    _close(lg, lm, 0.0, "GQA LSE")


def _paged_case(r, B=3, Lq=2, Hq=4, Hkv=2, d=8, page=4, lens=(9, 4, 1)):
    npages = [(L + page - 1) // page for L in lens]
    P = sum(npages) + 3
    perm = r.permutation(P)
    maxp = max(npages) + 1
    bt = np.zeros((B, maxp), dtype=np.int32)
    pos = 0
    for b, n in enumerate(npages):
        bt[b, :n] = perm[pos:pos + n]
        pos += n
    kp = r.standard_normal((P, page, Hkv, d))
    vp = r.standard_normal((P, page, Hkv, d))
    q = r.standard_normal((B, Lq, Hq, d))
    return q, kp, vp, bt, np.array(lens, dtype=np.int32)


def _contiguous_from_paged(kp, bt, lens, b, page):
    L = lens[b]
    rows = [kp[bt[b, j // page], j % page] for j in range(L)]  # [L][Hkv][d]
    return np.array(rows).transpose(1, 0, 2)  # [Hkv][L][d]


def pin_paged_equals_contiguous(mutant=0):
    """A shuffled pool + block table gives bit-identically the contiguous result."""
    r = _rng(11)
    page = 4
    q, kp, vp, bt, lens = _paged_case(r, page=page)
    slopes = np.abs(r.standard_normal((len(lens), q.shape[2])))
    for causal, tl, al in ((False, False, None), (True, False, None), (True, True, slopes),
                           (False, False, slopes)):
        o, lse = oracle.attn_paged(q, kp, vp, bt, lens, 0.4, causal, mutant=mutant, top_left=tl,
                                   alibi=al)
        for b in range(len(lens)):
            kc = _contiguous_from_paged(kp, bt, lens, b, page)[None]
            vc = _contiguous_from_paged(vp, bt, lens, b, page)[None]
            qd = q[b].transpose(1, 0, 2)[None]  # [1][Hq][Lq][d]
            od, ld = oracle.attn_dense(qd, kc, vc, 0.4, causal, mutant=mutant, top_left=tl,
                                       alibi=None if al is None else al[b:b + 1])
            _close(o[b].transpose(1, 0, 2), od[0], 0.0, "paged O")
            _close(lse[b], ld[0], 0.0, "paged LSE")


def pin_splits_combine_to_unsplit(mutant=0):
    """Split-KV partials merged by the combine equal the unsplit result (1e-12),
    including empty splits, the sink added once in the merge, causal Lq > 1 and
    window bands (splits laid from the band's first page)."""
    r = _rng(12)
    page = 4
    q, kp, vp, bt, lens = _paged_case(r, page=page, lens=(9, 4, 1))
    sink = r.standard_normal(4)
    # With a left window the splits start at the page of the first kept key;
    # every layout below spans at least the pages the band can reach.
    slopes = np.abs(r.standard_normal((len(lens), 4)))
    for causal, window, tl, al in ((False, (-1, -1), False, None), (True, (-1, -1), False, None),
                                   (True, (2, -1), False, None), (False, (1, 1), False, None),
                                   (False, (5, 0), False, None), (True, (2, -1), True, slopes),
                                   (False, (-1, -1), False, slopes)):
        for num_splits, chunk in ((1, 3), (2, 2), (4, 1), (3, 2)):
            op, lp = oracle.attn_paged_partials(q, kp, vp, bt, lens, num_splits, chunk, 0.4,
                                                causal, mutant=mutant, window=window,
                                                top_left=tl, alibi=al)
            B, Lq, Hq, d = q.shape
            rows = B * Hq * Lq
            sink_rows = np.broadcast_to(sink[None, :, None], (B, Hq, Lq)).reshape(-1)
            o, lse = oracle.combine(op.reshape(num_splits, rows, d), lp.reshape(num_splits, rows),
                                    sink_rows, mutant=mutant)
            o_ref, l_ref = oracle.attn_paged(q, kp, vp, bt, lens, 0.4, causal, sink=sink,
                                             mutant=mutant, window=window, top_left=tl,
                                             alibi=al)
            _close(o.reshape(B, Hq, Lq, d), o_ref.transpose(0, 2, 1, 3), 1e-12, "combine O")
            _close(lse.reshape(B, Hq, Lq), l_ref, 1e-12, "combine LSE")


def pin_varlen_equals_per_sequence(mutant=0):
    """Group mode: each packed sequence gives its own dense result."""
    r = _rng(13)
    lq, lk = [3, 1, 6], [5, 2, 6]
    Hq, Hkv, d = 4, 2, 4
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    q = r.standard_normal((cu_q[-1], Hq, d))
    k = r.standard_normal((cu_k[-1], Hkv, d))
    v = r.standard_normal((cu_k[-1], Hkv, d))
    sink = r.standard_normal(Hq)
    slopes = np.abs(r.standard_normal((3, Hq)))
    for tl, al in ((False, None), (True, slopes), (False, slopes)):
        o, lse = oracle.attn_varlen(q, k, v, cu_q, cu_k, 0.5, True, 0.7, sink, mutant=mutant,
                                    top_left=tl, alibi=al)
        for b in range(3):
            qs = q[cu_q[b]:cu_q[b + 1]].transpose(1, 0, 2)[None]
            ks = k[cu_k[b]:cu_k[b + 1]].transpose(1, 0, 2)[None]
            vs = v[cu_k[b]:cu_k[b + 1]].transpose(1, 0, 2)[None]
            od, ld = oracle.attn_dense(qs, ks, vs, 0.5, True, 0.7, sink, mutant=mutant,
                                       top_left=tl, alibi=None if al is None else al[b:b + 1])
            _close(o[cu_q[b]:cu_q[b + 1]].transpose(1, 0, 2), od[0], 0.0, "varlen O")
            _close(lse[:, cu_q[b]:cu_q[b + 1]], ld[0], 0.0, "varlen LSE")


def pin_window(mutant=0):
    """Sliding window (bottom-right aligned, CK window_size_left/right):
    brute force agrees; (-1,-1) is no mask; (-1,0) is causal; (0,0) keeps only
    key i + (Lk - Lq), so O_i = V[i + Lk - Lq] and LSE_i is that one score."""
    r = _rng(14)
    for (Lq, Lk, wl, wr, causal, cap, sink) in ((6, 9, 2, 1, False, 0.0, False),
                                               (9, 6, 3, 0, True, 0.0, True),
                                               (5, 5, 0, 2, False, 1.5, False),
                                               (4, 11, 1, -1, False, 0.0, True)):
        q = r.standard_normal((1, 2, Lq, 4))
        k = r.standard_normal((1, 1, Lk, 4))
        v = r.standard_normal((1, 1, Lk, 4))
        sk = r.standard_normal(2) if sink else None
        o, lse = oracle.attn_dense(q, k, v, 0.6, causal, cap, sk, mutant=mutant, window=(wl, wr))
        bo, bl = _brute.dense(q.tolist(), k.tolist(), v.tolist(), 0.6, causal, cap,
                              None if sk is None else sk.tolist(), window=(wl, wr))
        _close(o, np.array(bo), 1e-12, f"window brute O {Lq, Lk, wl, wr}")
        _close(lse, np.array(bl), 1e-12, f"window brute LSE {Lq, Lk, wl, wr}")
    q = r.standard_normal((1, 2, 7, 4))
    k = r.standard_normal((1, 2, 10, 4))
    v = r.standard_normal((1, 2, 10, 4))
    o0, l0 = oracle.attn_dense(q, k, v, 0.5, mutant=mutant)
    o1, l1 = oracle.attn_dense(q, k, v, 0.5, mutant=mutant, window=(-1, -1))
    _close(o1, o0, 0.0, "window unbounded")
    oc, lc = oracle.attn_dense(q, k, v, 0.5, causal=True, mutant=mutant)
    o2, l2 = oracle.attn_dense(q, k, v, 0.5, mutant=mutant, window=(-1, 0))
    _close(o2, oc, 0.0, "window (-1, 0) is causal")
    _close(l2, lc, 0.0, "window (-1, 0) is causal, LSE")
    o3, l3 = oracle.attn_dense(q, k, v, 0.5, mutant=mutant, window=(0, 0))
    _close(o3, v[:, :, 3:10], 0.0, "width-one window")
    _close(l3, 0.5 * np.einsum("bhid,bhid->bhi", q, k[:, :, 3:10]), 1e-14, "width-one LSE")


def pin_bias_alibi_top_left(mutant=0):
    """Additive bias, ALiBi and the top-left mask alignment (Composable Kernel
    FMHA forward: bias kargs, ALiBi slope per (batch, head) aligned like the
    mask, MASK_FROM_TOP_LEFT): brute force agrees; a per-row constant bias only
    shifts the LSE; a bias of -inf above the diagonal is the causal mask; ALiBi
    equals the explicit bias -slope*|diag - j| built here; a two-key closed form
    fixes the ALiBi sign; top-left equals bottom-right when Lq = Lk and keeps
    only key 0 for row 0 under causal."""
    r = _rng(21)
    for (Lq, Lk, causal, win, tl) in ((5, 7, True, (-1, -1), False), (7, 5, True, (-1, -1), True),
                                      (6, 6, False, (2, 1), True), (4, 9, False, (-1, -1), False)):
        q = r.standard_normal((2, 2, Lq, 4))
        k = r.standard_normal((2, 1, Lk, 4))
        v = r.standard_normal((2, 1, Lk, 4))
        al = np.abs(r.standard_normal((2, 2))) * 0.3
        bias = r.standard_normal((2, 2, Lq, Lk))
        o, lse = oracle.attn_dense(q, k, v, 0.5, causal, mutant=mutant, window=win, top_left=tl,
                                   alibi=al, bias=bias)
        bo, bl = _brute.dense(q.tolist(), k.tolist(), v.tolist(), 0.5, causal, window=win,
                              top_left=tl, alibi=al.tolist(), bias=bias.tolist())
        _close(o, np.array(bo), 1e-12, f"bias/alibi brute O {Lq, Lk, causal, win, tl}")
        _close(lse, np.array(bl), 1e-12, f"bias/alibi brute LSE {Lq, Lk, causal, win, tl}")
    q = r.standard_normal((1, 2, 6, 4))
    k = r.standard_normal((1, 2, 8, 4))
    v = r.standard_normal((1, 2, 8, 4))
    o0, l0 = oracle.attn_dense(q, k, v, 0.5, mutant=mutant)
    c = r.standard_normal((1, 2, 6, 1))
    o1, l1 = oracle.attn_dense(q, k, v, 0.5, mutant=mutant, bias=np.broadcast_to(c, (1, 2, 6, 8)))
    _close(o1, o0, 1e-13, "row-constant bias leaves O")
    _close(l1, l0 + c[..., 0], 1e-13, "row-constant bias shifts LSE")
    i = np.arange(6)[:, None]
    j = np.arange(8)[None, :]
    diag = i + (8 - 6)
    neg = np.where(j > diag, -np.inf, 0.0)
    oc, lc = oracle.attn_dense(q, k, v, 0.5, causal=True, mutant=mutant)
    o2, l2 = oracle.attn_dense(q, k, v, 0.5, mutant=mutant, bias=neg)
    _close(o2, oc, 1e-13, "-inf bias above the diagonal is causal")
    _close(l2, lc, 1e-13, "-inf bias above the diagonal is causal, LSE")
    slopes = np.array([[0.25, 0.7]])
    explicit = -slopes[0][None, :, None, None] * np.abs(diag - j)[None, None]
    o3, l3 = oracle.attn_dense(q, k, v, 0.5, mutant=mutant, alibi=slopes)
    o4, l4 = oracle.attn_dense(q, k, v, 0.5, mutant=mutant, bias=explicit)
    _close(o3, o4, 1e-13, "ALiBi equals its explicit bias")
    _close(l3, l4, 1e-13, "ALiBi equals its explicit bias, LSE")
    o5, _ = oracle.attn_dense(q, k, v, 0.5, mutant=mutant, alibi=np.zeros((1, 2)))
    _close(o5, o0, 0.0, "zero slope is no ALiBi")
    # Two identical keys, one query on the diagonal of key 1 (bottom-right):
    # weights e^{-m} (key 0, distance 1) and 1 (key 1).
    m = 0.9
    kk = np.ones((1, 1, 2, 4))
    vv = np.array([[[[1.0, 0, 0, 0], [0, 1.0, 0, 0]]]])
    qq = np.ones((1, 1, 1, 4))
    o6, l6 = oracle.attn_dense(qq, kk, vv, 0.5, mutant=mutant, alibi=np.array([[m]]))
    w0 = math.exp(-m) / (math.exp(-m) + 1.0)
    _close(o6[0, 0, 0], [w0, 1.0 - w0, 0, 0], 1e-14, "ALiBi two-key closed form")
    _close(l6[0, 0, 0], 2.0 + math.log(math.exp(-m) + 1.0), 1e-14, "ALiBi two-key LSE")
    ob, lb = oracle.attn_dense(q[:, :, :6], k[:, :, :6], v[:, :, :6], 0.5, causal=True,
                               mutant=mutant)
    ot, lt = oracle.attn_dense(q[:, :, :6], k[:, :, :6], v[:, :, :6], 0.5, causal=True,
                               mutant=mutant, top_left=True)
    _close(ot, ob, 0.0, "top-left equals bottom-right when Lq = Lk")
    o7, _ = oracle.attn_dense(q, k, v, 0.5, causal=True, mutant=mutant, top_left=True)
    _close(o7[:, :, 0], v[:, :, 0], 1e-14, "top-left causal row 0 is V[0]")


def pin_output_scale(mutant=0):
    """FP8 static quantisation's output scale (Composable Kernel
    FmhaFwdFp8StaticQuantKargs: O's accumulator times scale_o, P times scale_p;
    reading: O = scale_o * scale_p * softmax(S) V and LSE is not scaled).  For
    dense and group mode: O(s) equals s * O(1) exactly (one fp64 multiply of
    the same value on both sides), LSE(s) equals LSE(1) exactly."""
    rng = _rng(77)
    q, k, v = (rng.standard_normal(sh) for sh in ((2, 4, 5, 8), (2, 2, 7, 8), (2, 2, 7, 8)))
    sink = rng.standard_normal(4)
    for s in (2.0, 0.3):
        o1, l1 = oracle.attn_dense(q, k, v, 0.4, True, 0.0, sink, mutant=mutant)
        os_, ls = oracle.attn_dense(q, k, v, 0.4, True, 0.0, sink, mutant=mutant, o_scale=s)
        _close(os_, s * o1, 0.0, f"dense O(o_scale={s}) = s O(1)")
        _close(ls, l1, 0.0, f"dense LSE(o_scale={s}) = LSE(1)")
    lens = [3, 0, 6]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    qv = rng.standard_normal((int(cu[-1]), 4, 8))
    kv_ = rng.standard_normal((int(cu[-1]), 2, 8))
    vv = rng.standard_normal((int(cu[-1]), 2, 8))
    for s in (2.0, 0.3):
        o1, l1 = oracle.attn_varlen(qv, kv_, vv, cu, cu, 0.4, True, 0.0, sink, mutant=mutant)
        os_, ls = oracle.attn_varlen(qv, kv_, vv, cu, cu, 0.4, True, 0.0, sink, mutant=mutant,
                                     o_scale=s)
        _close(os_, s * o1, 0.0, f"varlen O(o_scale={s}) = s O(1)")
        _close(ls, l1, 0.0, f"varlen LSE(o_scale={s}) = LSE(1)")


PINS = [pin_golden, pin_rows_sum_to_one, pin_identical_keys, pin_one_hot, pin_lse_fsum,
        pin_causal_row0, pin_empty_rows, pin_brute_force, pin_softcap_limits, pin_sink_limits,
        pin_gqa_equals_repeated_mha, pin_paged_equals_contiguous, pin_splits_combine_to_unsplit,
        pin_varlen_equals_per_sequence, pin_window, pin_bias_alibi_top_left,
        pin_output_scale]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(0)


@pytest.mark.parametrize("mutant", oracle.MUTANTS)
def test_mutants_are_caught(mutant):
    assert oracle.mutant_id(mutant) == mutant
    failed = []
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted mistake {mutant} passed every pin"
