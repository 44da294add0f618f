"""A second, independent statement of the attention forward in plain Python
floats (fp64), used only to pin the C oracle on tiny shapes.

Written straight from the definition (Composable Kernel
fmha_fwd_pagedkv_kernel.hpp header comment: S = Q K^T, S' = S * scale,
S'' = S' + Bias, P = softmax(S''), O = P V), with the readings of the soft-cap,
sink, ALiBi, mask alignment and empty rows stated in the oracle.  No numpy, no
shared code.
"""
import math


def row(qv, keys, vals, scale, qi, Lq, causal, softcap, sink, window=(-1, -1), top_left=False,
        slope=0.0, bias_row=None):
    Lk = len(keys)
    scores = []
    diag = qi if top_left else qi + (Lk - Lq)
    for j in range(Lk):
        if causal and j > diag:
            continue
        if window[1] >= 0 and j > diag + window[1]:
            continue
        if window[0] >= 0 and j < diag - window[0]:
            continue
        s = scale * math.fsum(a * b for a, b in zip(qv, keys[j]))
        if softcap > 0:
            s = softcap * math.tanh(s / softcap)
        if bias_row is not None:
            s += bias_row[j]
        s -= slope * abs(diag - j)
        scores.append((j, s))
    logits = [s for _, s in scores] + ([sink] if sink is not None else [])
    d = len(qv)
    if not logits:
        return [0.0] * d, -math.inf
    m = max(logits)
    z = math.fsum(math.exp(x - m) for x in logits)
    lse = m + math.log(z)
    out = [0.0] * d
    for t in range(d):
        out[t] = math.fsum(math.exp(s - lse) * vals[j][t] for j, s in scores)
    return out, lse


def dense(q, k, v, scale, causal=False, softcap=0.0, sink=None, window=(-1, -1), top_left=False,
          alibi=None, bias=None):
    """q [B][Hq][Lq][d], k/v [B][Hkv][Lk][d] nested lists -> (o, lse).
    alibi: slopes [B][Hq] or None; bias: [B][Hq][Lq][Lk] or None."""
    B, Hq = len(q), len(q[0])
    Hkv = len(k[0])
    g = Hq // Hkv
    o = [[None] * Hq for _ in range(B)]
    lse = [[None] * Hq for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            Lq = len(q[b][h])
            rows = [row(q[b][h][i], k[b][h // g], v[b][h // g], scale, i, Lq, causal, softcap,
                        None if sink is None else sink[h], window, top_left,
                        0.0 if alibi is None else alibi[b][h],
                        None if bias is None else bias[b][h][i]) for i in range(Lq)]
            o[b][h] = [r[0] for r in rows]
            lse[b][h] = [r[1] for r in rows]
    return o, lse
