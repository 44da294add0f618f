"""The work counts behind the bench's TFLOP/s and GB/s, checked on the CPU
against brute force over the mask and against the closed forms the
measurement section states (headline: 4 * d * B * H * L(L+1)/2 FLOP;
decode: K and V of every cached key once, plus Q, O and LSE)."""
import numpy as np
import pytest

import bench


def _kept(Lq, Lk, left, right):
    """Brute-force count of kept (i, j): bottom-right band, -1 = unbounded."""
    i = np.arange(Lq)[:, None] + (Lk - Lq)
    j = np.arange(Lk)[None, :]
    keep = np.ones((Lq, Lk), dtype=bool)
    if right >= 0:
        keep &= j <= i + right
    if left >= 0:
        keep &= j >= i - left
    return int(keep.sum())


@pytest.mark.parametrize("Lq,Lk", [(1, 1), (4, 4), (4, 2), (2, 7), (130, 300), (300, 130)])
def test_causal_pairs_brute_force(Lq, Lk):
    assert bench.causal_pairs(Lq, Lk) == _kept(Lq, Lk, -1, 0)


@pytest.mark.parametrize("Lq,Lk,left,right", [(8, 8, 2, 0), (8, 8, -1, 3), (50, 70, 10, 5),
                                              (70, 50, 0, 0), (64, 64, -1, -1), (1, 100, 7, 0)])
def test_window_pairs_brute_force(Lq, Lk, left, right):
    assert bench.window_pairs(Lq, Lk, left, right) == _kept(Lq, Lk, left, right)


def test_headline_flops_closed_form():
    """B4 H16 L2048 d128 causal: 4 * 128 * 4 * 16 * 2048 * 2049 / 2 = 68.75 GFLOP."""
    assert bench.dense_flops(4, 16, 2048, 2048, 128, True) == 4 * 128 * 4 * 16 * 2048 * 2049 // 2
    assert bench.dense_flops(1, 16, 2048, 2048, 128, False) == 4 * 128 * 16 * 2048 * 2048


def test_varlen_flops_sums_sequences():
    lens = [5, 0, 17]
    expect = sum(4 * 64 * 3 * L * (L + 1) // 2 for L in lens)
    assert bench.varlen_flops(lens, 3, 64, True) == expect


def test_paged_bytes():
    """Each cached key's K and V rows once per kv head (not per query head),
    Q read and O written once, fp32 LSE."""
    lens, Hkv, d, Lq, Hq = [100, 7], 2, 128, 1, 8
    kv = (100 + 7) * Hkv * d * 2 * 2
    qo = 2 * 2 * Lq * Hq * d * 2
    lse = 2 * Hq * Lq * 4
    assert bench.paged_bytes(lens, Hkv, d, Lq, Hq) == kv + qo + lse
