"""fp64 CPU oracle for the fused attention forward (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product library never links or
calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, one query row at a
time, S and P materialised).  This module only compiles that file with gcc and
marshals numpy arrays into it.  Every function takes fp64 arrays holding the
exact values of the fp16/bf16 inputs (the widening is exact).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, a pure-Python brute force, invariants and planted mutants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int32)


def lib_path(mutant: int = 0) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (optionally a planted-mistake variant) with gcc."""
    path = lib_path(mutant)
    if not force and os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(_SRC):
        return path
    os.makedirs(_BUILD, exist_ok=True)
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    if mutant:
        cmd.insert(1, f"-DORACLE_MUTANT={mutant}")
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def _lib(mutant: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutant not in _libs:
            lib = ctypes.CDLL(build(mutant))
            m = [ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double]
            x = [ctypes.c_int, _D]  # top_left, alibi slopes [B][Hq]
            lib.oracle_attn_dense.argtypes = [_D, _D, _D, _D, _D] + [ctypes.c_int] * 6 + m + [
                _D, _D, _D] + x + [_D, ctypes.c_double]
            lib.oracle_attn_varlen.argtypes = [_D, _D, _D, _D, _D, _I, _I] + [ctypes.c_int] * 4 + m + [
                _D] + x + [ctypes.c_double]
            lib.oracle_attn_paged.argtypes = [_D, _D, _D, _I, _I, _D, _D] + [ctypes.c_int] * 7 + m + [
                _D] + x
            lib.oracle_attn_paged_partials.argtypes = [_D, _D, _D, _I, _I, _D, _D] + [
                ctypes.c_int] * 9 + m + x
            lib.oracle_combine.argtypes = [_D, _D, ctypes.c_int, ctypes.c_long, ctypes.c_int, _D,
                                           _D, _D]
            lib.oracle_mutant_id.restype = ctypes.c_int
            _libs[mutant] = lib
        return _libs[mutant]


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a):
    if a is None:
        return None
    if a.dtype == np.float64:
        return a.ctypes.data_as(_D)
    return a.ctypes.data_as(_I)


def _alibi(alibi, B, Hq):
    """ALiBi slopes broadcast to [B][Hq] (a [Hq] vector is shared by all batches)."""
    if alibi is None:
        return None
    return _f64(np.broadcast_to(np.asarray(alibi, dtype=np.float64), (B, Hq)))


def _check(rc: int, fn: str):
    if rc != 0:
        raise ValueError(f"oracle {fn}: invalid arguments")


def attn_dense(q, k, v, scale, causal=False, softcap=0.0, sink=None, want_sp=False, mutant=0,
               window=(-1, -1), top_left=False, alibi=None, bias=None, o_scale=1.0):
    """Dense attention.  q [B,Hq,Lq,d], k/v [B,Hkv,Lk,d] -> (o [B,Hq,Lq,d], lse [B,Hq,Lq])
    and, if ``want_sp``, the materialised S and P [B,Hq,Lq,Lk].  ``alibi``: slopes
    [B,Hq] or [Hq]; ``bias``: additive bias broadcastable to [B,Hq,Lq,Lk]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Lq, d = q.shape
    _, Hkv, Lk, _ = k.shape
    o = np.zeros((B, Hq, Lq, d))
    lse = np.zeros((B, Hq, Lq))
    sk = _f64(sink) if sink is not None else None
    s_out = np.zeros((B, Hq, Lq, Lk)) if want_sp else None
    p_out = np.zeros((B, Hq, Lq, Lk)) if want_sp else None
    al = _alibi(alibi, B, Hq)
    bi = None if bias is None else _f64(np.broadcast_to(np.asarray(bias, np.float64),
                                                        (B, Hq, Lq, Lk)))
    rc = _lib(mutant).oracle_attn_dense(_p(q), _p(k), _p(v), _p(o), _p(lse), B, Hq, Hkv, Lq, Lk,
                                        d, float(scale), int(bool(causal)), int(window[0]),
                                        int(window[1]), float(softcap), _p(sk), _p(s_out),
                                        _p(p_out), int(bool(top_left)), _p(al), _p(bi),
                                        float(o_scale))
    _check(rc, "attn_dense")
    if want_sp:
        return o, lse, s_out, p_out
    return o, lse


def attn_varlen(q, k, v, cu_q, cu_k, scale, causal=False, softcap=0.0, sink=None, mutant=0,
                window=(-1, -1), top_left=False, alibi=None, o_scale=1.0):
    """Varlen attention.  q [total_q,Hq,d], k/v [total_k,Hkv,d], cu int32 [B+1]
    -> (o [total_q,Hq,d], lse [Hq,total_q])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    total_q, Hq, d = q.shape
    Hkv = k.shape[1]
    B = cu_q.shape[0] - 1
    o = np.zeros((total_q, Hq, d))
    lse = np.zeros((Hq, total_q))
    sk = _f64(sink) if sink is not None else None
    rc = _lib(mutant).oracle_attn_varlen(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(cu_q), _p(cu_k),
                                         B, Hq, Hkv, d, float(scale), int(bool(causal)),
                                         int(window[0]), int(window[1]), float(softcap), _p(sk),
                                         int(bool(top_left)), _p(_alibi(alibi, B, Hq)),
                                         float(o_scale))
    _check(rc, "attn_varlen")
    return o, lse


def attn_paged(q, k_pool, v_pool, block_table, seqlens_k, scale, causal=False, softcap=0.0,
               sink=None, mutant=0, window=(-1, -1), top_left=False, alibi=None):
    """Paged-KV attention.  q [B,Lq,Hq,d], pools [P,page,Hkv,d], block_table int32
    [B,max_pages], seqlens_k int32 [B] -> (o [B,Lq,Hq,d], lse [B,Hq,Lq])."""
    q, kp, vp = _f64(q), _f64(k_pool), _f64(v_pool)
    bt, sl = _i32(block_table), _i32(seqlens_k)
    B, Lq, Hq, d = q.shape
    _, page, Hkv, _ = kp.shape
    o = np.zeros((B, Lq, Hq, d))
    lse = np.zeros((B, Hq, Lq))
    sk = _f64(sink) if sink is not None else None
    rc = _lib(mutant).oracle_attn_paged(_p(q), _p(kp), _p(vp), _p(bt), _p(sl), _p(o), _p(lse),
                                        B, Lq, Hq, Hkv, d, page, bt.shape[1], float(scale),
                                        int(bool(causal)), int(window[0]), int(window[1]),
                                        float(softcap), _p(sk), int(bool(top_left)),
                                        _p(_alibi(alibi, B, Hq)))
    _check(rc, "attn_paged")
    return o, lse


def attn_paged_partials(q, k_pool, v_pool, block_table, seqlens_k, num_splits, chunk_pages,
                        scale, causal=False, softcap=0.0, mutant=0, window=(-1, -1),
                        top_left=False, alibi=None):
    """Split-KV partials of the paged problem -> (o_part [S,B,Hq,Lq,d], lse_part [S,B,Hq,Lq])."""
    q, kp, vp = _f64(q), _f64(k_pool), _f64(v_pool)
    bt, sl = _i32(block_table), _i32(seqlens_k)
    B, Lq, Hq, d = q.shape
    _, page, Hkv, _ = kp.shape
    o = np.zeros((num_splits, B, Hq, Lq, d))
    lse = np.zeros((num_splits, B, Hq, Lq))
    rc = _lib(mutant).oracle_attn_paged_partials(
        _p(q), _p(kp), _p(vp), _p(bt), _p(sl), _p(o), _p(lse), B, Lq, Hq, Hkv, d, page,
        bt.shape[1], int(num_splits), int(chunk_pages), float(scale), int(bool(causal)),
        int(window[0]), int(window[1]), float(softcap), int(bool(top_left)),
        _p(_alibi(alibi, B, Hq)))
    _check(rc, "attn_paged_partials")
    return o, lse


def combine(o_part, lse_part, sink_rows=None, mutant=0):
    """Merge split partials.  o_part [S,rows,d], lse_part [S,rows] -> (o [rows,d], lse [rows])."""
    op, lp = _f64(o_part), _f64(lse_part)
    S, rows, d = op.shape
    o = np.zeros((rows, d))
    lse = np.zeros((rows,))
    sr = _f64(sink_rows) if sink_rows is not None else None
    rc = _lib(mutant).oracle_combine(_p(op), _p(lp), S, rows, d, _p(sr), _p(o), _p(lse))
    _check(rc, "combine")
    return o, lse


def mutant_id(mutant: int) -> int:
    return _lib(mutant).oracle_mutant_id()


MUTANTS = tuple(range(1, 14))
