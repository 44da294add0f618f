"""Seeded synthetic inputs for the attention forward workloads.

This module draws random numbers and lays them out; it holds none of the
attention arithmetic, so both the CUDA path (tests, benchmark) and the fp64
oracle consume exactly the same bits from here.

Recipe (the workloads are shaped like the ones the pages' kernels target:
the dense [B,H,N,d] contract of the DefTruth FA2 kernel, the GQA / causal
problems of the FlashAttention-3 epilogue, the Composable Kernel paged-KV and
group-mode problems):

* One ``torch.Generator`` seeded with ``seed``.  Integers (sequence lengths,
  the page permutation) are drawn first, on the CPU, in this order:
  lengths, block-table permutation.  Then Q, K, V (and the sink logits) are
  drawn as fp32 N(0,1) on ``device`` from a generator with the same seed,
  multiplied by ``value_scale`` and rounded to fp16/bf16 (round to nearest
  even, torch's cast).
* Large tensors are drawn in chunks of at most 2^26 elements so the fp32
  staging buffer stays small; chunking does not change the stream.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

_CHUNK = 1 << 26

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}


def _randn(shape, gen, device, dtype, value_scale=1.0):
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if value_scale != 1.0:
            x.mul_(value_scale)
        flat[s:e].copy_(x)
    return out


def _gens(seed, device):
    cpu = torch.Generator(device="cpu")
    cpu.manual_seed(seed)
    dev = torch.Generator(device=device)
    dev.manual_seed(seed)
    return cpu, dev


@dataclass
class DenseInputs:
    q: torch.Tensor  # [B, Hq, Lq, d]
    k: torch.Tensor  # [B, Hkv, Lk, d]
    v: torch.Tensor  # [B, Hkv, Lk, d]
    causal: bool = False
    softcap: float = 0.0
    sink: torch.Tensor | None = None  # [Hq] fp32


@dataclass
class VarlenInputs:
    q: torch.Tensor  # [total_q, Hq, d]
    k: torch.Tensor  # [total_k, Hkv, d]
    v: torch.Tensor  # [total_k, Hkv, d]
    cu_seqlens_q: torch.Tensor  # int32 [B+1] (CPU)
    cu_seqlens_k: torch.Tensor  # int32 [B+1] (CPU)
    max_seqlen_q: int
    max_seqlen_k: int
    causal: bool = False
    softcap: float = 0.0
    sink: torch.Tensor | None = None


@dataclass
class PagedInputs:
    q: torch.Tensor  # [B, Lq, Hq, d]
    k_pool: torch.Tensor  # [num_pages, page, Hkv, d]
    v_pool: torch.Tensor  # [num_pages, page, Hkv, d]
    block_table: torch.Tensor  # int32 [B, max_pages] (CPU)
    seqlens_k: torch.Tensor  # int32 [B] (CPU)
    page_size: int
    causal: bool = False
    softcap: float = 0.0
    sink: torch.Tensor | None = None
    extra: dict = field(default_factory=dict)


def dense(B, Hq, Hkv, Lq, Lk, d, dtype="bf16", seed=0, device="cpu", value_scale=1.0,
          causal=False, softcap=0.0, with_sink=False) -> DenseInputs:
    dt = DTYPES[dtype]
    _, gen = _gens(seed, device)
    q = _randn((B, Hq, Lq, d), gen, device, dt, value_scale)
    k = _randn((B, Hkv, Lk, d), gen, device, dt, value_scale)
    v = _randn((B, Hkv, Lk, d), gen, device, dt, value_scale)
    sink = _randn((Hq,), gen, device, torch.float32) if with_sink else None
    return DenseInputs(q, k, v, causal, softcap, sink)


def varlen(lens_q, lens_k, Hq, Hkv, d, dtype="bf16", seed=0, device="cpu", value_scale=1.0,
           causal=False, softcap=0.0, with_sink=False) -> VarlenInputs:
    """Packed [total, H, d] sequences with the given per-sequence lengths."""
    dt = DTYPES[dtype]
    _, gen = _gens(seed, device)
    lens_q = [int(x) for x in lens_q]
    lens_k = [int(x) for x in lens_k]
    cu_q = torch.zeros(len(lens_q) + 1, dtype=torch.int32)
    cu_k = torch.zeros(len(lens_k) + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(torch.tensor(lens_q, dtype=torch.int64), 0).to(torch.int32)
    cu_k[1:] = torch.cumsum(torch.tensor(lens_k, dtype=torch.int64), 0).to(torch.int32)
    q = _randn((int(cu_q[-1]), Hq, d), gen, device, dt, value_scale)
    k = _randn((int(cu_k[-1]), Hkv, d), gen, device, dt, value_scale)
    v = _randn((int(cu_k[-1]), Hkv, d), gen, device, dt, value_scale)
    sink = _randn((Hq,), gen, device, torch.float32) if with_sink else None
    return VarlenInputs(q, k, v, cu_q, cu_k, max(lens_q, default=0), max(lens_k, default=0),
                        causal, softcap, sink)


def random_lengths(n, lo, hi, seed=None, cpu_gen=None):
    """n integers uniform in [lo, hi] from ``cpu_gen`` (or a CPU generator of ``seed``)."""
    g = cpu_gen
    if g is None:
        g = torch.Generator(device="cpu")
        g.manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def paged(seqlens_k, Lq, Hq, Hkv, d, page_size, num_pages, max_pages=None, dtype="bf16", seed=0,
          device="cpu", value_scale=1.0, causal=False, softcap=0.0, with_sink=False,
          shuffle=True, cpu_gen=None) -> PagedInputs:
    """A K/V page pool and a block table.

    Sequence b owns ceil(L_b / page) pages, taken as consecutive chunks of a
    random permutation of the pool (or of 0..P-1 when ``shuffle`` is False);
    unused table columns are 0.
    """
    dt = DTYPES[dtype]
    cpu, gen = _gens(seed, device)
    if cpu_gen is not None:
        cpu = cpu_gen
    seqlens_k = [int(x) for x in seqlens_k]
    npages = [(L + page_size - 1) // page_size for L in seqlens_k]
    if max_pages is None:
        max_pages = max(npages, default=1)
    if sum(npages) > num_pages:
        raise ValueError("pool too small for the requested sequences")
    perm = torch.randperm(num_pages, generator=cpu) if shuffle else torch.arange(num_pages)
    bt = torch.zeros(len(seqlens_k), max(max_pages, 1), dtype=torch.int32)
    pos = 0
    for b, n in enumerate(npages):
        bt[b, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    q = _randn((len(seqlens_k), Lq, Hq, d), gen, device, dt, value_scale)
    kp = _randn((num_pages, page_size, Hkv, d), gen, device, dt, value_scale)
    vp = _randn((num_pages, page_size, Hkv, d), gen, device, dt, value_scale)
    sink = _randn((Hq,), gen, device, torch.float32) if with_sink else None
    return PagedInputs(q, kp, vp, bt, torch.tensor(seqlens_k, dtype=torch.int32), page_size,
                       causal, softcap, sink)


# ---------------------------------------------------------------------------
# The five workloads.  Seeds are 1000 + the workload number (1..5).
# ---------------------------------------------------------------------------
WORKLOADS = {
    1: "tiny dense B1 H2 L128 d64 fp16 non-causal",
    2: "dense causal prefill B4 H16 L2048 d128 bf16",
    3: "GQA causal prefill B2 Hq32 Hkv8 L8192 d128 bf16",
    4: "paged-KV decode B64 Hq32 Hkv8 d128 page64 L~U[512,8192] bf16",
    5: "varlen causal prefill 16 seqs L~U[128,4096] H16 d64 bf16 softcap30 sink",
}


def workload(n: int, device="cpu"):
    seed = 1000 + n
    if n == 1:
        return dense(1, 2, 2, 128, 128, 64, "f16", seed, device)
    if n == 2:
        return dense(4, 16, 16, 2048, 2048, 128, "bf16", seed, device, causal=True)
    if n == 3:
        return dense(2, 32, 8, 8192, 8192, 128, "bf16", seed, device, causal=True)
    if n == 4:
        cpu = torch.Generator(device="cpu")
        cpu.manual_seed(seed)
        lens = random_lengths(64, 512, 8192, cpu_gen=cpu)
        return paged(lens, 1, 32, 8, 128, 64, 10240, max_pages=128, dtype="bf16", seed=seed,
                     device=device, cpu_gen=cpu)
    if n == 5:
        lens = random_lengths(16, 128, 4096, seed)
        return varlen(lens, lens, 16, 16, 64, "bf16", seed, device, value_scale=2.0,
                      causal=True, softcap=30.0, with_sink=True)
    raise KeyError(n)
