"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module draws random numbers and fixes shapes; it holds none of the
attention arithmetic.  Every tensor is drawn on the CPU from a
``torch.Generator`` seeded per workload, as fp32 N(0, 1), then rounded to
bf16, so the CUDA library and the fp64 oracle see bit-identical values.
Integer lengths (decode ``kv_lens``, packed ``cu_seqlens``) come from the same
generator.

The named workloads follow the attention shapes the source pages discuss:
single-token decode over long KV caches with grouped-query heads, and
prefill at 4k-8k tokens, causal and non-causal, dense and packed.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Workload", "WORKLOADS", "make_prefill", "make_decode", "make_decode_multi", "make_varlen", "make_pages",
           "randn_bf16", "rope_tables"]


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "prefill" | "decode" | "decode_multi" | "varlen"
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    L: int = 0  # prefill Lq == Lkv; decode Lmax
    Lq: int = 1  # decode_multi: new tokens per sequence
    causal: bool = True
    out_f32: bool = False
    kv_lens: tuple = ()  # decode: fixed lengths, or () to draw from kv_range
    kv_range: tuple = ()  # decode: inclusive (lo, hi) for uniform integer lengths
    seq_range: tuple = ()  # varlen: inclusive (lo, hi) of sequence lengths
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_causal", "prefill", 1000, B=1, Hq=2, Hkv=2, D=64, L=128, causal=True, out_f32=True),
        Workload("decode_gqa", "decode", 1001, B=8, Hq=32, Hkv=8, D=128, L=4096, kv_range=(512, 4096)),
        Workload("decode_gqa_paged16", "decode", 1001, B=8, Hq=32, Hkv=8, D=128, L=4096, kv_range=(512, 4096),
                 extra={"page_size": 16}),
        Workload("decode_gqa_rope", "decode", 1001, B=8, Hq=32, Hkv=8, D=128, L=4096, kv_range=(512, 4096),
                 extra={"rope": "half"}),
        Workload("decode_long", "decode", 1002, B=4, Hq=32, Hkv=8, D=128, L=131072,
                 kv_lens=(32768, 65536, 98304, 131072)),
        Workload("decode_multi_gqa", "decode_multi", 1006, B=8, Hq=32, Hkv=8, D=128, L=4096, Lq=8,
                 kv_range=(512, 4096)),
        Workload("decode_multi_long", "decode_multi", 1007, B=4, Hq=32, Hkv=8, D=128, L=131072, Lq=8,
                 kv_lens=(32768, 65536, 98304, 131072)),
        Workload("prefill_causal", "prefill", 1003, B=4, Hq=32, Hkv=32, D=128, L=4096, causal=True),
        Workload("prefill_causal_rope", "prefill", 1003, B=4, Hq=32, Hkv=32, D=128, L=4096, causal=True,
                 extra={"rope": "half"}),
        Workload("prefill_ragged_gqa", "varlen", 1004, B=16, Hq=32, Hkv=8, D=128, causal=True,
                 seq_range=(256, 8192)),
        Workload("prefill_noncausal_d64", "prefill", 1005, B=2, Hq=16, Hkv=16, D=64, L=8192, causal=False),
    ]
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, g: torch.Generator, chunk_elems: int = 1 << 26) -> torch.Tensor:
    """N(0,1) drawn in fp32 and rounded to bf16, produced in chunks to bound host memory."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.bfloat16)
    for start in range(0, n, chunk_elems):
        stop = min(n, start + chunk_elems)
        out[start:stop] = torch.randn(stop - start, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def make_prefill(B, Hq, Hkv, Lq, Lkv, D, seed):
    """Dense prefill inputs: q [B,Hq,Lq,D], k/v [B,Hkv,Lkv,D], bf16."""
    g = _gen(seed)
    q = randn_bf16((B, Hq, Lq, D), g)
    k = randn_bf16((B, Hkv, Lkv, D), g)
    v = randn_bf16((B, Hkv, Lkv, D), g)
    return q, k, v


def make_decode(B, Hq, Hkv, Lmax, D, seed, kv_lens=None, kv_range=None):
    """Decode inputs: q [B,Hq,D], caches [B,Hkv,Lmax,D] bf16, kv_lens int32 [B].

    ``kv_lens`` fixes the lengths; otherwise they are drawn uniformly from the
    inclusive ``kv_range`` with the same generator (after the tensors); with
    neither, every sequence uses the whole cache.
    """
    g = _gen(seed)
    q = randn_bf16((B, Hq, D), g)
    kc = randn_bf16((B, Hkv, Lmax, D), g)
    vc = randn_bf16((B, Hkv, Lmax, D), g)
    if kv_lens is not None and len(kv_lens) > 0:
        lens = torch.tensor(list(kv_lens), dtype=torch.int32)
    elif kv_range is None:
        lens = torch.full((B,), int(Lmax), dtype=torch.int32)
    else:
        lo, hi = kv_range
        lens = torch.randint(int(lo), int(hi) + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    return q, kc, vc, lens


def make_decode_multi(B, Hq, Hkv, Lq, Lmax, D, seed, kv_lens=None, kv_range=None):
    """Multi-token decode inputs: q [B,Hq,Lq,D], caches [B,Hkv,Lmax,D] bf16, kv_lens int32 [B].

    Lengths as in :func:`make_decode`; they count every cached key, the Lq new
    tokens' own keys included.
    """
    g = _gen(seed)
    q = randn_bf16((B, Hq, Lq, D), g)
    kc = randn_bf16((B, Hkv, Lmax, D), g)
    vc = randn_bf16((B, Hkv, Lmax, D), g)
    if kv_lens is not None and len(kv_lens) > 0:
        lens = torch.tensor(list(kv_lens), dtype=torch.int32)
    elif kv_range is None:
        lens = torch.full((B,), int(Lmax), dtype=torch.int32)
    else:
        lo, hi = kv_range
        lens = torch.randint(int(lo), int(hi) + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    return q, kc, vc, lens


def make_varlen(nseq, Hq, Hkv, D, seed, seqlens=None, seq_range=None):
    """Packed (THD) inputs: q [total,Hq,D], k/v [total,Hkv,D] bf16 and int32 cu_seqlens [nseq+1].

    Query and key lengths are equal per sequence.  ``seqlens`` fixes the
    lengths; otherwise they are drawn uniformly from the inclusive ``seq_range``.
    """
    g = _gen(seed)
    if seqlens is None:
        lo, hi = seq_range
        seqlens = torch.randint(int(lo), int(hi) + 1, (nseq,), generator=g, dtype=torch.int64).tolist()
    seqlens = [int(s) for s in seqlens]
    cu = [0]
    for s in seqlens:
        cu.append(cu[-1] + s)
    total = cu[-1]
    q = randn_bf16((total, Hq, D), g)
    k = randn_bf16((total, Hkv, D), g)
    v = randn_bf16((total, Hkv, D), g)
    return q, k, v, torch.tensor(cu, dtype=torch.int32)


def make_pages(kcache, vcache, page_size, seed, spare_pages=3, fill_unused=float("nan")):
    """Scatter a contiguous cache [B,Hkv,Lmax,D] into a page pool [num_pages,Hkv,page_size,D].

    Pages are placed at a seeded random permutation of pool slots; block_table
    [B, max_pages] (int32) lists them per sequence.  Pool pages no sequence uses,
    and rows past Lmax in the last page, hold ``fill_unused`` (NaN by default) so
    a read of them shows up in the output.
    """
    B, Hkv, Lmax, D = kcache.shape
    max_pages = (Lmax + page_size - 1) // page_size
    num_pages = B * max_pages + spare_pages
    g = _gen(seed)
    perm = torch.randperm(num_pages, generator=g)
    kp = torch.full((num_pages, Hkv, page_size, D), fill_unused, dtype=kcache.dtype)
    vp = torch.full((num_pages, Hkv, page_size, D), fill_unused, dtype=vcache.dtype)
    table = torch.empty((B, max_pages), dtype=torch.int32)
    for b in range(B):
        for i in range(max_pages):
            pid = int(perm[b * max_pages + i])
            table[b, i] = pid
            lo, hi = i * page_size, min(Lmax, (i + 1) * page_size)
            kp[pid, :, : hi - lo] = kcache[b, :, lo:hi]
            vp[pid, :, : hi - lo] = vcache[b, :, lo:hi]
    return kp, vp, table


def rope_tables(max_pos: int, D: int, base: float = 10000.0):
    """Rotary-embedding tables (model constants handed to the kernels as data): fp32 [max_pos, D/2] cosines
    and sines of the angles p * base^(-2i/D), the usual frequency ladder, evaluated in fp64."""
    inv = base ** (-torch.arange(0, D // 2, dtype=torch.float64) * 2.0 / D)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.cos(ang).float().contiguous(), torch.sin(ang).float().contiguous()
