"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the method: it only draws random numbers,
lays them out in the paged cache format and builds block tables.  Both the CUDA
path and the CPU oracle are fed from here; neither imports the other.

Recipe (stated once, used everywhere):
  * generator: ``torch.Generator('cpu').manual_seed(seed)``;
  * q, K, V, query windows: N(0, 1) drawn in fp32, then cast to the workload
    dtype (the oracle reads the cast values, upcast exactly to fp32);
  * sequence lengths: uniform integers in [lo, hi] unless given;
  * physical blocks: a seeded permutation of the pool, so a sequence's pages
    are scattered, never contiguous;
  * block tables: int32 [B][table_stride], unused entries = -1.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch

DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}


@dataclasses.dataclass
class PagedCase:
    """One layer (or several) of a paged cache plus the sequences living in it."""

    h_q: int
    h_kv: int
    d: int
    b: int
    dtype: str
    n_total: int               # blocks in the pool
    seq_lens: torch.Tensor     # int32 [B]
    block_table: torch.Tensor  # int32 [B][table_stride]
    k_cache: torch.Tensor      # [layers][N_total][b][h_kv][d] (dtype)
    v_cache: torch.Tensor      # same
    q: torch.Tensor            # [B][h_q][d] (dtype)
    free_blocks: torch.Tensor  # int32: pool blocks not referenced by any table
    ref: torch.Tensor          # int32 [N_total]: references per block
    layers: int = 1

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def table_stride(self) -> int:
        return int(self.block_table.shape[1])


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, seed_or_gen, dtype: str = "f32") -> torch.Tensor:
    g = _gen(seed_or_gen) if isinstance(seed_or_gen, int) else seed_or_gen
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    return x.to(DTYPES[dtype])


def make_paged_case(seed: int, B: int, h_q: int, h_kv: int, d: int, b: int,
                    lens: Optional[Sequence[int]] = None, len_range=(1, 64),
                    dtype: str = "f32", spare_blocks: int = 0,
                    table_stride: Optional[int] = None, layers: int = 1,
                    shared_prefix_blocks: int = 0, device=None) -> PagedCase:
    """Random paged cache with ``B`` sequences.

    ``shared_prefix_blocks`` > 0 makes every sequence start with the same
    physical blocks (a shared prompt prefix, reference count B); each sequence
    then needs at least that many full blocks of its own length.
    ``device``: draw K, V and q there (a torch generator of that device seeded
    from ``seed``) instead of on the host -- for caches of several GB; lengths,
    tables and the free list are drawn on the host as always.
    """
    g = _gen(seed)
    if lens is None:
        lo, hi = len_range
        seq_lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    else:
        seq_lens = torch.as_tensor(list(lens), dtype=torch.int64)
        assert seq_lens.numel() == B
    n_blocks = (seq_lens + b - 1) // b
    P = int(shared_prefix_blocks)
    if P:
        assert int(seq_lens.min()) >= P * b, "every sequence must cover the shared prefix"
    own = n_blocks - P
    n_total = int(own.sum()) + P + int(spare_blocks)
    stride = int(table_stride) if table_stride is not None else max(int(n_blocks.max()), 1)
    assert stride >= int(n_blocks.max())
    perm = torch.randperm(n_total, generator=g).to(torch.int32)
    table = torch.full((B, stride), -1, dtype=torch.int32)
    ref = torch.zeros(n_total, dtype=torch.int32)
    cursor = 0
    prefix = perm[cursor:cursor + P]
    cursor += P
    for s in range(B):
        nb = int(n_blocks[s])
        if P:
            table[s, :P] = prefix
        m = nb - P
        table[s, P:nb] = perm[cursor:cursor + m]
        cursor += m
        ref[table[s, :nb].long()] += 1
    free = perm[cursor:].clone()
    dt = DTYPES[dtype]
    if device is not None:
        gd = torch.Generator(device=device).manual_seed(seed + 0x5EED)
        k = torch.empty(layers, n_total, b, h_kv, d, dtype=dt, device=device)
        v = torch.empty(layers, n_total, b, h_kv, d, dtype=dt, device=device)
        for arr in (k, v):  # layer by layer: no fp32 copy of the whole cache
            for layer in range(layers):
                arr[layer].copy_(torch.randn(n_total, b, h_kv, d, generator=gd, device=device))
        q = torch.randn(B, h_q, d, generator=gd, device=device)
        return PagedCase(h_q=h_q, h_kv=h_kv, d=d, b=b, dtype=dtype, n_total=n_total,
                         seq_lens=seq_lens.to(torch.int32), block_table=table,
                         k_cache=k, v_cache=v, q=q.to(dt), free_blocks=free, ref=ref, layers=layers)
    k = torch.randn(layers, n_total, b, h_kv, d, generator=g, dtype=torch.float32)
    v = torch.randn(layers, n_total, b, h_kv, d, generator=g, dtype=torch.float32)
    q = torch.randn(B, h_q, d, generator=g, dtype=torch.float32)
    return PagedCase(h_q=h_q, h_kv=h_kv, d=d, b=b, dtype=dtype, n_total=n_total,
                     seq_lens=seq_lens.to(torch.int32), block_table=table,
                     k_cache=k.to(dt), v_cache=v.to(dt), q=q.to(dt), free_blocks=free,
                     ref=ref, layers=layers)


def plant_duplicates(case: PagedCase, seed: int, frac: float = 0.1, noise: float = 0.05,
                     layer: int = 0) -> None:
    """Make about ``frac`` of the keys near-copies of an earlier key of the same block.

    For a chosen token t at slot j > 0 of its block, k_t <- k_{t-delta} + noise*eps
    with delta uniform in [1, j], so the pair falls inside one block.  Gaussian
    keys at d = 128 are nearly orthogonal; this gives the redundancy score pairs
    above its threshold.
    """
    g = _gen(seed)
    K = case.k_cache[layer].float()
    for s in range(case.B):
        L = int(case.seq_lens[s])
        pick = torch.rand(L, generator=g) < frac
        for t in torch.nonzero(pick).flatten().tolist():
            j = t % case.b
            if j == 0:
                continue
            delta = int(torch.randint(1, j + 1, (1,), generator=g))
            src = t - delta
            bt, bs = int(case.block_table[s, t // case.b]), t % case.b
            st, ss = int(case.block_table[s, src // case.b]), src % case.b
            eps = torch.randn(case.h_kv, case.d, generator=g)
            K[bt, bs] = K[st, ss] + noise * eps
    case.k_cache[layer] = K.to(case.k_cache.dtype)


def gather_tokens(cache_layer: torch.Tensor, table_row: torch.Tensor, L: int, b: int) -> torch.Tensor:
    """Logical view [L][h_kv][d] of one sequence's rows of a paged cache layer."""
    t = torch.arange(L)
    blocks = table_row[(t // b)].long()
    return cache_layer[blocks, t % b]
