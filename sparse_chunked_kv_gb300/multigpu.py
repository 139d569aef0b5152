"""Host logic of the multi-GPU split of the path (one process per GPU).

Prefill ("Chunked Prefill and KV Caching": chunks are processed
independently) shards by chunk range: rank r prefills the chunks of its
range into its own pool and table, with no exchange.  Decode ("Attention
Kernel Optimization": the KV dimension is partitioned, parts processed
independently, merged by log-sum-exp) needs one exchange: every rank
computes the partial state (pfd_decode_partial) of the selected chunks that
live in its pool -- the live block's keys only on the owner -- the partials
are gathered to the owner, and the owner merges them (pfd_lse_merge).

This module holds the bookkeeping and the gather; every computation runs in
libpfd's kernels.  Nothing here is on the single-GPU path.
"""
from __future__ import annotations

OWNER = 0   # the rank that holds the live block and merges


def chunk_range(n_chunks: int, rank: int, world: int) -> tuple:
    """Rank's contiguous range [lo, hi) of a sequence's n_chunks chunks (the
    first n_chunks % world ranks hold one more)."""
    base, extra = divmod(n_chunks, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def owner_of(chunk: int, n_chunks: int, world: int) -> int:
    """The rank whose prefill range holds in-sequence chunk `chunk`."""
    for r in range(world):
        lo, hi = chunk_range(n_chunks, r, world)
        if lo <= chunk < hi:
            return r
    raise ValueError(f"chunk {chunk} outside [0, {n_chunks})")


def local_selection(sel, cu_k, cu_n, rank: int, world: int) -> tuple:
    """The selected chunks rank must attend to, per sequence, in selection
    order.  sel holds table indices (sequence b's chunks are table entries
    cu_n[b] .. cu_n[b+1]-1, its selection sel[cu_k[b] .. cu_k[b+1]-1]).
    Returns (sel_local, cu_k_local) as Python lists; the union over ranks is
    sel, each entry on exactly one rank."""
    sel = [int(x) for x in sel]
    out, cu_out = [], [0]
    for b in range(len(cu_k) - 1):
        n_b = int(cu_n[b + 1]) - int(cu_n[b])
        for c in sel[int(cu_k[b]):int(cu_k[b + 1])]:
            if owner_of(c - int(cu_n[b]), n_b, world) == rank:
                out.append(c)
        cu_out.append(len(out))
    return out, cu_out


def self_keys_on(rank: int) -> int:
    """1 on the rank whose partial includes the live block's keys."""
    return 1 if rank == OWNER else 0


def gather_partials(part_o, part_lse, world: int, group=None):
    """All-gathers every rank's partial (o [rows, Hq, D], lse [rows, Hq])
    into [world, rows, Hq, D] and [world, rows, Hq], rank order: the layout
    pfd_lse_merge takes (n_parts = world).  One collective per tensor; the
    owner merges, the other ranks may drop the result."""
    import torch
    import torch.distributed as dist
    o_all = torch.empty((world,) + tuple(part_o.shape), dtype=part_o.dtype, device=part_o.device)
    l_all = torch.empty((world,) + tuple(part_lse.shape), dtype=part_lse.dtype,
                        device=part_lse.device)
    # list form: works on every backend (NCCL on GPUs, gloo on CPU)
    dist.all_gather(list(o_all.unbind(0)), part_o.contiguous(), group=group)
    dist.all_gather(list(l_all.unbind(0)), part_lse.contiguous(), group=group)
    return o_all, l_all
