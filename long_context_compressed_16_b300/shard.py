"""Multi-rank partition of the compressed-attention path (one process per GPU).

Decode shards the batch: sequences are independent, so rank r owns a contiguous range of them
and there is no exchange on the data path.

Prefill shards the chunk's tokens into contiguous ranges (context parallelism, "DeepSeek-V4"
technical-report pages, the long-context parallelism section).  Range boundaries fall on multiples
of `align` (128 = lcm of the CSA block m = 4 and the HCA block m' = 128), so no compressed block
straddles two ranks.  Two exchanges make every later step local:

  1. halo, point to point from rank r-1 to rank r:
       - the last m rows of the overlapped compressor's second stream (C^b, Z^b): rank r's first
         entry mixes its own first block of C^a/Z^a with the previous block of C^b/Z^b;
       - the last window-1 per-token window rows: rank r's first queries attend to them.
  2. all-gather of the compressed entries (attention cache and indexer keys), T/m rows in all.

After that, scoring, top-k and attention for a rank's own queries need only its own rows.

The arithmetic stays in the caller's per-rank functions (the library's CUDA calls on a GPU);
this module holds only the index arithmetic and the torch.distributed exchanges.  With the halo
prepended, a rank's compressor call sees exactly the rows a single-rank call would see for each
of its entries, so the partitioned result equals the single-rank one entry by entry.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.distributed as dist

ALIGN = 128


def batch_range(B: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous share [lo, hi) of B independent sequences for `rank`; sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world or B < 0:
        raise ValueError(f"bad partition: B={B} world={world} rank={rank}")
    return (B * rank) // world, (B * (rank + 1)) // world


@dataclass(frozen=True)
class TokenRange:
    lo: int            # first token position owned by the rank
    hi: int            # one past the last
    halo_b: int        # rows of C^b/Z^b received from rank-1 (m for CSA, 0 on rank 0)
    halo_win: int      # window rows received from rank-1 (window-1, clipped at lo)

    @property
    def tokens(self) -> int:
        return self.hi - self.lo


def token_range(T: int, world: int, rank: int, m: int, window: int, align: int = ALIGN) -> TokenRange:
    """Rank `rank`'s tokens of a T-token chunk: whole `align`-blocks, split as evenly as possible.

    Every rank must own at least one block, and the previous rank at least window-1 tokens so the
    window halo comes from one neighbour; both hold when T >= world * align and window <= align + 1."""
    if T % align or align % m:
        raise ValueError(f"T={T} and align={align} must be multiples of m={m} and align respectively")
    nb = T // align
    if nb < world:
        raise ValueError(f"T={T} gives {nb} blocks of {align} tokens for {world} ranks")
    if window - 1 > align:
        raise ValueError(f"window={window} needs a halo longer than one {align}-token block")
    lo = align * ((nb * rank) // world)
    hi = align * ((nb * (rank + 1)) // world)
    return TokenRange(lo, hi, m if rank > 0 else 0, min(window - 1, lo))


def _send_tail(t: torch.Tensor, rows: int, dst: int, group=None) -> None:
    dist.send(t[:, t.shape[1] - rows:].contiguous(), dst, group=group)


def _recv(shape, dtype, src: int, group=None) -> torch.Tensor:
    buf = torch.empty(shape, dtype=dtype)
    dist.recv(buf, src, group=group)
    return buf


def halo_exchange(r: TokenRange, streams: dict, rows_of: dict, group=None) -> dict:
    """Exchange 1.  streams: name -> this rank's [B, tokens, ...] CPU tensor; rows_of: name -> how
    many trailing rows the next rank needs.  Returns name -> [B, rows, ...] received from rank-1
    (zero rows on rank 0).  Sends go to rank+1 first (even ranks) or after receiving (odd ranks),
    so the blocking point-to-point calls pair up without a cycle."""
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    recvd = {}

    def do_recv():
        for name in sorted(streams):
            t = streams[name]
            rows = rows_of[name] if rank > 0 else 0
            shape = (t.shape[0], rows) + tuple(t.shape[2:])
            recvd[name] = _recv(shape, t.dtype, rank - 1, group) if rows else t.new_empty(shape)

    def do_send():
        if rank + 1 < world:
            for name in sorted(streams):
                if rows_of[name]:
                    if streams[name].shape[1] < rows_of[name]:
                        raise ValueError(f"{name}: rank {rank} holds {streams[name].shape[1]} rows, "
                                         f"the next rank needs {rows_of[name]}")
                    _send_tail(streams[name], rows_of[name], rank + 1, group)

    if rank % 2 == 0:
        do_send()
        do_recv()
    else:
        do_recv()
        do_send()
    return recvd


def allgather_rows(local: torch.Tensor, group=None) -> torch.Tensor:
    """Exchange 2.  Concatenate every rank's [B, n_r, ...] rows along dim 1 in rank order (the
    ranks' n_r may differ; shorter ones are padded for the collective and trimmed after)."""
    world = dist.get_world_size(group)
    n = torch.tensor([local.shape[1]], dtype=torch.int64)
    counts = [torch.zeros_like(n) for _ in range(world)]
    dist.all_gather(counts, n, group=group)
    counts = [int(c) for c in counts]
    nmax = max(counts)
    pad = local.new_zeros((local.shape[0], nmax) + tuple(local.shape[2:]))
    pad[:, :local.shape[1]] = local
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad.contiguous(), group=group)
    return torch.cat([p[:, :c] for p, c in zip(parts, counts)], dim=1)


def with_b_halo(r: TokenRange, m: int, Ca, Za, Cb, Zb, halo_Cb, halo_Zb):
    """Compressor inputs of rank r with the b-stream halo block prepended.

    Returns (Ca, Za, Cb, Zb, pos_shift, drop): compress these rows with RoPE position
    m*i + pos_shift for local entry i, then drop the first `drop` entries.  The prepended block's
    own a-stream rows are zeros: they feed only the dropped entry."""
    if r.halo_b == 0:
        return Ca, Za, Cb, Zb, r.lo, 0
    if halo_Cb.shape[1] != m or halo_Zb.shape[1] != m:
        raise ValueError("the b-stream halo must hold exactly one block of m rows")
    z = Ca.new_zeros((Ca.shape[0], m) + tuple(Ca.shape[2:]))
    cat = lambda h, x: torch.cat([h, x], dim=1)
    return cat(z, Ca), cat(z, Za), cat(halo_Cb, Cb), cat(halo_Zb, Zb), r.lo - m, 1


def window_ring(r: TokenRange, halo_win: torch.Tensor, own_win: torch.Tensor):
    """Per-token window rows for positions [lo - halo_win, hi) as a ring indexed by position mod
    Wcap (the layout the attention call reads), with Wcap = hi - lo + halo_win so no two of
    those positions share a slot.  Returns (ring [B, Wcap, d], Wcap)."""
    rows = torch.cat([halo_win, own_win], dim=1)
    Wcap = rows.shape[1]
    first = r.lo - halo_win.shape[1]
    slots = (torch.arange(first, r.hi) % Wcap).tolist()
    ring = torch.empty_like(rows)
    ring[:, slots] = rows
    return ring, Wcap
