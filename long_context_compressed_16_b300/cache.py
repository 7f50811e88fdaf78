"""Hybrid KV cache of one attention layer (B sequences advancing together).

"DeepSeek V4 模型技术大全", hybrid KV cache passage: the cache splits into
  - a state cache: the SWA window (the last n_win = 128 uncompressed rows) and the compressor
    tails (rows of blocks that have not closed yet, plus the block before them, whose second
    stream the next CSA entry still reads);
  - a classical cache: the closed CSA entries and indexer keys, or the closed HCA entries.
A prefix of P tokens is reusable up to P_closed = lcm(4, 128) floor(P / lcm) = 128 floor(P / 128);
the tail tau = P - P_closed is appended again (closed_prefix).

Every append goes through the library's csa_cache_append (compression of the entries that close,
ring and window writes, all in its kernels); this module holds the buffers and the token count.
"""
from __future__ import annotations

import math

import torch

from . import capi as C

M_CSA = 4
M_HCA = 128
N_WIN = 128
LCM = M_CSA * M_HCA // math.gcd(M_CSA, M_HCA)   # 128: common boundary of both compressors


def closed_prefix(P: int, m: int = M_CSA, m_hca: int = M_HCA) -> tuple[int, int]:
    """(P_closed, tau) for a prefix of P tokens: the longest prefix on an lcm(m, m') boundary
    (every CSA and HCA block inside it closed) and the tail that has to be recomputed."""
    if P < 0:
        raise ValueError("negative prefix length")
    step = m * m_hca // math.gcd(m, m_hca)
    closed = step * (P // step)
    return closed, P - closed


def closing_entries(t0: int, n: int, m: int) -> range:
    """Entries whose block closes while tokens t0 .. t0+n-1 are appended: entry i closes at
    token m(i+1) - 1."""
    return range(t0 // m, (t0 + n) // m)


class LayerCache:
    """kind "csa": overlapped m = 4 compressor with indexer keys (kv [B, N, d], kI [B, N, dI]);
    kind "hca": m' = 128 single-stream compressor (kv [B, N, d]).  win [B, Wcap, d] is the
    window ring csa_attend / hca_attend read (token u at slot u mod Wcap).

    params: the compressor weights as csa_cache_append takes them (bias_a, bias_b, gamma and the
    indexer's bias_a_I, bias_b_I, gamma_I), fp32 device tensors or absent."""

    def __init__(self, kind: str, B: int, n_tokens: int, d: int = 512, dI: int = 128, Wcap: int = N_WIN,
                 rope_dims: int = 64, theta: float = 160000.0, eps: float = 1e-6, norm: bool = True,
                 params: dict | None = None, device="cuda"):
        if kind not in ("csa", "hca"):
            raise ValueError("kind is 'csa' or 'hca'")
        self.kind = kind
        self.m = M_CSA if kind == "csa" else M_HCA
        self.B, self.d, self.dI = B, d, (dI if kind == "csa" else 0)
        self.cap = n_tokens
        self.t = 0
        self.params = dict(params or {})
        self.desc = C.csa_cache_desc(B=B, d=d, dI=self.dI, m=self.m, overlap=1 if kind == "csa" else 0, Wcap=Wcap,
                                     N_cap=n_tokens // self.m, rope_dims=rope_dims, rope_theta=theta,
                                     inv_freq=None, eps=eps,
                                     flags=(C.CSA_COMPRESS_NORM if norm else 0) | (C.CSA_COMPRESS_ROPE if rope_dims else 0),
                                     index_flags=C.CSA_COMPRESS_NORM if norm else 0)
        sb = C.csa_cache_state_bytes(self.desc)
        if sb == 0:
            raise ValueError("unsupported cache shape")
        dev = torch.device(device)
        N = n_tokens // self.m
        self.kv = torch.zeros((B, N, d), dtype=torch.bfloat16, device=dev)
        self.kI = torch.zeros((B, N, self.dI), dtype=torch.bfloat16, device=dev) if self.dI else None
        self.win = torch.zeros((B, Wcap, d), dtype=torch.bfloat16, device=dev)
        self.state = torch.zeros(sb, dtype=torch.uint8, device=dev)

    @property
    def n_closed(self) -> int:
        """Closed entries so far: floor(t / m)."""
        return self.t // self.m

    def append(self, rows: dict, snapshots: dict | None = None, stream=None) -> range:
        """Append the next n tokens.  rows: bf16 [B, n, width] tensors named as csa_cache_rows
        (CSA: Ca, Cb, Za, Zb, Ca_I, Cb_I, Za_I, Zb_I, win; HCA: Ca, Za, win).  With `snapshots`,
        the chunk is cut at every 128-token boundary it crosses and a checkpoint is stored there
        under its token count.  Returns the entries that closed."""
        names = (("Ca", "Cb", "Za", "Zb", "Ca_I", "Cb_I", "Za_I", "Zb_I") if self.kind == "csa" else ("Ca", "Za")) + ("win",)
        missing = [k for k in names if k not in rows]
        if missing:
            raise ValueError(f"rows missing: {missing}")
        n = rows["win"].shape[1]
        for k in names:
            r = rows[k]
            width = self.dI if k.endswith("_I") else self.d
            if (r.dtype != torch.bfloat16 or not r.is_cuda or not r.is_contiguous()
                    or tuple(r.shape) != (self.B, n, width)):
                raise ValueError(f"rows[{k!r}] must be a contiguous CUDA bf16 tensor of shape {(self.B, n, width)}")
        if self.t + n > self.cap:
            raise ValueError("cache is full")
        t_first = self.t
        bufs = {"kv": self.kv, "kI": self.kI, "win": self.win, "state": self.state}
        cuts = [n]
        if snapshots is not None:
            cuts = [b - t_first for b in range((t_first // LCM + 1) * LCM, t_first + n, LCM)] + [n]
        lo = 0
        for hi in cuts:
            part = rows if (lo, hi) == (0, n) else {k: v[:, lo:hi].contiguous() for k, v in rows.items()}
            C.check(C.csa_cache_append(self.desc, self.t, hi - lo, part, self.params, bufs, stream),
                    "csa_cache_append")
            self.t += hi - lo
            if snapshots is not None and self.t % LCM == 0:
                snapshots[self.t] = self.checkpoint()
            lo = hi
        return closing_entries(t_first, n, self.m)

    def checkpoint(self) -> dict:
        """Snapshot of the state cache at an lcm(4, 128) boundary: enough, with the classical
        entries before it, to resume appending from token t."""
        if self.t % LCM:
            raise ValueError("checkpoints sit on 128-token boundaries")
        return {"t": self.t, "state": self.state.clone(), "win": self.win.clone()}

    @classmethod
    def from_prefix(cls, source: "LayerCache", P: int, snapshots: dict) -> tuple["LayerCache", int]:
        """A cache of source's first P_closed tokens (closed entries copied, state restored from
        the snapshot taken at P_closed); returns it with tau, the tail the caller appends again."""
        closed, tau = closed_prefix(P)
        if closed > source.t:
            raise ValueError("the prefix is longer than the source cache")
        c = cls.__new__(cls)
        c.__dict__.update({k: v for k, v in source.__dict__.items()
                           if k not in ("kv", "kI", "win", "state", "t")})
        c.kv = torch.zeros_like(source.kv)
        c.kI = torch.zeros_like(source.kI) if source.kI is not None else None
        c.win = torch.zeros_like(source.win)
        c.state = torch.zeros_like(source.state)
        if closed:
            snap = snapshots[closed]
            nc = closed // source.m
            c.kv[:, :nc].copy_(source.kv[:, :nc])
            if c.kI is not None:
                c.kI[:, :nc].copy_(source.kI[:, :nc])
            c.state.copy_(snap["state"])
            c.win.copy_(snap["win"])
        c.t = closed
        return c, tau
