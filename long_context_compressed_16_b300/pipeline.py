"""Tensor-level calls over the C ABI: allocate outputs and workspaces with torch, fill the
descriptors, call libcsa.so, raise CsaError on a non-zero status.  All arithmetic happens in
the library's CUDA kernels."""
from __future__ import annotations

import torch

from . import capi as C


def _dev_check(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("inputs must be contiguous CUDA tensors")


def _ws(nbytes: int, device) -> torch.Tensor:
    # zero-filled: the status word at its start must begin cleared (it is sticky)
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def compress(Ca, Za, m, Cb=None, Zb=None, bias_a=None, bias_b=None, gamma=None, norm=True, rope=True,
             rope_dims=64, theta=160000.0, inv_freq=None, pos_shift=0, eps=1e-6, out=None, stream=None):
    """Token-level compressor (CSA when Cb/Zb are given, HCA otherwise). Returns bf16 [B, T//m, d]."""
    _dev_check(Ca, Za, Cb, Zb, bias_a, bias_b, gamma)
    B, T, d = Ca.shape
    N = T // m
    if out is None:
        out = torch.empty((B, N, d), dtype=torch.bfloat16, device=Ca.device)
    tab = C.float_table(inv_freq)
    desc = C.csa_compress_desc(B=B, T=T, d=d, m=m, overlap=1 if Cb is not None else 0, rope_dims=rope_dims,
                               rope_theta=theta, inv_freq=tab, pos_shift=pos_shift, eps=eps,
                               flags=(C.CSA_COMPRESS_NORM if norm else 0) | (C.CSA_COMPRESS_ROPE if rope else 0),
                               out_fmt=C.CSA_FMT_BF16)
    C.check(C.csa_compress(desc, Ca, Cb, Za, Zb, bias_a, bias_b, gamma, out, stream), "csa_compress")
    return out


def index_desc(B, Tq, N, nI, dI, k, m, fp8=False, lowp=False, bf16_scores=False, select_mode=0):
    """select_mode: C.CSA_SELECT_AUTO (0), C.CSA_SELECT_FUSED or C.CSA_SELECT_STORED."""
    fmt = C.CSA_FMT_FP8_ROWSCALE_LOWP if lowp else (C.CSA_FMT_FP8_ROWSCALE if fp8 else C.CSA_FMT_BF16)
    return C.csa_index_desc(B=B, Tq=Tq, N=N, n_heads=nI, head_dim=dI, k=k, m=m, key_fmt=fmt,
                            score_fmt=C.CSA_SCORE_BF16 if bf16_scores else C.CSA_SCORE_FP32,
                            select_mode=select_mode)


def index_topk(qI, w, kI, q_pos, m, k, kI_scale=None, score_out=None, idx_out=None, workspace=None,
               stream=None, lowp=False, bf16_scores=False, select_mode=0):
    """Lightning-indexer scores + per-query top-k. Returns int32 [B, Tq, k] (-1 padded).
    lowp: the low-precision indexer (FP8 keys with kI_scale, the query quantised to e4m3).
    bf16_scores: scores rounded to bf16 before the selection.
    select_mode: where the selection runs (same result): C.CSA_SELECT_AUTO, _FUSED or _STORED."""
    _dev_check(qI, w, kI, q_pos, kI_scale, score_out)
    B, Tq, nI, dI = qI.shape
    N = kI.shape[1]
    if lowp and kI_scale is None:
        raise ValueError("the low-precision indexer takes e4m3 keys with row scales")
    desc = index_desc(B, Tq, N, nI, dI, k, m, fp8=kI_scale is not None, lowp=lowp, bf16_scores=bf16_scores,
                      select_mode=select_mode)
    if idx_out is None:
        idx_out = torch.empty((B, Tq, k), dtype=torch.int32, device=qI.device)
    if workspace is None:
        workspace = _ws(C.csa_index_topk_workspace(desc), qI.device)
    C.check(C.csa_index_topk(desc, qI, w, kI, kI_scale, q_pos, idx_out, score_out, workspace, stream=stream),
            "csa_index_topk")
    return idx_out


def attend_desc(B, Tq, N, H, d, k=0, m=1, Wcap=128, window=128, rope_dims=64, theta=160000.0, scale=0.0,
                eps=1e-6, fp8=False, q_norm_rope=True, out_unrotate=True, write_lse=False, inv_freq_tab=None):
    flags = ((C.CSA_ATTEND_Q_NORM_ROPE if q_norm_rope else 0) | (C.CSA_ATTEND_OUT_UNROTATE if out_unrotate else 0)
             | (C.CSA_ATTEND_WRITE_LSE if write_lse else 0))
    return C.csa_attend_desc(B=B, Tq=Tq, N=N, H=H, d=d, rope_dims=rope_dims, k=k, m=m, Wcap=Wcap, window=window,
                             scale=scale, rope_theta=theta, inv_freq=inv_freq_tab, eps=eps,
                             kv_fmt=C.CSA_FMT_FP8_MIXED if fp8 else C.CSA_FMT_BF16, flags=flags)


def _attend(csa_mode, q, kv, idx, win, sink, q_pos, m, window, rope_dims, theta, scale, fp8, q_norm_rope,
            out_unrotate, want_lse, inv_freq, out, lse, workspace, stream, d_model=None):
    _dev_check(q, kv, idx, win, sink, q_pos)
    B, Tq, H, d = q.shape
    N = kv.shape[1]
    Wcap = win.shape[1]
    tab = C.float_table(inv_freq)
    desc = attend_desc(B, Tq, N, H, d, k=idx.shape[2] if csa_mode else 0, m=m, Wcap=Wcap, window=window,
                       rope_dims=rope_dims, theta=theta, scale=scale, fp8=fp8, q_norm_rope=q_norm_rope,
                       out_unrotate=out_unrotate, write_lse=want_lse, inv_freq_tab=tab)
    if out is None:
        out = torch.empty((B, Tq, H, d), dtype=torch.bfloat16, device=q.device)
    if want_lse and lse is None:
        lse = torch.empty((B, Tq, H), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _ws(C.csa_attend_workspace(desc) if csa_mode else C.hca_attend_workspace(desc), q.device)
    if csa_mode:
        st = C.csa_attend(desc, q, kv, idx, win, sink, q_pos, out, lse, workspace, stream=stream)
    else:
        st = C.hca_attend(desc, q, kv, win, sink, q_pos, out, lse, workspace, stream=stream)
    C.check(st, "csa_attend" if csa_mode else "hca_attend")
    return out, lse, workspace


def csa_attend(q, kv, idx, win, sink, q_pos, window=128, rope_dims=64, theta=160000.0, scale=0.0, fp8=False,
               q_norm_rope=True, out_unrotate=True, want_lse=False, inv_freq=None, out=None, lse=None,
               workspace=None, stream=None):
    """Sparse shared-KV attention over idx rows + window + sink. Returns (out bf16, lse|None, workspace)."""
    return _attend(True, q, kv, idx, win, sink, q_pos, 1, window, rope_dims, theta, scale, fp8, q_norm_rope,
                   out_unrotate, want_lse, inv_freq, out, lse, workspace, stream)


def hca_attend(q, kv, win, sink, q_pos, m=128, window=128, rope_dims=64, theta=160000.0, scale=0.0, fp8=False,
               q_norm_rope=True, out_unrotate=True, want_lse=False, inv_freq=None, out=None, lse=None,
               workspace=None, stream=None):
    """Dense shared-KV attention over all closed entries + window + sink."""
    return _attend(False, q, kv, None, win, sink, q_pos, m, window, rope_dims, theta, scale, fp8, q_norm_rope,
                   out_unrotate, want_lse, inv_freq, out, lse, workspace, stream)


def out_proj(O, W_down, groups, W_proj=None, z=None, y=None, workspace=None, stream=None):
    """Grouped output projection.  O: bf16 [T, n_heads, head_dim] (or [B, Tq, H, d]);
    W_down: bf16 [groups, rank, (n_heads/groups) head_dim]; W_proj: bf16 [d_out, groups rank] or
    None.  Returns (z [T, groups rank], y [T, d_out] or None)."""
    _dev_check(O, W_down, W_proj, z, y)
    H, d = O.shape[-2], O.shape[-1]
    T = O.numel() // (H * d)
    G, rank, K = W_down.shape
    d_out = 0 if W_proj is None else W_proj.shape[0]
    # the library takes plain pointers: every extent it reads or writes is checked here
    if any(t is not None and t.dtype != torch.bfloat16 for t in (O, W_down, W_proj, z, y)):
        raise ValueError("out_proj takes bf16 tensors")
    if G != groups or H % G != 0 or K != (H // G) * d:
        raise ValueError(f"W_down must be [groups, rank, (n_heads/groups) head_dim] = [{groups}, r, {H // max(groups, 1) * d}]")
    if W_proj is not None and tuple(W_proj.shape) != (d_out, G * rank):
        raise ValueError(f"W_proj must be [d_out, groups rank] = [d_out, {G * rank}]")
    if z is not None and tuple(z.shape) != (T, G * rank):
        raise ValueError(f"z must be [{T}, {G * rank}]")
    if y is not None and d_out and tuple(y.shape) != (T, d_out):
        raise ValueError(f"y must be [{T}, {d_out}]")
    desc = C.csa_out_proj_desc(T=T, n_heads=H, head_dim=d, groups=G, rank=rank, d_out=d_out)
    if z is None:
        z = torch.empty((T, G * rank), dtype=torch.bfloat16, device=O.device)
    if y is None and d_out:
        y = torch.empty((T, d_out), dtype=torch.bfloat16, device=O.device)
    if workspace is None:
        n = C.csa_out_proj_workspace(desc)
        if n == 0:
            raise C.CsaError(C.CSA_ERR_UNSUPPORTED, "csa_out_proj")
        workspace = _ws(n, O.device)
    C.check(C.csa_out_proj(desc, O, W_down, W_proj, z, y, workspace, stream=stream), "csa_out_proj")
    return z, y
