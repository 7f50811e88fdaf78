"""Oracle for DeepSeek-V4 hybrid compressed attention (CSA / HCA) -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 NumPy restatement of what the method computes, written from the
equations of "DeepSeek V4 模型技术大全" (wineandchord.com), chapter "Hybrid Attention":
the CSA compressor (the overlapped-softmax equations), the lightning indexer and
top-k (the I_{t,s} and TopK equations), the HCA compressor and visibility set, the
attention sink, the SWA window set and the partial-RoPE / RMSNorm table rows.

Only the test suite, the package's smoke check and the benchmark's CPU-baseline leg
may import this module.  It shares no code with the CUDA library: it decodes bf16
and e4m3 bytes with its own routines and uses NumPy matmul / sort as its only
library primitives.  Readings of points the pages leave open are stated at each
function (numbered R1..R19; the same numbers are used in the design notes).

Parity pins: every function here is pinned by the CPU tests (tests/test_oracle.py)
against closed forms, invariants, brute force and the pages' own worked numbers.
"""
from __future__ import annotations

import math

import numpy as np

# ------------------------------------------------------------------------------------------------
# storage decoding (own implementations, from the format definitions)
# ------------------------------------------------------------------------------------------------


def bf16_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16/int16 array) -> fp64. bf16 is the top half of an IEEE fp32."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def bf16_round(x) -> np.ndarray:
    """fp64 -> bf16 bit patterns (uint16): RNE to fp32, then RNE to 8 significant bits.
    Used when the oracle itself stores a compressed cache in bf16 for a later step."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return (r & np.uint64(0xFFFF)).astype(np.uint16)


def e4m3_to_f64(codes) -> np.ndarray:
    """OCP FP8 E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0 is subnormal
    (f/8 * 2^-6); S.1111.111 is NaN; no infinities.  Largest finite 448."""
    c = np.asarray(codes).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    f = c & 7
    mag = np.where(e == 0, (f / 8.0) * 2.0 ** -6, (1.0 + f / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (f == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def fp8_mixed_row_to_f64(rows) -> np.ndarray:
    """Decode mixed-precision cache rows (uint8 [..., 608]) -> fp64 [..., 512].
    Layout (the cache stores the RoPE dims in BF16 and the rest in FP8): bytes [0,448)
    e4m3 codes of dims 0..447, bytes [448,576) bf16 of dims 448..511, bytes [576,604)
    seven fp32 scales, one per 64-dim block of the e4m3 part; value = code * scale."""
    r = np.asarray(rows, dtype=np.uint8)
    lead = r.shape[:-1]
    r2 = r.reshape(-1, 608)
    codes = e4m3_to_f64(r2[:, :448]).reshape(-1, 7, 64)
    scales = np.ascontiguousarray(r2[:, 576:604]).view(np.float32).astype(np.float64).reshape(-1, 7, 1)
    nope = (codes * scales).reshape(-1, 448)
    rope = bf16_to_f64(np.ascontiguousarray(r2[:, 448:576]).view(np.uint16))
    return np.concatenate([nope, rope], axis=1).reshape(*lead, 512)


# ------------------------------------------------------------------------------------------------
# normalisation and rotation
# ------------------------------------------------------------------------------------------------


def rmsnorm(x, eps=1e-6, gamma=None):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gamma   (eps 1e-6 per the config
    table 'RMSNorm eps').  gamma=None means unit weight (R4)."""
    x = np.asarray(x, dtype=np.float64)
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    if gamma is not None:
        y = y * np.asarray(gamma, dtype=np.float64)
    return y


def rope_inv_freq(theta: float, rope_dims: int) -> np.ndarray:
    """inv_freq_i = theta^(-2i/r), i < r/2: the original rotary definition (R7)."""
    i = np.arange(rope_dims // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / rope_dims)


def rope(x, pos, inv_freq, rope_dims=64):
    """Partial RoPE: rotate the last r dims of x by angle pos*inv_freq_i on adjacent pairs
    (2i, 2i+1) of that slice (R7); the config table gives r = 64 of d = 512.  pos may be a scalar or
    broadcast against x's leading axes; a negative pos is the reverse rotation."""
    x = np.array(x, dtype=np.float64, copy=True)
    if rope_dims == 0:
        return x
    d = x.shape[-1]
    assert 0 < rope_dims <= d and rope_dims % 2 == 0
    sl = x[..., d - rope_dims:]
    ev = sl[..., 0::2].copy()
    od = sl[..., 1::2].copy()
    ang = np.asarray(pos, dtype=np.float64)[..., None] * np.asarray(inv_freq, dtype=np.float64)
    c, s = np.cos(ang), np.sin(ang)
    sl[..., 0::2] = ev * c - od * s
    sl[..., 1::2] = ev * s + od * c
    x[..., d - rope_dims:] = sl
    return x


# ------------------------------------------------------------------------------------------------
# compressor (CSA overlapped, HCA single-stream)
# ------------------------------------------------------------------------------------------------


def compress(Ca, Za, m, Cb=None, Zb=None, bias_a=None, bias_b=None, gamma=None, norm=True,
             rope_on=True, rope_dims=64, theta=160000.0, inv_freq=None, pos_shift=0, eps=1e-6):
    """Token-level compressor.

    CSA (Cb, Zb given; overlapped 2m rows): for entry i, per channel, softmax over the 2m logits
    [Z^a_{mi..m(i+1)-1} + B^a ; Z^b_{m(i-1)..mi-1} + B^b] weights the matching rows of C^a / C^b and
    the weighted rows are summed (the Softmax_row / C^Comp equations of the CSA path).
    HCA (Cb=None): softmax over the m' rows Z_{m'i..m'(i+1)-1} + B weighting C (the HCA equation).
    R1: Softmax_row normalises each channel separately over the token rows.
    R2: entry 0 has no block -1; its softmax runs over the m 'a' logits only.
    R3: B^a, B^b, B are [m, d] inputs indexed by the row's offset inside its block; None = 0.
    Then (R4/R5/R6) RMSNorm with weight gamma (None = 1) and RoPE at position m*i + pos_shift on
    the last rope_dims dims, base theta (compressed-branch base 160000).

    Inputs fp64 [B, T, d]; returns fp64 [B, N, d] with N = floor(T/m) (closed blocks only)."""
    Ca = np.asarray(Ca, dtype=np.float64)
    Za = np.asarray(Za, dtype=np.float64)
    B, T, d = Ca.shape
    N = T // m
    overlap = Cb is not None
    ba = np.zeros((m, d)) if bias_a is None else np.asarray(bias_a, dtype=np.float64)
    bb = np.zeros((m, d)) if bias_b is None else np.asarray(bias_b, dtype=np.float64)
    out = np.empty((B, N, d))
    for i in range(N):
        logits = [Za[:, m * i:m * (i + 1), :] + ba]
        values = [Ca[:, m * i:m * (i + 1), :]]
        if overlap and i >= 1:
            logits.append(np.asarray(Zb[:, m * (i - 1):m * i, :], dtype=np.float64) + bb)
            values.append(np.asarray(Cb[:, m * (i - 1):m * i, :], dtype=np.float64))
        L = np.concatenate(logits, axis=1)               # [B, rows, d]
        V = np.concatenate(values, axis=1)
        e = np.exp(L - L.max(axis=1, keepdims=True))
        S = e / e.sum(axis=1, keepdims=True)             # per-channel softmax over the rows
        out[:, i, :] = (S * V).sum(axis=1)
    if norm:
        out = rmsnorm(out, eps, gamma)
    elif gamma is not None:
        out = out * np.asarray(gamma, dtype=np.float64)
    if rope_on and rope_dims > 0:
        f = rope_inv_freq(theta, rope_dims) if inv_freq is None else np.asarray(inv_freq, np.float64)
        pos = (m * np.arange(N) + pos_shift).astype(np.float64)
        out = rope(out, pos[None, :], f, rope_dims)
    return out


# ------------------------------------------------------------------------------------------------
# lightning indexer and top-k
# ------------------------------------------------------------------------------------------------


def n_visible(t: int, m: int, N: int) -> int:
    """Closed compressed blocks visible to query position t: s < floor((t+1)/m), capped at N."""
    return max(0, min(N, (int(t) + 1) // m))


def index_scores(qI, w, kI, q_pos, m):
    """Lightning-indexer score I_{t,s} = sum_h w_{t,h} * ReLU(q^I_{t,h} . K^I_s) for s < floor((t+1)/m).
    R13: no scale and no rotation on q^I / K^I inside the score.

    qI fp64 [B, Tq, nI, dI], w [B, Tq, nI], kI fp64 [B, N, dI] (already dequantised), q_pos [B, Tq].
    Returns fp64 [B, Tq, N]; invisible entries are -inf."""
    qI = np.asarray(qI, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    kI = np.asarray(kI, dtype=np.float64)
    B, Tq = qI.shape[:2]
    N = kI.shape[1]
    out = np.full((B, Tq, N), -np.inf)
    for b in range(B):
        for t in range(Tq):
            nv = n_visible(q_pos[b][t], m, N)
            if nv == 0:
                continue
            dots = kI[b, :nv] @ qI[b, t].T               # [nv, nI]
            out[b, t, :nv] = np.maximum(dots, 0.0) @ w[b, t]
    return out


def e4m3_encode_rne(x32) -> np.ndarray:
    """fp32 values -> OCP FP8 E4M3 codes (uint8): round to nearest, ties to even, saturating to
    +-448 (the largest finite code); finite input never becomes NaN.  Written from the format
    definition: normals (1 + f/8) 2^(e-7) for e = 1..15 (S.1111.111 excluded), subnormals
    (f/8) 2^-6."""
    x = np.asarray(x32, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x)
    v = np.abs(x)
    out = np.zeros(v.shape, dtype=np.int64)
    sub = v < 2.0 ** -6
    # subnormal range: units of 2^-9; rounding up to 8 units gives the smallest normal (code 8)
    out = np.where(sub, np.rint(v / 2.0 ** -9).astype(np.int64), out)
    vn = np.where(sub, 1.0, v)
    mant, ex = np.frexp(vn)                        # vn = mant * 2^ex, mant in [0.5, 1)
    e = ex - 1                                     # vn = (2 mant) 2^e, 2 mant in [1, 2)
    f = np.rint((2.0 * mant - 1.0) * 8.0).astype(np.int64)
    e = np.where(f == 8, e + 1, e)
    f = np.where(f == 8, 0, f)
    code = (e + 7) * 8 + f
    code = np.where(code > 0x7E, 0x7E, code)       # above 448 (or onto the NaN pattern): 448
    out = np.where(sub, out, code)
    return (out | np.where(sign, 0x80, 0)).astype(np.uint8)


def quantize_query_e4m3(qI):
    """Low-precision indexer query (the pages' FP4/FP8 indexer, 5.4 of the technical-report
    digest): each (query, head) row of q^I gets scale = amax / 448 in fp32 (1 when the row is all
    zero) and codes = e4m3_RNE(q / scale) with the quotient rounded to fp32, the precision the
    GPU divides in.  Returns (codes uint8 [..., dI], scale fp32 [...])."""
    q = np.asarray(qI, dtype=np.float64)
    amax = np.max(np.abs(q), axis=-1).astype(np.float32)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    y = (q.astype(np.float32) / scale[..., None]).astype(np.float32)
    return e4m3_encode_rne(y), scale


def index_scores_lowp(qI, w, kI, q_pos, m):
    """Indexer scores with the query quantised by quantize_query_e4m3 (the keys are already the
    dequantised FP8 keys): I_{t,s} = sum_h w_{t,h} ReLU(q8_{t,h} . K_s) in fp64 over the exact
    dequantised operands."""
    codes, scale = quantize_query_e4m3(qI)
    q8 = e4m3_to_f64(codes) * scale.astype(np.float64)[..., None]
    return index_scores(q8, w, kI, q_pos, m)


def round_scores_bf16(scores):
    """Index scores held in BF16 instead of FP32 ("DeepSeek-V4 技术报告深度解读" 5.4 and the
    indexer QK-path row of "DeepSeek V4 模型技术大全": the top-k selector works on BF16 scores):
    every score rounded to the nearest bf16 value, ties to even, by this module's own rounding;
    -inf stays -inf.  The selection then runs topk_select on the rounded scores, where ties (which
    the rounding makes common) go to the smaller s (R14)."""
    return bf16_to_f64(bf16_round(np.asarray(scores, dtype=np.float64)))


def topk_select(scores, q_pos, m, k):
    """TopK_k over the visible scores of each query.  R14: ties go to the smaller s; with fewer
    than k visible entries all are taken and the row is padded with -1.
    Returns int64 [B, Tq, k] ordered by (score desc, s asc)."""
    scores = np.asarray(scores)
    B, Tq, N = scores.shape
    out = np.full((B, Tq, k), -1, dtype=np.int64)
    for b in range(B):
        for t in range(Tq):
            nv = n_visible(q_pos[b][t], m, N)
            s = np.arange(nv)
            order = np.lexsort((s, -scores[b, t, :nv]))   # primary: score desc; secondary: s asc
            take = order[:min(k, nv)]
            out[b, t, :take.size] = take
    return out


# ------------------------------------------------------------------------------------------------
# core attention: shared K=V MQA over selected / all closed entries + SWA window + sink
# ------------------------------------------------------------------------------------------------


def window_positions(t: int, window: int):
    """SWA window W_t = {u | t - n_win + 1 <= u <= t}, clipped at 0 (R9: includes t itself)."""
    return list(range(max(0, t - window + 1), t + 1))


def attend_query(q, t, kv, entries, win, window, sink, scale=None, rope_dims=64, theta=160000.0,
                 inv_freq=None, q_norm_rope=True, out_unrotate=True, eps=1e-6):
    """One query position t, all heads.

    q fp64 [H, d]; kv fp64 [N, d] compressed entries (K = V); entries: iterable of entry indices
    (the CSA top-k set with -1 pads dropped, or all closed HCA entries); win fp64 [Wcap, d] ring
    of uncompressed per-token KV (slot = position mod Wcap, R8); sink fp64 [H] logits a_h.
      q_hat = RoPE_t(RMSNorm(q))                      (R11, unit weight)
      z_j   = scale * q_hat . K_j   over entries u window   (R10: scale 1/sqrt(d); R9: no dedupe)
      p_j   = exp(z_j) / (exp(a_h) + sum_u exp(z_u))   (the attention-sink equation)
      o     = sum_j p_j K_j ;  o[d-r:] rotated by -t   (R12: reverse rotation of the output)
    Returns (o [H, d], lse [H]) with lse = log(exp(a_h) + sum_u exp(z_u))."""
    q = np.asarray(q, dtype=np.float64)
    H, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    f = rope_inv_freq(theta, rope_dims) if inv_freq is None else np.asarray(inv_freq, np.float64)
    qh = q
    if q_norm_rope:
        qh = rope(rmsnorm(q, eps), float(t), f, rope_dims)
    ent = [int(j) for j in entries if int(j) >= 0]
    Wcap = win.shape[0]
    rows = [kv[j] for j in ent] + [win[u % Wcap] for u in window_positions(t, window)]
    sink = np.asarray(sink, dtype=np.float64)
    if len(rows) == 0:
        return np.zeros((H, d)), sink.copy()
    K = np.stack(rows)                                   # [n, d]
    z = scale * (qh @ K.T)                               # [H, n]
    M = np.maximum(z.max(axis=1), sink)                  # stabiliser includes the sink logit
    e = np.exp(z - M[:, None])
    es = np.exp(sink - M)
    den = es + e.sum(axis=1)
    p = e / den[:, None]
    o = p @ K
    lse = M + np.log(den)
    if out_unrotate:
        o = rope(o, -float(t), f, rope_dims)
    return o, lse


def attend(q, kv, win, sink, q_pos, m, window, idx=None, query_subset=None, **kw):
    """Batched driver over attend_query.  idx None = HCA dense over all closed entries
    j < floor((t+1)/m) (the HCA visibility set); otherwise the CSA selected set idx[b, t].
    q fp64 [B, Tq, H, d]; kv fp64 [B, N, d]; win fp64 [B, Wcap, d]; q_pos [B, Tq].
    query_subset: optional list of (b, t) pairs; other outputs are left NaN."""
    q = np.asarray(q, dtype=np.float64)
    B, Tq, H, d = q.shape
    N = kv.shape[1]
    o = np.full((B, Tq, H, d), np.nan)
    lse = np.full((B, Tq, H), np.nan)
    pairs = query_subset if query_subset is not None else [(b, t) for b in range(B) for t in range(Tq)]
    for b, t in pairs:
        pos = int(q_pos[b][t])
        ents = range(n_visible(pos, m, N)) if idx is None else idx[b][t]
        o[b, t], lse[b, t] = attend_query(q[b, t], pos, kv[b], ents, win[b], window, sink, **kw)
    return o, lse


# ------------------------------------------------------------------------------------------------
# grouped output projection
# ------------------------------------------------------------------------------------------------


def out_proj(O, W_down, W_proj=None):
    """Grouped output projection ("DeepSeek V4 模型技术大全", the grouped output projection
    equations: O = Concat of the n_h head outputs split into g groups O^[u] of n_h/g consecutive
    heads; z^[u] = O^[u] W_down^[u]; y = Proj(Concat_u z^[u])).

    O: [T, n_h, d_h]; W_down: [g, r_o, (n_h/g) d_h], group u's matrix stored transposed (row n
    holds column n of W_down^[u]); W_proj: [d_out, g r_o] or None (Proj stored the same way).
    R26: z is kept in bf16 between the two products (rounded here with the oracle's own
    bf16 rounding), so y is the product of that rounded z.
    Returns (z fp64 [T, g r_o] before rounding, y fp64 [T, d_out] or None)."""
    O = np.asarray(O, dtype=np.float64)
    W_down = np.asarray(W_down, dtype=np.float64)
    T, n_h, d_h = O.shape
    g, r_o, K = W_down.shape
    assert n_h % g == 0 and K == (n_h // g) * d_h
    heads = n_h // g
    z = np.empty((T, g * r_o))
    for u in range(g):
        Ou = O[:, u * heads:(u + 1) * heads, :].reshape(T, K)     # O^[u]: the group's heads side by side
        z[:, u * r_o:(u + 1) * r_o] = Ou @ W_down[u].T              # O^[u] W_down^[u]
    if W_proj is None:
        return z, None
    y = bf16_to_f64(bf16_round(z)) @ np.asarray(W_proj, dtype=np.float64).T
    return z, y
