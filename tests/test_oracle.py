"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
closed forms, invariants, brute force on tiny inputs, library decoders and the
numbers the pages print (tests/golden/page_numbers.json).  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import csa_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))
rng = np.random.default_rng(1234)


def rnd(*shape):
    return rng.standard_normal(shape)


# ------------------------------------------------------------------ storage decoders

def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 97, dtype=np.uint16)
    ours = O.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ours)
    assert np.array_equal(ours[ok], ref[ok])


def test_bf16_round_matches_torch_and_is_nearest():
    x = rng.standard_normal(20000) * 10.0 ** rng.integers(-3, 4, 20000)
    ours = O.bf16_round(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # nearest: no other bf16 neighbour is closer to the fp32 value
    v = O.bf16_to_f64(ours)
    up = O.bf16_to_f64(ours + 1)
    dn = O.bf16_to_f64(ours - 1)
    f = x.astype(np.float32).astype(np.float64)
    assert np.all(np.abs(v - f) <= np.abs(up - f)) and np.all(np.abs(v - f) <= np.abs(dn - f))


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ours)
    assert np.array_equal(ours[ok], ref[ok])


def test_e4m3_known_values():
    v = O.e4m3_to_f64(np.array([0x7E, 0x38, 0x01, 0x08, 0xB8, 0x00, 0x80, 0x7F], dtype=np.uint8))
    assert v[0] == 448.0 and v[1] == 1.0 and v[2] == 2.0 ** -9 and v[3] == 2.0 ** -6
    assert v[4] == -1.0 and v[5] == 0.0 and v[6] == 0.0 and np.isnan(v[7])


def test_fp8_mixed_row_roundtrip_within_half_ulp():
    from long_context_compressed_16_b300 import synth
    x = torch.from_numpy(rnd(6, 512))
    x[:, 17] *= 20.0
    rows = synth.pack_kv_fp8_mixed(x).numpy()
    y = O.fp8_mixed_row_to_f64(rows)
    xs = x.numpy()
    # bf16 part: RNE of the fp32 value
    assert np.array_equal(O.bf16_round(xs[:, 448:]), O.bf16_round(y[:, 448:]))
    # e4m3 part: |x/scale - code| <= half the e4m3 spacing at that magnitude
    scales = rows[:, 576:604].copy().view(np.float32).astype(np.float64)
    for b in range(7):
        blk = xs[:, 64 * b:64 * (b + 1)]
        sc = scales[:, b:b + 1]
        v = blk / sc
        q = y[:, 64 * b:64 * (b + 1)] / sc
        e = np.maximum(np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6))), -6)
        half_ulp = 2.0 ** (e - 3) / 2
        assert np.all(np.abs(v - q) <= half_ulp * (1 + 1e-12))
        assert np.isclose(np.max(np.abs(v)), 448.0)


# ------------------------------------------------------------------ RMSNorm / RoPE

def test_rmsnorm_closed_forms():
    # constant vector c: c / sqrt(c^2 + eps); with c = 1e-3, eps = 1e-6 this is 1/sqrt(2)
    y = O.rmsnorm(np.full((3, 64), 1e-3), eps=1e-6)
    assert np.allclose(y, 1.0 / math.sqrt(2.0), rtol=0, atol=1e-15)
    x = rnd(5, 512)
    y = O.rmsnorm(x, eps=0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-14)
    g = rnd(512)
    assert np.allclose(O.rmsnorm(x, 1e-6, g), O.rmsnorm(x, 1e-6) * g, atol=1e-14)


def test_rope_unit_vector_at_position_one():
    d, r = 128, 64
    x = np.zeros(d)
    x[d - r] = 1.0                                   # first RoPE pair, inv_freq_0 = theta^0 = 1
    y = O.rope(x, 1.0, O.rope_inv_freq(160000.0, r), r)
    expect = np.zeros(d)
    expect[d - r] = math.cos(1.0)
    expect[d - r + 1] = math.sin(1.0)
    assert np.allclose(y, expect, atol=1e-15)
    # a non-RoPE dim never moves
    x = np.zeros(d)
    x[d - r - 1] = 1.0
    assert np.array_equal(O.rope(x, 12345.0, O.rope_inv_freq(160000.0, r), r), x)


def test_rope_invariants():
    r = 64
    f = O.rope_inv_freq(160000.0, r)
    assert f[0] == 1.0 and np.all(np.diff(f) < 0)
    assert np.isclose(f[-1], 160000.0 ** (-62 / 64))
    x, y = rnd(512), rnd(512)
    p1, p2 = 1000.0, 131072.0
    a = O.rope(x, p1, f, r)
    # norm of every pair preserved
    pa = a[448:].reshape(32, 2)
    px = x[448:].reshape(32, 2)
    assert np.allclose(np.linalg.norm(pa, axis=1), np.linalg.norm(px, axis=1), atol=1e-12)
    # reverse rotation is the inverse
    assert np.allclose(O.rope(a, -p1, f, r), x, atol=1e-12)
    # relative property: <R_p1 x, R_p2 y> = <R_{p1-p2} x, y>
    lhs = O.rope(x, p1, f, r) @ O.rope(y, p2, f, r)
    rhs = O.rope(x, p1 - p2, f, r) @ y
    assert np.isclose(lhs, rhs, rtol=1e-10, atol=1e-9)


# ------------------------------------------------------------------ compressor

def _plain(**kw):
    return dict(norm=False, rope_on=False, **kw)


def test_compress_uniform_gates_is_mean_pooling():
    m, d, T = 4, 16, 24
    Ca, Cb = rnd(1, T, d), rnd(1, T, d)
    Z = np.zeros((1, T, d))
    out = O.compress(Ca, Z, m, Cb=Cb, Zb=Z, **_plain())
    assert out.shape == (1, T // m, d)
    assert np.allclose(out[0, 0], Ca[0, 0:4].mean(axis=0), atol=1e-15)      # entry 0: m 'a' rows only
    for i in range(1, T // m):
        rows = np.concatenate([Ca[0, m * i:m * i + m], Cb[0, m * (i - 1):m * i]])
        assert np.allclose(out[0, i], rows.mean(axis=0), atol=1e-15)
    # HCA: m' rows, single stream
    C = rnd(1, 256, d)
    out = O.compress(C, np.zeros((1, 256, d)), 128, **_plain())
    assert np.allclose(out[0, 1], C[0, 128:256].mean(axis=0), atol=1e-14)


def test_compress_one_hot_gate_selects_the_right_row():
    m, d, T = 4, 8, 20
    Ca, Cb = rnd(2, T, d), rnd(2, T, d)
    Za, Zb = np.zeros((2, T, d)), np.zeros((2, T, d))
    i, c = 3, 5
    Za[1, m * i + 2, c] = 800.0        # a-stream row 2 of block i wins channel c of entry i
    Zb[1, m * i + 1, 2] = 800.0        # b-stream row 1 of block i wins channel 2 of entry i+1
    out = O.compress(Ca, Za, m, Cb=Cb, Zb=Zb, **_plain())
    assert out[1, i, c] == Ca[1, m * i + 2, c]
    assert out[1, i + 1, 2] == Cb[1, m * i + 1, 2]
    # biases: B^a row 2 / B^b row 1 dominate every channel
    ba = np.zeros((m, d))
    ba[2] = 800.0
    out = O.compress(Ca, np.zeros_like(Za), m, Cb=Cb, Zb=np.zeros_like(Zb), bias_a=ba, **_plain())
    assert np.array_equal(out[0, :, :], Ca[0, 2:T:m, :])
    bb = np.zeros((m, d))
    bb[1] = 800.0
    out = O.compress(Ca, np.zeros_like(Za), m, Cb=Cb, Zb=np.zeros_like(Zb), bias_b=bb, **_plain())
    for i in range(1, T // m):
        assert np.array_equal(out[0, i], Cb[0, m * (i - 1) + 1])
    assert np.allclose(out[0, 0], Ca[0, 0:4].mean(axis=0))    # entry 0 has no b block


def test_compress_two_rows_is_logistic_mix():
    # m = 1 with overlap: entry i mixes Ca_i and Cb_{i-1} with weight sigmoid(Za_i + ba - Zb_{i-1} - bb)
    d, T = 6, 9
    Ca, Cb, Za, Zb = rnd(1, T, d), rnd(1, T, d), rnd(1, T, d) * 3, rnd(1, T, d) * 3
    ba, bb = rnd(1, d), rnd(1, d)
    out = O.compress(Ca, Za, 1, Cb=Cb, Zb=Zb, bias_a=ba, bias_b=bb, **_plain())
    for i in range(1, T):
        g = 1.0 / (1.0 + np.exp(-((Za[0, i] + ba[0]) - (Zb[0, i - 1] + bb[0]))))
        assert np.allclose(out[0, i], g * Ca[0, i] + (1 - g) * Cb[0, i - 1], atol=1e-14)
    assert np.allclose(out[0, 0], Ca[0, 0])


def test_compress_weights_sum_to_one_and_norm_rope_stage():
    m, d, T = 4, 128, 64
    ones = np.ones((1, T, d))
    Za, Zb = rnd(1, T, d) * 4, rnd(1, T, d) * 4
    out = O.compress(ones, Za, m, Cb=ones, Zb=Zb, **_plain())
    assert np.allclose(out, 1.0, atol=1e-14)
    Ca, Cb = rnd(1, T, d), rnd(1, T, d)
    raw = O.compress(Ca, Za, m, Cb=Cb, Zb=Zb, **_plain())
    full = O.compress(Ca, Za, m, Cb=Cb, Zb=Zb, rope_dims=64, theta=160000.0)
    # the norm+rope stage: RMS 1 per entry (rotation keeps the norm) and un-rotating gives RMSNorm(raw)
    assert np.allclose(np.sqrt(np.mean(full ** 2, axis=-1)), np.sqrt(1.0 / (1.0 + 1e-6 / np.mean(raw ** 2, -1))),
                       atol=1e-12)
    f = O.rope_inv_freq(160000.0, 64)
    back = O.rope(full, -(m * np.arange(T // m, dtype=np.float64))[None, :], f, 64)
    assert np.allclose(back, O.rmsnorm(raw), atol=1e-12)


def test_compress_is_causal():
    m, d, T = 4, 128, 40
    a = [rnd(1, T, d) for _ in range(4)]
    ref = O.compress(a[0], a[2], m, Cb=a[1], Zb=a[3])
    t0 = 22                       # perturb tokens >= t0: entries whose blocks end before t0 are unchanged
    b = [x.copy() for x in a]
    for x in b:
        x[:, t0:] = rnd(1, T - t0, d)
    out = O.compress(b[0], b[2], m, Cb=b[1], Zb=b[3])
    closed = (t0 + 1) // m - 1    # last entry whose block ends at or before t0 - 1
    assert np.array_equal(out[:, :closed + 1], ref[:, :closed + 1])
    assert not np.allclose(out[:, closed + 1], ref[:, closed + 1])


# ------------------------------------------------------------------ indexer + top-k

def test_visibility_and_page_numbers():
    with open(os.path.join(HERE, "golden", "page_numbers.json")) as f:
        g = {c["id"]: c for c in json.load(f)["cases"]}
    c = g["closed_prefix_P1000"]
    assert O.n_visible(c["P"] - 1, c["m_hca"], 10 ** 9) * c["m_hca"] == c["P_closed"]
    assert c["P"] - O.n_visible(c["P"] - 1, c["m_hca"], 10 ** 9) * c["m_hca"] == c["tau"]
    for key in ("lcm_block_entries", "vllm_block_256"):
        c = g[key]
        assert O.n_visible(c["tokens"] - 1, c["m_csa"], 10 ** 9) == c["csa_entries"]
        assert O.n_visible(c["tokens"] - 1, c["m_hca"], 10 ** 9) == c["hca_entries"]
    c = g["hca_1m_entries"]
    assert round(O.n_visible(c["tokens"] - 1, c["m_hca"], 10 ** 9) / 1000, 1) == c["entries_approx_thousands"]
    c = g["window_128"]
    W = O.window_positions(c["t"], c["n_win"])
    assert (W[0], W[-1], len(W)) == (c["first"], c["last"], c["size"])
    c = g["partial_rope_ratio"]
    assert c["d_rope"] / c["d_h"] == c["rho"]
    # only closed blocks: t = m-2 sees nothing, t = m-1 sees block 0
    assert O.n_visible(2, 4, 100) == 0 and O.n_visible(3, 4, 100) == 1
    assert O.n_visible(126, 128, 100) == 0 and O.n_visible(127, 128, 100) == 1
    assert O.window_positions(5, 128) == list(range(0, 6))


def test_index_score_exact_integer_cases():
    # two heads, integer vectors: dots are exact
    N, dI = 6, 4
    kI = np.zeros((1, N, dI))
    for s in range(N):
        kI[0, s, s % dI] = s + 1
    qI = np.zeros((1, 1, 2, dI))
    qI[0, 0, 0] = [1, -1, 2, 0]
    qI[0, 0, 1] = [-3, 1, 0, 1]
    w = np.array([[[2.0, 3.0]]])
    t = 4 * N - 1
    sc = O.index_scores(qI, w, kI, [[t]], 4)
    for s in range(N):
        d0 = qI[0, 0, 0] @ kI[0, s]
        d1 = qI[0, 0, 1] @ kI[0, s]
        assert sc[0, 0, s] == 2 * max(d0, 0) + 3 * max(d1, 0)
    # visibility: query at t = 9 with m = 4 sees entries 0, 1 only
    sc = O.index_scores(qI, w, kI, [[9]], 4)
    assert np.isfinite(sc[0, 0, :2]).all() and np.isneginf(sc[0, 0, 2:]).all()
    # ReLU is per head: negating head 1 only removes head 1's positive part
    q2 = qI.copy()
    q2[0, 0, 1] *= -1
    a = O.index_scores(qI, w, kI, [[t]], 4)[0, 0]
    b = O.index_scores(q2, w, kI, [[t]], 4)[0, 0]
    h0 = 2 * np.maximum(kI[0] @ qI[0, 0, 0], 0)
    assert np.allclose(a - h0, 3 * np.maximum(kI[0] @ qI[0, 0, 1], 0))
    assert np.allclose(b - h0, 3 * np.maximum(-(kI[0] @ qI[0, 0, 1]), 0))


def test_index_query_equal_to_a_key_ranks_it_first():
    N, dI = 200, 32
    kI = rnd(1, N, dI)
    kI /= np.linalg.norm(kI, axis=-1, keepdims=True)
    j = 137
    qI = kI[0, j][None, None, None, :]
    sc = O.index_scores(qI, np.ones((1, 1, 1)), kI, [[4 * N]], 4)
    assert int(np.argmax(sc[0, 0])) == j
    assert O.topk_select(sc, [[4 * N]], 4, 1)[0, 0, 0] == j


def test_topk_brute_force_subsets():
    for trial in range(40):
        N = int(rng.integers(1, 11))
        k = int(rng.integers(1, 5))
        vals = rng.integers(0, 4, N).astype(np.float64)      # many exact ties
        sc = vals[None, None, :]
        got = O.topk_select(sc, [[4 * N - 1]], 4, k)[0, 0]
        nv = N
        if k >= nv:
            assert sorted(got[:nv].tolist()) == list(range(nv)) and np.all(got[nv:] == -1)
            continue
        best = None
        for sub in itertools.combinations(range(N), k):
            key = (-vals[list(sub)].sum(), sum(sub))                 # max score sum, then smallest indices
            if best is None or key < best[0]:
                best = (key, sub)
        assert sorted(got.tolist()) == list(best[1])


def test_topk_pads_with_minus_one():
    sc = np.arange(10, dtype=np.float64)[None, None, :]
    got = O.topk_select(sc, [[11]], 4, 5)[0, 0]      # t = 11 -> 3 visible
    assert got.tolist() == [2, 1, 0, -1, -1]


# ------------------------------------------------------------------ attention

def _attn_inputs(H=2, d=128, N=8, Wcap=64):
    q = rnd(H, d)
    kv = O.rmsnorm(rnd(N, d))
    win = O.rmsnorm(rnd(Wcap, d))
    sink = rnd(H)
    return q, kv, win, sink


def test_attend_textbook_softmax_when_extras_off():
    H, d, N = 3, 64, 20
    q, kv, win, _ = _attn_inputs(H, d, N)
    sink = np.full(H, -np.inf)
    o, lse = O.attend_query(q, 100, kv, range(N), win, 0, sink, rope_dims=0, q_norm_rope=False,
                            out_unrotate=False)
    logits = q @ kv.T / math.sqrt(d)
    import scipy.special
    P = scipy.special.softmax(logits, axis=1)
    assert np.allclose(o, P @ kv, atol=1e-13)
    assert np.allclose(lse, scipy.special.logsumexp(logits, axis=1), atol=1e-12)


def test_attend_sink_identity():
    H, d, N = 4, 128, 12
    q, kv, win, _ = _attn_inputs(H, d, N)
    t = 40
    kw = dict(rope_dims=64, out_unrotate=True)
    o0, lse0 = O.attend_query(q, t, kv, range(N), win, 128, np.full(H, -np.inf), **kw)
    S = np.exp(lse0)                              # sum of exp(z) without the sink
    for a in (-3.0, 0.0, 2.5, 9.0):
        oa, lsea = O.attend_query(q, t, kv, range(N), win, 128, np.full(H, a), **kw)
        assert np.allclose(oa, o0 * (S / (S + math.exp(a)))[:, None], atol=1e-13)
        assert np.allclose(np.exp(lsea), S + math.exp(a), rtol=1e-12)
    ob, _ = O.attend_query(q, t, kv, range(N), win, 128, np.full(H, 80.0), **kw)
    assert np.max(np.abs(ob)) < 1e-25


def test_attend_identical_rows_and_reverse_rotation_sign():
    H, d, r = 3, 128, 64
    f = O.rope_inv_freq(160000.0, r)
    u = O.rmsnorm(rnd(d))
    p, t = 37.0, 1000
    v = O.rope(u, p, f, r)
    N, Wcap = 10, 256
    kv = np.tile(v, (N, 1))
    win = np.tile(v, (Wcap, 1))
    q = rnd(H, d)
    sink = rnd(H)
    o, _ = O.attend_query(q, t, kv, range(N), win, 128, sink, rope_dims=r, out_unrotate=False)
    z = (O.rope(O.rmsnorm(q), float(t), f, r) @ v) / math.sqrt(d)
    n = N + 128
    psink = np.exp(sink) / (np.exp(sink) + n * np.exp(z))
    assert np.allclose(o, (1 - psink)[:, None] * v[None, :], atol=1e-13)
    o2, _ = O.attend_query(q, t, kv, range(N), win, 128, sink, rope_dims=r, out_unrotate=True)
    # un-rotation by -t: RoPE_{p-t}(u) scaled by the non-sink mass
    assert np.allclose(o2, (1 - psink)[:, None] * O.rope(u, p - t, f, r)[None, :], atol=1e-12)


def test_attend_window_bounds():
    H, d = 1, 64
    Wcap = 512
    q = np.zeros((H, d))
    q[0, 0] = 1.0
    t = 300
    for u0, inside in ((t, True), (t - 127, True), (t - 128, False), (t + 1, False)):
        win = np.zeros((Wcap, d))
        win[u0 % Wcap, 0] = 5.0
        o, _ = O.attend_query(q, t, np.zeros((0, d)), [], win, 128, np.array([-np.inf]), rope_dims=0,
                              q_norm_rope=False, out_unrotate=False)
        if inside:
            pe = math.exp(5.0 / 8.0) / (math.exp(5.0 / 8.0) + 127)
            assert np.isclose(o[0, 0], 5.0 * pe, rtol=1e-13)
        else:
            assert o[0, 0] == 0.0


def test_attend_topk_covering_all_equals_dense():
    B, Tq, H, d, N, m = 1, 3, 2, 128, 16, 4
    q = rnd(B, Tq, H, d)
    kv = O.rmsnorm(rnd(B, N, d))
    win = O.rmsnorm(rnd(B, 128, d))
    sink = rnd(H)
    q_pos = [[30, 45, 63]]
    dense, l1 = O.attend(q, kv, win, sink, q_pos, m, 128)
    idx = np.full((B, Tq, N), -1)
    for t in range(Tq):
        nv = O.n_visible(q_pos[0][t], m, N)
        idx[0, t, :nv] = rng.permutation(nv)
    sparse, l2 = O.attend(q, kv, win, sink, q_pos, m, 128, idx=idx)
    assert np.allclose(dense, sparse, atol=1e-13) and np.allclose(l1, l2, atol=1e-12)


def test_attend_brute_force_masked_matrix():
    """Full dense logit matrix over [entries | tokens | sink] with masks written from the
    visibility / selection / window definitions, against the per-query list-based oracle."""
    T, H, d, r, m, W, k = 32, 2, 128, 64, 4, 8, 3
    f = O.rope_inv_freq(160000.0, r)
    N = T // m
    q = rnd(1, T, H, d)
    kv = O.rmsnorm(rnd(1, N, d))
    win = O.rmsnorm(rnd(1, T, d))
    sink = rnd(H)
    q_pos = [list(range(T))]
    idx = np.full((1, T, k), -1)
    for t in range(T):
        nv = O.n_visible(t, m, N)
        sel = rng.permutation(nv)[:k]
        idx[0, t, :sel.size] = sel
    o, lse = O.attend(q, kv, win, sink, q_pos, m, W, idx=idx)
    K = np.concatenate([kv[0], win[0]])                  # [N + T, d]
    for h in range(H):
        Q = np.stack([O.rope(O.rmsnorm(q[0, t, h]), float(t), f, r) for t in range(T)])
        L = Q @ K.T / math.sqrt(d)                          # [T, N + T]
        mask = np.zeros_like(L, dtype=bool)
        for t in range(T):
            for s in idx[0, t]:
                if s >= 0:
                    mask[t, s] = True
            for u in range(T):
                mask[t, N + u] = (t - W < u <= t)
        Lm = np.where(mask, L, -np.inf)
        full = np.concatenate([Lm, np.full((T, 1), sink[h])], axis=1)
        P = np.exp(full - full.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        ref = P[:, :-1] @ K
        ref = np.stack([O.rope(ref[t], -float(t), f, r) for t in range(T)])
        assert np.allclose(o[0, :, h], ref, atol=1e-12)
        lref = np.log(np.exp(full - full.max(1, keepdims=True)).sum(1)) + full.max(1)
        assert np.allclose(lse[0, :, h], lref, atol=1e-12)


def test_whole_path_is_causal():
    """Perturbing tokens after t leaves the output at t unchanged through compress, indexer,
    top-k and attention."""
    T, m, d, dI, H, nI, k = 48, 4, 128, 32, 2, 2, 3
    streams = [rnd(1, T, d) for _ in range(4)]
    istreams = [rnd(1, T, dI) for _ in range(4)]
    q, qI, w = rnd(1, T, H, d), rnd(1, T, nI, dI), np.abs(rnd(1, T, nI))
    win = rnd(1, T, d)
    sink = rnd(H)
    q_pos = [list(range(T))]

    def run(st, ist, win):
        kv = O.compress(st[0], st[2], m, Cb=st[1], Zb=st[3])
        kI = O.compress(ist[0], ist[2], m, Cb=ist[1], Zb=ist[3], rope_on=False)
        sc = O.index_scores(qI, w, kI, q_pos, m)
        idx = O.topk_select(sc, q_pos, m, k)
        return O.attend(q, kv, win, sink, q_pos, m, 16, idx=idx)[0]

    ref = run(streams, istreams, win)
    t = 29
    st2 = [x.copy() for x in streams]
    ist2 = [x.copy() for x in istreams]
    win2 = win.copy()
    for x in st2 + ist2 + [win2]:
        x[:, t + 1:] = rnd(*x[:, t + 1:].shape)
    out = run(st2, ist2, win2)
    assert np.array_equal(out[0, :t + 1], ref[0, :t + 1])
    assert not np.allclose(out[0, t + 1:], ref[0, t + 1:])


# ------------------------------------------------------------------ low-precision indexer query

def test_e4m3_encoder_round_trips_every_code_and_rounds_half_to_even():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)   # no NaNs
    vals = O.e4m3_to_f64(codes)
    assert np.array_equal(O.e4m3_encode_rne(vals.astype(np.float32)), codes)
    # midpoints between neighbouring positive codes round to the even mantissa
    pos = np.arange(0, 0x7E)
    lo, hi = O.e4m3_to_f64(pos), O.e4m3_to_f64(pos + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    got = O.e4m3_encode_rne(mid).astype(np.int64)
    want = np.where(pos % 2 == 0, pos, pos + 1)
    exact = mid.astype(np.float64) == (lo + hi) / 2          # midpoints exactly representable in fp32
    assert np.array_equal(got[exact], want[exact])
    # saturation and underflow
    assert O.e4m3_encode_rne(np.float32([448.0, 460.0, 1e6, -1e6])).tolist() == [0x7E, 0x7E, 0x7E, 0xFE]
    assert O.e4m3_encode_rne(np.float32([2.0 ** -10, -2.0 ** -10, 0.0])).tolist() == [0, 0x80, 0]


def test_e4m3_encoder_matches_torch_in_range():
    x = (rng.standard_normal(50000) * 10.0 ** rng.integers(-3, 3, 50000)).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode_rne(x), ref)


def test_query_quantisation_scale_and_amax_code():
    q = rnd(3, 5, 128)
    codes, scale = O.quantize_query_e4m3(q)
    amax = np.max(np.abs(q), axis=-1)
    assert np.allclose(scale, amax / 448.0, rtol=1e-6)
    # the largest element of every row maps to the largest code
    i = np.argmax(np.abs(q), axis=-1)
    top = np.take_along_axis(codes, i[..., None], axis=-1)[..., 0] & 0x7F
    assert np.all(top == 0x7E)
    # dequantised values are within half an e4m3 step (relative 2^-4) of the inputs
    deq = O.e4m3_to_f64(codes) * scale[..., None]
    big = np.abs(q) > amax[..., None] * 2.0 ** -6
    assert np.all(np.abs(deq - q)[big] <= np.abs(q)[big] * 2.0 ** -4 + 1e-12)
    zc, zs = O.quantize_query_e4m3(np.zeros((2, 128)))
    assert np.all(zc == 0) and np.all(zs == 1.0)


def test_index_scores_lowp_by_hand():
    """Low-precision indexer scores, computed by hand from the e4m3 format (1 sign, 4 exponent
    bits with bias 7, 3 mantissa bits; subnormals in units of 2^-9) and the per-(query, head)
    scale amax/448 ("DeepSeek-V4 技术报告深度解读" 5.4, FP4/FP8 indexer; the I_{t,s} equation).

    head 0: q = (896, 3, 0.3, -10): amax 896 -> scale 2 exactly; q/2 = (448, 1.5, 0.15, -5).
            0.15 lies in [2^-3, 2^-2), step 2^-6: 0.15 = 9.6 steps -> 10 steps = 0.15625, so the
            dequantised row is (896, 3, 0.3125, -10).
    head 1: q = (1, -2, 0.01, 14): amax 14 -> scale 1/32 exactly; q*32 = (32, -64, 0.32, 448).
            0.32 lies in [2^-2, 2^-1), step 2^-5: 10.24 steps -> 10 = 0.3125, dequantised
            0.3125/32 = 0.009765625.  (With head 0's scale instead, 0.005 would be subnormal and
            come back as 3 * 2^-9 * 2 = 0.01171875: the per-row scale is visible.)
    keys: K_0 = (1, 1, 1, 1), K_1 = (0, 1, -4, 1); weights w = (0.5, 2).
      s = 0: head 0 889.3125, head 1 13.009765625 -> 0.5*889.3125 + 2*13.009765625 = 470.67578125
      s = 1: head 0 -8.25 -> ReLU 0, head 1 11.9609375 -> 2*11.9609375 = 23.921875"""
    qI = np.array([[[[896.0, 3.0, 0.3, -10.0], [1.0, -2.0, 0.01, 14.0]]]])
    w = np.array([[[0.5, 2.0]]])
    kI = np.array([[[1.0, 1.0, 1.0, 1.0], [0.0, 1.0, -4.0, 1.0]]])
    q_pos = [[8]]
    codes, scale = O.quantize_query_e4m3(qI)
    np.testing.assert_array_equal(scale[0, 0], np.array([2.0, 1.0 / 32.0], dtype=np.float32))
    np.testing.assert_array_equal(O.e4m3_to_f64(codes[0, 0, 0]), [448.0, 1.5, 0.15625, -5.0])
    np.testing.assert_array_equal(O.e4m3_to_f64(codes[0, 0, 1]), [32.0, -64.0, 0.3125, 448.0])
    got = O.index_scores_lowp(qI, w, kI, q_pos, 4)
    np.testing.assert_array_equal(got[0, 0], [470.67578125, 23.921875])
    # the unquantised query gives different scores (0.5*889.3 + 2*13.01 = 470.67 and 23.92):
    # the quantisation is really applied
    plain = O.index_scores(qI, w, kI, q_pos, 4)
    assert plain[0, 0, 0] != got[0, 0, 0] and plain[0, 0, 1] != got[0, 0, 1]


def test_bf16_scores_round_to_nearest_even_and_ties_go_to_the_smaller_entry():
    """bf16 keeps 8 significant bits: in [1, 2) the spacing is 2^-7.
      s0 = 1            -> 1
      s1 = 1 + 2^-8     -> halfway between 1 and 1 + 2^-7: ties to even -> 1
      s2 = 1 + 3 2^-8   -> halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even) -> 1 + 2^-6
      s3 = 1 + 2^-7 + 2^-10 -> nearest 1 + 2^-7
    In fp64 the order is s2 > s3 > s1 > s0 (top-3 = {2, 3, 1}); after rounding s0 and s1 tie at
    1 and the smaller index wins (top-3 = {2, 3, 0}); -inf stays -inf."""
    sc = np.array([[[1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -7 + 2.0 ** -10, -np.inf]]])
    r = O.round_scores_bf16(sc)
    np.testing.assert_array_equal(r[0, 0], [1.0, 1.0, 1.0 + 2.0 ** -6, 1.0 + 2.0 ** -7, -np.inf])
    q_pos = [[4 * 4 - 1]]                         # m = 4: entries 0..3 visible
    assert sorted(O.topk_select(sc, q_pos, 4, 3)[0, 0].tolist()) == [1, 2, 3]
    assert sorted(O.topk_select(r, q_pos, 4, 3)[0, 0].tolist()) == [0, 2, 3]
    assert O.topk_select(r, q_pos, 4, 1)[0, 0].tolist() == [2]


# ------------------------------------------------------------------------------------------------ grouped output projection

def test_out_proj_equals_one_block_diagonal_product():
    """Grouping heads u*n_h/g .. (u+1)*n_h/g - 1 with their own W_down^[u] is one product of the
    flattened O with the block-diagonal matrix diag(W_down^[1], .., W_down^[g])."""
    from scipy.linalg import block_diag
    rng = np.random.default_rng(5)
    T, n_h, d_h, g, r_o = 7, 6, 4, 3, 5
    Oa = rng.standard_normal((T, n_h, d_h))
    Wd = rng.standard_normal((g, r_o, (n_h // g) * d_h))
    z, y = O.out_proj(Oa, Wd)
    assert y is None
    dense = block_diag(*[Wd[u].T for u in range(g)])            # [n_h d_h, g r_o]
    np.testing.assert_allclose(z, Oa.reshape(T, n_h * d_h) @ dense, rtol=1e-12, atol=1e-12)


def test_out_proj_tiny_by_hand_and_bf16_intermediate():
    """n_h = 4 heads of d_h = 1, g = 2, r_o = 1: z = (1*1 + 2*10, 3*100 + 4*1000) = (21, 4300);
    z is held in bf16 (4300 -> 4288, the bf16 spacing at 4096 is 32) before Proj."""
    Oa = np.array([[[1.0], [2.0], [3.0], [4.0]]])
    Wd = np.array([[[1.0, 10.0]], [[100.0, 1000.0]]])
    Wp = np.array([[1.0, 1.0], [2.0, -1.0]])
    z, y = O.out_proj(Oa, Wd, Wp)
    np.testing.assert_array_equal(z, [[21.0, 4300.0]])
    np.testing.assert_array_equal(y, [[21.0 + 4288.0, 42.0 - 4288.0]])


def test_out_proj_page_configuration():
    """Flash: n_h = 64 heads of d_h = 512, g = 8, r_o = 1024, hidden 4096: each W_down^[u] is
    (n_h/g) d_h x r_o = 4096 x 1024, and the two products have equal work per token."""
    with open(os.path.join(HERE, "golden", "page_numbers.json")) as f:
        c = next(x for x in json.load(f)["cases"] if x["id"] == "out_proj_flash")
    K = c["n_h"] // c["g"] * c["d_h"]
    assert K == c["w_down_rows"] and c["r_o"] == c["w_down_cols"]
    assert c["n_h"] * c["d_h"] * c["r_o"] == c["g"] * c["r_o"] * c["hidden"]
