"""GPU parity: each C-ABI call against the fp64 oracle on the same seeded inputs.

Every call gets inputs that come from the seeded generator or from the oracle itself (never from
the CUDA path): the attention calls receive the oracle's own top-k sets, the indexer receives
the oracle's compressed keys rounded to bf16 by the oracle."""
import math

import numpy as np
import pytest
import torch

from long_context_compressed_16_b300 import capi as C
from long_context_compressed_16_b300 import pipeline as P
from long_context_compressed_16_b300 import synth as S
from oracle import csa_oracle as O
from tests.helpers import assert_close, assert_lse, check_topk_row, f64, nvis_of

pytestmark = pytest.mark.gpu
DEV = "cuda"
THETA = 160000.0


def _oracle_compress(inp, names, m, d, rope=True, overlap=True, **kw):
    Ca, Cb, Za, Zb = (f64(inp[n]) for n in names) if overlap else (f64(inp[names[0]]), None,
                                                                     f64(inp[names[1]]), None)
    return O.compress(Ca, Za, m, Cb=Cb, Zb=Zb, rope_on=rope, rope_dims=64 if rope else 0, theta=THETA, **kw)


def _to_dev_bf16(x64: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(O.bf16_round(x64).view(np.int16)).view(torch.bfloat16).to(DEV)


# ------------------------------------------------------------------------------------------------ compress

@pytest.mark.parametrize("B,T,d,m,overlap,rope,bias", [
    (1, 2048, 128, 4, True, True, False),       # tiny workload main stream
    (1, 2048, 64, 4, True, False, False),       # tiny workload indexer keys (RMSNorm, no RoPE)
    (2, 2050, 512, 4, True, True, True),        # ragged tail, batch 2, biases and gamma
    (1, 1000, 128, 1, True, True, True),        # m = 1 (two-row logistic mix)
    (2, 4096 + 77, 512, 128, False, True, True),  # HCA, ragged
    (1, 640, 1024, 8, True, True, False),       # widest supported row
    # whole-sequence m = 4 calls at every stage shape of the streamed kernel: d = 1024 (one entry
    # of 32 KB per stage, 3 groups), d = 256 (two entries per stage), a null b-bias read as zeros,
    # gamma without biases, and batch 2 with ~55 stages per CTA crossing the sequence boundary
    (3, 4096 + 8, 1024, 4, True, True, "a_only"),
    (2, 8192 + 4, 256, 4, True, True, "gamma_only"),
    (2, 16384 + 12, 512, 4, True, True, True),
])
def test_compress_parity(B, T, d, m, overlap, rope, bias):
    g = torch.Generator().manual_seed(T + d)
    names = ("Ca", "Cb", "Za", "Zb")
    inp = {n: S.normal_bf16((B, T, d), 7, S.TID[n], DEV) for n in names}
    ba = bb = gam = None
    kw = {}
    if bias:
        ba = torch.randn(m, d, generator=g).float().to(DEV)
        bb = torch.randn(m, d, generator=g).float().to(DEV)
        gam = (1 + 0.1 * torch.randn(d, generator=g)).float().to(DEV)
        if bias == "a_only":
            bb = None
        if bias == "gamma_only":
            ba = bb = None
        np_ = lambda t: None if t is None else t.double().cpu().numpy()
        kw = dict(bias_a=np_(ba), bias_b=np_(bb) if overlap else None, gamma=np_(gam))
    out = P.compress(inp["Ca"], inp["Za"], m, Cb=inp["Cb"] if overlap else None, Zb=inp["Zb"] if overlap else None,
                     bias_a=ba, bias_b=bb if overlap else None, gamma=gam, rope=rope,
                     rope_dims=64 if rope else 0, theta=THETA)
    torch.cuda.synchronize()
    if overlap:
        ref = O.compress(f64(inp["Ca"]), f64(inp["Za"]), m, Cb=f64(inp["Cb"]), Zb=f64(inp["Zb"]), rope_on=rope,
                         rope_dims=64 if rope else 0, theta=THETA, **kw)
    else:
        ref = O.compress(f64(inp["Ca"]), f64(inp["Za"]), m, rope_on=rope, rope_dims=64 if rope else 0, theta=THETA,
                         **{k: v for k, v in kw.items() if k != "bias_b"})
    assert_close(out, ref, f"compress B{B} T{T} d{d} m{m}")


def test_compress_rope_far_positions_and_table():
    """RoPE angles reduced in 64-bit integer phase: entries at positions past 2^21 (pos_shift),
    and a host frequency table with values above one radian per position (the reduction modulo a
    revolution) and far below it, against the oracle's fp64 angles."""
    B, T, d, m = 2, 2048 + 12, 512, 4
    g = torch.Generator().manual_seed(77)
    inp = {n: S.normal_bf16((B, T, d), 9, S.TID[n], DEV) for n in ("Ca", "Cb", "Za", "Zb")}
    inv = [3.7, 1.0, 0.5, 2.0 ** -0.5] + [float(160000.0 ** (-2.0 * j / 64)) for j in range(4, 32)]
    inv = [float(np.float32(v)) for v in inv]                 # the table is fp32 on the host side
    shift = 3 * (1 << 20) + 5
    out = P.compress(inp["Ca"], inp["Za"], m, Cb=inp["Cb"], Zb=inp["Zb"], inv_freq=inv, pos_shift=shift)
    torch.cuda.synchronize()
    ref = O.compress(f64(inp["Ca"]), f64(inp["Za"]), m, Cb=f64(inp["Cb"]), Zb=f64(inp["Zb"]),
                     inv_freq=np.asarray(inv, np.float64), pos_shift=shift)
    assert_close(out, ref, "compress, far positions, frequency table")


def test_compress_degenerate_sizes():
    x = S.normal_bf16((1, 3, 128), 0, 1, DEV)
    out = P.compress(x, x, 4, Cb=x, Zb=x)             # T < m: no closed block
    assert out.shape == (1, 0, 128)
    x = S.normal_bf16((0, 64, 128), 0, 1, DEV)
    assert P.compress(x, x, 4, Cb=x, Zb=x).shape == (0, 16, 128)


def test_compress_full_size_prefill_streams():
    """The 65536-token prefill chunk: main stream d=512 and indexer stream d=128, every entry."""
    w = S.WORKLOADS["csa_prefill_t65536"]
    inp = {n: S.normal_bf16((1, w.T, w.d), w.seed, S.TID[n], DEV) for n in ("Ca", "Cb", "Za", "Zb")}
    inp.update({n: S.normal_bf16((1, w.T, w.dI), w.seed, S.TID[n], DEV) for n in ("Ca_I", "Cb_I", "Za_I", "Zb_I")})
    kv = P.compress(inp["Ca"], inp["Za"], 4, Cb=inp["Cb"], Zb=inp["Zb"], theta=THETA)
    kI = P.compress(inp["Ca_I"], inp["Za_I"], 4, Cb=inp["Cb_I"], Zb=inp["Zb_I"], rope=False, rope_dims=0)
    torch.cuda.synchronize()
    ref = _oracle_compress(inp, ("Ca", "Cb", "Za", "Zb"), 4, 512)
    assert_close(kv, ref, "compress T=65536 d=512")
    ref = _oracle_compress(inp, ("Ca_I", "Cb_I", "Za_I", "Zb_I"), 4, 128, rope=False)
    assert_close(kI, ref, "compress T=65536 d=128 (indexer keys)")


# ------------------------------------------------------------------------------------------------ indexer + top-k

def _index_case(qI, w, kI, q_pos, m, k, kI_scale=None, with_scores=True, sample=None):
    B, Tq = qI.shape[:2]
    N = kI.shape[1]
    sc = torch.empty((B, Tq, N), dtype=torch.float32, device=DEV) if with_scores else None
    idx = P.index_topk(qI, w, kI, q_pos, m, k, kI_scale=kI_scale, score_out=sc)
    torch.cuda.synchronize()
    qpos = q_pos.cpu().numpy()
    gi = idx.cpu().numpy()
    gs = sc.cpu().numpy() if with_scores else None
    pairs = sample if sample is not None else [(b, t) for b in range(B) for t in range(Tq)]
    near = 0
    for b in range(B):
        rows = [t for (bb, t) in pairs if bb == b]
        if not rows:
            continue
        if kI_scale is None:
            kb = f64(kI[b:b + 1])
        else:
            kb = O.e4m3_to_f64(kI[b:b + 1].cpu().numpy()) * kI_scale[b:b + 1].cpu().double().numpy()[..., None]
        qb = f64(qI[b:b + 1, rows])
        wb = f64(w[b:b + 1, rows])
        ref = O.index_scores(qb, wb, kb, [qpos[b, rows]], m)
        for j, t in enumerate(rows):
            nv = nvis_of(qpos[b, t], m, N)
            if with_scores:
                row_ref = ref[0, j]
                tol = 1e-5 * max(1.0, float(np.max(np.abs(row_ref[:nv])))) if nv else 1e-6
                assert np.all(np.abs(gs[b, t, :nv] - row_ref[:nv]) <= tol), f"scores b{b} t{t}"
                assert np.all(np.isneginf(gs[b, t, nv:])), f"invisible scores b{b} t{t}"
            near += check_topk_row(gi[b, t], ref[0, j, :nv], nv, k, f"topk b{b} t{t}")
    return near


def test_index_topk_tiny_prefill_all_queries():
    w = S.WORKLOADS["tiny_csa_prefill_t2048"]
    inp = S.make_inputs(w, DEV)
    kI64 = _oracle_compress(inp, ("Ca_I", "Cb_I", "Za_I", "Zb_I"), 4, 64, rope=False)
    kI = _to_dev_bf16(kI64)
    _index_case(inp["qI"], inp["w"], kI, inp["q_pos"], 4, w.k)


@pytest.mark.parametrize("B,Tq,N,nI,dI,k,m", [
    (2, 37, 1000, 20, 128, 48, 4),     # ragged tiles, heads not a multiple of 16, prefill groups
    (3, 1, 129, 64, 128, 512, 4),      # k > N visible: take all + pad
    (1, 9, 300, 64, 64, 7, 4),         # dI = 64
    (2, 1, 5000, 8, 128, 2048, 4),     # largest k
])
def test_index_topk_shapes(B, Tq, N, nI, dI, k, m):
    qI = S.normal_bf16((B, Tq, nI, dI), 3, S.TID["qI"], DEV)
    w = S.uniform_f64((B, Tq, nI), 3, S.TID["w"], DEV).float()
    kI = S.normal_bf16((B, N, dI), 3, S.TID["kI"], DEV)
    gen = torch.Generator().manual_seed(N)
    q_pos = torch.randint(0, 4 * N + 8, (B, Tq), generator=gen).int()
    q_pos[0, 0] = 2          # a query with nothing visible
    _index_case(qI, w, kI, q_pos.to(DEV), m, k)


def test_index_topk_no_entries():
    qI = S.normal_bf16((2, 3, 8, 64), 1, 1, DEV)
    w = torch.ones((2, 3, 8), device=DEV)
    kI = torch.empty((2, 0, 64), dtype=torch.bfloat16, device=DEV)
    q_pos = torch.full((2, 3), 100, dtype=torch.int32, device=DEV)
    idx = P.index_topk(qI, w, kI, q_pos, 4, 5)
    assert torch.all(idx == -1)


def test_index_topk_decode_128k_full():
    w = S.WORKLOADS["csa_decode_128k_b32"]
    inp = S.make_inputs(w, DEV)
    _index_case(inp["qI"], inp["w"], inp["kI"], inp["q_pos"], 4, w.k)


def test_index_topk_decode_1m_fp8_full():
    w = S.WORKLOADS["csa_decode_1m_b4_fp8"]
    inp = S.make_inputs(w, DEV)
    _index_case(inp["qI"], inp["w"], inp["kI"], inp["q_pos"], 4, w.k, kI_scale=inp["kI_scale"])


@pytest.mark.parametrize("B,Tq,N,nI,dI,k", [
    (32, 1, 32768, 64, 128, 512),      # decode: rows split into slices, then merged
    (1, 300, 2000, 64, 128, 512),      # prefill-like rows, one stage
    (2, 5, 777, 16, 64, 40),           # ragged
])
def test_split_score_and_topk_calls_equal_fused_call(B, Tq, N, nI, dI, k):
    qI = S.normal_bf16((B, Tq, nI, dI), 5, S.TID["qI"], DEV)
    w = S.uniform_f64((B, Tq, nI), 5, S.TID["w"], DEV).float()
    kI = S.normal_bf16((B, N, dI), 5, S.TID["kI"], DEV)
    q_pos = (4 * N - 4 * Tq + 4 * torch.arange(Tq, dtype=torch.int32, device=DEV)).repeat(B, 1).contiguous()
    q_pos[0, 0] = 6                              # a short row (k > visible entries)
    desc = P.index_desc(B, Tq, N, nI, dI, k, 4)
    sc_f = torch.empty((B, Tq, N), dtype=torch.float32, device=DEV)
    idx_f = P.index_topk(qI, w, kI, q_pos, 4, k, score_out=sc_f)
    sc = torch.full((B, Tq, N), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(max(C.csa_index_score_workspace(desc), C.csa_topk_workspace(desc)), dtype=torch.uint8,
                     device=DEV)
    C.check(C.csa_index_score(desc, qI, w, kI, None, q_pos, sc, ws), "csa_index_score")
    idx = torch.full((B, Tq, k), -7, dtype=torch.int32, device=DEV)
    C.check(C.csa_topk(desc, sc, q_pos, idx, ws), "csa_topk")
    torch.cuda.synchronize()
    assert C.csa_read_device_status(ws)[0] == C.CSA_OK
    nv = torch.clamp((q_pos.long() + 1) // 4, max=N)
    mask = torch.arange(N, device=DEV)[None, None, :] >= nv[..., None]
    assert torch.equal(sc[~mask], sc_f[~mask])            # visible scores, bit for bit
    assert torch.all(torch.isnan(sc[mask]))               # the rest of each row is left untouched
    assert torch.equal(idx, idx_f)
    # the selector reads visible entries only: garbage past N_vis changes nothing
    sc2 = torch.where(mask, torch.full_like(sc, 3.0e38), sc)
    idx2 = torch.full_like(idx, -7)
    C.check(C.csa_topk(desc, sc2, q_pos, idx2, ws), "csa_topk")
    torch.cuda.synchronize()
    assert torch.equal(idx2, idx_f)


@pytest.mark.parametrize("B,Tq,N,nI,k", [
    (4, 1, 5000, 64, 1024),            # decode rows, sliced selection
    (1, 37, 700, 20, 64),              # prefill groups, heads not a multiple of 16
    (2, 3, 300, 16, 40),               # ragged tiles
])
def test_index_lowp_scores_and_topk(B, Tq, N, nI, k):
    """Low-precision indexer: the query quantised to e4m3 per (query, head), FP8 tensor cores.
    Scores against the oracle's quantised-query scores; top-k sets with the usual near-tie rule;
    the split score call gives the fused call's scores bit for bit."""
    dI, m = 128, 4
    qI = S.normal_bf16((B, Tq, nI, dI), 7, S.TID["qI"], DEV)
    w = S.uniform_f64((B, Tq, nI), 7, S.TID["w"], DEV).float()
    kf = S.normal_f64((B, N, dI), 7, S.TID["kI"], "cpu")
    k8, ks = S.quantize_rows_e4m3(kf)
    k8, ks = k8.to(DEV), ks.to(DEV)
    gen = torch.Generator().manual_seed(N + 1)
    q_pos = torch.randint(0, 4 * N + 8, (B, Tq), generator=gen).int()
    q_pos[0, 0] = 2
    q_pos = q_pos.to(DEV)
    sc = torch.empty((B, Tq, N), dtype=torch.float32, device=DEV)
    idx = P.index_topk(qI, w, k8, q_pos, m, k, kI_scale=ks, score_out=sc, lowp=True)
    desc = P.index_desc(B, Tq, N, nI, dI, k, m, lowp=True)
    sc2 = torch.full_like(sc, float("nan"))
    ws = torch.zeros(C.csa_index_score_workspace(desc), dtype=torch.uint8, device=DEV)
    C.check(C.csa_index_score(desc, qI, w, k8, ks, q_pos, sc2, ws), "csa_index_score")
    torch.cuda.synchronize()
    qpos = q_pos.cpu().numpy()
    gs, gs2, gi = sc.cpu().numpy(), sc2.cpu().numpy(), idx.cpu().numpy()
    for b in range(B):
        kb = O.e4m3_to_f64(k8[b:b + 1].cpu().numpy()) * ks[b:b + 1].cpu().double().numpy()[..., None]
        ref = O.index_scores_lowp(f64(qI[b:b + 1]), f64(w[b:b + 1]), kb, [qpos[b]], m)
        for t in range(Tq):
            nv = nvis_of(qpos[b, t], m, N)
            row = ref[0, t, :nv]
            tol = 1e-5 * max(1.0, float(np.max(np.abs(row)))) if nv else 1e-6
            assert np.all(np.abs(gs[b, t, :nv] - row) <= tol), f"lowp scores b{b} t{t}"
            assert np.array_equal(gs2[b, t, :nv], gs[b, t, :nv]), f"split call b{b} t{t}"
            check_topk_row(gi[b, t], row, nv, k, f"lowp topk b{b} t{t}")


def test_index_lowp_recall_against_exact_query():
    """The quantised query changes only near-ties: top-k recall against the same FP8 keys with the
    bf16 query, on the 1M-context FP8 decode inputs (the pages report 99.7% for their FP4
    indexer)."""
    w = S.WORKLOADS["csa_decode_1m_b4_fp8"]
    inp = S.make_inputs(w, DEV)
    exact = P.index_topk(inp["qI"], inp["w"], inp["kI"], inp["q_pos"], 4, w.k, kI_scale=inp["kI_scale"])
    lowp = P.index_topk(inp["qI"], inp["w"], inp["kI"], inp["q_pos"], 4, w.k, kI_scale=inp["kI_scale"], lowp=True)
    torch.cuda.synchronize()
    hits = sum(len(set(exact[b, 0].tolist()) & set(lowp[b, 0].tolist())) for b in range(w.B))
    recall = hits / (w.B * w.k)
    print(f"low-precision indexer recall@{w.k}: {recall:.4f}")
    assert recall >= 0.95


# ------------------------------------------------------------------------------------------------ attention

def _oracle_attend_rows(inp, idx_np, m, window, pairs, fp8=False, dense=False, **kw):
    """Oracle outputs for (b, t) pairs, decoding only the kv rows each query uses."""
    q_pos = inp["q_pos"].cpu().numpy()
    N = inp["kv"].shape[1]
    outs, lses = [], []
    for b, t in pairs:
        pos = int(q_pos[b, t])
        if dense:
            ents = list(range(nvis_of(pos, m, N)))
        else:
            ents = [int(e) for e in idx_np[b, t] if e >= 0]
        rows = inp["kv"][b, ents] if ents else inp["kv"][b, :0]
        kvr = O.fp8_mixed_row_to_f64(rows.cpu().numpy()) if fp8 else f64(rows)
        win = f64(inp["win"][b])
        o, l = O.attend_query(f64(inp["q"][b, t]), pos, kvr, range(len(ents)), win, window,
                              f64(inp["sink"]), theta=THETA, **kw)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def _oracle_topk(inp, m, k, pairs):
    """The oracle's own top-k rows for the given queries (fp64 scores over the generator's keys)."""
    q_pos = inp["q_pos"].cpu().numpy()
    N = inp["kI"].shape[1]
    B, Tq = inp["q"].shape[:2]
    idx = np.full((B, Tq, k), -1, dtype=np.int64)
    for b in sorted({p[0] for p in pairs}):
        rows = [t for (bb, t) in pairs if bb == b]
        if "kI_scale" in inp:
            kb = O.e4m3_to_f64(inp["kI"][b:b + 1].cpu().numpy()) * inp["kI_scale"][b:b + 1].cpu().double().numpy()[..., None]
        else:
            kb = f64(inp["kI"][b:b + 1])
        sc = O.index_scores(f64(inp["qI"][b:b + 1, rows]), f64(inp["w"][b:b + 1, rows]), kb, [q_pos[b, rows]], m)
        sel = O.topk_select(sc, [q_pos[b, rows]], m, k)
        for j, t in enumerate(rows):
            idx[b, t] = sel[0, j]
    return idx


def _decode_attend_case(name, fp8=False):
    w = S.WORKLOADS[name]
    inp = S.make_inputs(w, DEV)
    pairs = [(b, 0) for b in range(w.B)]
    idx_np = _oracle_topk(inp, w.m, w.k, pairs)
    idx = torch.from_numpy(idx_np.astype(np.int32)).to(DEV)
    out, lse, ws = P.csa_attend(inp["q"], inp["kv"], idx, inp["win"], inp["sink"], inp["q_pos"], fp8=fp8,
                                want_lse=True)
    torch.cuda.synchronize()
    assert C.csa_read_device_status(ws)[0] == C.CSA_OK
    ref, lref = _oracle_attend_rows(inp, idx_np, w.m, w.window, pairs, fp8=fp8)
    assert_close(out[:, 0], ref, name)
    assert_lse(lse[:, 0], lref, "lse")


def test_attend_decode_128k_full():
    _decode_attend_case("csa_decode_128k_b32")


def test_attend_decode_1m_fp8_full():
    _decode_attend_case("csa_decode_1m_b4_fp8", fp8=True)


@pytest.mark.parametrize("k,splits", [(60, 1), (100, 2), (320, 3), (1024, 6)])
def test_attend_decode_split_counts(k, splits):
    """Decode with k + 128 window slots cut into 192-slot splits: one split (no merge) and 2, 3, 6
    splits merged in a thread-block cluster (each CTA owns whole dim pairs of the output, so a
    rotated pair is merged and turned back in one place; 3 and 6 do not divide the 256 pairs
    evenly).  Selections are seeded random rows; a few queries see fewer entries than k."""
    assert (k + 128 + 191) // 192 == splits
    B, H, d, N, m = 4, 64, 512, 4096, 4
    q_pos = torch.tensor([[4 * N - 1], [4 * N - 77], [4 * k // 2], [4 * N // 3]], dtype=torch.int32, device=DEV)
    q = S.normal_bf16((B, 1, H, d), 17, 1, DEV)
    kv = S.normal_bf16((B, N, d), 17, 2, DEV)
    win = S.normal_bf16((B, 128, d), 17, 3, DEV)
    sink = S.normal_f64((H,), 17, 4).float().to(DEV)
    rng = np.random.default_rng(k)
    idx_np = np.full((B, 1, k), -1, dtype=np.int64)
    for b in range(B):
        nv = nvis_of(int(q_pos[b, 0]), m, N)
        take = min(k, nv)
        idx_np[b, 0, :take] = np.sort(rng.permutation(nv)[:take])
    idx = torch.from_numpy(idx_np.astype(np.int32)).to(DEV)
    out, lse, ws = P.csa_attend(q, kv, idx, win, sink, q_pos, want_lse=True)
    torch.cuda.synchronize()
    assert C.csa_read_device_status(ws)[0] == C.CSA_OK
    inp = dict(q=q, kv=kv, win=win, sink=sink, q_pos=q_pos)
    ref, lref = _oracle_attend_rows(inp, idx_np, m, 128, [(b, 0) for b in range(B)])
    assert_close(out[:, 0], ref, f"decode, {splits} splits")
    assert_lse(lse[:, 0], lref, "lse")
    # the same call again gives the same bits (fixed split order)
    out2, lse2, _ = P.csa_attend(q, kv, idx, win, sink, q_pos, want_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_attend_tiny_prefill_all_queries():
    w = S.WORKLOADS["tiny_csa_prefill_t2048"]
    inp = S.make_inputs(w, DEV)
    kI64 = _oracle_compress(inp, ("Ca_I", "Cb_I", "Za_I", "Zb_I"), 4, 64, rope=False)
    kv64 = _oracle_compress(inp, ("Ca", "Cb", "Za", "Zb"), 4, 128)
    inp["kI"] = _to_dev_bf16(kI64)
    inp["kv"] = _to_dev_bf16(kv64)
    pairs = [(0, t) for t in range(w.T)]
    idx_np = _oracle_topk(inp, 4, w.k, pairs)
    idx = torch.from_numpy(idx_np.astype(np.int32)).to(DEV)
    out, lse, _ = P.csa_attend(inp["q"], inp["kv"], idx, inp["win"], inp["sink"], inp["q_pos"], want_lse=True)
    torch.cuda.synchronize()
    ref, lref = _oracle_attend_rows(inp, idx_np, 4, w.window, pairs)
    assert_close(out[0], ref, "tiny prefill attend")
    assert_lse(lse[0], lref, "lse")


def test_attend_hca_decode_1m_full():
    w = S.WORKLOADS["hca_decode_1m_b8"]
    inp = S.make_inputs(w, DEV)
    out, lse, _ = P.hca_attend(inp["q"], inp["kv"], inp["win"], inp["sink"], inp["q_pos"], m=128, want_lse=True)
    torch.cuda.synchronize()
    pairs = [(b, 0) for b in range(w.B)]
    ref, lref = _oracle_attend_rows(inp, None, 128, w.window, pairs, dense=True)
    assert_close(out[:, 0], ref, "hca decode")
    assert_lse(lse[:, 0], lref, "lse")


def test_attend_hca_prefill_sampled():
    w = S.WORKLOADS["hca_prefill_t32768"]
    inp = S.make_inputs(w, DEV)
    kv = P.compress(inp["C"], inp["Z"], 128, theta=THETA)
    out, _, _ = P.hca_attend(inp["q"], kv, inp["win"], inp["sink"], inp["q_pos"], m=128)
    torch.cuda.synchronize()
    kv64 = O.compress(f64(inp["C"]), f64(inp["Z"]), 128, theta=THETA)
    assert_close(kv, kv64, "hca prefill compress")
    inp["kv"] = _to_dev_bf16(kv64)
    out2, _, _ = P.hca_attend(inp["q"], inp["kv"], inp["win"], inp["sink"], inp["q_pos"], m=128)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    ts = sorted(set([0, 1, 126, 127, 128, 129, 255, 256, 4095, w.T - 1] + rng.integers(0, w.T, 54).tolist()))
    pairs = [(0, t) for t in ts]
    ref, _ = _oracle_attend_rows(inp, None, 128, w.window, pairs, dense=True)
    assert_close(out2[0, ts], ref, "hca prefill attend (sampled)")


@pytest.mark.parametrize("flags,H", [((True, True), 32), ((False, False), 32), ((True, False), 32),
                                     ((True, True), 64), ((False, False), 128), ((True, False), 64)])
def test_attend_flags_and_edges(flags, H):
    """Small decode-like case: -1 pads, windows clipped at 0, ring wrap, sink, flags off, lse,
    with 32 heads (16 per CTA) and 64 / 128 heads (64 per CTA when the grid is large enough)."""
    qnr, unrot = flags
    B, d, N, k, Wcap = 3, 512, 300, 40, 160
    q = S.normal_bf16((B, 1, H, d), 11, 1, DEV)
    kv = S.normal_bf16((B, N, d), 11, 2, DEV)
    win = S.normal_bf16((B, Wcap, d), 11, 3, DEV)
    sink = (S.normal_f64((H,), 11, 4) * 3).float().to(DEV)
    q_pos = torch.tensor([[5], [1199], [1000]], dtype=torch.int32, device=DEV)   # t=5: window clipped
    rng = np.random.default_rng(0)
    idx_np = np.full((B, 1, k), -1)
    for b in range(B):
        nv = nvis_of(int(q_pos[b, 0]), 4, N)
        sel = rng.permutation(nv)[:k - 3]
        idx_np[b, 0, :sel.size] = sel
    idx = torch.from_numpy(idx_np.astype(np.int32)).to(DEV)
    out, lse, _ = P.csa_attend(q, kv, idx, win, sink, q_pos, q_norm_rope=qnr, out_unrotate=unrot, want_lse=True)
    torch.cuda.synchronize()
    inp = dict(q=q, kv=kv, win=win, sink=sink, q_pos=q_pos)
    ref, lref = _oracle_attend_rows(inp, idx_np, 4, 128, [(b, 0) for b in range(B)], q_norm_rope=qnr,
                                    out_unrotate=unrot)
    assert_close(out[:, 0], ref, f"flags {flags}")
    assert_lse(lse[:, 0], lref, "lse")


@pytest.mark.parametrize("H,d", [(16, 128), (64, 512)])
def test_attend_bad_index_is_reported_and_skipped(H, d):
    B, N, k = 1, 64, 8
    q = S.normal_bf16((B, 1, H, d), 12, 1, DEV)
    kv = S.normal_bf16((B, N, d), 12, 2, DEV)
    win = S.normal_bf16((B, 128, d), 12, 3, DEV)
    sink = torch.zeros(H, device=DEV)
    q_pos = torch.tensor([[256]], dtype=torch.int32, device=DEV)
    good = np.array([[[3, 9, 27, 40, 41, -1, 60, 2]]])
    bad = good.copy()
    bad[0, 0, 5] = N + 5
    out_b, _, ws = P.csa_attend(q, kv, torch.from_numpy(bad.astype(np.int32)).to(DEV), win, sink, q_pos)
    st, detail = C.csa_read_device_status(ws)
    assert st == C.CSA_ERR_DEVICE_CHECK and detail == N + 5
    out_g, _, ws2 = P.csa_attend(q, kv, torch.from_numpy(good.astype(np.int32)).to(DEV), win, sink, q_pos)
    assert C.csa_read_device_status(ws2)[0] == C.CSA_OK
    assert torch.equal(out_b, out_g)


def test_attend_prefill_rows_and_large_logits():
    """Prefill-shaped call (one split per query, 640 slots) where late entries have much larger
    logits, so the running maximum of the online softmax jumps between chunks.  The query is the
    oracle's own normalised and rotated q_hat rounded to bf16 and passed with the query
    preprocessing off, so both sides use identical logits and the comparison isolates the
    attention arithmetic."""
    B, T, H, d, N, k = 1, 96, 64, 512, 200, 512
    q_pos = (torch.arange(T, dtype=torch.int32) * 8 + 7)[None]
    q_raw = S.normal_f64((B, T, H, d), 13, 1).numpy()
    inv = O.rope_inv_freq(THETA, 64)
    qhat = np.stack([O.rope(O.rmsnorm(q_raw[0, t]), float(q_pos[0, t]), inv, 64) for t in range(T)])[None]
    q = _to_dev_bf16(qhat)
    kv64 = S.normal_f64((B, N, d), 13, 2, DEV)
    kv64[:, 150:] *= 4.0                              # late entries give much larger logits
    kv = S.f64_to_bf16(kv64)
    win = S.normal_bf16((B, 1024, d), 13, 3, DEV)     # ring of 1024 slots covers positions <= 767
    sink = S.normal_f64((H,), 13, 4).float().to(DEV)
    q_pos = q_pos.to(DEV)
    idx_np = np.full((B, T, k), -1, dtype=np.int32)
    for t in range(T):
        nv = nvis_of(int(q_pos[0, t]), 4, N)
        idx_np[0, t, :nv] = np.arange(nv)             # small logits first, the large ones chunks later
    idx = torch.from_numpy(idx_np).to(DEV)
    out, lse, _ = P.csa_attend(q, kv, idx, win, sink, q_pos, q_norm_rope=False, want_lse=True)
    torch.cuda.synchronize()
    inp = dict(q=q, kv=kv, win=win, sink=sink, q_pos=q_pos)
    ts = list(range(0, T, 5)) + [T - 1]
    ref, lref = _oracle_attend_rows(inp, idx_np, 4, 128, [(0, t) for t in ts], q_norm_rope=False)
    assert_close(out[0, ts], ref, "prefill rows, large logits")
    assert_lse(lse[0, ts], lref, "lse")


def test_attend_persistent_items_and_empty_rows():
    """Many more work items than CTAs (one CTA runs several queries and head groups in turn), two
    head groups, and queries that see no rows at all (t < 127 with no window: the output is zero
    and the LSE is the sink logit) interleaved with queries of up to 64 entries."""
    B, T, H, d, N, m = 1, 400, 128, 512, 64, 128
    rng = np.random.default_rng(17)
    ts = np.concatenate([np.arange(0, 40), rng.integers(0, N * m, T - 40)])
    rng.shuffle(ts)
    q_pos = torch.from_numpy(ts.astype(np.int32))[None].to(DEV)
    q = S.normal_bf16((B, T, H, d), 14, 1, DEV)
    kv = S.normal_bf16((B, N, d), 14, 2, DEV)
    win = S.normal_bf16((B, 128, d), 14, 3, DEV)
    sink = (S.normal_f64((H,), 14, 4) * 2).float().to(DEV)
    out, lse, ws = P.hca_attend(q, kv, win, sink, q_pos, m=m, window=0, want_lse=True)
    torch.cuda.synchronize()
    assert C.csa_read_device_status(ws)[0] == C.CSA_OK
    inp = dict(q=q, kv=kv, win=win, sink=sink, q_pos=q_pos)
    pick = sorted(set(rng.integers(0, T, 60).tolist()) | {int(np.argmin(ts)), int(np.argmax(ts))})
    ref, lref = _oracle_attend_rows(inp, None, m, 0, [(0, t) for t in pick], dense=True)
    assert_close(out[0, pick], ref, "persistent items")
    assert_lse(lse[0, pick], lref, "lse")
    empty = [i for i in range(T) if ts[i] < m - 1]
    assert torch.count_nonzero(out[0, empty]) == 0
    assert torch.equal(lse[0, empty], sink[None].expand(len(empty), H))


def test_attend_decode_splits_with_empty_splits():
    """Decode with fixed 512-slot splits where short contexts leave later splits without rows
    (their partials are empty and the merge skips them)."""
    B, H, d, N, m = 6, 64, 512, 2048, 128
    q_pos = torch.tensor([[200], [70000], [N * m - 1], [5000], [130], [N * m - 300]], dtype=torch.int32, device=DEV)
    q = S.normal_bf16((B, 1, H, d), 15, 1, DEV)
    kv = S.normal_bf16((B, N, d), 15, 2, DEV)
    win = S.normal_bf16((B, 128, d), 15, 3, DEV)
    sink = S.normal_f64((H,), 15, 4).float().to(DEV)
    out, lse, ws = P.hca_attend(q, kv, win, sink, q_pos, m=m, want_lse=True)
    torch.cuda.synchronize()
    assert C.csa_read_device_status(ws)[0] == C.CSA_OK
    inp = dict(q=q, kv=kv, win=win, sink=sink, q_pos=q_pos)
    ref, lref = _oracle_attend_rows(inp, None, m, 128, [(b, 0) for b in range(B)], dense=True)
    assert_close(out[:, 0], ref, "decode with empty splits")
    assert_lse(lse[:, 0], lref, "lse")


# ------------------------------------------------------------------------------------------------ whole path

def test_prefill_chain_small_end_to_end():
    """compress -> index/top-k -> attend on the GPU against the same chain in the oracle (which
    stores its compressed caches in bf16).  Top-k sets follow the near-tie rule; outputs are
    compared on every query whose selected set matches the oracle's exactly."""
    w = S.scaled(S.WORKLOADS["csa_prefill_t65536"], T=2048, N=512)
    inp = S.make_inputs(w, DEV)
    kv = P.compress(inp["Ca"], inp["Za"], 4, Cb=inp["Cb"], Zb=inp["Zb"], theta=THETA)
    kI = P.compress(inp["Ca_I"], inp["Za_I"], 4, Cb=inp["Cb_I"], Zb=inp["Zb_I"], rope=False, rope_dims=0)
    idx = P.index_topk(inp["qI"], inp["w"], kI, inp["q_pos"], 4, w.k)
    out, _, _ = P.csa_attend(inp["q"], kv, idx, inp["win"], inp["sink"], inp["q_pos"])
    torch.cuda.synchronize()
    kv64 = O.bf16_to_f64(O.bf16_round(_oracle_compress(inp, ("Ca", "Cb", "Za", "Zb"), 4, 512)))
    kI64 = O.bf16_to_f64(O.bf16_round(_oracle_compress(inp, ("Ca_I", "Cb_I", "Za_I", "Zb_I"), 4, 128, rope=False)))
    rng = np.random.default_rng(1)
    ts = sorted(set([0, 3, 4, 127, 128, 2047] + rng.integers(0, w.T, 40).tolist()))
    qpos = inp["q_pos"].cpu().numpy()
    sc = O.index_scores(f64(inp["qI"][:, ts]), f64(inp["w"][:, ts]), kI64, [qpos[0, ts]], 4)
    sel = O.topk_select(sc, [qpos[0, ts]], 4, w.k)
    gi = idx.cpu().numpy()
    same = []
    for j, t in enumerate(ts):
        nv = nvis_of(t, 4, w.N)
        n = check_topk_row(gi[0, t], sc[0, j, :nv], nv, w.k, f"chain t{t}")
        if n == 0:
            same.append((j, t))
    assert len(same) >= len(ts) // 2
    for j, t in same:
        o, _ = O.attend_query(f64(inp["q"][0, t]), t, kv64[0], sel[0, j], f64(inp["win"][0]), 128,
                              f64(inp["sink"]), theta=THETA)
        assert_close(out[0, t], o, f"chain attend t{t}")


def test_batch_invariance_and_determinism():
    """The same sequence decoded alone or inside a batch of 32 gives bit-identical indices and
    outputs; two runs are bit-identical."""
    w = S.WORKLOADS["csa_decode_128k_b32"]
    inp = S.make_inputs(S.scaled(w, B=8, N=8192), DEV)
    args = (inp["qI"], inp["w"], inp["kI"], inp["q_pos"], 4, 512)
    idx_a = P.index_topk(*args)
    idx_b = P.index_topk(*args)
    out_a, _, _ = P.csa_attend(inp["q"], inp["kv"], idx_a, inp["win"], inp["sink"], inp["q_pos"])
    out_b, _, _ = P.csa_attend(inp["q"], inp["kv"], idx_a, inp["win"], inp["sink"], inp["q_pos"])
    assert torch.equal(idx_a, idx_b) and torch.equal(out_a, out_b)
    b = 5
    one = lambda t: t[b:b + 1].contiguous()
    idx_1 = P.index_topk(one(inp["qI"]), one(inp["w"]), one(inp["kI"]), one(inp["q_pos"]), 4, 512)
    out_1, _, _ = P.csa_attend(one(inp["q"]), one(inp["kv"]), idx_1, one(inp["win"]), inp["sink"], one(inp["q_pos"]))
    assert torch.equal(idx_1[0], idx_a[b]) and torch.equal(out_1[0], out_a[b])


def test_gpu_path_is_causal():
    """Perturbing every input after position t leaves outputs at positions <= t bit-identical."""
    w = S.WORKLOADS["tiny_csa_prefill_t2048"]
    inp = S.make_inputs(w, DEV)

    def run(d):
        kv = P.compress(d["Ca"], d["Za"], 4, Cb=d["Cb"], Zb=d["Zb"], theta=THETA)
        kI = P.compress(d["Ca_I"], d["Za_I"], 4, Cb=d["Cb_I"], Zb=d["Zb_I"], rope=False, rope_dims=0)
        idx = P.index_topk(d["qI"], d["w"], kI, d["q_pos"], 4, w.k)
        return P.csa_attend(d["q"], kv, idx, d["win"], d["sink"], d["q_pos"])[0]

    ref = run(inp)
    t = 1234
    pert = {k: v.clone() for k, v in inp.items()}
    for k in ("Ca", "Cb", "Za", "Zb", "Ca_I", "Cb_I", "Za_I", "Zb_I", "q", "qI", "w", "win"):
        x = pert[k]
        x[:, t + 1:] = (torch.randn_like(x[:, t + 1:].float()) * 3).to(x.dtype)
    out = run(pert)
    assert torch.equal(out[:, :t + 1], ref[:, :t + 1])
    assert not torch.equal(out[:, t + 1:], ref[:, t + 1:])


def _prefill_sample_ts(T, n, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 3, 4, 5, 127, 128, 2047, 2048, 4095, 4096, T // 2, T - 2, T - 1]
    return sorted(set(fixed + rng.integers(0, T, n).tolist()))


def test_index_topk_prefill_65536_sampled():
    """Full 65536-token chunk through the chunked score workspace; sampled queries checked."""
    w = S.WORKLOADS["csa_prefill_t65536"]
    ist = {n: S.normal_bf16((1, w.T, w.dI), w.seed, S.TID[n], DEV) for n in ("Ca_I", "Cb_I", "Za_I", "Zb_I")}
    kI64 = _oracle_compress(ist, ("Ca_I", "Cb_I", "Za_I", "Zb_I"), 4, 128, rope=False)
    kI = _to_dev_bf16(kI64)
    qI = S.normal_bf16((1, w.T, w.nI, w.dI), w.seed, S.TID["qI"], DEV)
    wt = S.uniform_f64((1, w.T, w.nI), w.seed, S.TID["w"], DEV).float()
    q_pos = torch.arange(w.T, dtype=torch.int32, device=DEV)[None]
    idx = P.index_topk(qI, wt, kI, q_pos, 4, w.k)
    torch.cuda.synchronize()
    ts = _prefill_sample_ts(w.T, 40, 3)
    kb = O.bf16_to_f64(O.bf16_round(kI64))
    sc = O.index_scores(f64(qI[:, ts]), f64(wt[:, ts]), kb, [ts], 4)
    gi = idx.cpu().numpy()
    for j, t in enumerate(ts):
        nv = nvis_of(t, 4, w.N)
        check_topk_row(gi[0, t], sc[0, j, :nv], nv, w.k, f"prefill topk t{t}")


def test_attend_prefill_65536_sampled():
    """Full 65536-query sparse attention launch; sampled queries carry the oracle's top-k rows."""
    w = S.WORKLOADS["csa_prefill_t65536"]
    st = {n: S.normal_bf16((1, w.T, w.d), w.seed, S.TID[n], DEV) for n in ("Ca", "Cb", "Za", "Zb")}
    kv64 = _oracle_compress(st, ("Ca", "Cb", "Za", "Zb"), 4, 512)
    del st
    kv = _to_dev_bf16(kv64)
    q = S.normal_bf16((1, w.T, w.H, w.d), w.seed, S.TID["q"], DEV)
    win = S.normal_bf16((1, w.T, w.d), w.seed, S.TID["win"], DEV)
    sink = S.normal_f64((w.H,), w.seed, S.TID["sink"], DEV).float()
    q_pos = torch.arange(w.T, dtype=torch.int32, device=DEV)[None]
    ts = _prefill_sample_ts(w.T, 24, 4)
    rng = np.random.default_rng(9)
    nv_all = np.minimum(w.N, (np.arange(w.T) + 1) // 4)
    cols = np.arange(w.k)[None, :]
    idx_np = np.where(cols < nv_all[:, None], (cols * 7919) % np.maximum(nv_all[:, None], 1), -1).astype(np.int32)
    idx_np = idx_np[None]
    for t in ts:
        nv = nvis_of(t, 4, w.N)
        sel = rng.permutation(nv)[:w.k]
        idx_np[0, t] = -1
        idx_np[0, t, :sel.size] = sel
    idx = torch.from_numpy(idx_np).to(DEV)
    out, _, _ = P.csa_attend(q, kv, idx, win, sink, q_pos)
    torch.cuda.synchronize()
    inp = dict(q=q, kv=kv, win=win, sink=sink, q_pos=q_pos)
    ref, _ = _oracle_attend_rows(inp, idx_np, 4, w.window, [(0, t) for t in ts])
    assert_close(out[0, ts], ref, "prefill attend T=65536 (sampled)")
