"""Fused prefill indexer + streaming top-k.

On prefill batches csa_index_topk selects inside the score kernel ("DeepSeek V4 模型技术大全",
CSA path: the I_{t,s} and TopK equations; the fused-indexer row of "DeepSeek-V4 技术报告深度解读"
5.4): the epilogue keeps, per query, every entry that can still be among its top k (a running
lower bound of the k-th score), and the CTA's selector warps select the exact top k from that
list; the score rows are never stored.  The selection is exact, so the result must equal, bit for
bit, the unfused path (csa_index_score, then csa_topk on the stored rows), which the oracle pins in
test_parity_gpu; a few rows per case are also checked against the oracle directly.

The cases force the fused path (select_mode CSA_SELECT_FUSED) on shapes small enough to check
quickly; CSA_SELECT_AUTO takes it only for rows of at least 16 k entries, which one test checks.
The cases reach both selector paths: the common one (the class of the k-th key holds few keys:
resolve only that class) and the general radix select over the whole list (heavy ties, or keys
that climb past the histogram's range), plus rows with nothing visible (groups the score kernel
skips), rows shorter than k, ragged groups, k = 2048, BF16 scores and the low-precision indexer."""
import numpy as np
import pytest
import torch

from long_context_compressed_16_b300 import capi as C
from long_context_compressed_16_b300 import pipeline as P
from long_context_compressed_16_b300 import synth as S
from oracle import csa_oracle as O
from tests.helpers import check_topk_row, f64, nvis_of

pytestmark = pytest.mark.gpu
DEV = "cuda"
M = 4


def _unfused(desc, qI, w, kI, kI_scale, q_pos):
    ws = torch.zeros(max(256, C.csa_index_score_workspace(desc), C.csa_topk_workspace(desc)), dtype=torch.uint8,
                     device=DEV)
    sc = torch.full((desc.B, desc.Tq, desc.N), float("nan"), dtype=torch.float32, device=DEV)
    C.check(C.csa_index_score(desc, qI, w, kI, kI_scale, q_pos, sc, ws), "csa_index_score")
    idx = torch.full((desc.B, desc.Tq, desc.k), -7, dtype=torch.int32, device=DEV)
    C.check(C.csa_topk(desc, sc, q_pos, idx, ws), "csa_topk")
    torch.cuda.synchronize()
    assert C.csa_read_device_status(ws)[0] == C.CSA_OK
    return idx


def _fused(desc, qI, w, kI, kI_scale, q_pos, expect_launches=None, fused=True):
    ws = torch.zeros(max(256, C.csa_index_topk_workspace(desc)), dtype=torch.uint8, device=DEV)
    idx = torch.full((desc.B, desc.Tq, desc.k), -7, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    n0 = C.csa_launch_count()
    C.check(C.csa_index_topk(desc, qI, w, kI, kI_scale, q_pos, idx, None, ws), "csa_index_topk")
    n1 = C.csa_launch_count()
    torch.cuda.synchronize()
    assert C.csa_read_device_status(ws)[0] == C.CSA_OK
    if expect_launches is not None:
        if fused:
            assert n1 - n0 == expect_launches, f"fused selection not taken ({n1 - n0} launches)"
        else:
            assert n1 - n0 >= 2, f"expected stored scores and a selector launch ({n1 - n0} launches)"
    return idx


def _causal_pos(B, Tq, N):
    """Prefill positions ending at the last closed block, plus rows that see nothing (a whole
    group at the start of sequence 0) and rows shorter than any k."""
    q_pos = (M * N - M * Tq + M * torch.arange(Tq, dtype=torch.int32, device=DEV)).repeat(B, 1).contiguous()
    q_pos[0, :8] = torch.tensor([0, 1, 2, 0, 1, 0, 2, 1], dtype=torch.int32)   # two groups: nothing visible
    q_pos[0, 8:12] = torch.tensor([6, 30, 100, 401], dtype=torch.int32)         # 1, 7, 25, 100 entries
    return q_pos


def _oracle_rows(B, Tq, n_rows, seed):
    rng = np.random.default_rng(seed)
    rows = [(int(b), int(t)) for b, t in zip(rng.integers(0, B, n_rows), rng.integers(0, Tq, n_rows))]
    return rows + [(0, 0), (0, 9), (B - 1, Tq - 1)]


def _check_oracle(idx, qI, w, kI, q_pos, k, N, rows):
    qp = q_pos.cpu().numpy()
    gi = idx.cpu().numpy()
    kb = f64(kI)
    for b, t in rows:
        nv = nvis_of(qp[b, t], M, N)
        sc = O.index_scores(f64(qI[b:b + 1, t:t + 1]), f64(w[b:b + 1, t:t + 1]), kb[b:b + 1], [[qp[b, t]]], M)
        check_topk_row(gi[b, t], sc[0, 0, :nv], nv, k, f"fused topk b{b} t{t}")


@pytest.mark.parametrize("B,Tq,N,nI,dI,k,fused", [
    (1, 2560, 2000, 64, 128, 512, True),     # 640 groups of 4 queries, rows up to 2000 entries
    (3, 1001, 777, 64, 128, 100, True),      # ragged: the last group of every sequence holds 1 query
    (1, 2400, 1500, 64, 64, 256, True),      # 64-dim indexer heads
    (2, 1200, 5000, 64, 128, 2048, True),    # the largest k
    (1, 2400, 32768, 64, 128, 512, True),    # the longest rows the fused selection takes
    (1, 4800, 3000, 32, 128, 64, False),     # 32 heads (groups of 8 queries): stored scores + selector
    (1, 2400, 32769, 64, 128, 512, False),   # rows past the fused selection's bitmap: stored scores
])
def test_fused_select_equals_unfused(B, Tq, N, nI, dI, k, fused):
    qI = S.normal_bf16((B, Tq, nI, dI), 41, S.TID["qI"], DEV)
    w = S.uniform_f64((B, Tq, nI), 41, S.TID["w"], DEV).float()
    kI = S.normal_bf16((B, N, dI), 41, S.TID["kI"], DEV)
    q_pos = _causal_pos(B, Tq, N)
    desc = P.index_desc(B, Tq, N, nI, dI, k, M, select_mode=C.CSA_SELECT_FUSED)
    got = _fused(desc, qI, w, kI, None, q_pos, expect_launches=1, fused=fused)
    ref = _unfused(desc, qI, w, kI, None, q_pos)
    assert torch.equal(got, ref)
    assert torch.all(got[0, :8] == -1)                        # nothing visible
    _check_oracle(got, qI, w, kI, q_pos, k, N, _oracle_rows(B, Tq, 6, B * Tq))


def test_fused_select_heavy_ties():
    """Keys that repeat with period 3 (three distinct scores per query, each held by a third of
    the row): the k-th key's class holds more keys than the selector keeps in shared memory, so
    the whole list is radix-selected, ties going to the smaller entry.  All-zero queries (every
    score equal) keep exactly their first k entries."""
    B, Tq, N, nI, dI, k = 1, 2400, 3000, 64, 128, 512
    qI = S.normal_bf16((B, Tq, nI, dI), 43, S.TID["qI"], DEV)
    qI[0, 100:140] = 0
    w = S.uniform_f64((B, Tq, nI), 43, S.TID["w"], DEV).float()
    base = S.normal_bf16((B, 3, dI), 43, S.TID["kI"], DEV)
    kI = base[:, torch.arange(N, device=DEV) % 3].contiguous()
    q_pos = _causal_pos(B, Tq, N)
    desc = P.index_desc(B, Tq, N, nI, dI, k, M, select_mode=C.CSA_SELECT_FUSED)
    fused = _fused(desc, qI, w, kI, None, q_pos, expect_launches=1)
    ref = _unfused(desc, qI, w, kI, None, q_pos)
    assert torch.equal(fused, ref)
    # an all-zero query scores every entry 0: its top k are the first k entries
    t = 139
    nv = nvis_of(int(q_pos[0, t]), M, N)
    assert nv > k
    assert fused[0, t].tolist() == list(range(k))


def test_fused_select_climbing_scores():
    """Key rows scaled by 2^(s/48): the scores climb far above the first tile's range, so later
    keys pile into the histogram's top bin and the selector falls back to the general path."""
    B, Tq, N, nI, dI, k = 1, 2400, 1500, 64, 128, 300
    qI = S.normal_bf16((B, Tq, nI, dI), 44, S.TID["qI"], DEV)
    w = S.uniform_f64((B, Tq, nI), 44, S.TID["w"], DEV).float()
    kI0 = S.normal_bf16((B, N, dI), 44, S.TID["kI"], DEV).float()
    scale = torch.pow(2.0, torch.arange(N, device=DEV, dtype=torch.float32) / 48.0)
    kI = (kI0 * scale[None, :, None]).to(torch.bfloat16).contiguous()
    q_pos = _causal_pos(B, Tq, N)
    desc = P.index_desc(B, Tq, N, nI, dI, k, M, select_mode=C.CSA_SELECT_FUSED)
    fused = _fused(desc, qI, w, kI, None, q_pos, expect_launches=1)
    ref = _unfused(desc, qI, w, kI, None, q_pos)
    assert torch.equal(fused, ref)
    _check_oracle(fused, qI, w, kI, q_pos, k, N, _oracle_rows(B, Tq, 4, 7))


def test_fused_select_bf16_scores():
    B, Tq, N, nI, dI, k = 1, 2560, 2000, 64, 128, 512
    qI = S.normal_bf16((B, Tq, nI, dI), 45, S.TID["qI"], DEV)
    w = S.uniform_f64((B, Tq, nI), 45, S.TID["w"], DEV).float()
    kI = S.normal_bf16((B, N, dI), 45, S.TID["kI"], DEV)
    q_pos = _causal_pos(B, Tq, N)
    desc = P.index_desc(B, Tq, N, nI, dI, k, M, bf16_scores=True, select_mode=C.CSA_SELECT_FUSED)
    fused = _fused(desc, qI, w, kI, None, q_pos, expect_launches=1)
    ref = _unfused(desc, qI, w, kI, None, q_pos)
    assert torch.equal(fused, ref)


def test_fused_select_lowp():
    """Low-precision indexer (e4m3 keys with row scales, the query quantised per chunk)."""
    B, Tq, N, nI, dI, k = 1, 2560, 2000, 64, 128, 512
    qI = S.normal_bf16((B, Tq, nI, dI), 46, S.TID["qI"], DEV)
    w = S.uniform_f64((B, Tq, nI), 46, S.TID["w"], DEV).float()
    kf = S.normal_f64((B, N, dI), 46, S.TID["kI"], "cpu")
    kI8, kI_scale = S.quantize_rows_e4m3(kf)
    kI8, kI_scale = kI8.to(DEV), kI_scale.to(DEV)
    q_pos = _causal_pos(B, Tq, N)
    desc = P.index_desc(B, Tq, N, nI, dI, k, M, lowp=True, select_mode=C.CSA_SELECT_FUSED)
    fused = _fused(desc, qI, w, kI8, kI_scale, q_pos, expect_launches=2)   # query quantisation + scores
    ref = _unfused(desc, qI, w, kI8, kI_scale, q_pos)
    assert torch.equal(fused, ref)


def test_fused_select_is_deterministic_and_batch_invariant():
    """A query's row does not depend on the batch around it or on the run: the same sequence
    alone and as the second of two gives the same rows."""
    B, Tq, N, nI, dI, k = 2, 1400, 2500, 64, 128, 512
    qI = S.normal_bf16((B, Tq, nI, dI), 47, S.TID["qI"], DEV)
    w = S.uniform_f64((B, Tq, nI), 47, S.TID["w"], DEV).float()
    kI = S.normal_bf16((B, N, dI), 47, S.TID["kI"], DEV)
    q_pos = (M * N - M * Tq + M * torch.arange(Tq, dtype=torch.int32, device=DEV)).repeat(B, 1).contiguous()
    F = C.CSA_SELECT_FUSED
    a = P.index_topk(qI, w, kI, q_pos, M, k, select_mode=F)
    b = P.index_topk(qI, w, kI, q_pos, M, k, select_mode=F)
    # sequence 1 alone (350 groups: too few for the fused path, so stored scores and the
    # selector kernels) and inside the batch (700 groups: fused)
    c = P.index_topk(qI[1:].contiguous(), w[1:].contiguous(), kI[1:].contiguous(), q_pos[1:].contiguous(), M, k,
                     select_mode=F)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(a[1:], c)


@pytest.mark.parametrize("N,auto_fused", [(8192, True), (8191, False)])
def test_select_mode_auto_and_stored(N, auto_fused):
    """CSA_SELECT_AUTO fuses the selection for rows of at least 16 k entries (k = 512: N >= 8192),
    where it is faster, and stores the rows otherwise; CSA_SELECT_STORED always stores them.  All
    give the same rows."""
    B, Tq, nI, dI, k = 1, 2400, 64, 128, 512
    qI = S.normal_bf16((B, Tq, nI, dI), 48, S.TID["qI"], DEV)
    w = S.uniform_f64((B, Tq, nI), 48, S.TID["w"], DEV).float()
    kI = S.normal_bf16((B, N, dI), 48, S.TID["kI"], DEV)
    q_pos = _causal_pos(B, Tq, N)
    auto = _fused(P.index_desc(B, Tq, N, nI, dI, k, M), qI, w, kI, None, q_pos, expect_launches=1, fused=auto_fused)
    stored = _fused(P.index_desc(B, Tq, N, nI, dI, k, M, select_mode=C.CSA_SELECT_STORED), qI, w, kI, None, q_pos,
                    expect_launches=1, fused=False)
    forced = _fused(P.index_desc(B, Tq, N, nI, dI, k, M, select_mode=C.CSA_SELECT_FUSED), qI, w, kI, None, q_pos,
                    expect_launches=1, fused=True)
    assert torch.equal(auto, stored) and torch.equal(auto, forced)
