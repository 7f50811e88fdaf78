"""BF16 index scores: the indexer variant whose scores are held in BF16 for a faster top-k selector
("DeepSeek-V4 技术报告深度解读" 5.4; the indexer QK-path row of "DeepSeek V4 模型技术大全").

The scores are the fp32 scores rounded to bf16 (checked bit for bit against torch's rounding of
the fp32 path, which is itself checked against the oracle); the selection is checked against the
oracle's own rounded scores (oracle.round_scores_bf16 + topk_select), allowing differences only
among entries whose oracle score lies within one bf16 step of the k-th rounded score (where the
fp32 and fp64 sums may round to different neighbours); recall against the fp32 selection is
reported on the 128K decode batch."""
import numpy as np
import pytest
import torch

from long_context_compressed_16_b300 import capi as C
from long_context_compressed_16_b300 import pipeline as P
from long_context_compressed_16_b300 import synth as S
from oracle import csa_oracle as O
from tests.helpers import f64, nvis_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(B, Tq, N, nI, dI, seed):
    qI = S.normal_bf16((B, Tq, nI, dI), seed, S.TID["qI"], DEV)
    w = S.uniform_f64((B, Tq, nI), seed, S.TID["w"], DEV).float()
    kI = S.normal_bf16((B, N, dI), seed, S.TID["kI"], DEV)
    q_pos = (4 * N - 4 * Tq + 4 * torch.arange(Tq, dtype=torch.int32, device=DEV)).repeat(B, 1).contiguous()
    q_pos[0, 0] = 6                                            # a short row
    return qI, w, kI, q_pos


def _scores(desc, qI, w, kI, q_pos):
    ws = torch.zeros(max(256, C.csa_index_score_workspace(desc)), dtype=torch.uint8, device=DEV)
    sc = torch.full((desc.B, desc.Tq, desc.N), float("nan"), dtype=torch.float32, device=DEV)
    C.check(C.csa_index_score(desc, qI, w, kI, None, q_pos, sc, ws), "csa_index_score")
    return sc


def _bf16_step(x):
    """Spacing of bf16 values at |x| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return 2.0 ** (e - 7)


@pytest.mark.parametrize("B,Tq,N,nI,dI", [(32, 1, 32768, 64, 128), (1, 130, 3000, 64, 128), (2, 9, 777, 20, 64)])
def test_bf16_scores_are_the_fp32_scores_rounded(B, Tq, N, nI, dI):
    qI, w, kI, q_pos = _inputs(B, Tq, N, nI, dI, 31)
    s32 = _scores(P.index_desc(B, Tq, N, nI, dI, 64, 4), qI, w, kI, q_pos)
    s16 = _scores(P.index_desc(B, Tq, N, nI, dI, 64, 4, bf16_scores=True), qI, w, kI, q_pos)
    torch.cuda.synchronize()
    nv = torch.clamp((q_pos.long() + 1) // 4, max=N)
    vis = torch.arange(N, device=DEV)[None, None, :] < nv[..., None]
    assert torch.equal(s16[vis], s32[vis].to(torch.bfloat16).float())
    assert torch.all(torch.isnan(s16[~vis]))                   # invisible entries untouched


@pytest.mark.parametrize("B,Tq,N,nI,dI,k", [
    (4, 1, 32768, 64, 128, 512),       # decode rows (cluster selection)
    (1, 64, 2000, 64, 128, 512),       # prefill-like rows, one CTA each
    (2, 5, 777, 16, 64, 40),           # ragged
    (2, 1, 75000, 64, 128, 1024),      # rows of several slices
])
def test_bf16_topk_against_oracle(B, Tq, N, nI, dI, k):
    qI, w, kI, q_pos = _inputs(B, Tq, N, nI, dI, 32)
    idx = P.index_topk(qI, w, kI, q_pos, 4, k, bf16_scores=True)
    # the fused call and the two split calls agree bit for bit
    desc = P.index_desc(B, Tq, N, nI, dI, k, 4, bf16_scores=True)
    sc = _scores(desc, qI, w, kI, q_pos)
    ws = torch.zeros(max(256, C.csa_topk_workspace(desc)), dtype=torch.uint8, device=DEV)
    idx2 = torch.full_like(idx, -7)
    C.check(C.csa_topk(desc, sc, q_pos, idx2, ws), "csa_topk")
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2)
    qpos = q_pos.cpu().numpy()
    gi = idx.cpu().numpy()
    rows = [(b, t) for b in range(B) for t in range(Tq)][:12]
    for b, t in rows:
        nv = nvis_of(qpos[b, t], 4, N)
        ref = O.index_scores(f64(qI[b:b + 1, t:t + 1]), f64(w[b:b + 1, t:t + 1]), f64(kI[b:b + 1]), [[qpos[b, t]]], 4)
        r16 = O.round_scores_bf16(ref)
        g = gi[b, t]
        if nv <= k:
            assert sorted(g[:nv].tolist()) == list(range(nv)) and np.all(g[nv:] == -1)
            continue
        sel = set(O.topk_select(r16, [[qpos[b, t]]], 4, k)[0, 0].tolist())
        scores = r16[0, 0, :nv]
        order = np.lexsort((np.arange(nv), -scores))
        ik = scores[order[k - 1]]
        assert len(set(g.tolist())) == k and np.all((g >= 0) & (g < nv))
        for s in set(g.tolist()) ^ sel:
            # only entries whose fp64 score sits within one bf16 step of the k-th rounded score
            assert abs(ref[0, 0, s] - ik) <= _bf16_step(ik), (b, t, s, ref[0, 0, s], ik)


def test_bf16_scores_recall_on_decode_128k():
    """Recall of the BF16-score selection against the fp32 selection on the 128K decode batch (the
    pages report 99.7% recall of KV entries)."""
    wl = S.WORKLOADS["csa_decode_128k_b32"]
    inp = S.make_inputs(wl, DEV)
    a = P.index_topk(inp["qI"], inp["w"], inp["kI"], inp["q_pos"], 4, wl.k)
    b = P.index_topk(inp["qI"], inp["w"], inp["kI"], inp["q_pos"], 4, wl.k, bf16_scores=True)
    torch.cuda.synchronize()
    hits = sum(len(set(a[i, 0].tolist()) & set(b[i, 0].tolist())) for i in range(wl.B))
    recall = hits / (wl.B * wl.k)
    print(f"bf16-score recall@{wl.k} against fp32 scores: {recall:.4f}")
    assert recall >= 0.97
