"""csa_index_topk_noalloc: the indexer + top-k call for callers that cannot allocate device memory.

Such callers (code running inside a host callback or an allocator hook, plug-ins that are handed
only their input and output buffers) cannot create the workspace that csa_index_topk needs, so
this variant uses a fixed scratch array that the library keeps in device memory.  These tests
check that it returns exactly what the workspace-taking call returns, on two calls in a row (the
second one sees the first one's leftovers in the shared array), and that requests larger than
the array are refused before any work is enqueued.

The file is named so that pytest collects it last."""
import ctypes

import pytest
import torch

from long_context_compressed_16_b300 import capi as C
from long_context_compressed_16_b300 import pipeline as P
from long_context_compressed_16_b300 import synth as S

FAKE = 0x10000   # an aligned address that host-side validation never dereferences


def test_noalloc_refuses_requests_beyond_the_scratch_array():
    big = P.index_desc(8, 1, 262144, 64, 128, 1024, 4)          # 8 MiB of scores + status word
    assert C.csa_index_topk_workspace(big) > C.CSA_NOALLOC_SCRATCH_BYTES
    st = C.lib.csa_index_topk_noalloc(ctypes.byref(big), FAKE, FAKE, FAKE, None, FAKE, FAKE, None, None)
    assert st == C.CSA_ERR_UNSUPPORTED
    bad = P.index_desc(2, 1, 1000, 64, 96, 64, 4)                # head_dim 96 is not supported
    st = C.lib.csa_index_topk_noalloc(ctypes.byref(bad), FAKE, FAKE, FAKE, None, FAKE, FAKE, None, None)
    assert st == C.CSA_ERR_INVALID_ARG


def _case(B, N, nI, dI, k, seed, fp8, Tq=1):
    dev = "cuda"
    qI = S.normal_bf16((B, Tq, nI, dI), seed, S.TID["qI"], dev)
    w = S.uniform_f64((B, Tq, nI), seed, S.TID["w"], dev).float()
    if fp8:
        codes, scale = S.quantize_rows_e4m3(S.normal_f64((B, N, dI), seed, S.TID["kI"], dev))
        kI, kI_scale = codes, scale
    else:
        kI, kI_scale = S.normal_bf16((B, N, dI), seed, S.TID["kI"], dev), None
    if Tq == 1:
        q_pos = torch.full((B, 1), 4 * N, dtype=torch.int32, device=dev)
        q_pos[0, 0] = 4 * (N // 3)                                # a shorter visible prefix
    else:
        # the last Tq tokens of a prefill chunk of 4 N tokens
        q_pos = (4 * N - Tq + torch.arange(Tq, dtype=torch.int32, device=dev)).repeat(B, 1).contiguous()
    return qI, w, kI, kI_scale, q_pos


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_twice_in_a_row():
    """Decode rows in the bf16, FP8 and low-precision key formats (the low-precision query and
    weight rows sit after the score rows in the scratch array), with and without score_out, and
    a prefill chunk whose workspace is close to the array's size: every call is compared bit for
    bit with csa_index_topk on a workspace of its own, twice in a row."""
    cases = [dict(B=4, N=20000, nI=64, dI=128, k=512, seed=21, fp8=False, lowp=False, Tq=1, scores=False),
             dict(B=3, N=9000, nI=32, dI=128, k=256, seed=22, fp8=True, lowp=False, Tq=1, scores=False),
             dict(B=4, N=30000, nI=64, dI=128, k=512, seed=23, fp8=True, lowp=True, Tq=1, scores=False),
             dict(B=2, N=12000, nI=64, dI=128, k=512, seed=24, fp8=False, lowp=False, Tq=1, scores=True),
             dict(B=1, N=4000, nI=64, dI=128, k=128, seed=25, fp8=False, lowp=False, Tq=512, scores=False)]
    for c in cases:
        qI, w, kI, kI_scale, q_pos = _case(c["B"], c["N"], c["nI"], c["dI"], c["k"], c["seed"], c["fp8"], c["Tq"])
        desc = P.index_desc(c["B"], c["Tq"], c["N"], c["nI"], c["dI"], c["k"], 4, fp8=c["fp8"], lowp=c["lowp"])
        need = C.csa_index_topk_workspace(desc)
        assert 0 < need <= C.CSA_NOALLOC_SCRATCH_BYTES
        if c["Tq"] > 1:
            assert need > 0.9 * C.CSA_NOALLOC_SCRATCH_BYTES, need      # the case is near the limit
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        shape = (c["B"], c["Tq"], c["k"])
        ref = torch.full(shape, -7, dtype=torch.int32, device="cuda")
        sc_ref = torch.full((c["B"], c["Tq"], c["N"]), -5.0, device="cuda") if c["scores"] else None
        C.check(C.csa_index_topk(desc, qI, w, kI, kI_scale, q_pos, ref, sc_ref, ws), "csa_index_topk")
        for rep in range(2):
            got = torch.full(shape, -7, dtype=torch.int32, device="cuda")
            sc = torch.full_like(sc_ref, -5.0) if c["scores"] else None
            C.check(C.csa_index_topk_noalloc(desc, qI, w, kI, kI_scale, q_pos, got, sc), "csa_index_topk_noalloc")
            torch.cuda.synchronize()
            assert torch.equal(got, ref), (c, rep)
            if c["scores"]:
                assert torch.equal(sc, sc_ref), (c, rep)
        assert int((ref >= 0).sum()) == c["B"] * c["Tq"] * c["k"]
