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


def _case(B, N, nI, dI, k, seed, fp8):
    dev = "cuda"
    qI = S.normal_bf16((B, 1, nI, dI), seed, S.TID["qI"], dev)
    w = S.uniform_f64((B, 1, nI), seed, S.TID["w"], dev).float()
    if fp8:
        codes, scale = S.quantize_rows_e4m3(S.normal_f64((B, N, dI), seed, S.TID["kI"], dev))
        kI, kI_scale = codes, scale
    else:
        kI, kI_scale = S.normal_bf16((B, N, dI), seed, S.TID["kI"], dev), None
    q_pos = torch.full((B, 1), 4 * N, dtype=torch.int32, device=dev)
    q_pos[0, 0] = 4 * (N // 3)                                    # a shorter visible prefix
    return qI, w, kI, kI_scale, q_pos


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_twice_in_a_row():
    cases = [dict(B=4, N=20000, nI=64, dI=128, k=512, seed=21, fp8=False),
             dict(B=3, N=9000, nI=32, dI=128, k=256, seed=22, fp8=True)]
    for c in cases:
        qI, w, kI, kI_scale, q_pos = _case(c["B"], c["N"], c["nI"], c["dI"], c["k"], c["seed"], c["fp8"])
        desc = P.index_desc(c["B"], 1, c["N"], c["nI"], c["dI"], c["k"], 4, fp8=c["fp8"])
        assert C.csa_index_topk_workspace(desc) <= C.CSA_NOALLOC_SCRATCH_BYTES
        ws = torch.zeros(C.csa_index_topk_workspace(desc), dtype=torch.uint8, device="cuda")
        ref = torch.full((c["B"], 1, c["k"]), -7, dtype=torch.int32, device="cuda")
        got = torch.full_like(ref, -7)
        C.check(C.csa_index_topk(desc, qI, w, kI, kI_scale, q_pos, ref, None, ws), "csa_index_topk")
        C.check(C.csa_index_topk_noalloc(desc, qI, w, kI, kI_scale, q_pos, got, None), "csa_index_topk_noalloc")
        torch.cuda.synchronize()
        assert torch.equal(got, ref), c
        assert int((ref >= 0).sum()) == c["B"] * c["k"]
