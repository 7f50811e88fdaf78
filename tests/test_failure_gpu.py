"""Failure detection without a GPU fault: a bounded device-side wait that nothing satisfies must
give up, report CSA_ERR_TIMEOUT through the workspace status word and leave the context usable."""
import pytest
import torch

from long_context_compressed_16_b300 import capi as C
from long_context_compressed_16_b300 import pipeline as P
from long_context_compressed_16_b300 import synth as S


def test_selftest_argument_checks_without_launch():
    assert C.lib.csa_selftest_bounded_wait(None, 256, 10_000_000, None) == C.CSA_ERR_WORKSPACE
    assert C.lib.csa_selftest_bounded_wait(0x10000, 100, 10_000_000, None) == C.CSA_ERR_WORKSPACE
    assert C.lib.csa_selftest_bounded_wait(0x10000, 256, 10, None) == C.CSA_ERR_INVALID_ARG
    assert C.lib.csa_selftest_bounded_wait(0x10000, 256, 3_000_000_000, None) == C.CSA_ERR_INVALID_ARG
    assert C.lib.csa_selftest_bounded_wait(0x10008, 256, 10_000_000, None) == C.CSA_ERR_INVALID_ARG


@pytest.mark.gpu
def test_unsatisfied_wait_times_out_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    limit_ms = 20
    C.check(C.csa_selftest_bounded_wait(ws, limit_ms * 1_000_000), "selftest")
    st, detail_us = C.csa_read_device_status(ws)
    assert st == C.CSA_ERR_TIMEOUT
    assert limit_ms * 1000 <= detail_us < 2_000_000
    # the status word is sticky until cleared, and the context still runs work correctly
    C.check(C.csa_clear_device_status(ws), "clear")
    assert C.csa_read_device_status(ws)[0] == C.CSA_OK
    qI = S.normal_bf16((1, 1, 16, 64), 9, 1, "cuda")
    kI = S.normal_bf16((1, 64, 64), 9, 2, "cuda")
    w = torch.ones((1, 1, 16), device="cuda")
    q_pos = torch.full((1, 1), 4 * 64, dtype=torch.int32, device="cuda")
    sc = torch.empty((1, 1, 64), dtype=torch.float32, device="cuda")
    idx = P.index_topk(qI, w, kI, q_pos, 4, 8, score_out=sc)
    torch.cuda.synchronize()
    ref = torch.relu(kI[0].float() @ qI[0, 0].float().T).sum(1)
    assert torch.allclose(sc[0, 0], ref, rtol=1e-5, atol=1e-4)
    assert sorted(idx[0, 0].tolist()) == sorted(torch.topk(sc[0, 0], 8).indices.tolist())
