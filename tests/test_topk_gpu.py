"""GPU parity of the top-k selection on rows split over several slices, where one thread-block
cluster selects a row (csa_topk on given scores).  Integer-valued scores make ties common, also
across slice boundaries, so the tie rule (smaller entry index first) decides many rows; the
visible counts put the end of the row everywhere: none, fewer than k, inside a slice, and on a
slice boundary.  The expected set is the oracle's; the library writes it in increasing index."""
import numpy as np
import pytest
import torch

from long_context_compressed_16_b300 import capi as C
from long_context_compressed_16_b300 import pipeline as P
from oracle import csa_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _expected(scores, q_pos, m, k):
    sel = O.topk_select(scores[None], [q_pos], m, k)[0]
    out = np.full_like(sel, -1)
    for t in range(sel.shape[0]):
        s = np.sort(sel[t][sel[t] >= 0])
        out[t, :s.size] = s
    return out


@pytest.mark.parametrize("Q,N,k,levels", [
    (8, 20000, 300, 50),       # 5 slices of 4096: a cluster of five CTAs, heavy ties
    (32, 32768, 512, 1000),    # the decode shape: 4 slices
    (6, 24576, 2048, 7),       # largest k, only 7 distinct values: the threshold bin is huge
    (2, 100000, 1024, 300),    # long rows: 13 two-stage slices re-cut into a cluster of 7
])
def test_topk_cluster_rows_with_ties(Q, N, k, levels):
    m = 4
    rng = np.random.default_rng(N + k)
    scores = rng.integers(0, levels, size=(Q, N)).astype(np.float32)
    scores[0, :] = 1.0                                    # one row where every score ties
    nv = [N, 0, k - 3, 4096 + 17, 8192, N - 1, 3 * 4096 - 1, 12345]   # visible entries per query
    nv = (nv * (Q // len(nv) + 1))[:Q]
    q_pos = np.array([max(0, v * m) for v in nv], dtype=np.int32)    # n_visible(t) = (t + 1) // m = v
    st = torch.from_numpy(scores).to(DEV).view(1, Q, N)
    qp = torch.from_numpy(q_pos).to(DEV).view(1, Q)
    desc = P.index_desc(1, Q, N, 1, 64, k, m)
    idx = torch.empty((1, Q, k), dtype=torch.int32, device=DEV)
    ws = torch.zeros(max(256, C.csa_topk_workspace(desc)), dtype=torch.uint8, device=DEV)
    C.check(C.csa_topk(desc, st, qp, idx, ws), "csa_topk")
    st_, det = C.csa_read_device_status(ws)
    assert st_ == C.CSA_OK, (st_, det)
    got = idx[0].cpu().numpy()
    exp = _expected(scores, q_pos, m, k)
    for t in range(Q):
        assert np.array_equal(got[t], exp[t]), f"row {t} (visible {O.n_visible(q_pos[t], m, N)})"
