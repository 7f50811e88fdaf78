"""Host logic of the hybrid KV cache (no GPU): the closed-prefix split, which entries close in a
chunk, and csa_cache_append's argument checks (calls that fail validation launch nothing)."""
import json
import os

import pytest

from long_context_compressed_16_b300 import capi as C
from long_context_compressed_16_b300.cache import closed_prefix, closing_entries

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")


def _case(cid):
    with open(GOLDEN) as f:
        return next(c for c in json.load(f)["cases"] if c["id"] == cid)


def test_closed_prefix_worked_example():
    c = _case("closed_prefix_P1000")
    assert closed_prefix(c["P"], 4, c["m_hca"]) == (c["P_closed"], c["tau"])


@pytest.mark.parametrize("cid", ["lcm_block_entries", "vllm_block_256"])
def test_entries_per_logical_block(cid):
    c = _case(cid)
    assert len(closing_entries(0, c["tokens"], c["m_csa"])) == c["csa_entries"]
    assert len(closing_entries(0, c["tokens"], c["m_hca"])) == c["hca_entries"]
    # a logical block of lcm tokens is itself a closed prefix
    assert closed_prefix(c["tokens"], c["m_csa"], c["m_hca"]) == (c["tokens"], 0)


def test_closed_prefix_properties():
    for P in range(0, 3000, 7):
        closed, tau = closed_prefix(P)
        assert closed + tau == P and 0 <= tau < 128 and closed % 4 == 0 and closed % 128 == 0
        # nothing longer on a common boundary of both ratios fits in P
        assert not any(q % 4 == 0 and q % 128 == 0 for q in range(closed + 1, P + 1))
    assert closed_prefix(12, 4, 6) == (12, 0) and closed_prefix(23, 4, 6) == (12, 11)
    with pytest.raises(ValueError):
        closed_prefix(-1)


def test_closing_entries_brute_force():
    for m in (1, 3, 4, 128):
        for t0 in range(0, 300, 13):
            for n in (0, 1, 2, 5, 128, 131):
                brute = [(u + 1) // m - 1 for u in range(t0, t0 + n) if (u + 1) % m == 0]
                assert list(closing_entries(t0, n, m)) == brute


FAKE = 1 << 20   # 16-byte aligned address that is never dereferenced: every case below is rejected


def _desc(**kw):
    base = dict(B=2, d=512, dI=128, m=4, overlap=1, Wcap=128, N_cap=256, rope_dims=64, rope_theta=160000.0,
                inv_freq=None, eps=1e-6, flags=C.CSA_COMPRESS_NORM | C.CSA_COMPRESS_ROPE,
                index_flags=C.CSA_COMPRESS_NORM)
    base.update(kw)
    return C.csa_cache_desc(**base)


def test_cache_state_bytes():
    # CSA: 8 rings of [B, 2m, width] bf16 (4 of width d, 4 of width dI)
    assert C.csa_cache_state_bytes(_desc()) == 4 * 2 * 8 * 512 * 2 + 4 * 2 * 8 * 128 * 2
    assert C.csa_cache_state_bytes(_desc(dI=0)) == 4 * 2 * 8 * 512 * 2
    # HCA: two rings of [B, m', d]
    assert C.csa_cache_state_bytes(_desc(dI=0, m=128, overlap=0)) == 2 * 2 * 128 * 512 * 2
    # ring sizes round up to 256 bytes each
    assert C.csa_cache_state_bytes(_desc(B=1, d=64, dI=0, m=1, rope_dims=0)) == 4 * 256
    for bad in (dict(d=100), dict(d=384), dict(dI=96), dict(dI=192), dict(m=0), dict(Wcap=0), dict(overlap=0),   # indexer needs overlap
                dict(index_flags=C.CSA_COMPRESS_ROPE), dict(rope_dims=6), dict(eps=-1.0)):
        assert C.csa_cache_state_bytes(_desc(**bad)) == 0, bad


def test_cache_append_validation():
    rows = {k: FAKE for k in ("Ca", "Cb", "Za", "Zb", "Ca_I", "Cb_I", "Za_I", "Zb_I", "win")}
    bufs = {k: FAKE for k in ("kv", "kI", "win", "state")}
    call = lambda desc, t0=0, n=4, r=rows, b=bufs, p=None: C.csa_cache_append(desc, t0, n, r, p, b, stream=0)
    assert call(_desc(), n=0) == C.CSA_OK                       # nothing to append: no launch
    assert call(_desc(B=0)) == C.CSA_OK
    assert call(_desc(), t0=-1) == C.CSA_ERR_INVALID_ARG
    assert call(_desc(), n=-1) == C.CSA_ERR_INVALID_ARG
    assert call(_desc(N_cap=1), t0=4, n=4) == C.CSA_ERR_INVALID_ARG   # entry 1 does not fit
    assert call(_desc(), t0=2 ** 31 - 2, n=4) == C.CSA_ERR_INVALID_ARG
    assert call(_desc(d=96)) == C.CSA_ERR_UNSUPPORTED
    assert call(_desc(overlap=0)) == C.CSA_ERR_UNSUPPORTED         # indexer keys without overlap
    assert call(_desc(index_flags=C.CSA_COMPRESS_ROPE)) == C.CSA_ERR_UNSUPPORTED
    assert call(_desc(), r={**rows, "Zb_I": None}) == C.CSA_ERR_INVALID_ARG
    assert call(_desc(), r={**rows, "win": FAKE + 8}) == C.CSA_ERR_INVALID_ARG
    assert call(_desc(), b={**bufs, "state": None}) == C.CSA_ERR_INVALID_ARG
    assert call(_desc(), b={**bufs, "kI": None}) == C.CSA_ERR_INVALID_ARG
    assert call(_desc(), p={"gamma": FAKE + 4}) == C.CSA_ERR_INVALID_ARG
    assert C.lib.csa_cache_append(None, 0, 1, None, None, None, None) == C.CSA_ERR_INVALID_ARG
