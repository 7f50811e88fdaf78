"""GPU parity of the hybrid KV cache (csa_cache_append): appending a sequence chunk by chunk (one
token at a time included) gives the entries the oracle computes from the whole sequence, and
bit for bit those of one whole-sequence csa_compress call; the window ring holds the last Wcap
rows; a prefix restored at its 128-token boundary and the tail appended again reproduces the
cache that never stopped."""
import numpy as np
import pytest
import torch

from long_context_compressed_16_b300 import pipeline as P
from long_context_compressed_16_b300 import synth as S
from long_context_compressed_16_b300.cache import LayerCache, closed_prefix
from oracle import csa_oracle as O
from tests.helpers import assert_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
THETA = 160000.0
CSA_STREAMS = ("Ca", "Cb", "Za", "Zb", "Ca_I", "Cb_I", "Za_I", "Zb_I")


def _chunks(T, seed):
    """Chunk lengths covering T tokens: single tokens, short odd runs, block-sized and long runs."""
    rng = np.random.default_rng(seed)
    out, t = [], 0
    menu = (1, 1, 1, 2, 3, 4, 5, 7, 8, 127, 128, 131)
    while t < T:
        n = min(int(rng.choice(menu)), T - t)
        out.append(n)
        t += n
    return out


def _inputs(kind, B, T, d, dI, seed):
    names = CSA_STREAMS if kind == "csa" else ("Ca", "Za")
    inp = {n: S.normal_bf16((B, T, dI if n.endswith("_I") else d), seed, S.TID[n], DEV) for n in names}
    inp["win"] = S.normal_bf16((B, T, d), seed, S.TID["win"], DEV)
    return inp


def _params(kind, d, dI, m, seed):
    g = torch.Generator().manual_seed(seed)
    p = {"bias_a": torch.randn(m, d, generator=g), "gamma": 1 + 0.1 * torch.randn(d, generator=g)}
    if kind == "csa":
        p.update(bias_b=torch.randn(m, d, generator=g), bias_a_I=torch.randn(m, dI, generator=g),
                 bias_b_I=torch.randn(m, dI, generator=g), gamma_I=1 + 0.1 * torch.randn(dI, generator=g))
    return {k: v.float().to(DEV) for k, v in p.items()}


def _fill(cache, inp, chunks, snapshots=None, t_from=0):
    t = t_from
    for n in chunks:
        closed = cache.append({k: v[:, t:t + n].contiguous() for k, v in inp.items()}, snapshots=snapshots)
        assert list(closed) == list(range(t // cache.m, (t + n) // cache.m))
        t += n
    assert cache.t == t


def _np(p, k):
    return None if k not in p else p[k].double().cpu().numpy()


@pytest.mark.parametrize("kind,B,T,d,dI,seed", [
    ("csa", 2, 700, 512, 128, 11),     # ragged tail (700 = 4*175), batch 2
    ("csa", 1, 261, 128, 64, 12),      # tiny workload widths
    ("hca", 2, 3 * 128 + 50, 512, 0, 13),
])
def test_chunked_append_matches_whole_sequence(kind, B, T, d, dI, seed):
    m = 4 if kind == "csa" else 128
    inp = _inputs(kind, B, T, d, dI, seed)
    prm = _params(kind, d, dI, m, seed)
    cache = LayerCache(kind, B, T + 64, d=d, dI=dI, params=prm, device=DEV)
    _fill(cache, inp, _chunks(T, seed))
    N = T // m
    torch.cuda.synchronize()
    ov = kind == "csa"
    whole = P.compress(inp["Ca"], inp["Za"], m, Cb=inp["Cb"] if ov else None, Zb=inp["Zb"] if ov else None,
                       bias_a=prm["bias_a"], bias_b=prm.get("bias_b"), gamma=prm["gamma"], theta=THETA)
    assert torch.equal(cache.kv[:, :N], whole), "cache entries differ from one whole-sequence call"
    assert not (cache.kv[:, N:] != 0).any(), "entries beyond the closed prefix were written"
    ref = O.compress(f64(inp["Ca"]), f64(inp["Za"]), m, Cb=f64(inp["Cb"]) if ov else None,
                     Zb=f64(inp["Zb"]) if ov else None, bias_a=_np(prm, "bias_a"), bias_b=_np(prm, "bias_b"),
                     gamma=_np(prm, "gamma"), rope_dims=64, theta=THETA)
    assert_close(cache.kv[:, :N], ref, f"{kind} cache entries")
    if ov:
        wI = P.compress(inp["Ca_I"], inp["Za_I"], m, Cb=inp["Cb_I"], Zb=inp["Zb_I"], bias_a=prm["bias_a_I"],
                        bias_b=prm["bias_b_I"], gamma=prm["gamma_I"], rope=False, rope_dims=0)
        assert torch.equal(cache.kI[:, :N], wI)
        refI = O.compress(f64(inp["Ca_I"]), f64(inp["Za_I"]), m, Cb=f64(inp["Cb_I"]), Zb=f64(inp["Zb_I"]),
                          bias_a=_np(prm, "bias_a_I"), bias_b=_np(prm, "bias_b_I"), gamma=_np(prm, "gamma_I"),
                          rope_on=False, rope_dims=0)
        assert_close(cache.kI[:, :N], refI, "cache indexer keys")
    # window ring: token u at slot u mod 128 for the last 128 tokens
    u = np.arange(T - 128, T)
    assert torch.equal(cache.win[:, u % 128], inp["win"][:, u])


def test_decode_append_one_token_at_a_time():
    """Decode: one token per call from an empty cache; every 4th token closes one CSA entry."""
    B, T, d, dI = 3, 137, 128, 64
    inp = _inputs("csa", B, T, d, dI, 21)
    cache = LayerCache("csa", B, T, d=d, dI=dI, device=DEV)
    for t in range(T):
        closed = cache.append({k: v[:, t:t + 1].contiguous() for k, v in inp.items()})
        assert list(closed) == ([t // 4] if (t + 1) % 4 == 0 else [])
    whole = P.compress(inp["Ca"], inp["Za"], 4, Cb=inp["Cb"], Zb=inp["Zb"], theta=THETA)
    torch.cuda.synchronize()
    assert torch.equal(cache.kv[:, :T // 4], whole)
    ref = O.compress(f64(inp["Ca"]), f64(inp["Za"]), 4, Cb=f64(inp["Cb"]), Zb=f64(inp["Zb"]), rope_dims=64,
                     theta=THETA)
    assert_close(cache.kv[:, :T // 4], ref, "decode-appended entries")


@pytest.mark.parametrize("kind", ["csa", "hca"])
def test_prefix_reuse_recomputes_only_the_tail(kind):
    """Prefix of P = 1000 tokens: reuse up to P_closed = 896, append the tau = 104 tail again."""
    B, P_len, d, dI = 2, 1000, 256, 64
    m = 4 if kind == "csa" else 128
    inp = _inputs(kind, B, P_len, d, dI, 31)
    prm = _params(kind, d, dI, m, 31)
    src = LayerCache(kind, B, 1024, d=d, dI=dI, params=prm, device=DEV)
    snaps = {}
    _fill(src, inp, _chunks(P_len, 31), snaps)
    assert sorted(snaps) == list(range(128, P_len + 1, 128))
    closed, tau = closed_prefix(P_len)
    assert (closed, tau) == (896, 104)
    re, tau2 = LayerCache.from_prefix(src, P_len, snaps)
    assert tau2 == tau and re.t == closed
    _fill(re, inp, [tau], t_from=closed)
    torch.cuda.synchronize()
    assert torch.equal(re.kv, src.kv)
    if kind == "csa":
        assert torch.equal(re.kI, src.kI)
    assert torch.equal(re.win, src.win)
    assert torch.equal(re.state, src.state)
