"""Multi-rank partition, run as two gloo ranks on the CPU.

Each rank computes its share with the fp64 oracle standing in for the per-rank library calls;
the partitioned results must equal the single-rank oracle.  The exchanges and the index
arithmetic are the ones the GPU ranks use (long_context_compressed_16_b300.shard)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from long_context_compressed_16_b300 import shard as SH
from long_context_compressed_16_b300 import synth as S

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _f64(t):
    return t.detach().to(torch.float64)


def _tiny(T=512):
    w = S.scaled(S.WORKLOADS["tiny_csa_prefill_t2048"], T=T, N=T // 4, d=128, H=2, nI=2, dI=32, k=16)
    return w, S.make_inputs(w, "cpu")


def _compress_csa(O, Ca, Za, Cb, Zb, m, pos_shift, rope_on):
    return O.compress(Ca.numpy(), Za.numpy(), m, Cb=Cb.numpy(), Zb=Zb.numpy(), rope_on=rope_on,
                      pos_shift=pos_shift)


def _single_rank(O, w, inp):
    f = {k: _f64(v) for k, v in inp.items()}
    kv = O.compress(f["Ca"].numpy(), f["Za"].numpy(), w.m, Cb=f["Cb"].numpy(), Zb=f["Zb"].numpy())
    kI = O.compress(f["Ca_I"].numpy(), f["Za_I"].numpy(), w.m, Cb=f["Cb_I"].numpy(), Zb=f["Zb_I"].numpy(),
                    rope_on=False)
    hca = O.compress(f["Ca"].numpy(), f["Za"].numpy(), 128)
    pos = inp["q_pos"].numpy()
    sc = O.index_scores(f["qI"].numpy(), f["w"].numpy(), kI, pos, w.m)
    idx = O.topk_select(sc, pos, w.m, w.k)
    o, lse = O.attend(f["q"].numpy(), kv, f["win"].numpy(), f["sink"].numpy(), pos, w.m, w.window, idx=idx)
    oh, _ = O.attend(f["q"].numpy(), hca, f["win"].numpy(), f["sink"].numpy(), pos, 128, w.window)
    return kv, kI, hca, idx, o, lse, oh


def _cp_rank(rank, port, T):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        from oracle import csa_oracle as O
        w, inp = _tiny(T)
        r = SH.token_range(T, WORLD, rank, w.m, w.window)
        f = {k: _f64(v) for k, v in inp.items()}
        own = {k: f[k][:, r.lo:r.hi] for k in ("Ca", "Za", "Cb", "Zb", "Ca_I", "Za_I", "Cb_I", "Zb_I", "win")}
        # exchange 1: b-stream tails and window rows from rank-1
        rows = {"Cb": w.m, "Zb": w.m, "Cb_I": w.m, "Zb_I": w.m, "win": w.window - 1}
        halo = SH.halo_exchange(r, {k: own[k] for k in rows}, rows)
        assert halo["Cb"].shape[1] == r.halo_b and halo["win"].shape[1] == r.halo_win

        def local(Ca, Za, Cb, Zb, hCb, hZb, rope_on):
            a, z, b, zb, shift, drop = SH.with_b_halo(r, w.m, Ca, Za, Cb, Zb, hCb, hZb)
            return torch.from_numpy(_compress_csa(O, a, z, b, zb, w.m, shift, rope_on)[:, drop:])

        kv_loc = local(own["Ca"], own["Za"], own["Cb"], own["Zb"], halo["Cb"], halo["Zb"], True)
        kI_loc = local(own["Ca_I"], own["Za_I"], own["Cb_I"], own["Zb_I"], halo["Cb_I"], halo["Zb_I"], False)
        hca_loc = torch.from_numpy(O.compress(own["Ca"].numpy(), own["Za"].numpy(), 128, pos_shift=r.lo))
        assert kv_loc.shape[1] == r.tokens // w.m and hca_loc.shape[1] == r.tokens // 128
        # exchange 2: all-gather of the compressed entries
        kv = SH.allgather_rows(kv_loc).numpy()
        kI = SH.allgather_rows(kI_loc).numpy()
        hca = SH.allgather_rows(hca_loc).numpy()
        # local queries against the gathered caches, window from halo + own rows
        ring, Wcap = SH.window_ring(r, halo["win"], own["win"])
        pos = inp["q_pos"][:, r.lo:r.hi].numpy()
        q = f["q"][:, r.lo:r.hi].numpy()
        sc = O.index_scores(f["qI"][:, r.lo:r.hi].numpy(), f["w"][:, r.lo:r.hi].numpy(), kI, pos, w.m)
        idx = O.topk_select(sc, pos, w.m, w.k)
        o, lse = O.attend(q, kv, ring.numpy(), f["sink"].numpy(), pos, w.m, w.window, idx=idx)
        oh, _ = O.attend(q, hca, ring.numpy(), f["sink"].numpy(), pos, 128, w.window)

        kv1, kI1, hca1, idx1, o1, lse1, oh1 = _single_rank(O, w, inp)
        np.testing.assert_allclose(kv, kv1, rtol=0, atol=1e-12)
        np.testing.assert_allclose(kI, kI1, rtol=0, atol=1e-12)
        np.testing.assert_allclose(hca, hca1, rtol=0, atol=1e-12)
        assert np.array_equal(idx, idx1[:, r.lo:r.hi])
        np.testing.assert_allclose(o, o1[:, r.lo:r.hi], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, lse1[:, r.lo:r.hi], rtol=0, atol=1e-12)
        np.testing.assert_allclose(oh, oh1[:, r.lo:r.hi], rtol=0, atol=1e-12)
    finally:
        dist.destroy_process_group()


def _decode_rank(rank, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        from oracle import csa_oracle as O
        w = S.scaled(S.WORKLOADS["csa_decode_128k_b32"], B=5, N=96, d=128, H=2, nI=2, dI=32, k=8)
        inp = S.make_inputs(w, "cpu")
        f = {k: _f64(v) for k, v in inp.items() if v.dtype != torch.int32}
        pos = inp["q_pos"].numpy()
        lo, hi = SH.batch_range(w.B, WORLD, rank)

        def run(b0, b1):
            sc = O.index_scores(f["qI"][b0:b1].numpy(), f["w"][b0:b1].numpy(), f["kI"][b0:b1].numpy(),
                                pos[b0:b1], w.m)
            idx = O.topk_select(sc, pos[b0:b1], w.m, w.k)
            o, _ = O.attend(f["q"][b0:b1].numpy(), f["kv"][b0:b1].numpy(), f["win"][b0:b1].numpy(),
                            f["sink"].numpy(), pos[b0:b1], w.m, w.window, idx=idx)
            return torch.from_numpy(idx), torch.from_numpy(o)

        idx, o = run(lo, hi)                      # no exchange on the data path
        idx_all, o_all = SH.allgather_rows(idx.transpose(0, 1)), SH.allgather_rows(o.transpose(0, 1))
        idx1, o1 = run(0, w.B)
        assert torch.equal(idx_all.transpose(0, 1), idx1)
        assert torch.equal(o_all.transpose(0, 1), o1)
    finally:
        dist.destroy_process_group()


def test_batch_range_covers_batch_evenly():
    for B in (0, 1, 5, 32, 33):
        for world in (1, 2, 3, 8):
            parts = [SH.batch_range(B, world, r) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == B
            assert all(parts[i][1] == parts[i + 1][0] for i in range(world - 1))
            sizes = [hi - lo for lo, hi in parts]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        SH.batch_range(4, 2, 2)


def test_token_range_alignment_and_halo():
    T, m, window = 65536, 4, 128
    for world in (1, 2, 3, 8):
        rs = [SH.token_range(T, world, r, m, window) for r in range(world)]
        assert rs[0].lo == 0 and rs[-1].hi == T
        for a, b in zip(rs, rs[1:]):
            assert a.hi == b.lo and b.lo % 128 == 0
            assert b.halo_b == m and b.halo_win == window - 1 and a.tokens >= window - 1
        assert rs[0].halo_b == 0 and rs[0].halo_win == 0
    with pytest.raises(ValueError):
        SH.token_range(256, 3, 0, 4, 128)         # two 128-token blocks for three ranks
    with pytest.raises(ValueError):
        SH.token_range(1000, 2, 0, 4, 128)        # not a whole number of blocks


def test_window_ring_slots():
    r = SH.TokenRange(lo=256, hi=512, halo_b=4, halo_win=127)
    halo = torch.arange(256 - 127, 256, dtype=torch.float64).view(1, -1, 1)
    own = torch.arange(256, 512, dtype=torch.float64).view(1, -1, 1)
    ring, Wcap = SH.window_ring(r, halo, own)
    assert Wcap == 383
    for p in range(256 - 127, 512):
        assert ring[0, p % Wcap, 0].item() == p


def test_context_parallel_prefill_two_gloo_ranks():
    mp.spawn(_cp_rank, args=(_free_port(), 512), nprocs=WORLD, join=True)


def test_batch_sharded_decode_two_gloo_ranks():
    mp.spawn(_decode_rank, args=(_free_port(),), nprocs=WORLD, join=True)
