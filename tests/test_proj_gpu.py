"""GPU parity of the grouped output projection (csa_out_proj) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from long_context_compressed_16_b300 import pipeline as P
from long_context_compressed_16_b300 import synth as S
from oracle import csa_oracle as O
from tests.helpers import assert_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(T, n_h, d_h, g, r_o, d_out, seed):
    K = n_h // g * d_h
    Oa = S.normal_bf16((T, n_h, d_h), seed, S.TID["O"], DEV)
    Wd = S.weight_bf16((g, r_o, K), seed, S.TID["W_down"], K, DEV)
    Wp = S.weight_bf16((d_out, g * r_o), seed, S.TID["W_proj"], g * r_o, DEV) if d_out else None
    return Oa, Wd, Wp


@pytest.mark.parametrize("T,n_h,d_h,g,r_o,d_out", [
    (300, 8, 128, 2, 128, 256),        # ragged rows (300 = 2 x 128 + 44)
    (1000, 64, 512, 8, 1024, 4096),    # Flash widths
    (32, 64, 512, 8, 1024, 4096),      # decode batch of 32 tokens
    (129, 16, 64, 4, 192, 64),         # rank 192: 64-wide tiles; one row past a tile
    (1, 8, 128, 8, 64, 0),             # one token, one head per group, z only
    (17, 8, 128, 2, 256, 128),         # few rows: weight-major tiles, 32-row activation tile, 15 masked
    (48, 16, 64, 4, 128, 256),         # 48-row activation tile
    (64, 64, 512, 8, 1024, 4096),      # 64 rows: the largest weight-major case
    (65, 16, 64, 4, 128, 256),         # 65 rows: back to activation-major tiles
])
def test_out_proj_parity(T, n_h, d_h, g, r_o, d_out):
    Oa, Wd, Wp = _inputs(T, n_h, d_h, g, r_o, d_out, T + n_h)
    z, y = P.out_proj(Oa, Wd, g, W_proj=Wp)
    torch.cuda.synchronize()
    zr, yr = O.out_proj(f64(Oa), f64(Wd), None if Wp is None else f64(Wp))
    assert_close(z, zr, f"z T{T} g{g}")
    if d_out:
        assert_close(y, yr, f"y T{T} d_out{d_out}")
    else:
        assert y is None


def test_out_proj_rows_are_batch_invariant_and_deterministic():
    """A token's outputs do not depend on how many other tokens share the call (different tile
    widths and tile counts), and repeated calls are bit-identical."""
    Oa, Wd, Wp = _inputs(1000, 64, 512, 8, 1024, 4096, 77)
    z1, y1 = P.out_proj(Oa, Wd, 8, W_proj=Wp)
    z2, y2 = P.out_proj(Oa, Wd, 8, W_proj=Wp)
    torch.cuda.synchronize()
    assert torch.equal(z1, z2) and torch.equal(y1, y2)
    for lo, n in ((200, 32), (500, 1), (7, 64), (900, 100)):   # weight-major and activation-major tiles
        zs, ys = P.out_proj(Oa[lo:lo + n].contiguous(), Wd, 8, W_proj=Wp)
        torch.cuda.synchronize()
        assert torch.equal(zs, z1[lo:lo + n]) and torch.equal(ys, y1[lo:lo + n]), (lo, n)


def test_out_proj_empty():
    Oa, Wd, Wp = _inputs(0, 8, 128, 2, 128, 256, 1)
    z, y = P.out_proj(Oa, Wd, 2, W_proj=Wp)
    assert z.shape == (0, 256) and y.shape == (0, 256)


def test_out_proj_full_size_sampled_rows():
    """The prefill size (65536 tokens, Flash widths) in one call; 40 sampled rows (first, last and
    seeded random ones, rows being independent) against the oracle."""
    T = 65536
    Oa, Wd, Wp = _inputs(T, 64, 512, 8, 1024, 4096, 3)
    z, y = P.out_proj(Oa, Wd, 8, W_proj=Wp)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, 127, 128, T - 1], np.random.default_rng(3).integers(0, T, 36)]))
    ri = torch.from_numpy(rows).to(DEV)
    zr, yr = O.out_proj(f64(Oa[ri]), f64(Wd), f64(Wp))
    assert_close(z[ri], zr, "z sampled rows")
    assert_close(y[ri], yr, "y sampled rows")
