"""Host-side checks of the C ABI that need no GPU: the library loads and exports every entry
point include/csa.h declares, the ctypes descriptors match the C layout field by field, and
invalid requests are rejected with their documented status before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

from long_context_compressed_16_b300 import capi as C

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")
FAKE = 0x10000          # an aligned address that host-side validation never dereferences


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_\w+|hca_\w+)\s*\(", src)))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("csa_compress", "csa_index_topk", "csa_attend", "hca_attend"):
        assert n in names


def test_library_exports_every_declared_symbol():
    out = subprocess.run(["nm", "-D", "--defined-only", C.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    assert set(C.EXPORTS) <= exported


def test_descriptor_layout_matches_c(tmp_path):
    structs = {"csa_compress_desc": C.csa_compress_desc, "csa_index_desc": C.csa_index_desc,
               "csa_attend_desc": C.csa_attend_desc, "csa_out_proj_desc": C.csa_out_proj_desc,
               "csa_cache_desc": C.csa_cache_desc, "csa_cache_rows": C.csa_cache_rows,
               "csa_cache_params": C.csa_cache_params, "csa_cache_buffers": C.csa_cache_buffers}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "csa.h"', "int main(void){"]
    for sname, cls in structs.items():
        lines.append(f'printf("{sname} size %zu\\n", sizeof({sname}));')
        for fname, _ in cls._fields_:
            lines.append(f'printf("{sname} {fname} %zu\\n", offsetof({sname}, {fname}));')
    lines.append("return 0;}")
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = {}
    for ln in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        s, f, v = ln.split()
        got[(s, f)] = int(v)
    for sname, cls in structs.items():
        assert got[(sname, "size")] == ctypes.sizeof(cls)
        for fname, _ in cls._fields_:
            assert got[(sname, fname)] == getattr(cls, fname).offset, (sname, fname)


def test_status_strings():
    for s in range(7):
        assert C.status_string(s)
    assert C.status_string(99) == "unknown status"


def _cdesc(**kw):
    d = dict(B=1, T=64, d=128, m=4, overlap=1, rope_dims=64, rope_theta=160000.0, inv_freq=None, pos_shift=0,
             eps=1e-6, flags=3, out_fmt=C.CSA_FMT_BF16)
    d.update(kw)
    return C.csa_compress_desc(**d)


def test_compress_validation():
    call = lambda desc, **p: C.lib.csa_compress(ctypes.byref(desc), p.get("Ca", FAKE), p.get("Cb", FAKE),
                                                p.get("Za", FAKE), p.get("Zb", FAKE), None, None, None,
                                                p.get("out", FAKE), None)
    assert call(_cdesc(d=100)) == C.CSA_ERR_UNSUPPORTED
    assert call(_cdesc(d=2048)) == C.CSA_ERR_UNSUPPORTED
    assert call(_cdesc(d=192)) == C.CSA_ERR_UNSUPPORTED     # widths are powers of two (norm reduction)
    assert call(_cdesc(m=0)) == C.CSA_ERR_INVALID_ARG
    assert call(_cdesc(rope_dims=60)) == C.CSA_ERR_UNSUPPORTED
    assert call(_cdesc(out_fmt=C.CSA_FMT_FP8_MIXED)) == C.CSA_ERR_UNSUPPORTED
    assert call(_cdesc(), Ca=None) == C.CSA_ERR_INVALID_ARG
    assert call(_cdesc(), Cb=None) == C.CSA_ERR_INVALID_ARG
    assert call(_cdesc(), Ca=FAKE + 4) == C.CSA_ERR_INVALID_ARG                # misaligned
    assert call(_cdesc(T=3)) == C.CSA_OK                                       # no closed block: nothing to do
    bad = C.float_table([float("nan")] + [0.5] * 31)                           # a non-finite frequency
    assert call(_cdesc(inv_freq=bad)) == C.CSA_ERR_INVALID_ARG
    inf = C.float_table([0.5] * 31 + [float("inf")])
    assert call(_cdesc(inv_freq=inf)) == C.CSA_ERR_INVALID_ARG


def _idesc(**kw):
    d = dict(B=2, Tq=1, N=1000, n_heads=64, head_dim=128, k=64, m=4, key_fmt=C.CSA_FMT_BF16)
    d.update(kw)
    return C.csa_index_desc(**d)


def test_index_validation_and_workspace():
    ws = C.lib.csa_index_topk_workspace(ctypes.byref(_idesc()))
    assert ws >= 256 + 2 * 1000 * 4
    assert C.lib.csa_index_topk_workspace(ctypes.byref(_idesc(head_dim=96))) == 0
    big = C.lib.csa_index_topk_workspace(ctypes.byref(_idesc(B=1, Tq=65536, N=16384)))
    assert 256 << 20 <= big <= (256 << 20) + 4096          # prefill scores are materialised in chunks

    def call(desc, ws_ptr=FAKE, ws_bytes=1 << 30, **p):
        return C.lib.csa_index_topk(ctypes.byref(desc), p.get("qI", FAKE), FAKE, p.get("kI", FAKE),
                                    p.get("kI_scale", None), FAKE, FAKE, None, ws_ptr, ws_bytes, None)
    assert call(_idesc(n_heads=65)) == C.CSA_ERR_INVALID_ARG
    assert call(_idesc(k=0)) == C.CSA_ERR_INVALID_ARG
    assert call(_idesc(k=4096)) == C.CSA_ERR_INVALID_ARG
    assert call(_idesc(N=300000)) == C.CSA_ERR_UNSUPPORTED
    assert call(_idesc(), ws_ptr=None) == C.CSA_ERR_WORKSPACE
    assert call(_idesc(), ws_bytes=100) == C.CSA_ERR_WORKSPACE
    assert call(_idesc(key_fmt=C.CSA_FMT_FP8_ROWSCALE)) == C.CSA_ERR_INVALID_ARG   # scales missing
    assert call(_idesc(score_fmt=2)) == C.CSA_ERR_INVALID_ARG                       # unknown score format
    assert call(_idesc(select_mode=3)) == C.CSA_ERR_INVALID_ARG                     # unknown selection mode
    assert C.lib.csa_index_topk_workspace(ctypes.byref(_idesc(score_fmt=C.CSA_SCORE_BF16))) == ws
    # the fused selection's candidate lists take the place of the score rows, so a call that may
    # take it never needs less workspace than one that stores the rows
    kw = dict(B=1, Tq=2400, N=32768, k=512)
    stored = C.lib.csa_index_topk_workspace(ctypes.byref(_idesc(select_mode=C.CSA_SELECT_STORED, **kw)))
    fused = C.lib.csa_index_topk_workspace(ctypes.byref(_idesc(select_mode=C.CSA_SELECT_FUSED, **kw)))
    assert stored > 0 and fused >= stored
    assert call(_idesc(B=0)) == C.CSA_OK


def test_split_index_calls_validation_and_workspace():
    assert C.lib.csa_index_score_workspace(ctypes.byref(_idesc())) == 256
    assert C.lib.csa_index_score_workspace(ctypes.byref(_idesc(head_dim=96))) == 0
    # decode rows longer than one selection slice keep (key, index) candidates of every slice
    ws = C.lib.csa_topk_workspace(ctypes.byref(_idesc(B=32, Tq=1, N=32768, k=512)))
    assert ws >= 256 + 32 * 2 * 512 * 8
    assert C.lib.csa_topk_workspace(ctypes.byref(_idesc(B=1, Tq=65536, N=16384))) == 256   # one stage
    sc = lambda desc, ws_ptr=FAKE, ws_bytes=1 << 30: C.lib.csa_index_score(
        ctypes.byref(desc), FAKE, FAKE, FAKE, None, FAKE, FAKE, ws_ptr, ws_bytes, None)
    assert sc(_idesc(n_heads=65)) == C.CSA_ERR_INVALID_ARG
    assert sc(_idesc(N=300000)) == C.CSA_ERR_UNSUPPORTED
    assert sc(_idesc(), ws_bytes=100) == C.CSA_ERR_WORKSPACE
    assert sc(_idesc(key_fmt=C.CSA_FMT_FP8_ROWSCALE)) == C.CSA_ERR_INVALID_ARG
    assert sc(_idesc(B=0)) == C.CSA_OK
    tk = lambda desc, ws_ptr=FAKE, ws_bytes=1 << 30: C.lib.csa_topk(
        ctypes.byref(desc), FAKE, FAKE, FAKE, ws_ptr, ws_bytes, None)
    assert tk(_idesc(k=0)) == C.CSA_ERR_INVALID_ARG
    assert tk(_idesc(), ws_ptr=None) == C.CSA_ERR_WORKSPACE
    assert tk(_idesc(B=32, Tq=1, N=32768, k=512), ws_bytes=256) == C.CSA_ERR_WORKSPACE
    assert tk(_idesc(B=0)) == C.CSA_OK


def _adesc(**kw):
    d = dict(B=2, Tq=1, N=1000, H=64, d=512, rope_dims=64, k=64, m=4, Wcap=128, window=128, scale=0.0,
             rope_theta=160000.0, inv_freq=None, eps=1e-6, kv_fmt=C.CSA_FMT_BF16, flags=3)
    d.update(kw)
    return C.csa_attend_desc(**d)


def test_attend_validation_and_workspace():
    # decode splits 640 slots into 192-slot pieces: partial results per split live in the workspace
    ws = C.lib.csa_attend_workspace(ctypes.byref(_adesc(k=512)))
    assert ws == 256 + 2 * 4 * 64 * (512 + 2) * 4
    assert C.lib.csa_attend_workspace(ctypes.byref(_adesc(Tq=8, k=512))) == 256     # prefill: one split

    def call(desc, ws_bytes=1 << 30, **p):
        return C.lib.csa_attend(ctypes.byref(desc), FAKE, FAKE, p.get("idx", FAKE), FAKE, FAKE, FAKE,
                                FAKE, None, FAKE, ws_bytes, None)
    assert call(_adesc(d=256)) == C.CSA_ERR_INVALID_ARG
    assert call(_adesc(H=24)) == C.CSA_ERR_INVALID_ARG
    assert call(_adesc(window=200)) == C.CSA_ERR_INVALID_ARG              # window > ring capacity
    assert call(_adesc(kv_fmt=C.CSA_FMT_FP8_MIXED, d=128)) == C.CSA_ERR_INVALID_ARG
    assert call(_adesc(), idx=None) == C.CSA_ERR_INVALID_ARG
    assert call(_adesc(k=512), ws_bytes=1024) == C.CSA_ERR_WORKSPACE
    assert call(_adesc(flags=7)) == C.CSA_ERR_INVALID_ARG                 # lse requested, pointer NULL
    assert call(_adesc(B=0)) == C.CSA_OK
    assert C.lib.hca_attend(ctypes.byref(_adesc(m=0)), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                            1 << 20, None) == C.CSA_ERR_INVALID_ARG


def test_binding_refuses_to_run_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(C, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        C._load()


def test_out_proj_validation_and_workspace():
    desc = lambda **kw: C.csa_out_proj_desc(**{**dict(T=300, n_heads=64, head_dim=512, groups=8, rank=1024,
                                                      d_out=4096), **kw})
    assert C.csa_out_proj_workspace(desc()) == 256
    for bad in (dict(groups=3), dict(rank=100), dict(d_out=100), dict(head_dim=12), dict(T=-1), dict(groups=0)):
        assert C.csa_out_proj_workspace(desc(**bad)) == 0, bad
    ws = FAKE
    call = lambda d, **p: C.csa_out_proj(d, p.get("O", FAKE), p.get("Wd", FAKE), p.get("Wp", FAKE),
                                         p.get("z", FAKE), p.get("y", FAKE), p.get("ws", ws), p.get("n", 256), stream=0)
    assert call(desc(T=0)) == C.CSA_OK                                  # no rows: no launch
    assert call(desc(groups=3)) == C.CSA_ERR_INVALID_ARG
    assert call(desc(rank=96)) == C.CSA_ERR_UNSUPPORTED
    assert call(desc(), n=128) == C.CSA_ERR_WORKSPACE
    assert call(desc(), ws=None) == C.CSA_ERR_WORKSPACE
    assert call(desc(), O=None) == C.CSA_ERR_INVALID_ARG
    assert call(desc(), O=FAKE + 8) == C.CSA_ERR_INVALID_ARG
    assert call(desc(), Wp=None) == C.CSA_ERR_INVALID_ARG              # d_out > 0 needs Proj
    assert call(desc(), y=None) == C.CSA_ERR_INVALID_ARG
    assert C.lib.csa_out_proj(None, None, None, None, None, None, None, 0, None) == C.CSA_ERR_INVALID_ARG
