"""Python binding of the C ABI in include/csa.h (ctypes; argument marshalling only).

Every function here has the name of the C entry point it calls and returns its csa_status.
Tensor arguments may be torch tensors (their data_ptr() is passed), raw integer device
addresses, or None (NULL).  All computation happens in libcsa.so's CUDA kernels; there is no
fallback: importing this module fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_int32, c_size_t, c_uint, c_uint64, c_void_p

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcsa.so")

# csa_status
CSA_OK = 0
CSA_ERR_INVALID_ARG = 1
CSA_ERR_UNSUPPORTED = 2
CSA_ERR_WORKSPACE = 3
CSA_ERR_CUDA = 4
CSA_ERR_DEVICE_CHECK = 5
CSA_ERR_TIMEOUT = 6
# csa_format
CSA_FMT_BF16 = 0
CSA_FMT_FP8_MIXED = 1
CSA_FMT_FP8_ROWSCALE = 2
CSA_FMT_FP8_ROWSCALE_LOWP = 3
CSA_FP8_MIXED_ROW_BYTES = 608
# csa_index_desc.score_fmt
CSA_SCORE_FP32 = 0
CSA_SCORE_BF16 = 1
# csa_index_desc.select_mode
CSA_SELECT_AUTO = 0
CSA_SELECT_FUSED = 1
CSA_SELECT_STORED = 2
CSA_NOALLOC_SCRATCH_BYTES = 8 << 20
# flags
CSA_COMPRESS_NORM = 1
CSA_COMPRESS_ROPE = 2
CSA_ATTEND_Q_NORM_ROPE = 1
CSA_ATTEND_OUT_UNROTATE = 2
CSA_ATTEND_WRITE_LSE = 4

EXPORTS = ("csa_compress", "csa_index_topk_workspace", "csa_index_topk", "csa_attend_workspace",
           "hca_attend_workspace", "csa_attend", "hca_attend", "csa_read_device_status", "csa_clear_device_status",
           "csa_status_string", "csa_launch_count", "csa_index_topk_noalloc", "csa_index_score_workspace",
           "csa_index_score", "csa_topk_workspace", "csa_topk", "csa_selftest_bounded_wait",
           "csa_cache_state_bytes", "csa_cache_append", "csa_out_proj_workspace", "csa_out_proj")


class csa_compress_desc(ctypes.Structure):
    _fields_ = [("B", c_int), ("T", c_int), ("d", c_int), ("m", c_int), ("overlap", c_int),
                ("rope_dims", c_int), ("rope_theta", c_float), ("inv_freq", POINTER(c_float)),
                ("pos_shift", c_int), ("eps", c_float), ("flags", c_uint), ("out_fmt", c_int)]


class csa_index_desc(ctypes.Structure):
    _fields_ = [("B", c_int), ("Tq", c_int), ("N", c_int), ("n_heads", c_int), ("head_dim", c_int),
                ("k", c_int), ("m", c_int), ("key_fmt", c_int), ("score_fmt", c_int), ("select_mode", c_int)]


class csa_attend_desc(ctypes.Structure):
    _fields_ = [("B", c_int), ("Tq", c_int), ("N", c_int), ("H", c_int), ("d", c_int),
                ("rope_dims", c_int), ("k", c_int), ("m", c_int), ("Wcap", c_int), ("window", c_int),
                ("scale", c_float), ("rope_theta", c_float), ("inv_freq", POINTER(c_float)),
                ("eps", c_float), ("kv_fmt", c_int), ("flags", c_uint)]


class csa_out_proj_desc(ctypes.Structure):
    _fields_ = [("T", c_int), ("n_heads", c_int), ("head_dim", c_int), ("groups", c_int), ("rank", c_int),
                ("d_out", c_int)]


class csa_cache_desc(ctypes.Structure):
    _fields_ = [("B", c_int), ("d", c_int), ("dI", c_int), ("m", c_int), ("overlap", c_int), ("Wcap", c_int),
                ("N_cap", c_int), ("rope_dims", c_int), ("rope_theta", c_float), ("inv_freq", POINTER(c_float)),
                ("eps", c_float), ("flags", c_uint), ("index_flags", c_uint)]


class csa_cache_rows(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("Ca", "Cb", "Za", "Zb", "Ca_I", "Cb_I", "Za_I", "Zb_I", "win")]


class csa_cache_params(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("bias_a", "bias_b", "gamma", "bias_a_I", "bias_b_I", "gamma_I")]


class csa_cache_buffers(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("kv", "kI", "win", "state")]


class CsaError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run long_context_compressed_16_b300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp = c_void_p
    lib.csa_compress.argtypes = [POINTER(csa_compress_desc), vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.csa_compress.restype = c_int
    lib.csa_index_topk_workspace.argtypes = [POINTER(csa_index_desc)]
    lib.csa_index_topk_workspace.restype = c_size_t
    lib.csa_index_topk.argtypes = [POINTER(csa_index_desc), vp, vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]
    lib.csa_index_topk.restype = c_int
    lib.csa_index_topk_noalloc.argtypes = [POINTER(csa_index_desc), vp, vp, vp, vp, vp, vp, vp, vp]
    lib.csa_index_topk_noalloc.restype = c_int
    lib.csa_index_score_workspace.argtypes = [POINTER(csa_index_desc)]
    lib.csa_index_score_workspace.restype = c_size_t
    lib.csa_index_score.argtypes = [POINTER(csa_index_desc), vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]
    lib.csa_index_score.restype = c_int
    lib.csa_topk_workspace.argtypes = [POINTER(csa_index_desc)]
    lib.csa_topk_workspace.restype = c_size_t
    lib.csa_topk.argtypes = [POINTER(csa_index_desc), vp, vp, vp, vp, c_size_t, vp]
    lib.csa_topk.restype = c_int
    lib.csa_attend_workspace.argtypes = [POINTER(csa_attend_desc)]
    lib.csa_attend_workspace.restype = c_size_t
    lib.hca_attend_workspace.argtypes = [POINTER(csa_attend_desc)]
    lib.hca_attend_workspace.restype = c_size_t
    lib.csa_attend.argtypes = [POINTER(csa_attend_desc), vp, vp, vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]
    lib.csa_attend.restype = c_int
    lib.hca_attend.argtypes = [POINTER(csa_attend_desc), vp, vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]
    lib.hca_attend.restype = c_int
    lib.csa_read_device_status.argtypes = [vp, vp, POINTER(c_int32)]
    lib.csa_read_device_status.restype = c_int
    lib.csa_clear_device_status.argtypes = [vp, vp]
    lib.csa_clear_device_status.restype = c_int
    lib.csa_status_string.argtypes = [c_int]
    lib.csa_status_string.restype = ctypes.c_char_p
    lib.csa_selftest_bounded_wait.argtypes = [vp, c_size_t, ctypes.c_int64, vp]
    lib.csa_selftest_bounded_wait.restype = c_int
    lib.csa_cache_state_bytes.argtypes = [POINTER(csa_cache_desc)]
    lib.csa_cache_state_bytes.restype = c_size_t
    lib.csa_cache_append.argtypes = [POINTER(csa_cache_desc), ctypes.c_int64, c_int, POINTER(csa_cache_rows),
                                     POINTER(csa_cache_params), POINTER(csa_cache_buffers), vp]
    lib.csa_cache_append.restype = c_int
    lib.csa_out_proj_workspace.argtypes = [POINTER(csa_out_proj_desc)]
    lib.csa_out_proj_workspace.restype = c_size_t
    lib.csa_out_proj.argtypes = [POINTER(csa_out_proj_desc), vp, vp, vp, vp, vp, vp, c_size_t, vp]
    lib.csa_out_proj.restype = c_int
    lib.csa_launch_count.argtypes = []
    lib.csa_launch_count.restype = c_uint64
    return lib


lib = _load()


def _p(x):
    """Device address of a tensor / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    return x.data_ptr() or None


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream


def _nbytes(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        raise TypeError("pass the workspace size explicitly for raw addresses")
    return x.numel() * x.element_size()


def float_table(values):
    """Host float array for a descriptor's inv_freq field (keep the returned object alive)."""
    if values is None:
        return None
    arr = (c_float * len(values))(*[float(v) for v in values])
    return arr


def status_string(status: int) -> str:
    return lib.csa_status_string(int(status)).decode()


def check(status: int, where: str = "csa") -> None:
    if status != CSA_OK:
        raise CsaError(status, where)


def csa_compress(desc, Ca, Cb, Za, Zb, bias_a, bias_b, gamma, out, stream=None) -> int:
    return lib.csa_compress(ctypes.byref(desc), _p(Ca), _p(Cb), _p(Za), _p(Zb), _p(bias_a), _p(bias_b),
                            _p(gamma), _p(out), _stream(stream))


def csa_index_topk_workspace(desc) -> int:
    return lib.csa_index_topk_workspace(ctypes.byref(desc))


def _check_index_tensors(desc, qI, w, kI, kI_scale, q_pos, idx_out, score_out):
    """The indexer calls take plain pointers: when torch tensors are passed, every extent the
    library reads or writes is checked against the descriptor first (raw addresses are the
    caller's responsibility)."""
    import torch
    B, Tq, N, nI, dI, k = desc.B, desc.Tq, desc.N, desc.n_heads, desc.head_dim, desc.k
    fp8 = desc.key_fmt in (CSA_FMT_FP8_ROWSCALE, CSA_FMT_FP8_ROWSCALE_LOWP)
    want = [("qI", qI, (B, Tq, nI, dI), torch.bfloat16), ("w", w, (B, Tq, nI), torch.float32),
            ("kI", kI, (B, N, dI), torch.uint8 if fp8 else torch.bfloat16),
            ("q_pos", q_pos, (B, Tq), torch.int32), ("idx_out", idx_out, (B, Tq, k), torch.int32),
            ("score_out", score_out, (B, Tq, N), torch.float32)]
    if fp8:
        want.append(("kI_scale", kI_scale, (B, N), torch.float32))
    for name, t, shape, dtype in want:
        if t is None or isinstance(t, int):
            continue
        if tuple(t.shape) != shape or t.dtype != dtype or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor of shape {shape}, "
                             f"got {t.dtype} {tuple(t.shape)} on {t.device}")


def csa_index_topk(desc, qI, w, kI, kI_scale, q_pos, idx_out, score_out, workspace, ws_bytes=None,
                   stream=None) -> int:
    _check_index_tensors(desc, qI, w, kI, kI_scale, q_pos, idx_out, score_out)
    n = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return lib.csa_index_topk(ctypes.byref(desc), _p(qI), _p(w), _p(kI), _p(kI_scale), _p(q_pos), _p(idx_out),
                              _p(score_out), _p(workspace), n, _stream(stream))


def csa_index_topk_noalloc(desc, qI, w, kI, kI_scale, q_pos, idx_out, score_out, stream=None) -> int:
    """csa_index_topk without a workspace argument: the library's fixed device scratch array is
    used instead (for callers that cannot allocate device memory; see include/csa.h)."""
    _check_index_tensors(desc, qI, w, kI, kI_scale, q_pos, idx_out, score_out)
    return lib.csa_index_topk_noalloc(ctypes.byref(desc), _p(qI), _p(w), _p(kI), _p(kI_scale), _p(q_pos),
                                      _p(idx_out), _p(score_out), _stream(stream))


def csa_index_score_workspace(desc) -> int:
    return lib.csa_index_score_workspace(ctypes.byref(desc))


def csa_index_score(desc, qI, w, kI, kI_scale, q_pos, score_out, workspace, ws_bytes=None, stream=None) -> int:
    n = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return lib.csa_index_score(ctypes.byref(desc), _p(qI), _p(w), _p(kI), _p(kI_scale), _p(q_pos), _p(score_out),
                               _p(workspace), n, _stream(stream))


def csa_topk_workspace(desc) -> int:
    return lib.csa_topk_workspace(ctypes.byref(desc))


def csa_topk(desc, scores, q_pos, idx_out, workspace, ws_bytes=None, stream=None) -> int:
    n = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return lib.csa_topk(ctypes.byref(desc), _p(scores), _p(q_pos), _p(idx_out), _p(workspace), n, _stream(stream))


def csa_attend_workspace(desc) -> int:
    return lib.csa_attend_workspace(ctypes.byref(desc))


def hca_attend_workspace(desc) -> int:
    return lib.hca_attend_workspace(ctypes.byref(desc))


def csa_attend(desc, q, kv, idx, win, sink, q_pos, out, lse, workspace, ws_bytes=None, stream=None) -> int:
    n = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return lib.csa_attend(ctypes.byref(desc), _p(q), _p(kv), _p(idx), _p(win), _p(sink), _p(q_pos), _p(out),
                          _p(lse), _p(workspace), n, _stream(stream))


def hca_attend(desc, q, kv, win, sink, q_pos, out, lse, workspace, ws_bytes=None, stream=None) -> int:
    n = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return lib.hca_attend(ctypes.byref(desc), _p(q), _p(kv), _p(win), _p(sink), _p(q_pos), _p(out), _p(lse),
                          _p(workspace), n, _stream(stream))


def csa_read_device_status(workspace, stream=None):
    detail = c_int32(0)
    st = lib.csa_read_device_status(_p(workspace), _stream(stream), ctypes.byref(detail))
    return st, detail.value


def csa_clear_device_status(workspace, stream=None) -> int:
    return lib.csa_clear_device_status(_p(workspace), _stream(stream))


def csa_selftest_bounded_wait(workspace, limit_ns, ws_bytes=None, stream=None) -> int:
    n = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return lib.csa_selftest_bounded_wait(_p(workspace), n, int(limit_ns), _stream(stream))


def csa_launch_count() -> int:
    return int(lib.csa_launch_count())


def csa_cache_state_bytes(desc) -> int:
    return lib.csa_cache_state_bytes(ctypes.byref(desc))


def csa_cache_append(desc, t0, n, rows, params, bufs, stream=None) -> int:
    """rows / params / bufs: dicts of tensors (or addresses) keyed by the C struct's field names;
    missing keys are NULL."""
    r = csa_cache_rows(**{k: _p(v) for k, v in rows.items()})
    p = csa_cache_params(**{k: _p(v) for k, v in (params or {}).items()})
    b = csa_cache_buffers(**{k: _p(v) for k, v in bufs.items()})
    return lib.csa_cache_append(ctypes.byref(desc), int(t0), int(n), ctypes.byref(r),
                                ctypes.byref(p) if params is not None else None, ctypes.byref(b), _stream(stream))


def csa_out_proj_workspace(desc) -> int:
    return lib.csa_out_proj_workspace(ctypes.byref(desc))


def csa_out_proj(desc, O, W_down, W_proj, z, y, workspace, ws_bytes=None, stream=None) -> int:
    n = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return lib.csa_out_proj(ctypes.byref(desc), _p(O), _p(W_down), _p(W_proj), _p(z), _p(y), _p(workspace), n,
                            _stream(stream))
