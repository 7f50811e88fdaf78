"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle harness.

Every tensor is drawn from a counter-based generator: splitmix64 keyed by
(seed, tensor id, flat element index), so any element can be regenerated on
its own and the same call gives the same bytes on CPU or GPU.  Normal values
come from the Box-Muller transform in fp64, uniforms from the top 53 bits.
Values are rounded once, round-to-nearest-even, to the storage format the
library consumes (bf16, or e4m3 with fp32 block/row scales) and both sides of
every parity check read those same bytes.

This module holds only data generation and storage encoding.  None of the
attention method's arithmetic (compression, normalisation, rotation,
scoring, selection or attention) lives here.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

_M64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB
_CHUNK = 1 << 25  # elements generated per pass (bounds the fp64/int64 temporaries)

# tensor ids: fixed so that each named input is its own stream
TID = {
    "Ca": 1, "Cb": 2, "Za": 3, "Zb": 4,
    "Ca_I": 5, "Cb_I": 6, "Za_I": 7, "Zb_I": 8,
    "C": 9, "Z": 10,
    "q": 11, "qI": 12, "w": 13, "kv": 14, "kI": 15, "win": 16, "sink": 17,
    "outlier_kv": 18, "outlier_kI": 19,
    "O": 20, "W_down": 21, "W_proj": 22,
    "Ba": 23, "Bb": 24, "Ba_I": 25, "Bb_I": 26, "gamma": 27, "gamma_I": 28, "B": 29,
}


def _s64(v: int) -> int:
    """Reinterpret an unsigned 64-bit constant as a signed int64 value."""
    v &= _M64
    return v - (1 << 64) if v >= (1 << 63) else v


def _srl(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 lanes (torch's >> is arithmetic)."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    """splitmix64 output function (wrapping 64-bit multiply)."""
    z = (z ^ _srl(z, 30)) * _s64(_MIX1)
    z = (z ^ _srl(z, 27)) * _s64(_MIX2)
    return z ^ _srl(z, 31)


def _mix64_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * _MIX1) & _M64
    z = ((z ^ (z >> 27)) * _MIX2) & _M64
    return z ^ (z >> 31)


def stream_key(seed: int, tensor_id: int) -> int:
    """Starting splitmix64 state of the stream for (seed, tensor id)."""
    return _mix64_int((seed << 32) ^ (tensor_id * 0x632BE59BD9B4E019))


def raw_bits(seed: int, tensor_id: int, start: int, n: int, device) -> torch.Tensor:
    """splitmix64 outputs number start..start+n-1 of one stream, as int64 lanes."""
    base = stream_key(seed, tensor_id)
    i = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    state = i * _s64(_GOLDEN) + _s64(base)
    return _mix64(state)


def _normal_chunk(bits: torch.Tensor) -> torch.Tensor:
    u1 = (_srl(bits, 38).to(torch.float64) + 0.5) * (2.0 ** -26)
    u2 = (((bits >> 12) & ((1 << 26) - 1)).to(torch.float64)) * (2.0 ** -26)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def _uniform_chunk(bits: torch.Tensor) -> torch.Tensor:
    return (_srl(bits, 11).to(torch.float64) + 0.5) * (2.0 ** -53)


def _fill(shape, seed, tensor_id, device, kind, encode):
    """Generate a tensor chunk by chunk and encode each chunk to its storage dtype."""
    n = 1
    for s in shape:
        n *= s
    out = None
    for start in range(0, max(n, 1), _CHUNK):
        cnt = min(_CHUNK, n - start)
        if cnt <= 0:
            break
        bits = raw_bits(seed, tensor_id, start, cnt, device)
        vals = _normal_chunk(bits) if kind == "normal" else _uniform_chunk(bits)
        enc = encode(vals)
        if out is None:
            out = torch.empty(n, dtype=enc.dtype, device=device)
        out[start:start + cnt] = enc
    if out is None:
        out = encode(torch.empty(0, dtype=torch.float64, device=device))
    return out.view(*shape)


def normal_f64(shape, seed, tensor_id, device="cpu") -> torch.Tensor:
    return _fill(shape, seed, tensor_id, device, "normal", lambda v: v)


def uniform_f64(shape, seed, tensor_id, device="cpu") -> torch.Tensor:
    return _fill(shape, seed, tensor_id, device, "uniform", lambda v: v)


# ----------------------------------------------------------------------------------------------
# storage encodings
# ----------------------------------------------------------------------------------------------

def f64_to_bf16(x: torch.Tensor) -> torch.Tensor:
    """fp64 -> fp32 (IEEE RNE) -> bf16 (RNE on the fp32 bit pattern). Returns a bfloat16 tensor."""
    b = x.to(torch.float32).contiguous().view(torch.int32).to(torch.int64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (r & 0xFFFF).to(torch.int32).to(torch.int16).view(torch.bfloat16)


def normal_bf16(shape, seed, tensor_id, device="cpu", scale_channels=None) -> torch.Tensor:
    """N(0,1) values rounded to bf16. scale_channels=(idx tensor, factor) multiplies those
    trailing-dim channels by factor before rounding (the seeded outlier recipe)."""
    def enc(v):
        return f64_to_bf16(v)
    if scale_channels is None:
        return _fill(shape, seed, tensor_id, device, "normal", enc)
    x = normal_f64(shape, seed, tensor_id, device)
    idx, factor = scale_channels
    x[..., idx.to(device)] *= factor
    return f64_to_bf16(x)


def weight_bf16(shape, seed, tensor_id, fan_in: int, device="cpu") -> torch.Tensor:
    """Random-init projection weights: N(0, 1/fan_in) values rounded to bf16."""
    return f64_to_bf16(normal_f64(shape, seed, tensor_id, device) / math.sqrt(fan_in))


def e4m3_encode(v: torch.Tensor) -> torch.Tensor:
    """OCP FP8 E4M3 (bias 7, largest finite 448, no infinities) code of fp64 values,
    round-to-nearest-even with saturation to +-448. Returns uint8 codes."""
    sign = (v < 0) | ((v == 0) & (torch.signbit(v)))
    a = v.abs().clamp(max=448.0)
    mant, ex = torch.frexp(a)                  # a = mant * 2^ex, mant in [0.5, 1)
    e = (ex - 1).clamp(min=-6)                 # binade exponent, subnormals share 2^-6's grid
    ulp = torch.pow(torch.tensor(2.0, dtype=torch.float64, device=v.device), (e - 3).to(torch.float64))
    q = torch.round(a / ulp) * ulp             # torch.round is half-to-even
    q = q.clamp(max=448.0)
    mant2, ex2 = torch.frexp(q)
    e2 = (ex2 - 1)
    normal = q >= 2.0 ** -6
    E = torch.where(normal, e2 + 7, torch.zeros_like(e2))
    Mn = torch.where(normal, torch.round(q / torch.pow(torch.tensor(2.0, dtype=torch.float64, device=v.device),
                                                        e2.to(torch.float64)) * 8.0) - 8.0,
                     torch.round(q / (2.0 ** -9)))
    code = (E.to(torch.int64) << 3) | Mn.to(torch.int64)
    code = torch.where(q == 0, torch.zeros_like(code), code)
    code = code | (sign.to(torch.int64) << 7)
    return code.to(torch.uint8)


FP8_ROW_BYTES = 608          # 448 e4m3 | 64 bf16 | 7 fp32 block scales | 4 pad
FP8_NOPE_DIMS = 448
FP8_BLOCK = 64


def pack_kv_fp8_mixed(x: torch.Tensor) -> torch.Tensor:
    """Mixed-precision cache row for d=512 entries.

    dims [0,448): e4m3 codes, one fp32 scale per 64-element block, scale = amax/448
    (1 when the block is all zero), code = RNE-saturate(x/scale);
    dims [448,512): bf16 (RNE);  bytes: [0,448) codes, [448,576) bf16, [576,604) scales, [604,608) zero.
    x: fp64 [..., 512]. Returns uint8 [..., 608]."""
    assert x.shape[-1] == 512
    lead = x.shape[:-1]
    xf = x.reshape(-1, 512)
    rows = xf.shape[0]
    out = torch.zeros(rows, FP8_ROW_BYTES, dtype=torch.uint8, device=x.device)
    step = 1 << 18
    for r0 in range(0, rows, step):
        xs = xf[r0:r0 + step]
        nope = xs[:, :FP8_NOPE_DIMS].reshape(-1, 7, FP8_BLOCK)
        amax = nope.abs().amax(dim=2)
        scale = (amax / 448.0).to(torch.float32)
        scale = torch.where(amax == 0, torch.ones_like(scale), scale)
        codes = e4m3_encode(nope / scale.to(torch.float64).unsqueeze(2)).reshape(-1, FP8_NOPE_DIMS)
        rope = f64_to_bf16(xs[:, FP8_NOPE_DIMS:]).contiguous().view(torch.uint8).reshape(-1, 128)
        sc = scale.contiguous().view(torch.uint8).reshape(-1, 28)
        o = out[r0:r0 + step]
        o[:, :448] = codes
        o[:, 448:576] = rope
        o[:, 576:604] = sc
    return out.view(*lead, FP8_ROW_BYTES)


def quantize_rows_e4m3(x: torch.Tensor):
    """Per-row e4m3 quantisation (indexer keys): scale = amax/448 per row (1 if zero).
    x: fp64 [..., D]. Returns (uint8 codes [..., D], fp32 scales [...])."""
    amax = x.abs().amax(dim=-1)
    scale = (amax / 448.0).to(torch.float32)
    scale = torch.where(amax == 0, torch.ones_like(scale), scale)
    codes = e4m3_encode(x / scale.to(torch.float64).unsqueeze(-1))
    return codes, scale


def outlier_channels(seed: int, tensor_id: int, d: int, frac: float = 0.01) -> torch.Tensor:
    """A seeded choice of max(1, round(frac*d)) channel indices (fixed for every row)."""
    n = max(1, int(round(frac * d)))
    bits = raw_bits(seed, tensor_id, 0, d, "cpu")
    order = torch.argsort(_srl(bits, 1), stable=True)
    return torch.sort(order[:n]).values


# ----------------------------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------------------------

@dataclass
class Workload:
    """Shapes and hyperparameters of one synthetic workload."""
    name: str
    kind: str                 # "csa_prefill" | "csa_decode" | "hca_decode" | "hca_prefill"
    B: int = 1
    T: int = 0                # prefill tokens (0 for decode)
    N: int = 0                # compressed entries (decode: cache length)
    d: int = 512
    m: int = 4
    rope_dims: int = 64
    H: int = 64
    nI: int = 64
    dI: int = 128
    k: int = 512
    window: int = 128
    theta: float = 160000.0
    eps: float = 1e-6
    fp8: bool = False
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def queries(self) -> int:
        return self.B * (self.T if self.kind.endswith("prefill") else 1)


# The five workloads the method is measured on (sizes from the pages' flash/pro configs).
WORKLOADS = {
    "tiny_csa_prefill_t2048": Workload("tiny_csa_prefill_t2048", "csa_prefill", B=1, T=2048, N=512, d=128,
                                       m=4, H=16, nI=4, dI=64, k=64),
    "csa_decode_128k_b32": Workload("csa_decode_128k_b32", "csa_decode", B=32, N=32768, d=512, m=4, H=64,
                                    nI=64, dI=128, k=512),
    "csa_prefill_t65536": Workload("csa_prefill_t65536", "csa_prefill", B=1, T=65536, N=16384, d=512, m=4,
                                   H=64, nI=64, dI=128, k=512),
    "hca_decode_1m_b8": Workload("hca_decode_1m_b8", "hca_decode", B=8, N=8192, d=512, m=128, H=64, k=0),
    "hca_prefill_t32768": Workload("hca_prefill_t32768", "hca_prefill", B=1, T=32768, N=256, d=512, m=128,
                                   H=64, k=0),
    "csa_decode_1m_b4_fp8": Workload("csa_decode_1m_b4_fp8", "csa_decode", B=4, N=262144, d=512, m=4, H=64,
                                     nI=64, dI=128, k=1024, fp8=True),
}


def scaled(w: Workload, **kw) -> Workload:
    """Same workload at other sizes (parity tests at sizes the oracle finishes quickly)."""
    d = dict(w.__dict__)
    d.update(kw)
    d["extra"] = dict(w.extra)
    return Workload(**d)


def make_inputs(w: Workload, device="cpu") -> dict:
    """All inputs of a workload as tensors on `device`.

    prefill: per-token streams Ca/Cb/Za/Zb [B,T,d] (CSA; HCA: C/Z), indexer streams [B,T,dI],
             q [B,T,H,d], qI [B,T,nI,dI], w [B,T,nI], win [B,T,d] (per-token window KV, slot=position),
             q_pos [B,T] = 0..T-1; the compressor's parameters: position biases Ba/Bb [m,d] (CSA; HCA: B)
             and Ba_I/Bb_I [m,dI] ~ 0.5 N(0,1), RMSNorm weights gamma [d], gamma_I [dI] ~ 1 + 0.1 N(0,1),
             all fp32.
    decode:  kv [B,N,d] (bf16, or packed mixed FP8 rows), kI [B,N,dI] (bf16, or e4m3 + row scales),
             q [B,1,H,d], qI [B,1,nI,dI], w [B,1,nI], win ring [B,128,d] (slot = position mod 128),
             q_pos [B,1] = m*N (the new token's index).
    sink [H] fp32 ~N(0,1) in every case; w ~U(0,1)."""
    s = w.seed
    out = {}
    g = lambda name, shape: normal_bf16(shape, s, TID[name], device)
    f32 = lambda name, shape, scale, shift: (shift + scale * normal_f64(shape, s, TID[name], device)).to(torch.float32)
    out["sink"] = normal_f64((w.H,), s, TID["sink"], device).to(torch.float32)
    if w.kind == "csa_prefill":
        B, T = w.B, w.T
        for nm in ("Ca", "Cb", "Za", "Zb"):
            out[nm] = g(nm, (B, T, w.d))
        for nm in ("Ca_I", "Cb_I", "Za_I", "Zb_I"):
            out[nm] = g(nm, (B, T, w.dI))
        out["q"] = g("q", (B, T, w.H, w.d))
        out["qI"] = g("qI", (B, T, w.nI, w.dI))
        out["w"] = uniform_f64((B, T, w.nI), s, TID["w"], device).to(torch.float32)
        out["win"] = g("win", (B, T, w.d))
        out["q_pos"] = torch.arange(T, dtype=torch.int32, device=device).repeat(B, 1)
        out["Ba"], out["Bb"] = f32("Ba", (w.m, w.d), 0.5, 0.0), f32("Bb", (w.m, w.d), 0.5, 0.0)
        out["Ba_I"], out["Bb_I"] = f32("Ba_I", (w.m, w.dI), 0.5, 0.0), f32("Bb_I", (w.m, w.dI), 0.5, 0.0)
        out["gamma"], out["gamma_I"] = f32("gamma", (w.d,), 0.1, 1.0), f32("gamma_I", (w.dI,), 0.1, 1.0)
    elif w.kind == "hca_prefill":
        B, T = w.B, w.T
        out["C"] = g("C", (B, T, w.d))
        out["Z"] = g("Z", (B, T, w.d))
        out["q"] = g("q", (B, T, w.H, w.d))
        out["win"] = g("win", (B, T, w.d))
        out["q_pos"] = torch.arange(T, dtype=torch.int32, device=device).repeat(B, 1)
        out["B"] = f32("B", (w.m, w.d), 0.5, 0.0)
        out["gamma"] = f32("gamma", (w.d,), 0.1, 1.0)
    elif w.kind in ("csa_decode", "hca_decode"):
        B, N = w.B, w.N
        if w.fp8:
            kv_ch = outlier_channels(s, TID["outlier_kv"], w.d)
            x = normal_f64((B, N, w.d), s, TID["kv"], device)
            x[..., kv_ch.to(device)] *= 20.0
            out["kv"] = pack_kv_fp8_mixed(x)
            del x
        else:
            out["kv"] = g("kv", (B, N, w.d))
        if w.kind == "csa_decode":
            if w.fp8:
                ki_ch = outlier_channels(s, TID["outlier_kI"], w.dI)
                x = normal_f64((B, N, w.dI), s, TID["kI"], device)
                x[..., ki_ch.to(device)] *= 20.0
                out["kI"], out["kI_scale"] = quantize_rows_e4m3(x)
                del x
            else:
                out["kI"] = g("kI", (B, N, w.dI))
            out["qI"] = g("qI", (B, 1, w.nI, w.dI))
            out["w"] = uniform_f64((B, 1, w.nI), s, TID["w"], device).to(torch.float32)
        out["q"] = g("q", (B, 1, w.H, w.d))
        out["win"] = g("win", (B, w.window, w.d))
        out["q_pos"] = torch.full((B, 1), w.m * N, dtype=torch.int32, device=device)
    else:
        raise ValueError(w.kind)
    return out
