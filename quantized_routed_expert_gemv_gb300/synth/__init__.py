"""Seeded synthetic workloads for the MoE FFN layer.

Draws expert records, router matrices, hidden states and per-expert logit
offsets in the library's record format from a counter-based SplitMix64
stream (``synth.c``).  It holds none of the layer's arithmetic, so the CUDA
library and the fp64 oracle can both be fed from it.  Every value depends
only on (seed, tensor, layer, expert/token, index), so single experts of a
12.7 GB layer can be regenerated on demand.

Workload shapes and value distributions (the MoE layers that the pages'
streaming engines run: 4-bit affine group-64 experts and an 8-bit router,
TurboFieldfare page, section "Belleği azaltan çalışma yapısı"; 16 routed
experts per K3 layer, WASTE page, section "RAM bütçesi ve dar performans
aralığı"):

* expert codes uniform 0..15; scale ~ U[0.005, 0.02] and bias ~ N(0, 0.05),
  both rounded to bf16;
* router codes uniform 0..255; scale ~ U[0.005, 0.02] / 16, bias ~ N(0, 0.05);
* hidden states ~ N(0, 1) rounded to bf16;
* skewed routing: per-expert logit offset beta ~ N(0, 1);
* streamed-cache routing: beta_e = ln p_{pi(e)}, p_r proportional to r^-1.1
  (Zipf), pi a seeded permutation.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_SRC = os.path.join(_HERE, "synth.c")

EXPERT_SCALE = (0.005, 0.02)
EXPERT_BIAS_SD = 0.05
ROUTER_SCALE = (0.005 / 16, 0.02 / 16)
ROUTER_BIAS_SD = 0.05

TAG_HIDDEN = 10
TAG_BETA = 11
TAG_PERM = 12
TAG_RVQ_CODES = 13
TAG_RVQ_CB = 14

# 3-bit residual VQ experts: codeword values ~ N(0, sd) per stage, rounded to
# bf16, each stage finer than the one before (the pages give no distribution;
# these give weights of about the spread of the 4-bit experts' dequantised
# values around their mean).
RVQ_STAGE_SD = (0.05, 0.02, 0.01)


def build(force: bool = False) -> str:
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC",
                               "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        u64, vp, i32, d = ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        L.synth_key.argtypes = [u64] * 5
        L.synth_key.restype = u64
        L.synth_draw.argtypes = [u64, u64]
        L.synth_draw.restype = u64
        L.synth_bf16_from_double.argtypes = [d]
        L.synth_bf16_from_double.restype = ctypes.c_uint16
        L.synth_fill_bytes.argtypes = [u64, vp, ctypes.c_size_t]
        L.synth_fill_bf16_uniform.argtypes = [u64, vp, ctypes.c_size_t, d, d]
        L.synth_fill_bf16_normal.argtypes = [u64, vp, ctypes.c_size_t, d, d]
        L.synth_fill_f64_uniform.argtypes = [u64, vp, ctypes.c_size_t]
        L.synth_fill_f64_normal.argtypes = [u64, vp, ctypes.c_size_t]
        L.synth_record_stride.argtypes = [i32, i32]
        L.synth_record_stride.restype = u64
        L.synth_expert_record.argtypes = [u64, i32, i32, i32, i32, d, d, d, vp]
        L.synth_router.argtypes = [u64, i32, i32, i32, d, d, d, vp, vp]
        _lib = L
    return _lib


@dataclass(frozen=True)
class Shape:
    """Layer shape: hidden H, routed experts E, top-k, expert FFN F, shared FFN Fs."""
    H: int
    E: int
    k: int
    F: int
    Fs: int


TINY = Shape(256, 8, 2, 128, 256)
MID = Shape(2048, 128, 8, 768, 2048)
LARGE = Shape(7168, 512, 16, 2048, 2048)


@dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    weight_seed: int      # seed of the weights
    input_seed: int       # seed of hidden states / routing offsets
    layers: int = 1
    beta: str = "none"    # "none" | "normal" | "zipf"


WORKLOADS = {
    "tiny": Workload("tiny", TINY, 0, 0),
    "mid-decode": Workload("mid-decode", MID, 1, 1),
    "mid-prefill": Workload("mid-prefill", MID, 1, 2, beta="normal"),
    "large-decode": Workload("large-decode", LARGE, 3, 3),
    "large-streamed": Workload("large-streamed", LARGE, 4, 4, layers=4, beta="zipf"),
}


def key(seed, tag, a=0, b=0, c=0) -> int:
    return lib().synth_key(seed, tag, a, b, c)


def record_stride(H: int, F: int) -> int:
    return int(lib().synth_record_stride(H, F))


def bf16_from_double(v: float) -> int:
    return int(lib().synth_bf16_from_double(v))


def expert_record(seed: int, layer: int, e: int, H: int, F: int, out: np.ndarray | None = None):
    """One expert record (the shared expert uses e = E) as uint8[stride]."""
    n = record_stride(H, F)
    if out is None:
        out = np.empty(n, np.uint8)
    assert out.nbytes >= n and out.flags["C_CONTIGUOUS"]
    lib().synth_expert_record(seed, layer, e, H, F, EXPERT_SCALE[0], EXPERT_SCALE[1],
                              EXPERT_BIAS_SD, out.ctypes.data)
    return out


def fill_records(seed: int, layer: int, experts, H: int, F: int, out: np.ndarray, threads=None):
    """Writes records of `experts` back to back into out (uint8, >= n*stride), in parallel."""
    stride = record_stride(H, F)
    experts = list(experts)
    assert out.nbytes >= stride * len(experts)
    base = out.ctypes.data
    L = lib()

    def one(i):
        L.synth_expert_record(seed, layer, experts[i], H, F, EXPERT_SCALE[0], EXPERT_SCALE[1],
                              EXPERT_BIAS_SD, base + i * stride)

    threads = threads or min(32, os.cpu_count() or 1)
    if len(experts) <= 1 or threads <= 1:
        for i in range(len(experts)):
            one(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(len(experts))))
    return out


def rvq_record_stride(H: int, F: int) -> int:
    """Stride of a 3-bit residual-VQ record: 3 code bytes per 8 weights of
    gate, up and down, rounded up to 4096 bytes."""
    return (3 * (3 * F * H // 8) + 4095) // 4096 * 4096


def rvq_expert_record(seed: int, layer: int, e: int, H: int, F: int, out: np.ndarray | None = None):
    """One RVQ expert record (the shared expert uses e = E) as uint8[stride]:
    uniform code bytes, zero padding."""
    n, payload = rvq_record_stride(H, F), 3 * (3 * F * H // 8)
    if out is None:
        out = np.empty(n, np.uint8)
    assert out.nbytes >= n and out.flags["C_CONTIGUOUS"]
    lib().synth_fill_bytes(key(seed, TAG_RVQ_CODES, layer, e), out.ctypes.data, payload)
    out[payload:n] = 0
    return out


def fill_rvq_records(seed: int, layer: int, experts, H: int, F: int, out: np.ndarray, threads=None):
    """RVQ records of `experts` back to back into out (uint8, >= n*stride)."""
    stride = rvq_record_stride(H, F)
    experts = list(experts)
    assert out.nbytes >= stride * len(experts)
    flat = out.reshape(-1)

    def one(i):
        rvq_expert_record(seed, layer, experts[i], H, F, flat[i * stride:(i + 1) * stride])

    threads = threads or min(32, os.cpu_count() or 1)
    if len(experts) <= 1 or threads <= 1:
        for i in range(len(experts)):
            one(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(len(experts))))
    return out


def rvq_codebooks(seed: int, layer: int) -> np.ndarray:
    """A layer's RVQ codebooks, bf16 bits uint16[3 kinds (gate, up, down)][3 stages][256][8]."""
    out = np.empty((3, 3, 256, 8), np.uint16)
    for kind in range(3):
        for st in range(3):
            lib().synth_fill_bf16_normal(key(seed, TAG_RVQ_CB, layer, kind, st), out[kind, st].ctypes.data,
                                         256 * 8, 0.0, RVQ_STAGE_SD[st])
    return out


def router(seed: int, layer: int, E: int, H: int):
    """(codes uint8[E][H], sb uint32[E][H/64])."""
    codes = np.empty((E, H), np.uint8)
    sb = np.empty((E, H // 64), np.uint32)
    lib().synth_router(seed, layer, E, H, ROUTER_SCALE[0], ROUTER_SCALE[1], ROUTER_BIAS_SD,
                       codes.ctypes.data, sb.ctypes.data)
    return codes, sb


def hidden(seed: int, stream: int, token: int, H: int, attempt: int = 0) -> np.ndarray:
    """One hidden state, bf16 bits uint16[H], ~ N(0,1)."""
    out = np.empty(H, np.uint16)
    lib().synth_fill_bf16_normal(key(seed, TAG_HIDDEN, stream, token, attempt), out.ctypes.data,
                                 H, 0.0, 1.0)
    return out


def hidden_chain(seed: int, token: int, H: int, layers: int, rho: float) -> np.ndarray:
    """Hidden states of one token at successive layers, bf16 bits
    uint16[layers][H], standing in for a residual stream that each layer
    changes only in part: x_0 = z_0 and x_{l+1} = bf16(f32(rho * x_l +
    sqrt(1 - rho^2) * z_{l+1})), with z_l = hidden(seed, l, token, H).  Every
    x_l stays ~ N(0, 1); rho = 0 gives the independent per-layer draws."""
    out = np.empty((layers, H), np.uint16)
    out[0] = hidden(seed, 0, token, H)
    c = float(np.sqrt(max(0.0, 1.0 - rho * rho)))
    for l in range(1, layers):
        prev = bf16_bits_to_float(out[l - 1]).astype(np.float64)
        z = bf16_bits_to_float(hidden(seed, l, token, H)).astype(np.float64)
        out[l] = float_to_bf16_bits((rho * prev + c * z).astype(np.float32))
    return out


def uniforms(k: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float64)
    lib().synth_fill_f64_uniform(k, out.ctypes.data, n)
    return out


def normals(k: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float64)
    lib().synth_fill_f64_normal(k, out.ctypes.data, n)
    return out


def beta_normal(seed: int, layer: int, E: int) -> np.ndarray:
    """Per-expert logit offset ~ N(0, 1) (skewed routing), float32[E]."""
    return normals(key(seed, TAG_BETA, layer), E).astype(np.float32)


def beta_zipf(seed: int, layer: int, E: int, s: float = 1.1) -> np.ndarray:
    """beta_e = ln p_{pi(e)}, p_r proportional to r^-s over ranks 1..E, float32[E]."""
    ranks = np.arange(1, E + 1, dtype=np.float64)
    w = ranks ** (-s)
    logp = np.log(w / w.sum())
    perm = np.argsort(uniforms(key(seed, TAG_PERM, layer), E), kind="stable")
    return logp[perm].astype(np.float32)


def beta_for(wl: Workload, layer: int = 0):
    E = wl.shape.E
    if wl.beta == "normal":
        return beta_normal(wl.input_seed, layer, E)
    if wl.beta == "zipf":
        return beta_zipf(wl.input_seed, layer, E)
    return None


def zipf_probabilities(E: int, s: float = 1.1) -> np.ndarray:
    r = np.arange(1, E + 1, dtype=np.float64)
    w = r ** (-s)
    return w / w.sum()


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (a format conversion)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def float_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bit patterns (finite inputs)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def pack_codes4(q: np.ndarray) -> np.ndarray:
    """[rows][cols] codes 0..15 -> [rows][cols/2] bytes, element j in byte j/2,
    low nibble for even j (the library's packing)."""
    q = np.asarray(q, np.uint8)
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)


def pack_sb(scale_bits: np.ndarray, bias_bits: np.ndarray) -> np.ndarray:
    return (np.asarray(scale_bits, np.uint32) | (np.asarray(bias_bits, np.uint32) << 16)).astype(
        np.uint32)


def assemble_record(H: int, F: int, gate_q, gate_s, gate_b, up_q, up_s, up_b, down_q, down_s,
                    down_b) -> np.ndarray:
    """Builds one record from explicit codes ([out][in], 0..15) and bf16 bit
    patterns of scale/bias ([out][in/64]) -- used for hand-built layers."""
    stride = record_stride(H, F)
    rec = np.zeros(stride, np.uint8)
    parts = [pack_codes4(gate_q), pack_codes4(up_q), pack_codes4(down_q),
             pack_sb(gate_s, gate_b), pack_sb(up_s, up_b), pack_sb(down_s, down_b)]
    off = 0
    for p in parts:
        b = np.ascontiguousarray(p).view(np.uint8).reshape(-1)
        rec[off:off + b.size] = b
        off += b.size
    return rec
