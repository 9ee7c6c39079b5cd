"""Host-side layer builders shared by the tests.

Everything here either draws data through ``synth`` or builds hand-made
layers whose outputs have closed forms.  The only arithmetic of the layer it
contains is the test-side dense dequantisation used to hand whole matrices
to library routines (numpy / torch) -- never to the CUDA path.
"""
from __future__ import annotations

import numpy as np

import oracle
from quantized_routed_expert_gemv_gb300 import synth


def unpack4(packed: np.ndarray, rows: int, cols: int) -> np.ndarray:
    b = np.asarray(packed, np.uint8).reshape(rows, cols // 2)
    q = np.empty((rows, cols), np.uint8)
    q[:, 0::2] = b & 0x0F
    q[:, 1::2] = b >> 4
    return q


def sb_split(words: np.ndarray):
    w = np.asarray(words, np.uint32)
    s = synth.bf16_bits_to_float((w & 0xFFFF).astype(np.uint16)).astype(np.float64)
    b = synth.bf16_bits_to_float((w >> 16).astype(np.uint16)).astype(np.float64)
    return s, b


def dense4(codes: np.ndarray, sb: np.ndarray, rows: int, cols: int) -> np.ndarray:
    q = unpack4(codes, rows, cols).astype(np.float64)
    s, b = sb_split(np.asarray(sb).reshape(rows, cols // 64))
    return q * np.repeat(s, 64, axis=1) + np.repeat(b, 64, axis=1)


def dense8(codes: np.ndarray, sb: np.ndarray, rows: int, cols: int) -> np.ndarray:
    q = np.asarray(codes, np.uint8).reshape(rows, cols).astype(np.float64)
    s, b = sb_split(np.asarray(sb).reshape(rows, cols // 64))
    return q * np.repeat(s, 64, axis=1) + np.repeat(b, 64, axis=1)


def record_mats(rec: np.ndarray, H: int, F: int):
    """Dense (W_g [F][H], W_u [F][H], W_d [H][F]) of one record."""
    L = oracle.record_layout(H, F)
    cg = rec[L["gate_codes"]:L["up_codes"]]
    cu = rec[L["up_codes"]:L["down_codes"]]
    cd = rec[L["down_codes"]:L["gate_sb"]]
    sg = rec[L["gate_sb"]:L["up_sb"]].view(np.uint32)
    su = rec[L["up_sb"]:L["down_sb"]].view(np.uint32)
    sd = rec[L["down_sb"]:L["bytes"]].view(np.uint32)
    return dense4(cg, sg, F, H), dense4(cu, su, F, H), dense4(cd, sd, H, F)


def dense_rvq(codes: np.ndarray, cb: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Dense [rows][cols] float64 of a 3-bit residual-VQ matrix, by numpy
    gathers: cb is one kind's codebooks [3][256][8] (bf16 bits)."""
    q = np.asarray(codes, np.uint8).reshape(rows, cols // 8, 3)
    c = synth.bf16_bits_to_float(np.asarray(cb, np.uint16)).astype(np.float64)
    return (c[0][q[..., 0]] + c[1][q[..., 1]] + c[2][q[..., 2]]).reshape(rows, cols)


def rvq_record_mats(rec: np.ndarray, cbs: np.ndarray, H: int, F: int):
    """Dense (W_g, W_u, W_d) of one RVQ record; cbs [3 kinds][3][256][8]."""
    L = oracle.rvq_layout(H, F)
    return (dense_rvq(rec[L["gate_codes"]:L["up_codes"]], cbs[0], F, H),
            dense_rvq(rec[L["up_codes"]:L["down_codes"]], cbs[1], F, H),
            dense_rvq(rec[L["down_codes"]:L["bytes"]], cbs[2], H, F))


class HostLayer:
    """A whole synthetic layer in host memory (small shapes only)."""

    def mats(self, rec: np.ndarray, F: int):
        return record_mats(rec, self.shape.H, F)

    def __init__(self, shape: synth.Shape, seed: int, layer: int = 0, beta=None):
        self.shape = shape
        H, E, F, Fs = shape.H, shape.E, shape.F, shape.Fs
        self.stride = synth.record_stride(H, F)
        self.records = np.zeros((E, self.stride), np.uint8)
        synth.fill_records(seed, layer, range(E), H, F, self.records)
        self.shared = synth.expert_record(seed, layer, E, H, Fs) if Fs else None
        self.router_codes, self.router_sb = synth.router(seed, layer, E, H)
        self.beta = beta

    def oracle(self) -> oracle.Layer:
        s = self.shape
        return oracle.Layer(s.H, s.E, s.k, s.F, s.Fs, {e: self.records[e] for e in range(s.E)},
                            self.shared, self.router_codes, self.router_sb, self.beta)


class HostLayerRVQ:
    """A synthetic layer of 3-bit residual-VQ experts in host memory."""

    def __init__(self, shape: synth.Shape, seed: int, layer: int = 0, beta=None):
        self.shape = shape
        H, E, F, Fs = shape.H, shape.E, shape.F, shape.Fs
        self.stride = synth.rvq_record_stride(H, F)
        self.records = np.zeros((E, self.stride), np.uint8)
        synth.fill_rvq_records(seed, layer, range(E), H, F, self.records)
        self.shared = synth.rvq_expert_record(seed, layer, E, H, Fs) if Fs else None
        self.codebooks = synth.rvq_codebooks(seed, layer)
        self.router_codes, self.router_sb = synth.router(seed, layer, E, H)
        self.beta = beta

    def mats(self, rec: np.ndarray, F: int):
        return rvq_record_mats(rec, self.codebooks, self.shape.H, F)

    def oracle(self) -> oracle.Layer:
        s = self.shape
        return oracle.Layer(s.H, s.E, s.k, s.F, s.Fs, {e: self.records[e] for e in range(s.E)},
                            self.shared, self.router_codes, self.router_sb, self.beta,
                            codebooks=self.codebooks)


def identity_layer_rvq(E: int = 8, k: int = 2, H: int = 64):
    """The identity-expert layer of identity_layer() in the RVQ format
    (H = F = Fs): stage 1 codeword 1 of the gate books is (8, 0, ..., 0),
    codewords 1..8 of the up books are the unit vectors, codeword 1 + 8a + i
    of the down books is 2^-(6 + a) e_i; every other codeword, and all of
    stages 2 and 3, is zero.  Gate rows use (1, 0, 0) in block 0, up row j
    codeword 1 + j%8 in block j/8, down row r of an expert with a = e mod 3
    codeword 1 + 8a + r%8 in block r/8; other blocks code 0.  With x_0 = 8,
        out = (1 + sum_i p_i 2^-a_{e_i}) x."""
    F = H
    cbs = np.zeros((3, 3, 256, 8), np.uint16)
    cbs[0, 0, 1, 0] = synth.bf16_from_double(8.0)
    for i in range(8):
        cbs[1, 0, 1 + i, i] = synth.bf16_from_double(1.0)
        for a in range(3):
            cbs[2, 0, 1 + 8 * a + i, i] = synth.bf16_from_double(2.0 ** -(6 + a))
    stride = synth.rvq_record_stride(H, F)

    def rec(a):
        g = np.zeros((F, H // 8, 3), np.uint8)
        g[:, 0, 0] = 1
        u = np.zeros((F, H // 8, 3), np.uint8)
        u[np.arange(F), np.arange(F) // 8, 0] = 1 + np.arange(F) % 8
        d = np.zeros((H, F // 8, 3), np.uint8)
        d[np.arange(H), np.arange(H) // 8, 0] = 1 + 8 * a + np.arange(H) % 8
        out = np.zeros(stride, np.uint8)
        body = np.concatenate([g.ravel(), u.ravel(), d.ravel()])
        out[:body.size] = body
        return out

    records = np.stack([rec(e % 3) for e in range(E)])
    shared = rec(0)
    rc, rsb = synth.router(12345, 0, E, H)
    return records, shared, rc, rsb, cbs


def margin_ok(logits: np.ndarray, k: int, margin: float = 1e-3) -> bool:
    if k >= logits.size:
        return True
    srt = np.sort(logits)[::-1]
    return (srt[k - 1] - srt[k]) >= margin


def hidden_with_margin(orc: oracle.Layer, seed: int, stream: int, token: int,
                       margin: float = 1e-3, max_attempts: int = 64) -> np.ndarray:
    """Draws the token's hidden state, redrawing (attempt 1, 2, ...) from the
    same stream until the oracle's k-th/(k+1)-th logit gap is >= margin."""
    for a in range(max_attempts):
        x = synth.hidden(seed, stream, token, orc.H, attempt=a)
        logits, _, _ = orc.route(x)
        if margin_ok(logits, orc.k, margin):
            return x
    raise RuntimeError("no hidden state with the required router margin")


def identity_layer(E: int = 8, k: int = 2, H: int = 64):
    """Identity-expert layer: H = F = Fs = 64.  Gate rows have code 8 at
    input 0 (scale 1, bias 0), up row j is the unit vector e_j, down is the
    diagonal with scale 2^-(6 + a) (a = e mod 3 for routed expert e, 0 for
    the shared expert).  With x_0 = 8: g_j = 64, silu(64) = 64 exactly in
    float64, h_j = 64 x_j and y_e = 2^-a_e x, so
        out = (1 + sum_i p_i 2^-a_{e_i}) x."""
    F = H
    one = synth.bf16_from_double(1.0)
    zero = synth.bf16_from_double(0.0)
    G = H // 64

    def rec(a):
        gq = np.zeros((F, H), np.uint8)
        gq[:, 0] = 8
        uq = np.zeros((F, H), np.uint8)
        uq[np.arange(F), np.arange(F)] = 1
        dq = np.zeros((H, F), np.uint8)
        dq[np.arange(H), np.arange(H)] = 1
        ones = np.full((F, G), one, np.uint16)
        zeros = np.full((F, G), zero, np.uint16)
        ds = np.full((H, F // 64), synth.bf16_from_double(2.0 ** -(6 + a)), np.uint16)
        return synth.assemble_record(H, F, gq, ones, zeros, uq, ones, zeros, dq, ds,
                                     np.full((H, F // 64), zero, np.uint16))

    records = np.stack([rec(e % 3) for e in range(E)])
    shared = rec(0)
    rc, rsb = synth.router(12345, 0, E, H)
    return records, shared, rc, rsb
