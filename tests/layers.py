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


class HostLayer:
    """A whole synthetic layer in host memory (small shapes only)."""

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
