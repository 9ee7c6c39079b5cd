"""fp64 CPU oracle of the MoE FFN layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library's product path never
touches it; it shares no code with the CUDA library (``oracle.c`` re-derives
the record layout and every formula on its own).

This module is a thin ctypes wrapper around ``oracle.c`` (plain single-thread
C, fp64).  See ``oracle.c`` for the formulas and the pages each one follows:
the TurboFieldfare page, sections "Belleği azaltan çalışma yapısı" (affine
4-bit group-64 experts, 8-bit router) and "Token üretim süreci" (router,
top-k, bounded LFU cache, shared expert, combine), and the WASTE page,
sections "Disk streaming mimarisi" (gate, up and down stored contiguously),
"Önceden okuma ve router tahmini" (router lookahead into the cache) and
"Quantization ve doğruluk" (3-bit residual-VQ experts).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")


GCC_FLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp"
        subprocess.check_call(["gcc", *GCC_FLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in
                ("gate_codes", "up_codes", "down_codes", "gate_sb", "up_sb", "down_sb",
                 "bytes", "stride")]


class _Layer(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("F", ctypes.c_int), ("Fs", ctypes.c_int),
                ("records", ctypes.POINTER(ctypes.c_void_p)),
                ("shared_record", ctypes.c_void_p),
                ("router_codes", ctypes.c_void_p),
                ("router_sb", ctypes.c_void_p),
                ("beta", ctypes.c_void_p),
                ("codebooks", ctypes.c_void_p)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Binds this wrapper to another build of oracle.c for the duration (the
    tests use it to run the pins against copies with a planted mistake)."""
    global _lib
    saved = lib()
    _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def _bind(L):
    """Declares the argument and result types of the oracle's C functions."""
    vp, i32, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.orc_bf16_to_double.restype = d
    L.orc_record_layout.argtypes = [i32, i32, ctypes.POINTER(_Layout)]
    L.orc_dequant4.argtypes = [vp, vp, i32, i32, i32]
    L.orc_dequant4.restype = d
    L.orc_dequant8.argtypes = [vp, vp, i32, i32, i32]
    L.orc_dequant8.restype = d
    L.orc_gemv4.argtypes = [vp, vp, i32, i32, vp, vp]
    L.orc_router_logits.argtypes = [vp, vp, vp, i32, i32, vp, vp]
    L.orc_topk.argtypes = [vp, i32, i32, vp, vp, vp]
    L.orc_silu.argtypes = [d]
    L.orc_silu.restype = d
    L.orc_expert.argtypes = [vp, i32, i32, vp, vp, vp]
    L.orc_route.argtypes = [ctypes.POINTER(_Layer), vp, vp, vp, vp, vp, vp]
    L.orc_moe_token.argtypes = [ctypes.POINTER(_Layer), vp, vp, vp, vp, vp, vp]
    L.orc_moe_token.restype = i32
    L.orc_moe_token_dense.argtypes = [ctypes.POINTER(_Layer), vp, vp, vp, vp, vp, vp]
    L.orc_moe_token_dense.restype = i32
    L.orc_lfu_step.argtypes = [i32, i32, vp, vp, vp, vp, i32, ctypes.c_int64, vp, vp]
    L.orc_lfu_step.restype = i32
    L.orc_lfu_lookahead.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp, i32, vp, vp]
    L.orc_lfu_lookahead.restype = i32
    L.orc_rvq_layout.argtypes = [i32, i32, ctypes.POINTER(_Layout)]
    L.orc_dequant_rvq.argtypes = [vp, vp, i32, i32, i32]
    L.orc_dequant_rvq.restype = d
    L.orc_gemv_rvq.argtypes = [vp, vp, i32, i32, vp, vp]
    L.orc_expert_rvq.argtypes = [vp, vp, i32, i32, vp, vp, vp]
    return L


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def bf16_to_double(h: int) -> float:
    return lib().orc_bf16_to_double(h)


def record_layout(H: int, F: int) -> dict:
    L = _Layout()
    lib().orc_record_layout(H, F, ctypes.byref(L))
    return {n: int(getattr(L, n)) for n, _ in _Layout._fields_}


def dequant4(codes: np.ndarray, sb: np.ndarray, cols: int, r: int, j: int) -> float:
    return lib().orc_dequant4(_p(codes), _p(sb), cols, r, j)


def dequant8(codes: np.ndarray, sb: np.ndarray, cols: int, r: int, j: int) -> float:
    return lib().orc_dequant8(_p(codes), _p(sb), cols, r, j)


def gemv4(codes: np.ndarray, sb: np.ndarray, rows: int, cols: int, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.zeros(rows, np.float64)
    lib().orc_gemv4(_p(codes), _p(sb), rows, cols, _p(x), _p(y))
    return y


def rvq_layout(H: int, F: int) -> dict:
    """Byte layout of a 3-bit residual-VQ expert record (see oracle.c)."""
    L = _Layout()
    lib().orc_rvq_layout(H, F, ctypes.byref(L))
    return {n: int(getattr(L, n)) for n, _ in _Layout._fields_}


def dequant_rvq(codes: np.ndarray, cb: np.ndarray, cols: int, r: int, j: int) -> float:
    """Weight (r, j) of an RVQ matrix; cb = one kind's codebooks [3][256][8] bf16."""
    return lib().orc_dequant_rvq(_p(codes), _p(np.ascontiguousarray(cb, np.uint16)), cols, r, j)


def gemv_rvq(codes: np.ndarray, cb: np.ndarray, rows: int, cols: int, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.zeros(rows, np.float64)
    lib().orc_gemv_rvq(_p(codes), _p(np.ascontiguousarray(cb, np.uint16)), rows, cols, _p(x), _p(y))
    return y


def expert_rvq(record: np.ndarray, codebooks: np.ndarray, H: int, F: int, x: np.ndarray) -> np.ndarray:
    """y = W_d(silu(W_g x) * W_u x) for one RVQ record; codebooks [3][3][256][8] bf16."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.zeros(H, np.float64)
    scr = np.zeros(3 * F, np.float64)
    lib().orc_expert_rvq(_p(record), _p(np.ascontiguousarray(codebooks, np.uint16)), H, F, _p(x),
                         _p(y), _p(scr))
    return y


def silu(z: float) -> float:
    return lib().orc_silu(z)


def expert(record: np.ndarray, H: int, F: int, x: np.ndarray) -> np.ndarray:
    """y = W_d(silu(W_g x) * W_u x) for one expert record (x in float64)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.zeros(H, np.float64)
    scr = np.zeros(3 * F, np.float64)
    lib().orc_expert(_p(record), H, F, _p(x), _p(y), _p(scr))
    return y


class Layer:
    """Host view of one layer for the oracle: every buffer is a numpy array in
    the library's record format.  ``records`` maps expert id -> record bytes;
    missing experts are allowed as long as the token does not select them."""

    def __init__(self, H, E, k, F, Fs, records, shared_record, router_codes, router_sb,
                 beta=None, codebooks=None):
        """codebooks: bf16 [3][3][256][8] for a layer of 3-bit residual-VQ
        experts; None for 4-bit affine experts."""
        self.H, self.E, self.k, self.F, self.Fs = H, E, k, F, Fs
        self._cb = None if codebooks is None else np.ascontiguousarray(codebooks, dtype=np.uint16)
        self._recs = dict(records)
        self._shared = shared_record
        self._rc = np.ascontiguousarray(router_codes, dtype=np.uint8)
        self._rsb = np.ascontiguousarray(router_sb, dtype=np.uint32)
        self._beta = None if beta is None else np.ascontiguousarray(beta, dtype=np.float32)
        self._ptrs = (ctypes.c_void_p * E)()
        for e in range(E):
            r = self._recs.get(e)
            self._ptrs[e] = None if r is None else r.ctypes.data
        self._c = _Layer(H, E, k, F, Fs,
                         ctypes.cast(self._ptrs, ctypes.POINTER(ctypes.c_void_p)),
                         None if shared_record is None else shared_record.ctypes.data,
                         self._rc.ctypes.data, self._rsb.ctypes.data,
                         None if self._beta is None else self._beta.ctypes.data,
                         None if self._cb is None else self._cb.ctypes.data)

    def set_record(self, e: int, rec: np.ndarray):
        self._recs[e] = rec
        self._ptrs[e] = rec.ctypes.data

    def route(self, x_bf16: np.ndarray):
        """Returns (logits[E], ids[k], p[k]) for one token."""
        x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
        xd = np.zeros(self.H, np.float64)
        logits = np.zeros(self.E, np.float64)
        ids = np.zeros(self.k, np.int32)
        p = np.zeros(self.k, np.float64)
        taken = np.zeros(self.E, np.uint8)
        lib().orc_route(ctypes.byref(self._c), _p(x), _p(xd), _p(logits), _p(ids), _p(p),
                        _p(taken))
        return logits, ids, p

    def _work(self):
        return np.zeros(2 * self.H + self.E + 3 * max(self.F, self.Fs, 1), np.float64)

    def token(self, x_bf16: np.ndarray, dense: bool = False):
        """Full layer for one token: returns (out[H] float64, ids[k], p[k])."""
        x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
        out = np.zeros(self.H, np.float64)
        ids = np.zeros(self.k, np.int32)
        p = np.zeros(self.k, np.float64)
        taken = np.zeros(self.E, np.uint8)
        work = self._work()
        if dense:
            rc = lib().orc_moe_token_dense(ctypes.byref(self._c), _p(x), _p(out), _p(work),
                                           _p(taken), _p(ids), _p(p))
        else:
            rc = lib().orc_moe_token(ctypes.byref(self._c), _p(x), _p(out), _p(ids), _p(p),
                                     _p(work), _p(taken))
        if rc != 0:
            raise KeyError("a selected expert's record is missing from the oracle layer")
        return out, ids, p


def waves(ids: np.ndarray, n_slots: int):
    """Splits a step's tokens into waves of consecutive tokens whose distinct
    experts fit the cache: a wave grows token by token while the union of
    its tokens' ids has at most n_slots experts.  ids[B][k]; returns the
    [t0, t1) bounds.  (The pages give a cache of fixed size and a router of
    k experts per token, and no rule for a step that needs more; reading:
    run it as several steps, tokens in order.)"""
    ids = np.asarray(ids)
    out, t0, have = [], 0, set()
    for t in range(ids.shape[0]):
        row = set(int(e) for e in ids[t])
        if len(have | row) > n_slots:
            out.append((t0, t))
            t0, have = t, set()
        have |= row
    if ids.shape[0]:
        out.append((t0, ids.shape[0]))
    return out


class LFU:
    """Replays the bounded LFU residency policy on an id stream, with the
    optional router lookahead between demand steps (see oracle.c).

    Cumulative counters, in the library's terms: hits, misses, evictions,
    lookahead_copies, lookahead_hits (demand hits on a record a lookahead
    copied and no demand step had used yet)."""

    def __init__(self, n_slots: int, E: int):
        self.n_slots, self.E = n_slots, E
        self.slot_expert = np.full(n_slots, -1, np.int32)
        self.count = np.zeros(E, np.int64)
        self.last_use = np.zeros(E, np.int64)
        self.pinned = np.zeros(E, np.uint8)   # lookahead pins, cleared by the next demand step
        self.fresh = np.zeros(E, np.uint8)    # copied by a lookahead, not yet used
        self.step_no = 0
        self.hits = self.misses = self.evictions = 0
        self.lookahead_copies = self.lookahead_hits = 0

    def step(self, ids: np.ndarray):
        """One demand step over the step's distinct ids (first-appearance
        order).  Returns (hit[k] bool, slot[k] int, misses)."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        k = ids.size
        hit = np.zeros(k, np.int32)
        slot = np.zeros(k, np.int32)
        empty = int((self.slot_expert < 0).sum())
        self.pinned[:] = 0
        self.step_no += 1
        m = lib().orc_lfu_step(self.n_slots, self.E, _p(self.slot_expert), _p(self.count),
                               _p(self.last_use), _p(ids), k, self.step_no, _p(hit), _p(slot))
        if m < 0:
            raise ValueError("more distinct experts in one step than slots")
        self.lookahead_hits += int(sum(1 for e, h in zip(ids, hit) if h and self.fresh[e]))
        self.fresh[ids] = 0
        gone = np.ones(self.E, bool)
        gone[self.slot_expert[self.slot_expert >= 0]] = False
        self.fresh[gone] = 0
        self.hits += int(hit.sum())
        self.misses += m
        self.evictions += m - min(m, empty)
        return hit.astype(bool), slot, m

    def lookahead(self, pred: np.ndarray, n_ahead: int):
        """A lookahead over predicted rankings pred[B][k] (each row in rank
        order), taking each token's first n_ahead.  Returns (slot[] of the
        visited predictions, -1 where dropped; copies; evictions)."""
        pred = np.asarray(pred, dtype=np.int32)
        if pred.ndim == 1:
            pred = pred[None]
        order = np.ascontiguousarray(pred[:, :n_ahead].T.reshape(-1))  # rank-major
        slot = np.zeros(order.size, np.int32)
        ev = ctypes.c_int(0)
        c = lib().orc_lfu_lookahead(self.n_slots, self.E, _p(self.slot_expert), _p(self.count),
                                    _p(self.last_use), _p(self.pinned), _p(self.fresh), _p(order),
                                    int(order.size), _p(slot), ctypes.byref(ev))
        self.lookahead_copies += c
        self.evictions += ev.value
        return slot, c, ev.value
