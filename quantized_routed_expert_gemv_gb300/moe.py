"""Python binding of the C ABI in ``include/moe.h`` (ctypes, marshalling only).

Every function keeps the C name and takes raw addresses (ints) for device and
host buffers, exactly like the C call.  No step of the layer runs here: if
``libmoe.so`` is missing the first call raises instead of falling back to
anything else.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_ARG = -1
MOE_ERR_ALIGN = -2
MOE_ERR_CUDA = -3
MOE_ERR_TIMEOUT = -4
MOE_ERR_RESIDENCY = -5
MOE_ERR_NOMEM = -6
MOE_ERR_UNSUPPORTED = -7

# bytes of the static device scratch behind moe_decode_noalloc (include/moe.h)
MOE_NOALLOC_SCRATCH_BYTES = 16 << 20

ERROR_NAMES = {0: "MOE_OK", -1: "MOE_ERR_ARG", -2: "MOE_ERR_ALIGN", -3: "MOE_ERR_CUDA",
               -4: "MOE_ERR_TIMEOUT", -5: "MOE_ERR_RESIDENCY", -6: "MOE_ERR_NOMEM",
               -7: "MOE_ERR_UNSUPPORTED"}


class moe_layer_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("hidden", "n_experts", "top_k", "ffn", "shared_ffn",
                                              "group", "wbits", "rbits", "max_tokens")]


class moe_record_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("gate_codes", "up_codes", "down_codes", "gate_sb",
                                               "up_sb", "down_sb", "bytes", "stride")]


class moe_layer_weights(ctypes.Structure):
    _fields_ = [("expert_records", ctypes.c_void_p), ("shared_record", ctypes.c_void_p),
                ("router_codes", ctypes.c_void_p), ("router_sb", ctypes.c_void_p),
                ("router_logit_bias", ctypes.c_void_p), ("expert_codebooks", ctypes.c_void_p)]


class moe_residency_stats_t(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_uint64), ("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64),
                ("evictions", ctypes.c_uint64), ("bytes_h2d", ctypes.c_uint64),
                ("lookaheads", ctypes.c_uint64), ("lookahead_copies", ctypes.c_uint64),
                ("lookahead_hits", ctypes.c_uint64), ("lookahead_bytes", ctypes.c_uint64)]


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where}: {ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None

_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t

# name -> (restype, argtypes)
SIGNATURES = {
    "moe_record_layout_of": (ctypes.c_int, [_i32, _i32, ctypes.POINTER(moe_record_layout)]),
    "moe_expert_bytes": (_sz, [ctypes.POINTER(moe_layer_desc), _i32]),
    "moe_open": (ctypes.c_int, [ctypes.POINTER(moe_layer_desc), ctypes.POINTER(moe_layer_weights),
                                ctypes.POINTER(_vp)]),
    "moe_close": (None, [_vp]),
    "moe_workspace_bytes": (_sz, [_vp, _i32]),
    "moe_workspace_init": (ctypes.c_int, [_vp, _vp, _sz, _vp]),
    "moe_decode": (ctypes.c_int, [_vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_prefill_chunk": (ctypes.c_int, [_vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_decode_host": (ctypes.c_int, [_vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_check": (ctypes.c_int, [_vp, _vp, _vp]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_set_profile_events": (ctypes.c_int, [_vp, ctypes.POINTER(_vp)]),
    "moe_residency_pool_bytes": (_sz, [_vp, _i32]),
    "moe_residency_open": (ctypes.c_int, [_vp, _vp, _i32, _vp, _sz, ctypes.POINTER(_vp)]),
    "moe_residency_decode": (ctypes.c_int, [_vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp,
                                            _vp]),
    "moe_residency_stats": (ctypes.c_int, [_vp, ctypes.POINTER(moe_residency_stats_t)]),
    "moe_residency_slots": (ctypes.c_int, [_vp, _vp, _i32]),
    "moe_residency_set_fault": (ctypes.c_int, [_vp, _i32]),
    "moe_residency_close": (None, [_vp]),
    "moe_decode_noalloc": (ctypes.c_int, [_vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp]),
    "moe_check_noalloc": (ctypes.c_int, [_vp, _vp]),
    "moe_decode_kernels": (_i32, [_vp, _i32]),
    "moe_residency_verify": (ctypes.c_int, [_vp, _vp]),
    "moe_crc32": (ctypes.c_uint32, [_vp, _sz]),
    "moe_residency_lookahead": (ctypes.c_int, [_vp, _vp, _i32, _i32, _vp, _vp, _vp, _sz, _vp, _vp]),
    "moe_rvq_record_layout_of": (ctypes.c_int, [_i32, _i32, ctypes.POINTER(moe_record_layout)]),
}


def lib():
    """Loads libmoe.so (built by ``quantized_routed_expert_gemv_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            if hasattr(L, name):
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def last_error() -> str:
    return lib().moe_last_error().decode()


def check(rc: int, where: str) -> int:
    if rc != MOE_OK:
        raise MoEError(rc, where, last_error())
    return rc


def desc(H, E, k, F, Fs, max_tokens=16, group=64, wbits=4, rbits=8) -> moe_layer_desc:
    return moe_layer_desc(H, E, k, F, Fs, group, wbits, rbits, max_tokens)


def moe_record_layout_of(hidden: int, ffn: int) -> dict:
    out = moe_record_layout()
    check(lib().moe_record_layout_of(hidden, ffn, ctypes.byref(out)), "moe_record_layout_of")
    return {n: int(getattr(out, n)) for n, _ in moe_record_layout._fields_}


def moe_expert_bytes(d: moe_layer_desc, ffn: int) -> int:
    return int(lib().moe_expert_bytes(ctypes.byref(d), ffn))


def moe_open(d: moe_layer_desc, w: moe_layer_weights) -> int:
    h = _vp()
    check(lib().moe_open(ctypes.byref(d), ctypes.byref(w), ctypes.byref(h)), "moe_open")
    return h.value


def moe_close(layer: int) -> None:
    lib().moe_close(layer)


def moe_workspace_bytes(layer: int, max_tokens: int) -> int:
    return int(lib().moe_workspace_bytes(layer, max_tokens))


def moe_workspace_init(layer: int, ws: int, nbytes: int, stream: int = 0) -> None:
    check(lib().moe_workspace_init(layer, ws, nbytes, stream), "moe_workspace_init")


def moe_decode(layer, x, B, out_bf16, out_f32, ids, weights, ws, ws_bytes, stream=0) -> None:
    check(lib().moe_decode(layer, x, B, out_bf16, out_f32, ids, weights, ws, ws_bytes, stream),
          "moe_decode")


def moe_prefill_chunk(layer, x, T, out_bf16, out_f32, ids, weights, ws, ws_bytes, stream=0) -> None:
    check(lib().moe_prefill_chunk(layer, x, T, out_bf16, out_f32, ids, weights, ws, ws_bytes,
                                  stream), "moe_prefill_chunk")


def moe_decode_host(layer, x, B, out_bf16, out_f32, ids, weights, ws, ws_bytes, stream=0) -> None:
    check(lib().moe_decode_host(layer, x, B, out_bf16, out_f32, ids, weights, ws, ws_bytes,
                                stream), "moe_decode_host")


def moe_decode_noalloc(layer, x, B, out_bf16, out_f32, ids, weights, stream=0) -> None:
    """moe_decode with the workspace in the library's static device scratch."""
    check(lib().moe_decode_noalloc(layer, x, B, out_bf16, out_f32, ids, weights, stream),
          "moe_decode_noalloc")


def moe_check_noalloc(layer: int, stream: int = 0) -> int:
    """Status of the static scratch of moe_decode_noalloc (moe_check's codes);
    clears its control block after an error."""
    return int(lib().moe_check_noalloc(layer, stream))


def moe_set_profile_events(layer: int, events) -> None:
    """events: four cudaEvent_t handles (ints) or None to switch the hook off."""
    arr = None if events is None else (_vp * 4)(*events)
    check(lib().moe_set_profile_events(layer, arr), "moe_set_profile_events")


MOE_RESIDENCY_FAULT_NONE, MOE_RESIDENCY_FAULT_TAG, MOE_RESIDENCY_FAULT_COPY = 0, 1, 2


def moe_residency_pool_bytes(layer: int, n_slots: int) -> int:
    return int(lib().moe_residency_pool_bytes(layer, n_slots))


def moe_residency_open(layer: int, host_records: int, n_slots: int, pool: int, pool_bytes: int) -> int:
    h = _vp()
    check(lib().moe_residency_open(layer, host_records, n_slots, pool, pool_bytes, ctypes.byref(h)),
          "moe_residency_open")
    return h.value


def moe_residency_decode(res, x, B, out_bf16, out_f32, ids, weights, ws, ws_bytes, main_stream=0,
                         copy_stream=0) -> None:
    check(lib().moe_residency_decode(res, x, B, out_bf16, out_f32, ids, weights, ws, ws_bytes,
                                     main_stream, copy_stream), "moe_residency_decode")


def moe_residency_lookahead(res, x, B, n_ahead, ids, weights, ws, ws_bytes, stream=0,
                            copy_stream=0) -> None:
    check(lib().moe_residency_lookahead(res, x, B, n_ahead, ids, weights, ws, ws_bytes, stream,
                                        copy_stream), "moe_residency_lookahead")


def moe_residency_stats(res: int) -> dict:
    out = moe_residency_stats_t()
    check(lib().moe_residency_stats(res, ctypes.byref(out)), "moe_residency_stats")
    return {n: int(getattr(out, n)) for n, _ in moe_residency_stats_t._fields_}


def moe_residency_slots(res: int, n_slots: int):
    arr = (ctypes.c_int32 * n_slots)()
    check(lib().moe_residency_slots(res, arr, n_slots), "moe_residency_slots")
    return list(arr)


def moe_residency_set_fault(res: int, mode: int) -> None:
    check(lib().moe_residency_set_fault(res, mode), "moe_residency_set_fault")


def moe_residency_close(res: int) -> None:
    lib().moe_residency_close(res)


def moe_check(layer: int, ws: int, stream: int = 0) -> int:
    """Returns the device-latched status code (MOE_OK, MOE_ERR_TIMEOUT, ...)."""
    return int(lib().moe_check(layer, ws, stream))
