"""C-ABI checks that need no GPU: the library loads, exports every function
include/*.h declares, computes the record layout the oracle derives on its
own, and rejects bad arguments on the host before any device work."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest
import torch

import oracle
from quantized_routed_expert_gemv_gb300 import build, moe, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(moe_\w+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def L():
    build.build()
    return moe.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert "moe_decode" in names and "moe_open" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported by libmoe.so"
        assert n in moe.SIGNATURES, f"{n} has no binding"


@pytest.mark.parametrize("H,F", [(256, 128), (2048, 768), (2048, 2048), (7168, 2048), (64, 64),
                                 (8192, 8192)])
def test_record_layout_matches_oracle(L, H, F):
    got = moe.moe_record_layout_of(H, F)
    assert got == oracle.record_layout(H, F)
    d = moe.desc(H, 8, 2, F, 0)
    assert moe.moe_expert_bytes(d, F) == synth.record_stride(H, F)


@pytest.mark.parametrize("H,F", [(256, 128), (2048, 768), (7168, 2048), (64, 64)])
def test_rvq_record_layout_matches_oracle(L, H, F):
    out = moe.moe_record_layout()
    assert L.moe_rvq_record_layout_of(H, F, ctypes.byref(out)) == moe.MOE_OK
    assert {n: int(getattr(out, n)) for n, _ in moe.moe_record_layout._fields_} == oracle.rvq_layout(H, F)
    d = moe.desc(H, 8, 2, F, 0, wbits=3)
    assert moe.moe_expert_bytes(d, F) == synth.rvq_record_stride(H, F)
    assert L.moe_rvq_record_layout_of(H + 32, F, ctypes.byref(out)) == moe.MOE_ERR_ARG


@pytest.mark.parametrize("H,F", [(0, 64), (96, 64), (64, 100), (8256, 64), (64, -64)])
def test_record_layout_rejects_bad_shapes(L, H, F):
    out = moe.moe_record_layout()
    assert L.moe_record_layout_of(H, F, ctypes.byref(out)) == moe.MOE_ERR_ARG
    assert "64" in moe.last_error()


def _weights(aligned=True):
    # Host addresses stand in for device pointers: validation never dereferences them.
    base = 1 << 20
    off = 0 if aligned else 8
    return moe.moe_layer_weights(base * 16 + off, None, base * 32 + off, base * 48, None)


BAD_DESCS = [
    dict(hidden=100), dict(hidden=0), dict(n_experts=0), dict(n_experts=2000), dict(top_k=0),
    dict(top_k=9), dict(ffn=65), dict(shared_ffn=10), dict(group=32), dict(wbits=5),
    dict(wbits=3),  # residual-VQ experts without codebooks
    dict(rbits=4),
    dict(max_tokens=0), dict(max_tokens=129),
]


@pytest.mark.parametrize("bad", BAD_DESCS, ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_open_rejects_bad_desc(L, bad):
    d = moe.desc(256, 8, 2, 128, 0)
    for k, v in bad.items():
        setattr(d, k, v)
    h = ctypes.c_void_p()
    rc = L.moe_open(ctypes.byref(d), ctypes.byref(_weights()), ctypes.byref(h))
    assert rc == moe.MOE_ERR_ARG, moe.last_error()
    assert h.value is None


def test_open_rejects_misaligned_and_missing(L):
    d = moe.desc(256, 8, 2, 128, 0)
    h = ctypes.c_void_p()
    assert L.moe_open(ctypes.byref(d), ctypes.byref(_weights(False)), ctypes.byref(h)) == \
        moe.MOE_ERR_ALIGN
    w = _weights()
    w.router_codes = None
    assert L.moe_open(ctypes.byref(d), ctypes.byref(w), ctypes.byref(h)) == moe.MOE_ERR_ARG
    d.shared_ffn = 256  # shared width without a shared record
    assert L.moe_open(ctypes.byref(d), ctypes.byref(_weights()), ctypes.byref(h)) == moe.MOE_ERR_ARG
    assert L.moe_open(None, ctypes.byref(_weights()), ctypes.byref(h)) == moe.MOE_ERR_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_open_without_gpu_fails_cleanly(L):
    d = moe.desc(256, 8, 2, 128, 0)
    h = ctypes.c_void_p()
    rc = L.moe_open(ctypes.byref(d), ctypes.byref(_weights()), ctypes.byref(h))
    assert rc in (moe.MOE_ERR_CUDA, moe.MOE_ERR_UNSUPPORTED)
    assert h.value is None and moe.last_error()


def test_calls_reject_invalid_handles(L):
    fake = (ctypes.c_uint8 * 4096)()   # zeroed host memory: wrong magic
    p = ctypes.addressof(fake)
    assert L.moe_workspace_bytes(None, 1) == 0
    assert L.moe_workspace_bytes(p, 1) == 0
    for fn in ("moe_decode", "moe_prefill_chunk", "moe_decode_host"):
        assert getattr(L, fn)(None, 0, 1, 0, 0, 0, 0, 0, 0, None) == moe.MOE_ERR_ARG
        assert getattr(L, fn)(p, 0, 1, 0, 0, 0, 0, 0, 0, None) == moe.MOE_ERR_ARG
    assert L.moe_check(None, p, None) == moe.MOE_ERR_ARG
    assert L.moe_workspace_init(None, p, 16, None) == moe.MOE_ERR_ARG
    L.moe_close(None)
    L.moe_close(p)          # wrong magic: ignored, not freed
    assert isinstance(moe.last_error(), str)


def test_residency_and_noalloc_calls_reject_invalid_handles(L):
    fake = (ctypes.c_uint8 * 4096)()
    p = ctypes.addressof(fake)
    assert L.moe_residency_pool_bytes(None, 4) == 0
    assert L.moe_residency_pool_bytes(p, 4) == 0
    h = ctypes.c_void_p()
    assert L.moe_residency_open(None, p, 4, p, 1 << 20, ctypes.byref(h)) == moe.MOE_ERR_ARG
    assert L.moe_residency_open(p, p, 4, p, 1 << 20, ctypes.byref(h)) == moe.MOE_ERR_ARG
    assert h.value is None
    for r in (None, p):
        assert L.moe_residency_decode(r, 0, 1, 0, 0, 0, 0, 0, 0, None, None) == moe.MOE_ERR_ARG
        st = moe.moe_residency_stats_t()
        assert L.moe_residency_stats(r, ctypes.byref(st)) == moe.MOE_ERR_ARG
        assert L.moe_residency_slots(r, (ctypes.c_int32 * 4)(), 4) == moe.MOE_ERR_ARG
        assert L.moe_residency_set_fault(r, 1) == moe.MOE_ERR_ARG
        assert L.moe_residency_verify(r, None) == moe.MOE_ERR_ARG
        assert L.moe_residency_lookahead(r, 0, 1, 6, 0, 0, 0, 0, None, None) == moe.MOE_ERR_ARG
        assert L.moe_decode_kernels(r, 1) == -1
        L.moe_residency_close(r)  # ignored
        assert L.moe_decode_noalloc(r, 0, 1, 0, 0, 0, 0, None) == moe.MOE_ERR_ARG
        assert L.moe_check_noalloc(r, None) == moe.MOE_ERR_ARG
    assert "invalid" in moe.last_error()


def test_crc32_check_value_and_zlib(L):
    """moe_crc32 is the IEEE 802.3 / zlib CRC-32: the published check value of
    "123456789" and zlib's own routine on random data of many lengths and
    start alignments (the eight-byte steps and the byte tail)."""
    import zlib
    msg = b"123456789"
    assert L.moe_crc32(msg, len(msg)) == 0xCBF43926
    assert L.moe_crc32(None, 0) == 0
    rng = np.random.default_rng(5)
    data = rng.integers(0, 256, 1 << 20, dtype=np.uint8)
    base = data.ctypes.data
    for off, n in [(0, 1), (1, 7), (3, 8), (5, 9), (0, 63), (7, 1000), (0, 1 << 20)]:
        n = min(n, data.size - off)
        assert L.moe_crc32(base + off, n) == zlib.crc32(data[off:off + n].tobytes()), (off, n)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(moe, "_lib", None)
    monkeypatch.setattr(moe, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        moe.lib()
