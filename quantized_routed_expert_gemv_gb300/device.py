"""Device-resident synthetic layers: torch owns the memory, libmoe does the work.

``DeviceLayer`` draws a layer with ``synth`` (in pinned host chunks, copied
to HBM), opens it through the C ABI and owns a zero-initialised workspace.
Its ``decode`` / ``prefill`` methods only allocate outputs and marshal
pointers to ``moe_decode`` / ``moe_prefill_chunk``.
"""
from __future__ import annotations

import numpy as np
import torch

from . import moe, synth


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """bf16 bit patterns (uint16) -> torch.bfloat16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class DeviceLayer:
    def __init__(self, shape: synth.Shape, weight_seed: int, layer: int = 0, beta=None,
                 max_tokens: int = 16, device="cuda:0", chunk_records: int = 32,
                 host_records: np.ndarray | None = None, host_shared: np.ndarray | None = None,
                 router=None, resident: bool = True, rvq: bool = False, codebooks=None):
        """rvq: the experts are 3-bit residual-VQ records (wbits = 3) with the
        layer's codebooks (synth.rvq_codebooks unless given)."""
        self.shape = s = shape
        self.device = torch.device(device)
        self.max_tokens = max_tokens
        self.rvq = rvq
        stride_of = synth.rvq_record_stride if rvq else synth.record_stride
        fill = synth.fill_rvq_records if rvq else synth.fill_records
        one = synth.rvq_expert_record if rvq else synth.expert_record
        self.stride = stride_of(s.H, s.F)
        if resident:
            self.records = torch.empty(s.E * self.stride, dtype=torch.uint8, device=self.device)
            if host_records is not None:
                self.records.copy_(torch.from_numpy(np.ascontiguousarray(host_records).reshape(-1)))
            else:
                n = min(chunk_records, s.E)
                pinned = torch.empty(n * self.stride, dtype=torch.uint8, pin_memory=True)
                view = pinned.numpy()
                for e0 in range(0, s.E, n):
                    cnt = min(n, s.E - e0)
                    fill(weight_seed, layer, range(e0, e0 + cnt), s.H, s.F, view)
                    self.records[e0 * self.stride:(e0 + cnt) * self.stride].copy_(
                        pinned[:cnt * self.stride])
        else:
            self.records = None
        if s.Fs:
            sh = host_shared if host_shared is not None else one(weight_seed, layer, s.E, s.H, s.Fs)
            self.shared = torch.from_numpy(np.ascontiguousarray(sh)).to(self.device)
        else:
            self.shared = None
        rc, rsb = router if router is not None else synth.router(weight_seed, layer, s.E, s.H)
        self.router_codes = torch.from_numpy(np.ascontiguousarray(rc)).to(self.device)
        self.router_sb = torch.from_numpy(np.ascontiguousarray(rsb).view(np.int32)).to(self.device)
        self.beta = None if beta is None else torch.from_numpy(
            np.ascontiguousarray(beta, np.float32)).to(self.device)
        self.codebooks = None
        if rvq:
            cb = codebooks if codebooks is not None else synth.rvq_codebooks(weight_seed, layer)
            self.codebooks = torch.from_numpy(np.ascontiguousarray(cb, np.uint16).view(np.int16)).to(self.device)
        self.desc = moe.desc(s.H, s.E, s.k, s.F, s.Fs, max_tokens=max_tokens, wbits=3 if rvq else 4)
        self.weights = moe.moe_layer_weights(
            self.records.data_ptr() if self.records is not None else None,
            self.shared.data_ptr() if self.shared is not None else None,
            self.router_codes.data_ptr(), self.router_sb.data_ptr(),
            self.beta.data_ptr() if self.beta is not None else None,
            self.codebooks.data_ptr() if self.codebooks is not None else None)
        self.handle = moe.moe_open(self.desc, self.weights)
        self.ws_bytes = moe.moe_workspace_bytes(self.handle, max_tokens)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        moe.moe_workspace_init(self.handle, self.ws.data_ptr(), self.ws_bytes,
                               torch.cuda.current_stream(self.device).cuda_stream)

    def outputs(self, T: int):
        s, dev = self.shape, self.device
        return (torch.empty(T, s.H, dtype=torch.bfloat16, device=dev),
                torch.empty(T, s.H, dtype=torch.float32, device=dev),
                torch.empty(T, s.k, dtype=torch.int32, device=dev),
                torch.empty(T, s.k, dtype=torch.float32, device=dev))

    def _call(self, fn, x: torch.Tensor, outs, stream):
        ob, of, ids, w = outs
        T = x.shape[0]
        st = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        fn(self.handle, x.data_ptr(), T, ob.data_ptr(), of.data_ptr() if of is not None else None,
           ids.data_ptr(), w.data_ptr(), self.ws.data_ptr(), self.ws_bytes, st)
        return ob, of, ids, w

    def decode(self, x: torch.Tensor, outs=None, stream=None):
        return self._call(moe.moe_decode, x, outs or self.outputs(x.shape[0]), stream)

    def prefill(self, x: torch.Tensor, outs=None, stream=None):
        return self._call(moe.moe_prefill_chunk, x, outs or self.outputs(x.shape[0]), stream)

    def check(self, stream=None) -> int:
        st = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        return moe.moe_check(self.handle, self.ws.data_ptr(), st)

    def close(self):
        if self.handle:
            moe.moe_close(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pinned_records(shape: synth.Shape, weight_seed: int, layer: int = 0,
                   host_records: np.ndarray | None = None, rvq: bool = False) -> torch.Tensor:
    """All E expert records of a layer in page-locked host memory (3-bit
    residual-VQ records when rvq)."""
    stride = (synth.rvq_record_stride if rvq else synth.record_stride)(shape.H, shape.F)
    t = torch.empty(shape.E * stride, dtype=torch.uint8, pin_memory=True)
    if host_records is not None:
        t.copy_(torch.from_numpy(np.ascontiguousarray(host_records).reshape(-1)))
    else:
        fill = synth.fill_rvq_records if rvq else synth.fill_records
        fill(weight_seed, layer, range(shape.E), shape.H, shape.F, t.numpy())
    return t


class CachedLayer:
    """A layer whose routed experts are read through the HBM expert cache
    (moe_residency_*): host records pinned, n_slots record slots on the GPU."""

    def __init__(self, dl: DeviceLayer, host_records: torch.Tensor, n_slots: int):
        self.dl = dl
        self.host = host_records
        self.n_slots = n_slots
        self.pool_bytes = moe.moe_residency_pool_bytes(dl.handle, n_slots)
        self.pool = torch.empty(self.pool_bytes, dtype=torch.uint8, device=dl.device)
        self.handle = moe.moe_residency_open(dl.handle, host_records.data_ptr(), n_slots,
                                             self.pool.data_ptr(), self.pool_bytes)
        self.copy_stream = torch.cuda.Stream(dl.device)
        self.ahead_ws = None

    def decode(self, x: torch.Tensor, outs=None, stream=None):
        ob, of, ids, w = outs or self.dl.outputs(x.shape[0])
        st = stream if stream is not None else torch.cuda.current_stream(self.dl.device).cuda_stream
        moe.moe_residency_decode(self.handle, x.data_ptr(), x.shape[0], ob.data_ptr(),
                                 of.data_ptr() if of is not None else None, ids.data_ptr(),
                                 w.data_ptr(), self.dl.ws.data_ptr(), self.dl.ws_bytes, st,
                                 self.copy_stream.cuda_stream)
        return ob, of, ids, w

    def lookahead(self, x: torch.Tensor, n_ahead: int, stream=None, copy_stream=None):
        """Runs this layer's router on an earlier hidden state x and reads the
        first n_ahead experts of each token's predicted ranking into the
        cache (moe_residency_lookahead).  Uses a workspace of its own, so it
        may run on another stream than the layer's steps.  Returns the
        predicted (ids, weights) [B][k] on the device."""
        dl = self.dl
        st = stream if stream is not None else torch.cuda.current_stream(dl.device).cuda_stream
        self.prepare_lookahead(st)
        B = x.shape[0]
        moe.moe_residency_lookahead(self.handle, x.data_ptr(), B, n_ahead, self.ahead_ids.data_ptr(),
                                    self.ahead_w.data_ptr(), self.ahead_ws.data_ptr(), dl.ws_bytes,
                                    st, (copy_stream or self.copy_stream).cuda_stream)
        return self.ahead_ids[:B], self.ahead_w[:B]

    def prepare_lookahead(self, stream) -> None:
        """Allocates the lookahead's workspace and predicted-routing buffers
        (once); stream orders the workspace initialisation."""
        if self.ahead_ws is None:
            dl = self.dl
            self.ahead_ws = torch.empty(dl.ws_bytes, dtype=torch.uint8, device=dl.device)
            moe.moe_workspace_init(dl.handle, self.ahead_ws.data_ptr(), dl.ws_bytes, stream)
            _, _, self.ahead_ids, self.ahead_w = dl.outputs(dl.desc.max_tokens)

    def check_lookahead(self, stream=None) -> int:
        """moe_check of the lookahead workspace (0 if none was made)."""
        if self.ahead_ws is None:
            return moe.MOE_OK
        st = stream if stream is not None else torch.cuda.current_stream(self.dl.device).cuda_stream
        return moe.moe_check(self.dl.handle, self.ahead_ws.data_ptr(), st)

    def stats(self) -> dict:
        return moe.moe_residency_stats(self.handle)

    def slots(self):
        return moe.moe_residency_slots(self.handle, self.n_slots)

    def set_fault(self, mode: int) -> None:
        moe.moe_residency_set_fault(self.handle, mode)

    def close(self):
        if self.handle:
            moe.moe_residency_close(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
