"""Layers of 3-bit residual-VQ experts (wbits = 3) through the C ABI.

WASTE page, section "Quantization ve doğruluk": each run of 8 weights along
a row is the sum of one codeword from each of 3 stages of 256-entry
codebooks.  moe_decode on such a layer is compared element by element with
the fp64 oracle (oracle.c, orc_expert_rvq) on seeded layers from tiny to the
mid shape, with ragged tile counts, no shared expert, k = E and k = 1; the
identity-expert layer in this format must give its closed form; prefill
chunks refuse the format.  Through the HBM expert cache (WASTE page, section
"Disk streaming mimarisi": the 3-bit records are what is streamed), Zipf
streams at B = 1 and 4 keep counters and slots equal to the oracle's LFU
replay, copy 3 bits per weight per miss, and give the oracle's outputs.
"""
import numpy as np
import pytest
import torch

import oracle
from layers import HostLayerRVQ, hidden_with_margin, identity_layer_rvq
from quantized_routed_expert_gemv_gb300 import moe, synth
from quantized_routed_expert_gemv_gb300.device import CachedLayer, DeviceLayer, bf16_bits, bf16_tensor

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS, P_TOL = 2e-3, 1e-4, 1e-5
DEV = "cuda:0"


def assert_token(t, out_f32, out_bf16, ids, w, ref_out, ref_ids, ref_p):
    assert np.array_equal(ids[t], ref_ids), (t, ids[t], ref_ids)
    assert np.abs(w[t].astype(np.float64) - ref_p).max() <= P_TOL, (t, w[t], ref_p)
    err = np.abs(out_f32[t].astype(np.float64) - ref_out).max()
    bound = TOL_REL * np.abs(ref_out).max() + TOL_ABS
    assert err <= bound, (t, err, bound)
    assert np.array_equal(out_bf16[t], synth.float_to_bf16_bits(out_f32[t]))


def run(dl: DeviceLayer, xs: np.ndarray):
    ob, of, ids, w = dl.decode(bf16_tensor(xs, DEV))
    torch.cuda.synchronize()
    assert dl.check() == moe.MOE_OK, moe.last_error()
    return of.cpu().numpy(), bf16_bits(ob), ids.cpu().numpy(), w.cpu().numpy()


def device_rvq(hl: HostLayerRVQ, max_tokens: int) -> DeviceLayer:
    return DeviceLayer(hl.shape, 0, beta=hl.beta, max_tokens=max_tokens, device=DEV,
                       host_records=hl.records, host_shared=hl.shared,
                       router=(hl.router_codes, hl.router_sb), rvq=True, codebooks=hl.codebooks)


SHAPES = [
    (synth.TINY, 1), (synth.TINY, 3),
    (synth.Shape(64, 4, 4, 64, 64), 2),        # E == k: every expert chosen
    (synth.Shape(128, 6, 3, 64, 0), 4),        # no shared expert
    (synth.Shape(192, 5, 1, 128, 64), 3),      # k = 1: weight exactly 1
    (synth.Shape(320, 16, 4, 192, 128), 5),    # ragged row tiles, F != Fs
    (synth.MID, 1), (synth.MID, 4),            # 2048 hidden, 128 experts, top-8
]


@pytest.mark.parametrize("shape,T", SHAPES, ids=lambda v: str(v))
def test_rvq_layer_matches_oracle(shape, T):
    hl = HostLayerRVQ(shape, seed=6, beta=synth.beta_normal(6, 0, shape.E))
    orc = hl.oracle()
    dl = device_rvq(hl, max(T, 1))
    xs = np.stack([hidden_with_margin(orc, 6, 0, t) for t in range(T)])
    of, ob, ids, w = run(dl, xs)
    for t in range(T):
        assert_token(t, of, ob, ids, w, *orc.token(xs[t]))
    assert moe.lib().moe_decode_kernels(dl.handle, T) == 4  # router, gate|up, down, combine
    dl.close()


@pytest.mark.parametrize("T", [1, 3])
def test_rvq_identity_expert_layer(T):
    records, shared, rc, rsb, cbs = identity_layer_rvq()
    E, k, H = 8, 2, 64
    shape = synth.Shape(H, E, k, H, H)
    dl = DeviceLayer(shape, 0, max_tokens=4, device=DEV, host_records=records, host_shared=shared,
                     router=(rc, rsb), rvq=True, codebooks=cbs)
    lay = oracle.Layer(H, E, k, H, H, {e: records[e] for e in range(E)}, shared, rc, rsb, codebooks=cbs)
    xs = np.stack([synth.hidden(3, 0, t, H) for t in range(T)])
    xs[:, 0] = synth.bf16_from_double(8.0)
    of, ob, ids, w = run(dl, xs)
    for t in range(T):
        ref, rids, rp = lay.token(xs[t])
        assert_token(t, of, ob, ids, w, ref, rids, rp)
        x = synth.bf16_bits_to_float(xs[t]).astype(np.float64)
        scale = 1.0 + sum(float(w[t, i]) * 2.0 ** -(int(ids[t, i]) % 3) for i in range(k))
        np.testing.assert_allclose(of[t], scale * x, rtol=2e-6, atol=1e-30)
    dl.close()


def test_rvq_refuses_prefill():
    hl = HostLayerRVQ(synth.TINY, seed=1)
    dl = device_rvq(hl, 4)
    x = bf16_tensor(np.stack([synth.hidden(1, 0, t, synth.TINY.H) for t in range(2)]), DEV)
    with pytest.raises(moe.MoEError) as ei:
        dl.prefill(x)
    assert ei.value.code == moe.MOE_ERR_ARG and "wbits=4" in str(ei.value)
    dl.close()


def first_appearance(ids):
    seen, order = set(), []
    for e in np.asarray(ids).reshape(-1):
        if int(e) not in seen:
            seen.add(int(e))
            order.append(int(e))
    return np.array(order, np.int32)


@pytest.mark.parametrize("B,steps,n_slots", [(1, 24, 8), (4, 10, 16)])
def test_rvq_records_through_the_cache(B, steps, n_slots):
    shape = synth.Shape(256, 64, 4, 128, 256)
    beta = synth.beta_zipf(4, 0, 64)
    hl = HostLayerRVQ(shape, seed=8, beta=beta)
    orc = hl.oracle()
    dl = DeviceLayer(shape, 0, beta=beta, max_tokens=B, device=DEV, host_records=hl.records,
                     host_shared=hl.shared, router=(hl.router_codes, hl.router_sb), rvq=True,
                     codebooks=hl.codebooks)
    host = torch.empty(hl.records.nbytes, dtype=torch.uint8, pin_memory=True)
    host.copy_(torch.from_numpy(hl.records.reshape(-1)))
    cl = CachedLayer(dl, host, n_slots)
    lfu = oracle.LFU(n_slots, shape.E)
    rec_bytes = oracle.rvq_layout(shape.H, shape.F)["bytes"]
    for s in range(steps):
        xs = np.stack([hidden_with_margin(orc, 19, s, t) for t in range(B)])
        ob, of, ids, w = cl.decode(bf16_tensor(xs, DEV))
        torch.cuda.synchronize()
        assert dl.check() == moe.MOE_OK, moe.last_error()
        ids = ids.cpu().numpy()
        for t0, t1 in oracle.waves(ids, n_slots):
            lfu.step(first_appearance(ids[t0:t1]))
        st = cl.stats()
        assert (st["hits"], st["misses"], st["evictions"]) == (lfu.hits, lfu.misses, lfu.evictions)
        assert st["bytes_h2d"] == st["misses"] * rec_bytes
        assert cl.slots() == list(lfu.slot_expert)
        got = (of.cpu().numpy(), bf16_bits(ob), ids, w.cpu().numpy())
        for t in range(B):
            assert_token(t, *got, *orc.token(xs[t]))
    st = cl.stats()
    assert st["evictions"] > 0 and st["hits"] > 0
    cl.close()
    dl.close()


@pytest.mark.parametrize("B", [1, 3])
def test_rvq_host_entry_matches_device_entry(B):
    """moe_decode_host on a 3-bit layer over several calls with changing
    inputs (the first call plain, later ones replaying the captured step:
    x staged by a kernel that the single-token router overlaps, outputs
    written into mapped host memory) equals moe_decode on the same inputs,
    and the oracle."""
    shape = synth.Shape(320, 16, 4, 192, 128)
    hl = HostLayerRVQ(shape, seed=12, beta=synth.beta_normal(12, 0, shape.E))
    orc = hl.oracle()
    dl = device_rvq(hl, 4)
    for rep in range(4):
        xs = np.stack([hidden_with_margin(orc, 12, rep, t) for t in range(B)])
        of, ob, ids, w = run(dl, xs)
        hob = np.zeros((B, shape.H), np.uint16)
        hof = np.zeros((B, shape.H), np.float32)
        hids = np.zeros((B, shape.k), np.int32)
        hw = np.zeros((B, shape.k), np.float32)
        moe.moe_decode_host(dl.handle, xs.ctypes.data, B, hob.ctypes.data, hof.ctypes.data, hids.ctypes.data,
                            hw.ctypes.data, dl.ws.data_ptr(), dl.ws_bytes, None)
        assert np.array_equal(hob, ob) and np.array_equal(hof, of)
        assert np.array_equal(hids, ids) and np.array_equal(hw, w)
        for t in range(B):
            assert_token(t, hof, hob, hids, hw, *orc.token(xs[t]))
    assert dl.check() == moe.MOE_OK, moe.last_error()
    dl.close()
