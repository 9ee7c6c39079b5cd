"""Parity of the CUDA decode / prefill path (through the C ABI) with the fp64
oracle, element by element, on seeded synthetic layers.

Bar (per token): expert ids bit-exact; routing weights within 1e-5;
max |out_f32 - ref| <= 2e-3 * max |ref| + 1e-4; out_bf16 bit-exact equal to
round-to-nearest-even(out_f32)."""
import numpy as np
import pytest
import torch

import oracle
from layers import HostLayer, hidden_with_margin, identity_layer
from quantized_routed_expert_gemv_gb300 import moe, synth
from quantized_routed_expert_gemv_gb300.device import DeviceLayer, bf16_bits, bf16_tensor

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


def run(dl: DeviceLayer, xs: np.ndarray, prefill=False):
    x = bf16_tensor(xs, DEV)
    ob, of, ids, w = (dl.prefill if prefill else dl.decode)(x)
    torch.cuda.synchronize()
    assert dl.check() == moe.MOE_OK, moe.last_error()
    return of.cpu().numpy(), bf16_bits(ob), ids.cpu().numpy(), w.cpu().numpy()


def device_from_host(hl: HostLayer, max_tokens=16):
    return DeviceLayer(hl.shape, 0, beta=hl.beta, max_tokens=max_tokens, device=DEV,
                       host_records=hl.records, host_shared=hl.shared,
                       router=(hl.router_codes, hl.router_sb))


def draw_tokens(orc, seed, stream, T):
    return np.stack([hidden_with_margin(orc, seed, stream, t) for t in range(T)])


# ---------------------------------------------------------------- closed form

@pytest.mark.parametrize("T", [1, 3])
def test_identity_expert_layer(T):
    records, shared, rc, rsb = identity_layer()
    E, k, H = 8, 2, 64
    shape = synth.Shape(H, E, k, H, H)
    dl = DeviceLayer(shape, 0, max_tokens=4, device=DEV, host_records=records, host_shared=shared,
                     router=(rc, rsb))
    lay = oracle.Layer(H, E, k, H, H, {e: records[e] for e in range(E)}, shared, rc, rsb)
    xs = np.stack([synth.hidden(3, 0, t, H) for t in range(T)])
    # Every |x| >= 1/16 keeps each 32-value chunk within 2^7 of its largest
    # magnitude (8), where the single-token kernels' 16-bit fixed-point
    # activations are exact, so the closed form holds to fp32 rounding.
    xf = synth.bf16_bits_to_float(xs)
    small = np.abs(xf) < 0.0625
    xs[small] = np.where(xf[small] < 0, synth.bf16_from_double(-0.0625),
                         synth.bf16_from_double(0.0625)).astype(np.uint16)
    xs[:, 0] = synth.bf16_from_double(8.0)
    of, ob, ids, w = run(dl, xs)
    for t in range(T):
        ref, rids, rp = lay.token(xs[t])
        assert_token(t, of, ob, ids, w, ref, rids, rp)
        x = synth.bf16_bits_to_float(xs[t]).astype(np.float64)
        scale = 1.0 + sum(float(w[t, i]) * 2.0 ** -(int(ids[t, i]) % 3) for i in range(k))
        np.testing.assert_allclose(of[t], scale * x, rtol=2e-6, atol=1e-30)


@pytest.mark.parametrize("T", [1, 3])
def test_identity_expert_layer_unclamped(T):
    """The identity-expert layer on hidden states as drawn (no clamp): small
    activations in a chunk with a large one are rounded by the fixed-point
    path, so the closed form holds within the parity bar, not exactly."""
    records, shared, rc, rsb = identity_layer()
    E, k, H = 8, 2, 64
    shape = synth.Shape(H, E, k, H, H)
    dl = DeviceLayer(shape, 0, max_tokens=4, device=DEV, host_records=records, host_shared=shared,
                     router=(rc, rsb))
    lay = oracle.Layer(H, E, k, H, H, {e: records[e] for e in range(E)}, shared, rc, rsb)
    xs = np.stack([synth.hidden(5, 0, t, H) for t in range(T)])
    xs[:, 0] = synth.bf16_from_double(8.0)
    of, ob, ids, w = run(dl, xs)
    for t in range(T):
        ref, rids, rp = lay.token(xs[t])
        assert_token(t, of, ob, ids, w, ref, rids, rp)
        x = synth.bf16_bits_to_float(xs[t]).astype(np.float64)
        scale = 1.0 + sum(float(w[t, i]) * 2.0 ** -(int(ids[t, i]) % 3) for i in range(k))
        closed = scale * x
        assert np.abs(of[t] - closed).max() <= TOL_REL * np.abs(closed).max() + TOL_ABS


# ---------------------------------------------------------------- small layers

SMALL = [
    (synth.TINY, 1), (synth.TINY, 2), (synth.TINY, 5), (synth.TINY, 16),
    (synth.Shape(64, 4, 4, 64, 64), 3),        # E == k: every expert chosen
    (synth.Shape(128, 6, 3, 64, 0), 4),        # no shared expert
    (synth.Shape(192, 5, 1, 128, 64), 7),      # k = 1: weight exactly 1
    (synth.Shape(320, 16, 4, 192, 128), 9),    # two gate|up tiles, ragged sizes
    (synth.Shape(1024, 40, 6, 448, 320), 11),  # several tiles, F != Fs
]


@pytest.mark.parametrize("shape,T", SMALL, ids=lambda v: str(v))
def test_small_layers(shape, T):
    hl = HostLayer(shape, seed=17, beta=synth.beta_normal(17, 0, shape.E))
    orc = hl.oracle()
    dl = device_from_host(hl)
    xs = draw_tokens(orc, 17, 1, T)
    of, ob, ids, w = run(dl, xs)
    for t in range(T):
        ref, rids, rp = orc.token(xs[t])
        assert_token(t, of, ob, ids, w, ref, rids, rp)
    if shape.k == 1:
        assert np.all(w == 1.0)


# Single-token geometries: 2, 3 (with idle warps) and 4 warps per row, no
# shared expert, and enough items per CTA to wrap the pipeline ring.
B1_SHAPES = [synth.Shape(2048, 64, 8, 2048, 2048), synth.Shape(3072, 24, 4, 1536, 512),
             synth.Shape(4096, 32, 4, 1024, 0)]


@pytest.mark.parametrize("shape", B1_SHAPES, ids=lambda s: f"H{s.H}F{s.F}Fs{s.Fs}")
def test_single_token_geometries(shape):
    hl = HostLayer(shape, seed=41, beta=synth.beta_normal(41, 0, shape.E))
    orc = hl.oracle()
    dl = device_from_host(hl)
    for t in range(2):
        xs = draw_tokens(orc, 41, 10 + t, 1)
        of, ob, ids, w = run(dl, xs)
        ref, rids, rp = orc.token(xs[0])
        assert_token(0, of, ob, ids, w, ref, rids, rp)


@pytest.mark.parametrize("T", [2, 4, 5, 16])
def test_few_tokens_sharing_every_expert(T):
    """Logit offsets steer every token to the same k experts, so each routed
    expert of the few-token kernel serves all T tokens (the most tokens an
    item holds, up to 16) and the shared expert too; a second call on the
    same workspace checks that the kernels left their counters at zero."""
    shape = synth.Shape(1024, 40, 6, 448, 320)
    beta = np.zeros(shape.E, np.float32)
    beta[[3, 7, 11, 19, 23, 31]] = 50.0
    hl = HostLayer(shape, seed=37, beta=beta)
    orc = hl.oracle()
    dl = device_from_host(hl)
    for rep in range(2):
        xs = draw_tokens(orc, 37, 5 + rep, T)
        of, ob, ids, w = run(dl, xs)
        assert set(np.unique(ids)) == {3, 7, 11, 19, 23, 31}
        for t in range(T):
            ref, rids, rp = orc.token(xs[t])
            assert_token(t, of, ob, ids, w, ref, rids, rp)


@pytest.mark.parametrize("outlier", [64.0, 4096.0])
def test_activation_outliers(outlier):
    # One huge activation per token (as real hidden states have): the single-
    # token path rounds the other activations of that 32-value chunk to
    # 2^-15 of the outlier; the result must still meet the parity bar.
    shape = synth.Shape(1024, 40, 6, 448, 320)
    hl = HostLayer(shape, seed=31)
    orc = hl.oracle()
    dl = device_from_host(hl)
    for t in range(3):
        x = synth.hidden(31, 7, t, shape.H)
        x[37 * (t + 1)] = synth.bf16_from_double(outlier * (-1) ** t)
        xs = x[None]
        of, ob, ids, w = run(dl, xs)
        ref, rids, rp = orc.token(xs[0])
        assert_token(0, of, ob, ids, w, ref, rids, rp)


def test_tiny_workload_config0():
    wl = synth.WORKLOADS["tiny"]
    hl = HostLayer(wl.shape, seed=wl.weight_seed)
    orc = hl.oracle()
    dl = device_from_host(hl)
    xs = draw_tokens(orc, wl.input_seed, 0, 1)
    of, ob, ids, w = run(dl, xs)
    ref, rids, rp = orc.token(xs[0])
    assert_token(0, of, ob, ids, w, ref, rids, rp)


def test_zero_tokens_is_a_no_op():
    hl = HostLayer(synth.TINY, seed=1)
    dl = device_from_host(hl)
    ob, of, ids, w = dl.outputs(1)
    rc = moe.lib().moe_decode(dl.handle, ob.data_ptr(), 0, ob.data_ptr(), of.data_ptr(),
                              ids.data_ptr(), w.data_ptr(), dl.ws.data_ptr(), dl.ws_bytes, None)
    assert rc == moe.MOE_OK


def test_too_many_tokens_and_small_workspace_rejected():
    hl = HostLayer(synth.TINY, seed=1)
    dl = device_from_host(hl, max_tokens=4)
    x = bf16_tensor(np.zeros((5, 256), np.uint16), DEV)
    ob, of, ids, w = dl.outputs(5)
    L = moe.lib()
    assert L.moe_decode(dl.handle, x.data_ptr(), 5, ob.data_ptr(), of.data_ptr(), ids.data_ptr(),
                        w.data_ptr(), dl.ws.data_ptr(), dl.ws_bytes, None) == moe.MOE_ERR_ARG
    assert L.moe_decode(dl.handle, x.data_ptr(), 2, ob.data_ptr(), of.data_ptr(), ids.data_ptr(),
                        w.data_ptr(), dl.ws.data_ptr(), 1024, None) == moe.MOE_ERR_ARG
    assert L.moe_decode(dl.handle, x.data_ptr() + 2, 2, ob.data_ptr(), of.data_ptr(),
                        ids.data_ptr(), w.data_ptr(), dl.ws.data_ptr(), dl.ws_bytes,
                        None) == moe.MOE_ERR_ALIGN


def test_deterministic_and_host_entry_matches():
    shape = synth.Shape(1024, 40, 6, 448, 320)
    hl = HostLayer(shape, seed=23)
    orc = hl.oracle()
    dl = device_from_host(hl)
    xs = draw_tokens(orc, 23, 2, 6)
    a = run(dl, xs)
    b = run(dl, xs)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    ob = np.zeros((6, shape.H), np.uint16)
    of = np.zeros((6, shape.H), np.float32)
    ids = np.zeros((6, shape.k), np.int32)
    w = np.zeros((6, shape.k), np.float32)
    moe.moe_decode_host(dl.handle, xs.ctypes.data, 6, ob.ctypes.data, of.ctypes.data,
                        ids.ctypes.data, w.ctypes.data, dl.ws.data_ptr(), dl.ws_bytes, None)
    assert np.array_equal(of, a[0]) and np.array_equal(ob, a[1])
    assert np.array_equal(ids, a[2]) and np.array_equal(w, a[3])


@pytest.mark.parametrize("B,f32", [(1, False), (1, True), (3, False)])
def test_host_entry_replays_match_device_entry(B, f32):
    """moe_decode_host over several calls with changing inputs: the first call
    runs plain launches and captures the step, later ones replay the graph;
    every call's outputs equal moe_decode's on the same inputs."""
    shape = synth.Shape(1024, 40, 6, 448, 320)
    hl = HostLayer(shape, seed=29)
    orc = hl.oracle()
    dl = device_from_host(hl)
    for rep in range(4):
        xs = draw_tokens(orc, 29, 40 + rep, B)
        ref = run(dl, xs)
        ob = np.zeros((B, shape.H), np.uint16)
        of = np.zeros((B, shape.H), np.float32)
        ids = np.zeros((B, shape.k), np.int32)
        w = np.zeros((B, shape.k), np.float32)
        moe.moe_decode_host(dl.handle, xs.ctypes.data, B, ob.ctypes.data, of.ctypes.data if f32 else None,
                            ids.ctypes.data, w.ctypes.data, dl.ws.data_ptr(), dl.ws_bytes, None)
        assert np.array_equal(ob, ref[1]) and np.array_equal(ids, ref[2]) and np.array_equal(w, ref[3])
        if f32:
            assert np.array_equal(of, ref[0])
    assert dl.check() == moe.MOE_OK, moe.last_error()


# ---------------------------------------------------------------- workloads

@pytest.fixture(scope="module")
def mid():
    wl = synth.WORKLOADS["mid-decode"]
    hl = HostLayer(wl.shape, seed=wl.weight_seed)
    return wl, hl, hl.oracle(), device_from_host(hl, max_tokens=128)


@pytest.mark.parametrize("B", [1, 4, 16, 32, 64])
def test_mid_decode(mid, B):
    wl, hl, orc, dl = mid
    xs = draw_tokens(orc, wl.input_seed, 100 + B, B)
    of, ob, ids, w = run(dl, xs)
    for t in range(B):
        ref, rids, rp = orc.token(xs[t])
        assert_token(t, of, ob, ids, w, ref, rids, rp)


@pytest.mark.parametrize("T", [128, 37])
def test_mid_prefill_skewed(mid, T):
    wl_p = synth.WORKLOADS["mid-prefill"]
    _, hl, _, _ = mid
    beta = synth.beta_for(wl_p)
    orc = oracle.Layer(hl.shape.H, hl.shape.E, hl.shape.k, hl.shape.F, hl.shape.Fs,
                       {e: hl.records[e] for e in range(hl.shape.E)}, hl.shared,
                       hl.router_codes, hl.router_sb, beta)
    dl = DeviceLayer(hl.shape, 0, beta=beta, max_tokens=128, device=DEV, host_records=hl.records,
                     host_shared=hl.shared, router=(hl.router_codes, hl.router_sb))
    xs = draw_tokens(orc, wl_p.input_seed, T, T)
    of, ob, ids, w = run(dl, xs, prefill=True)
    counts = np.bincount(ids.reshape(-1), minlength=hl.shape.E)
    assert counts.max() > 2 * counts[counts > 0].mean()   # the skew shows up
    sample = sorted(set(range(0, T, max(1, T // 20))) | {T - 1})
    for t in range(T):
        _, rids, rp = orc.route(xs[t])
        assert np.array_equal(ids[t], rids)
        assert np.abs(w[t] - rp).max() <= P_TOL
    for t in sample:
        ref, rids, rp = orc.token(xs[t])
        assert_token(t, of, ob, ids, w, ref, rids, rp)


@pytest.fixture(scope="module")
def large():
    wl = synth.WORKLOADS["large-decode"]
    s = wl.shape
    dl = DeviceLayer(s, wl.weight_seed, max_tokens=128, device=DEV)
    rc, rsb = synth.router(wl.weight_seed, 0, s.E, s.H)
    shared = synth.expert_record(wl.weight_seed, 0, s.E, s.H, s.Fs)
    orc = oracle.Layer(s.H, s.E, s.k, s.F, s.Fs, {}, shared, rc, rsb)
    yield wl, dl, orc
    dl.close()
    del dl
    torch.cuda.empty_cache()


def _oracle_with_records(orc, wl, ids):
    s = wl.shape
    for e in set(int(v) for v in ids):
        if e not in orc._recs:
            orc.set_record(e, synth.expert_record(wl.weight_seed, 0, e, s.H, s.F))


@pytest.mark.parametrize("B,sample", [(1, [0]), (4, [0, 3]), (16, [0, 9, 15]), (32, [0, 31]), (64, [5, 63])])
def test_large_decode(large, B, sample):
    wl, dl, orc = large
    xs = draw_tokens(orc, wl.input_seed, 200 + B, B)
    of, ob, ids, w = run(dl, xs)
    for t in range(B):
        _, rids, rp = orc.route(xs[t])
        assert np.array_equal(ids[t], rids)
        assert np.abs(w[t] - rp).max() <= P_TOL
    for t in sample:
        _oracle_with_records(orc, wl, ids[t])
        ref, rids, rp = orc.token(xs[t])
        assert_token(t, of, ob, ids, w, ref, rids, rp)


def test_large_prefill_chunk(large):
    wl, dl, orc = large
    T = 128
    xs = draw_tokens(orc, wl.input_seed, 300, T)
    of, ob, ids, w = run(dl, xs, prefill=True)
    for t in range(T):
        _, rids, rp = orc.route(xs[t])
        assert np.array_equal(ids[t], rids)
    for t in (0, 64, 127):
        _oracle_with_records(orc, wl, ids[t])
        ref, rids, rp = orc.token(xs[t])
        assert_token(t, of, ob, ids, w, ref, rids, rp)


def test_decode_kernel_counts(large):
    """moe_decode_kernels follows the dispatch: one token runs the router and
    the fused gate|up + down kernel; 2..16 tokens the router, the few-token
    fused kernel and the combine; 32 tokens over 512 experts one single-token
    pass per token; 64 tokens (64 * 16 > 512) the five tensor-core chunk
    kernels."""
    _, dl, _ = large
    L = moe.lib()
    assert L.moe_decode_kernels(dl.handle, 0) == 0
    assert L.moe_decode_kernels(dl.handle, 1) == 2
    for B in (2, 4, 16):
        assert L.moe_decode_kernels(dl.handle, B) == 3
    assert L.moe_decode_kernels(dl.handle, 32) == 64
    assert L.moe_decode_kernels(dl.handle, 64) == 5
    assert L.moe_decode_kernels(dl.handle, 129) == -1
    assert L.moe_decode_kernels(None, 1) == -1


def test_router_exact_ties_over_512_experts():
    """Router rows repeat every 40 experts, so each logit value is shared by
    15 experts.  The selection by (logit descending, id ascending) must take
    the lowest ids of the tied classes, over E = 600 > 512 candidates (two
    candidates per thread in the top-k's first sorts) and k = 32."""
    shape = synth.Shape(256, 600, 32, 64, 0)
    hl = HostLayer(shape, seed=61)
    for e in range(40, shape.E):
        hl.router_codes[e] = hl.router_codes[e % 40]
        hl.router_sb[e] = hl.router_sb[e % 40]
    orc = hl.oracle()
    for attempt in range(64):  # distinct classes at least 1e-3 apart
        x = synth.hidden(61, 0, 0, shape.H, attempt=attempt)
        lg = orc.route(x)[0]
        if np.diff(np.sort(lg[:40])).min() >= 1e-3:
            break
    else:
        raise RuntimeError("no hidden state with separated logit classes")
    dl = device_from_host(hl, max_tokens=1)
    of, ob, ids, w = run(dl, x[None])
    ref, rids, rp = orc.token(x)
    assert_token(0, of, ob, ids, w, ref, rids, rp)
    chosen = set(int(i) for i in ids[0])
    for i in chosen:  # every lower id of the same class is chosen too
        assert all(j in chosen for j in range(i % 40, i, 40))
