"""Prefill chunks on the tensor-core path (T >= 32 tokens) through the C ABI.

Every token and every element of moe_prefill_chunk's output is compared with
moe_decode on the same tokens (the decode kernels, themselves pinned to the
oracle in test_decode_gpu.py) at the parity bar, and sampled tokens with the
fp64 oracle directly.  Cases: skewed routing at the mid shape for several T,
a hot expert whose tokens span two 64-token blocks, a layer without a shared
expert, the tiny shape, and an identity-expert layer with a closed form.
"""
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


def run(dl, xs, prefill):
    x = bf16_tensor(xs, DEV)
    ob, of, ids, w = (dl.prefill if prefill else dl.decode)(x)
    torch.cuda.synchronize()
    assert dl.check() == moe.MOE_OK, moe.last_error()
    return of.cpu().numpy(), bf16_bits(ob), ids.cpu().numpy(), w.cpu().numpy()


def assert_rows(of, ob, ids, w, ref_of, ref_ids, ref_w):
    assert np.array_equal(ids, ref_ids)
    assert np.abs(w.astype(np.float64) - ref_w).max() <= P_TOL
    for t in range(of.shape[0]):
        err = np.abs(of[t].astype(np.float64) - ref_of[t]).max()
        bound = TOL_REL * np.abs(ref_of[t].astype(np.float64)).max() + TOL_ABS
        assert err <= bound, (t, err, bound)
    assert np.array_equal(ob, synth.float_to_bf16_bits(of))


def check_layer(hl, T, seed, stream, sample=4):
    orc = hl.oracle()
    dl = DeviceLayer(hl.shape, 0, beta=hl.beta, max_tokens=128, device=DEV, host_records=hl.records,
                     host_shared=hl.shared, router=(hl.router_codes, hl.router_sb))
    xs = np.stack([hidden_with_margin(orc, seed, stream, t) for t in range(T)])
    got = run(dl, xs, prefill=True)
    ref = run(dl, xs, prefill=False)
    assert_rows(*got, *ref[:1], ref[2], ref[3])
    of, ob, ids, w = got
    for t in sorted(set(np.linspace(0, T - 1, sample).astype(int).tolist())):
        r, rids, rp = orc.token(xs[t])
        assert np.array_equal(ids[t], rids)
        assert np.abs(w[t] - rp).max() <= P_TOL
        err = np.abs(of[t].astype(np.float64) - r).max()
        assert err <= TOL_REL * np.abs(r).max() + TOL_ABS, (t, err)
    dl.close()
    return ids


@pytest.fixture(scope="module")
def mid_host():
    wl = synth.WORKLOADS["mid-prefill"]
    return HostLayer(wl.shape, wl.weight_seed, beta=synth.beta_for(wl))


@pytest.mark.parametrize("T", [32, 33, 64, 100, 128])
def test_mid_skewed_all_tokens(mid_host, T):
    check_layer(mid_host, T, 41, T)


def test_hot_expert_spans_blocks():
    shape = synth.Shape(512, 16, 2, 256, 256)
    beta = np.zeros(16, np.float32)
    beta[3], beta[7] = 30.0, 20.0   # every token routes to experts 3 and 7
    hl = HostLayer(shape, 8, beta=beta)
    ids = check_layer(hl, 128, 43, 0)
    assert set(ids.reshape(-1).tolist()) == {3, 7}


def test_without_shared_expert():
    hl = HostLayer(synth.Shape(256, 16, 4, 128, 0), 9, beta=synth.beta_normal(9, 0, 16))
    check_layer(hl, 48, 44, 0)


def test_tiny_shape():
    hl = HostLayer(synth.TINY, 0, beta=synth.beta_normal(1, 0, synth.TINY.E))
    check_layer(hl, 40, 45, 0)


def test_identity_experts_closed_form():
    E, k, H = 8, 2, 128
    records, shared, rc, rsb = identity_layer(E, k, H)
    shape = synth.Shape(H, E, k, H, H)
    dl = DeviceLayer(shape, 0, max_tokens=64, device=DEV, host_records=records, host_shared=shared,
                     router=(rc, rsb))
    T = 32
    xs = np.stack([synth.hidden(6, 0, t, H) for t in range(T)])
    xs[:, 0] = synth.bf16_from_double(8.0)
    of, ob, ids, w = run(dl, xs, prefill=True)
    for t in range(T):
        x = synth.bf16_bits_to_float(xs[t]).astype(np.float64)
        scale = 1.0 + sum(float(w[t, i]) * 2.0 ** -(int(ids[t, i]) % 3) for i in range(k))
        # every product and partial sum is exact until the final fp32 combine
        np.testing.assert_allclose(of[t], scale * x, rtol=2e-6, atol=1e-30)
    dl.close()


def test_wide_hidden_router_token_blocks():
    """H = 8192 with E = 8: a router row spans 16 warps, so a token pass holds
    2 tokens and a 128-token chunk has 64 passes over 2 row blocks of 4
    experts.  The router then runs at its cap of 48 token blocks, some of
    them two passes long; the last row-block CTA of each token block takes
    that block's top-k and the last token block groups every pair.  Every
    token's ids and weights are checked against the oracle's routing, and
    sampled outputs against the oracle."""
    shape = synth.Shape(8192, 8, 2, 128, 128)
    hl = HostLayer(shape, 12, beta=synth.beta_normal(12, 0, 8))
    orc = hl.oracle()
    T = 128
    xs = np.stack([hidden_with_margin(orc, 47, 0, t) for t in range(T)])
    for prefill, n in ((True, T), (False, 16)):
        dl = DeviceLayer(shape, 0, beta=hl.beta, max_tokens=128, device=DEV, host_records=hl.records,
                         host_shared=hl.shared, router=(hl.router_codes, hl.router_sb))
        of, ob, ids, w = run(dl, xs[:n], prefill)
        for t in range(n):
            _, rids, rp = orc.route(xs[t])
            assert np.array_equal(ids[t], rids), (prefill, t, ids[t], rids)
            assert np.abs(w[t] - rp).max() <= P_TOL
        assert np.array_equal(ob, synth.float_to_bf16_bits(of))
        for t in (0, n // 2, n - 1):
            r, _, _ = orc.token(xs[t])
            err = np.abs(of[t].astype(np.float64) - r).max()
            assert err <= TOL_REL * np.abs(r).max() + TOL_ABS, (prefill, t, err)
        dl.close()
