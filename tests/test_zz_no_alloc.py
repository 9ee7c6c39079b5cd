"""moe_decode_noalloc (workspace in the library's static device scratch)
against moe_decode (caller-allocated workspace), through the C ABI, and
moe_check_noalloc, the scratch's status call.

Callers that cannot allocate device memory while serving use this entry
point; these tests check that it computes what moe_decode computes, on
consecutive calls, across layers of both expert formats sharing the one
scratch, and up to the batch limit the header states for the large layer.

Same bar as the oracle parity tests: expert ids identical, routing weights
within 1e-5, max |out - out_ref| <= 2e-3 * max |out_ref| + 1e-4, bf16 output
equal to round-to-nearest-even of the fp32 output."""
import numpy as np
import pytest
import torch

from quantized_routed_expert_gemv_gb300 import moe, synth
from quantized_routed_expert_gemv_gb300.device import DeviceLayer, bf16_bits, bf16_tensor

# The largest batch of the large layer (H=7168, E=512, top-16, F=Fs=2048)
# whose workspace fits the 16 MiB static scratch, as include/moe.h states it.
LARGE_NOALLOC_MAX_B = 31

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS, P_TOL = 2e-3, 1e-4, 1e-5
DEV = "cuda:0"


@pytest.fixture(scope="module")
def layer():
    dl = DeviceLayer(synth.MID, 11, max_tokens=128, device=DEV)
    yield dl
    dl.close()


def noalloc(dl, x):
    ob, of, ids, w = dl.outputs(x.shape[0])
    st = torch.cuda.current_stream(dl.device).cuda_stream
    moe.moe_decode_noalloc(dl.handle, x.data_ptr(), x.shape[0], ob.data_ptr(), of.data_ptr(),
                           ids.data_ptr(), w.data_ptr(), st)
    return ob, of, ids, w


def host(outs):
    ob, of, ids, w = outs
    return bf16_bits(ob), of.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


def assert_same(got, ref):
    gb, gf, gi, gw = got
    rb, rf, ri, rw = ref
    assert np.array_equal(gi, ri)
    assert np.abs(gw.astype(np.float64) - rw).max() <= P_TOL
    for t in range(gf.shape[0]):
        err = np.abs(gf[t].astype(np.float64) - rf[t]).max()
        bound = TOL_REL * np.abs(rf[t].astype(np.float64)).max() + TOL_ABS
        assert err <= bound, (t, err, bound)
    assert np.array_equal(gb, synth.float_to_bf16_bits(gf))


def test_two_calls_in_a_row_match_moe_decode(layer):
    H = layer.shape.H
    x1 = bf16_tensor(np.stack([synth.hidden(21, 0, 0, H)]), DEV)
    x2 = bf16_tensor(np.stack([synth.hidden(21, 1, t, H) for t in range(4)]), DEV)
    got1 = noalloc(layer, x1)
    got2 = noalloc(layer, x2)
    torch.cuda.synchronize()
    got1, got2 = host(got1), host(got2)
    ref1 = host(layer.decode(x1))
    ref2 = host(layer.decode(x2))
    torch.cuda.synchronize()
    assert layer.check() == moe.MOE_OK, moe.last_error()
    assert_same(got1, ref1)
    assert_same(got2, ref2)


def test_oversize_batch_is_rejected(layer):
    B = 128
    assert moe.moe_workspace_bytes(layer.handle, B) > moe.lib().moe_workspace_bytes(layer.handle, 1)
    assert moe.moe_workspace_bytes(layer.handle, B) > moe.MOE_NOALLOC_SCRATCH_BYTES
    x = bf16_tensor(np.stack([synth.hidden(21, 2, t, layer.shape.H) for t in range(B)]), DEV)
    with pytest.raises(moe.MoEError) as ei:
        noalloc(layer, x)
    assert ei.value.code == moe.MOE_ERR_ARG
    assert "static scratch" in str(ei.value)


def test_status_after_normal_steps_is_ok(layer):
    H = layer.shape.H
    for s in range(3):
        x = bf16_tensor(np.stack([synth.hidden(23, s, t, H) for t in range(1 + s)]), DEV)
        noalloc(layer, x)
    st = torch.cuda.current_stream(layer.device).cuda_stream
    assert moe.moe_check_noalloc(layer.handle, st) == moe.MOE_OK, moe.last_error()


def test_layers_of_both_formats_alternate_on_the_scratch():
    """A 4-bit affine layer and a 3-bit residual-VQ layer take turns on the
    one scratch (one stream, B = 1 and 3): each output equals moe_decode's
    with that layer's own workspace, so no kernel family leaves the shared
    control block in a state the other cannot use."""
    shape = synth.TINY
    a = DeviceLayer(shape, 5, max_tokens=4, device=DEV)
    b = DeviceLayer(shape, 6, max_tokens=4, device=DEV, rvq=True)
    try:
        for s in range(3):
            for dl in (a, b, a):
                for B in (1, 3):
                    x = bf16_tensor(np.stack([synth.hidden(29, 10 * s + B, t, shape.H) for t in range(B)]), DEV)
                    got = host(noalloc(dl, x))
                    ref = host(dl.decode(x))
                    torch.cuda.synchronize()
                    assert_same(got, ref)
        st = torch.cuda.current_stream(a.device).cuda_stream
        assert moe.moe_check_noalloc(a.handle, st) == moe.MOE_OK, moe.last_error()
        assert a.check() == moe.MOE_OK and b.check() == moe.MOE_OK, moe.last_error()
    finally:
        a.close()
        b.close()


def test_large_layer_at_the_stated_batch_limit():
    """The header's limit for the large layer is exact: its workspace fits the
    scratch at B = LARGE_NOALLOC_MAX_B and not one token more; a call at the
    limit equals moe_decode, and one above it is refused before any launch."""
    wl = synth.WORKLOADS["large-decode"]
    s = wl.shape
    dl = DeviceLayer(s, wl.weight_seed, max_tokens=LARGE_NOALLOC_MAX_B + 1, device=DEV)
    try:
        n = LARGE_NOALLOC_MAX_B
        assert moe.moe_workspace_bytes(dl.handle, n) <= moe.MOE_NOALLOC_SCRATCH_BYTES
        assert moe.moe_workspace_bytes(dl.handle, n + 1) > moe.MOE_NOALLOC_SCRATCH_BYTES
        for r in range(2):
            x = bf16_tensor(np.stack([synth.hidden(wl.input_seed, 70 + r, t, s.H) for t in range(n)]), DEV)
            got = host(noalloc(dl, x))
            ref = host(dl.decode(x))
            torch.cuda.synchronize()
            assert_same(got, ref)
        x = bf16_tensor(np.stack([synth.hidden(wl.input_seed, 72, t, s.H) for t in range(n + 1)]), DEV)
        with pytest.raises(moe.MoEError) as ei:
            noalloc(dl, x)
        assert ei.value.code == moe.MOE_ERR_ARG
        st = torch.cuda.current_stream(dl.device).cuda_stream
        assert moe.moe_check_noalloc(dl.handle, st) == moe.MOE_OK, moe.last_error()
        assert dl.check() == moe.MOE_OK, moe.last_error()
    finally:
        dl.close()
