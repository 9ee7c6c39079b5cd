"""moe_decode_noalloc (workspace in the library's static device scratch)
against moe_decode (caller-allocated workspace), through the C ABI.

Same bar as the oracle parity tests: expert ids identical, routing weights
within 1e-5, max |out - out_ref| <= 2e-3 * max |out_ref| + 1e-4, bf16 output
equal to round-to-nearest-even of the fp32 output."""
import numpy as np
import pytest
import torch

from quantized_routed_expert_gemv_gb300 import moe, synth
from quantized_routed_expert_gemv_gb300.device import DeviceLayer, bf16_bits, bf16_tensor

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
    assert moe.moe_workspace_bytes(layer.handle, B) > (4 << 20)
    x = bf16_tensor(np.stack([synth.hidden(21, 2, t, layer.shape.H) for t in range(B)]), DEV)
    with pytest.raises(moe.MoEError) as ei:
        noalloc(layer, x)
    assert ei.value.code == moe.MOE_ERR_ARG
    assert "static scratch" in str(ei.value)
