"""The HBM expert cache (moe_residency_*) through the C ABI.

* The hand-worked LFU trace (tests/golden/lfu_trace.txt) replayed on the GPU
  path: the router is steered to the trace's ids by a large per-expert logit
  offset; slot contents and hit/miss counts must follow the trace exactly.
* Zipf-biased streams at B=1 (single-token kernels split around the cache
  update) and B=4 (general kernels): hits, misses and slot contents equal
  the oracle's LFU replay of the ids the GPU chose; outputs equal
  moe_decode's with every expert resident, and the fp64 oracle's within the
  parity bar.
* Host-side fault injection: a wrong slot tag is caught by the kernels
  (MOE_ERR_RESIDENCY through moe_check); a failed copy returns MOE_ERR_CUDA,
  leaves the slot empty, and the next step recovers.
* A step needing more experts than slots runs as waves of consecutive
  tokens, replayed exactly by the oracle.
* The streamed workload's own layer shape (H=7168, F=Fs=2048, top-16,
  Zipf(1.1) router offsets; E cut to 64, 24 slots): B=1 steps with
  evictions and a B=4 step in waves, every output against the oracle.
* The optional CRC-32 check of host records: a wrong checksum refuses the
  step that would upload the record, with the cache state unchanged.
* Router lookahead (moe_residency_lookahead): the hand-worked trace
  (tests/golden/lfu_lookahead_trace.txt, its one-token rows) replayed with a
  steered router; Zipf streams at B=1 and B=4, the lookahead on its own
  streams in the second, whose slots and counters equal the oracle's replay
  of the ids the GPU predicted and chose, with outputs unchanged; a failed
  lookahead copy and a record failing its checksum.
"""
import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from layers import HostLayer, hidden_with_margin
from quantized_routed_expert_gemv_gb300 import moe, synth
from quantized_routed_expert_gemv_gb300.device import (CachedLayer, DeviceLayer, bf16_bits,
                                                       bf16_tensor, pinned_records)

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS, P_TOL = 2e-3, 1e-4, 1e-5
DEV = "cuda:0"
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def host(outs):
    ob, of, ids, w = outs
    torch.cuda.synchronize()
    return bf16_bits(ob), of.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


def assert_close(got, ref):
    gb, gf, gi, gw = got
    rb, rf, ri, rw = ref
    assert np.array_equal(gi, ri)
    assert np.abs(gw.astype(np.float64) - rw).max() <= P_TOL
    for t in range(gf.shape[0]):
        err = np.abs(gf[t].astype(np.float64) - rf[t]).max()
        assert err <= TOL_REL * np.abs(rf[t].astype(np.float64)).max() + TOL_ABS
    assert np.array_equal(gb, synth.float_to_bf16_bits(gf))


def assert_oracle(got, t, ref_out, ref_ids, ref_p):
    gb, gf, gi, gw = got
    assert np.array_equal(gi[t], ref_ids)
    assert np.abs(gw[t].astype(np.float64) - ref_p).max() <= P_TOL
    err = np.abs(gf[t].astype(np.float64) - ref_out).max()
    assert err <= TOL_REL * np.abs(ref_out).max() + TOL_ABS


def make(shape, seed, beta, n_slots, max_tokens=4):
    hl = HostLayer(shape, seed, beta=beta)
    dl = DeviceLayer(shape, seed, beta=beta, max_tokens=max_tokens, device=DEV,
                     host_records=hl.records, host_shared=hl.shared,
                     router=(hl.router_codes, hl.router_sb))
    cl = CachedLayer(dl, pinned_records(shape, seed, host_records=hl.records), n_slots)
    return hl, dl, cl


def first_appearance(ids):
    seen, order = set(), []
    for e in np.asarray(ids).reshape(-1):
        if int(e) not in seen:
            seen.add(int(e))
            order.append(int(e))
    return np.array(order, np.int32)


def test_hand_trace_on_gpu():
    rows = [l.split("|") for l in open(os.path.join(GOLDEN, "lfu_trace.txt"))
            if l.strip() and not l.startswith("#")]
    shape = synth.Shape(64, 6, 2, 64, 64)
    hl, dl, cl = make(shape, 5, np.zeros(6, np.float32), 3, max_tokens=1)
    x = bf16_tensor(synth.hidden(5, 0, 0, 64)[None], DEV)
    prev = cl.stats()
    for r in rows:
        ids = [int(t) for t in r[1].split()]
        hits = [int(t) for t in r[2].split()]
        beta = np.zeros(6, np.float32)
        beta[ids[0]], beta[ids[1]] = 200.0, 100.0
        dl.beta.copy_(torch.from_numpy(beta))
        got = host(cl.decode(x))
        assert list(got[2][0]) == ids
        assert cl.slots() == [int(t) for t in r[4].split()]
        st = cl.stats()
        assert st["hits"] - prev["hits"] == sum(hits)
        assert st["misses"] - prev["misses"] == len(ids) - sum(hits)
        prev = st
        ref = host(dl.decode(x))
        assert_close(got, ref)
    assert dl.check() == moe.MOE_OK, moe.last_error()
    assert prev["steps"] == len(rows)
    assert prev["bytes_h2d"] == prev["misses"] * oracle.record_layout(64, 64)["bytes"]
    cl.close()
    dl.close()


@pytest.mark.parametrize("B,steps,n_slots", [(1, 40, 8), (4, 16, 16)])
def test_zipf_stream_matches_lfu_replay_and_oracle(B, steps, n_slots):
    shape = synth.Shape(256, 64, 4, 128, 256)
    beta = synth.beta_zipf(4, 0, 64)
    hl, dl, cl = make(shape, 7, beta, n_slots, max_tokens=B)
    orc = hl.oracle()
    lfu = oracle.LFU(n_slots, 64)
    prev = cl.stats()
    for s in range(steps):
        xs = np.stack([hidden_with_margin(orc, 9, s, t) for t in range(B)])
        x = bf16_tensor(xs, DEV)
        got = host(cl.decode(x))
        hit, _, m = lfu.step(first_appearance(got[2]))
        st = cl.stats()
        assert st["misses"] - prev["misses"] == m
        assert st["hits"] - prev["hits"] == int(hit.sum())
        assert cl.slots() == list(lfu.slot_expert)
        prev = st
        assert_close(got, host(dl.decode(x)))
        if s % 8 == 0 or s == steps - 1:
            for t in range(B):
                assert_oracle(got, t, *orc.token(xs[t]))
    assert dl.check() == moe.MOE_OK, moe.last_error()
    assert prev["evictions"] > 0 and prev["hits"] > 0
    cl.close()
    dl.close()


def test_faults_are_caught_and_recovered():
    shape = synth.Shape(256, 16, 2, 128, 256)
    hl, dl, cl = make(shape, 3, None, 4, max_tokens=2)
    orc = hl.oracle()
    xs = [np.stack([hidden_with_margin(orc, 13, s, 0)]) for s in range(4)]
    # a copy that fails: MOE_ERR_CUDA, its slot left empty, nothing counted twice
    cl.set_fault(moe.MOE_RESIDENCY_FAULT_COPY)
    with pytest.raises(moe.MoEError) as ei:
        cl.decode(bf16_tensor(xs[0], DEV))
    assert ei.value.code == moe.MOE_ERR_CUDA
    torch.cuda.synchronize()
    assert cl.slots().count(-1) >= 3
    got = host(cl.decode(bf16_tensor(xs[0], DEV)))
    assert dl.check() == moe.MOE_OK, moe.last_error()
    assert_oracle(got, 0, *orc.token(xs[0][0]))
    # a wrong slot tag: the kernels refuse the slot and latch MOE_ERR_RESIDENCY
    cl.set_fault(moe.MOE_RESIDENCY_FAULT_TAG)
    cl.decode(bf16_tensor(xs[1], DEV))
    assert dl.check() == moe.MOE_ERR_RESIDENCY
    # moe_check cleared the workspace's persistent counters with the error:
    # the single-token kernels of a plain decode run on the same workspace
    got = host(dl.decode(bf16_tensor(xs[1], DEV)))
    assert dl.check() == moe.MOE_OK, moe.last_error()
    assert_oracle(got, 0, *orc.token(xs[1][0]))
    got = host(cl.decode(bf16_tensor(xs[2], DEV)))
    assert dl.check() == moe.MOE_OK, moe.last_error()
    assert_oracle(got, 0, *orc.token(xs[2][0]))
    cl.close()
    dl.close()


def test_waves_when_a_step_needs_more_experts_than_slots():
    """A step whose tokens need more distinct experts than there are slots
    runs as waves of consecutive tokens (each a cache step): slots and
    counters equal the oracle's LFU replay of the waves oracle.waves cuts
    from the GPU's ids; outputs equal moe_decode's and the oracle's."""
    shape = synth.Shape(256, 64, 4, 128, 256)
    beta = synth.beta_zipf(4, 0, 64)
    B, n_slots = 8, 8
    hl, dl, cl = make(shape, 9, beta, n_slots, max_tokens=B)
    orc = hl.oracle()
    lfu = oracle.LFU(n_slots, 64)
    n_waves = 0
    for s in range(6):
        xs = np.stack([hidden_with_margin(orc, 31, s, t) for t in range(B)])
        x = bf16_tensor(xs, DEV)
        got = host(cl.decode(x))
        ws = oracle.waves(got[2], n_slots)
        assert len(ws) > 1
        for t0, t1 in ws:
            lfu.step(first_appearance(got[2][t0:t1]))
        n_waves += len(ws)
        st = cl.stats()
        assert st["steps"] == n_waves
        assert (st["hits"], st["misses"], st["evictions"]) == (lfu.hits, lfu.misses, lfu.evictions)
        assert cl.slots() == list(lfu.slot_expert)
        assert_close(got, host(dl.decode(x)))
        for t in (0, B - 1):
            assert_oracle(got, t, *orc.token(xs[t]))
    assert dl.check() == moe.MOE_OK, moe.last_error()
    cl.close()
    dl.close()


def test_record_checksums():
    """moe_residency_verify, the optional CRC-32 payload check: with the true
    checksums every step runs and matches the oracle; a wrong value for one
    expert refuses the first step that uploads its record (MOE_ERR_RESIDENCY
    naming the expert, cache state unchanged); switched off, that step runs."""
    shape = synth.Shape(256, 16, 2, 128, 256)
    hl, dl, cl = make(shape, 4, None, 4, max_tokens=2)
    orc = hl.oracle()
    L = moe.lib()
    lay = moe.moe_record_layout()
    assert L.moe_record_layout_of(shape.H, shape.F, ctypes.byref(lay)) == moe.MOE_OK
    base = cl.host.data_ptr()
    crc = np.array([L.moe_crc32(base + e * lay.stride, lay.bytes) for e in range(shape.E)], np.uint32)
    assert L.moe_residency_verify(cl.handle, crc.ctypes.data) == moe.MOE_OK
    x0 = np.stack([hidden_with_margin(orc, 17, 0, 0)])
    got = host(cl.decode(bf16_tensor(x0, DEV)))
    assert dl.check() == moe.MOE_OK, moe.last_error()
    assert_oracle(got, 0, *orc.token(x0[0]))
    # a token that needs a record not yet resident
    resident = set(cl.slots())
    for s in range(1, 64):
        x1 = np.stack([hidden_with_margin(orc, 17, s, 0)])
        need = [int(e) for e in orc.route(x1[0])[1] if int(e) not in resident]
        if need:
            break
    else:
        pytest.fail("no token needing a non-resident expert")
    bad = crc.copy()
    bad[need[0]] ^= 1
    assert L.moe_residency_verify(cl.handle, bad.ctypes.data) == moe.MOE_OK  # resident records still match
    before, slots = cl.stats(), cl.slots()
    with pytest.raises(moe.MoEError) as ei:
        cl.decode(bf16_tensor(x1, DEV))
    assert ei.value.code == moe.MOE_ERR_RESIDENCY
    assert f"expert {need[0]} " in str(ei.value)
    torch.cuda.synchronize()
    assert cl.stats() == before and cl.slots() == slots
    assert L.moe_residency_verify(cl.handle, None) == moe.MOE_OK
    got = host(cl.decode(bf16_tensor(x1, DEV)))
    assert dl.check() == moe.MOE_OK, moe.last_error()
    assert_oracle(got, 0, *orc.token(x1[0]))
    cl.close()
    dl.close()


def test_lookahead_hand_trace_on_gpu():
    rows = [[c.strip() for c in l.split("|")]
            for l in open(os.path.join(GOLDEN, "lfu_lookahead_trace.txt"))
            if l.strip() and not l.startswith("#")]
    rows = [r for r in rows if ";" not in r[3]]  # one-token rows: the router is steered per expert
    assert len(rows) >= 8
    shape = synth.Shape(64, 6, 2, 64, 64)
    hl, dl, cl = make(shape, 5, np.zeros(6, np.float32), 3, max_tokens=1)
    x = bf16_tensor(synth.hidden(5, 0, 0, 64)[None], DEV)
    keys = ("hits", "misses", "lookahead_copies", "lookahead_hits", "evictions")
    for r in rows[:8]:                                   # rows 1-8 run back to back
        ids = [int(t) for t in r[3].split()]
        beta = np.zeros(6, np.float32)
        beta[ids[0]], beta[ids[1]] = 200.0, 100.0
        dl.beta.copy_(torch.from_numpy(beta))
        prev = cl.stats()
        if r[1] == "D":
            got = host(cl.decode(x))
            assert list(got[2][0]) == ids
            assert_close(got, host(dl.decode(x)))
        else:
            pids, _ = cl.lookahead(x, int(r[2]))
            torch.cuda.synchronize()
            assert list(pids.cpu().numpy()[0]) == ids
        st = cl.stats()
        assert [st[k] - prev[k] for k in keys] == [int(t) for t in r[4:9]], f"row {r[0]}"
        assert cl.slots() == [int(t) for t in r[9].split()], f"row {r[0]}"
    st = cl.stats()
    rec = oracle.record_layout(64, 64)["bytes"]
    assert st["lookaheads"] == sum(1 for r in rows[:8] if r[1] == "P")
    assert st["lookahead_bytes"] == st["lookahead_copies"] * rec
    assert st["bytes_h2d"] == st["misses"] * rec
    assert dl.check() == moe.MOE_OK, moe.last_error()
    assert cl.check_lookahead() == moe.MOE_OK, moe.last_error()
    cl.close()
    dl.close()


@pytest.mark.parametrize("B,steps,n_slots,n_ahead,own_streams", [(1, 40, 8, 2, False),
                                                                 (4, 16, 16, 2, True)])
def test_lookahead_zipf_stream_matches_replay(B, steps, n_slots, n_ahead, own_streams):
    shape = synth.Shape(256, 64, 4, 128, 256)
    beta = synth.beta_zipf(4, 0, 64)
    hl, dl, cl = make(shape, 7, beta, n_slots, max_tokens=B)
    orc = hl.oracle()
    lfu = oracle.LFU(n_slots, 64)
    ls = torch.cuda.Stream(DEV) if own_streams else None
    lc = torch.cuda.Stream(DEV) if own_streams else None
    keys = ("hits", "misses", "evictions", "lookahead_copies", "lookahead_hits")
    for s in range(steps):
        # the "earlier" hidden state of the lookahead and the step's own
        xp = bf16_tensor(np.stack([hidden_with_margin(orc, 21, s, t) for t in range(B)]), DEV)
        xs = np.stack([hidden_with_margin(orc, 9, s, t) for t in range(B)])
        x = bf16_tensor(xs, DEV)
        if own_streams:
            ls.wait_stream(torch.cuda.current_stream(DEV))
            pids, _ = cl.lookahead(xp, n_ahead, stream=ls.cuda_stream, copy_stream=lc)
            torch.cuda.current_stream(DEV).wait_stream(ls)
        else:
            pids, _ = cl.lookahead(xp, n_ahead)
        pred = pids.cpu().numpy()
        assert np.array_equal(pred, host(dl.decode(xp))[2])    # the layer's own router on xp
        lfu.lookahead(pred, n_ahead)
        assert cl.slots() == list(lfu.slot_expert)
        got = host(cl.decode(x))
        lfu.step(first_appearance(got[2]))
        st = cl.stats()
        assert [st[k] for k in keys] == [getattr(lfu, k) for k in keys]
        assert cl.slots() == list(lfu.slot_expert)
        assert_close(got, host(dl.decode(x)))
        if s % 8 == 0 or s == steps - 1:
            for t in range(B):
                assert_oracle(got, t, *orc.token(xs[t]))
    assert dl.check() == moe.MOE_OK, moe.last_error()
    assert cl.check_lookahead() == moe.MOE_OK, moe.last_error()
    st = cl.stats()
    assert st["lookahead_copies"] > 0 and st["lookahead_hits"] >= 0 and st["lookaheads"] == steps
    cl.close()
    dl.close()


def test_lookahead_faults():
    """A lookahead copy that fails: MOE_ERR_CUDA, its slot left empty, and
    the next step still matches the oracle.  A predicted record that fails
    its CRC-32 check: MOE_ERR_RESIDENCY, cache state unchanged."""
    shape = synth.Shape(256, 16, 2, 128, 256)
    hl, dl, cl = make(shape, 3, None, 4, max_tokens=1)
    orc = hl.oracle()
    x0 = np.stack([hidden_with_margin(orc, 23, 0, 0)])
    cl.set_fault(moe.MOE_RESIDENCY_FAULT_COPY)
    with pytest.raises(moe.MoEError) as ei:
        cl.lookahead(bf16_tensor(x0, DEV), 2)
    assert ei.value.code == moe.MOE_ERR_CUDA
    torch.cuda.synchronize()
    assert cl.slots().count(-1) == 4
    got = host(cl.decode(bf16_tensor(x0, DEV)))
    assert dl.check() == moe.MOE_OK, moe.last_error()
    assert_oracle(got, 0, *orc.token(x0[0]))
    # checksums: a wrong value for a predicted, non-resident expert
    L = moe.lib()
    lay = moe.moe_record_layout()
    assert L.moe_record_layout_of(shape.H, shape.F, ctypes.byref(lay)) == moe.MOE_OK
    base = cl.host.data_ptr()
    crc = np.array([L.moe_crc32(base + e * lay.stride, lay.bytes) for e in range(shape.E)], np.uint32)
    resident = set(cl.slots())
    for s in range(1, 64):
        x1 = np.stack([hidden_with_margin(orc, 23, s, 0)])
        need = [int(e) for e in orc.route(x1[0])[1] if int(e) not in resident]
        if need:
            break
    else:
        pytest.fail("no token needing a non-resident expert")
    bad = crc.copy()
    bad[need[0]] ^= 1
    assert L.moe_residency_verify(cl.handle, bad.ctypes.data) == moe.MOE_OK
    before, slots = cl.stats(), cl.slots()
    with pytest.raises(moe.MoEError) as ei:
        cl.lookahead(bf16_tensor(x1, DEV), 2)
    assert ei.value.code == moe.MOE_ERR_RESIDENCY and f"expert {need[0]} " in str(ei.value)
    assert cl.stats() == before and cl.slots() == slots
    assert L.moe_residency_verify(cl.handle, crc.ctypes.data) == moe.MOE_OK
    cl.lookahead(bf16_tensor(x1, DEV), 2)
    got = host(cl.decode(bf16_tensor(x1, DEV)))
    assert dl.check() == moe.MOE_OK, moe.last_error()
    assert cl.check_lookahead() == moe.MOE_OK, moe.last_error()
    assert_oracle(got, 0, *orc.token(x1[0]))
    st = cl.stats()
    assert st["lookahead_hits"] >= 1 and st["misses"] - before["misses"] == 0
    cl.close()
    dl.close()


def test_streamed_workload_shape_through_the_cache():
    """The cache at the streamed workload's layer shape, where its kernels
    run the large tile plan (gate|up of the shared expert during the copies,
    then the routed gate|up and the down + combine).  E is cut to 64 and the
    cache to 24 slots so that the layer fits a test (1.6 GB of records).
    Six B=1 steps (two fill the cache, the rest evict) and one B=4 step (64
    pairs over more distinct experts than slots: waves).  Every token of
    every step: ids bit-exact, weights within 1e-5 and out_f32 within the
    parity bar of the fp64 oracle; counters and slots equal the oracle's LFU
    replay of the waves it cuts from the GPU's ids."""
    E, n_slots = 64, 24
    shape = synth.Shape(7168, E, 16, 2048, 2048)
    beta = synth.beta_zipf(4, 0, E)
    hl, dl, cl = make(shape, 4, beta, n_slots, max_tokens=4)
    orc = hl.oracle()
    lfu = oracle.LFU(n_slots, E)
    n_waves = 0
    with ThreadPoolExecutor(max_workers=8) as pool:   # the oracle's C code runs outside the GIL
        for s, B in enumerate([1, 1, 1, 1, 1, 1, 4]):
            xs = np.stack([hidden_with_margin(orc, 43, s, t) for t in range(B)])
            refs = pool.map(orc.token, list(xs))
            got = host(cl.decode(bf16_tensor(xs, DEV)))
            assert dl.check() == moe.MOE_OK, moe.last_error()
            for t, ref in enumerate(refs):
                assert_oracle(got, t, *ref)
            assert np.array_equal(got[0], synth.float_to_bf16_bits(got[1]))
            ws = oracle.waves(got[2], n_slots)
            for t0, t1 in ws:
                lfu.step(first_appearance(got[2][t0:t1]))
            n_waves += len(ws)
            st = cl.stats()
            assert st["steps"] == n_waves
            assert (st["hits"], st["misses"], st["evictions"]) == (lfu.hits, lfu.misses, lfu.evictions)
            assert cl.slots() == list(lfu.slot_expert)
    st = cl.stats()
    assert st["evictions"] > 0 and st["hits"] > 0 and n_waves > 7
    assert st["bytes_h2d"] == st["misses"] * oracle.record_layout(shape.H, shape.F)["bytes"]
    cl.close()
    dl.close()
