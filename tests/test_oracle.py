"""Pins of the fp64 oracle against things other than itself: hand-worked
closed forms, library routines (numpy / scipy / torch float64), brute force
and invariants.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from layers import (HostLayer, HostLayerRVQ, dense4, dense8, hidden_with_margin, identity_layer,
                    identity_layer_rvq,
                    record_mats)
from quantized_routed_expert_gemv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_blocks():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "dequant_blocks.txt"))
             if l.strip() and not l.startswith("#")]
    blocks = []
    for i in range(0, len(lines), 4):
        hdr, codes, byts, exp = lines[i:i + 4]
        assert hdr[0] == "block" and codes[0] == "codes" and byts[0] == "bytes"
        blocks.append(dict(bits=int(hdr[1]), s_bits=int(hdr[2], 16), s=float(hdr[3]),
                           b_bits=int(hdr[4], 16), b=float(hdr[5]),
                           codes=[int(t) for t in codes[1:]],
                           bytes=np.array([int(t, 16) for t in byts[1:]], np.uint8),
                           expect=[float(t) for t in exp[1:]]))
    return blocks


# ---- bf16 and dequantisation --------------------------------------------------

@pytest.mark.parametrize("bits,val", [(0x3F80, 1.0), (0xC000, -2.0), (0x3E00, 0.125),
                                      (0x0000, 0.0), (0x8000, -0.0), (0x3EAB, 0.333984375),
                                      (0x7F7F, 3.3895313892515355e38), (0x0001, 2.0 ** -133)])
def test_bf16_widening(bits, val):
    assert oracle.bf16_to_double(bits) == val


@pytest.mark.parametrize("blk", _golden_blocks(), ids=lambda b: f"{b['bits']}bit")
def test_dequant_hand_blocks(blk):
    sb = np.array([blk["s_bits"] | (blk["b_bits"] << 16)], np.uint32)
    codes = blk["bytes"]
    assert oracle.bf16_to_double(blk["s_bits"]) == blk["s"]
    assert oracle.bf16_to_double(blk["b_bits"]) == blk["b"]
    for j in range(64):
        if blk["bits"] == 4:
            got = oracle.dequant4(codes, sb, 64, 0, j)
        else:
            got = oracle.dequant8(codes, sb, 64, 0, j)
        assert got == blk["expect"][j], (j, got)


def test_dequant_group_boundary():
    # Two groups per row, two rows: each (row, group) has its own scale/bias,
    # so a wrong group or row index picks the wrong pair.
    cols, rows = 128, 2
    q = np.full((rows, cols), 3, np.uint8)
    scales = [[1.0, 2.0], [4.0, 8.0]]
    biases = [[0.0, 0.5], [-1.0, 0.25]]
    s_bits = np.array([[synth.bf16_from_double(v) for v in r] for r in scales], np.uint16)
    b_bits = np.array([[synth.bf16_from_double(v) for v in r] for r in biases], np.uint16)
    codes = synth.pack_codes4(q)
    sb = synth.pack_sb(s_bits, b_bits)
    for r in range(rows):
        for j in (0, 63, 64, 127):
            g = j // 64
            assert oracle.dequant4(codes, sb, cols, r, j) == 3 * scales[r][g] + biases[r][g]


def test_gemv_orientation_single_weight():
    # One non-zero weight at (r0, j0): y must be x[j0] at row r0 only.
    rows, cols = 5, 128
    r0, j0 = 3, 77
    q = np.zeros((rows, cols), np.uint8)
    q[r0, j0] = 1
    one, zero = synth.bf16_from_double(1.0), synth.bf16_from_double(0.0)
    sb = synth.pack_sb(np.full((rows, 2), one, np.uint16), np.full((rows, 2), zero, np.uint16))
    x = np.arange(cols, dtype=np.float64) * 0.5 + 1.0
    y = oracle.gemv4(synth.pack_codes4(q), sb, rows, cols, x)
    expect = np.zeros(rows)
    expect[r0] = x[j0]
    assert np.array_equal(y, expect)


def test_gemv_bias_term():
    # All codes 0: y_r = sum_g b_{r,g} * sum_{j in g} x_j (closed form).
    rows, cols = 3, 192
    q = np.zeros((rows, cols), np.uint8)
    bvals = np.array([[0.5, -1.0, 2.0], [0.25, 0.0, -0.5], [1.0, 1.0, 1.0]])
    b_bits = np.vectorize(synth.bf16_from_double)(bvals).astype(np.uint16)
    s_bits = np.full((rows, 3), synth.bf16_from_double(1.0), np.uint16)
    x = np.linspace(-1, 1, cols)
    y = oracle.gemv4(synth.pack_codes4(q), synth.pack_sb(s_bits, b_bits), rows, cols, x)
    gs = x.reshape(3, 64).sum(axis=1)
    np.testing.assert_allclose(y, bvals @ gs, rtol=1e-14, atol=1e-14)


# ---- SiLU -----------------------------------------------------------------------

def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(64.0) == 64.0            # e^-64 vanishes against 1 in float64
    assert math.isclose(oracle.silu(math.log(3.0)), 0.75 * math.log(3.0), rel_tol=1e-15)
    for z in (0.3, 1.7, 5.0, 11.0):
        # silu(-z) = silu(z) - z
        assert abs(oracle.silu(-z) - (oracle.silu(z) - z)) <= 4e-16 * z
    assert oracle.silu(-800.0) == -0.0 or abs(oracle.silu(-800.0)) < 1e-300


# ---- router, top-k and weights ---------------------------------------------------

def _topk_via_layer(logits, k):
    """Route through the oracle with a router whose logits equal `logits`:
    H=64, all codes 0, scale 1, bias 0 -> W x = 0, so l = beta exactly."""
    E = logits.size
    H = 64
    rc = np.zeros((E, H), np.uint8)
    sb = synth.pack_sb(np.full((E, 1), synth.bf16_from_double(1.0), np.uint16),
                       np.zeros((E, 1), np.uint16))
    lay = oracle.Layer(H, E, k, 64, 0, {}, None, rc, sb, np.asarray(logits, np.float32))
    return lay.route(np.zeros(H, np.uint16))


def test_topk_ties_go_to_lower_id():
    logits = np.array([1.0, 3.0, 2.0, 3.0, 0.5, 2.0], np.float32)
    _, ids, p = _topk_via_layer(logits, 4)
    assert list(ids) == [1, 3, 2, 5]
    assert p[0] == p[1] and p[2] == p[3]


def test_topk_k1_weight_is_exactly_one():
    _, ids, p = _topk_via_layer(np.array([0.1, -2.0, 7.5, 7.0], np.float32), 1)
    assert list(ids) == [2] and p[0] == 1.0


@pytest.mark.parametrize("E,k", [(8, 2), (128, 8), (512, 16), (64, 64)])
def test_topk_against_library(E, k):
    rng = np.random.default_rng(E * 31 + k)
    logits = rng.normal(0, 3, E).astype(np.float32)
    lg, ids, p = _topk_via_layer(logits, k)
    l64 = logits.astype(np.float64)
    assert np.array_equal(lg, l64)
    order = np.lexsort((np.arange(E), -l64))[:k]          # library sort: (desc, id asc)
    assert np.array_equal(ids, order)
    sm = torch.softmax(torch.tensor(l64, dtype=torch.float64), 0).numpy()
    ref = sm[order] / sm[order].sum()                       # softmax over all, renormalised
    np.testing.assert_allclose(p, ref, rtol=1e-13, atol=0)
    assert abs(p.sum() - 1.0) < 1e-12
    assert np.all(np.diff(p) <= 0)


def test_router_logits_vs_numpy_dense():
    E, H = 16, 256
    rc, rsb = synth.router(7, 0, E, H)
    beta = synth.beta_normal(7, 0, E)
    x = synth.hidden(7, 0, 0, H)
    lay = oracle.Layer(H, E, 4, 64, 0, {}, None, rc, rsb, beta)
    logits, _, _ = lay.route(x)
    W = dense8(rc, rsb, E, H)
    xd = synth.bf16_bits_to_float(x).astype(np.float64)
    np.testing.assert_allclose(logits, W @ xd + beta.astype(np.float64), rtol=1e-12, atol=1e-12)


# ---- whole layer --------------------------------------------------------------------

def _torch_layer(hl, x_bits):
    """The layer from library routines in float64: torch.matmul, F.silu,
    torch.softmax, torch.topk (stable ordering enforced by id tie-break)."""
    s = hl.shape
    xd = torch.tensor(synth.bf16_bits_to_float(x_bits).astype(np.float64))
    Wr = torch.tensor(dense8(hl.router_codes, hl.router_sb, s.E, s.H))
    logits = Wr @ xd
    if hl.beta is not None:
        logits = logits + torch.tensor(hl.beta.astype(np.float64))
    order = np.lexsort((np.arange(s.E), -logits.numpy()))[:s.k]
    pr = torch.softmax(logits, 0)[order]
    pr = pr / pr.sum()

    def ffn(rec, F):
        Wg, Wu, Wd = (torch.tensor(m) for m in hl.mats(rec, F))
        return Wd @ (torch.nn.functional.silu(Wg @ xd) * (Wu @ xd))

    out = ffn(hl.shared, s.Fs) if s.Fs else torch.zeros(s.H, dtype=torch.float64)
    for i, e in enumerate(order):
        out = out + pr[i] * ffn(hl.records[e], s.F)
    return out.numpy(), order, pr.numpy()


SMALL = [synth.TINY, synth.Shape(64, 4, 4, 64, 64), synth.Shape(128, 6, 3, 64, 0),
         synth.Shape(192, 5, 1, 128, 64)]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: f"H{s.H}E{s.E}k{s.k}F{s.F}Fs{s.Fs}")
def test_layer_vs_torch_float64(shape):
    hl = HostLayer(shape, seed=0, beta=synth.beta_normal(0, 0, shape.E))
    orc = hl.oracle()
    for t in range(2):
        x = synth.hidden(0, 99, t, shape.H)
        out, ids, p = orc.token(x)
        ref, rids, rp = _torch_layer(hl, x)
        assert np.array_equal(ids, rids)
        np.testing.assert_allclose(p, rp, rtol=1e-12)
        scale = np.abs(ref).max()
        assert np.abs(out - ref).max() <= 1e-12 * scale


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: f"H{s.H}E{s.E}k{s.k}F{s.F}Fs{s.Fs}")
def test_masked_dense_equals_sparse(shape):
    hl = HostLayer(shape, seed=5)
    orc = hl.oracle()
    x = synth.hidden(5, 1, 0, shape.H)
    a, ids, p = orc.token(x)
    b, ids2, p2 = orc.token(x, dense=True)
    assert np.array_equal(ids, ids2) and np.array_equal(p, p2)
    assert np.abs(a - b).max() <= 1e-12 * np.abs(b).max()


def test_identity_expert_layer():
    records, shared, rc, rsb = identity_layer()
    E, k, H = 8, 2, 64
    lay = oracle.Layer(H, E, k, H, H, {e: records[e] for e in range(E)}, shared, rc, rsb)
    xs = synth.hidden(3, 0, 0, H)
    xs[0] = synth.bf16_from_double(8.0)
    out, ids, p = lay.token(xs)
    x = synth.bf16_bits_to_float(xs).astype(np.float64)
    scale = 1.0 + sum(p[i] * 2.0 ** -(int(ids[i]) % 3) for i in range(k))
    np.testing.assert_allclose(out, scale * x, rtol=1e-15, atol=0)
    assert abs(p.sum() - 1.0) < 1e-12


# ---- 3-bit residual VQ ------------------------------------------------------------------

def _rvq_golden():
    cb = np.zeros((3, 256, 8), np.uint16)
    rows, expect = {}, {}
    for line in open(os.path.join(GOLDEN, "rvq_blocks.txt")):
        f = line.split("|")[0].split()
        if not f or f[0].startswith("#"):
            continue
        if f[0] == "cb":
            cb[int(f[1]) - 1, int(f[2])] = [int(h, 16) for h in f[3:11]]
        elif f[0] == "row":
            rows[int(f[1])] = [int(v) for v in f[3:]]
        elif f[0] == "expect":
            expect[int(f[1])] = [float(v) for v in f[2:]]
    codes = np.array([rows[r] for r in sorted(rows)], np.uint8)
    W = np.array([expect[r] for r in sorted(expect)], np.float64)
    return cb, codes, W


def test_rvq_hand_blocks():
    cb, codes, W = _rvq_golden()
    rows, cols = W.shape
    for r in range(rows):
        for j in range(cols):
            assert oracle.dequant_rvq(codes, cb, cols, r, j) == W[r, j], (r, j)
    for j in range(cols):                                     # unit inputs pick columns
        x = np.zeros(cols)
        x[j] = 1.0
        assert np.array_equal(oracle.gemv_rvq(codes, cb, rows, cols, x), W[:, j])
    x = np.linspace(-1, 1, cols)
    np.testing.assert_allclose(oracle.gemv_rvq(codes, cb, rows, cols, x), W @ x, rtol=1e-14)


def test_rvq_layout():
    for H, F in [(256, 128), (2048, 768), (7168, 2048), (64, 64)]:
        L = oracle.rvq_layout(H, F)
        assert L["up_codes"] == 3 * F * H // 8 and L["down_codes"] == 2 * L["up_codes"]
        assert L["bytes"] == 9 * F * H // 8 and L["stride"] % 4096 == 0
        assert L["stride"] == synth.rvq_record_stride(H, F)
    # 3 bits per weight: three code bytes per 8 weights of each matrix
    assert oracle.rvq_layout(7168, 2048)["bytes"] * 8 == 3 * 3 * 7168 * 2048


def test_rvq_identity_layer():
    records, shared, rc, rsb, cbs = identity_layer_rvq()
    E, k, H = 8, 2, 64
    lay = oracle.Layer(H, E, k, H, H, {e: records[e] for e in range(E)}, shared, rc, rsb,
                       codebooks=cbs)
    xs = synth.hidden(3, 0, 0, H)
    xs[0] = synth.bf16_from_double(8.0)
    out, ids, p = lay.token(xs)
    x = synth.bf16_bits_to_float(xs).astype(np.float64)
    scale = 1.0 + sum(p[i] * 2.0 ** -(int(ids[i]) % 3) for i in range(k))
    np.testing.assert_allclose(out, scale * x, rtol=1e-15, atol=0)


@pytest.mark.parametrize("shape", SMALL[:3], ids=lambda s: f"H{s.H}E{s.E}k{s.k}F{s.F}Fs{s.Fs}")
def test_rvq_layer_vs_torch_float64(shape):
    hl = HostLayerRVQ(shape, seed=2, beta=synth.beta_normal(2, 0, shape.E))
    orc = hl.oracle()
    for t in range(2):
        x = synth.hidden(2, 99, t, shape.H)
        out, ids, p = orc.token(x)
        ref, rids, rp = _torch_layer(hl, x)
        assert np.array_equal(ids, rids)
        np.testing.assert_allclose(p, rp, rtol=1e-12)
        assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()
        dense, _, _ = orc.token(x, dense=True)
        assert np.abs(out - dense).max() <= 1e-12 * np.abs(dense).max()


def test_missing_selected_record_raises():
    hl = HostLayer(synth.TINY, seed=0)
    s = synth.TINY
    lay = oracle.Layer(s.H, s.E, s.k, s.F, s.Fs, {}, hl.shared, hl.router_codes, hl.router_sb)
    with pytest.raises(KeyError):
        lay.token(synth.hidden(0, 0, 0, s.H))


def test_margin_redraw_meets_margin():
    hl = HostLayer(synth.TINY, seed=0)
    orc = hl.oracle()
    for t in range(4):
        x = hidden_with_margin(orc, 0, 0, t)
        logits, _, _ = orc.route(x)
        srt = np.sort(logits)[::-1]
        assert srt[1] - srt[2] >= 1e-3


# ---- record format -----------------------------------------------------------------

def test_record_layout_closed_form():
    # Large layer: H=7168, F=2048 -> 22,020,096 code bytes + 2,752,512 sb bytes.
    L = oracle.record_layout(7168, 2048)
    assert L["bytes"] == 24_772_608 and L["stride"] == 24_772_608
    assert L["up_codes"] == 2048 * 3584 and L["down_codes"] == 2 * 2048 * 3584
    assert L["gate_sb"] == 22_020_096 and L["down_sb"] - L["up_sb"] == 2048 * 112 * 4
    T = oracle.record_layout(256, 128)
    assert T["bytes"] == 55_296 and T["stride"] == 57_344
    for H, F in [(256, 128), (2048, 768), (7168, 2048), (64, 64)]:
        assert oracle.record_layout(H, F)["stride"] == synth.record_stride(H, F)
        assert synth.record_stride(H, F) % 4096 == 0


# ---- LFU policy ----------------------------------------------------------------------

def test_lfu_hand_trace():
    rows = [l.split("|") for l in open(os.path.join(GOLDEN, "lfu_trace.txt"))
            if l.strip() and not l.startswith("#")]
    lfu = oracle.LFU(3, 6)
    for r in rows:
        ids = np.array(r[1].split(), np.int32)
        hit, slot, m = lfu.step(ids)
        assert list(hit.astype(int)) == [int(t) for t in r[2].split()]
        assert list(slot) == [int(t) for t in r[3].split()]
        assert list(lfu.slot_expert) == [int(t) for t in r[4].split()]
        assert m == int((~hit).sum())


def test_lfu_invariants_random_stream():
    rng = np.random.default_rng(3)
    n_slots, E, k = 8, 40, 4
    lfu = oracle.LFU(n_slots, E)
    total_miss = 0
    for _ in range(300):
        ids = rng.choice(E, size=k, replace=False).astype(np.int32)
        before = set(int(e) for e in lfu.slot_expert if e >= 0)
        hit, slot, m = lfu.step(ids)
        after = list(lfu.slot_expert)
        for i, e in enumerate(ids):
            assert after[slot[i]] == e                         # every id resident
            assert hit[i] == (int(e) in before)
        assert len(set(e for e in after if e >= 0)) == sum(1 for e in after if e >= 0)
        total_miss += m
    assert lfu.count.sum() == 300 * k
    assert total_miss < 300 * k


def test_waves_hand_example():
    # 4 slots, top-2.  Worked by hand: {0,1} then {1,2} -> 3 experts; {3,4}
    # would make 5 -> new wave; {3,4} {4,5} {0,5} -> {0,3,4,5} = 4 fits; then
    # {1,2} makes 6 -> new wave.
    ids = np.array([[0, 1], [1, 2], [3, 4], [4, 5], [0, 5], [1, 2]])
    assert oracle.waves(ids, 4) == [(0, 2), (2, 5), (5, 6)]
    assert oracle.waves(ids, 6) == [(0, 6)]
    assert oracle.waves(ids, 2) == [(0, 1), (1, 2), (2, 3), (3, 4), (4, 5), (5, 6)]
    assert oracle.waves(ids[:0], 4) == []


def test_lfu_lookahead_hand_trace():
    rows = [[c.strip() for c in l.split("|")]
            for l in open(os.path.join(GOLDEN, "lfu_lookahead_trace.txt"))
            if l.strip() and not l.startswith("#")]
    lfu = oracle.LFU(3, 6)
    for r in rows:
        before = (lfu.hits, lfu.misses, lfu.lookahead_copies, lfu.lookahead_hits, lfu.evictions)
        counts = lfu.count.copy()
        if r[1] == "D":
            lfu.step(np.array(r[3].split(), np.int32))
        else:
            pred = np.array([t.split() for t in r[3].split(";")], np.int32)
            lfu.lookahead(pred, int(r[2]))
            assert np.array_equal(lfu.count, counts)          # no use counted
        after = (lfu.hits, lfu.misses, lfu.lookahead_copies, lfu.lookahead_hits, lfu.evictions)
        assert [a - b for a, b in zip(after, before)] == [int(t) for t in r[4:9]], f"row {r[0]}"
        assert list(lfu.slot_expert) == [int(t) for t in r[9].split()], f"row {r[0]}"


def test_lfu_lookahead_with_exact_predictions_moves_every_miss():
    """A lookahead told exactly the next step's ids (one token, n = k) pins the
    same experts the step pins and sees the same counts among the others, so
    it must choose the very victims the demand step would: the cache ends in
    the same state as without it, and every miss becomes a lookahead copy
    that the step then hits."""
    rng = np.random.default_rng(5)
    n_slots, E, k = 8, 40, 4
    plain, ahead = oracle.LFU(n_slots, E), oracle.LFU(n_slots, E)
    for _ in range(300):
        ids = rng.choice(E, size=k, replace=False).astype(np.int32)
        plain.step(ids)
        ahead.lookahead(ids[None], k)
        hit, _, m = ahead.step(ids)
        assert m == 0 and hit.all()
        assert list(ahead.slot_expert) == list(plain.slot_expert)
    assert ahead.lookahead_copies == plain.misses > 0
    assert ahead.lookahead_hits == ahead.lookahead_copies
    assert ahead.evictions == plain.evictions and ahead.misses == 0


def test_lfu_lookahead_invariants_random_stream():
    rng = np.random.default_rng(6)
    n_slots, E, k = 6, 30, 3
    lfu = oracle.LFU(n_slots, E)
    for it in range(400):
        if it % 2:
            B, n = int(rng.integers(1, 4)), int(rng.integers(0, k + 1))
            pred = np.stack([rng.choice(E, size=k, replace=False) for _ in range(B)]).astype(np.int32)
            counts, pinned0 = lfu.count.copy(), lfu.pinned.copy()
            slot, c, ev = lfu.lookahead(pred, n)
            order = pred[:, :n].T.reshape(-1)
            assert np.array_equal(lfu.count, counts)
            assert all(lfu.pinned[e] for e in order) and (lfu.pinned >= pinned0).all()
            for i, e in enumerate(order):
                if slot[i] >= 0:
                    assert lfu.slot_expert[slot[i]] == e       # resident where it says
                else:                                          # dropped: no slot was free
                    assert all(lfu.pinned[x] for x in lfu.slot_expert if x >= 0)
                    assert (lfu.slot_expert >= 0).all()
            assert ev <= c
        else:
            ids = rng.choice(E, size=k, replace=False).astype(np.int32)
            hit, slot, m = lfu.step(ids)
            assert not lfu.pinned.any()
            assert all(lfu.slot_expert[slot[i]] == e for i, e in enumerate(ids))
        live = [e for e in lfu.slot_expert if e >= 0]
        assert len(set(live)) == len(live)
        assert not any(lfu.fresh[e] for e in range(E) if e not in live)


# ---- generator --------------------------------------------------------------------------

def test_synth_bf16_rounding():
    assert synth.bf16_from_double(1.0) == 0x3F80
    assert synth.bf16_from_double(1.0 / 3.0) == 0x3EAB
    assert synth.bf16_from_double(1.0 + 2.0 ** -8) == 0x3F80     # tie -> even
    assert synth.bf16_from_double(1.0 + 3 * 2.0 ** -8) == 0x3F82  # tie -> even (up)
    assert synth.bf16_from_double(-0.75) == 0xBF40


def test_synth_hidden_chain():
    H = 4096
    ind = synth.hidden_chain(3, 5, H, 4, 0.0)
    for l in range(4):
        assert np.array_equal(ind[l], synth.hidden(3, l, 5, H))   # rho = 0: independent draws
    ch = synth.hidden_chain(3, 5, H, 4, 0.9)
    assert np.array_equal(ch[0], ind[0])
    xs = synth.bf16_bits_to_float(ch).astype(np.float64)
    for l in range(4):
        assert abs(xs[l].std() - 1.0) < 0.05
    for l in range(1, 4):
        assert abs(np.corrcoef(xs[l - 1], xs[l])[0, 1] - 0.9) < 0.02


def test_synth_rvq_records_and_codebooks():
    H, F = 256, 128
    stride = synth.rvq_record_stride(H, F)
    buf = np.zeros((3, stride), np.uint8)
    synth.fill_rvq_records(11, 2, [5, 0, 7], H, F, buf)
    assert np.array_equal(buf[2], synth.rvq_expert_record(11, 2, 7, H, F))   # random access
    assert not np.array_equal(buf[0], buf[1])
    payload = oracle.rvq_layout(H, F)["bytes"]
    assert not buf[0, payload:].any()                                        # zero padding
    counts = np.bincount(buf[0, :payload], minlength=256)
    assert counts.min() > 0.6 * payload / 256                                # uniform codes
    cb = synth.rvq_codebooks(11, 2)
    assert cb.shape == (3, 3, 256, 8) and np.array_equal(cb, synth.rvq_codebooks(11, 2))
    w = synth.bf16_bits_to_float(cb).astype(np.float64)
    for st, sd in enumerate(synth.RVQ_STAGE_SD):
        assert abs(w[:, st].std() - sd) < 0.1 * sd and abs(w[:, st].mean()) < 0.1 * sd
    assert not np.array_equal(cb[0], cb[1]) and not np.array_equal(cb, synth.rvq_codebooks(11, 3))


def test_synth_random_access_and_distributions():
    H, F = 256, 128
    buf = np.zeros((3, synth.record_stride(H, F)), np.uint8)
    synth.fill_records(11, 2, [5, 0, 7], H, F, buf)
    assert np.array_equal(buf[2], synth.expert_record(11, 2, 7, H, F))
    assert not np.array_equal(buf[0], buf[1])
    L = oracle.record_layout(H, F)
    q = np.concatenate([buf[0][:L["gate_sb"]] & 15, buf[0][:L["gate_sb"]] >> 4])
    counts = np.bincount(q, minlength=16)
    assert counts.min() > 0.8 * q.size / 16
    x = synth.bf16_bits_to_float(synth.hidden(1, 0, 0, 65536)).astype(np.float64)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    sb = buf[0][L["gate_sb"]:L["bytes"]].view(np.uint32)
    s = synth.bf16_bits_to_float((sb & 0xFFFF).astype(np.uint16))
    assert s.min() >= 0.0049 and s.max() <= 0.0201
