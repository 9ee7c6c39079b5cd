"""The oracle's pins catch plausible mistakes.

Each case copies oracle.c, plants one mistake by replacing one exact piece
of its text (a swapped nibble order, a dropped bias, a tie going the wrong
way, a sign error, gate and up exchanged, ...), builds the copy with the
oracle's own compiler flags, binds the oracle wrapper to it and runs the
pins that should notice.  At least one of them must fail: a pin that passes
on both the oracle and a broken copy pins nothing.  The oracle itself is
never changed; everything happens on the CPU in a temporary directory.
"""
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle as pins
from quantized_routed_expert_gemv_gb300 import synth

HAND4 = [b for b in pins._golden_blocks() if b["bits"] == 4][0]
HAND8 = [b for b in pins._golden_blocks() if b["bits"] == 8][0]

# (name, text in oracle.c, replacement, pins that must notice: (function, args))
MUTANTS = [
    ("4-bit nibble order swapped",
     "int q = (j % 2 == 0) ? (byte & 0x0F) : (byte >> 4);",
     "int q = (j % 2 == 0) ? (byte >> 4) : (byte & 0x0F);",
     [(pins.test_dequant_hand_blocks, (HAND4,)), (pins.test_gemv_orientation_single_weight, ())]),
    ("4-bit bias subtracted",
     "    return s * (double)q + b;\n}\n\n/* Weight (r, j) of the 8-bit router",
     "    return s * (double)q - b;\n}\n\n/* Weight (r, j) of the 8-bit router",
     [(pins.test_dequant_hand_blocks, (HAND4,)), (pins.test_gemv_bias_term, ())]),
    ("router (8-bit) bias dropped",
     "    return s * (double)q + b;\n}\n\n/* y[r] = sum_j",
     "    return s * (double)q;\n}\n\n/* y[r] = sum_j",
     [(pins.test_dequant_hand_blocks, (HAND8,)), (pins.test_router_logits_vs_numpy_dense, ())]),
    ("GEMV input reversed",
     "acc += orc_dequant4(codes, sb, cols, r, j) * x[j];",
     "acc += orc_dequant4(codes, sb, cols, r, j) * x[cols - 1 - j];",
     [(pins.test_gemv_orientation_single_weight, ())]),
    ("router ignores the logit offset",
     "logits[e] = acc + (beta ? (double)beta[e] : 0.0);",
     "logits[e] = acc;",
     [(pins.test_layer_vs_torch_float64, (synth.TINY,))]),
    ("top-k ties go to the higher id",
     "if (best < 0 || logits[e] > logits[best])",
     "if (best < 0 || logits[e] >= logits[best])",
     [(pins.test_topk_ties_go_to_lower_id, ())]),
    ("weights not renormalised",
     "p[i] = exp(logits[ids[i]] - lmax) / z;",
     "p[i] = exp(logits[ids[i]] - lmax);",
     [(pins.test_topk_against_library, (8, 2))]),
    ("SiLU sign error",
     "double orc_silu(double z) { return z / (1.0 + exp(-z)); }",
     "double orc_silu(double z) { return z / (1.0 + exp(z)); }",
     [(pins.test_silu_closed_forms, ())]),
    ("gate and up exchanged",
     "    orc_gemv4(rec + L.up_codes, rec + L.up_sb, F, H, x, u);\n    for (int j = 0; j < F; ++j)\n"
     "        h[j] = orc_silu(g[j]) * u[j];",
     "    orc_gemv4(rec + L.up_codes, rec + L.up_sb, F, H, x, u);\n    for (int j = 0; j < F; ++j)\n"
     "        h[j] = orc_silu(u[j]) * g[j];",
     [(pins.test_identity_expert_layer, ()), (pins.test_layer_vs_torch_float64, (synth.TINY,))]),
    ("shared expert weighted like a routed one",
     "            out[r] = y[r];",
     "            out[r] = p[0] * y[r];",
     [(pins.test_identity_expert_layer, ())]),
    ("residual-VQ stages read from the wrong codebook",
     "cb[((size_t)s * 256 + blk[s]) * 8 + (size_t)(j % 8)]",
     "cb[((size_t)(2 - s) * 256 + blk[s]) * 8 + (size_t)(j % 8)]",
     [(pins.test_rvq_hand_blocks, ())]),
    ("residual-VQ block taken from the element index",
     "(size_t)(j / 8) * 3;",
     "(size_t)(j % 8 % (cols / 8)) * 3;",
     [(pins.test_rvq_hand_blocks, ())]),
    ("residual-VQ elements of a codeword reversed",
     "cb[((size_t)s * 256 + blk[s]) * 8 + (size_t)(j % 8)]",
     "cb[((size_t)s * 256 + blk[s]) * 8 + (size_t)(7 - j % 8)]",
     [(pins.test_rvq_hand_blocks, ()), (pins.test_rvq_identity_layer, ())]),
    ("LFU ties go to the higher id",
     "(last_use[e] == last_use[v] && e < v))))",
     "(last_use[e] == last_use[v] && e > v))))",
     [(pins.test_lfu_hand_trace, ())]),
    ("LFU counts not cumulative",
     "        count[ids[i]] += 1;",
     "        count[ids[i]] = 1;",
     [(pins.test_lfu_hand_trace, ())]),
    ("LFU ignores recency",
     "(count[e] == count[v] &&\n                     (last_use[e] < last_use[v] ||",
     "(count[e] == count[v] &&\n                     (last_use[e] > last_use[v] ||",
     [(pins.test_lfu_hand_trace, ())]),
    ("lookahead ties go to the higher id",
     "(last_use[r] == last_use[v] && r < v))))",
     "(last_use[r] == last_use[v] && r > v))))",
     [(pins.test_lfu_lookahead_hand_trace, ())]),
    ("lookahead does not pin resident predictions",
     "        if (where >= 0) {\n            slot[i] = where;",
     "        if (where >= 0) {\n            pinned[e] = 0;\n            slot[i] = where;",
     [(pins.test_lfu_lookahead_hand_trace, ()), (pins.test_lfu_lookahead_invariants_random_stream, ())]),
]


@pytest.fixture(scope="module")
def src():
    with open(oracle._SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(src, tmp_path, name, old, new, checks):
    assert src.count(old) == 1, f"the text to replace must occur once in oracle.c ({name})"
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", *oracle.GCC_FLAGS, str(mutant), "-o", str(so), "-lm"])
    caught = []
    with oracle.using_library(str(so)):
        for fn, args in checks:
            try:
                fn(*args)
            except (AssertionError, ValueError, KeyError):
                caught.append(fn.__name__)
    assert caught, f"no pin noticed: {name}"


def test_unmodified_copy_passes_every_listed_pin(src, tmp_path):
    """The harness itself: the same copy-build-bind route with nothing
    planted passes all the pins the mutants use."""
    c = tmp_path / "oracle_copy.c"
    c.write_text(src)
    so = tmp_path / "liboracle_copy.so"
    subprocess.check_call(["gcc", *oracle.GCC_FLAGS, str(c), "-o", str(so), "-lm"])
    seen = set()
    with oracle.using_library(str(so)):
        for _, _, _, checks in MUTANTS:
            for fn, args in checks:
                key = (fn.__name__, repr(args)[:40])
                if key not in seen:
                    seen.add(key)
                    fn(*args)
    assert np.isfinite(oracle.silu(1.0))
