"""Writes streamed_lfu_counts.txt: the expert-cache counters the oracle's
fp64 router and LFU replay give for the streamed workload that bench.py
times (4 large layers, H=7168, E=512, top-16, 64 slots per layer, Zipf(1.1)
router offsets, 256 single-token steps from a cold cache).

Three runs, as in the benchmark: hidden states drawn independently per step
and layer with no lookahead; hidden states chained across layers (rho 0.9)
without and with the router lookahead (layer l+1's router on layer l's
hidden state, its first 6 experts read ahead).  Calls only the oracle and
the seeded input generators.  About two minutes on one core:

    python tests/golden/make_streamed_lfu_counts.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from quantized_routed_expert_gemv_gb300 import synth  # noqa: E402

SLOTS, STEPS, RHO, N_AHEAD = 64, 256, 0.9, 6
KEYS = ("hits", "misses", "evictions", "lookahead_copies", "lookahead_hits")


def replay(layers, inputs, ahead):
    nl = len(layers)
    caches = [oracle.LFU(SLOTS, layers[0].E) for _ in range(nl)]
    for t in range(STEPS):
        xs = inputs(t)
        for l in range(nl):
            if ahead and l > 0:
                caches[l].lookahead(layers[l].route(xs[l - 1])[1][None], N_AHEAD)
            caches[l].step(layers[l].route(xs[l])[1])
    return [[getattr(c, k) for k in KEYS] for c in caches]


def main():
    wl = synth.WORKLOADS["large-streamed"]
    s, nl = wl.shape, wl.layers
    layers = []
    for l in range(nl):
        rc, rsb = synth.router(wl.weight_seed, l, s.E, s.H)
        layers.append(oracle.Layer(s.H, s.E, s.k, s.F, s.Fs, {}, None, rc, rsb, synth.beta_for(wl, l)))
    chain = {}

    def chained(t):
        if t not in chain:
            chain.clear()
            chain[t] = synth.hidden_chain(wl.input_seed, t, s.H, nl, RHO)
        return chain[t]

    runs = {
        "independent": replay(layers, lambda t: [synth.hidden(wl.input_seed, l, t, s.H) for l in range(nl)],
                              False),
        "chained_off": replay(layers, chained, False),
        "chained_on": replay(layers, chained, True),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "streamed_lfu_counts.txt")
    with open(path, "w") as f:
        f.write("# Expert-cache counters of the streamed workload from the oracle's fp64 router\n"
                "# and LFU replay (written by make_streamed_lfu_counts.py; see its docstring).\n"
                f"# slots {SLOTS}, steps {STEPS}, rho {RHO}, n_ahead {N_AHEAD}\n"
                "# run | layer | " + " | ".join(KEYS) + "\n")
        for name, rows in runs.items():
            for l, row in enumerate(rows):
                f.write(f"{name} | {l} | " + " | ".join(str(v) for v in row) + "\n")
    print(open(path).read())


if __name__ == "__main__":
    main()
