"""Writes stack28_T8192_mirror_drift.txt: how far the oracle's own bf16-mirror result of the
28-layer T = 8192 workload moves when its input moves by one rounding unit.

    python tests/golden/make_stack28_drift.py        # fp64 NumPy only; tens of minutes

Calls only the oracle (and the seeded input generator). The mirror rounds to bf16 at every
storage point of the contract (LayerNorm outputs, q/k/v, the attention output, the SwiGLU
product), so a difference smaller than one bf16 rounding anywhere upstream flips some of those
roundings, and the flips then travel through the residual stream of all later layers. Two
faithful implementations of the contract therefore differ after 28 layers by at least what
the mirror differs from itself under the smallest perturbation of its input. The script
measures that, layer by layer, for two perturbations of the input hidden state (every element
moved by one unit in the last place, in a seeded random direction):

  fp32_ulp   one float32 ulp: the storage precision of the residual stream on the GPU;
  bf16_ulp   one bf16 ulp: the precision of the stored activations.

For each it records the max-abs and mean-abs difference of the final hidden state and of the
logits (and their ratio to the largest logit), and the mean-abs difference after every layer.
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import decoder as O          # noqa: E402
from synth import Inputs                 # noqa: E402
from synth.configs import stack28_T8192  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "stack28_T8192_mirror_drift.txt")


def nudge(x, ulp_bits, seed):
    """x moved by one unit in the last place of a format with `ulp_bits` fraction bits
    (23: float32, 7: bf16), up or down by a seeded coin, per element."""
    x = np.asarray(x, np.float64)
    rng = np.random.default_rng(seed)
    sign = np.where(rng.random(x.shape) < 0.5, -1.0, 1.0)
    e = np.floor(np.log2(np.abs(np.where(x == 0, 1.0, x))))
    return x + sign * np.exp2(e - ulp_bits)


def run(inp, hidden):
    wl = inp.wl
    shape = O.shape_dict(inp.shape)
    pos, _ = O.positions(wl.seq_lens, [(i.seq, i.start, i.grid_t, i.grid_h, i.grid_w)
                                       for i in wl.images])
    ds = [inp.ds(i) for i in range(wl.n_deepstack)]
    h, hs = O.prefill(hidden, inp.layer, shape, pos, inp.cu_seqlens, inp.ds_rows, ds, True,
                      return_all=True)
    lg = O.logits(h[inp.head_rows], inp.final_ln, inp.embed, shape, True)
    return hs, lg


def main():
    t0 = time.time()
    inp = Inputs(stack28_T8192())
    base_h, base_lg = run(inp, inp.hidden)
    print(f"base run {time.time() - t0:.0f} s", flush=True)
    lines = []
    for name, bits, seed in (("fp32_ulp", 23, 101), ("bf16_ulp", 7, 102)):
        t1 = time.time()
        hs, lg = run(inp, nudge(inp.hidden, bits, seed))
        d = np.abs(hs[-1] - base_h[-1])
        dl = np.abs(lg - base_lg)
        per_layer = [float(np.abs(a - b).mean()) for a, b in zip(hs, base_h)]
        lines += [
            f"{name}_hidden_max: {d.max():.6g}",
            f"{name}_hidden_mean: {d.mean():.6g}",
            f"{name}_logits_max: {dl.max():.6g}",
            f"{name}_logits_mean: {dl.mean():.6g}",
            f"{name}_logits_rel: {dl.max() / np.abs(base_lg).max():.6g}",
            f"{name}_hidden_mean_per_layer: " + ", ".join(f"{x:.4g}" for x in per_layer),
        ]
        print(f"{name}: hidden max {d.max():.4g} mean {d.mean():.4g}, logits max "
              f"{dl.max():.4g} ({time.time() - t1:.0f} s)", flush=True)
        del hs
    head = [
        "# The oracle's bf16-mirror result of the 28-layer T = 8192 workload (stack28_T8192:",
        "# 28 layers 3:1 sliding:full, three 32x32 images, deepstack after layers 0-2, head on",
        "# the last token) against the same mirror run on an input hidden state moved by one",
        "# float32 ulp (fp32_ulp) or one bf16 ulp (bf16_ulp) per element, seeded direction.",
        "# max / mean: absolute differences of the final hidden state and of the logits;",
        "# logits_rel: max-abs logit difference over the largest |logit|.",
        "# Written by: python tests/golden/make_stack28_drift.py (calls only oracle/ and synth/).",
    ]
    with open(OUT, "w") as f:
        f.write("\n".join(head + lines) + "\n")
    print(f"wrote {OUT} in {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main()
