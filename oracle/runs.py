"""Runs the oracle over a whole workload. TEST INFRASTRUCTURE ONLY (see oracle/__init__).

``inp`` is any object with the fields of synth.Inputs; positions are computed here by
the oracle's own rule, never taken from the CUDA path.
"""
from __future__ import annotations

import numpy as np

from . import decoder as O


def run_prefill(inp, mirror_bf16=None, return_all=False, hidden=None):
    """Final residual stream h [T, H] and logits of the head rows, both float64 (``hidden``:
    the stack's input instead of the workload's hidden states)."""
    wl = inp.wl
    shape = O.shape_dict(inp.shape)
    if mirror_bf16 is None:
        mirror_bf16 = inp.shape.dtype == "bf16"
    spans = [(i.seq, i.start, i.grid_t, i.grid_h, i.grid_w) for i in inp.images]
    pos, _ = O.positions(wl.seq_lens, spans)
    ds = [inp.ds(i) for i in range(wl.n_deepstack)]
    out = O.prefill(inp.hidden if hidden is None else hidden, inp.layer, shape, pos,
                    inp.cu_seqlens, inp.ds_rows, ds,
                    mirror_bf16, return_all=return_all)
    h, hs = (out if return_all else (out, None))
    logits = O.logits(h[inp.head_rows], inp.final_ln, inp.embed, shape, mirror_bf16)
    return (h, logits, hs) if return_all else (h, logits)


def run_decode(inp, mirror_bf16=True):
    shape = O.shape_dict(inp.shape)
    h = O.decode_step(inp.hidden, inp.layer, shape, inp.seq_lens, inp.rope_delta, inp.page_table,
                      inp.kv, inp.wl.page_size, mirror_bf16)
    logits = O.logits(h[inp.head_rows], inp.final_ln, inp.embed, shape, mirror_bf16)
    return h, logits


def run(inp, mirror_bf16=None):
    if inp.wl.mode == "decode":
        return run_decode(inp, True if mirror_bf16 is None else mirror_bf16)
    return run_prefill(inp, mirror_bf16)


def dequantized_q4(triple):
    """A 4-bit affine matrix as the GPU path multiplies it: dequantised exactly, then rounded
    to bf16 (the reading of the mlx affine weights in a bf16 tensor-core product)."""
    return O.round_bf16(O.dequantize_affine(*triple))


def run_decode_q4(inp, mirror_bf16=True):
    """run_decode with the workload's 4-bit affine layers and embedding (inp.layer_q4,
    inp.embed_q4) in place of the bf16 ones."""
    shape = O.shape_dict(inp.shape)

    def layer(i):
        q = inp.layer_q4(i)
        out = {"ln": q["ln"]}
        for key in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
            out[key] = dequantized_q4(q[key])
        return out

    h = O.decode_step(inp.hidden, layer, shape, inp.seq_lens, inp.rope_delta, inp.page_table,
                      inp.kv, inp.wl.page_size, mirror_bf16)
    embed = dequantized_q4(inp.embed_q4)
    logits = O.logits(h[inp.head_rows], inp.final_ln, embed, shape, mirror_bf16)
    return h, logits
