"""Puts one workload's host arrays on the device and drives the C-ABI over it.

``inp`` is any object with the fields of synth.Inputs (hidden, layer(i), final_ln, embed,
images, cu_seqlens, ds_rows, ds(i), head_rows and, for decode, kv(i), page_table,
seq_lens, rope_delta). Position ids come from the library's own host helpers.
Marshalling only: no step of the decoder is computed here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib as L
from .model import DecoderStack, to_device


class GpuWorkload:
    def __init__(self, inp, device="cuda", max_tokens=None, stack=None):
        self.inp = inp
        wl = inp.wl
        self.wl = wl
        self.shape = inp.shape
        self.device = device
        T = wl.total_tokens
        self.T = T
        self.stack = stack or DecoderStack(self.shape, inp.layer, inp.final_ln, inp.embed,
                                           max_tokens or max(T, 1), page_size=wl.page_size,
                                           device=device)
        self.hidden0 = to_device(inp.hidden, device)
        self.head_rows = to_device(inp.head_rows, device)
        if wl.mode == "prefill":
            spans = [(i.seq, i.start, i.grid_t, i.grid_h, i.grid_w) for i in inp.images]
            pos, self.rope_delta = L.cc_build_mrope_positions(spans, wl.seq_lens)
            self.pos = torch.tensor(pos, dtype=torch.int32, device=device)
            self.cu = to_device(inp.cu_seqlens, device)
            self.n_seqs = len(wl.seq_lens)
            self.n_ds = wl.n_deepstack
            self.ds_rows = to_device(inp.ds_rows, device) if self.n_ds else None
            self.ds_feats = [to_device(inp.ds(i), device) for i in range(self.n_ds)]
        else:
            pos = L.cc_build_decode_positions(inp.seq_lens.tolist(), inp.rope_delta.tolist())
            self.pos = torch.tensor(pos, dtype=torch.int32, device=device)
            self.seq_lens = to_device(inp.seq_lens, device)
            self.page_table = to_device(inp.page_table, device)
            self.max_pages = inp.max_pages
            self.kpools, self.vpools = [], []
            for i in range(self.shape.num_layers):
                k, v = inp.kv(i)
                self.kpools.append(to_device(k, device))
                self.vpools.append(to_device(v, device))
            self.kv = L.make_kv_pool(self.kpools, self.vpools, inp.n_pages)

    def fresh_hidden(self):
        return self.hidden0.clone()

    def prefill(self, hidden, stream=None, kv=None, page_table=None, max_pages=0):
        self.stack.prefill(hidden, self.pos, self.cu, self.n_seqs, self.ds_rows, self.ds_feats,
                           kv=kv, page_table=page_table, max_pages=max_pages, stream=stream)
        return hidden

    def decode(self, hidden, stream=None):
        self.stack.decode(hidden, self.pos, self.seq_lens, self.page_table, self.max_pages, self.kv,
                          stream=stream)
        return hidden

    def logits(self, hidden, out=None, stream=None):
        n = int(self.head_rows.numel())
        if out is None:
            out = torch.empty(n, self.shape.vocab_size, dtype=torch.float32, device=self.device)
        self.stack.logits(hidden, self.head_rows, n, out, stream=stream)
        return out

    def step(self, hidden, logits_out=None, stream=None):
        """One whole pass of the path: the layer stack (prefill or decode) and the head."""
        if self.wl.mode == "prefill":
            self.prefill(hidden, stream)
        else:
            self.decode(hidden, stream)
        return self.logits(hidden, logits_out, stream)

    def sync(self):
        self.stack.sync()

    def close(self):
        self.stack.close()


def as_numpy(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)
