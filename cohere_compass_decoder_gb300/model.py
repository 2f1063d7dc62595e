"""Device-side owner of one decoder stack: uploads and packs the weights, holds the plan.

Memory management and argument marshalling around the C-ABI; every step of the forward
runs in the library's kernels (see include/cc.h).
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib as L


def to_device(arr: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 arrays are bf16 bit patterns; float32 stays float32; int32 stays int32."""
    if arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


class DecoderStack:
    """Weights of every layer packed on the device plus a cc_layer_plan.

    ``layer(i)`` returns the checkpoint matrices of layer i (ln, wq, wk, wv, wo, wg, wu, wd)
    as numpy arrays (uint16 bf16 bits or float32)."""

    def __init__(self, shape, layer, final_ln, embed, max_tokens, page_size=16, device="cuda"):
        self.shape = shape
        self.device = device
        self.cfg = L.make_config(shape, max_tokens, page_size)
        self.bf16 = shape.dtype == "bf16"
        H, d, I = shape.hidden_size, shape.head_dim, shape.intermediate_size
        nq, nkv = shape.num_attention_heads, shape.num_key_value_heads
        self.N1 = (nq + 2 * nkv) * d + 2 * I
        self.K2 = nq * d + I
        dt = torch.bfloat16 if self.bf16 else torch.float32
        self.ln, self.w1, self.w2 = [], [], []
        for i in range(shape.num_layers):
            w = layer(i)
            dev = {k: to_device(v, device) for k, v in w.items()}
            w1 = torch.empty(self.N1, H, dtype=dt, device=device)
            w2 = torch.empty(H, self.K2, dtype=dt, device=device)
            L.cc_pack_layer_weights(self.cfg, dev["wq"], dev["wk"], dev["wv"], dev["wo"], dev["wg"],
                                    dev["wu"], dev["wd"], w1, w2)
            torch.cuda.current_stream().synchronize()
            self.ln.append(dev["ln"])
            self.w1.append(w1)
            self.w2.append(w2)
            del dev
        self.final_ln = to_device(final_ln, device)
        self.embed = to_device(embed, device)
        self.plan = L.cc_layer_plan_create(self.cfg, list(zip(self.ln, self.w1, self.w2)),
                                           self.final_ln, self.embed)

    def attach_q4(self, layer_q4, embed_q4):
        """Uploads and tiles the 4-bit affine weights (``layer_q4(i)``: ln and a (words,
        scales, biases) triple per matrix; ``embed_q4`` one triple) for decode_q4/logits_q4."""
        H = self.shape.hidden_size
        u32 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(self.device)
        tiled = lambda rows, k: torch.empty(L.cc_q4_tiled_bytes(rows, k), dtype=torch.uint8,
                                            device=self.device)
        names = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")
        self.q4 = []
        for i in range(self.shape.num_layers):
            w = layer_q4(i)
            words = [u32(w[k][0]) for k in names]
            scales = [to_device(w[k][1], self.device) for k in names]
            biases = [to_device(w[k][2], self.device) for k in names]
            w1 = tiled(self.N1, H)
            w2 = tiled(H, self.K2)
            L.cc_pack_layer_weights_q4(self.cfg, words, scales, biases, w1, w2)
            torch.cuda.current_stream().synchronize()
            self.q4.append((to_device(w["ln"], self.device), w1, w2))
        ew, es, eb = embed_q4
        V = ew.shape[0]
        self.embed_q4 = tiled(V, H)
        L.cc_pack_q4_tiles(u32(ew), to_device(es, self.device), to_device(eb, self.device), V, H,
                           self.embed_q4)
        torch.cuda.current_stream().synchronize()
        L.cc_layer_plan_attach_q4(self.plan, self.q4, self.embed_q4)

    def decode_q4(self, hidden, pos, seq_lens, page_table, max_pages, kv, stream=None):
        L.cc_decode_step_q4(self.plan, hidden, pos, seq_lens, page_table, max_pages,
                            hidden.shape[0], kv, stream)

    def logits_q4(self, hidden, rows, n_rows, out, stream=None):
        L.cc_logits_q4(self.plan, hidden, rows, n_rows, out, stream)

    def prefill(self, hidden, pos, cu_seqlens, n_seqs, ds_rows=None, ds_feats=(), kv=None,
                page_table=None, max_pages=0, stream=None):
        n_ds_rows = 0 if ds_rows is None else int(ds_rows.numel())
        L.cc_prefill_forward(self.plan, hidden, pos, cu_seqlens, n_seqs, hidden.shape[0], ds_rows,
                             n_ds_rows, list(ds_feats), kv, page_table, max_pages, stream)

    def prefill_tokens(self, token_ids, mm_rows, mm_embeds, hidden, pos, cu_seqlens, n_seqs,
                       ds_rows=None, ds_feats=(), kv=None, page_table=None, max_pages=0,
                       stream=None):
        n_mm = 0 if mm_rows is None else int(mm_rows.numel())
        n_ds_rows = 0 if ds_rows is None else int(ds_rows.numel())
        L.cc_prefill_forward_tokens(self.plan, token_ids, mm_rows, mm_embeds, n_mm, hidden, pos,
                                    cu_seqlens, n_seqs, hidden.shape[0], ds_rows, n_ds_rows,
                                    list(ds_feats), kv, page_table, max_pages, stream)

    def decode(self, hidden, pos, seq_lens, page_table, max_pages, kv, stream=None):
        L.cc_decode_step(self.plan, hidden, pos, seq_lens, page_table, max_pages, hidden.shape[0],
                         kv, stream)

    def logits(self, hidden, rows, n_rows, out, stream=None):
        L.cc_logits(self.plan, hidden, rows, n_rows, out, stream)

    def sync(self, stream=None):
        L.cc_sync(self.plan, stream)

    def close(self):
        if self.plan:
            L.cc_layer_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
