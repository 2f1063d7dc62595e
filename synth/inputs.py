"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This module draws random numbers and lays them out; it holds none of the decoder's
arithmetic. Weights are N(0, 0.02), LayerNorm gains 1 + N(0, 0.02), hidden inputs
N(0, 1), deepstack features N(0, 0.1) and, for the decode workload, the cached K/V
N(0, 1). For bf16 workloads every drawn value is rounded (round-to-nearest-even) to
bf16 once, here, and stored as raw bf16 bit patterns (uint16); hidden states are
handed over as float32 holding those bf16 values.

Layer ``i``'s tensors come from their own generator seeded by (seed, 1, i), so a
layer can be regenerated without drawing the layers before it.
"""
from __future__ import annotations

import numpy as np

from .configs import Workload, ModelShape, ImageSpan


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even) and return the uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _draw(rng, shape, std, mean=0.0, bf16=True):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    x *= np.float32(std)
    if mean:
        x += np.float32(mean)
    return f32_to_bf16_bits(x) if bf16 else x


class Inputs:
    """All tensors of one workload, drawn lazily and cached.

    Storage conventions (row-major numpy arrays):
      hidden      float32 [T, H]
      layer(i)    dict: ln [H]; wq [nq*d, H]; wk, wv [nkv*d, H]; wo [H, nq*d];
                  wg, wu [I, H]; wd [H, I]   (uint16 bf16 bits, or float32 for f32 shapes)
      final_ln    [H]; embed [V, H]
      ds_rows     int32 [R]  token rows of all image tokens, in token order
      ds(i)       [R, H]     deepstack tensor added after layer i
      cu_seqlens  int32 [B+1]; head_rows int32 [N]
    decode only:
      kv(i)       (K, V) each [n_pages, nkv, page, d] bf16 bits: the cache of layer i
      page_table  int32 [B, max_pages]; seq_lens int32 [B]; rope_delta int32 [B]
    """

    def __init__(self, wl: Workload):
        self.wl = wl
        self.shape: ModelShape = wl.shape
        self.bf16 = wl.shape.dtype == "bf16"
        self._layers = {}
        self._ds = {}
        self._kv = {}
        self._misc = None

    # ---- sequence structure -------------------------------------------------------
    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.wl.seq_lens)]).astype(np.int32)

    @property
    def images(self):
        return list(self.wl.images)

    @property
    def ds_rows(self) -> np.ndarray:
        cu = self.cu_seqlens
        rows = []
        for im in sorted(self.wl.images, key=lambda s: (s.seq, s.start)):
            base = int(cu[im.seq]) + im.start
            rows.extend(range(base, base + im.n_tokens))
        return np.asarray(rows, dtype=np.int32)

    @property
    def head_rows(self) -> np.ndarray:
        if self.wl.head_rows == "all":
            return np.arange(self.wl.total_tokens, dtype=np.int32)
        if self.wl.mode == "decode":
            return np.arange(self.wl.decode_batch, dtype=np.int32)
        return (self.cu_seqlens[1:] - 1).astype(np.int32)

    # ---- tensors ---------------------------------------------------------------------
    def _misc_draw(self):
        if self._misc is None:
            s = self.shape
            rng = np.random.default_rng((self.wl.seed, 0))
            T = self.wl.total_tokens
            hid = rng.standard_normal(size=(T, s.hidden_size), dtype=np.float32)
            if self.bf16:
                hid = bf16_bits_to_f32(f32_to_bf16_bits(hid))
            final_ln = _draw(rng, (s.hidden_size,), 0.02, 1.0, self.bf16)
            self._misc = dict(hidden=hid, final_ln=final_ln)
        return self._misc

    @property
    def hidden(self) -> np.ndarray:
        return self._misc_draw()["hidden"]

    @property
    def final_ln(self) -> np.ndarray:
        return self._misc_draw()["final_ln"]

    @property
    def embed(self) -> np.ndarray:
        if "embed" not in self._ds:
            s = self.shape
            rng = np.random.default_rng((self.wl.seed, 2))
            self._ds["embed"] = _draw(rng, (s.vocab_size, s.hidden_size), 0.02, 0.0, self.bf16)
        return self._ds["embed"]

    def layer(self, i: int) -> dict:
        if i not in self._layers:
            s = self.shape
            rng = np.random.default_rng((self.wl.seed, 1, i))
            H, d, I = s.hidden_size, s.head_dim, s.intermediate_size
            nq, nkv = s.num_attention_heads, s.num_key_value_heads
            w = {}
            w["ln"] = _draw(rng, (H,), 0.02, 1.0, self.bf16)
            w["wq"] = _draw(rng, (nq * d, H), 0.02, 0.0, self.bf16)
            w["wk"] = _draw(rng, (nkv * d, H), 0.02, 0.0, self.bf16)
            w["wv"] = _draw(rng, (nkv * d, H), 0.02, 0.0, self.bf16)
            w["wo"] = _draw(rng, (H, nq * d), 0.02, 0.0, self.bf16)
            w["wg"] = _draw(rng, (I, H), 0.02, 0.0, self.bf16)
            w["wu"] = _draw(rng, (I, H), 0.02, 0.0, self.bf16)
            w["wd"] = _draw(rng, (H, I), 0.02, 0.0, self.bf16)
            self._layers[i] = w
        return self._layers[i]

    def ds(self, i: int) -> np.ndarray:
        assert i < self.wl.n_deepstack
        key = ("ds", i)
        if key not in self._ds:
            rng = np.random.default_rng((self.wl.seed, 3, i))
            R = len(self.ds_rows)
            self._ds[key] = _draw(rng, (R, self.shape.hidden_size), 0.1, 0.0, self.bf16)
        return self._ds[key]

    # ---- 4-bit affine weights (the mlx conversion's storage form) ------------------------
    def _affine_q4(self, rng, rows, cols):
        """(words uint32 [rows, cols / 8], scales, biases bf16 bits [rows, cols / 64]).
        Words are uniform 32-bit values, so every 4-bit field is uniform on 0..15; scales
        are (0.02 / 4.6) * U(0.5, 1.5) and biases -7.5 * scale + N(0, 0.002), so a weight
        spreads about as widely as the N(0, 0.02) bf16 weights."""
        words = rng.integers(0, 1 << 32, size=(rows, cols // 8), dtype=np.uint64).astype(np.uint32)
        sc = (np.float32(0.02 / 4.6) * rng.uniform(0.5, 1.5, size=(rows, cols // 64))).astype(np.float32)
        sc_bits = f32_to_bf16_bits(sc)
        bias = np.float32(-7.5) * bf16_bits_to_f32(sc_bits) + _draw(rng, sc.shape, 0.002, 0.0, False)
        return words, sc_bits, f32_to_bf16_bits(bias)

    def layer_q4(self, i: int) -> dict:
        """Layer i in 4-bit affine form, group 64: ln [H] (bf16 bits, as layer(i)) and, for
        each of wq, wk, wv, wo, wg, wu, wd, a (words, scales, biases) triple of the same
        [out, in] matrix shape. Drawn from their own generator (seed, 9, i)."""
        key = ("q4", i)
        if key not in self._ds:
            s = self.shape
            rng = np.random.default_rng((self.wl.seed, 9, i))
            H, d, I = s.hidden_size, s.head_dim, s.intermediate_size
            nq, nkv = s.num_attention_heads, s.num_key_value_heads
            w = {"ln": self.layer(i)["ln"]}
            for name, (r, c) in (("wq", (nq * d, H)), ("wk", (nkv * d, H)), ("wv", (nkv * d, H)),
                                 ("wo", (H, nq * d)), ("wg", (I, H)), ("wu", (I, H)),
                                 ("wd", (H, I))):
                w[name] = self._affine_q4(rng, r, c)
            self._ds[key] = w
        return self._ds[key]

    @property
    def embed_q4(self):
        """The tied embedding [V, H] in 4-bit affine form (seed, 10)."""
        if "embed_q4" not in self._ds:
            s = self.shape
            rng = np.random.default_rng((self.wl.seed, 10))
            self._ds["embed_q4"] = self._affine_q4(rng, s.vocab_size, s.hidden_size)
        return self._ds["embed_q4"]

    # ---- token-id input (the embedding merge before the path) ----------------------------
    @property
    def token_ids(self) -> np.ndarray:
        """int32 [T], uniform over the vocabulary (placeholder ids at image rows are
        irrelevant: those rows take the image features)."""
        if "tok" not in self._ds:
            rng = np.random.default_rng((self.wl.seed, 7))
            self._ds["tok"] = rng.integers(0, self.shape.vocab_size, size=self.wl.total_tokens,
                                           dtype=np.int64).astype(np.int32)
        return self._ds["tok"]

    @property
    def mm_rows(self) -> np.ndarray:
        """The image rows (those of every image span), in order."""
        return self.ds_rows

    @property
    def mm_embeds(self) -> np.ndarray:
        """Projected vision features of the image rows, N(0, 1) (bf16 workloads: bf16)."""
        if "mm" not in self._ds:
            rng = np.random.default_rng((self.wl.seed, 8))
            self._ds["mm"] = _draw(rng, (len(self.mm_rows), self.shape.hidden_size), 1.0, 0.0,
                                   self.bf16)
        return self._ds["mm"]

    # ---- decode state ------------------------------------------------------------------
    @property
    def max_pages(self) -> int:
        wl = self.wl
        return (wl.cache_len + 1 + wl.page_size - 1) // wl.page_size

    @property
    def n_pages(self) -> int:
        return self.wl.decode_batch * self.max_pages

    @property
    def page_table(self) -> np.ndarray:
        rng = np.random.default_rng((self.wl.seed, 4))
        perm = rng.permutation(self.n_pages).astype(np.int32)
        return perm.reshape(self.wl.decode_batch, self.max_pages)

    @property
    def seq_lens(self) -> np.ndarray:
        return np.full(self.wl.decode_batch, self.wl.cache_len, dtype=np.int32)

    @property
    def rope_delta(self) -> np.ndarray:
        # per-sequence rope delta left over from the (image-bearing) prefill: <= 0
        rng = np.random.default_rng((self.wl.seed, 5))
        return rng.integers(-self.wl.cache_len // 2, 1, size=self.wl.decode_batch).astype(np.int32)

    def kv(self, i: int):
        if i not in self._kv:
            s = self.shape
            rng = np.random.default_rng((self.wl.seed, 6, i))
            shp = (self.n_pages, s.num_key_value_heads, self.wl.page_size, s.head_dim)
            k = _draw(rng, shp, 1.0, 0.0, True)
            v = _draw(rng, shp, 1.0, 0.0, True)
            self._kv[i] = (k, v)
        return self._kv[i]
