"""The workloads the decoder stack is exercised on: model shapes and sequence layouts.

Nothing here computes any part of the method; these are plain descriptions of the
model hyper-parameters (the ``text_config`` keys of the Compass checkpoint, see the
"Config (config.json)" and "Text decoder forward" sections of the mlxcel issue
"feat(vlm): add Cohere Compass / North-Micro-Vision (cohere_compass) VLM") and of
where the image spans sit in each synthetic sequence.

Five named workloads follow the five configurations the stack is specified on, plus
small shapes used by the parity tests (several tiles and a ragged tail, but cheap
enough for the fp64 oracle).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

SLIDING = "sliding_attention"
FULL = "full_attention"


@dataclass(frozen=True)
class ModelShape:
    num_layers: int
    hidden_size: int
    num_attention_heads: int
    num_key_value_heads: int
    head_dim: int
    intermediate_size: int
    vocab_size: int
    sliding_window: int
    mrope_section: Tuple[int, int, int]
    rope_theta: float
    layer_types: Tuple[str, ...]
    layer_norm_eps: float = 1e-5
    logit_scale: float = 0.0625
    dtype: str = "bf16"  # "bf16" or "f32": storage type of weights and activations
    mrope_layout: str = "interleaved"  # or "sections_hwt" (contiguous [H, W, T] sections)

    def __post_init__(self):
        assert len(self.layer_types) == self.num_layers
        assert sum(self.mrope_section) == self.head_dim // 2
        assert self.num_attention_heads % self.num_key_value_heads == 0


@dataclass(frozen=True)
class ImageSpan:
    """One image inside sequence ``seq``: merged grid (t, h, w) starting at token ``start``
    (offset within that sequence). It occupies t*h*w consecutive tokens."""
    seq: int
    start: int
    grid_t: int
    grid_h: int
    grid_w: int

    @property
    def n_tokens(self) -> int:
        return self.grid_t * self.grid_h * self.grid_w


@dataclass
class Workload:
    name: str
    shape: ModelShape
    mode: str                      # "prefill" or "decode"
    seq_lens: List[int]            # prefill: lengths of the packed sequences
    images: List[ImageSpan] = field(default_factory=list)
    n_deepstack: int = 0           # deepstack tensors, added after layers 0..n_deepstack-1
    head_rows: str = "last"        # "all" or "last" (last token of every sequence)
    seed: int = 0
    # decode only
    decode_batch: int = 0
    cache_len: int = 0
    page_size: int = 16

    @property
    def total_tokens(self) -> int:
        return self.decode_batch if self.mode == "decode" else sum(self.seq_lens)


def _pattern_3to1(n):
    # full attention at every 4th layer (i % 4 == 3), sliding elsewhere
    return tuple(FULL if i % 4 == 3 else SLIDING for i in range(n))


SHAPE_LAYER_FP32 = ModelShape(
    num_layers=1, hidden_size=256, num_attention_heads=4, num_key_value_heads=1,
    head_dim=64, intermediate_size=512, vocab_size=1024, sliding_window=32,
    mrope_section=(12, 10, 10), rope_theta=1e4, layer_types=(SLIDING,),
    layer_norm_eps=1e-5, logit_scale=0.0625, dtype="f32")

# the two-layer pair's per-layer shapes (also used by the 28-layer stack, the decode step
# and the varlen prefill); rope theta 50000 as in the real model.
_C2 = dict(hidden_size=2048, num_attention_heads=16, num_key_value_heads=4, head_dim=128,
           intermediate_size=8192, vocab_size=256000, mrope_section=(24, 20, 20),
           rope_theta=50000.0, layer_norm_eps=1e-5, logit_scale=0.0625, dtype="bf16")

SHAPE_PAIR = ModelShape(num_layers=2, sliding_window=512, layer_types=(SLIDING, FULL), **_C2)
SHAPE_STACK28 = ModelShape(num_layers=28, sliding_window=4096, layer_types=_pattern_3to1(28), **_C2)
SHAPE_PAIR_W4096 = ModelShape(num_layers=2, sliding_window=4096, layer_types=(SLIDING, FULL), **_C2)


def layer_fp32_T128() -> Workload:
    return Workload("layer_fp32_T128", SHAPE_LAYER_FP32, "prefill", [128],
                    images=[ImageSpan(0, 48, 1, 4, 4)], n_deepstack=1, head_rows="all", seed=1)


def pair_T2048() -> Workload:
    return Workload("pair_bf16_T2048", SHAPE_PAIR, "prefill", [2048],
                    images=[ImageSpan(0, 300, 1, 16, 16)], n_deepstack=1, head_rows="last", seed=2)


def stack28_T8192() -> Workload:
    # three 32x32 images interleaved with text at fixed offsets
    imgs = [ImageSpan(0, s, 1, 32, 32) for s in (1280, 3584, 5888)]
    return Workload("stack28_bf16_T8192", SHAPE_STACK28, "prefill", [8192],
                    images=imgs, n_deepstack=3, head_rows="last", seed=3)


def decode_B64_cache4096() -> Workload:
    return Workload("decode_B64_cache4096", SHAPE_PAIR_W4096, "decode", [],
                    n_deepstack=0, head_rows="all", seed=4,
                    decode_batch=64, cache_len=4096, page_size=16)


def varlen_images(seq_lens, seed=5) -> List[ImageSpan]:
    """Seeded image layout of the varlen workload: per sequence 1-4 square merged grids
    of side 24..48, separated by text gaps of at least 64 tokens."""
    import numpy as np
    out = []
    for s, L in enumerate(seq_lens):
        rng = np.random.default_rng((seed, 100 + s))
        while True:
            n = int(rng.integers(1, 5))
            g = [int(x) for x in rng.integers(24, 49, size=n)]
            if sum(x * x for x in g) <= L - 64 * (n + 1):
                break
        extra = L - sum(x * x for x in g) - 64 * (n + 1)
        cuts = np.sort(rng.integers(0, extra + 1, size=n))
        parts = np.diff(np.concatenate([[0], cuts, [extra]]))
        gaps = [64 + int(p) for p in parts]
        pos = 0
        for i in range(n):
            pos += gaps[i]
            out.append(ImageSpan(s, pos, 1, g[i], g[i]))
            pos += g[i] * g[i]
        assert pos + gaps[n] == L
    return out


def varlen_T32768() -> Workload:
    lens = [4096, 8192, 12288, 8192]
    # The 2-layer stack has no layer 2, so deepstack goes after layers 0 and 1 only.
    return Workload("varlen_bf16_T32768", SHAPE_PAIR_W4096, "prefill", lens,
                    images=varlen_images(lens), n_deepstack=2, head_rows="last", seed=5)


WORKLOADS = {"layer_fp32_T128": layer_fp32_T128, "pair_T2048": pair_T2048,
             "stack28_T8192": stack28_T8192, "decode_B64_cache4096": decode_B64_cache4096,
             "varlen_T32768": varlen_T32768}


def small_shape(num_layers=2, layer_types=None, window=64, dtype="bf16", hidden=256,
                heads=(4, 2), head_dim=128, inter=384, vocab=640, section=None,
                theta=50000.0, logit_scale=0.0625, mrope_layout="interleaved") -> ModelShape:
    """A reduced model for parity tests; head_dim stays 128 unless asked otherwise."""
    if layer_types is None:
        layer_types = tuple(FULL if i % 4 == 3 else SLIDING for i in range(num_layers))
    if section is None:
        half = head_dim // 2
        s1 = (half * 5) // 16
        section = (half - 2 * s1, s1, s1)
    return ModelShape(num_layers=num_layers, hidden_size=hidden, num_attention_heads=heads[0],
                      num_key_value_heads=heads[1], head_dim=head_dim, intermediate_size=inter,
                      vocab_size=vocab, sliding_window=window, mrope_section=tuple(section),
                      rope_theta=theta, layer_types=tuple(layer_types), dtype=dtype,
                      logit_scale=logit_scale, mrope_layout=mrope_layout)
