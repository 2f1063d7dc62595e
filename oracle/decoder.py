"""Plain, slow fp64 CPU oracle of the Compass-style parallel decoder stack.

TEST INFRASTRUCTURE ONLY. This module exists to check the CUDA path; only the test
suite, the package's smoke check and the bench's CPU-baseline leg may import it. It
shares no code, tables or helpers with the CUDA library, and nothing in it is tuned.

Every function follows the definition on the pages, cited by page and section:

  [Compass issue]   mlxcel issue "feat(vlm): add Cohere Compass / North-Micro-Vision
                    (cohere_compass) VLM" -- sections "Text decoder forward" (the block,
                    the attention of layer i, the interleaved MRoPE, the position ids),
                    "Validation" (the unit-test list) and "Acceptance criteria".
  [Kernel story]    C-Kernel-Engine "Cohere Kernel Story", section 1 (parallel block,
                    3:1 layer split, final_logit_scale footer) and section 3 (outputs
                    rounded to BF16 exactly where the contract says).
  [mlxcel VLM manual]  mlxcel user guide "Vision-Language Models", "Stage 4: Embedding
                    Merge".
  [FreeToken PR 454]   FreeToken pull request "feat(mm): serve image input on the Qwen
                    families", "How it fits together".

Arithmetic is float64 throughout. With ``mirror_bf16=True`` (bf16 workloads) values are
rounded to bf16 at exactly the points where the GPU path stores bf16 and nowhere else:
the LayerNorm outputs, q/k after rotation and v, the attention output and the SwiGLU
product (the residual stream and the logits stay unrounded).

Readings of points the pages leave open (window edge, GQA grouping, LayerNorm variance,
...) are stated in the docstrings where they are used.
"""
from __future__ import annotations

import numpy as np

SLIDING = "sliding_attention"
FULL = "full_attention"

_BF16_DROP = np.uint64(45)                      # 52 - 7 fraction bits dropped
_BF16_HALF = np.uint64((1 << 44) - 1)
_BF16_MASK = np.uint64(~((1 << 45) - 1) & 0xFFFFFFFFFFFFFFFF)


# ----------------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------------
def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned as float64.

    bf16 keeps 7 of float64's 52 fraction bits; the dropped 45 bits are rounded to
    nearest-even on the bit pattern. Inputs are finite and far from the bf16 subnormal
    range (|x| >= 2**-126 or 0), which holds for every tensor of the method.
    """
    a = np.ascontiguousarray(x, dtype=np.float64)
    b = a.view(np.uint64)
    lsb = (b >> _BF16_DROP) & np.uint64(1)
    r = (b + _BF16_HALF + lsb) & _BF16_MASK
    return r.view(np.float64)


def from_storage(x) -> np.ndarray:
    """uint16 bf16 bit patterns, or float32/float64 values, as float64."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


# ----------------------------------------------------------------------------------
# a0: position ids  ([Compass issue], "Position ids (get_rope_index)")
# ----------------------------------------------------------------------------------
def rope_index(seq_len: int, images):
    """(t, h, w) position ids of one sequence and its rope_delta.

    ``images`` holds (start, grid_t, grid_h, grid_w) per image, merged grid, start
    being the token offset inside the sequence. Text tokens take max(previous
    positions) + 1 on all three axes (0 for the first token). The t*h*w image tokens of
    an image, in row-major (t, h, w) order, take offset + (t_idx, h_idx, w_idx), where
    offset = max(previous positions) + 1. rope_delta = max position + 1 - seq_len.
    """
    pos = np.zeros((3, seq_len), dtype=np.int64)
    starts = {s: (t, h, w) for (s, t, h, w) in images}
    nxt = 0
    k = 0
    while k < seq_len:
        if k in starts:
            gt, gh, gw = starts[k]
            off = nxt
            for ti in range(gt):
                for hi in range(gh):
                    for wi in range(gw):
                        pos[:, k] = (off + ti, off + hi, off + wi)
                        k += 1
            nxt = int(pos[:, k - gt * gh * gw:k].max()) + 1
        else:
            pos[:, k] = nxt
            nxt += 1
            k += 1
    if seq_len == 0:          # no positions: rope_delta taken as 0 (max+1 - L with max = -1)
        return pos, 0
    return pos, int(pos.max()) + 1 - seq_len


def positions(seq_lens, images):
    """Packed positions [3, T] of several sequences (restarting at 0 for each) and the
    per-sequence rope deltas. ``images`` holds (seq, start, grid_t, grid_h, grid_w)."""
    cols, deltas = [], []
    for s, L in enumerate(seq_lens):
        ims = [(st, t, h, w) for (sq, st, t, h, w) in images if sq == s]
        p, dl = rope_index(L, ims)
        cols.append(p)
        deltas.append(dl)
    return np.concatenate(cols, axis=1), np.asarray(deltas, dtype=np.int64)


def decode_positions(seq_lens, rope_delta):
    """Decode token position: offset + rope_delta on all three axes, offset being the
    number of tokens already cached ([Compass issue], "Position ids")."""
    p = np.asarray(seq_lens, np.int64) + np.asarray(rope_delta, np.int64)
    return np.stack([p, p, p])


def image_token_count(grid_thw, merge=2):
    """Image-pad tokens of an image of patch grid (t, h, w): t * (h/merge) * (w/merge)."""
    t, h, w = grid_thw
    return t * (h // merge) * (w // merge)


# ----------------------------------------------------------------------------------
# a1 / a4: interleaved MRoPE and the split rotate-half ([Compass issue], "Text decoder
# forward": the interleaved MRoPE paragraph and the attention of layer i)
# ----------------------------------------------------------------------------------
def mrope_axis(half: int, section):
    """Axis of frequency j (0 = t, 1 = h, 2 = w): h when j % 3 == 1 and j < 3*section[1],
    w when j % 3 == 2 and j < 3*section[2], t otherwise."""
    ax = np.zeros(half, dtype=np.int64)
    for j in range(half):
        if j % 3 == 1 and j < 3 * section[1]:
            ax[j] = 1
        elif j % 3 == 2 and j < 3 * section[2]:
            ax[j] = 2
    return ax


def mrope_sections_hwt(half: int, section):
    """The contiguous-section layout ([Compass issue], "Acceptance criteria", the correction
    to the RoPE item: the checkpoint's rotary class pre-permutes inv_freq and gives the axes
    contiguous [H, W, T] sections). The pages name the layout but not the permutation. Reading
    (parity unpinned): the rotary index k runs first over the frequencies the interleaved rule
    sends to h, in increasing frequency index, then over those it sends to w, then over those
    it sends to t -- the same (axis, frequency) pairs as the interleaved layout, in contiguous
    sections of sizes section[1], section[2], section[0].
    Returns (axis[k], freq_index[k]) for k < half."""
    ax_int = mrope_axis(half, section)
    order = [j for a in (1, 2, 0) for j in range(half) if ax_int[j] == a]
    return ax_int[order], np.asarray(order, dtype=np.int64)


MROPE_LAYOUTS = ("interleaved", "sections_hwt")


def mrope_cos_sin(pos, head_dim: int, theta: float, section, layout: str = "interleaved"):
    """cos, sin of shape [T, head_dim]: inv_freq[j] = theta**(-2j/head_dim),
    freqs[:, k] = pos[axis(k)] * inv_freq[f(k)], then cos/sin of concat(freqs, freqs).
    layout "interleaved" (the contract): axis(k) = mrope_axis, f(k) = k; "sections_hwt":
    mrope_sections_hwt."""
    half = head_dim // 2
    j = np.arange(half, dtype=np.float64)
    inv_freq = float(theta) ** (-2.0 * j / head_dim)
    if layout == "interleaved":
        ax, fidx = mrope_axis(half, section), np.arange(half)
    elif layout == "sections_hwt":
        ax, fidx = mrope_sections_hwt(half, section)
    else:
        raise ValueError(f"unknown MRoPE layout {layout!r}")
    pos = np.asarray(pos, dtype=np.float64)
    freqs = np.empty((pos.shape[1], half), dtype=np.float64)
    for jj in range(half):
        freqs[:, jj] = pos[ax[jj]] * inv_freq[fidx[jj]]
    emb = np.concatenate([freqs, freqs], axis=1)
    return np.cos(emb), np.sin(emb)


def rotate_half_split(x):
    """concat(-x2, x1) over the two halves of the last axis (not pairwise)."""
    half = x.shape[-1] // 2
    return np.concatenate([-x[..., half:], x[..., :half]], axis=-1)


def apply_rope(x, cos, sin):
    """x * cos + rotate_half_split(x) * sin; x is [T, heads, d], cos/sin [T, d]."""
    return x * cos[:, None, :] + rotate_half_split(x) * sin[:, None, :]


# ----------------------------------------------------------------------------------
# the step before the path: embedding lookup and image-row merge ([Compass issue] "Text
# decoder forward": h = embed_tokens(tokens); [mlxcel VLM manual] "Stage 4: Embedding
# Merge": the projected image features take the rows of the image placeholder tokens;
# [FreeToken PR 454] "How it fits together", scheduler and engine: the rows arrive as a
# row list (mm_rows) with the gathered features (mm_embeds), merged by one index copy)
# ----------------------------------------------------------------------------------
def embed_merge(token_ids, embed, mm_rows=None, mm_embeds=None):
    """h[t] = embed[token_ids[t]] for every row, then h[mm_rows[r]] = mm_embeds[r].

    Reading: the row list names distinct rows (an index copy with a repeated row has no
    single result); a token id outside the vocabulary is an error.
    """
    token_ids = np.asarray(token_ids, dtype=np.int64)
    embed = np.asarray(embed, dtype=np.float64)
    if token_ids.size and (token_ids.min() < 0 or token_ids.max() >= embed.shape[0]):
        raise ValueError("token id outside the vocabulary")
    h = np.empty((token_ids.size, embed.shape[1]), dtype=np.float64)
    for t, tok in enumerate(token_ids):
        h[t] = embed[tok]
    if mm_rows is not None and len(mm_rows):
        mm_rows = np.asarray(mm_rows, dtype=np.int64)
        if len(set(mm_rows.tolist())) != mm_rows.size:
            raise ValueError("repeated image row")
        if mm_rows.min() < 0 or mm_rows.max() >= token_ids.size:
            raise ValueError("image row outside the sequence")
        feats = np.asarray(mm_embeds, dtype=np.float64)
        for r, row in enumerate(mm_rows):
            h[row] = feats[r]
    return h


# ----------------------------------------------------------------------------------
# 4-bit affine weights ([Compass issue] "Config (config.json)": quantization {group_size 64,
# bits 4, mode affine} in the mlx conversion that the reference checkpoint ships)
# ----------------------------------------------------------------------------------
def dequantize_affine(packed, scales, biases, group=64, bits=4):
    """w[n, k] = scales[n, k // group] * q[n, k] + biases[n, k // group].

    Readings: q[n, k] is the bits-wide field at bit offset bits * (k % (32 // bits)) of the
    32-bit word packed[n, k // (32 // bits)] (lowest bits first); scales and biases are the
    stored values (bf16 bit patterns or floats). The result is exact (float64).
    """
    packed = np.asarray(packed, dtype=np.uint32)
    per = 32 // bits
    N, W = packed.shape
    K = W * per
    q = np.empty((N, K), dtype=np.float64)
    mask = np.uint32((1 << bits) - 1)
    for i in range(per):
        q[:, i::per] = ((packed >> np.uint32(bits * i)) & mask).astype(np.float64)
    s = from_storage(scales)
    b = from_storage(biases)
    if s.shape != (N, K // group) or b.shape != (N, K // group):
        raise ValueError("scales / biases must hold one value per group of each row")
    return np.repeat(s, group, axis=1) * q + np.repeat(b, group, axis=1)


# ----------------------------------------------------------------------------------
# a2: LayerNorm ([Compass issue], "Text decoder forward": weight only, no bias)
# ----------------------------------------------------------------------------------
def layer_norm(x, gamma, eps):
    """gamma * (x - mean) / sqrt(var + eps) per row; var is the biased (1/n) variance."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * gamma


def silu(x):
    """x * sigmoid(x) = x / (1 + e^-x), the SwiGLU gate activation (reading: the block's
    "SwiGLU" is the usual silu-gated linear unit)."""
    return x / (1.0 + np.exp(-x))


def swiglu(a, wg, wu, wd, rb=lambda x: x):
    """The MLP branch of the block ([Compass issue] "Text decoder forward": mlp = SwiGLU(a)):
    down_proj(silu(gate_proj(a)) * up_proj(a)), with gate_proj = ``wg``, up_proj = ``wu``,
    down_proj = ``wd`` (output-major [out, in] matrices). ``rb`` rounds the gated product
    before down_proj (bf16 in the mirror mode, where the GPU stores it)."""
    act = rb(silu(a @ wg.T) * (a @ wu.T))
    return act @ wd.T


# ----------------------------------------------------------------------------------
# a5: causal / sliding-window GQA attention ([Compass issue], "Text decoder forward")
# ----------------------------------------------------------------------------------
def attention(q, k, v, cu_seqlens, window, scale, row_block=1024):
    """Softmax attention per packed sequence and per query head.

    q [T, nq, d], k/v [T, nkv, d]. Query head h reads KV head h // (nq // nkv).
    Key j is visible to query i (both within one sequence) iff j <= i and, for a
    sliding layer (window not None), i - j < window: the last ``window`` keys
    including the query's own. Scores are scaled by ``scale``; masked keys get -inf.
    Rows are evaluated ``row_block`` at a time; each row's softmax runs over all of
    that row's visible keys, so the blocking changes no row's definition.
    """
    T, nq, d = q.shape
    nkv = k.shape[1]
    group = nq // nkv
    out = np.zeros((T, nq, v.shape[2]), dtype=np.float64)
    cu = [int(c) for c in cu_seqlens]
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for r0 in range(a, b, row_block):
            r1 = min(b, r0 + row_block)
            k0 = a if window is None else max(a, r0 - window + 1)
            i = np.arange(r0, r1)[:, None]
            j = np.arange(k0, r1)[None, :]
            vis = j <= i
            if window is not None:
                vis &= (i - j) < window
            for h in range(nq):
                g = h // group
                S = (q[r0:r1, h, :] @ k[k0:r1, g, :].T) * scale
                S = np.where(vis, S, -np.inf)
                S = S - S.max(axis=1, keepdims=True)
                P = np.exp(S)
                P /= P.sum(axis=1, keepdims=True)
                out[r0:r1, h, :] = P @ v[k0:r1, g, :]
    return out


# ----------------------------------------------------------------------------------
# one parallel block ([Compass issue] "Text decoder forward"; [Kernel story] section 1)
# ----------------------------------------------------------------------------------
def _w(layer, key):
    return from_storage(layer[key])


def block(h, layer, layer_type, shape, cos_sin, cu_seqlens, mirror_bf16):
    """h + Attn(a) + SwiGLU(a) with a = LayerNorm(h): one shared norm, no post-norm.

    ``layer`` holds ln, wq, wk, wv, wo, wg, wu, wd (output-major [out, in] matrices);
    ``shape`` is a dict of the model hyper-parameters.
    """
    rb = round_bf16 if mirror_bf16 else (lambda x: x)
    T = h.shape[0]
    nq, nkv, d = shape["num_attention_heads"], shape["num_key_value_heads"], shape["head_dim"]
    a = rb(layer_norm(h, _w(layer, "ln"), shape["layer_norm_eps"]))
    q = (a @ _w(layer, "wq").T).reshape(T, nq, d)
    k = (a @ _w(layer, "wk").T).reshape(T, nkv, d)
    v = (a @ _w(layer, "wv").T).reshape(T, nkv, d)
    if layer_type == SLIDING:
        cos, sin = cos_sin
        q = apply_rope(q, cos, sin)
        k = apply_rope(k, cos, sin)
        window = shape["sliding_window"]
    else:
        window = None                       # full layers: no rotation, plain causal
    q, k, v = rb(q), rb(k), rb(v)
    o = rb(attention(q, k, v, cu_seqlens, window, d ** -0.5))
    attn = o.reshape(T, nq * d) @ _w(layer, "wo").T
    mlp = swiglu(a, _w(layer, "wg"), _w(layer, "wu"), _w(layer, "wd"), rb)
    return h + attn + mlp


def prefill(hidden, layers, shape, pos, cu_seqlens, ds_rows=None, ds=(), mirror_bf16=True,
            return_all=False):
    """The layer stack over packed sequences; returns the final residual stream h [T, H].

    After layer i < len(ds): h[ds_rows] += ds[i] ([Compass issue] "Text decoder forward":
    deepstack after layers 0, 1, 2 only). ``layers`` is a sequence (or a callable
    i -> layer dict), ``pos`` the [3, T] position ids.
    """
    h = np.array(hidden, dtype=np.float64)
    cos_sin = mrope_cos_sin(pos, shape["head_dim"], shape["rope_theta"], shape["mrope_section"],
                            shape["mrope_layout"])
    get = layers if callable(layers) else (lambda i: layers[i])
    hs = []
    for i in range(shape["num_layers"]):
        h = block(h, get(i), shape["layer_types"][i], shape, cos_sin, cu_seqlens, mirror_bf16)
        if i < len(ds):
            h[np.asarray(ds_rows)] += from_storage(ds[i])
        if return_all:
            hs.append(h.copy())
    return (h, hs) if return_all else h


def logits(h_rows, final_ln, embed, shape, mirror_bf16=True):
    """logit_scale * (LayerNorm(h) @ embed.T): the tied head with its scale footer."""
    rb = round_bf16 if mirror_bf16 else (lambda x: x)
    a = rb(layer_norm(h_rows, from_storage(final_ln), shape["layer_norm_eps"]))
    return (a @ from_storage(embed).T) * shape["logit_scale"]


# ----------------------------------------------------------------------------------
# a9: one decode step over a paged KV cache
# ----------------------------------------------------------------------------------
def gather_cache(pool, page_table_row, n_tokens, page_size):
    """Tokens 0..n_tokens-1 of one sequence from a [pages, nkv, page, d] pool."""
    idx = np.arange(n_tokens)
    pages = np.asarray(page_table_row)[idx // page_size]
    return from_storage(pool[pages, :, idx % page_size, :])        # [n, nkv, d]


def decode_attention(q, K, V, window, scale):
    """Attention of the newest of the L = K.shape[0] tokens of one sequence: q [nq, d] is
    query index L - 1, K and V [L, nkv, d] its keys and values in position order. Key j is
    visible iff (L - 1) - j < window (sliding layers) or always (full, window None); query head
    h reads KV head h // (nq // nkv) ([Compass issue] "Text decoder forward")."""
    L, nkv = K.shape[0], K.shape[1]
    nq = q.shape[0]
    lo = 0 if window is None else max(0, L - window)    # first key with (L - 1) - j < window
    out = np.zeros((nq, V.shape[2]))
    for hq in range(nq):
        g = hq // (nq // nkv)
        s = (K[lo:, g, :] @ q[hq, :]) * scale
        p = np.exp(s - s.max())
        out[hq] = (p / p.sum()) @ V[lo:, g, :]
    return out


def decode_step(hidden, layers, shape, seq_lens, rope_delta, page_table, kv, page_size,
                mirror_bf16=True):
    """One new token per sequence. ``kv(i)`` returns layer i's (K, V) pools holding
    post-rotation keys. Sequence b attends over its seq_lens[b] cached tokens plus the new
    one (query index i = seq_lens[b]); sliding layers see only keys with i - j < window.
    The pools are read, never written: the new K/V are appended to gathered copies."""
    rb = round_bf16 if mirror_bf16 else (lambda x: x)
    h = np.array(hidden, dtype=np.float64)
    B = h.shape[0]
    nq, nkv, d = shape["num_attention_heads"], shape["num_key_value_heads"], shape["head_dim"]
    pos = decode_positions(seq_lens, rope_delta)
    cos, sin = mrope_cos_sin(pos, d, shape["rope_theta"], shape["mrope_section"],
                             shape["mrope_layout"])
    get = layers if callable(layers) else (lambda i: layers[i])
    for li in range(shape["num_layers"]):
        layer = get(li)
        a = rb(layer_norm(h, _w(layer, "ln"), shape["layer_norm_eps"]))
        q = (a @ _w(layer, "wq").T).reshape(B, nq, d)
        k = (a @ _w(layer, "wk").T).reshape(B, nkv, d)
        v = (a @ _w(layer, "wv").T).reshape(B, nkv, d)
        sliding = shape["layer_types"][li] == SLIDING
        if sliding:
            q = apply_rope(q, cos, sin)
            k = apply_rope(k, cos, sin)
        q, k, v = rb(q), rb(k), rb(v)
        kpool, vpool = kv(li)
        win = shape["sliding_window"] if sliding else None
        o = np.zeros((B, nq, d))
        for b in range(B):
            n = int(seq_lens[b])                 # the new token is query index n
            K = np.concatenate([gather_cache(kpool, page_table[b], n, page_size), k[b:b + 1]])
            V = np.concatenate([gather_cache(vpool, page_table[b], n, page_size), v[b:b + 1]])
            o[b] = decode_attention(q[b], K, V, win, d ** -0.5)
        o = rb(o)
        attn = o.reshape(B, nq * d) @ _w(layer, "wo").T
        h = h + attn + swiglu(a, _w(layer, "wg"), _w(layer, "wu"), _w(layer, "wd"), rb)
    return h


def shape_dict(shape) -> dict:
    """Model hyper-parameters as a plain dict (accepts any object with those attributes)."""
    keys = ["num_layers", "hidden_size", "num_attention_heads", "num_key_value_heads",
            "head_dim", "intermediate_size", "vocab_size", "sliding_window", "mrope_section",
            "rope_theta", "layer_types", "layer_norm_eps", "logit_scale"]
    get = (lambda k, d=None: shape.get(k, d)) if isinstance(shape, dict) else \
        (lambda k, d=None: getattr(shape, k, d))
    out = {k: get(k) for k in keys}
    out["mrope_layout"] = get("mrope_layout", "interleaved")
    return out


__all__ = [n for n in dir() if not n.startswith("_") and n != "np"]
