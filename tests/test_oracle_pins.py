"""Pins of the fp64 oracle against what the pages and the mathematics fix (no GPU).

Each test ties one part of the oracle to something other than itself: a worked example
printed on the pages (``tests/golden``), a closed form, a textbook formulation written
differently (complex rotation for RoPE, per-element Python loops for attention), a
library routine (torch's bf16 cast) or an invariant the pages state (parallel block
without post-norm, logits linear in logit_scale, deepstack on the first layers only,
causal prefix, decode equals the last prefill row).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import decoder as O
from synth import Inputs, Workload, ImageSpan, small_shape, SLIDING, FULL
from synth.configs import SHAPE_STACK28, layer_fp32_T128, varlen_T32768

from conftest import read_golden


def sd(shape):
    return O.shape_dict(shape)


# ----------------------------------------------------------------------------- bf16
def test_round_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    # add exact ties: bf16 value + half an ulp
    b = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    ulp = np.abs(b) * 2.0 ** -7
    ties = (b + 0.5 * ulp).astype(np.float32)
    for arr in (x, ties):
        want = torch.from_numpy(arr).to(torch.bfloat16).double().numpy()
        got = O.round_bf16(arr.astype(np.float64))
        assert np.array_equal(got, want)


def test_round_bf16_single_rounding_from_float64():
    # ties go to even; a value just above a tie rounds up even where a detour through
    # float32 would have created a tie
    assert O.round_bf16(1 + 2.0 ** -8) == 1.0
    assert O.round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    assert O.round_bf16(1 + 2.0 ** -8 + 2.0 ** -30) == 1 + 2.0 ** -7
    assert O.round_bf16(-(1 + 2.0 ** -8 + 2.0 ** -30)) == -(1 + 2.0 ** -7)
    assert O.round_bf16(0.0) == 0.0


# ----------------------------------------------------------------------------- MRoPE
def test_interleaved_selector_matches_page():
    g = read_golden("mrope_selector_section_24_20_20.txt")
    ax = O.mrope_axis(64, (24, 20, 20))
    assert sorted(np.nonzero(ax == 1)[0].tolist()) == g["h"]
    assert sorted(np.nonzero(ax == 2)[0].tolist()) == g["w"]
    assert sorted(np.nonzero(ax == 0)[0].tolist()) == g["t"]


@pytest.mark.parametrize("section", [(24, 20, 20), (12, 10, 10), (16, 8, 8)])
def test_selector_counts_match_section(section):
    ax = O.mrope_axis(sum(section), section)
    assert [(ax == a).sum() for a in range(3)] == list(section)


def test_split_rotate_half_matches_page():
    g = read_golden("rotate_half_split.txt")
    q = np.asarray(g["q"], dtype=np.float64)[None, None, :]
    cos = np.full((1, 4), float(g["cos"][0]))
    sin = np.full((1, 4), float(g["sin"][0]))
    out = O.apply_rope(q, cos, sin)[0, 0]
    assert out.tolist() == g["expected"]
    assert out.tolist() != g["not_expected"]


def test_mrope_with_equal_axes_is_1d_rope():
    """t = h = w reduces the interleaved MRoPE to plain 1-D rotary embedding (split
    halves), here written as a complex rotation of (x_j + i x_{j+d/2})."""
    rng = np.random.default_rng(1)
    d, theta, T = 128, 50000.0, 37
    p = rng.integers(0, 40000, size=T)
    pos = np.stack([p, p, p])
    cos, sin = O.mrope_cos_sin(pos, d, theta, (24, 20, 20))
    x = rng.standard_normal((T, 3, d))
    got = O.apply_rope(x, cos, sin)
    half = d // 2
    z = x[..., :half] + 1j * x[..., half:]
    ang = p[:, None] * np.exp(-np.log(theta) * 2 * np.arange(half) / d)[None, :]
    zr = z * np.exp(1j * ang)[:, None, :]
    want = np.concatenate([zr.real, zr.imag], axis=-1)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-9)


def test_mrope_reads_the_selected_axis():
    # positions differ per axis; frequency j must rotate by pos[axis(j)] * theta^(-2j/d)
    g = read_golden("mrope_selector_section_24_20_20.txt")
    pos = np.array([[7], [1000], [123456]])
    cos, sin = O.mrope_cos_sin(pos, 128, 50000.0, (24, 20, 20))
    for axis, name in enumerate("thw"):
        for j in g[name]:
            ang = pos[axis, 0] * 50000.0 ** (-j / 64.0)
            assert math.isclose(cos[0, j], math.cos(ang), abs_tol=1e-9)
            assert math.isclose(sin[0, j + 64], math.sin(ang), abs_tol=1e-9)


def test_sections_layout_is_contiguous_hwt():
    """The corrected layout's structure ([Compass issue] "Acceptance criteria": contiguous
    [H, W, T] sections): the first section[1] rotary indices read h, the next section[2] w,
    the remaining section[0] t."""
    for section in [(24, 20, 20), (12, 10, 10), (16, 8, 8)]:
        half = sum(section)
        ax, _ = O.mrope_sections_hwt(half, section)
        want = [1] * section[1] + [2] * section[2] + [0] * section[0]
        assert ax.tolist() == want


def test_sections_layout_reads_the_page_frequencies_per_axis():
    """Reading of the pre-permuted inv_freq: each section takes, in increasing order, the
    frequency indices the page's interleaved rule gives to its axis (the page's lists)."""
    g = read_golden("mrope_selector_section_24_20_20.txt")
    ax, fidx = O.mrope_sections_hwt(64, (24, 20, 20))
    assert fidx.tolist() == g["h"] + g["w"] + g["t"]
    pos = np.array([[7], [1000], [123456]])
    cos, sin = O.mrope_cos_sin(pos, 128, 50000.0, (24, 20, 20), "sections_hwt")
    k = 0
    for axis, name in [(1, "h"), (2, "w"), (0, "t")]:
        for j in g[name]:
            ang = pos[axis, 0] * 50000.0 ** (-j / 64.0)
            assert math.isclose(cos[0, k], math.cos(ang), abs_tol=1e-9)
            assert math.isclose(sin[0, k + 64], math.sin(ang), abs_tol=1e-9)
            k += 1
    assert k == 64


def test_sections_layout_is_a_permutation_of_the_interleaved_pairs():
    """Both layouts rotate by the same (axis, frequency) pairs: on any positions the columns of
    one cos/sin table are a permutation of the other's."""
    rng = np.random.default_rng(4)
    pos = rng.integers(0, 9000, size=(3, 23))
    ci, si = O.mrope_cos_sin(pos, 128, 50000.0, (24, 20, 20))
    cs, ss = O.mrope_cos_sin(pos, 128, 50000.0, (24, 20, 20), "sections_hwt")
    _, fidx = O.mrope_sections_hwt(64, (24, 20, 20))
    np.testing.assert_array_equal(cs[:, :64], ci[:, fidx])
    np.testing.assert_array_equal(ss[:, 64:], si[:, 64 + fidx])
    assert not np.allclose(cs, ci)


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(2)
    pos = rng.integers(0, 5000, size=(3, 50))
    cos, sin = O.mrope_cos_sin(pos, 64, 1e4, (12, 10, 10))
    x = rng.standard_normal((50, 2, 64))
    y = O.apply_rope(x, cos, sin)
    n0 = x[..., :32] ** 2 + x[..., 32:] ** 2
    n1 = y[..., :32] ** 2 + y[..., 32:] ** 2
    np.testing.assert_allclose(n0, n1, rtol=1e-12)


# ----------------------------------------------------------------------------- positions
def test_positions_closed_form_single_layer_workload():
    wl = layer_fp32_T128()
    pos, delta = O.positions(wl.seq_lens, [(i.seq, i.start, i.grid_t, i.grid_h, i.grid_w)
                                           for i in wl.images])
    want = np.zeros((3, 128), dtype=np.int64)
    want[:, :48] = np.arange(48)
    for r in range(4):
        for c in range(4):
            want[:, 48 + 4 * r + c] = (48, 48 + r, 48 + c)
    want[:, 64:] = np.arange(52, 116)
    assert np.array_equal(pos, want)
    assert delta.tolist() == [-12]


def test_positions_hand_worked_two_images():
    # 2 text, a 2x3 image (offset 2), 2 text, a 1x2 image, 1 text
    L = 13
    pos, delta = O.rope_index(L, [(2, 1, 2, 3), (10, 1, 1, 2)])
    t = [0, 1, 2, 2, 2, 2, 2, 2, 5, 6, 7, 7, 9]
    h = [0, 1, 2, 2, 2, 3, 3, 3, 5, 6, 7, 7, 9]
    w = [0, 1, 2, 3, 4, 2, 3, 4, 5, 6, 7, 8, 9]
    assert pos.tolist() == [t, h, w]
    assert delta == 9 + 1 - 13


def test_image_pad_token_count_matches_page():
    g = read_golden("image_pad_tokens.txt")
    assert O.image_token_count(tuple(g["grid_thw"])) == g["tokens"][0]


def test_decode_positions_add_rope_delta():
    p = O.decode_positions([4096, 10], [-12, 0])
    assert p.tolist() == [[4084, 10]] * 3


def test_layer_pattern_matches_page():
    g = read_golden("layer_pattern_28.txt")
    full = [i for i, t in enumerate(SHAPE_STACK28.layer_types) if t == FULL]
    assert full == g["full"]


def test_varlen_layout_is_valid():
    wl = varlen_T32768()
    for s, L in enumerate(wl.seq_lens):
        ims = sorted([i for i in wl.images if i.seq == s], key=lambda i: i.start)
        assert 1 <= len(ims) <= 4
        prev_end = 0
        for im in ims:
            assert 24 <= im.grid_h <= 48 and im.grid_h == im.grid_w
            assert im.start - prev_end >= 64
            prev_end = im.start + im.n_tokens
        assert L - prev_end >= 64


# ----------------------------------------------------------------------------- LayerNorm
def test_layer_norm_closed_form():
    # rows [-1, 1]: mean 0, biased variance 1 -> x / sqrt(1 + eps)
    eps = 1e-5
    x = np.array([[-1.0, 1.0], [3.0, 5.0]])
    got = O.layer_norm(x, np.array([1.0, 2.0]), eps)
    s = 1.0 / math.sqrt(1.0 + eps)
    np.testing.assert_allclose(got, [[-s, 2 * s], [-s, 2 * s]], rtol=1e-15)


def test_layer_norm_moments_and_affine_invariance():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((16, 300)) * 4 + 2
    y = O.layer_norm(x, np.ones(300), 0.0)
    np.testing.assert_allclose(y.mean(axis=1), 0, atol=1e-12)
    np.testing.assert_allclose((y ** 2).mean(axis=1), 1, atol=1e-12)
    np.testing.assert_allclose(O.layer_norm(7 * x - 3, np.ones(300), 0.0), y, atol=1e-12)


# ----------------------------------------------------------------------------- attention
def _rand_qkv(rng, T, nq, nkv, d):
    return (rng.standard_normal((T, nq, d)), rng.standard_normal((T, nkv, d)),
            rng.standard_normal((T, nkv, d)))


@pytest.mark.parametrize("window", [None, 1, 5, 16])
def test_attention_zero_query_is_mean_of_visible_values(window):
    rng = np.random.default_rng(4)
    T, d = 40, 8
    q = np.zeros((T, 2, d))
    _, k, v = _rand_qkv(rng, T, 2, 1, d)
    out = O.attention(q, k, v, [0, T], window, 0.3)
    for i in range(T):
        lo = 0 if window is None else max(0, i - window + 1)
        np.testing.assert_allclose(out[i, 0], v[lo:i + 1, 0].mean(axis=0), atol=1e-12)


def test_attention_first_row_is_first_value():
    rng = np.random.default_rng(5)
    q, k, v = _rand_qkv(rng, 9, 4, 2, 16)
    out = O.attention(q, k, v, [0, 9], 3, 0.25)
    np.testing.assert_allclose(out[0, 0], v[0, 0], atol=1e-14)
    np.testing.assert_allclose(out[0, 3], v[0, 1], atol=1e-14)


@pytest.mark.parametrize("window", [None, 4])
def test_attention_matches_elementwise_loops(window):
    rng = np.random.default_rng(6)
    T, nq, nkv, d = 11, 4, 2, 5
    q, k, v = _rand_qkv(rng, T, nq, nkv, d)
    scale = d ** -0.5
    out = O.attention(q, k, v, [0, 6, 11], window, scale)
    for s0, s1 in ((0, 6), (6, 11)):
        for i in range(s0, s1):
            for h in range(nq):
                g = h // (nq // nkv)
                js = [j for j in range(s0, i + 1) if window is None or i - j < window]
                sc = [sum(q[i, h, c] * k[j, g, c] for c in range(d)) * scale for j in js]
                m = max(sc)
                e = [math.exp(x - m) for x in sc]
                z = sum(e)
                for c in range(d):
                    want = sum(e[n] * v[js[n], g, c] for n in range(len(js))) / z
                    assert abs(out[i, h, c] - want) < 1e-12



def test_attention_row_blocking_changes_nothing():
    """The oracle evaluates query rows in blocks whose key range starts at the block's first
    row minus the window; any block size gives every row the same visible keys."""
    rng = np.random.default_rng(10)
    q, k, v = _rand_qkv(rng, 45, 4, 2, 8)
    for window in (None, 1, 6, 20):
        a = O.attention(q, k, v, [0, 19, 45], window, 0.3, row_block=1024)
        for rb in (1, 4, 7):
            b = O.attention(q, k, v, [0, 19, 45], window, 0.3, row_block=rb)
            np.testing.assert_allclose(a, b, atol=1e-14)

def test_window_at_least_sequence_equals_full_causal():
    rng = np.random.default_rng(7)
    q, k, v = _rand_qkv(rng, 70, 4, 1, 16)
    full = O.attention(q, k, v, [0, 70], None, 0.25)
    np.testing.assert_array_equal(O.attention(q, k, v, [0, 70], 70, 0.25), full)
    np.testing.assert_array_equal(O.attention(q, k, v, [0, 70], 1000, 0.25), full)


def test_gqa_equals_mha_with_repeated_kv():
    rng = np.random.default_rng(8)
    q, k, v = _rand_qkv(rng, 30, 6, 2, 8)
    g = O.attention(q, k, v, [0, 30], 7, 0.3)
    m = O.attention(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), [0, 30], 7, 0.3)
    np.testing.assert_allclose(g, m, atol=1e-14)


def test_varlen_packed_equals_separate():
    rng = np.random.default_rng(9)
    q, k, v = _rand_qkv(rng, 50, 4, 2, 8)
    packed = O.attention(q, k, v, [0, 17, 50], 9, 0.3)
    a = O.attention(q[:17], k[:17], v[:17], [0, 17], 9, 0.3)
    b = O.attention(q[17:], k[17:], v[17:], [0, 33], 9, 0.3)
    np.testing.assert_allclose(packed, np.concatenate([a, b]), atol=1e-14)


# ----------------------------------------------------------------------------- blocks
def _tiny(num_layers=1, types=None, T=24, window=8, n_ds=0, images=()):
    shape = small_shape(num_layers=num_layers, layer_types=types, window=window, hidden=64,
                        heads=(4, 2), head_dim=16, inter=48, vocab=50)
    wl = Workload("tiny", shape, "prefill", [T], images=list(images), n_deepstack=n_ds,
                  head_rows="all", seed=11)
    inp = Inputs(wl)
    pos, _ = O.positions(wl.seq_lens, [(i.seq, i.start, i.grid_t, i.grid_h, i.grid_w)
                                       for i in wl.images])
    return shape, inp, pos


def _zeroed(layer, keys):
    out = dict(layer)
    for k in keys:
        out[k] = np.zeros_like(layer[k])
    return out


def test_parallel_block_has_no_post_norm():
    shape, inp, pos = _tiny(types=(SLIDING,), images=[ImageSpan(0, 5, 1, 2, 3)])
    s = sd(shape)
    cs = O.mrope_cos_sin(pos, s["head_dim"], s["rope_theta"], s["mrope_section"])
    h = inp.hidden.astype(np.float64)
    L = inp.layer(0)
    both = O.block(h, L, SLIDING, s, cs, [0, 24], False)
    attn_only = O.block(h, _zeroed(L, ["wg", "wu", "wd"]), SLIDING, s, cs, [0, 24], False)
    mlp_only = O.block(h, _zeroed(L, ["wo"]), SLIDING, s, cs, [0, 24], False)
    np.testing.assert_allclose(both - h, (attn_only - h) + (mlp_only - h), atol=1e-12)
    # zero o_proj and down_proj leave h unchanged
    same = O.block(h, _zeroed(L, ["wo", "wd"]), SLIDING, s, cs, [0, 24], False)
    np.testing.assert_array_equal(same, h)
    # all-zero MLP weights: h + o_proj(attention(q, k, v)) from the same normed input
    a = O.layer_norm(h, O.from_storage(L["ln"]), s["layer_norm_eps"])
    q = (a @ O.from_storage(L["wq"]).T).reshape(24, 4, 16)
    k = (a @ O.from_storage(L["wk"]).T).reshape(24, 2, 16)
    v = (a @ O.from_storage(L["wv"]).T).reshape(24, 2, 16)
    q, k = O.apply_rope(q, *cs), O.apply_rope(k, *cs)
    o = O.attention(q, k, v, [0, 24], 8, 0.25)
    want = h + o.reshape(24, 64) @ O.from_storage(L["wo"]).T
    np.testing.assert_allclose(attn_only, want, atol=1e-12)


def test_full_layers_ignore_positions():
    shape, inp, pos = _tiny(types=(FULL,))
    s = sd(shape)
    h = inp.hidden.astype(np.float64)
    a = O.prefill(h, [inp.layer(0)], s, pos, [0, 24], mirror_bf16=False)
    b = O.prefill(h, [inp.layer(0)], s, pos * 7 + 3, [0, 24], mirror_bf16=False)
    np.testing.assert_array_equal(a, b)
    shape2, inp2, _ = _tiny(types=(SLIDING,))
    c = O.prefill(h, [inp2.layer(0)], sd(shape2), pos, [0, 24], mirror_bf16=False)
    e = O.prefill(h, [inp2.layer(0)], sd(shape2), pos * 7 + 3, [0, 24], mirror_bf16=False)
    assert np.abs(c - e).max() > 1e-6


def test_deepstack_first_layers_only():
    img = [ImageSpan(0, 4, 1, 2, 4)]
    shape, inp, pos = _tiny(num_layers=4, types=(SLIDING, SLIDING, SLIDING, FULL), n_ds=3,
                            images=img)
    s = sd(shape)
    h = inp.hidden.astype(np.float64)
    rows = inp.ds_rows
    layers = [inp.layer(i) for i in range(4)]
    ds = [inp.ds(i) for i in range(3)]
    with_ds, hs = O.prefill(h, layers, s, pos, [0, 24], rows, ds, False, return_all=True)
    _, hs0 = O.prefill(h, layers, s, pos, [0, 24], rows, [], False, return_all=True)
    zero = [np.zeros_like(x) for x in ds]
    np.testing.assert_array_equal(O.prefill(h, layers, s, pos, [0, 24], rows, zero, False),
                                  hs0[-1])
    # after layer 0 the difference is exactly ds_0 at the image rows
    diff = hs[0] - hs0[0]
    want = np.zeros_like(diff)
    want[rows] = O.from_storage(ds[0])
    np.testing.assert_allclose(diff, want, atol=1e-12)
    # a fourth tensor is never read: layer 3 gets no deepstack add
    extra = ds + [np.full_like(ds[0], 7)]
    np.testing.assert_array_equal(O.prefill(h, layers, s, pos, [0, 24], rows, extra[:3], False),
                                  with_ds)


def test_logits_linear_in_logit_scale():
    shape, inp, pos = _tiny()
    s = sd(shape)
    h = inp.hidden.astype(np.float64)
    l1 = O.logits(h, inp.final_ln, inp.embed, dict(s, logit_scale=0.0625), False)
    l4 = O.logits(h, inp.final_ln, inp.embed, dict(s, logit_scale=0.25), False)
    np.testing.assert_allclose(l4, 4 * l1, rtol=1e-15)
    assert l1.shape == (24, 50)


def test_silu_against_its_closed_form():
    """silu(0) = 0; silu(x) - silu(-x) = x (x * (sigmoid(x) + sigmoid(-x)) = x); silu(1) =
    sigmoid(1) = 1 / (1 + 1/e); silu(x) -> x for large x and -> 0 for very negative x.
    A sigmoid, a gelu or a tanh gate fails at least one of these."""
    assert O.silu(np.float64(0.0)) == 0.0
    x = np.linspace(-30.0, 30.0, 6001)
    np.testing.assert_allclose(O.silu(x) - O.silu(-x), x, rtol=0, atol=1e-13)
    assert O.silu(np.float64(1.0)) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert O.silu(np.float64(40.0)) == pytest.approx(40.0, rel=1e-15)
    assert abs(O.silu(np.float64(-40.0))) < 1e-15


def test_swiglu_branch_golden():
    """The hand-worked SwiGLU example (tests/golden/swiglu_tiny.txt): gate and up read
    different inputs, so their order is fixed."""
    g = read_golden("swiglu_tiny.txt")
    a = np.array([g["a"]])
    wg, wu, wd = np.array([g["wg"]]), np.array([g["wu"]]), np.array([g["wd"]])
    got = O.swiglu(a, wg, wu, wd)
    assert got.shape == (1, 1)
    assert got[0, 0] == pytest.approx(g["swiglu"][0], rel=1e-15)
    assert abs(got[0, 0] - g["swapped"][0]) > 0.2


def test_block_swiglu_golden():
    """One whole block on the hand-worked input of tests/golden/swiglu_tiny.txt: attention
    weights zero, so the block adds exactly the SwiGLU branch of a = LayerNorm(h). Fails if
    the block swaps gate and up, or gates with sigmoid instead of silu."""
    g = read_golden("swiglu_tiny.txt")
    shape = {"num_attention_heads": 1, "num_key_value_heads": 1, "head_dim": 2,
             "layer_norm_eps": 0.0, "sliding_window": 4}
    z = np.zeros((2, 2))
    layer = {"ln": np.ones(2), "wq": z, "wk": z, "wv": z, "wo": z,
             "wg": np.array([[1.0, 0.0]]), "wu": np.array([[0.0, 1.0]]),
             "wd": np.array([[1.0], [0.0]])}
    h = np.array([g["block_h"]])
    out = O.block(h, layer, FULL, shape, None, [0, 1], False)
    np.testing.assert_allclose(out[0], g["block_out"], rtol=0, atol=1e-15)
    for wrong in ("block_swapped", "block_sigmoid"):
        assert np.abs(out[0] - np.array(g[wrong])).max() > 0.4
    # the decode step runs the same branch: one cached-free token, same result
    kv = np.zeros((1, 1, 16, 2), np.float64)
    dec = O.decode_step(h, [layer], dict(shape, num_layers=1, layer_types=(FULL,),
                                         rope_theta=1e4, mrope_section=(1, 0, 0),
                                         mrope_layout="interleaved"),
                        [0], [0], np.zeros((1, 1), np.int64), lambda i: (kv, kv), 16, False)
    np.testing.assert_allclose(dec[0], g["block_out"], rtol=0, atol=1e-15)


def test_head_final_layer_norm_golden():
    """The head on the hand-worked input of tests/golden/head_final_ln_tiny.txt: the final
    LayerNorm (with its own gain) runs before the tied embedding and the logit_scale footer.
    Fails if the norm is dropped or its gain ignored."""
    g = read_golden("head_final_ln_tiny.txt")
    h = np.array([g["h"]])
    embed = np.array([g["embed_row0"], g["embed_row1"], g["embed_row2"]])
    shape = {"layer_norm_eps": 0.0, "logit_scale": g["logit_scale"][0]}
    for mirror in (False, True):    # every value on this path is exact in bf16
        got = O.logits(h, np.array(g["final_ln"]), embed, shape, mirror)
        np.testing.assert_array_equal(got[0], g["logits"])
    for wrong in ("logits_no_final_ln", "logits_no_gain"):
        assert np.abs(got[0] - np.array(g[wrong])).max() >= 0.25
    # with the workloads' eps = 1e-5, a row of mean 0 and variance 1 scales by 1/sqrt(1 + eps)
    eps = 1e-5
    row = np.array([[-1.0, 1.0, -1.0, 1.0]])
    got = O.logits(row, np.array(g["final_ln"]), embed, dict(shape, layer_norm_eps=eps), False)
    gam = np.array(g["final_ln"])
    want = g["logit_scale"][0] * np.array([gam[1], -gam[2], -gam[0] + gam[3]]) / math.sqrt(1 + eps)
    np.testing.assert_allclose(got[0], want, rtol=1e-14)


def test_text_prefill_is_causal():
    """First 48 logits of a 96-token prefill equal a 48-token prefill (4 layers, 3 sliding
    and 1 full), as in the pages' text_prefill_is_causal test."""
    types = (SLIDING, SLIDING, SLIDING, FULL)
    shape, inp, pos = _tiny(num_layers=4, types=types, T=96, window=20)
    s = sd(shape)
    layers = [inp.layer(i) for i in range(4)]
    h = inp.hidden.astype(np.float64)
    full = O.prefill(h, layers, s, pos, [0, 96], mirror_bf16=False)
    half = O.prefill(h[:48], layers, s, pos[:, :48], [0, 48], mirror_bf16=False)
    l96 = O.logits(full[:48], inp.final_ln, inp.embed, s, False)
    l48 = O.logits(half, inp.final_ln, inp.embed, s, False)
    np.testing.assert_allclose(l96, l48, atol=1e-4)
    np.testing.assert_allclose(l96, l48, atol=1e-12)


def _cache_from_prefill(shape, inp, h_in, layers, pos, n, page, table, n_pages):
    """Post-rotation K and V of tokens 0..n-1 of each layer written into paged pools."""
    s = sd(shape)
    cs = O.mrope_cos_sin(pos, s["head_dim"], s["rope_theta"], s["mrope_section"])
    nkv, d = s["num_key_value_heads"], s["head_dim"]
    _, hs = O.prefill(h_in, layers, s, pos, [0, h_in.shape[0]], mirror_bf16=False,
                      return_all=True)
    ins = [h_in] + hs[:-1]
    pools = []
    for i, L in enumerate(layers):
        a = O.layer_norm(ins[i], O.from_storage(L["ln"]), s["layer_norm_eps"])
        k = (a @ O.from_storage(L["wk"]).T).reshape(-1, nkv, d)
        v = (a @ O.from_storage(L["wv"]).T).reshape(-1, nkv, d)
        if s["layer_types"][i] == SLIDING:
            k = O.apply_rope(k, *cs)
        K = np.zeros((n_pages, nkv, page, d))
        V = np.zeros((n_pages, nkv, page, d))
        for t in range(n):
            K[table[t // page], :, t % page] = k[t]
            V[table[t // page], :, t % page] = v[t]
        pools.append((K, V))
    return pools, hs[-1]


@pytest.mark.parametrize("window", [5, 64])
def test_decode_equals_last_row_of_prefill(window):
    types = (SLIDING, FULL)
    n = 21                       # cached tokens; the decoded token is number n
    shape, inp, pos = _tiny(num_layers=2, types=types, T=n + 1, window=window)
    s = sd(shape)
    layers = [inp.layer(i) for i in range(2)]
    h = inp.hidden.astype(np.float64)
    page, n_pages = 4, 9
    table = np.random.default_rng(12).permutation(n_pages)[:6]
    pools, h_pref = _cache_from_prefill(shape, inp, h, layers, pos, n, page, table, n_pages)
    out = O.decode_step(h[n:n + 1], layers, s, [n], [0], table[None, :],
                        lambda i: pools[i], page, mirror_bf16=False)
    np.testing.assert_allclose(out[0], h_pref[n], atol=1e-10)
    # relabelling the pool's pages (and the table with them) changes nothing
    perm = np.random.default_rng(13).permutation(n_pages)
    inv = np.argsort(perm)
    pools2 = [(K[inv], V[inv]) for K, V in pools]
    out2 = O.decode_step(h[n:n + 1], layers, s, [n], [0], perm[table][None, :],
                         lambda i: pools2[i], page, mirror_bf16=False)
    np.testing.assert_array_equal(out2, out)


# ---------------------------------------------------------------- embedding merge
def test_embed_merge_worked_example():
    g = read_golden("embed_merge_tiny.txt")
    embed = np.array([[v, 10 * v, -v] for v in range(4)], dtype=np.float64)
    h = O.embed_merge(g["tokens"], embed, g["mm_rows"], [g["mm_feat0"], g["mm_feat1"]])
    for t in range(5):
        assert h[t].tolist() == [float(x) for x in g[f"h{t}"]]


def test_embed_merge_without_images_is_the_lookup_and_rejects_bad_input():
    rng = np.random.default_rng(7)
    embed = rng.standard_normal((11, 8))
    toks = rng.integers(0, 11, size=20)
    h = O.embed_merge(toks, embed)
    # each row is some embedding row, the one its token names (checked column by column)
    for t in range(20):
        assert np.array_equal(h[t], embed[toks[t]])
    with pytest.raises(ValueError):
        O.embed_merge([11], embed)
    with pytest.raises(ValueError):
        O.embed_merge([1, 2, 3], embed, [1, 1], np.zeros((2, 8)))
    with pytest.raises(ValueError):
        O.embed_merge([1, 2, 3], embed, [3], np.zeros((1, 8)))


# ---------------------------------------------------------------- 4-bit affine weights
def test_dequantize_affine_worked_example():
    g = read_golden("affine_q4_row.txt")
    packed = np.array([g["words"]], dtype=np.uint64).astype(np.uint32)
    w = O.dequantize_affine(packed, np.array([g["scales"]]), np.array([g["biases"]]))
    assert w.shape == (1, 128)
    assert w[0, :16].tolist() == g["w_first16"]
    assert w[0, 32:36].tolist() == g["w_32_35"]
    assert np.all(w[0, 64:] == g["w_group1"][0])
    # the descending half of group 0: q = 15 - (k - 16)
    assert w[0, 16:32].tolist() == [0.5 * (15 - i) - 2.0 for i in range(16)]
    assert np.all(w[0, 48:64] == 0.5 * 7 - 2.0)


def test_drift_script_moves_each_element_by_one_unit_in_the_last_place():
    """The perturbation behind the 28-layer end-to-end bound (tests/golden/
    make_stack28_drift.py) moves every element by exactly one float32 (or bf16) ulp."""
    import importlib.util, os
    from conftest import GOLDEN
    spec = importlib.util.spec_from_file_location("make_drift",
                                                  os.path.join(GOLDEN, "make_stack28_drift.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    x = np.random.default_rng(3).standard_normal(5000).astype(np.float32).astype(np.float64)
    y = mod.nudge(x, 23, 1)
    up = np.nextafter(x.astype(np.float32), np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(x.astype(np.float32), np.float32(-np.inf)).astype(np.float64)
    # one ulp of the binade of x (at a power of two, the step down is half as large: still one
    # unit in the last place of x's own binade)
    ok = (y == up) | (y == dn) | (np.abs(y - x) == np.abs(up - x))
    assert ok.all()
    xb = O.round_bf16(x)
    yb = mod.nudge(xb, 7, 2)
    assert np.array_equal(O.round_bf16(yb), yb)            # still a bf16 value
    assert (np.abs(yb - xb) == np.exp2(np.floor(np.log2(np.abs(xb))) - 7)).all()
