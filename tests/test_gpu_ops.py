"""Parity of the single CUDA operations (through the C-ABI) against the fp64 oracle.

Inputs are seeded; sizes span several tiles and end in ragged tails. Tolerances:
LayerNorm and the MRoPE table are compared at their storage precision; the GEMM at fp32
accumulation accuracy; attention (bf16 P and bf16 output) within the stack tolerance
max-abs 2e-2 / mean-abs 2e-3 (tighter in practice).
"""
import numpy as np
import pytest
import torch

import cohere_compass_decoder_gb300._lib as L
from oracle import decoder as O

from gpu_util import require_gpu, bf16_dev, f64, err_stats, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _sync():
    torch.cuda.synchronize()
    L.cc_op_sync()


# --------------------------------------------------------------------------- LayerNorm
@pytest.mark.parametrize("rows,H", [(300, 2048), (5, 256), (129, 1024), (1, 128), (33, 640),
                                    (17, 4096), (9, 3968)])
def test_layernorm_matches_oracle(rows, H):
    rng = np.random.default_rng(rows + H)
    x = (rng.standard_normal((rows + 7, H)) * 3 + 0.5).astype(np.float32)
    g = bf16_dev(1 + 0.02 * rng.standard_normal(H))
    idx = rng.permutation(rows + 7)[:rows].astype(np.int32)
    out = torch.empty(rows, H, dtype=torch.bfloat16, device="cuda")
    xd = torch.from_numpy(x).cuda()
    L.cc_op_layernorm(xd, g, out, rows, H, 1e-5, torch.from_numpy(idx).cuda())
    _sync()
    want = O.round_bf16(O.layer_norm(x[idx].astype(np.float64), f64(g), 1e-5))
    got = f64(out)
    ulp = np.abs(want) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(got - want) <= ulp * 1.01)
    assert np.mean(got != want) < 0.01


# --------------------------------------------------------------------------- embedding merge
@pytest.mark.parametrize("T,H,V,n_img", [(300, 256, 1000, 37), (1, 128, 7, 0), (513, 2048, 4000, 200),
                                         (70, 640, 300, 9), (20, 4096, 50, 3)])
def test_embed_merge_matches_oracle(T, H, V, n_img):
    rng = np.random.default_rng(T + H)
    embed = bf16_dev(0.5 * rng.standard_normal((V, H)))
    tok = rng.integers(0, V, size=T).astype(np.int32)
    rows = rng.permutation(T)[:n_img].astype(np.int32)
    feats = bf16_dev(rng.standard_normal((max(n_img, 1), H)))[:n_img]
    g = bf16_dev(1 + 0.02 * rng.standard_normal(H))
    h = torch.empty(T, H, dtype=torch.float32, device="cuda")
    a = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    tok_d = torch.from_numpy(tok).cuda()
    rows_d = torch.from_numpy(rows).cuda() if n_img else None
    L.cc_op_embed_merge(tok_d, T, embed, V, H, rows_d, feats if n_img else None, n_img, h, g, 1e-5, a)
    _sync()
    want = O.embed_merge(tok, f64(embed), rows if n_img else None, f64(feats) if n_img else None)
    assert np.array_equal(f64(h), want)               # a copy: bit-exact
    # the fused LayerNorm is the standalone one, bit for bit
    a2 = torch.empty_like(a)
    L.cc_op_layernorm(h, g, a2, T, H, 1e-5, None)
    _sync()
    assert torch.equal(a, a2)
    ln_ref = O.round_bf16(O.layer_norm(want, f64(g), 1e-5))
    assert np.abs(f64(a) - ln_ref).max() <= np.abs(ln_ref).max() * 2.0 ** -7


def test_embed_merge_reports_a_token_outside_the_vocabulary():
    V, H, T = 50, 128, 20
    embed = torch.zeros(V, H, dtype=torch.bfloat16, device="cuda")
    tok = torch.arange(T, dtype=torch.int32, device="cuda")
    tok[5] = V
    h = torch.empty(T, H, dtype=torch.float32, device="cuda")
    L.cc_op_embed_merge(tok, T, embed, V, H, None, None, 0, h)
    with pytest.raises(L.CCError) as e:
        L.cc_op_sync()
    assert e.value.status == L.CC_ERR_DEVICE_CHECK
    assert torch.count_nonzero(h[5]) == 0


# --------------------------------------------------------------------------- MRoPE table
@pytest.mark.parametrize("section,theta", [((24, 20, 20), 50000.0), ((12, 10, 10), 1e4)])
def test_mrope_table_matches_oracle(section, theta):
    rng = np.random.default_rng(3)
    T = 777
    pos = rng.integers(0, 40000, size=(3, T)).astype(np.int32)
    d = 2 * sum(section)
    table = torch.empty(T, d // 2, 2, dtype=torch.float32, device="cuda")
    L.cc_op_mrope_table(torch.from_numpy(pos).cuda(), T, d, theta, section, table)
    _sync()
    cos, sin = O.mrope_cos_sin(pos, d, theta, section)
    got = f64(table)
    assert np.abs(got[..., 0] - cos[:, :d // 2]).max() < 2e-6
    assert np.abs(got[..., 1] - sin[:, :d // 2]).max() < 2e-6


@pytest.mark.parametrize("section,theta", [((24, 20, 20), 50000.0), ((12, 10, 10), 1e4),
                                           ((16, 8, 8), 1e6)])
def test_mrope_table_sections_layout_matches_oracle(section, theta):
    """The contiguous [H, W, T]-section layout (parity unpinned: the oracle states a reading)."""
    rng = np.random.default_rng(4)
    T = 501
    pos = rng.integers(0, 40000, size=(3, T)).astype(np.int32)
    d = 2 * sum(section)
    table = torch.empty(T, d // 2, 2, dtype=torch.float32, device="cuda")
    L.cc_op_mrope_table_layout(torch.from_numpy(pos).cuda(), T, d, theta, section,
                               "sections_hwt", table)
    _sync()
    cos, sin = O.mrope_cos_sin(pos, d, theta, section, "sections_hwt")
    got = f64(table)
    assert np.abs(got[..., 0] - cos[:, :d // 2]).max() < 2e-6
    assert np.abs(got[..., 1] - sin[:, :d // 2]).max() < 2e-6


# --------------------------------------------------------------------------- GEMM
@pytest.mark.parametrize("m,n,k", [(128, 128, 64), (300, 384, 640), (64, 2560, 2048),
                                   (1, 1280, 128), (1000, 512, 1024)])
def test_gemm_matches_oracle(m, n, k):
    rng = np.random.default_rng(m * 7 + n + k)
    a = bf16_dev(rng.standard_normal((m, k)))
    b = bf16_dev(rng.standard_normal((n, k)))
    c = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    L.cc_op_gemm_bf16(a, b, c, m, n, k, 0.5, 0)
    _sync()
    want = 0.5 * (f64(a) @ f64(b).T)
    got = f64(c)
    rel = np.abs(got - want).max() / np.abs(want).max()
    assert np.all(np.isfinite(got))
    assert rel < 1e-5, rel


def test_gemm_accumulates():
    rng = np.random.default_rng(11)
    m, n, k = 200, 256, 512
    a, b = bf16_dev(rng.standard_normal((m, k))), bf16_dev(rng.standard_normal((n, k)))
    c0 = rng.standard_normal((m, n)).astype(np.float32)
    c = torch.from_numpy(c0).cuda()
    L.cc_op_gemm_bf16(a, b, c, m, n, k, 1.0, 1)
    _sync()
    want = c0 + f64(a) @ f64(b).T
    assert np.abs(f64(c) - want).max() / np.abs(want).max() < 1e-5


# --------------------------------------------------------------------------- 4-bit affine GEMM
def _bits(x):
    """float values -> bf16 bit patterns (round to nearest even), as the test's own input."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def _u16_dev(u):
    return torch.from_numpy(np.ascontiguousarray(u).view(np.int16)).cuda().view(torch.bfloat16)


def _u32_dev(u):
    return torch.from_numpy(np.ascontiguousarray(u, dtype=np.uint32).view(np.int32)).cuda()


def _q4_matrix(rng, n, k):
    """Uniform 4-bit fields; scales of both signs and several binades; biases around
    -7.5 scale (the mlx conversion's typical offset) plus spread."""
    words = rng.integers(0, 1 << 32, size=(n, k // 8), dtype=np.uint64).astype(np.uint32)
    sc = _bits(0.01 * rng.standard_normal((n, k // 64)) * rng.choice([0.25, 1, 4], (n, k // 64)))
    sf = (sc.astype(np.uint32) << 16).view(np.float32)
    bi = _bits(-7.5 * sf + 0.01 * rng.standard_normal(sf.shape))
    return words, sc, bi


def _tile_host(words, sc, bi):
    """The tiled block layout of include/cc.h, written out on the host (a rearrangement)."""
    rows, W = words.shape
    G = sc.shape[1]
    kqt = (G + 1) // 2
    wpad = np.zeros((rows, kqt * 16), np.uint32)
    wpad[:, :W] = words
    sbpad = np.zeros((rows, kqt * 2), np.uint32)
    sbpad[:, :G] = sc.astype(np.uint32) | (bi.astype(np.uint32) << 16)
    out = np.zeros((rows // 128, kqt, 2304), np.uint32)
    for t in range(rows // 128):
        for j in range(kqt):
            blk = wpad[128 * t:128 * t + 128, 16 * j:16 * j + 16]          # [row, word]
            out[t, j, :2048] = blk.reshape(128, 4, 4).transpose(1, 0, 2).reshape(-1)
            out[t, j, 2048:] = sbpad[128 * t:128 * t + 128, 2 * j:2 * j + 2].T.reshape(-1)
    return out.reshape(-1)


def _q4_upload(words, sc, bi):
    n, g = sc.shape
    out = torch.empty(L.cc_q4_tiled_bytes(n, 64 * g), dtype=torch.uint8, device="cuda")
    L.cc_pack_q4_tiles(_u32_dev(words), _u16_dev(sc), _u16_dev(bi), n, 64 * g, out)
    return out


@pytest.mark.parametrize("rows,k", [(256, 640), (128, 64), (384, 192)])
def test_q4_tiles_layout(rows, k):
    rng = np.random.default_rng(rows + k)
    words = rng.integers(0, 1 << 32, size=(rows, k // 8), dtype=np.uint64).astype(np.uint32)
    sc = rng.integers(0, 1 << 16, size=(rows, k // 64), dtype=np.uint16)
    bi = rng.integers(0, 1 << 16, size=(rows, k // 64), dtype=np.uint16)
    out = _q4_upload(words, sc, bi)
    _sync()
    assert out.numel() == (rows // 128) * ((k // 64 + 1) // 2) * 9216
    assert np.array_equal(out.cpu().numpy().view(np.uint32), _tile_host(words, sc, bi))


@pytest.mark.parametrize("m,n,k,acc", [(64, 256, 2048, 0), (1, 128, 64, 0), (128, 384, 640, 0),
                                       (100, 1280, 1024, 0), (64, 2048, 10240, 1),
                                       (5, 512, 4096, 1), (16, 256, 192, 0), (64, 256, 1472, 1),
                                       (33, 128 * 160, 256, 0), (128, 128 * 400, 384, 0),
                                       (100, 128 * 320, 640, 0)])
def test_gemm_q4_matches_oracle(m, n, k, acc):
    from oracle.runs import dequantized_q4
    rng = np.random.default_rng(m + 3 * n + 7 * k)
    a = bf16_dev(rng.standard_normal((m, k)))
    words, sc, bi = _q4_matrix(rng, n, k)
    wt = _q4_upload(words, sc, bi)
    c0 = rng.standard_normal((m, n)).astype(np.float32)
    c = torch.from_numpy(c0).cuda() if acc else torch.full((m, n), float("nan"), device="cuda")
    L.cc_op_gemm_q4(a, wt, c, m, n, k, 0.5, acc)
    _sync()
    want = 0.5 * (f64(a) @ dequantized_q4((words, sc, bi)).T) + (c0 if acc else 0.0)
    got = f64(c)
    assert np.all(np.isfinite(got))
    rel = np.abs(got - want).max() / np.abs(want).max()
    assert rel < 1e-5, rel


def test_pack_layer_weights_q4_layout():
    """w1's rows q | k | v | 64-row gate/up blocks and w2's columns o | down, in tiled form:
    a byte-exact rearrangement of the seven checkpoint matrices."""
    from synth import small_shape
    shape = small_shape(num_layers=1, heads=(4, 2), inter=192)
    cfg = L.make_config(shape, 16, 16)
    H, d, I = shape.hidden_size, shape.head_dim, shape.intermediate_size
    nq, nkv = shape.num_attention_heads, shape.num_key_value_heads
    dims = [(nq * d, H), (nkv * d, H), (nkv * d, H), (H, nq * d), (I, H), (I, H), (H, I)]
    rng = np.random.default_rng(5)
    mats = [(rng.integers(0, 1 << 32, size=(r, c // 8), dtype=np.uint64).astype(np.uint32),
             rng.integers(0, 1 << 16, size=(r, c // 64), dtype=np.uint16),
             rng.integers(0, 1 << 16, size=(r, c // 64), dtype=np.uint16)) for r, c in dims]
    N1, K2 = (nq + 2 * nkv) * d + 2 * I, nq * d + I
    w1 = torch.empty(L.cc_q4_tiled_bytes(N1, H), dtype=torch.uint8, device="cuda")
    w2 = torch.empty(L.cc_q4_tiled_bytes(H, K2), dtype=torch.uint8, device="cuda")
    L.cc_pack_layer_weights_q4(cfg, [_u32_dev(m[0]) for m in mats], [_u16_dev(m[1]) for m in mats],
                               [_u16_dev(m[2]) for m in mats], w1, w2)
    _sync()

    def rows_w1(x):
        q, k_, v, o, g, u, dn = x
        gu = np.stack([g.reshape(I // 64, 64, -1), u.reshape(I // 64, 64, -1)], 1).reshape(2 * I, -1)
        return np.concatenate([q, k_, v, gu])

    fused1 = [rows_w1([m[p] for m in mats]) for p in range(3)]
    fused2 = [np.concatenate([mats[3][p], mats[6][p]], 1) for p in range(3)]
    assert np.array_equal(w1.cpu().numpy().view(np.uint32), _tile_host(*fused1))
    assert np.array_equal(w2.cpu().numpy().view(np.uint32), _tile_host(*fused2))


# --------------------------------------------------------------------------- prefill attention
def _attn_case(lens, nq, nkv, window, seed, qscale=1.0, ramp=0.0):
    """ramp > 0 adds a score bias growing with the key index (so the running max keeps
    moving and the output rescaling runs): k[j] += ramp * j / T * u with q . u > 0."""
    rng = np.random.default_rng(seed)
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    qn = rng.standard_normal((T, nq * 128)) * qscale
    kn = rng.standard_normal((T, nkv * 128))
    if ramp:
        qn[:, ::128] = np.abs(qn[:, ::128]) + 1.0
        kn[:, ::128] += ramp * np.arange(T)[:, None] / T
    q = bf16_dev(qn)
    k = bf16_dev(kn)
    v = bf16_dev(rng.standard_normal((T, nkv * 128)))
    ld = nq * 128 + 64
    out = torch.full((T, ld), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.cc_op_attention_prefill(q, k, v, out, ld, torch.from_numpy(cu).cuda(), len(lens), T, nq,
                              nkv, window)
    _sync()
    want = O.attention(f64(q).reshape(T, nq, 128), f64(k).reshape(T, nkv, 128),
                       f64(v).reshape(T, nkv, 128), cu, window if window > 0 else None,
                       128 ** -0.5)
    got = f64(out)[:, :nq * 128].reshape(T, nq, 128)
    assert np.all(np.isnan(f64(out)[:, nq * 128:]))   # nothing written past the heads
    return got, want


@pytest.mark.parametrize("lens,nq,nkv,window", [
    ([300], 4, 2, 0),
    ([300], 4, 1, 64),
    ([100, 260, 37], 2, 2, 100),
    ([1], 2, 1, 0),
    ([1000], 16, 4, 512),
    ([129, 128, 127], 8, 1, 0),
    ([300], 16, 1, 0),
    ([260, 77], 16, 1, 100),
])
def test_attention_prefill_matches_oracle(lens, nq, nkv, window):
    got, want = _attn_case(lens, nq, nkv, window, seed=sum(lens) + nq + window)
    assert_close(got, want, 2e-2, 2e-3, "attention")


@pytest.mark.parametrize("lens,window,qscale,ramp", [
    ([700], 0, 4.0, 0.0), ([700], 300, 4.0, 0.0), ([900], 0, 1.0, 300.0), ([513, 400], 0, 2.0, 200.0),
])
def test_attention_prefill_large_scores(lens, window, qscale, ramp):
    got, want = _attn_case(lens, 4, 2, window, seed=77 + len(lens), qscale=qscale, ramp=ramp)
    assert_close(got, want, 2e-2, 2e-3, "attention (large scores)")


def test_attention_window_at_least_sequence_equals_full():
    rng = np.random.default_rng(5)
    T, nq, nkv = 333, 4, 2
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    q, k, v = (bf16_dev(rng.standard_normal((T, n * 128))) for n in (nq, nkv, nkv))
    outs = []
    for w in (0, T, 5000):
        o = torch.empty(T, nq * 128, dtype=torch.bfloat16, device="cuda")
        L.cc_op_attention_prefill(q, k, v, o, nq * 128, cu, 1, T, nq, nkv, w)
        outs.append(o)
    _sync()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])



# --------------------------------------------------------------------------- mask membership
# With zero queries every score is 0, so every visible key gets weight exactly 1 and P V
# sums exact integers. With V[j] = e_(j mod 128) (one-hot by key position), output column c
# of a query is (its visible keys j with j = c mod 128) / (its visible keys): a closed form
# of the visible set. One key too many or too few moves that key's column by at least a
# third, far outside one bf16 rounding, so this checks the causal / window / sequence masks
# key by key (the random-input parity tests bound such an error only through the tolerance).
def _onehot_by_position(n, nkv):
    v = np.zeros((n, nkv, 128))
    v[np.arange(n), :, np.arange(n) % 128] = 1.0
    return v


def _visible_fraction(lo, hi):
    """Column c: #{lo <= j <= hi : j = c mod 128} / (hi - lo + 1)."""
    c = np.arange(128)
    first = lo + (c - lo) % 128
    cnt = np.where(first <= hi, (hi - first) // 128 + 1, 0)
    return cnt / (hi - lo + 1)


def _assert_one_rounding(got, want, what):
    # bf16(count * fp32(1/n)): within one bf16 rounding (2^-8 relative); absent keys give 0
    bad = np.abs(got - want) > want * 2.0 ** -8 * 1.01
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, first at {np.argwhere(bad)[0]}"


@pytest.mark.parametrize("lens,window", [
    ([1000], 0), ([1000], 1), ([1000], 127), ([1000], 128), ([1000], 129), ([1000], 300),
    ([1000], 512), ([1000], 513), ([2048], 512), ([2048], 0),
    ([129, 300, 1, 700], 256), ([129, 300, 1, 700], 0), ([128, 128, 255], 128)])
def test_attention_prefill_mask_membership(lens, window):
    nq, nkv = 4, 2
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rng = np.random.default_rng(T + window)
    q = torch.zeros(T, nq * 128, dtype=torch.bfloat16, device="cuda")
    k = bf16_dev(rng.standard_normal((T, nkv * 128)))
    vp = np.zeros((T, nkv, 128))
    for s0, s1 in zip(cu[:-1], cu[1:]):
        vp[s0:s1] = _onehot_by_position(s1 - s0, nkv)
    v = bf16_dev(vp.reshape(T, nkv * 128))
    out = torch.empty(T, nq * 128, dtype=torch.bfloat16, device="cuda")
    L.cc_op_attention_prefill(q, k, v, out, nq * 128, torch.from_numpy(cu).cuda(), len(lens), T,
                              nq, nkv, window)
    _sync()
    want = np.zeros((T, nq, 128))
    for s0, s1 in zip(cu[:-1], cu[1:]):
        for i in range(s1 - s0):
            lo = max(0, i - window + 1) if window > 0 else 0
            want[s0 + i] = _visible_fraction(lo, i)
    got = f64(out).reshape(T, nq, 128)
    _assert_one_rounding(got, want, f"prefill mask lens={lens} window={window}")
    # the oracle's masks give the same visible sets
    ref = O.attention(np.zeros((T, nq, 128)), f64(k).reshape(T, nkv, 128), vp, cu,
                      window if window > 0 else None, 128 ** -0.5)
    np.testing.assert_allclose(ref, want, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("window", [0, 1, 16, 127, 128, 129, 1024, 4096])
def test_attention_decode_mask_membership(window):
    nq, nkv, ps = 8, 2, 16
    n_keys = np.array([1, 15, 16, 17, 127, 128, 129, 1023, 1024, 1025, 4096, 4097],
                      dtype=np.int32)
    B = len(n_keys)
    max_pages = (int(n_keys.max()) + ps - 1) // ps
    n_pages = B * max_pages + 3
    rng = np.random.default_rng(window + 11)
    table = rng.permutation(n_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    vp = np.zeros((n_pages, nkv, ps, 128))
    for b in range(B):
        j = np.arange(int(n_keys[b]))
        vp[table[b][j // ps], :, j % ps, j % 128] = 1.0
    kp = bf16_dev(rng.standard_normal((n_pages, nkv, ps, 128)))
    q = torch.zeros(B, nq * 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(B, nq * 128, dtype=torch.bfloat16, device="cuda")
    L.cc_op_attention_decode(q, kp, bf16_dev(vp), n_pages, torch.from_numpy(table).cuda(),
                             max_pages, torch.from_numpy(n_keys).cuda(), B, nq, nkv, ps, window,
                             out, nq * 128)
    _sync()
    want = np.zeros((B, nq, 128))
    for b in range(B):
        n = int(n_keys[b])
        lo = max(0, n - window) if window > 0 else 0
        want[b] = _visible_fraction(lo, n - 1)
    _assert_one_rounding(f64(out).reshape(B, nq, 128), want, f"decode mask window={window}")


# --------------------------------------------------------------------------- decode attention
@pytest.mark.parametrize("nq,nkv,window,max_pages", [
    (8, 2, 0, 44), (8, 2, 200, 44), (16, 4, 0, 44), (4, 4, 37, 44), (8, 1, 0, 44),
    (16, 1, 0, 44), (16, 4, 0, 300), (16, 4, 1500, 300)])
def test_attention_decode_matches_oracle(nq, nkv, window, max_pages):
    rng = np.random.default_rng(nq * 13 + nkv + window + max_pages)
    B, ps = 7, 16
    n_pages = B * max_pages + 5
    n_keys = rng.integers(1, max_pages * ps + 1, size=B).astype(np.int32)
    n_keys[0] = 1
    n_keys[1] = max_pages * ps
    table = rng.permutation(n_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    kp = bf16_dev(rng.standard_normal((n_pages, nkv, ps, 128)))
    vp = bf16_dev(rng.standard_normal((n_pages, nkv, ps, 128)))
    q = bf16_dev(rng.standard_normal((B, nq * 128)))
    out = torch.empty(B, nq * 128, dtype=torch.bfloat16, device="cuda")
    L.cc_op_attention_decode(q, kp, vp, n_pages, torch.from_numpy(table).cuda(), max_pages,
                             torch.from_numpy(n_keys).cuda(), B, nq, nkv, ps, window, out,
                             nq * 128)
    _sync()
    K, V, Q = f64(kp), f64(vp), f64(q).reshape(B, nq, 128)
    want = np.zeros((B, nq, 128))
    for b in range(B):
        n = int(n_keys[b])
        idx = np.arange(n)
        Kb = K[table[b][idx // ps], :, idx % ps, :]
        Vb = V[table[b][idx // ps], :, idx % ps, :]
        qi = np.zeros((n, nq, 128))
        qi[n - 1] = Q[b]
        want[b] = O.attention(qi, Kb, Vb, [0, n], window if window > 0 else None,
                              128 ** -0.5, row_block=n)[n - 1]
    got = f64(out).reshape(B, nq, 128)
    assert_close(got, want, 2e-2, 2e-3, "decode attention")


def test_attention_decode_flags_bad_page_ids():
    B, nq, nkv, ps, max_pages = 2, 4, 1, 16, 4
    n_pages = 8
    table = torch.tensor([[0, 1, 2, 3], [4, 5, 99, 7]], dtype=torch.int32, device="cuda")
    kp = torch.zeros(n_pages, nkv, ps, 128, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    q = torch.zeros(B, nq * 128, dtype=torch.bfloat16, device="cuda")
    nk = torch.tensor([64, 64], dtype=torch.int32, device="cuda")
    out = torch.empty(B, nq * 128, dtype=torch.bfloat16, device="cuda")
    L.cc_op_attention_decode(q, kp, vp, n_pages, table, max_pages, nk, B, nq, nkv, ps, 0, out,
                             nq * 128)
    torch.cuda.synchronize()
    with pytest.raises(L.CCError) as e:
        L.cc_op_sync()
    assert e.value.status == L.CC_ERR_DEVICE_CHECK
    L.cc_op_sync()   # the flag was cleared
