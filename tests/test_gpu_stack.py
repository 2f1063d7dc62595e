"""Parity of the whole path (layer stack + head, through the C-ABI) against the oracle.

bf16 workloads compare against the oracle's bf16-mirror mode (rounding at the GPU's
storage points) with the benchmark spec's tolerance on the outputs: max-abs <= 2e-2 and
mean-abs <= 2e-3 on the final hidden state and on the logits; the logits also have to
agree to 2% of their largest magnitude, which is the stricter test for them. The fp32
workload compares against pure fp64 at fp32-level tolerance (1e-4).
"""
import numpy as np
import pytest
import torch

from oracle import runs as R
from synth import Inputs, Workload, ImageSpan, small_shape, SLIDING, FULL
from synth.configs import layer_fp32_T128, pair_T2048, stack28_T8192, decode_B64_cache4096, varlen_T32768
from cohere_compass_decoder_gb300.workload import GpuWorkload, as_numpy
from cohere_compass_decoder_gb300.model import to_device
import cohere_compass_decoder_gb300._lib as L

from gpu_util import require_gpu, assert_close, err_stats
from conftest import read_golden

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN = 2e-2, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _check(inp, gw, h_gpu, lg_gpu, tol=(TOL_MAX, TOL_MEAN), lg_rel=2e-2):
    h_ref, lg_ref = R.run(inp)
    h = as_numpy(h_gpu)
    lg = as_numpy(lg_gpu)
    mx, mn = assert_close(h, h_ref, tol[0], tol[1], "hidden")
    lmx, lmn = assert_close(lg, lg_ref, tol[0], tol[1], "logits")
    rel = lmx / max(np.abs(lg_ref).max(), 1e-30)
    assert rel <= lg_rel, f"logits relative error {rel:.3g}"
    return dict(h_max=mx, h_mean=mn, lg_max=lmx, lg_mean=lmn, lg_rel=rel)


def _run(inp, max_tokens=None):
    gw = GpuWorkload(inp, max_tokens=max_tokens)
    h = gw.fresh_hidden()
    lg = gw.step(h)
    gw.sync()
    return gw, h, lg


def _small(name, seq_lens, images, n_ds, types=(SLIDING, FULL), window=64, head_rows="all",
           seed=21, **kw):
    shape = small_shape(num_layers=len(types), layer_types=types, window=window, **kw)
    return Inputs(Workload(name, shape, "prefill", seq_lens, images=images, n_deepstack=n_ds,
                           head_rows=head_rows, seed=seed))


# ------------------------------------------------------------------------- small bf16 stacks
def test_small_stack_single_sequence():
    inp = _small("small1", [300], [ImageSpan(0, 37, 1, 8, 8)], 2)
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg)


def test_small_stack_varlen_and_gqa_variants():
    imgs = [ImageSpan(0, 10, 1, 5, 6), ImageSpan(1, 0, 1, 4, 4), ImageSpan(2, 50, 1, 3, 3),
            ImageSpan(2, 70, 1, 2, 5)]
    inp = _small("small2", [100, 200, 157], imgs, 2, types=(SLIDING, SLIDING, FULL, SLIDING),
                 window=90, heads=(8, 2), hidden=384, inter=256, vocab=384, seed=22)
    gw, h, lg = _run(inp, max_tokens=600)
    _check(inp, gw, h, lg)


def test_small_stack_sections_mrope_layout():
    """Prefill and decode with the contiguous [H, W, T]-section MRoPE layout (parity unpinned:
    the oracle states a reading of the permutation)."""
    inp = _small("small_sec", [260], [ImageSpan(0, 20, 1, 6, 8)], 1,
                 types=(SLIDING, FULL, SLIDING), mrope_layout="sections_hwt", seed=27)
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg)
    shape = small_shape(num_layers=2, layer_types=(SLIDING, FULL), window=70, heads=(8, 2),
                        mrope_layout="sections_hwt")
    dec = Inputs(Workload("dec_sec", shape, "decode", [], head_rows="all", seed=28,
                          decode_batch=6, cache_len=120, page_size=16))
    gw, h, lg = _run(dec)
    _check(dec, gw, h, lg)


def test_small_stack_with_empty_sequences():
    """Empty sequences inside a packed batch (equal cu_seqlens entries) contribute no tokens,
    no positions and no work; the others are unaffected (reading: an empty sequence has no
    positions and rope_delta 0)."""
    inp = _small("small_empty", [0, 150, 0, 0, 91, 0], [ImageSpan(1, 30, 1, 4, 5),
                                                          ImageSpan(4, 0, 1, 3, 3)], 2,
                 types=(SLIDING, FULL), window=70, seed=29)
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg)



def test_small_stack_hidden_640_prefill_and_decode():
    """A hidden size that is a multiple of 128 but not of 256 (640: five 128-column blocks per
    LayerNorm row, 128-wide output tiles in the residual GEMM), through prefill, the head and a
    decode step."""
    inp = _small("small_h640", [200], [ImageSpan(0, 25, 1, 4, 6)], 1,
                 types=(SLIDING, FULL), window=50, hidden=640, inter=320, seed=24)
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg)
    shape = small_shape(num_layers=2, layer_types=(SLIDING, FULL), window=70, hidden=640,
                        inter=320)
    dec = Inputs(Workload("dec_h640", shape, "decode", [], head_rows="all", seed=25,
                          decode_batch=5, cache_len=90, page_size=16))
    gw, h, lg = _run(dec)
    _check(dec, gw, h, lg)

def test_a_device_wait_that_runs_out_reports_timeout_and_the_plan_recovers():
    """The bounded-wait error path on the GPU: the test hook makes the first GEMM of a forward
    wait on a barrier that nothing arrives on. That wait gives up, cc_sync reports
    CC_ERR_TIMEOUT (and clears the flag), and the next forward on the same plan is complete
    and matches the oracle."""
    inp = _small("small_stall", [260], [ImageSpan(0, 30, 1, 6, 6)], 1, seed=31)
    gw = GpuWorkload(inp)
    h = gw.fresh_hidden()
    lg = gw.step(h)
    gw.sync()
    _check(inp, gw, h, lg)
    L.cc_test_stall_next_gemm()
    h_bad = gw.fresh_hidden()
    gw.step(h_bad)
    with pytest.raises(L.CCError) as e:
        gw.sync()
    assert e.value.status == L.CC_ERR_TIMEOUT
    h2 = gw.fresh_hidden()
    lg2 = gw.step(h2)
    gw.sync()
    _check(inp, gw, h2, lg2)
    gw.close()


def test_small_stack_single_row_block_splits_the_output_projection():
    """T = 100 (one row block) at the pair's hidden size: the output projection splits K and
    adds with reductions, and each layer's LayerNorm runs as its own kernel."""
    inp = _small("small_rb1", [100], [ImageSpan(0, 20, 1, 4, 6)], 2,
                 types=(SLIDING, FULL, SLIDING), hidden=2048, inter=1024, heads=(16, 4),
                 vocab=256, seed=34)
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg)


def test_small_stack_mha_and_no_images():
    inp = _small("small3", [130], [], 0, types=(FULL, SLIDING), window=33, heads=(2, 2),
                 hidden=128, inter=128, vocab=256, seed=23)
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg)


def test_prefill_from_token_ids():
    """The embedding merge fused with layer 0's LayerNorm gives the same stack output, bit for
    bit, as the merge op followed by the hidden-state prefill, and the oracle's merge + stack."""
    inp = _small("small_tok", [300], [ImageSpan(0, 37, 1, 8, 8)], 2, seed=29)
    gw = GpuWorkload(inp)
    st = gw.stack
    s = inp.shape
    tok = torch.from_numpy(inp.token_ids).cuda()
    rows = torch.from_numpy(inp.mm_rows.astype(np.int32)).cuda()
    feats = to_device(inp.mm_embeds)
    T = inp.wl.total_tokens
    h1 = torch.empty(T, s.hidden_size, dtype=torch.float32, device="cuda")
    st.prefill_tokens(tok, rows, feats, h1, gw.pos, gw.cu, gw.n_seqs, gw.ds_rows, gw.ds_feats)
    h2 = torch.empty_like(h1)
    L.cc_op_embed_merge(tok, T, st.embed, s.vocab_size, s.hidden_size, rows, feats,
                        int(rows.numel()), h2)
    L.cc_op_sync()
    gw.prefill(h2)
    gw.sync()
    assert torch.equal(h1, h2)
    from oracle import decoder as OD
    h0 = OD.embed_merge(inp.token_ids, OD.from_storage(inp.embed), inp.mm_rows,
                        OD.from_storage(inp.mm_embeds))
    h_ref, _ = R.run_prefill(inp, hidden=h0)
    assert_close(as_numpy(h1), h_ref, TOL_MAX, TOL_MEAN, "hidden")


def test_causal_prefix_on_gpu():
    """First 48 logits of a 96-token prefill equal those of a 48-token prefill (pages'
    text_prefill_is_causal), here on the GPU path (3 sliding + 1 full layer)."""
    types = (SLIDING, SLIDING, SLIDING, FULL)
    a = _small("c96", [96], [], 0, types=types, window=20, head_rows="all", seed=24)
    b = _small("c48", [48], [], 0, types=types, window=20, head_rows="all", seed=24)
    # same weights by seed; the 48-token run takes the first 48 rows and the same final gain
    b._misc = dict(hidden=a.hidden[:48].copy(), final_ln=a.final_ln)
    _, ha, la = _run(a)
    _, hb, lb = _run(b)
    mx, _ = err_stats(as_numpy(la)[:48], as_numpy(lb))
    assert mx <= 1e-4, mx
    mx, _ = err_stats(as_numpy(ha)[:48], as_numpy(hb))
    assert mx <= 1e-4, mx


# ------------------------------------------------------------------------- the five workloads
def test_single_layer_fp32_T128():
    inp = Inputs(layer_fp32_T128())
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg, tol=(1e-4, 1e-5), lg_rel=1e-4)


def test_two_layer_pair_T2048():
    inp = Inputs(pair_T2048())
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg)


def _small_decode(seed=31, B=5, types=(SLIDING, FULL), window=70, heads=(8, 2)):
    shape = small_shape(num_layers=len(types), layer_types=types, window=window, heads=heads)
    wl = Workload("dec_small", shape, "decode", [], head_rows="all", seed=seed, decode_batch=B,
                  cache_len=150, page_size=16)
    return Inputs(wl)


def test_small_decode_step():
    inp = _small_decode()
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg)


def test_small_decode_step_q4():
    """The decode step and head on 4-bit affine weights (group 64) against the oracle run on
    the same weights dequantised and rounded to bf16."""
    inp = _small_decode(seed=37, B=7)
    gw = GpuWorkload(inp)
    gw.stack.attach_q4(inp.layer_q4, inp.embed_q4)
    h = gw.fresh_hidden()
    gw.stack.decode_q4(h, gw.pos, gw.seq_lens, gw.page_table, gw.max_pages, gw.kv)
    n = int(gw.head_rows.numel())
    lg = torch.empty(n, inp.shape.vocab_size, dtype=torch.float32, device="cuda")
    gw.stack.logits_q4(h, gw.head_rows, n, lg)
    gw.sync()
    h_ref, lg_ref = R.run_decode_q4(inp)
    assert_close(as_numpy(h), h_ref, TOL_MAX, TOL_MEAN, "hidden")
    lmx, _ = assert_close(as_numpy(lg), lg_ref, TOL_MAX, TOL_MEAN, "logits")
    assert lmx / np.abs(lg_ref).max() <= 2e-2
    # the bf16 and 4-bit weights differ, so must the results
    assert np.abs(as_numpy(h) - R.run_decode(inp)[0]).max() > 1e-2


def _graph_replay(gw, step):
    """step(hidden, logits) captured into a CUDA graph after one eager call (which sizes the
    plan's scratch), replayed on a fresh hidden state; returns (eager h, eager logits, replayed
    h, replayed logits)."""
    h_e = gw.fresh_hidden()
    lg_e = step(h_e, None)
    gw.sync()
    h = gw.fresh_hidden()
    lg = torch.empty_like(lg_e)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        step(h, lg)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):                       # replays start from the same input each time
        h.copy_(gw.hidden0)
        g.replay()
    torch.cuda.synchronize()
    gw.sync()
    return h_e, lg_e, h, lg


def test_decode_step_replays_from_a_cuda_graph():
    """The decode step and the head make no allocation and no host synchronisation once the
    plan's scratch fits the call: captured into a CUDA graph, a replay gives the eager results
    (up to the order of the split-K atomic adds into h)."""
    inp = _small_decode(seed=41, B=5)
    gw = GpuWorkload(inp)
    h_e, lg_e, h, lg = _graph_replay(gw, lambda hid, out: gw.step(hid, out))
    assert_close(as_numpy(h), as_numpy(h_e), 1e-4, 1e-6, "hidden (graph vs eager)")
    assert_close(as_numpy(lg), as_numpy(lg_e), 1e-4, 1e-6, "logits (graph vs eager)")
    gw.close()


def test_decode_step_q4_replays_from_a_cuda_graph():
    inp = _small_decode(seed=43, B=6)
    gw = GpuWorkload(inp)
    gw.stack.attach_q4(inp.layer_q4, inp.embed_q4)
    n = int(gw.head_rows.numel())

    def step(hid, out):
        if out is None:
            out = torch.empty(n, inp.shape.vocab_size, dtype=torch.float32, device="cuda")
        gw.stack.decode_q4(hid, gw.pos, gw.seq_lens, gw.page_table, gw.max_pages, gw.kv)
        gw.stack.logits_q4(hid, gw.head_rows, n, out)
        return out
    h_e, lg_e, h, lg = _graph_replay(gw, step)
    assert_close(as_numpy(h), as_numpy(h_e), 1e-4, 1e-6, "hidden (q4 graph vs eager)")
    assert_close(as_numpy(lg), as_numpy(lg_e), 1e-4, 1e-6, "logits (q4 graph vs eager)")
    gw.close()


def test_prefill_replays_from_a_cuda_graph():
    inp = _small("small_graph", [200, 77], [ImageSpan(0, 40, 1, 4, 6)], 2, seed=45)
    gw = GpuWorkload(inp)
    h_e, lg_e, h, lg = _graph_replay(gw, lambda hid, out: gw.step(hid, out))
    assert_close(as_numpy(h), as_numpy(h_e), 1e-4, 1e-6, "hidden (prefill graph vs eager)")
    assert_close(as_numpy(lg), as_numpy(lg_e), 1e-4, 1e-6, "logits (prefill graph vs eager)")
    gw.close()


def test_decode_step_B64_cache4096():
    inp = Inputs(decode_B64_cache4096())
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg)


def test_decode_step_q4_B64_cache4096():
    """The 4-bit decode step and head at the size the bench times (64 sequences x 4096 cached
    tokens, the two-layer pair, vocab 256000) against the oracle on the dequantised weights."""
    inp = Inputs(decode_B64_cache4096())
    gw = GpuWorkload(inp)
    gw.stack.attach_q4(inp.layer_q4, inp.embed_q4)
    h = gw.fresh_hidden()
    n = int(gw.head_rows.numel())
    lg = torch.empty(n, inp.shape.vocab_size, dtype=torch.float32, device="cuda")
    gw.stack.decode_q4(h, gw.pos, gw.seq_lens, gw.page_table, gw.max_pages, gw.kv)
    gw.stack.logits_q4(h, gw.head_rows, n, lg)
    gw.sync()
    h_ref, lg_ref = R.run_decode_q4(inp)
    assert_close(as_numpy(h), h_ref, TOL_MAX, TOL_MEAN, "hidden")
    lmx, _ = assert_close(as_numpy(lg), lg_ref, TOL_MAX, TOL_MEAN, "logits")
    assert lmx / np.abs(lg_ref).max() <= 2e-2
    gw.close()


def test_decode_continues_prefill_on_gpu():
    """Prefill of L tokens fills the paged cache; decoding token L+1 then matches the last
    row of an (L+1)-token prefill (both on the GPU)."""
    import cohere_compass_decoder_gb300._lib as L
    types = (SLIDING, FULL, SLIDING)
    Lc = 77
    full = _small("dcp_full", [Lc + 1], [ImageSpan(0, 10, 1, 3, 4)], 0, types=types, window=40,
                  head_rows="all", seed=41)
    gw_full, h_full, lg_full = _run(full)
    # same weights and inputs, first Lc tokens only, with a paged cache
    pre = _small("dcp_pre", [Lc], [ImageSpan(0, 10, 1, 3, 4)], 0, types=types, window=40,
                 head_rows="all", seed=41)
    gw = GpuWorkload(pre, max_tokens=Lc + 1)
    ps, max_pages = 16, (Lc + 1 + 15) // 16
    n_pages = max_pages + 3
    table = torch.tensor(np.random.default_rng(1).permutation(n_pages)[:max_pages][None, :],
                         dtype=torch.int32, device="cuda")
    shape = pre.shape
    kp = [torch.zeros(n_pages, shape.num_key_value_heads, ps, 128, dtype=torch.bfloat16,
                      device="cuda") for _ in types]
    vp = [torch.zeros_like(t) for t in kp]
    kv = L.make_kv_pool(kp, vp, n_pages)
    h = gw.fresh_hidden()
    gw.prefill(h, kv=kv, page_table=table, max_pages=max_pages)
    # the decode token: the (Lc+1)-th input row, position from rope_delta
    x = torch.from_numpy(full.hidden[Lc:Lc + 1].copy()).cuda()
    _, delta = L.cc_build_mrope_positions([(0, 10, 1, 3, 4)], [Lc])
    pos = torch.tensor(L.cc_build_decode_positions([Lc], delta), dtype=torch.int32, device="cuda")
    seq_lens = torch.tensor([Lc], dtype=torch.int32, device="cuda")
    gw.stack.decode(x, pos, seq_lens, table, max_pages, kv)
    gw.sync()
    mx, mn = err_stats(as_numpy(x)[0], as_numpy(h_full)[Lc])
    assert mx <= TOL_MAX and mn <= TOL_MEAN, (mx, mn)


def test_chunked_prefill_over_a_paged_prefix():
    """Two sequences prefilled in two chunks each (an image span crosses each boundary,
    deepstack rows on both sides): the first chunk fills the paged cache, the second
    continues it through cc_prefill_forward_chunk. Both chunks' rows equal the rows of the
    whole prefill (on the GPU and in the oracle)."""
    types = (SLIDING, FULL, SLIDING)
    lens, cut = [300, 200], [130, 77]
    imgs = [ImageSpan(0, 120, 1, 4, 6), ImageSpan(1, 60, 1, 5, 5), ImageSpan(1, 150, 1, 2, 3)]
    full = _small("chunked", lens, imgs, 1, types=types, window=90, head_rows="all", seed=43)
    gw, h_full, _ = _run(full)
    h_ref, _ = R.run_prefill(full)
    st = gw.stack
    s = full.shape
    starts = np.concatenate([[0], np.cumsum(lens)])
    rows1 = np.concatenate([np.arange(starts[i], starts[i] + cut[i]) for i in range(2)])
    rows2 = np.concatenate([np.arange(starts[i] + cut[i], starts[i + 1]) for i in range(2)])
    pos_full = gw.pos.cpu().numpy()
    ds_rows_full = full.ds_rows
    ps, max_pages = 16, (max(lens) + 15) // 16
    n_pages = 2 * max_pages + 3
    table = torch.tensor(np.random.default_rng(2).permutation(n_pages)[:2 * max_pages]
                         .reshape(2, max_pages), dtype=torch.int32, device="cuda")
    kp = [torch.zeros(n_pages, s.num_key_value_heads, ps, 128, dtype=torch.bfloat16,
                      device="cuda") for _ in types]
    vp = [torch.zeros_like(t) for t in kp]
    kv = L.make_kv_pool(kp, vp, n_pages)

    def chunk_inputs(rows, seq_lens):
        h = torch.from_numpy(full.hidden[rows].copy()).cuda()
        pos = torch.from_numpy(np.ascontiguousarray(pos_full[:, rows])).cuda()
        cu = torch.tensor(np.concatenate([[0], np.cumsum(seq_lens)]), dtype=torch.int32,
                          device="cuda")
        where = {int(r): k for k, r in enumerate(rows)}
        sel = [k for k, r in enumerate(ds_rows_full) if int(r) in where]
        ds_rows = torch.tensor([where[int(ds_rows_full[k])] for k in sel], dtype=torch.int32,
                               device="cuda")
        ds = [to_device(full.ds(0)[sel])]
        return h, pos, cu, ds_rows, ds

    h1, pos1, cu1, dr1, ds1 = chunk_inputs(rows1, cut)
    L.cc_prefill_forward(st.plan, h1, pos1, cu1, 2, len(rows1), dr1, int(dr1.numel()), ds1, kv,
                         table, max_pages)
    len2 = [lens[i] - cut[i] for i in range(2)]
    h2, pos2, cu2, dr2, ds2 = chunk_inputs(rows2, len2)
    prefix = torch.tensor(cut, dtype=torch.int32, device="cuda")
    L.cc_prefill_forward_chunk(st.plan, h2, pos2, cu2, 2, len(rows2), prefix, kv, table,
                               max_pages, dr2, int(dr2.numel()), ds2)
    st.sync()
    hf = as_numpy(h_full)
    for got, rows in ((h1, rows1), (h2, rows2)):
        assert_close(as_numpy(got), hf[rows], TOL_MAX, TOL_MEAN, "chunk vs whole prefill")
        assert_close(as_numpy(got), h_ref[rows], TOL_MAX, TOL_MEAN, "chunk vs oracle")


def test_prefill_from_token_ids_pair_T2048():
    """The token-id prefill (embedding merge fused with layer 0's LayerNorm) at the size the
    bench times: the two-layer pair, 2048 tokens, one 16x16 image, vocab 256000."""
    from oracle import decoder as OD
    inp = Inputs(pair_T2048())
    gw = GpuWorkload(inp)
    s = inp.shape
    T = inp.wl.total_tokens
    tok = torch.from_numpy(inp.token_ids).cuda()
    rows = torch.from_numpy(inp.mm_rows.astype(np.int32)).cuda()
    feats = to_device(inp.mm_embeds)
    h = torch.empty(T, s.hidden_size, dtype=torch.float32, device="cuda")
    gw.stack.prefill_tokens(tok, rows, feats, h, gw.pos, gw.cu, gw.n_seqs, gw.ds_rows, gw.ds_feats)
    gw.sync()
    h0 = OD.embed_merge(inp.token_ids, OD.from_storage(inp.embed), inp.mm_rows,
                        OD.from_storage(inp.mm_embeds))
    h_ref, _ = R.run_prefill(inp, hidden=h0)
    assert_close(as_numpy(h), h_ref, TOL_MAX, TOL_MEAN, "hidden")
    gw.close()


def test_chunked_prefill_pair_2048_after_2048():
    """The chunked prefill at the size the bench times: a 4096-token sequence of the two-layer
    pair, the first 2048 tokens prefilled into the paged cache, the next 2048 continuing them
    (an image span crosses the boundary); both chunks equal the rows of the oracle's whole
    prefill."""
    from synth.configs import SHAPE_PAIR
    T, cut = 4096, 2048
    inp = Inputs(Workload("pair_T4096_chunked", SHAPE_PAIR, "prefill", [T],
                          images=[ImageSpan(0, 300, 1, 16, 16), ImageSpan(0, 1900, 1, 16, 16)],
                          n_deepstack=1, head_rows="last", seed=47))
    h_ref, _ = R.run_prefill(inp)
    gw = GpuWorkload(inp, max_tokens=cut)
    st = gw.stack
    s = inp.shape
    ps, max_pages = 16, T // 16
    table = torch.tensor(np.random.default_rng(3).permutation(max_pages + 5)[:max_pages]
                         .reshape(1, max_pages), dtype=torch.int32, device="cuda")
    kp = [torch.zeros(max_pages + 5, s.num_key_value_heads, ps, 128, dtype=torch.bfloat16,
                      device="cuda") for _ in range(s.num_layers)]
    vp = [torch.zeros_like(t) for t in kp]
    kv = L.make_kv_pool(kp, vp, max_pages + 5)
    pos_full = gw.pos.cpu().numpy()
    ds_rows = inp.ds_rows

    def chunk(lo, hi):
        h = torch.from_numpy(inp.hidden[lo:hi].copy()).cuda()
        pos = torch.from_numpy(np.ascontiguousarray(pos_full[:, lo:hi])).cuda()
        cu = torch.tensor([0, hi - lo], dtype=torch.int32, device="cuda")
        sel = [k for k, r in enumerate(ds_rows) if lo <= int(r) < hi]
        dr = torch.tensor([int(ds_rows[k]) - lo for k in sel], dtype=torch.int32, device="cuda")
        ds = [to_device(inp.ds(0)[sel])]
        return h, pos, cu, dr, ds

    h1, pos1, cu1, dr1, ds1 = chunk(0, cut)
    L.cc_prefill_forward(st.plan, h1, pos1, cu1, 1, cut, dr1, int(dr1.numel()), ds1, kv, table,
                         max_pages)
    h2, pos2, cu2, dr2, ds2 = chunk(cut, T)
    prefix = torch.tensor([cut], dtype=torch.int32, device="cuda")
    L.cc_prefill_forward_chunk(st.plan, h2, pos2, cu2, 1, T - cut, prefix, kv, table, max_pages,
                               dr2, int(dr2.numel()), ds2)
    st.sync()
    assert_close(as_numpy(h1), h_ref[:cut], TOL_MAX, TOL_MEAN, "first chunk vs oracle")
    assert_close(as_numpy(h2), h_ref[cut:], TOL_MAX, TOL_MEAN, "second chunk vs oracle")
    gw.close()


@pytest.fixture(scope="module")
def stack28_oracle():
    """The 28-layer workload's inputs and the oracle's residual stream after every layer."""
    from oracle import decoder as O
    inp = Inputs(stack28_T8192())
    wl = inp.wl
    pos, _ = O.positions(wl.seq_lens, [(i.seq, i.start, i.grid_t, i.grid_h, i.grid_w)
                                       for i in wl.images])
    ds = [inp.ds(i) for i in range(wl.n_deepstack)]
    h, hs = O.prefill(inp.hidden, inp.layer, O.shape_dict(inp.shape), pos, inp.cu_seqlens,
                      inp.ds_rows, ds, True, return_all=True)
    lg = O.logits(h[inp.head_rows], inp.final_ln, inp.embed, O.shape_dict(inp.shape), True)
    return inp, hs, lg


class _OneLayer(Inputs):
    """Layer i of the 28-layer workload alone, fed with a given residual stream."""

    def __init__(self, base, i, hidden):
        import dataclasses
        shape = dataclasses.replace(base.shape, num_layers=1,
                                    layer_types=(base.shape.layer_types[i],), vocab_size=128)
        n_ds = 1 if i < base.wl.n_deepstack else 0
        super().__init__(dataclasses.replace(base.wl, shape=shape, n_deepstack=n_ds))
        self.base, self.i = base, i
        self._misc = dict(hidden=hidden.astype(np.float32), final_ln=base.final_ln)
        self._ds["embed"] = np.zeros((128, shape.hidden_size), np.uint16)

    def layer(self, j):
        return self.base.layer(self.i)

    def ds(self, j):
        return self.base.ds(self.i)


@pytest.mark.slow
def test_stack28_every_layer_from_oracle_input(stack28_oracle):
    """Each of the 28 layers (with its deepstack add) on the GPU, started from the oracle's
    residual stream before it, matches the oracle's stream after it within the stack
    tolerance (2e-2 max-abs, 2e-3 mean-abs)."""
    inp, hs, _ = stack28_oracle
    prev = inp.hidden.astype(np.float64)
    worst = []
    for i in range(inp.shape.num_layers):
        one = _OneLayer(inp, i, prev)
        gw = GpuWorkload(one)
        h = gw.fresh_hidden()
        gw.prefill(h)
        gw.sync()
        mx, mn = assert_close(as_numpy(h), hs[i], TOL_MAX, TOL_MEAN, f"layer {i}")
        worst.append((mx, mn))
        gw.close()
        prev = hs[i]
    print("per-layer max/mean:", worst)


@pytest.mark.slow
def test_stack28_T8192(stack28_oracle):
    """The whole 28-layer stack and the head, end to end, within a bound derived from the
    oracle alone (tests/golden/stack28_T8192_mirror_drift.txt, written by
    tests/golden/make_stack28_drift.py). Moving every input element by one float32 ulp (the
    resolution of the GPU's fp32 residual stream) flips some of the bf16 roundings the
    contract prescribes, and the oracle's own mirror result then drifts by a mean-abs that grows
    about linearly with depth, to the recorded floor after 28 layers; the GPU, whose fp32
    accumulation differs from the oracle's fp64 at every layer, sits on the same growth. Bound:
    1.25x the floor on the mean-abs and 1.5x on the max-abs (an extreme value over 16.8 M
    elements) of the final hidden state; the logits keep the benchmark spec's bound (2e-2 max-abs,
    2e-3 mean-abs) and 2% of their largest magnitude, twice the floor's 1%."""
    g = read_golden("stack28_T8192_mirror_drift.txt")
    inp, hs, lg_ref = stack28_oracle
    gw, h, lg = _run(inp)
    mx, mn = assert_close(as_numpy(h), hs[-1], 1.5 * g["fp32_ulp_hidden_max"][0],
                          1.25 * g["fp32_ulp_hidden_mean"][0], "hidden after 28 layers")
    lmx, _ = assert_close(as_numpy(lg), lg_ref, TOL_MAX, TOL_MEAN, "logits")
    rel = lmx / np.abs(lg_ref).max()
    print(f"hidden max {mx:.4g} mean {mn:.4g} (floor {g['fp32_ulp_hidden_max'][0]:.4g} / "
          f"{g['fp32_ulp_hidden_mean'][0]:.4g}); logits rel {rel:.4g}")
    assert rel <= 2e-2, f"logits relative error {rel:.3g}"


def test_pair_shapes_with_a_ragged_row_block_past_one_round():
    """The two-layer pair's shapes at T = 2610: 21 row blocks of 128 x 256 output tiles (the
    last one ragged) in the output projection with the fused next-layer LayerNorm, more row
    blocks than one round of tiles holds. The two row blocks past the first round (the ragged
    one, and image rows that take the deepstack add) run as 128-column tile halves."""
    from synth.configs import SHAPE_PAIR
    inp = Inputs(Workload("pair_T2610", SHAPE_PAIR, "prefill", [2610],
                          images=[ImageSpan(0, 2300, 1, 12, 16)], n_deepstack=1,
                          head_rows="last", seed=33))
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg)


def test_pair_shapes_with_a_last_round_more_than_half_full():
    """The two-layer pair's shapes at T = 3700: 29 row blocks (the last one ragged), 232 output
    tiles of 128 x 256 in the output projection with the fused next-layer LayerNorm. The
    second round holds 80 tiles on 152 CTAs, more than half, so it runs as whole tiles (as
    halves it would take two rounds of 128-column tiles); image rows there take the deepstack
    add."""
    from synth.configs import SHAPE_PAIR
    inp = Inputs(Workload("pair_T3700", SHAPE_PAIR, "prefill", [3700],
                          images=[ImageSpan(0, 3000, 1, 12, 16)], n_deepstack=1,
                          head_rows="last", seed=34))
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg)


@pytest.mark.slow
def test_varlen_T32768():
    inp = Inputs(varlen_T32768())
    gw, h, lg = _run(inp)
    _check(inp, gw, h, lg)
