"""ctypes binding of libcc.so: the C-ABI entry points under the same names.

Argument marshalling only: torch tensors (or raw integer addresses) become pointers,
Python sequences become ctypes arrays, and a non-OK status raises CCError. Every step
of the decoder runs in the library's CUDA kernels; nothing here computes.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcc.so")

CC_OK, CC_ERR_INVALID_ARG, CC_ERR_UNSUPPORTED, CC_ERR_OOM, CC_ERR_CUDA, CC_ERR_TIMEOUT, \
    CC_ERR_DEVICE_CHECK = range(7)
CC_SLIDING, CC_FULL = 0, 1
CC_F32, CC_BF16 = 0, 1
MROPE_LAYOUTS = ("interleaved", "sections_hwt")      # cc_mrope_layout values 0, 1

EXPORTS = [
    "cc_status_string", "cc_build_mrope_positions", "cc_build_decode_positions",
    "cc_pack_layer_weights", "cc_layer_plan_create", "cc_layer_plan_destroy",
    "cc_prefill_forward", "cc_decode_step", "cc_logits", "cc_sync", "cc_op_layernorm",
    "cc_op_mrope_table", "cc_op_gemm_bf16", "cc_op_attention_prefill",
    "cc_op_attention_decode", "cc_op_sync", "cc_profile_enable", "cc_profile_read",
    "cc_kernel_class_name", "cc_op_attention_decode_noalloc", "cc_prefill_forward_tokens",
    "cc_op_embed_merge", "cc_prefill_forward_chunk", "cc_q4_tiled_bytes", "cc_pack_q4_tiles",
    "cc_pack_layer_weights_q4", "cc_layer_plan_attach_q4", "cc_decode_step_q4", "cc_logits_q4",
    "cc_op_gemm_q4", "cc_op_mrope_table_layout", "cc_test_stall_next_gemm",
]
KERNEL_CLASSES = ["rope_table", "row_maps", "layernorm", "gemm_qkv_mlp", "attn_prefill",
                  "gemm_out_resid", "attn_decode", "gemm_head", "f32_path", "embed_merge"]


class CCError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class cc_model_config(C.Structure):
    _fields_ = [("num_layers", C.c_int32), ("hidden_size", C.c_int32),
                ("n_q_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("intermediate_size", C.c_int32),
                ("vocab_size", C.c_int32), ("sliding_window", C.c_int32),
                ("mrope_section", C.c_int32 * 3), ("kv_page_size", C.c_int32),
                ("max_tokens", C.c_int32), ("dtype", C.c_int32),
                ("layer_types", C.POINTER(C.c_int32)), ("rope_theta", C.c_double),
                ("layer_norm_eps", C.c_float), ("logit_scale", C.c_float),
                ("mrope_layout", C.c_int32)]


class cc_layer_weights(C.Structure):
    _fields_ = [("ln_w", C.c_void_p), ("w1", C.c_void_p), ("w2", C.c_void_p)]


class cc_layer_weights_q4(C.Structure):
    _fields_ = [("ln_w", C.c_void_p), ("w1", C.c_void_p), ("w2", C.c_void_p)]


class cc_kv_pool(C.Structure):
    _fields_ = [("k", C.POINTER(C.c_void_p)), ("v", C.POINTER(C.c_void_p)),
                ("n_pages", C.c_int32)]


class cc_kernel_time(C.Structure):
    _fields_ = [("launches", C.c_int32), ("total_ms", C.c_double)]


class cc_image_span(C.Structure):
    _fields_ = [("seq", C.c_int32), ("start", C.c_int32), ("grid_t", C.c_int32),
                ("grid_h", C.c_int32), ("grid_w", C.c_int32)]


_lib = None


def lib() -> C.CDLL:
    """The loaded library. Raises ImportError (loudly) when libcc.so has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it first with "
                              "`python -m cohere_compass_decoder_gb300.build`")
        L = C.CDLL(LIB_PATH)
        vp, i32, p32 = C.c_void_p, C.c_int32, C.POINTER(C.c_int32)
        sig = {
            "cc_status_string": (C.c_char_p, [C.c_int]),
            "cc_build_mrope_positions": (C.c_int, [C.POINTER(cc_image_span), i32, p32, i32, p32, p32]),
            "cc_build_decode_positions": (C.c_int, [p32, p32, i32, p32]),
            "cc_pack_layer_weights": (C.c_int, [C.POINTER(cc_model_config)] + [vp] * 10),
            "cc_layer_plan_create": (C.c_int, [C.POINTER(cc_model_config),
                                               C.POINTER(cc_layer_weights), vp, vp,
                                               C.POINTER(vp)]),
            "cc_layer_plan_destroy": (None, [vp]),
            "cc_prefill_forward": (C.c_int, [vp, vp, vp, vp, i32, i32, vp, i32,
                                             C.POINTER(vp), i32, C.POINTER(cc_kv_pool), vp,
                                             i32, vp]),
            "cc_prefill_forward_tokens": (C.c_int, [vp, vp, vp, vp, i32, vp, vp, vp, i32, i32, vp,
                                                    i32, C.POINTER(vp), i32,
                                                    C.POINTER(cc_kv_pool), vp, i32, vp]),
            "cc_prefill_forward_chunk": (C.c_int, [vp, vp, vp, vp, i32, i32, vp, vp, i32,
                                                   C.POINTER(vp), i32, C.POINTER(cc_kv_pool), vp,
                                                   i32, vp]),
            "cc_decode_step": (C.c_int, [vp, vp, vp, vp, vp, i32, i32, C.POINTER(cc_kv_pool), vp]),
            "cc_logits": (C.c_int, [vp, vp, vp, i32, vp, vp]),
            "cc_sync": (C.c_int, [vp, vp]),
            "cc_q4_tiled_bytes": (C.c_size_t, [i32, i32]),
            "cc_pack_q4_tiles": (C.c_int, [vp, vp, vp, i32, i32, vp, vp]),
            "cc_pack_layer_weights_q4": (C.c_int, [C.POINTER(cc_model_config), C.POINTER(vp),
                                                   C.POINTER(vp), C.POINTER(vp), vp, vp, vp]),
            "cc_layer_plan_attach_q4": (C.c_int, [vp, C.POINTER(cc_layer_weights_q4), vp]),
            "cc_decode_step_q4": (C.c_int, [vp, vp, vp, vp, vp, i32, i32, C.POINTER(cc_kv_pool),
                                            vp]),
            "cc_logits_q4": (C.c_int, [vp, vp, vp, i32, vp, vp]),
            "cc_op_gemm_q4": (C.c_int, [vp, vp, vp, i32, i32, i32, C.c_float, i32, vp]),
            "cc_op_layernorm": (C.c_int, [vp, vp, vp, i32, i32, C.c_float, vp, vp]),
            "cc_op_embed_merge": (C.c_int, [vp, i32, vp, i32, i32, vp, vp, i32, vp, vp, C.c_float,
                                            vp, vp]),
            "cc_op_mrope_table": (C.c_int, [vp, i32, i32, C.c_double, p32, vp, vp]),
            "cc_op_mrope_table_layout": (C.c_int, [vp, i32, i32, C.c_double, p32, i32, vp, vp]),
            "cc_op_gemm_bf16": (C.c_int, [vp, vp, vp, i32, i32, i32, C.c_float, i32, vp]),
            "cc_op_attention_prefill": (C.c_int, [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                                  i32, vp]),
            "cc_op_attention_decode": (C.c_int, [vp, vp, vp, i32, vp, i32, vp, i32, i32, i32,
                                                 i32, i32, vp, i32, vp]),
            "cc_op_sync": (C.c_int, [vp]),
            "cc_op_attention_decode_noalloc": (C.c_int, [vp, vp, vp, i32, vp, i32, vp, i32, i32,
                                                         i32, i32, i32, vp, i32, vp, vp]),
            "cc_profile_enable": (C.c_int, [vp, i32]),
            "cc_profile_read": (C.c_int, [vp, C.POINTER(cc_kernel_time)]),
            "cc_kernel_class_name": (C.c_char_p, [i32]),
            "cc_test_stall_next_gemm": (None, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# ------------------------------------------------------------------------ marshalling
def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status, where):
    if status != CC_OK:
        raise CCError(status, where)


def status_string(status: int) -> str:
    return lib().cc_status_string(status).decode()


def _i32_array(values):
    arr = (C.c_int32 * len(values))(*[int(v) for v in values])
    return arr


# ------------------------------------------------------------------------ host helpers
def cc_build_mrope_positions(spans, seq_lens):
    """spans: iterable of (seq, start, grid_t, grid_h, grid_w); returns (pos [3][T] list of
    lists, rope_delta list). Host-only call (no GPU needed)."""
    spans = list(spans)
    sp = (cc_image_span * max(1, len(spans)))()
    for i, s in enumerate(spans):
        sp[i] = cc_image_span(*[int(v) for v in s])
    lens = _i32_array(seq_lens)
    T = int(sum(int(x) for x in seq_lens))
    pos = (C.c_int32 * max(1, 3 * T))()
    delta = (C.c_int32 * max(1, len(lens)))()
    st = lib().cc_build_mrope_positions(sp, len(spans), lens, len(lens), pos, delta)
    _check(st, "cc_build_mrope_positions")
    flat = list(pos)[:3 * T]
    return [flat[0:T], flat[T:2 * T], flat[2 * T:3 * T]], list(delta)[:len(lens)]


def cc_build_decode_positions(seq_lens, rope_delta):
    B = len(seq_lens)
    pos = (C.c_int32 * max(1, 3 * B))()
    st = lib().cc_build_decode_positions(_i32_array(seq_lens), _i32_array(rope_delta), B, pos)
    _check(st, "cc_build_decode_positions")
    flat = list(pos)[:3 * B]
    return [flat[0:B], flat[B:2 * B], flat[2 * B:3 * B]]


# ------------------------------------------------------------------------ plan API
def make_config(shape, max_tokens, page_size=16):
    """cc_model_config from an object with the model hyper-parameters (see synth.configs).
    The returned struct keeps its layer_types array alive."""
    types = _i32_array([CC_SLIDING if t == "sliding_attention" else CC_FULL
                        for t in shape.layer_types])
    cfg = cc_model_config()
    cfg.num_layers = shape.num_layers
    cfg.hidden_size = shape.hidden_size
    cfg.n_q_heads = shape.num_attention_heads
    cfg.n_kv_heads = shape.num_key_value_heads
    cfg.head_dim = shape.head_dim
    cfg.intermediate_size = shape.intermediate_size
    cfg.vocab_size = shape.vocab_size
    cfg.sliding_window = shape.sliding_window
    cfg.mrope_section = (C.c_int32 * 3)(*shape.mrope_section)
    cfg.kv_page_size = page_size
    cfg.max_tokens = max_tokens
    cfg.dtype = CC_BF16 if shape.dtype == "bf16" else CC_F32
    cfg.layer_types = C.cast(types, C.POINTER(C.c_int32))
    cfg.rope_theta = float(shape.rope_theta)
    cfg.layer_norm_eps = float(shape.layer_norm_eps)
    cfg.logit_scale = float(shape.logit_scale)
    cfg.mrope_layout = MROPE_LAYOUTS.index(getattr(shape, "mrope_layout", "interleaved"))
    cfg._keep = types
    return cfg


def cc_pack_layer_weights(cfg, wq, wk, wv, wo, wg, wu, wd, w1_out, w2_out, stream=None):
    st = lib().cc_pack_layer_weights(C.byref(cfg), *[_ptr(t) for t in (wq, wk, wv, wo, wg, wu, wd,
                                                                       w1_out, w2_out)],
                                     _stream(stream))
    _check(st, "cc_pack_layer_weights")


def cc_layer_plan_create(cfg, layers, final_ln_w, embed):
    """layers: sequence of (ln_w, w1, w2) tensors. Returns the plan handle (int)."""
    arr = (cc_layer_weights * len(layers))()
    for i, (ln, w1, w2) in enumerate(layers):
        arr[i] = cc_layer_weights(_ptr(ln), _ptr(w1), _ptr(w2))
    out = C.c_void_p()
    st = lib().cc_layer_plan_create(C.byref(cfg), arr, _ptr(final_ln_w), _ptr(embed), C.byref(out))
    _check(st, "cc_layer_plan_create")
    return out.value


def cc_layer_plan_destroy(plan):
    if plan:
        lib().cc_layer_plan_destroy(plan)


def make_kv_pool(k_list, v_list, n_pages):
    ka = (C.c_void_p * len(k_list))(*[_ptr(t) for t in k_list])
    va = (C.c_void_p * len(v_list))(*[_ptr(t) for t in v_list])
    pool = cc_kv_pool(C.cast(ka, C.POINTER(C.c_void_p)), C.cast(va, C.POINTER(C.c_void_p)),
                      int(n_pages))
    pool._keep = (ka, va)
    return pool


def cc_prefill_forward(plan, hidden, pos_thw, cu_seqlens, n_seqs, total_tokens, ds_rows=None,
                       n_ds_rows=0, ds_feats=(), kv=None, page_table=None, max_pages=0,
                       stream=None):
    feats = (C.c_void_p * max(1, len(ds_feats)))(*[_ptr(t) for t in ds_feats])
    st = lib().cc_prefill_forward(plan, _ptr(hidden), _ptr(pos_thw), _ptr(cu_seqlens), n_seqs,
                                  total_tokens, _ptr(ds_rows), n_ds_rows, feats, len(ds_feats),
                                  C.byref(kv) if kv is not None else None, _ptr(page_table),
                                  max_pages, _stream(stream))
    _check(st, "cc_prefill_forward")


def cc_prefill_forward_tokens(plan, token_ids, mm_rows, mm_embeds, n_mm_rows, hidden, pos_thw,
                              cu_seqlens, n_seqs, total_tokens, ds_rows=None, n_ds_rows=0,
                              ds_feats=(), kv=None, page_table=None, max_pages=0, stream=None):
    feats = (C.c_void_p * max(1, len(ds_feats)))(*[_ptr(t) for t in ds_feats])
    st = lib().cc_prefill_forward_tokens(plan, _ptr(token_ids), _ptr(mm_rows), _ptr(mm_embeds),
                                         n_mm_rows, _ptr(hidden), _ptr(pos_thw), _ptr(cu_seqlens),
                                         n_seqs, total_tokens, _ptr(ds_rows), n_ds_rows, feats,
                                         len(ds_feats),
                                         C.byref(kv) if kv is not None else None,
                                         _ptr(page_table), max_pages, _stream(stream))
    _check(st, "cc_prefill_forward_tokens")


def cc_prefill_forward_chunk(plan, hidden, pos_thw, cu_seqlens, n_seqs, total_tokens, prefix_lens,
                             kv, page_table, max_pages, ds_rows=None, n_ds_rows=0, ds_feats=(),
                             stream=None):
    feats = (C.c_void_p * max(1, len(ds_feats)))(*[_ptr(t) for t in ds_feats])
    st = lib().cc_prefill_forward_chunk(plan, _ptr(hidden), _ptr(pos_thw), _ptr(cu_seqlens), n_seqs,
                                        total_tokens, _ptr(prefix_lens), _ptr(ds_rows), n_ds_rows,
                                        feats, len(ds_feats), C.byref(kv), _ptr(page_table),
                                        max_pages, _stream(stream))
    _check(st, "cc_prefill_forward_chunk")


def cc_decode_step(plan, hidden, pos_thw, seq_lens, page_table, max_pages, batch, kv,
                   stream=None):
    st = lib().cc_decode_step(plan, _ptr(hidden), _ptr(pos_thw), _ptr(seq_lens),
                              _ptr(page_table), max_pages, batch, C.byref(kv), _stream(stream))
    _check(st, "cc_decode_step")


def cc_logits(plan, hidden, rows, n_rows, logits, stream=None):
    st = lib().cc_logits(plan, _ptr(hidden), _ptr(rows), n_rows, _ptr(logits), _stream(stream))
    _check(st, "cc_logits")


def cc_q4_tiled_bytes(rows, k):
    return int(lib().cc_q4_tiled_bytes(rows, k))


def cc_pack_q4_tiles(words, scales, biases, rows, k, out, stream=None):
    _check(lib().cc_pack_q4_tiles(_ptr(words), _ptr(scales), _ptr(biases), rows, k, _ptr(out),
                                  _stream(stream)), "cc_pack_q4_tiles")


def cc_pack_layer_weights_q4(cfg, packed, scales, biases, w1_out, w2_out, stream=None):
    """packed / scales / biases: 7 tensors each, in the order q, k, v, o, gate, up, down."""
    arrs = [(C.c_void_p * 7)(*[_ptr(t) for t in group]) for group in (packed, scales, biases)]
    st = lib().cc_pack_layer_weights_q4(C.byref(cfg), *arrs, _ptr(w1_out), _ptr(w2_out),
                                        _stream(stream))
    _check(st, "cc_pack_layer_weights_q4")


def cc_layer_plan_attach_q4(plan, layers, embed_q4):
    """layers: sequence of (ln_w, w1, w2) tensors (tiled 4-bit weights)."""
    arr = (cc_layer_weights_q4 * len(layers))()
    for i, t in enumerate(layers):
        arr[i] = cc_layer_weights_q4(*[_ptr(x) for x in t])
    _check(lib().cc_layer_plan_attach_q4(plan, arr, _ptr(embed_q4)), "cc_layer_plan_attach_q4")


def cc_decode_step_q4(plan, hidden, pos_thw, seq_lens, page_table, max_pages, batch, kv,
                      stream=None):
    st = lib().cc_decode_step_q4(plan, _ptr(hidden), _ptr(pos_thw), _ptr(seq_lens),
                                 _ptr(page_table), max_pages, batch, C.byref(kv), _stream(stream))
    _check(st, "cc_decode_step_q4")


def cc_logits_q4(plan, hidden, rows, n_rows, logits, stream=None):
    st = lib().cc_logits_q4(plan, _ptr(hidden), _ptr(rows), n_rows, _ptr(logits), _stream(stream))
    _check(st, "cc_logits_q4")


def cc_sync(plan, stream=None):
    _check(lib().cc_sync(plan, _stream(stream)), "cc_sync")


def cc_test_stall_next_gemm():
    """Test hook: the next bf16 GEMM launch takes its bounded-wait timeout path."""
    lib().cc_test_stall_next_gemm()


# ------------------------------------------------------------------------ single ops
def cc_op_sync(stream=None):
    _check(lib().cc_op_sync(_stream(stream)), "cc_op_sync")


def cc_op_layernorm(x, gamma, out, rows, hidden, eps, row_idx=None, stream=None):
    _check(lib().cc_op_layernorm(_ptr(x), _ptr(gamma), _ptr(out), rows, hidden, eps, _ptr(row_idx),
                                 _stream(stream)), "cc_op_layernorm")


def cc_op_mrope_table(pos, tokens, head_dim, theta, section, table, stream=None):
    _check(lib().cc_op_mrope_table(_ptr(pos), tokens, head_dim, float(theta), _i32_array(section),
                                   _ptr(table), _stream(stream)), "cc_op_mrope_table")


def cc_op_mrope_table_layout(pos, tokens, head_dim, theta, section, layout, table, stream=None):
    _check(lib().cc_op_mrope_table_layout(_ptr(pos), tokens, head_dim, float(theta),
                                          _i32_array(section), MROPE_LAYOUTS.index(layout),
                                          _ptr(table), _stream(stream)),
           "cc_op_mrope_table_layout")


def cc_op_gemm_bf16(a, b, c, m, n, k, alpha=1.0, accumulate=0, stream=None):
    _check(lib().cc_op_gemm_bf16(_ptr(a), _ptr(b), _ptr(c), m, n, k, alpha, accumulate,
                                 _stream(stream)), "cc_op_gemm_bf16")


def cc_op_gemm_q4(a, w_tiled, c, m, n, k, alpha=1.0, accumulate=0, stream=None):
    _check(lib().cc_op_gemm_q4(_ptr(a), _ptr(w_tiled), _ptr(c), m, n, k, alpha, accumulate,
                               _stream(stream)), "cc_op_gemm_q4")


def cc_op_embed_merge(token_ids, tokens, embed, vocab, hidden_size, mm_rows, mm_embeds,
                      n_mm_rows, hidden, ln_w=None, eps=1e-5, ln_out=None, stream=None):
    _check(lib().cc_op_embed_merge(_ptr(token_ids), tokens, _ptr(embed), vocab, hidden_size,
                                   _ptr(mm_rows), _ptr(mm_embeds), n_mm_rows, _ptr(hidden),
                                   _ptr(ln_w), eps, _ptr(ln_out), _stream(stream)),
           "cc_op_embed_merge")


def cc_op_attention_prefill(q, k, v, out, ld_out, cu_seqlens, n_seqs, tokens, n_q, n_kv, window,
                            stream=None):
    _check(lib().cc_op_attention_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(out), ld_out,
                                         _ptr(cu_seqlens), n_seqs, tokens, n_q, n_kv, window,
                                         _stream(stream)), "cc_op_attention_prefill")


def cc_op_attention_decode(q, k_pool, v_pool, n_pages, page_table, max_pages, n_keys, batch, n_q,
                           n_kv, page_size, window, out, ld_out, stream=None):
    _check(lib().cc_op_attention_decode(_ptr(q), _ptr(k_pool), _ptr(v_pool), n_pages,
                                        _ptr(page_table), max_pages, _ptr(n_keys), batch, n_q, n_kv,
                                        page_size, window, _ptr(out), ld_out, _stream(stream)),
           "cc_op_attention_decode")


def cc_op_attention_decode_noalloc(q, k_pool, v_pool, n_pages, page_table, max_pages, n_keys,
                                   batch, n_q, n_kv, page_size, window, out, ld_out,
                                   err_flag=None, stream=None):
    """Decode attention with the library's fixed scratch: allocates no device memory."""
    _check(lib().cc_op_attention_decode_noalloc(_ptr(q), _ptr(k_pool), _ptr(v_pool), n_pages,
                                                _ptr(page_table), max_pages, _ptr(n_keys), batch,
                                                n_q, n_kv, page_size, window, _ptr(out), ld_out,
                                                _ptr(err_flag), _stream(stream)),
           "cc_op_attention_decode_noalloc")


# ------------------------------------------------------------------------ profiling
def cc_profile_enable(plan, enable=True):
    _check(lib().cc_profile_enable(plan, 1 if enable else 0), "cc_profile_enable")


def cc_profile_read(plan):
    """{kernel class name: (launches, total ms)} since the last read."""
    arr = (cc_kernel_time * len(KERNEL_CLASSES))()
    _check(lib().cc_profile_read(plan, arr), "cc_profile_read")
    return {lib().cc_kernel_class_name(i).decode(): (arr[i].launches, arr[i].total_ms)
            for i in range(len(KERNEL_CLASSES))}
