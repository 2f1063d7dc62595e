/*
 * cc.h -- C-ABI of the GB300 (sm_103a) Compass-style parallel decoder stack.
 *
 * The library computes the forward pass of the Cohere2/Compass parallel decoder layer
 * stack over a merged image+text sequence, as defined by the mlxcel issue
 * "feat(vlm): add Cohere Compass / North-Micro-Vision (cohere_compass) VLM", section
 * "Text decoder forward":
 *
 *   for each layer i:  a = LayerNorm_i(h)                      (weight only, f32 statistics)
 *                      h = h + Attn_i(a) + SwiGLU_i(a)         (parallel block, no post-norm)
 *                      if i < n_deepstack: h[image rows] += deepstack[i]
 *   logits = logit_scale * (LayerNorm_f(h) @ embed^T)          (tied head)
 *
 * Sliding layers rotate q and k with the interleaved 3-axis MRoPE (split rotate-half)
 * and attend causally over the last `sliding_window` keys; full layers use no position
 * encoding and plain causal attention. Attention is grouped-query (query head h reads
 * KV head h / (n_q / n_kv)) with scale head_dim^-0.5.
 *
 * Conventions for every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller unless the comment says
 *    "host". Matrices are row-major and dense (leading dimension = row length) unless a
 *    leading dimension is passed.
 *  - `stream` is a cudaStream_t passed as void*; every call is stream-ordered and
 *    asynchronous (no host synchronisation), except the host helpers.
 *  - Errors found on the host return a status and launch nothing. Errors found on the
 *    device (a bounded wait that ran out, a bad index) set a sticky device flag that
 *    cc_sync / cc_op_sync returns; the results of the affected calls are undefined.
 *  - No call aborts the process or throws across the ABI.
 *  - bf16 tensors hold raw bfloat16 bit patterns; f32 tensors hold IEEE floats.
 *  - A process drives the library on one CUDA device: each kernel's shared-memory limit
 *    is configured once, on the device current at its first launch. Calls on one plan
 *    come from one host thread at a time (they reuse the plan's workspace).
 */
#ifndef CC_H_
#define CC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CC_OK = 0,
  CC_ERR_INVALID_ARG = 1,   /* a host-detectable argument error                       */
  CC_ERR_UNSUPPORTED = 2,   /* a valid configuration this build does not implement    */
  CC_ERR_OOM = 3,           /* device allocation failed                               */
  CC_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch, copy, attribute)    */
  CC_ERR_TIMEOUT = 5,       /* device: a bounded inter-warp wait gave up              */
  CC_ERR_DEVICE_CHECK = 6   /* device: an index check failed (page id, row map)       */
} cc_status;

typedef enum { CC_SLIDING = 0, CC_FULL = 1 } cc_layer_type;
typedef enum { CC_F32 = 0, CC_BF16 = 1 } cc_dtype;

/* Which rotary index reads which position axis at which frequency (the half-dimension index
 * k < head_dim/2, inv_freq[j] = theta^(-2j/head_dim)):
 *  CC_MROPE_INTERLEAVED   mlxcel issue, "Text decoder forward", interleaved MRoPE: k reads
 *                         axis h when k % 3 == 1 and k < 3 section[1], w when k % 3 == 2 and
 *                         k < 3 section[2], else t, at frequency k.
 *  CC_MROPE_SECTIONS_HWT  the same issue's acceptance notes (the RoPE correction): contiguous
 *                         [H, W, T] sections with pre-permuted inv_freq. The permutation is
 *                         not on the pages; read as: the H section (section[1] indices) takes,
 *                         in increasing order, the frequencies the interleaved rule sends to h,
 *                         then W (section[2]) those sent to w, then T the rest. */
typedef enum { CC_MROPE_INTERLEAVED = 0, CC_MROPE_SECTIONS_HWT = 1 } cc_mrope_layout;

/* Model hyper-parameters: the text_config keys of the Compass checkpoint (mlxcel issue,
 * "Config (config.json)" and "Text decoder forward"). `layer_types` points to
 * num_layers entries of cc_layer_type and is copied by cc_layer_plan_create.
 * Requirements (else CC_ERR_INVALID_ARG): mrope_section sums to head_dim/2;
 * n_q_heads % n_kv_heads == 0; sliding_window > 0; all sizes > 0.
 * All plans need hidden_size a multiple of 128 and at most 4096, intermediate_size a
 * multiple of 64 (else CC_ERR_UNSUPPORTED). bf16 plans also need head_dim == 128,
 * vocab_size a multiple of 128, kv_page_size == 16 and n_q / n_kv one of 1, 2, 4, 8, 16.
 * f32 plans need head_dim <= 128. */
typedef struct {
  int32_t num_layers;
  int32_t hidden_size;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t intermediate_size;
  int32_t vocab_size;
  int32_t sliding_window;
  int32_t mrope_section[3];   /* frequencies on the t, h, w axes                        */
  int32_t kv_page_size;       /* tokens per KV page (paged cache), e.g. 16              */
  int32_t max_tokens;         /* largest token count of one call; sizes the workspace   */
  int32_t dtype;              /* cc_dtype of weights and stored activations             */
  const int32_t* layer_types; /* host [num_layers]                                     */
  double rope_theta;
  float layer_norm_eps;
  float logit_scale;
  int32_t mrope_layout;       /* cc_mrope_layout (0: interleaved)                        */
} cc_model_config;

/* One layer's weights, packed by cc_pack_layer_weights:
 *  ln_w [H]                    LayerNorm gain
 *  w1   [N1, H], N1 = (n_q + 2 n_kv) d + 2 I: rows q | k | v | then the SwiGLU gate and
 *       up rows interleaved in blocks of 64 (gate 0..63, up 0..63, gate 64..127, ...)
 *  w2   [H, K2], K2 = n_q d + I: columns o_proj | down_proj
 * The plan borrows these pointers; they must outlive it. */
typedef struct {
  const void* ln_w;
  const void* w1;
  const void* w2;
} cc_layer_weights;

/* Paged KV cache of every layer: k[i], v[i] point to [n_pages, n_kv, page_size, head_dim]
 * bf16 pools (caller-owned, host array of device pointers, num_layers entries each).
 * Keys are stored after rotation (sliding layers) or as projected (full layers).
 * Token t of sequence b lives in page page_table[b * max_pages + t / page_size], slot
 * t % page_size. */
typedef struct {
  void* const* k;
  void* const* v;
  int32_t n_pages;
} cc_kv_pool;

/* One image inside a packed batch: merged grid (t, h, w) occupying t*h*w consecutive
 * tokens of sequence `seq`, starting at token offset `start` of that sequence. */
typedef struct {
  int32_t seq;
  int32_t start;
  int32_t grid_t;
  int32_t grid_h;
  int32_t grid_w;
} cc_image_span;

typedef struct cc_layer_plan cc_layer_plan;

/* ---------------------------------------------------------------------------------- */
const char* cc_status_string(cc_status s);

/* Host helper (no device work). Position ids of packed sequences, mlxcel issue
 * "Text decoder forward", paragraph "Position ids (get_rope_index)": text tokens take
 * max(previous positions)+1 on all three axes (0 for a sequence's first token); the
 * t*h*w tokens of an image take offset + (t_idx, h_idx, w_idx) in row-major grid order,
 * offset = max(previous positions)+1; rope_delta = max position + 1 - length.
 * seq_lens: host [n_seqs]; spans: host [n_spans] (any order, must not overlap or leave
 * their sequence); pos_out: host [3, sum(seq_lens)] (t row, h row, w row);
 * rope_delta_out: host [n_seqs]. Bit-exact integer arithmetic. */
cc_status cc_build_mrope_positions(const cc_image_span* spans, int32_t n_spans,
                                   const int32_t* seq_lens, int32_t n_seqs,
                                   int32_t* pos_out, int32_t* rope_delta_out);

/* Host helper: decode position of each sequence's new token, offset + rope_delta on all
 * three axes (same paragraph). seq_lens/rope_delta host [batch]; pos_out host [3, batch]. */
cc_status cc_build_decode_positions(const int32_t* seq_lens, const int32_t* rope_delta,
                                    int32_t batch, int32_t* pos_out);

/* Packs one layer's projection matrices into the w1/w2 layout of cc_layer_weights
 * (device-to-device copies on `stream`). Inputs are the checkpoint's [out, in] matrices:
 * wq [n_q d, H], wk/wv [n_kv d, H], wo [H, n_q d], wg/wu [I, H], wd [H, I].
 * w1_out [N1, H] and w2_out [H, K2] are caller-allocated. Element size from cfg->dtype. */
cc_status cc_pack_layer_weights(const cc_model_config* cfg, const void* wq, const void* wk,
                                const void* wv, const void* wo, const void* wg,
                                const void* wu, const void* wd, void* w1_out, void* w2_out,
                                void* stream);

/* Creates a plan: copies cfg and layer_types, borrows the weights (layers[num_layers],
 * final_ln_w [H], embed [V, H], the tied embedding used as the LM head), allocates its
 * device workspace for cfg->max_tokens tokens and builds the weight TMA descriptors.
 * Uses the current CUDA device. On error *out is NULL. */
cc_status cc_layer_plan_create(const cc_model_config* cfg, const cc_layer_weights* layers,
                               const void* final_ln_w, const void* embed,
                               cc_layer_plan** out);
void cc_layer_plan_destroy(cc_layer_plan* plan);

/* Prefill forward over packed sequences; updates hidden in place.
 *  hidden      f32 [T, H] residual stream (input embeddings in, final h out; not normed)
 *  pos_thw     int32 [3, T] position ids (cc_build_mrope_positions)
 *  cu_seqlens  int32 [n_seqs + 1], cu_seqlens[0] = 0, non-decreasing, last = T
 *  ds_rows     int32 [n_ds_rows] token rows of the image tokens (distinct), may be NULL
 *              when n_deepstack == 0
 *  ds_feats    host array of n_deepstack device pointers, each [n_ds_rows, H] in the
 *              plan's dtype; tensor i is added after layer i (n_deepstack <= num_layers)
 *  kv          optional paged cache to fill with every token's K/V (NULL: none);
 *  page_table  int32 [n_seqs, max_pages] when kv is given
 * T <= max_tokens. The last CTA of every row-tile is bounded by T; no host sync. */
cc_status cc_prefill_forward(cc_layer_plan* plan, float* hidden, const int32_t* pos_thw,
                             const int32_t* cu_seqlens, int32_t n_seqs, int32_t total_tokens,
                             const int32_t* ds_rows, int32_t n_ds_rows,
                             const void* const* ds_feats, int32_t n_deepstack,
                             const cc_kv_pool* kv, const int32_t* page_table,
                             int32_t max_pages, void* stream);

/* The step before the path fused with it: cc_prefill_forward starting from token ids.
 * The embedding merge (Compass issue, "Text decoder forward": h = embed_tokens(tokens);
 * mlxcel VLM manual "Stage 4: Embedding Merge" and FreeToken PR 454 "How it fits together":
 * the image placeholder rows take the projected vision features, given as a row list and
 * the gathered features) runs in one kernel with layer 0's LayerNorm, then the stack runs
 * as in cc_prefill_forward.
 *  token_ids int32 [T] in [0, vocab) (device); mm_rows int32 [n_mm_rows] distinct rows in
 *  [0, T) and mm_embeds bf16 [n_mm_rows, H] (both NULL when n_mm_rows == 0); hidden f32
 *  [T, H] receives h (it is not read). The other arguments are those of cc_prefill_forward.
 * bf16 plans only (CC_ERR_UNSUPPORTED otherwise). A token id outside the vocabulary or an
 * image row outside [0, T) sets the device error flag (cc_sync); that row's h is zero. */
cc_status cc_prefill_forward_tokens(cc_layer_plan* plan, const int32_t* token_ids,
                                    const int32_t* mm_rows, const void* mm_embeds,
                                    int32_t n_mm_rows, float* hidden, const int32_t* pos_thw,
                                    const int32_t* cu_seqlens, int32_t n_seqs,
                                    int32_t total_tokens, const int32_t* ds_rows,
                                    int32_t n_ds_rows, const void* const* ds_feats,
                                    int32_t n_deepstack, const cc_kv_pool* kv,
                                    const int32_t* page_table, int32_t max_pages, void* stream);

/* Chunked prefill (the step after a prefill chunk, before decode): as cc_prefill_forward,
 * but the tokens of sequence s continue prefix_lens[s] keys already in the paged cache,
 * at positions prefix_lens[s] .. prefix_lens[s] + L_s - 1 (pos_thw holds their absolute
 * position ids, e.g. the slice of the whole sequence's ids, so an image span may cross the
 * chunk boundary). Their keys and values are written to the cache at those slots and every
 * query attends over the cached keys it sees (causal, window on sliding layers) through the
 * page table; the result equals the rows of a prefill of the whole sequences.
 *  prefix_lens int32 [n_seqs] (device); kv and page_table required,
 *  prefix_lens[s] + L_s <= max_pages * 16. bf16 plans with head_dim 128 and 16-token pages
 *  only (CC_ERR_UNSUPPORTED otherwise). */
cc_status cc_prefill_forward_chunk(cc_layer_plan* plan, float* hidden, const int32_t* pos_thw,
                                   const int32_t* cu_seqlens, int32_t n_seqs,
                                   int32_t total_tokens, const int32_t* prefix_lens,
                                   const int32_t* ds_rows, int32_t n_ds_rows,
                                   const void* const* ds_feats, int32_t n_deepstack,
                                   const cc_kv_pool* kv, const int32_t* page_table,
                                   int32_t max_pages, void* stream);

/* One decode step: one new token per sequence.
 *  hidden    f32 [batch, H] (in: the new tokens' embeddings; out: final h)
 *  pos_thw   int32 [3, batch] (cc_build_decode_positions)
 *  seq_lens  int32 [batch] tokens already cached; the new token's K/V are written at
 *            slot seq_lens[b] and it attends over seq_lens[b] + 1 keys (sliding layers:
 *            the last sliding_window of them). seq_lens[b] + 1 <= max_pages * page_size.
 *  page_table int32 [batch, max_pages]; kv the cache (required). The caller advances
 *  seq_lens afterwards. */
cc_status cc_decode_step(cc_layer_plan* plan, float* hidden, const int32_t* pos_thw,
                         const int32_t* seq_lens, const int32_t* page_table,
                         int32_t max_pages, int32_t batch, const cc_kv_pool* kv,
                         void* stream);

/* Tied LM head: logits[r] = logit_scale * (LayerNorm_f(hidden[rows[r]]) @ embed^T).
 * hidden f32 [*, H]; rows int32 [n_rows] (NULL: rows 0..n_rows-1); logits f32 [n_rows, V].
 * n_rows <= max_tokens. */
cc_status cc_logits(cc_layer_plan* plan, const float* hidden, const int32_t* rows,
                    int32_t n_rows, float* logits, void* stream);

/* ---------------------------------------------------------------- 4-bit affine weights
 * The mlx conversion of the checkpoint stores the projections and the embedding in 4-bit
 * affine form with group size 64 (Compass issue, "Config (config.json)", quantization
 * {group_size 64, bits 4, mode affine}): w[n, k] = scale[n, k / 64] * q[n, k] +
 * bias[n, k / 64], q[n, k] the 4-bit field at bit 4 * (k % 8) of the 32-bit word
 * packed[n, k / 8] (lowest bits first), scale and bias bf16. The decode-step GEMMs below read
 * these weights directly (about a quarter of the bf16 bytes) and turn each group into bf16
 * on chip: the dequantised weight is rounded to bf16 (scale * q + bias rounded once), then
 * multiplied with fp32 accumulation.
 *
 * Tiled form (what the GEMMs read): a [rows, K] matrix, rows % 128 == 0, K % 64 == 0, is cut
 * into blocks of 128 rows x 128 K, block (t, j) at byte (t * ceil(K / 128) + j) * 9216:
 *   bytes [0, 8192)     the 16 packed words of each of the 128 rows, chunk-major: the
 *                       16-byte chunk c (words 4c .. 4c + 3 of the row's 16) of row r at
 *                       byte (c * 128 + r) * 16
 *   bytes [8192, 9216)  one 32-bit word per group and row, group g (of the block's two) and
 *                       row r at byte 8192 + (g * 128 + r) * 4: scale's bf16 bits in the low
 *                       half, bias's in the high half
 * Words and groups past K are zero. Each block is one contiguous read of the weight stream. */
typedef struct {
  const void* ln_w;  /* bf16 [H] LayerNorm gain                                          */
  const void* w1;    /* tiled [N1, H]: rows arranged as w1 of cc_layer_weights            */
  const void* w2;    /* tiled [H, K2]: columns arranged as w2                             */
} cc_layer_weights_q4;

/* Bytes of the tiled form of a [rows, k] matrix (0 unless rows % 128 == 0, k % 64 == 0). */
size_t cc_q4_tiled_bytes(int32_t rows, int32_t k);

/* Tiles one checkpoint matrix: words uint32 [rows, k / 8], scales and biases bf16
 * [rows, k / 64] (device) -> out (cc_q4_tiled_bytes(rows, k) bytes, caller-allocated,
 * 16-byte aligned). rows % 128 == 0 and k % 64 == 0, else CC_ERR_UNSUPPORTED. */
cc_status cc_pack_q4_tiles(const void* words, const void* scales, const void* biases,
                           int32_t rows, int32_t k, void* out, void* stream);

/* cc_pack_layer_weights for 4-bit affine matrices: packed[i], scales[i], biases[i] (host
 * arrays of 7 device pointers, in the order q, k, v, o, gate, up, down) are the checkpoint's
 * [out, in / 8] uint32 words and [out, in / 64] bf16 scales and biases. Writes w1 and w2 of
 * cc_layer_weights_q4 (cc_q4_tiled_bytes(N1, H) and cc_q4_tiled_bytes(H, K2) bytes,
 * caller-allocated) with w1's row and w2's column arrangement. Uses stream-ordered scratch
 * the size of the larger fused matrix. */
cc_status cc_pack_layer_weights_q4(const cc_model_config* cfg, const void* const* packed,
                                   const void* const* scales, const void* const* biases,
                                   void* w1_out, void* w2_out, void* stream);

/* Gives a bf16 plan the tiled 4-bit affine weights of every layer (layers[num_layers]) and
 * of the tied embedding (embed_q4: tiled [V, H]) for cc_decode_step_q4 and cc_logits_q4.
 * Borrowed like the bf16 weights (16-byte aligned). A second call replaces the first. */
cc_status cc_layer_plan_attach_q4(cc_layer_plan* plan, const cc_layer_weights_q4* layers,
                                  const void* embed_q4);

/* cc_decode_step with the attached 4-bit weights (same arguments and result up to the
 * weights' rounding). batch <= 128. CC_ERR_INVALID_ARG when nothing is attached. */
cc_status cc_decode_step_q4(cc_layer_plan* plan, float* hidden, const int32_t* pos_thw,
                            const int32_t* seq_lens, const int32_t* page_table,
                            int32_t max_pages, int32_t batch, const cc_kv_pool* kv,
                            void* stream);

/* cc_logits with the attached 4-bit embedding as the LM head. n_rows <= 128. */
cc_status cc_logits_q4(cc_layer_plan* plan, const float* hidden, const int32_t* rows,
                       int32_t n_rows, float* logits, void* stream);

/* CUDA graphs: cc_prefill_forward, cc_prefill_forward_tokens, cc_prefill_forward_chunk,
 * cc_decode_step(_q4) and cc_logits(_q4) enqueue kernels (and, for a split head, one memset)
 * on `stream` only: no allocation and no host synchronisation, except that cc_decode_step
 * grows the plan's split-KV scratch (cudaMalloc after a stream synchronize) the first time a
 * call needs more. After one eager call of the same shape they can be captured into a CUDA
 * graph by stream capture and replayed; the arguments (device pointers, sizes) are baked in. */

/* Waits for `stream`, then returns and clears the plan's sticky device error flag
 * (CC_ERR_TIMEOUT / CC_ERR_DEVICE_CHECK), or CC_ERR_CUDA if the stream failed. */
cc_status cc_sync(cc_layer_plan* plan, void* stream);

/* Per-kernel timing of a plan's calls (no counterpart on the pages; a measurement aid).
 * While enabled, every kernel launch of cc_prefill_forward / cc_decode_step / cc_logits is
 * bracketed by CUDA events recorded on the launching stream. cc_profile_read waits for
 * those events and returns, per kernel class, the launch count and summed device time;
 * it then clears the records. Enabling costs two event records per launch. */
typedef enum {
  CC_K_ROPE_TABLE = 0,     /* MRoPE cos/sin table                                   */
  CC_K_ROW_MAPS = 1,       /* deepstack row map, KV slots, attention tile lists      */
  CC_K_LAYERNORM = 2,      /* pre-block and final LayerNorm                          */
  CC_K_GEMM_QKV_MLP = 3,   /* [q|k|v|gate,up] projection + rotation + SwiGLU epilogue */
  CC_K_ATTN_PREFILL = 4,   /* causal / sliding flash attention                       */
  CC_K_GEMM_OUT = 5,       /* [o|down] projection + residual (+ deepstack)           */
  CC_K_ATTN_DECODE = 6,    /* paged decode attention + split combine                 */
  CC_K_GEMM_HEAD = 7,      /* tied head x logit_scale                                */
  CC_K_F32_PATH = 8,       /* kernels of the fp32 variant                            */
  CC_K_EMBED_MERGE = 9,    /* embedding lookup + image rows + layer 0 LayerNorm      */
  CC_K_COUNT = 10
} cc_kernel_class;

typedef struct {
  int32_t launches;
  double total_ms;
} cc_kernel_time;

cc_status cc_profile_enable(cc_layer_plan* plan, int32_t enable);
/* out: CC_K_COUNT entries indexed by cc_kernel_class. */
cc_status cc_profile_read(cc_layer_plan* plan, cc_kernel_time* out);
const char* cc_kernel_class_name(int32_t kernel_class);

/* ------------------------------- single operations ---------------------------------
 * The steps of the path as separate calls, for composition and testing. They use a
 * library-wide device error flag read by cc_op_sync. Scratch memory they need is
 * taken with cudaMallocAsync/cudaFreeAsync on `stream`. */

/* Embedding merge, optionally fused with a LayerNorm (see cc_prefill_forward_tokens):
 * hidden[t] = f32(embed[token_ids[t]]), then hidden[mm_rows[r]] = f32(mm_embeds[r]); when
 * ln_w is not NULL also ln_out[t] = bf16(LayerNorm(hidden[t]) * ln_w) with the arithmetic
 * of cc_op_layernorm. token_ids int32 [T]; embed bf16 [vocab, H]; mm_rows int32 [R]
 * distinct (which of two equal rows wins is unspecified); mm_embeds bf16 [R, H]; hidden
 * f32 [T, H]; ln_w bf16 [H]; ln_out bf16 [T, H]. H % 128 == 0, H <= 4096. Bad indices set the
 * op error flag (cc_op_sync). */
cc_status cc_op_embed_merge(const int32_t* token_ids, int32_t tokens, const void* embed,
                            int32_t vocab, int32_t hidden_size, const int32_t* mm_rows,
                            const void* mm_embeds, int32_t n_mm_rows, float* hidden,
                            const void* ln_w, float eps, void* ln_out, void* stream);

/* LayerNorm (Compass issue, "Text decoder forward": weight only, no bias, f32 statistics,
 * biased variance, eps inside the square root): out[r] = bf16(gamma * (x[src] - mean) /
 * sqrt(var + eps)), src = row_idx ? row_idx[r] : r. x f32 [*, H]; gamma bf16 [H];
 * out bf16 [rows, H]. H % 128 == 0 and H <= 4096 (else CC_ERR_UNSUPPORTED). */
cc_status cc_op_layernorm(const float* x, const void* gamma, void* out, int32_t rows,
                          int32_t hidden, float eps, const int32_t* row_idx, void* stream);

/* Interleaved MRoPE cos/sin table (Compass issue, "Text decoder forward", interleaved
 * MRoPE paragraph): table[t, j] = (cos, sin)(pos[axis(j), t] * theta^(-2j/head_dim)) for
 * j < head_dim/2, axis(j) = h if j%3==1 and j<3*section[1], w if j%3==2 and
 * j<3*section[2], else t. pos int32 [3, T]; table f32 [T, head_dim/2, 2]. */
cc_status cc_op_mrope_table(const int32_t* pos, int32_t tokens, int32_t head_dim,
                            double theta, const int32_t* section_host, float* table,
                            void* stream);

/* cc_op_mrope_table for a given cc_mrope_layout (the table of CC_MROPE_SECTIONS_HWT puts at
 * rotary index k the axis and frequency of that layout). */
cc_status cc_op_mrope_table_layout(const int32_t* pos, int32_t tokens, int32_t head_dim,
                                   double theta, const int32_t* section_host, int32_t layout,
                                   float* table, void* stream);

/* The 4-bit affine GEMM of cc_decode_step_q4: C[M, N] = alpha * A[M, K] @ W^T (+ C when
 * accumulate != 0), W [N, K] in tiled form (cc_pack_q4_tiles), each weight rounded to bf16
 * after dequantisation. A bf16 [M, K]; C f32 [M, N]. M <= 128, K % 64 == 0, N % 128 == 0;
 * A and W 16-byte aligned. */
cc_status cc_op_gemm_q4(const void* a, const void* w_tiled, float* c, int32_t m, int32_t n,
                        int32_t k, float alpha, int32_t accumulate, void* stream);

/* Dense bf16 GEMM on the tcgen05 tensor cores: C[M, N] = alpha * A[M, K] @ B[N, K]^T
 * (+ C when accumulate != 0). A, B bf16 row-major (K contiguous); C f32 [M, N].
 * K % 64 == 0, N % 128 == 0; A and B 16-byte aligned. */
cc_status cc_op_gemm_bf16(const void* a, const void* b, float* c, int32_t m, int32_t n,
                          int32_t k, float alpha, int32_t accumulate, void* stream);

/* Prefill attention (causal, or sliding window when window > 0) over packed sequences,
 * grouped-query, scale head_dim^-0.5, on the tcgen05 tensor cores.
 * q bf16 [T, n_q * 128]; k, v bf16 [T, n_kv * 128]; out bf16 rows of leading dimension
 * ld_out (head h at columns h*128 .. h*128+127). head_dim must be 128. */
cc_status cc_op_attention_prefill(const void* q, const void* k, const void* v, void* out,
                                  int32_t ld_out, const int32_t* cu_seqlens, int32_t n_seqs,
                                  int32_t tokens, int32_t n_q, int32_t n_kv, int32_t window,
                                  void* stream);

/* Decode attention of one query token per sequence over a paged cache (split-KV):
 * q bf16 [batch, n_q * 128]; k_pool, v_pool bf16 [n_pages, n_kv, page_size, 128];
 * page_table int32 [batch, max_pages] (ids outside [0, n_pages) set the device flag
 * CC_ERR_DEVICE_CHECK and their keys are skipped); n_keys int32 [batch] keys to attend
 * over (token n_keys-1 is the query's own, n_keys <= max_pages * page_size);
 * window > 0: only the last `window` keys; out bf16 rows of leading dimension ld_out.
 * page_size must be 16 and n_q / n_kv one of 1, 2, 4, 8, 16 (else CC_ERR_UNSUPPORTED). */
cc_status cc_op_attention_decode(const void* q, const void* k_pool, const void* v_pool,
                                 int32_t n_pages, const int32_t* page_table, int32_t max_pages,
                                 const int32_t* n_keys, int32_t batch, int32_t n_q,
                                 int32_t n_kv, int32_t page_size, int32_t window, void* out,
                                 int32_t ld_out, void* stream);

/* Waits for `stream`; returns and clears the library-wide device error flag of the
 * single operations. */
cc_status cc_op_sync(void* stream);

/* Test hook of the device error path (the pages have no counterpart). The next bf16 tensor-
 * core GEMM launched in this process, by any plan or single operation, starts with its MMA
 * thread waiting on a barrier that nothing arrives on. That bounded wait gives up within
 * about a second and records CC_ERR_TIMEOUT in the launch's error flag; the launch's other
 * warps then stop waiting, its copies in flight land and its tensor memory is released, so
 * the context stays usable. The call's outputs are wrong (cc_sync / cc_op_sync returns
 * CC_ERR_TIMEOUT and clears the flag); later calls are unaffected. For tests only. */
void cc_test_stall_next_gemm(void);

/* Decode attention that allocates no device memory. The pages have no counterpart to
 * this call; it exists for callers that cannot call cudaMalloc: a serving runtime whose
 * memory pool has already reserved the device (a fresh allocation fails or fragments it),
 * a decode loop that must not take the device-wide synchronisation cudaMalloc/cudaFree
 * may impose, or a host that is not allowed to allocate at all.
 * Same inputs, outputs and result as cc_op_attention_decode. Its split-KV scratch is one
 * fixed array inside the library (16 MiB, held on every GPU that loads the library until
 * the process exits): it needs batch * n_q * ceil(max_pages / 64) * 130 floats, at most
 * 4194304; larger problems return CC_ERR_INVALID_ARG and launch nothing.
 * The first call on a device looks up that array's device address (with that device
 * current) and caches it; make that first call before any stream capture. All calls share
 * the array, so calls that may overlap on the GPU (other streams, other threads) race and
 * must be serialised by the caller. err_flag: optional caller-owned device int32 that
 * receives CC_ERR_TIMEOUT / CC_ERR_DEVICE_CHECK (first error wins; the caller clears it);
 * NULL: device-side problems are not reported. A split whose bounded wait gave up counts as
 * empty (it never merges a partial left in the array by an earlier call), so the output of
 * a call that reported CC_ERR_TIMEOUT is wrong but holds nothing of another call. */
cc_status cc_op_attention_decode_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                         int32_t n_pages, const int32_t* page_table,
                                         int32_t max_pages, const int32_t* n_keys, int32_t batch,
                                         int32_t n_q, int32_t n_kv, int32_t page_size,
                                         int32_t window, void* out, int32_t ld_out,
                                         int32_t* err_flag, void* stream);

#ifdef __cplusplus
}
#endif

#endif  /* CC_H_ */
