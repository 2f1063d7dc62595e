// Internal launchers of the cc kernels (not part of the C-ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "common.h"

namespace cc {

// ---------------------------------------------------------------- GEMM (tcgen05)
enum EpiMode : int {
  EPI_F32 = 0,      // c = alpha * acc (+ c)
  EPI_RESID = 1,    // h += acc (+ deepstack row)
  EPI_QKV_MLP = 2,  // column-typed: q / k / v heads (+ rotation, + paged K/V), SwiGLU
  EPI_RESID_LN = 3, // EPI_RESID, then the next layer's LayerNorm of the updated rows
};

struct EpiParams {
  // EPI_F32 and EPI_RESID: fp32 output / residual, leading dimension ldc
  float* c = nullptr;
  int ldc = 0;
  float alpha = 1.f;
  int accumulate = 0;
  // EPI_RESID: deepstack add, ds_map[row] = index into ds (or -1)
  const int32_t* ds_map = nullptr;
  const __nv_bfloat16* ds = nullptr;
  // EPI_QKV_MLP: columns [0, q_cols) q heads, then kv_cols of k, kv_cols of v, then the
  // SwiGLU region in 128-column blocks (64 gate columns, then the 64 matching up columns)
  int q_cols = 0, kv_cols = 0, n_kv = 0;
  const float2* rope = nullptr;          // [M, 64] (cos, sin), null: no rotation
  __nv_bfloat16* q_out = nullptr;        // [M, ld_q]
  int ld_q = 0;
  __nv_bfloat16* k_out = nullptr;        // [M, ld_kv] contiguous copy (nullable)
  __nv_bfloat16* v_out = nullptr;
  int ld_kv = 0;
  __nv_bfloat16* k_pool = nullptr;       // paged copy (nullable)
  __nv_bfloat16* v_pool = nullptr;
  const int32_t* kv_slot = nullptr;      // [M] flat slot page*page_size + offset, <0: skip
  int page_size = 16;
  __nv_bfloat16* act_out = nullptr;      // [M, ld_act]
  int ld_act = 0;
  // EPI_RESID_LN: ln_out[row] = bf16(LayerNorm(h[row]) * ln_gamma) of the updated rows. Each
  // output tile stores its rows' (mean, M2) per 128-column slot in ln_part [M, N / 128] and
  // adds its slot count to ln_cnt[m-tile] (zero when the launch starts; left at N / 128); the
  // tiles of a row block meet there and each normalises its own columns.
  const __nv_bfloat16* ln_gamma = nullptr;
  __nv_bfloat16* ln_out = nullptr;       // [M, ldc]
  float2* ln_part = nullptr;
  int32_t* ln_cnt = nullptr;
  float ln_eps = 0.f;
  // test hook (cc_test_stall_next_gemm): the MMA thread first waits on a barrier that
  // nothing arrives on, so the launch takes its timeout path
  int test_stall = 0;
};

// C[M,N] (epilogue) = A[M,K] @ B[N,K]^T with A, B given by TMA maps (bf16, box 64 x 128
// for A and 64 x BN for B, 128-byte swizzle). bn is 128 or 256; splits divides the
// K loop (splits > 1 needs an additive epilogue: EPI_RESID or EPI_F32 with accumulate).
// tb_half (optional): the same weights with a 128-row box; with it a 256-wide EPI_RESID_LN
// launch runs a last round that is at most half full as 128-column halves of its tiles.
cc_status launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K, int bn,
                      int splits, int epi, const EpiParams& ep, int* err, cudaStream_t s,
                      const CUtensorMap* tb_half = nullptr);

// Test hook: the next launch_gemm call (any thread) stalls its MMA thread (EpiParams::test_stall).
void test_stall_next_gemm();

// Picks bn / splits for a problem (used by every caller of launch_gemm).
void gemm_choose(int M, int N, int K, int epi, int* bn, int* splits);
// Whether launch_gemm runs EPI_RESID_LN for an [M, N] output (it needs one K split and an
// output row block's N / bn tiles on distinct resident CTAs).
bool gemm_resid_ln_ok(int M, int N, int K);

// Tiled 4-bit affine weights of a [rows, K] matrix (rows % 128 == 0, K % 64 == 0): block
// (t, j), t < rows / 128, j < ceil(K / 128), is kQ4TileBlockBytes contiguous bytes at
// (t * ceil(K / 128) + j) * kQ4TileBlockBytes holding rows 128 t .. 128 t + 127 and
// K = 128 j .. 128 j + 127:
//   bytes [0, 8192)     the rows' packed words (16 per row), chunk-major: the 16-byte chunk
//                       c (words 4c .. 4c + 3) of row r at (c * 128 + r) * 16
//   bytes [8192, 9216)  (scale, bias) words of groups 2 j and 2 j + 1: group g, row r at
//                       (g * 128 + r) * 4, scale's bf16 bits in the low half
// Words and groups past K are zero.
constexpr uint32_t kQ4TileBlockBytes = 9216;
size_t q4_tiled_bytes(int rows, int K);
// words uint32 [rows, K / 8] (checkpoint order), scales / biases bf16 [rows, K / 64]
cc_status launch_q4_tile(const uint32_t* words, const uint16_t* scales, const uint16_t* biases,
                         int rows, int K, uint8_t* out, cudaStream_t s);

// The GEMM with W in 4-bit affine form (group 64 along K), weight-stationary for M <= 128:
// tx maps the bf16 activations X [M, K] with box 64 x gemm_q4_token_tile(M) rows (128-byte
// swizzle); w_tiled holds W [N, K] tiled as above (16-byte aligned). N % 128 == 0,
// K % 64 == 0.
int gemm_q4_token_tile(int M);
cc_status launch_gemm_q4(const CUtensorMap& tx, const void* w_tiled, int M, int N, int K,
                         int epi, const EpiParams& ep, int* err, cudaStream_t s);

// ---------------------------------------------------------------- attention
// One work item of the prefill attention, for every head group: a 128-query tile and the
// key tiles [kt0, kt1) it reads. A query tile whose key range is long next to the launch's
// average work per SM is cut into n_chunks items; each writes a partial (running max, sum,
// unnormalised O) and the last one to finish merges them.
struct AttnTile {
  int32_t seq_start;  // first token of the sequence in the packed batch
  int32_t seq_len;
  int32_t q0;         // first query (relative to the sequence) of this 128-row tile
  int32_t kt0, kt1;   // key tiles of this item
  int32_t chunk;      // index among the query tile's n_chunks items
  int32_t n_chunks;
  int32_t slot0;      // partial slot of chunk 0 (chunk c uses slot0 + c); -1 when unsplit
  int32_t split;      // ordinal of the split query tile (its arrival counters); -1 unsplit
  int32_t prefix;     // keys of the sequence before this call's tokens (chunked prefill)
  int32_t seq;        // the sequence (its page-table row)
  int32_t pad;
};

// K and V of a chunked prefill: the paged pool [page][kv head][16][128] read through the
// page table (pt null: contiguous K and V of the call's own tokens).
struct AttnPaged {
  const int32_t* pt = nullptr;  // [n_seqs, max_pages]
  int max_pages = 0;
  int n_pages = 0;
};

// Scratch of one prefill attention launch. `counters` and `sched` must be zero when the
// launch starts; the kernel leaves the counters at zero and advances `sched`.
struct AttnScratch {
  float* part_o = nullptr;      // [slots][n_q][128 rows][128] unnormalised partial outputs
  float2* part_ml = nullptr;    // [slots][n_q][128 rows] running max (log2 units), sum
  int32_t* counters = nullptr;  // [split tiles][head groups][1 + max chunks] arrivals, flags
  int32_t* sched = nullptr;     // next work item (one counter per launch)
};

// Head groups of a launch: pairs of query heads sharing a KV head, else single heads.
int attn_groups(int n_q, int n_kv);
// Capacities of the split bookkeeping for a launch with `groups` head groups (bounds that
// hold for every cu_seqlens, from the splitting rule of the tile builder).
int attn_split_slots(int groups);
int attn_split_tiles(int groups);
size_t attn_part_o_floats(int n_q, int n_kv);
size_t attn_part_ml_pairs(int n_q, int n_kv);

// Ints of split bookkeeping (per split tile and head group: an arrival count and one ready
// flag per chunk) of a launch with `groups` head groups.
int attn_counter_ints(int groups);

// Builds the work lists of all sequences (query tiles, long ones cut into chunks), heaviest
// first, for launches with `groups` head groups: list a with window_a and, when tiles_b is
// not null, list b with window_b, in one launch that also zeroes zero[0 .. n_zero).
// prefix (nullable, [n_seqs]): the tokens of sequence s continue a cached prefix of
// prefix[s] keys (chunked prefill); the key tiles are then absolute key positions.
cc_status launch_attn_tiles(const int32_t* cu_seqlens, int n_seqs, int tokens, int groups,
                            int window_a, AttnTile* tiles_a, int32_t* n_tiles_a, int window_b,
                            AttnTile* tiles_b, int32_t* n_tiles_b, int32_t* zero, int n_zero,
                            cudaStream_t s, const int32_t* prefix = nullptr, int max_prefix = 0);
int attn_max_tiles(int tokens, int n_seqs);
// Rows (keys) of the K and V boxes the prefill attention kernel loads.
int attn_kv_box_rows();

// tk, tv: [T, n_kv * 128] (contiguous) or, with paged.pt, the pools as
// [n_pages * n_kv * 16, 128] with 16-row boxes.
cc_status launch_attn_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              __nv_bfloat16* out, int ld_out, const AttnTile* tiles,
                              const int32_t* n_tiles, int max_tiles, int n_q, int n_kv,
                              int window, const AttnScratch& sc, int* err, cudaStream_t s,
                              const AttnPaged& paged = AttnPaged());

// ---------------------------------------------------------------- decode attention
struct DecodeScratch {
  float* part_o = nullptr;   // [batch, n_q, splits, 128]
  float* part_ml = nullptr;  // [batch, n_q, splits, 2]
};
int decode_splits(int max_pages);
size_t decode_scratch_floats(int batch, int n_q, int max_pages);
cc_status launch_attn_decode(const __nv_bfloat16* q, int ld_q, const __nv_bfloat16* k_pool,
                             const __nv_bfloat16* v_pool, int n_pages, const int32_t* page_table,
                             int max_pages, const int32_t* n_keys, int batch, int n_q, int n_kv,
                             int page_size, int window, DecodeScratch scr, __nv_bfloat16* out,
                             int ld_out, int* err, cudaStream_t s);

// ---------------------------------------------------------------- small kernels
cc_status launch_layernorm_bf16(const float* x, const __nv_bfloat16* gamma, __nv_bfloat16* out,
                                int rows, int H, float eps, const int32_t* row_idx,
                                cudaStream_t s);
cc_status launch_layernorm_f32(const float* x, const float* gamma, float* out, int rows, int H,
                               float eps, const int32_t* row_idx, cudaStream_t s);
cc_status launch_mrope_table(const int32_t* pos, int T, int head_dim, double theta,
                             const int32_t section[3], int layout, float2* table, cudaStream_t s);
// h[row] = f32(mm_embeds[mm_map[row]]) when mm_map[row] >= 0, else f32(embed[tok[row]]);
// ln_out (nullable) = bf16(LayerNorm(h row) * ln_w). Out-of-range token ids set err.
cc_status launch_embed_ln(const int32_t* tok, const __nv_bfloat16* embed, int V,
                          const int32_t* mm_map, const __nv_bfloat16* mm_embeds, int rows, int H,
                          float* h, const __nv_bfloat16* ln_w, float eps, __nv_bfloat16* ln_out,
                          int* err, cudaStream_t s);
cc_status launch_ds_map(const int32_t* rows, int n_rows, int T, int32_t* map, int* err,
                        cudaStream_t s);
// kv_slot for prefill tokens: page_table[seq, t / ps] * ps + t % ps
// slots[t] = cache slot of token t: position prefix[s] + (t - cu[s]) of its sequence s
// (prefix nullable: 0).
cc_status launch_kv_slots_prefill(const int32_t* cu_seqlens, int n_seqs, int T,
                                  const int32_t* page_table, int max_pages, int page_size,
                                  int n_pages, int32_t* slots, int* err, cudaStream_t s,
                                  const int32_t* prefix = nullptr);
// kv_slot of decode rows: the new token of sequence b goes to slot seq_lens[b]
cc_status launch_kv_slots_decode(const int32_t* seq_lens, int batch, const int32_t* page_table,
                                 int max_pages, int page_size, int n_pages, int32_t* slots,
                                 int32_t* n_keys, int* err, cudaStream_t s);

// ---------------------------------------------------------------- fp32 (CUDA-core) path
cc_status launch_gemm_f32(const float* a, int lda, const float* b, int ldb, float* c, int ldc,
                          int M, int N, int K, float alpha, int accumulate, cudaStream_t s);
cc_status launch_qkv_mlp_f32(const float* y, int ldy, int M, int q_cols, int kv_cols,
                             int head_dim, int inter, const float2* rope, float* q, float* k,
                             float* v, float* act, int ld_act, cudaStream_t s);
cc_status launch_attn_f32(const float* q, const float* k, const float* v, float* out,
                          int ld_out, const int32_t* cu_seqlens, int n_seqs, int T, int n_q,
                          int n_kv, int head_dim, int window, cudaStream_t s);
cc_status launch_ds_add_f32(float* h, int H, const int32_t* rows, int n_rows, const float* ds,
                            cudaStream_t s);

}  // namespace cc
