// The C-ABI: argument checks, the layer plan (configuration, borrowed weights, owned
// workspace, weight TMA descriptors) and the stream-ordered sequence of kernels of each
// entry point. The forward follows the mlxcel issue "Cohere Compass /
// North-Micro-Vision", section "Text decoder forward":
//   per layer  LayerNorm -> [q|k|v|gate,up] projection (+ rotation on sliding layers,
//              + K/V into the paged cache, + SwiGLU) -> attention -> [o|down] projection
//              + residual (+ deepstack rows after the first layers)
//   head       LayerNorm_f on the selected rows -> tied embedding GEMM x logit_scale.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "kernels.h"

namespace cc {

cudaError_t& last_cuda_error() {
  static cudaError_t e = cudaSuccess;
  return e;
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      n = v;
    else
      n = kNumSMsFallback;
  }
  return n;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint64_t ld, uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !base || rows == 0 || cols == 0) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (ld * 2) % 16 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw =
      (box_cols * 2 == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// library-wide error flag of the single operations (one per process; single device)
static int* op_error_flag() {
  static int* flag = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    if (cudaMalloc(&flag, sizeof(int)) != cudaSuccess) flag = nullptr;
    else cudaMemset(flag, 0, sizeof(int));
  });
  return flag;
}

static cc_status read_and_clear(int* flag, cudaStream_t s) {
  CC_CHECK_CUDA(cudaStreamSynchronize(s));
  if (!flag) return CC_OK;
  int h = 0;
  CC_CHECK_CUDA(cudaMemcpy(&h, flag, sizeof(int), cudaMemcpyDeviceToHost));
  if (h != 0) {
    CC_CHECK_CUDA(cudaMemset(flag, 0, sizeof(int)));
    return static_cast<cc_status>(h);
  }
  return CC_OK;
}

// Per-kernel-class timing with CUDA events recorded on the launching stream.
struct Profiler {
  bool on = false;
  struct Rec {
    int cls;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> spare;
  cudaEvent_t get() {
    if (!spare.empty()) {
      cudaEvent_t e = spare.back();
      spare.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) e = nullptr;
    return e;
  }
  ~Profiler() {
    for (auto& r : recs) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
    for (auto e : spare) cudaEventDestroy(e);
  }
};

class ProfScope {
 public:
  ProfScope(Profiler& p, int cls, cudaStream_t s) : p_(p), cls_(cls), s_(s) {
    if (p_.on) {
      a_ = p_.get();
      if (a_) cudaEventRecord(a_, s_);
    }
  }
  ~ProfScope() {
    if (!p_.on || !a_) return;
    cudaEvent_t b = p_.get();
    if (!b) return;
    cudaEventRecord(b, s_);
    p_.recs.push_back({cls_, a_, b});
  }

 private:
  Profiler& p_;
  int cls_;
  cudaStream_t s_;
  cudaEvent_t a_ = nullptr;
};

}  // namespace cc

using namespace cc;

#define CC_TIMED(plan, cls, stream, expr)              \
  do {                                                 \
    ProfScope ps_((plan)->prof, (cls), (stream));      \
    CC_CHECK_STATUS(expr);                             \
  } while (0)

struct cc_layer_plan {
  Profiler prof;
  cc_model_config cfg{};
  std::vector<int32_t> types;
  std::vector<cc_layer_weights> layers;
  const void* final_ln = nullptr;
  const void* embed = nullptr;
  bool bf16 = true;
  int H = 0, nq = 0, nkv = 0, d = 0, I = 0, V = 0, N1 = 0, K2 = 0, q_cols = 0, kv_cols = 0;
  int T_max = 0;
  // weight TMA descriptors, box heights 128 and 256
  std::vector<CUtensorMap> w1_128, w1_256, w2_128, w2_256;
  CUtensorMap emb_128{}, emb_256{};
  // workspace (one allocation)
  uint8_t* ws = nullptr;
  int* err = nullptr;
  __nv_bfloat16 *a = nullptr, *q = nullptr, *k = nullptr, *v = nullptr, *a2 = nullptr;
  float *af = nullptr, *yf = nullptr, *qf = nullptr, *kf = nullptr, *vf = nullptr, *a2f = nullptr;
  float2* rope = nullptr;
  int32_t *ds_map = nullptr, *mm_map = nullptr, *kv_slot = nullptr, *n_keys = nullptr,
          *n_tiles = nullptr;
  AttnTile *tiles_s = nullptr, *tiles_f = nullptr;
  int max_tiles = 0;
  // prefill attention: partials of split query tiles, then [arrival counters | one item
  // counter per layer], zeroed before each forward
  float* attn_part_o = nullptr;
  float2* attn_part_ml = nullptr;
  int32_t* attn_cnt = nullptr;
  size_t attn_cnt_ints = 0;
  int attn_groups_n = 1;
  // the residual + LayerNorm epilogue: per-row partial statistics [T, H / 128] and one
  // arrival counter per row block and layer (inside attn_cnt, zeroed before each forward)
  float2* ln_part = nullptr;
  int32_t* ln_cnt = nullptr;
  int ln_row_blocks = 0;
  // tiled 4-bit affine weights (cc_layer_plan_attach_q4)
  std::vector<cc_layer_weights_q4> layers_q4;
  const void* embed_q4 = nullptr;
  // decode split-KV scratch, grown on demand
  float* dec_scratch = nullptr;
  size_t dec_scratch_floats = 0;

  ~cc_layer_plan() {
    if (ws) cudaFree(ws);
    if (dec_scratch) cudaFree(dec_scratch);
  }
  const CUtensorMap& w1(int i, int bn) const { return bn == 256 ? w1_256[i] : w1_128[i]; }
  const CUtensorMap& w2(int i, int bn) const { return bn == 256 ? w2_256[i] : w2_128[i]; }
  const CUtensorMap& emb(int bn) const { return bn == 256 ? emb_256 : emb_128; }
};

extern "C" const char* cc_status_string(cc_status s) {
  switch (s) {
    case CC_OK: return "ok";
    case CC_ERR_INVALID_ARG: return "invalid argument";
    case CC_ERR_UNSUPPORTED: return "unsupported configuration";
    case CC_ERR_OOM: return "device out of memory";
    case CC_ERR_CUDA: return "CUDA error";
    case CC_ERR_TIMEOUT: return "device wait timed out";
    case CC_ERR_DEVICE_CHECK: return "device index check failed";
  }
  return "unknown status";
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static cc_status check_config(const cc_model_config* c) {
  if (!c || !c->layer_types) return CC_ERR_INVALID_ARG;
  if (c->num_layers <= 0 || c->hidden_size <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 ||
      c->head_dim <= 0 || c->intermediate_size <= 0 || c->vocab_size <= 0 ||
      c->sliding_window <= 0 || c->max_tokens <= 0 || c->kv_page_size <= 0)
    return CC_ERR_INVALID_ARG;
  if (c->n_q_heads % c->n_kv_heads != 0) return CC_ERR_INVALID_ARG;
  if (c->head_dim % 2 != 0) return CC_ERR_INVALID_ARG;
  if (c->mrope_section[0] < 0 || c->mrope_section[1] < 0 || c->mrope_section[2] < 0 ||
      c->mrope_section[0] + c->mrope_section[1] + c->mrope_section[2] != c->head_dim / 2)
    return CC_ERR_INVALID_ARG;
  if (c->dtype != CC_BF16 && c->dtype != CC_F32) return CC_ERR_INVALID_ARG;
  if (c->mrope_layout != CC_MROPE_INTERLEAVED && c->mrope_layout != CC_MROPE_SECTIONS_HWT)
    return CC_ERR_INVALID_ARG;
  if (!(c->rope_theta > 0.0) || !(c->layer_norm_eps >= 0.f)) return CC_ERR_INVALID_ARG;
  for (int i = 0; i < c->num_layers; ++i)
    if (c->layer_types[i] != CC_SLIDING && c->layer_types[i] != CC_FULL) return CC_ERR_INVALID_ARG;
  if (c->intermediate_size % 64 != 0) return CC_ERR_UNSUPPORTED;
  if (c->hidden_size % 128 != 0 || c->hidden_size > 4096) return CC_ERR_UNSUPPORTED;
  if (c->dtype == CC_BF16) {
    if (c->head_dim != 128 || c->vocab_size % 128 != 0 || c->kv_page_size != 16)
      return CC_ERR_UNSUPPORTED;
    const int g = c->n_q_heads / c->n_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return CC_ERR_UNSUPPORTED;
  } else {
    if (c->head_dim > 128) return CC_ERR_UNSUPPORTED;
  }
  return CC_OK;
}

extern "C" cc_status cc_pack_layer_weights(const cc_model_config* cfg, const void* wq,
                                           const void* wk, const void* wv, const void* wo,
                                           const void* wg, const void* wu, const void* wd,
                                           void* w1_out, void* w2_out, void* stream) {
  CC_CHECK_STATUS(check_config(cfg));
  if (!wq || !wk || !wv || !wo || !wg || !wu || !wd || !w1_out || !w2_out)
    return CC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t es = cfg->dtype == CC_BF16 ? 2 : 4;
  const size_t H = cfg->hidden_size, d = cfg->head_dim, I = cfg->intermediate_size;
  const size_t qr = cfg->n_q_heads * d, kr = cfg->n_kv_heads * d;
  uint8_t* w1 = static_cast<uint8_t*>(w1_out);
  const size_t row = H * es;
  CC_CHECK_CUDA(cudaMemcpyAsync(w1, wq, qr * row, cudaMemcpyDeviceToDevice, s));
  CC_CHECK_CUDA(cudaMemcpyAsync(w1 + qr * row, wk, kr * row, cudaMemcpyDeviceToDevice, s));
  CC_CHECK_CUDA(cudaMemcpyAsync(w1 + (qr + kr) * row, wv, kr * row, cudaMemcpyDeviceToDevice, s));
  uint8_t* mlp = w1 + (qr + 2 * kr) * row;
  // 64-row blocks: gate block b at rows 128 b, up block b at rows 128 b + 64
  CC_CHECK_CUDA(cudaMemcpy2DAsync(mlp, 128 * row, wg, 64 * row, 64 * row, I / 64,
                                  cudaMemcpyDeviceToDevice, s));
  CC_CHECK_CUDA(cudaMemcpy2DAsync(mlp + 64 * row, 128 * row, wu, 64 * row, 64 * row, I / 64,
                                  cudaMemcpyDeviceToDevice, s));
  const size_t K2 = qr + I;
  uint8_t* w2 = static_cast<uint8_t*>(w2_out);
  CC_CHECK_CUDA(cudaMemcpy2DAsync(w2, K2 * es, wo, qr * es, qr * es, H, cudaMemcpyDeviceToDevice, s));
  CC_CHECK_CUDA(cudaMemcpy2DAsync(w2 + qr * es, K2 * es, wd, I * es, I * es, H,
                                  cudaMemcpyDeviceToDevice, s));
  return CC_OK;
}

extern "C" cc_status cc_layer_plan_create(const cc_model_config* cfg, const cc_layer_weights* layers,
                                          const void* final_ln_w, const void* embed,
                                          cc_layer_plan** out) {
  if (!out) return CC_ERR_INVALID_ARG;
  *out = nullptr;
  CC_CHECK_STATUS(check_config(cfg));
  if (!layers || !final_ln_w || !embed) return CC_ERR_INVALID_ARG;
  for (int i = 0; i < cfg->num_layers; ++i)
    if (!layers[i].ln_w || !layers[i].w1 || !layers[i].w2) return CC_ERR_INVALID_ARG;

  cc_layer_plan* p = new (std::nothrow) cc_layer_plan();
  if (!p) return CC_ERR_OOM;
  p->cfg = *cfg;
  p->types.assign(cfg->layer_types, cfg->layer_types + cfg->num_layers);
  p->cfg.layer_types = p->types.data();
  p->layers.assign(layers, layers + cfg->num_layers);
  p->final_ln = final_ln_w;
  p->embed = embed;
  p->bf16 = cfg->dtype == CC_BF16;
  p->H = cfg->hidden_size;
  p->nq = cfg->n_q_heads;
  p->nkv = cfg->n_kv_heads;
  p->d = cfg->head_dim;
  p->I = cfg->intermediate_size;
  p->V = cfg->vocab_size;
  p->q_cols = p->nq * p->d;
  p->kv_cols = p->nkv * p->d;
  p->N1 = p->q_cols + 2 * p->kv_cols + 2 * p->I;
  p->K2 = p->q_cols + p->I;
  p->T_max = cfg->max_tokens;
  const size_t T = p->T_max;
  p->max_tiles = attn_max_tiles(p->T_max, p->T_max);

  // workspace layout
  std::vector<std::pair<void**, size_t>> parts;
  parts.push_back({reinterpret_cast<void**>(&p->err), 256});
  parts.push_back({reinterpret_cast<void**>(&p->rope), T * (p->d / 2) * sizeof(float2)});
  parts.push_back({reinterpret_cast<void**>(&p->ds_map), T * 4});
  parts.push_back({reinterpret_cast<void**>(&p->mm_map), T * 4});
  parts.push_back({reinterpret_cast<void**>(&p->kv_slot), T * 4});
  parts.push_back({reinterpret_cast<void**>(&p->n_keys), T * 4});
  parts.push_back({reinterpret_cast<void**>(&p->n_tiles), 256});
  parts.push_back({reinterpret_cast<void**>(&p->tiles_s), p->max_tiles * sizeof(AttnTile)});
  parts.push_back({reinterpret_cast<void**>(&p->tiles_f), p->max_tiles * sizeof(AttnTile)});
  if (p->bf16) {
    p->attn_groups_n = attn_groups(p->nq, p->nkv);
    p->ln_row_blocks = (p->T_max + 127) / 128;
    // [split counters | one item counter per layer | LayerNorm arrivals per layer, row block]
    p->attn_cnt_ints = (size_t)attn_counter_ints(p->attn_groups_n) + cfg->num_layers +
                       (size_t)cfg->num_layers * p->ln_row_blocks;
    parts.push_back({reinterpret_cast<void**>(&p->ln_part), T * (p->H / 128) * sizeof(float2)});
    parts.push_back({reinterpret_cast<void**>(&p->attn_part_o),
                     attn_part_o_floats(p->nq, p->nkv) * sizeof(float)});
    parts.push_back({reinterpret_cast<void**>(&p->attn_part_ml),
                     attn_part_ml_pairs(p->nq, p->nkv) * sizeof(float2)});
    parts.push_back({reinterpret_cast<void**>(&p->attn_cnt), p->attn_cnt_ints * 4});
    parts.push_back({reinterpret_cast<void**>(&p->a), T * p->H * 2});
    parts.push_back({reinterpret_cast<void**>(&p->q), T * p->q_cols * 2});
    parts.push_back({reinterpret_cast<void**>(&p->k), T * p->kv_cols * 2});
    parts.push_back({reinterpret_cast<void**>(&p->v), T * p->kv_cols * 2});
    parts.push_back({reinterpret_cast<void**>(&p->a2), T * p->K2 * 2});
  } else {
    parts.push_back({reinterpret_cast<void**>(&p->af), T * p->H * 4});
    parts.push_back({reinterpret_cast<void**>(&p->yf), T * p->N1 * 4});
    parts.push_back({reinterpret_cast<void**>(&p->qf), T * p->q_cols * 4});
    parts.push_back({reinterpret_cast<void**>(&p->kf), T * p->kv_cols * 4});
    parts.push_back({reinterpret_cast<void**>(&p->vf), T * p->kv_cols * 4});
    parts.push_back({reinterpret_cast<void**>(&p->a2f), T * p->K2 * 4});
  }
  size_t total = 0;
  for (auto& pr : parts) total += align256(pr.second);
  if (cudaMalloc(&p->ws, total) != cudaSuccess) {
    delete p;
    return CC_ERR_OOM;
  }
  size_t off = 0;
  for (auto& pr : parts) {
    *pr.first = p->ws + off;
    off += align256(pr.second);
  }
  // finite contents everywhere (rows past a call's tokens are read by full tiles)
  if (cudaMemset(p->ws, 0, total) != cudaSuccess) {
    delete p;
    return CC_ERR_CUDA;
  }
  if (p->bf16)
    p->ln_cnt = p->attn_cnt + attn_counter_ints(p->attn_groups_n) + cfg->num_layers;
  if (p->bf16) {
    const int L = cfg->num_layers;
    p->w1_128.resize(L);
    p->w1_256.resize(L);
    p->w2_128.resize(L);
    p->w2_256.resize(L);
    bool ok = true;
    for (int i = 0; i < L; ++i) {
      ok &= make_tmap_bf16_2d(&p->w1_128[i], layers[i].w1, p->N1, p->H, p->H, 128, 64);
      ok &= make_tmap_bf16_2d(&p->w1_256[i], layers[i].w1, p->N1, p->H, p->H, 256, 64);
      ok &= make_tmap_bf16_2d(&p->w2_128[i], layers[i].w2, p->H, p->K2, p->K2, 128, 64);
      ok &= make_tmap_bf16_2d(&p->w2_256[i], layers[i].w2, p->H, p->K2, p->K2, 256, 64);
    }
    ok &= make_tmap_bf16_2d(&p->emb_128, embed, p->V, p->H, p->H, 128, 64);
    ok &= make_tmap_bf16_2d(&p->emb_256, embed, p->V, p->H, p->H, 256, 64);
    if (!ok) {
      delete p;
      return CC_ERR_INVALID_ARG;  // misaligned weights or no driver entry point
    }
  }
  *out = p;
  return CC_OK;
}

extern "C" void cc_layer_plan_destroy(cc_layer_plan* plan) { delete plan; }

extern "C" size_t cc_q4_tiled_bytes(int32_t rows, int32_t k) {
  if (rows <= 0 || k <= 0 || rows % 128 != 0 || k % 64 != 0) return 0;
  return q4_tiled_bytes(rows, k);
}

extern "C" cc_status cc_pack_q4_tiles(const void* words, const void* scales, const void* biases,
                                      int32_t rows, int32_t k, void* out, void* stream) {
  if (rows < 0 || k < 0) return CC_ERR_INVALID_ARG;
  if (rows == 0 || k == 0) return CC_OK;
  if (rows % 128 != 0 || k % 64 != 0) return CC_ERR_UNSUPPORTED;
  if (!words || !scales || !biases || !out) return CC_ERR_INVALID_ARG;
  return launch_q4_tile(static_cast<const uint32_t*>(words), static_cast<const uint16_t*>(scales),
                        static_cast<const uint16_t*>(biases), rows, k, static_cast<uint8_t*>(out),
                        static_cast<cudaStream_t>(stream));
}

extern "C" cc_status cc_pack_layer_weights_q4(const cc_model_config* cfg, const void* const* packed,
                                              const void* const* scales, const void* const* biases,
                                              void* w1_out, void* w2_out, void* stream) {
  CC_CHECK_STATUS(check_config(cfg));
  if (cfg->dtype != CC_BF16) return CC_ERR_UNSUPPORTED;
  if (!packed || !scales || !biases || !w1_out || !w2_out) return CC_ERR_INVALID_ARG;
  for (int i = 0; i < 7; ++i)
    if (!packed[i] || !scales[i] || !biases[i]) return CC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t H = cfg->hidden_size, d = cfg->head_dim, I = cfg->intermediate_size;
  const size_t qr = cfg->n_q_heads * d, kr = cfg->n_kv_heads * d, K2 = qr + I;
  const size_t N1 = qr + 2 * kr + 2 * I;
  // the fused matrices in checkpoint (row-major) form first: w1 [N1, H] rows q | k | v | gate
  // and up in 64-row blocks, w2 [H, K2] columns o | down; then their tiles
  const size_t w1_words = N1 * H / 8, w1_groups = N1 * H / 64;
  const size_t w2_words = H * K2 / 8, w2_groups = H * K2 / 64;
  uint8_t* tmp = nullptr;
  const size_t tmp_bytes = std::max(w1_words * 4 + 2 * w1_groups * 2, w2_words * 4 + 2 * w2_groups * 2);
  CC_CHECK_CUDA(cudaMallocAsync(&tmp, tmp_bytes, s));
  cc_status st = CC_OK;
  auto fail = [&](cudaError_t e) {
    if (e != cudaSuccess && st == CC_OK) {
      last_cuda_error() = e;
      st = CC_ERR_CUDA;
    }
  };
  const cudaMemcpyKind dd = cudaMemcpyDeviceToDevice;
  {
    // three parts with the row arrangement of w1: words (H / 2 bytes per row), scales and
    // biases (H / 32 bytes per row)
    uint8_t* parts[3] = {tmp, tmp + w1_words * 4, tmp + w1_words * 4 + w1_groups * 2};
    const size_t row_b[3] = {H / 2, H / 32, H / 32};
    const void* const* src[3] = {packed, scales, biases};
    for (int q = 0; q < 3; ++q) {
      uint8_t* base = parts[q];
      const size_t row = row_b[q];
      fail(cudaMemcpyAsync(base, src[q][0], qr * row, dd, s));
      fail(cudaMemcpyAsync(base + qr * row, src[q][1], kr * row, dd, s));
      fail(cudaMemcpyAsync(base + (qr + kr) * row, src[q][2], kr * row, dd, s));
      uint8_t* mlp = base + (qr + 2 * kr) * row;
      fail(cudaMemcpy2DAsync(mlp, 128 * row, src[q][4], 64 * row, 64 * row, I / 64, dd, s));
      fail(cudaMemcpy2DAsync(mlp + 64 * row, 128 * row, src[q][5], 64 * row, 64 * row, I / 64, dd, s));
    }
    if (st == CC_OK)
      st = launch_q4_tile(reinterpret_cast<const uint32_t*>(parts[0]),
                          reinterpret_cast<const uint16_t*>(parts[1]),
                          reinterpret_cast<const uint16_t*>(parts[2]), static_cast<int>(N1),
                          static_cast<int>(H), static_cast<uint8_t*>(w1_out), s);
  }
  if (st == CC_OK) {
    // w2's columns: o then down, per part (words: 1/2 byte per column; scales, biases: 1/32)
    uint8_t* parts[3] = {tmp, tmp + w2_words * 4, tmp + w2_words * 4 + w2_groups * 2};
    const void* const* src[3] = {packed, scales, biases};
    for (int q = 0; q < 3; ++q) {
      const size_t per = q == 0 ? 2 : 32;   // columns per byte of the part
      fail(cudaMemcpy2DAsync(parts[q], K2 / per, src[q][3], qr / per, qr / per, H, dd, s));
      fail(cudaMemcpy2DAsync(parts[q] + qr / per, K2 / per, src[q][6], I / per, I / per, H, dd, s));
    }
    if (st == CC_OK)
      st = launch_q4_tile(reinterpret_cast<const uint32_t*>(parts[0]),
                          reinterpret_cast<const uint16_t*>(parts[1]),
                          reinterpret_cast<const uint16_t*>(parts[2]), static_cast<int>(H),
                          static_cast<int>(K2), static_cast<uint8_t*>(w2_out), s);
  }
  fail(cudaFreeAsync(tmp, s));
  return st;
}

extern "C" cc_status cc_layer_plan_attach_q4(cc_layer_plan* p, const cc_layer_weights_q4* layers,
                                             const void* embed_q4) {
  if (!p || !layers || !embed_q4) return CC_ERR_INVALID_ARG;
  if (!p->bf16) return CC_ERR_UNSUPPORTED;
  auto aligned = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  const int L = p->cfg.num_layers;
  for (int i = 0; i < L; ++i)
    if (!layers[i].ln_w || !layers[i].w1 || !layers[i].w2 || !aligned(layers[i].w1) ||
        !aligned(layers[i].w2))
      return CC_ERR_INVALID_ARG;
  if (!aligned(embed_q4)) return CC_ERR_INVALID_ARG;
  p->layers_q4.assign(layers, layers + L);
  p->embed_q4 = embed_q4;
  return CC_OK;
}

// one GEMM with the plan's tile choice; `b128`/`b256` are the weight maps
// Rows declared in the tensor map of a workspace activation (a, a2) for an m-row GEMM: at
// least one 128-row tile of real memory, so a short m (the head's last token, a decode
// batch) is fetched as plain rows instead of a mostly out-of-bounds box, which the TMA
// fills far more slowly. Rows past m hold stale data; they only reach accumulator rows the
// epilogues never store.
static int act_rows(const cc_layer_plan* p, int m) { return std::max(m, std::min(128, p->T_max)); }

static cc_status plan_gemm(const CUtensorMap& ta, const CUtensorMap& b128, const CUtensorMap& b256,
                           int M, int N, int K, int epi, const EpiParams& ep, int* err,
                           cudaStream_t s) {
  int bn, splits;
  gemm_choose(M, N, K, epi, &bn, &splits);
  return launch_gemm(ta, bn == 256 ? b256 : b128, M, N, K, bn, splits, epi, ep, err, s,
                     bn == 256 ? &b128 : nullptr);
}

// Token-id input of the prefill: the embedding merge fused with layer 0's LayerNorm.
struct EmbedIn {
  const int32_t* tok;
  const int32_t* mm_rows;
  const __nv_bfloat16* mm_embeds;
  int n_mm_rows;
};

static cc_status prefill_bf16(cc_layer_plan* p, float* hidden, const int32_t* pos,
                              const int32_t* cu, int n_seqs, int T, const int32_t* ds_rows,
                              int n_ds_rows, const void* const* ds_feats, int n_ds,
                              const cc_kv_pool* kv, const int32_t* page_table, int max_pages,
                              cudaStream_t s, const EmbedIn* emb = nullptr,
                              const int32_t* prefix = nullptr) {
  const cc_model_config& c = p->cfg;
  // chunked prefill: the tokens continue cached prefixes; attention reads every key from the
  // paged cache, which the projection epilogue fills with this call's keys first
  const bool chunked = prefix != nullptr;
  if (emb) {
    // h = embed[tok] with the image rows replaced, and layer 0's a = LayerNorm(h), in one pass
    if (emb->n_mm_rows > 0)
      CC_TIMED(p, CC_K_ROW_MAPS, s, launch_ds_map(emb->mm_rows, emb->n_mm_rows, T, p->mm_map, p->err, s));
    CC_TIMED(p, CC_K_EMBED_MERGE, s,
             launch_embed_ln(emb->tok, static_cast<const __nv_bfloat16*>(p->embed), p->V,
                             emb->n_mm_rows > 0 ? p->mm_map : nullptr, emb->mm_embeds, T, p->H,
                             hidden, static_cast<const __nv_bfloat16*>(p->layers[0].ln_w),
                             c.layer_norm_eps, p->a, p->err, s));
  }
  CC_TIMED(p, CC_K_ROPE_TABLE, s, launch_mrope_table(pos, T, p->d, c.rope_theta, c.mrope_section, c.mrope_layout, p->rope, s));
  if (n_ds > 0) CC_TIMED(p, CC_K_ROW_MAPS, s, launch_ds_map(ds_rows, n_ds_rows, T, p->ds_map, p->err, s));
  if (kv)
    CC_TIMED(p, CC_K_ROW_MAPS, s, launch_kv_slots_prefill(cu, n_seqs, T, page_table, max_pages, c.kv_page_size,
                                            kv->n_pages, p->kv_slot, p->err, s, prefix));
  // both work lists (sliding, full) in one launch, which also clears the attention counters
  CC_TIMED(p, CC_K_ROW_MAPS, s, launch_attn_tiles(cu, n_seqs, T, p->attn_groups_n, c.sliding_window,
                                                 p->tiles_s, p->n_tiles, 0, p->tiles_f,
                                                 p->n_tiles + 1, p->attn_cnt,
                                                 static_cast<int>(p->attn_cnt_ints), s, prefix,
                                                 chunked ? max_pages * c.kv_page_size : 0));
  const int32_t* layer_sched0 = p->attn_cnt + (p->attn_cnt_ints - c.num_layers);
  CUtensorMap ta, ta2, tq, tk, tv;
  if (!make_tmap_bf16_2d(&ta, p->a, act_rows(p, T), p->H, p->H, 128, 64) ||
      !make_tmap_bf16_2d(&ta2, p->a2, act_rows(p, T), p->K2, p->K2, 128, 64) ||
      !make_tmap_bf16_2d(&tq, p->q, T, p->q_cols, p->q_cols, 128, 64) ||
      !make_tmap_bf16_2d(&tk, p->k, T, p->kv_cols, p->kv_cols, attn_kv_box_rows(), 64) ||
      !make_tmap_bf16_2d(&tv, p->v, T, p->kv_cols, p->kv_cols, attn_kv_box_rows(), 64))
    return CC_ERR_CUDA;
  const int tiles = attn_max_tiles(T, n_seqs);
  // the output projection's epilogue also normalises the updated rows for the next layer
  const bool ln_fused = gemm_resid_ln_ok(T, p->H, p->K2);
  for (int i = 0; i < c.num_layers; ++i) {
    const bool sliding = p->types[i] == CC_SLIDING;
    // layer 0's LayerNorm: with token input it ran with the embedding merge; later layers'
    // ran in the previous layer's output projection when ln_fused
    const bool a_ready = i == 0 ? emb != nullptr : ln_fused;
    if (!a_ready)
      CC_TIMED(p, CC_K_LAYERNORM, s, launch_layernorm_bf16(hidden, static_cast<const __nv_bfloat16*>(p->layers[i].ln_w),
                                            p->a, T, p->H, c.layer_norm_eps, nullptr, s));
    EpiParams e1;
    e1.q_cols = p->q_cols;
    e1.kv_cols = p->kv_cols;
    e1.n_kv = p->nkv;
    e1.rope = sliding ? p->rope : nullptr;
    e1.q_out = p->q;
    e1.ld_q = p->q_cols;
    e1.k_out = p->k;
    e1.v_out = p->v;
    e1.ld_kv = p->kv_cols;
    if (kv) {
      e1.k_pool = static_cast<__nv_bfloat16*>(kv->k[i]);
      e1.v_pool = static_cast<__nv_bfloat16*>(kv->v[i]);
      e1.kv_slot = p->kv_slot;
      e1.page_size = c.kv_page_size;
    }
    e1.act_out = p->a2 + p->q_cols;
    e1.ld_act = p->K2;
    CC_TIMED(p, CC_K_GEMM_QKV_MLP, s, plan_gemm(ta, p->w1_128[i], p->w1_256[i], T, p->N1, p->H, EPI_QKV_MLP, e1,
                              p->err, s));
    AttnScratch sc;
    sc.part_o = p->attn_part_o;
    sc.part_ml = p->attn_part_ml;
    sc.counters = p->attn_cnt;
    sc.sched = const_cast<int32_t*>(layer_sched0) + i;
    AttnPaged paged;
    CUtensorMap pk = tk, pv = tv;
    if (chunked) {
      const uint64_t pool_rows = (uint64_t)kv->n_pages * p->nkv * c.kv_page_size;
      if (!make_tmap_bf16_2d(&pk, kv->k[i], pool_rows, p->d, p->d, 16, 64) ||
          !make_tmap_bf16_2d(&pv, kv->v[i], pool_rows, p->d, p->d, 16, 64))
        return CC_ERR_CUDA;
      paged.pt = page_table;
      paged.max_pages = max_pages;
      paged.n_pages = kv->n_pages;
    }
    CC_TIMED(p, CC_K_ATTN_PREFILL, s, launch_attn_prefill(tq, pk, pv, p->a2, p->K2, sliding ? p->tiles_s : p->tiles_f,
                                        p->n_tiles + (sliding ? 0 : 1), tiles, p->nq, p->nkv,
                                        sliding ? c.sliding_window : 0, sc, p->err, s, paged));
    EpiParams e2;
    e2.c = hidden;
    e2.ldc = p->H;
    if (i < n_ds) {
      e2.ds_map = p->ds_map;
      e2.ds = static_cast<const __nv_bfloat16*>(ds_feats[i]);
    }
    int epi2 = EPI_RESID;
    if (ln_fused && i + 1 < c.num_layers) {
      epi2 = EPI_RESID_LN;
      e2.ln_gamma = static_cast<const __nv_bfloat16*>(p->layers[i + 1].ln_w);
      e2.ln_out = p->a;   // layer i + 1's GEMM-1 operand (layer i's GEMM-1 has read it)
      e2.ln_part = p->ln_part;
      e2.ln_cnt = p->ln_cnt + (size_t)i * p->ln_row_blocks;
      e2.ln_eps = c.layer_norm_eps;
    }
    CC_TIMED(p, CC_K_GEMM_OUT, s, plan_gemm(ta2, p->w2_128[i], p->w2_256[i], T, p->H, p->K2, epi2, e2,
                              p->err, s));
  }
  return CC_OK;
}

static cc_status prefill_f32(cc_layer_plan* p, float* hidden, const int32_t* pos, const int32_t* cu,
                             int n_seqs, int T, const int32_t* ds_rows, int n_ds_rows,
                             const void* const* ds_feats, int n_ds, cudaStream_t s) {
  const cc_model_config& c = p->cfg;
  CC_TIMED(p, CC_K_ROPE_TABLE, s, launch_mrope_table(pos, T, p->d, c.rope_theta, c.mrope_section, c.mrope_layout, p->rope, s));
  for (int i = 0; i < c.num_layers; ++i) {
    const bool sliding = p->types[i] == CC_SLIDING;
    CC_TIMED(p, CC_K_F32_PATH, s, launch_layernorm_f32(hidden, static_cast<const float*>(p->layers[i].ln_w), p->af,
                                         T, p->H, c.layer_norm_eps, nullptr, s));
    CC_TIMED(p, CC_K_F32_PATH, s, launch_gemm_f32(p->af, p->H, static_cast<const float*>(p->layers[i].w1), p->H,
                                    p->yf, p->N1, T, p->N1, p->H, 1.f, 0, s));
    CC_TIMED(p, CC_K_F32_PATH, s, launch_qkv_mlp_f32(p->yf, p->N1, T, p->q_cols, p->kv_cols, p->d, p->I,
                                       sliding ? p->rope : nullptr, p->qf, p->kf, p->vf,
                                       p->a2f + p->q_cols, p->K2, s));
    CC_TIMED(p, CC_K_F32_PATH, s, launch_attn_f32(p->qf, p->kf, p->vf, p->a2f, p->K2, cu, n_seqs, T, p->nq,
                                    p->nkv, p->d, sliding ? c.sliding_window : 0, s));
    CC_TIMED(p, CC_K_F32_PATH, s, launch_gemm_f32(p->a2f, p->K2, static_cast<const float*>(p->layers[i].w2),
                                    p->K2, hidden, p->H, T, p->H, p->K2, 1.f, 1, s));
    if (i < n_ds)
      CC_TIMED(p, CC_K_F32_PATH, s, launch_ds_add_f32(hidden, p->H, ds_rows, n_ds_rows,
                                        static_cast<const float*>(ds_feats[i]), s));
  }
  return CC_OK;
}

extern "C" cc_status cc_prefill_forward(cc_layer_plan* p, float* hidden, const int32_t* pos_thw,
                                        const int32_t* cu_seqlens, int32_t n_seqs,
                                        int32_t total_tokens, const int32_t* ds_rows,
                                        int32_t n_ds_rows, const void* const* ds_feats,
                                        int32_t n_deepstack, const cc_kv_pool* kv,
                                        const int32_t* page_table, int32_t max_pages,
                                        void* stream) {
  if (!p) return CC_ERR_INVALID_ARG;
  if (total_tokens < 0 || total_tokens > p->T_max || n_seqs < 1 || n_deepstack < 0 ||
      n_deepstack > p->cfg.num_layers || n_ds_rows < 0)
    return CC_ERR_INVALID_ARG;
  if (total_tokens == 0) return CC_OK;
  if (!hidden || !pos_thw || !cu_seqlens) return CC_ERR_INVALID_ARG;
  if (n_deepstack > 0 && n_ds_rows > 0) {
    if (!ds_rows || !ds_feats) return CC_ERR_INVALID_ARG;
    for (int i = 0; i < n_deepstack; ++i)
      if (!ds_feats[i]) return CC_ERR_INVALID_ARG;
  }
  const int n_ds = n_ds_rows > 0 ? n_deepstack : 0;
  if (kv) {
    if (!p->bf16) return CC_ERR_UNSUPPORTED;
    if (!kv->k || !kv->v || kv->n_pages <= 0 || !page_table || max_pages <= 0)
      return CC_ERR_INVALID_ARG;
    for (int i = 0; i < p->cfg.num_layers; ++i)
      if (!kv->k[i] || !kv->v[i]) return CC_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p->bf16)
    return prefill_bf16(p, hidden, pos_thw, cu_seqlens, n_seqs, total_tokens, ds_rows, n_ds_rows,
                        ds_feats, n_ds, kv, page_table, max_pages, s);
  return prefill_f32(p, hidden, pos_thw, cu_seqlens, n_seqs, total_tokens, ds_rows, n_ds_rows,
                     ds_feats, n_ds, s);
}

extern "C" cc_status cc_prefill_forward_tokens(
    cc_layer_plan* p, const int32_t* token_ids, const int32_t* mm_rows, const void* mm_embeds,
    int32_t n_mm_rows, float* hidden, const int32_t* pos_thw, const int32_t* cu_seqlens,
    int32_t n_seqs, int32_t total_tokens, const int32_t* ds_rows, int32_t n_ds_rows,
    const void* const* ds_feats, int32_t n_deepstack, const cc_kv_pool* kv,
    const int32_t* page_table, int32_t max_pages, void* stream) {
  if (!p) return CC_ERR_INVALID_ARG;
  if (!p->bf16) return CC_ERR_UNSUPPORTED;
  if (total_tokens < 0 || total_tokens > p->T_max || n_seqs < 1 || n_deepstack < 0 ||
      n_deepstack > p->cfg.num_layers || n_ds_rows < 0 || n_mm_rows < 0)
    return CC_ERR_INVALID_ARG;
  if (total_tokens == 0) return CC_OK;
  if (!token_ids || !hidden || !pos_thw || !cu_seqlens) return CC_ERR_INVALID_ARG;
  if (n_mm_rows > 0 && (!mm_rows || !mm_embeds)) return CC_ERR_INVALID_ARG;
  if (n_deepstack > 0 && n_ds_rows > 0) {
    if (!ds_rows || !ds_feats) return CC_ERR_INVALID_ARG;
    for (int i = 0; i < n_deepstack; ++i)
      if (!ds_feats[i]) return CC_ERR_INVALID_ARG;
  }
  if (kv) {
    if (!kv->k || !kv->v || kv->n_pages <= 0 || !page_table || max_pages <= 0)
      return CC_ERR_INVALID_ARG;
    for (int i = 0; i < p->cfg.num_layers; ++i)
      if (!kv->k[i] || !kv->v[i]) return CC_ERR_INVALID_ARG;
  }
  const EmbedIn emb{token_ids, mm_rows, static_cast<const __nv_bfloat16*>(mm_embeds), n_mm_rows};
  const int n_ds = n_ds_rows > 0 ? n_deepstack : 0;
  return prefill_bf16(p, hidden, pos_thw, cu_seqlens, n_seqs, total_tokens, ds_rows, n_ds_rows,
                      ds_feats, n_ds, kv, page_table, max_pages, static_cast<cudaStream_t>(stream),
                      &emb);
}

extern "C" cc_status cc_prefill_forward_chunk(
    cc_layer_plan* p, float* hidden, const int32_t* pos_thw, const int32_t* cu_seqlens,
    int32_t n_seqs, int32_t total_tokens, const int32_t* prefix_lens, const int32_t* ds_rows,
    int32_t n_ds_rows, const void* const* ds_feats, int32_t n_deepstack, const cc_kv_pool* kv,
    const int32_t* page_table, int32_t max_pages, void* stream) {
  if (!p) return CC_ERR_INVALID_ARG;
  if (!p->bf16) return CC_ERR_UNSUPPORTED;
  if (p->cfg.kv_page_size != 16 || p->d != 128) return CC_ERR_UNSUPPORTED;
  if (total_tokens < 0 || total_tokens > p->T_max || n_seqs < 1 || n_deepstack < 0 ||
      n_deepstack > p->cfg.num_layers || n_ds_rows < 0)
    return CC_ERR_INVALID_ARG;
  if (total_tokens == 0) return CC_OK;
  if (!hidden || !pos_thw || !cu_seqlens || !prefix_lens || !kv || !page_table || max_pages <= 0)
    return CC_ERR_INVALID_ARG;
  if (!kv->k || !kv->v || kv->n_pages <= 0) return CC_ERR_INVALID_ARG;
  for (int i = 0; i < p->cfg.num_layers; ++i)
    if (!kv->k[i] || !kv->v[i]) return CC_ERR_INVALID_ARG;
  if (n_deepstack > 0 && n_ds_rows > 0) {
    if (!ds_rows || !ds_feats) return CC_ERR_INVALID_ARG;
    for (int i = 0; i < n_deepstack; ++i)
      if (!ds_feats[i]) return CC_ERR_INVALID_ARG;
  }
  const int n_ds = n_ds_rows > 0 ? n_deepstack : 0;
  return prefill_bf16(p, hidden, pos_thw, cu_seqlens, n_seqs, total_tokens, ds_rows, n_ds_rows,
                      ds_feats, n_ds, kv, page_table, max_pages, static_cast<cudaStream_t>(stream),
                      nullptr, prefix_lens);
}

static cc_status decode_step(cc_layer_plan* p, float* hidden, const int32_t* pos_thw,
                             const int32_t* seq_lens, const int32_t* page_table, int32_t max_pages,
                             int32_t batch, const cc_kv_pool* kv, void* stream, bool q4) {
  if (!p) return CC_ERR_INVALID_ARG;
  if (!p->bf16) return CC_ERR_UNSUPPORTED;
  if (batch < 0 || batch > p->T_max) return CC_ERR_INVALID_ARG;
  if (q4 && (p->layers_q4.empty() || batch > 128)) return CC_ERR_INVALID_ARG;
  if (batch == 0) return CC_OK;
  if (!hidden || !pos_thw || !seq_lens || !page_table || max_pages <= 0 || !kv || !kv->k ||
      !kv->v || kv->n_pages <= 0)
    return CC_ERR_INVALID_ARG;
  for (int i = 0; i < p->cfg.num_layers; ++i)
    if (!kv->k[i] || !kv->v[i]) return CC_ERR_INVALID_ARG;
  const cc_model_config& c = p->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t need = decode_scratch_floats(batch, p->nq, max_pages);
  if (need > p->dec_scratch_floats) {
    if (p->dec_scratch) {
      CC_CHECK_CUDA(cudaStreamSynchronize(s));
      cudaFree(p->dec_scratch);
      p->dec_scratch = nullptr;
      p->dec_scratch_floats = 0;
    }
    if (cudaMalloc(&p->dec_scratch, need * sizeof(float)) != cudaSuccess) return CC_ERR_OOM;
    p->dec_scratch_floats = need;
  }
  DecodeScratch scr;
  scr.part_o = p->dec_scratch;
  scr.part_ml = p->dec_scratch + (size_t)batch * p->nq * decode_splits(max_pages) * 128;

  CC_TIMED(p, CC_K_ROPE_TABLE, s, launch_mrope_table(pos_thw, batch, p->d, c.rope_theta, c.mrope_section, c.mrope_layout, p->rope, s));
  CC_TIMED(p, CC_K_ROW_MAPS, s, launch_kv_slots_decode(seq_lens, batch, page_table, max_pages, c.kv_page_size,
                                         kv->n_pages, p->kv_slot, p->n_keys, p->err, s));
  CUtensorMap ta, ta2;
  const uint32_t box = q4 ? static_cast<uint32_t>(gemm_q4_token_tile(batch)) : 128u;
  if (!make_tmap_bf16_2d(&ta, p->a, act_rows(p, batch), p->H, p->H, box, 64) ||
      !make_tmap_bf16_2d(&ta2, p->a2, act_rows(p, batch), p->K2, p->K2, box, 64))
    return CC_ERR_CUDA;
  for (int i = 0; i < c.num_layers; ++i) {
    const bool sliding = p->types[i] == CC_SLIDING;
    const void* ln_w = q4 ? p->layers_q4[i].ln_w : p->layers[i].ln_w;
    CC_TIMED(p, CC_K_LAYERNORM, s, launch_layernorm_bf16(hidden, static_cast<const __nv_bfloat16*>(ln_w),
                                          p->a, batch, p->H, c.layer_norm_eps, nullptr, s));
    EpiParams e1;
    e1.q_cols = p->q_cols;
    e1.kv_cols = p->kv_cols;
    e1.n_kv = p->nkv;
    e1.rope = sliding ? p->rope : nullptr;
    e1.q_out = p->q;
    e1.ld_q = p->q_cols;
    e1.k_pool = static_cast<__nv_bfloat16*>(kv->k[i]);
    e1.v_pool = static_cast<__nv_bfloat16*>(kv->v[i]);
    e1.kv_slot = p->kv_slot;
    e1.page_size = c.kv_page_size;
    e1.act_out = p->a2 + p->q_cols;
    e1.ld_act = p->K2;
    if (q4)
      CC_TIMED(p, CC_K_GEMM_QKV_MLP, s, launch_gemm_q4(ta, p->layers_q4[i].w1, batch, p->N1, p->H,
                                                      EPI_QKV_MLP, e1, p->err, s));
    else
      CC_TIMED(p, CC_K_GEMM_QKV_MLP, s, plan_gemm(ta, p->w1_128[i], p->w1_256[i], batch, p->N1, p->H, EPI_QKV_MLP, e1,
                                p->err, s));
    CC_TIMED(p, CC_K_ATTN_DECODE, s, launch_attn_decode(p->q, p->q_cols, static_cast<const __nv_bfloat16*>(kv->k[i]),
                                       static_cast<const __nv_bfloat16*>(kv->v[i]), kv->n_pages,
                                       page_table, max_pages, p->n_keys, batch, p->nq, p->nkv,
                                       c.kv_page_size, sliding ? c.sliding_window : 0, scr, p->a2,
                                       p->K2, p->err, s));
    EpiParams e2;
    e2.c = hidden;
    e2.ldc = p->H;
    if (q4)
      CC_TIMED(p, CC_K_GEMM_OUT, s, launch_gemm_q4(ta2, p->layers_q4[i].w2, batch, p->H, p->K2,
                                                  EPI_RESID, e2, p->err, s));
    else
      CC_TIMED(p, CC_K_GEMM_OUT, s, plan_gemm(ta2, p->w2_128[i], p->w2_256[i], batch, p->H, p->K2, EPI_RESID, e2,
                                p->err, s));
  }
  return CC_OK;
}

extern "C" cc_status cc_decode_step(cc_layer_plan* p, float* hidden, const int32_t* pos_thw,
                                    const int32_t* seq_lens, const int32_t* page_table,
                                    int32_t max_pages, int32_t batch, const cc_kv_pool* kv,
                                    void* stream) {
  return decode_step(p, hidden, pos_thw, seq_lens, page_table, max_pages, batch, kv, stream, false);
}

extern "C" cc_status cc_decode_step_q4(cc_layer_plan* p, float* hidden, const int32_t* pos_thw,
                                       const int32_t* seq_lens, const int32_t* page_table,
                                       int32_t max_pages, int32_t batch, const cc_kv_pool* kv,
                                       void* stream) {
  return decode_step(p, hidden, pos_thw, seq_lens, page_table, max_pages, batch, kv, stream, true);
}

extern "C" cc_status cc_logits_q4(cc_layer_plan* p, const float* hidden, const int32_t* rows,
                                  int32_t n_rows, float* logits, void* stream) {
  if (!p) return CC_ERR_INVALID_ARG;
  if (!p->bf16) return CC_ERR_UNSUPPORTED;
  if (p->layers_q4.empty() || n_rows < 0 || n_rows > p->T_max || n_rows > 128)
    return CC_ERR_INVALID_ARG;
  if (n_rows == 0) return CC_OK;
  if (!hidden || !logits) return CC_ERR_INVALID_ARG;
  const cc_model_config& c = p->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CC_TIMED(p, CC_K_LAYERNORM, s, launch_layernorm_bf16(hidden, static_cast<const __nv_bfloat16*>(p->final_ln),
                                        p->a, n_rows, p->H, c.layer_norm_eps, rows, s));
  CUtensorMap ta;
  if (!make_tmap_bf16_2d(&ta, p->a, act_rows(p, n_rows), p->H, p->H,
                         static_cast<uint32_t>(gemm_q4_token_tile(n_rows)), 64))
    return CC_ERR_CUDA;
  EpiParams e;
  e.c = logits;
  e.ldc = p->V;
  e.alpha = c.logit_scale;
  ProfScope ps_(p->prof, CC_K_GEMM_HEAD, s);
  return launch_gemm_q4(ta, p->embed_q4, n_rows, p->V, p->H, EPI_F32, e, p->err, s);
}

extern "C" cc_status cc_logits(cc_layer_plan* p, const float* hidden, const int32_t* rows,
                               int32_t n_rows, float* logits, void* stream) {
  if (!p) return CC_ERR_INVALID_ARG;
  if (n_rows < 0 || n_rows > p->T_max) return CC_ERR_INVALID_ARG;
  if (n_rows == 0) return CC_OK;
  if (!hidden || !logits) return CC_ERR_INVALID_ARG;
  const cc_model_config& c = p->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p->bf16) {
    CC_TIMED(p, CC_K_LAYERNORM, s, launch_layernorm_bf16(hidden, static_cast<const __nv_bfloat16*>(p->final_ln),
                                          p->a, n_rows, p->H, c.layer_norm_eps, rows, s));
    CUtensorMap ta;
    if (!make_tmap_bf16_2d(&ta, p->a, act_rows(p, n_rows), p->H, p->H, 128, 64)) return CC_ERR_CUDA;
    EpiParams e;
    e.c = logits;
    e.ldc = p->V;
    e.alpha = c.logit_scale;
    int bn, splits;
    gemm_choose(n_rows, p->V, p->H, EPI_F32, &bn, &splits);
    if (splits > 1) CC_CHECK_CUDA(cudaMemsetAsync(logits, 0, (size_t)n_rows * p->V * 4, s));
    { ProfScope ps_(p->prof, CC_K_GEMM_HEAD, s); return launch_gemm(ta, p->emb(bn), n_rows, p->V, p->H, bn, splits, EPI_F32, e, p->err, s); }
  }
  CC_TIMED(p, CC_K_LAYERNORM, s, launch_layernorm_f32(hidden, static_cast<const float*>(p->final_ln), p->af, n_rows,
                                       p->H, c.layer_norm_eps, rows, s));
  { ProfScope ps_(p->prof, CC_K_GEMM_HEAD, s); return launch_gemm_f32(p->af, p->H, static_cast<const float*>(p->embed), p->H, logits, p->V,
                         n_rows, p->V, p->H, c.logit_scale, 0, s); }
}

extern "C" cc_status cc_sync(cc_layer_plan* p, void* stream) {
  if (!p) return CC_ERR_INVALID_ARG;
  return read_and_clear(p->err, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ single operations
extern "C" cc_status cc_op_sync(void* stream) {
  return read_and_clear(op_error_flag(), static_cast<cudaStream_t>(stream));
}

extern "C" cc_status cc_op_layernorm(const float* x, const void* gamma, void* out, int32_t rows,
                                     int32_t hidden, float eps, const int32_t* row_idx,
                                     void* stream) {
  if (rows < 0 || hidden <= 0) return CC_ERR_INVALID_ARG;
  if (rows == 0) return CC_OK;
  if (!x || !gamma || !out) return CC_ERR_INVALID_ARG;
  return launch_layernorm_bf16(x, static_cast<const __nv_bfloat16*>(gamma),
                               static_cast<__nv_bfloat16*>(out), rows, hidden, eps, row_idx,
                               static_cast<cudaStream_t>(stream));
}

extern "C" cc_status cc_op_embed_merge(const int32_t* token_ids, int32_t tokens,
                                       const void* embed, int32_t vocab, int32_t hidden_size,
                                       const int32_t* mm_rows, const void* mm_embeds,
                                       int32_t n_mm_rows, float* hidden, const void* ln_w,
                                       float eps, void* ln_out, void* stream) {
  if (tokens < 0 || vocab <= 0 || hidden_size <= 0 || n_mm_rows < 0) return CC_ERR_INVALID_ARG;
  if (tokens == 0) return CC_OK;
  if (!token_ids || !embed || !hidden || (n_mm_rows > 0 && (!mm_rows || !mm_embeds)) ||
      (ln_w != nullptr) != (ln_out != nullptr))
    return CC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* map = nullptr;
  if (n_mm_rows > 0) CC_CHECK_CUDA(cudaMallocAsync(&map, (size_t)tokens * 4, s));
  cc_status st = CC_OK;
  if (map) st = launch_ds_map(mm_rows, n_mm_rows, tokens, map, op_error_flag(), s);
  if (st == CC_OK)
    st = launch_embed_ln(token_ids, static_cast<const __nv_bfloat16*>(embed), vocab, map,
                         static_cast<const __nv_bfloat16*>(mm_embeds), tokens, hidden_size, hidden,
                         static_cast<const __nv_bfloat16*>(ln_w), eps,
                         static_cast<__nv_bfloat16*>(ln_out), op_error_flag(), s);
  if (map) CC_CHECK_CUDA(cudaFreeAsync(map, s));
  return st;
}

extern "C" cc_status cc_op_mrope_table_layout(const int32_t* pos, int32_t tokens,
                                              int32_t head_dim, double theta,
                                              const int32_t* section_host, int32_t layout,
                                              float* table, void* stream) {
  if (tokens < 0 || head_dim <= 0 || head_dim % 2 || !section_host || !(theta > 0))
    return CC_ERR_INVALID_ARG;
  if (section_host[0] < 0 || section_host[1] < 0 || section_host[2] < 0 ||
      section_host[0] + section_host[1] + section_host[2] != head_dim / 2)
    return CC_ERR_INVALID_ARG;
  if (layout != CC_MROPE_INTERLEAVED && layout != CC_MROPE_SECTIONS_HWT) return CC_ERR_INVALID_ARG;
  if (tokens == 0) return CC_OK;
  if (!pos || !table) return CC_ERR_INVALID_ARG;
  return launch_mrope_table(pos, tokens, head_dim, theta, section_host, layout,
                            reinterpret_cast<float2*>(table), static_cast<cudaStream_t>(stream));
}

extern "C" cc_status cc_op_mrope_table(const int32_t* pos, int32_t tokens, int32_t head_dim,
                                       double theta, const int32_t* section_host, float* table,
                                       void* stream) {
  return cc_op_mrope_table_layout(pos, tokens, head_dim, theta, section_host,
                                  CC_MROPE_INTERLEAVED, table, stream);
}

extern "C" cc_status cc_op_gemm_bf16(const void* a, const void* b, float* c, int32_t m, int32_t n,
                                     int32_t k, float alpha, int32_t accumulate, void* stream) {
  if (m < 0 || n <= 0 || k <= 0) return CC_ERR_INVALID_ARG;
  if (m == 0) return CC_OK;
  if (!a || !b || !c) return CC_ERR_INVALID_ARG;
  if (k % 64 != 0 || n % 128 != 0) return CC_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int bn, splits;
  gemm_choose(m, n, k, EPI_F32, &bn, &splits);
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, a, m, k, k, 128, 64) || !make_tmap_bf16_2d(&tb, b, n, k, k, bn, 64))
    return CC_ERR_INVALID_ARG;
  if (splits > 1 && !accumulate) CC_CHECK_CUDA(cudaMemsetAsync(c, 0, (size_t)m * n * 4, s));
  EpiParams e;
  e.c = c;
  e.ldc = n;
  e.alpha = alpha;
  e.accumulate = accumulate || splits > 1;
  return launch_gemm(ta, tb, m, n, k, bn, splits, EPI_F32, e, op_error_flag(), s);
}

extern "C" cc_status cc_op_gemm_q4(const void* a, const void* w_tiled, float* c, int32_t m,
                                   int32_t n, int32_t k, float alpha, int32_t accumulate,
                                   void* stream) {
  if (m < 0 || n <= 0 || k <= 0) return CC_ERR_INVALID_ARG;
  if (m == 0) return CC_OK;
  if (!a || !w_tiled || !c) return CC_ERR_INVALID_ARG;
  if (m > 128 || k % 64 != 0 || n % 128 != 0) return CC_ERR_UNSUPPORTED;
  CUtensorMap ta;
  if (!make_tmap_bf16_2d(&ta, a, m, k, k, static_cast<uint32_t>(gemm_q4_token_tile(m)), 64))
    return CC_ERR_INVALID_ARG;
  EpiParams e;
  e.c = c;
  e.ldc = n;
  e.alpha = alpha;
  e.accumulate = accumulate != 0;
  return launch_gemm_q4(ta, w_tiled, m, n, k, EPI_F32, e, op_error_flag(),
                        static_cast<cudaStream_t>(stream));
}

extern "C" cc_status cc_op_attention_prefill(const void* q, const void* k, const void* v, void* out,
                                             int32_t ld_out, const int32_t* cu_seqlens,
                                             int32_t n_seqs, int32_t tokens, int32_t n_q,
                                             int32_t n_kv, int32_t window, void* stream) {
  if (tokens < 0 || n_seqs < 1 || n_q <= 0 || n_kv <= 0 || n_q % n_kv || window < 0 ||
      ld_out < n_q * 128)
    return CC_ERR_INVALID_ARG;
  if (tokens == 0) return CC_OK;
  if (!q || !k || !v || !out || !cu_seqlens) return CC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bf16_2d(&tq, q, tokens, n_q * 128, n_q * 128, 128, 64) ||
      !make_tmap_bf16_2d(&tk, k, tokens, n_kv * 128, n_kv * 128, attn_kv_box_rows(), 64) ||
      !make_tmap_bf16_2d(&tv, v, tokens, n_kv * 128, n_kv * 128, attn_kv_box_rows(), 64))
    return CC_ERR_INVALID_ARG;
  const int max_tiles = attn_max_tiles(tokens, n_seqs);
  const int groups = attn_groups(n_q, n_kv);
  // one stream-ordered allocation: [n_tiles | split counters, item counter | tiles |
  // partial (max, sum) | partial O]
  const size_t cnt_ints = (size_t)attn_counter_ints(groups) + 1;
  const size_t off_tiles = align256(256 + cnt_ints * 4);
  const size_t off_ml = align256(off_tiles + (size_t)max_tiles * sizeof(AttnTile));
  const size_t off_o = align256(off_ml + attn_part_ml_pairs(n_q, n_kv) * sizeof(float2));
  const size_t bytes = off_o + attn_part_o_floats(n_q, n_kv) * sizeof(float);
  void* scratch = nullptr;
  CC_CHECK_CUDA(cudaMallocAsync(&scratch, bytes, s));
  uint8_t* base = static_cast<uint8_t*>(scratch);
  int32_t* n_tiles = reinterpret_cast<int32_t*>(base);
  AttnScratch sc;
  sc.counters = reinterpret_cast<int32_t*>(base + 256);
  sc.sched = sc.counters + (cnt_ints - 1);
  sc.part_ml = reinterpret_cast<float2*>(base + off_ml);
  sc.part_o = reinterpret_cast<float*>(base + off_o);
  AttnTile* tiles = reinterpret_cast<AttnTile*>(base + off_tiles);
  cc_status st = launch_attn_tiles(cu_seqlens, n_seqs, tokens, groups, window, tiles, n_tiles, 0,
                                   nullptr, nullptr, sc.counters, static_cast<int>(cnt_ints), s);
  if (st == CC_OK)
    st = launch_attn_prefill(tq, tk, tv, static_cast<__nv_bfloat16*>(out), ld_out, tiles, n_tiles,
                             max_tiles, n_q, n_kv, window, sc, op_error_flag(), s);
  CC_CHECK_CUDA(cudaFreeAsync(scratch, s));
  return st;
}

extern "C" cc_status cc_op_attention_decode(const void* q, const void* k_pool, const void* v_pool,
                                            int32_t n_pages, const int32_t* page_table,
                                            int32_t max_pages,
                                            const int32_t* n_keys, int32_t batch, int32_t n_q,
                                            int32_t n_kv, int32_t page_size, int32_t window,
                                            void* out, int32_t ld_out, void* stream) {
  if (batch < 0 || n_q <= 0 || n_kv <= 0 || n_q % n_kv || max_pages <= 0 || window < 0 ||
      page_size <= 0 || ld_out < n_q * 128 || n_pages <= 0)
    return CC_ERR_INVALID_ARG;
  if (batch == 0) return CC_OK;
  if (!q || !k_pool || !v_pool || !page_table || !n_keys || !out) return CC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t floats = decode_scratch_floats(batch, n_q, max_pages);
  void* scratch = nullptr;
  CC_CHECK_CUDA(cudaMallocAsync(&scratch, floats * sizeof(float), s));
  DecodeScratch scr;
  scr.part_o = static_cast<float*>(scratch);
  scr.part_ml = scr.part_o + (size_t)batch * n_q * decode_splits(max_pages) * 128;
  const cc_status st = launch_attn_decode(
      static_cast<const __nv_bfloat16*>(q), n_q * 128, static_cast<const __nv_bfloat16*>(k_pool),
      static_cast<const __nv_bfloat16*>(v_pool), n_pages, page_table, max_pages, n_keys, batch,
      n_q, n_kv, page_size, window, scr, static_cast<__nv_bfloat16*>(out), ld_out,
      op_error_flag(), s);
  CC_CHECK_CUDA(cudaFreeAsync(scratch, s));
  return st;
}

extern "C" void cc_test_stall_next_gemm(void) { test_stall_next_gemm(); }

extern "C" cc_status cc_profile_enable(cc_layer_plan* p, int32_t enable) {
  if (!p) return CC_ERR_INVALID_ARG;
  p->prof.on = enable != 0;
  return CC_OK;
}

extern "C" cc_status cc_profile_read(cc_layer_plan* p, cc_kernel_time* out) {
  if (!p || !out) return CC_ERR_INVALID_ARG;
  for (int i = 0; i < CC_K_COUNT; ++i) out[i] = cc_kernel_time{0, 0.0};
  cc_status st = CC_OK;
  for (auto& r : p->prof.recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
      st = CC_ERR_CUDA;
    if (r.cls >= 0 && r.cls < CC_K_COUNT) {
      out[r.cls].launches += 1;
      out[r.cls].total_ms += ms;
    }
    p->prof.spare.push_back(r.a);
    p->prof.spare.push_back(r.b);
  }
  p->prof.recs.clear();
  return st;
}

extern "C" const char* cc_kernel_class_name(int32_t k) {
  static const char* names[CC_K_COUNT] = {"rope_table", "row_maps", "layernorm", "gemm_qkv_mlp",
                                          "attn_prefill", "gemm_out_resid", "attn_decode",
                                          "gemm_head", "f32_path", "embed_merge"};
  return (k >= 0 && k < CC_K_COUNT) ? names[k] : "unknown";
}
