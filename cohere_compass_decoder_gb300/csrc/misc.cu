// Memory-bound helpers of the path: LayerNorm, the MRoPE cos/sin table, row maps.
#include <algorithm>
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace cc {

namespace {

// ---------------------------------------------------------------------- LayerNorm
// mlxcel issue "Cohere Compass / North-Micro-Vision", "Text decoder forward": LayerNorm
// with weight only (no bias), statistics in f32; biased variance, eps inside the root.
// One warp per row; two passes over the row (mean, then centred second moment) kept in
// registers (H / 128 float4 per lane, any multiple of 128 up to 128 * kMaxV4).
constexpr int kMaxV4 = 32;  // H <= 4096 in the register-resident variant

// LayerNorm of one row held by a warp (lane owns columns 4 (lane + 32 i) .. +3, i < NV4):
// mean, then the centred second moment, both reduced across the warp; out = (v - mean) *
// rstd * gamma.
template <int NV4, typename OutT>
__device__ __forceinline__ void ln_row(const float4 (&v)[NV4], const void* __restrict__ gamma,
                                       int gamma_bf16, int H, float eps, OutT* __restrict__ out_row,
                                       int lane) {
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NV4; ++i) s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mean = s / H;
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < NV4; ++i) {
    const float a = v[i].x - mean, b = v[i].y - mean, c = v[i].z - mean, d = v[i].w - mean;
    q += (a * a + b * b) + (c * c + d * d);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
  const float rstd = rsqrtf(q / H + eps);
#pragma unroll
  for (int i = 0; i < NV4; ++i) {
    const int c0 = 4 * (lane + 32 * i);
    float g0, g1, g2, g3;
    if (gamma_bf16) {
      const __nv_bfloat162* gp = reinterpret_cast<const __nv_bfloat162*>(
          reinterpret_cast<const __nv_bfloat16*>(gamma) + c0);
      const float2 a = __bfloat1622float2(gp[0]), b = __bfloat1622float2(gp[1]);
      g0 = a.x; g1 = a.y; g2 = b.x; g3 = b.y;
    } else {
      const float4 gg = reinterpret_cast<const float4*>(gamma)[c0 / 4];
      g0 = gg.x; g1 = gg.y; g2 = gg.z; g3 = gg.w;
    }
    const float y0 = (v[i].x - mean) * rstd * g0, y1 = (v[i].y - mean) * rstd * g1;
    const float y2 = (v[i].z - mean) * rstd * g2, y3 = (v[i].w - mean) * rstd * g3;
    if constexpr (sizeof(OutT) == 2) {
      uint2 pk;
      pk.x = pack_bf16x2(y0, y1);
      pk.y = pack_bf16x2(y2, y3);
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out_row) + c0) = pk;
    } else {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(out_row) + c0) =
          make_float4(y0, y1, y2, y3);
    }
  }
}

template <int NV4, typename OutT>
__global__ void __launch_bounds__(256)
    k_layernorm(const float* __restrict__ x, const void* __restrict__ gamma,
                OutT* __restrict__ out, int rows, int H, float eps,
                const int32_t* __restrict__ row_idx, int gamma_bf16) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int src = row_idx ? row_idx[row] : row;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)src * H);
  float4 v[NV4];
#pragma unroll
  for (int i = 0; i < NV4; ++i) v[i] = xr[lane + 32 * i];
  ln_row<NV4, OutT>(v, gamma, gamma_bf16, H, eps, out + (size_t)row * H, lane);
}

// ---------------------------------------------------------------------- embedding merge
// The step before the path (mlxcel issue "Text decoder forward": h = embed_tokens(tokens);
// mlxcel VLM manual "Stage 4: Embedding Merge"; FreeToken PR 454 "How it fits together":
// the image rows take the gathered features, mm_rows -> mm_embeds, by one index copy),
// fused with the first LayerNorm: one warp per row reads the bf16 source row (the image
// feature when mm_map[row] >= 0, else the token's embedding row), writes it to h in f32 and,
// when ln_out is not null, writes LayerNorm(h row) with the same arithmetic as k_layernorm.
template <int NV4>
__global__ void __launch_bounds__(256)
    k_embed_ln(const int32_t* __restrict__ tok, const __nv_bfloat16* __restrict__ embed, int V,
               const int32_t* __restrict__ mm_map, const __nv_bfloat16* __restrict__ mm_embeds,
               int rows, int H, float* __restrict__ h, const __nv_bfloat16* __restrict__ ln_w,
               float eps, __nv_bfloat16* __restrict__ ln_out, int* err) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int f = mm_map ? mm_map[row] : -1;
  const __nv_bfloat16* src = nullptr;
  if (f >= 0) {
    src = mm_embeds + (size_t)f * H;
  } else {
    const int t = tok[row];
    if (t >= 0 && t < V) src = embed + (size_t)t * H;
    else if (lane == 0) set_error(err, CC_DEV_CHECK);   // the row becomes zeros
  }
  float4 v[NV4];
#pragma unroll
  for (int i = 0; i < NV4; ++i) {
    const int c0 = 4 * (lane + 32 * i);
    if (src) {
      const uint2 raw = *reinterpret_cast<const uint2*>(src + c0);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
      v[i] = make_float4(a.x, a.y, b.x, b.y);
    } else {
      v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    *reinterpret_cast<float4*>(h + (size_t)row * H + c0) = v[i];
  }
  if (ln_out) ln_row<NV4, __nv_bfloat16>(v, ln_w, 1, H, eps, ln_out + (size_t)row * H, lane);
}

template <typename OutT>
cc_status launch_ln(const float* x, const void* gamma, OutT* out, int rows, int H, float eps,
                    const int32_t* row_idx, int gamma_bf16, cudaStream_t s) {
  if (rows <= 0) return CC_OK;
  if (H % 128 != 0 || H > 128 * kMaxV4) return CC_ERR_UNSUPPORTED;
  const int nv4 = H / 128;
  const dim3 grid((rows + 7) / 8);
  cudaError_t e = cudaSuccess;
#define CC_LN_CASE(N) \
  case N: e = launch_pdl(k_layernorm<N, OutT>, grid, dim3(256), 0, s, x, gamma, out, rows, H, eps, row_idx, gamma_bf16); break;
  switch (nv4) {
    CC_LN_CASE(1) CC_LN_CASE(2) CC_LN_CASE(3) CC_LN_CASE(4) CC_LN_CASE(5) CC_LN_CASE(6) CC_LN_CASE(7) CC_LN_CASE(8)
    CC_LN_CASE(9) CC_LN_CASE(10) CC_LN_CASE(11) CC_LN_CASE(12) CC_LN_CASE(13) CC_LN_CASE(14) CC_LN_CASE(15) CC_LN_CASE(16)
    CC_LN_CASE(17) CC_LN_CASE(18) CC_LN_CASE(19) CC_LN_CASE(20) CC_LN_CASE(21) CC_LN_CASE(22) CC_LN_CASE(23) CC_LN_CASE(24)
    CC_LN_CASE(25) CC_LN_CASE(26) CC_LN_CASE(27) CC_LN_CASE(28) CC_LN_CASE(29) CC_LN_CASE(30) CC_LN_CASE(31) CC_LN_CASE(32)
    default: return CC_ERR_UNSUPPORTED;
  }
#undef CC_LN_CASE
  CC_CHECK_CUDA(e);
  return CC_OK;
}

// ---------------------------------------------------------------------- MRoPE table
// mlxcel issue "Text decoder forward", interleaved MRoPE: frequency j (< d/2) reads the h
// axis when j % 3 == 1 and j < 3 s_h, the w axis when j % 3 == 2 and j < 3 s_w, else t;
// angle = pos[axis] * theta^(-2j/d). theta^(-2j/d) is evaluated once per call on the host
// in double precision; the angle (up to ~1e5 rad) is formed and reduced modulo 2*pi in
// double precision; sincosf then sees |r| <= pi.
// per rotary index k: the position axis it reads and its inverse frequency
struct MropeTbl {
  double v[64];
  int32_t axis[64];
};

__global__ void k_mrope_table(const int32_t* __restrict__ pos, int T, int half, const MropeTbl f,
                              float2* __restrict__ table) {
  pdl_trigger();
  pdl_wait();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= T * half) return;
  const int t = idx / half, j = idx - t * half;
  const double ang = static_cast<double>(pos[f.axis[j] * T + t]) * f.v[j];
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  const double r = fma(-two_pi, rint(ang * inv_two_pi), ang);
  float sn, cs;
  sincosf(static_cast<float>(r), &sn, &cs);
  table[idx] = make_float2(cs, sn);
}

// ---------------------------------------------------------------------- row maps
__global__ void k_fill_i32(int32_t* p, int n, int32_t v) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = v;
}

__global__ void k_ds_map(const int32_t* __restrict__ rows, int n_rows, int T,
                         int32_t* __restrict__ map, int* err) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n_rows) return;
  const int t = rows[r];
  if (t < 0 || t >= T) {
    set_error(err, CC_DEV_CHECK);
    return;
  }
  map[t] = r;
}

// Both steps in one block when the map is short: -1 everywhere, then the row entries.
__global__ void __launch_bounds__(1024)
    k_row_map_1blk(const int32_t* __restrict__ rows, int n_rows, int T,
                   int32_t* __restrict__ map, int* err) {
  pdl_trigger();
  pdl_wait();
  for (int t = threadIdx.x; t < T; t += blockDim.x) map[t] = -1;
  __syncthreads();
  for (int r = threadIdx.x; r < n_rows; r += blockDim.x) {
    const int t = rows[r];
    if (t < 0 || t >= T) set_error(err, CC_DEV_CHECK);
    else map[t] = r;
  }
}

__global__ void k_kv_slots_prefill(const int32_t* __restrict__ cu, int n_seqs, int T,
                                   const int32_t* __restrict__ pt, int max_pages, int ps,
                                   int n_pages, int32_t* __restrict__ slots, int* err,
                                   const int32_t* __restrict__ prefix) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int lo = 0, hi = n_seqs;  // sequence s with cu[s] <= t < cu[s+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid;
  }
  const int pos = t - cu[lo] + (prefix ? prefix[lo] : 0);
  const int pi = pos / ps;
  int slot = -1;
  if (pos >= 0 && pi < max_pages) {
    const int page = pt[(size_t)lo * max_pages + pi];
    if (page >= 0 && page < n_pages) slot = page * ps + (pos - pi * ps);
  }
  if (slot < 0) set_error(err, CC_DEV_CHECK);
  slots[t] = slot;
}

__global__ void k_kv_slots_decode(const int32_t* __restrict__ seq_lens, int batch,
                                  const int32_t* __restrict__ pt, int max_pages, int ps,
                                  int n_pages, int32_t* __restrict__ slots,
                                  int32_t* __restrict__ n_keys, int* err) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int pos = seq_lens[b];
  const int pi = pos / ps;
  int slot = -1;
  if (pos >= 0 && pi < max_pages) {
    const int page = pt[(size_t)b * max_pages + pi];
    if (page >= 0 && page < n_pages) slot = page * ps + (pos - pi * ps);
  }
  if (slot < 0) set_error(err, CC_DEV_CHECK);
  slots[b] = slot;
  n_keys[b] = slot < 0 ? 0 : pos + 1;
}


// The tiled 4-bit weight blocks (layout in kernels.h), one output word per thread-step.
__global__ void k_q4_tile(const uint32_t* __restrict__ words, const uint16_t* __restrict__ scales,
                          const uint16_t* __restrict__ biases, int rows, int K,
                          uint32_t* __restrict__ out) {
  pdl_wait();
  const int G = K / 64, W = K / 8, kqt = (G + 1) / 2;
  constexpr int kWordsPerBlock = kQ4TileBlockBytes / 4;   // 2048 packed + 256 (scale, bias)
  const size_t total = (size_t)(rows / 128) * kqt * kWordsPerBlock;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t b = i / kWordsPerBlock;
    const int e = static_cast<int>(i - b * kWordsPerBlock);
    const int t = static_cast<int>(b / kqt), j = static_cast<int>(b - (size_t)t * kqt);
    uint32_t v = 0;
    if (e < 2048) {
      const int c = e >> 9, r = (e >> 2) & 127, w = 4 * c + (e & 3);
      const int col = 16 * j + w;
      if (col < W) v = words[(size_t)(128 * t + r) * W + col];
    } else {
      const int g = (e - 2048) >> 7, r = (e - 2048) & 127;
      const int grp = 2 * j + g;
      if (grp < G) {
        const size_t src = (size_t)(128 * t + r) * G + grp;
        v = static_cast<uint32_t>(scales[src]) | (static_cast<uint32_t>(biases[src]) << 16);
      }
    }
    out[i] = v;
  }
}

}  // namespace

cc_status launch_layernorm_bf16(const float* x, const __nv_bfloat16* gamma, __nv_bfloat16* out,
                                int rows, int H, float eps, const int32_t* row_idx,
                                cudaStream_t s) {
  return launch_ln<__nv_bfloat16>(x, gamma, out, rows, H, eps, row_idx, 1, s);
}

cc_status launch_layernorm_f32(const float* x, const float* gamma, float* out, int rows, int H,
                               float eps, const int32_t* row_idx, cudaStream_t s) {
  return launch_ln<float>(x, gamma, out, rows, H, eps, row_idx, 0, s);
}

cc_status launch_embed_ln(const int32_t* tok, const __nv_bfloat16* embed, int V,
                          const int32_t* mm_map, const __nv_bfloat16* mm_embeds, int rows, int H,
                          float* h, const __nv_bfloat16* ln_w, float eps, __nv_bfloat16* ln_out,
                          int* err, cudaStream_t s) {
  if (rows <= 0) return CC_OK;
  if (H % 128 != 0 || H > 128 * kMaxV4) return CC_ERR_UNSUPPORTED;
  const dim3 grid((rows + 7) / 8);
  cudaError_t e = cudaSuccess;
#define CC_EMB_CASE(N)                                                                     \
  case N:                                                                                  \
    e = launch_pdl(k_embed_ln<N>, grid, dim3(256), 0, s, tok, embed, V, mm_map, mm_embeds, \
                   rows, H, h, ln_w, eps, ln_out, err);                                    \
    break;
  switch (H / 128) {
    CC_EMB_CASE(1) CC_EMB_CASE(2) CC_EMB_CASE(3) CC_EMB_CASE(4) CC_EMB_CASE(5) CC_EMB_CASE(6) CC_EMB_CASE(7) CC_EMB_CASE(8)
    CC_EMB_CASE(9) CC_EMB_CASE(10) CC_EMB_CASE(11) CC_EMB_CASE(12) CC_EMB_CASE(13) CC_EMB_CASE(14) CC_EMB_CASE(15) CC_EMB_CASE(16)
    CC_EMB_CASE(17) CC_EMB_CASE(18) CC_EMB_CASE(19) CC_EMB_CASE(20) CC_EMB_CASE(21) CC_EMB_CASE(22) CC_EMB_CASE(23) CC_EMB_CASE(24)
    CC_EMB_CASE(25) CC_EMB_CASE(26) CC_EMB_CASE(27) CC_EMB_CASE(28) CC_EMB_CASE(29) CC_EMB_CASE(30) CC_EMB_CASE(31) CC_EMB_CASE(32)
    default: return CC_ERR_UNSUPPORTED;
  }
#undef CC_EMB_CASE
  CC_CHECK_CUDA(e);
  return CC_OK;
}

cc_status launch_mrope_table(const int32_t* pos, int T, int head_dim, double theta,
                             const int32_t section[3], int layout, float2* table, cudaStream_t s) {
  if (T <= 0) return CC_OK;
  const int half = head_dim / 2;
  if (half > 64) return CC_ERR_UNSUPPORTED;
  if (layout != CC_MROPE_INTERLEAVED && layout != CC_MROPE_SECTIONS_HWT) return CC_ERR_INVALID_ARG;
  // the interleaved assignment: index j reads h when j % 3 == 1 and j < 3 section[1], w when
  // j % 3 == 2 and j < 3 section[2], else t, at frequency j
  int axis_il[64];
  for (int j = 0; j < half; ++j)
    axis_il[j] = (j % 3 == 1 && j < 3 * section[1]) ? 1 : (j % 3 == 2 && j < 3 * section[2]) ? 2 : 0;
  MropeTbl f{};
  if (layout == CC_MROPE_INTERLEAVED) {
    for (int j = 0; j < half; ++j) {
      f.axis[j] = axis_il[j];
      f.v[j] = std::pow(theta, -2.0 * j / head_dim);
    }
  } else {
    // contiguous sections h, w, t, each holding its axis's frequencies in increasing order
    int k = 0;
    const int order[3] = {1, 2, 0};
    for (int a : order)
      for (int j = 0; j < half; ++j)
        if (axis_il[j] == a) {
          f.axis[k] = a;
          f.v[k] = std::pow(theta, -2.0 * j / head_dim);
          ++k;
        }
  }
  const int n = T * half;
  CC_CHECK_CUDA(launch_pdl(k_mrope_table, dim3((n + 255) / 256), dim3(256), 0, s, pos, T, half, f,
                            table));
  return CC_OK;
}

cc_status launch_ds_map(const int32_t* rows, int n_rows, int T, int32_t* map, int* err,
                        cudaStream_t s) {
  if (T <= 0) return CC_OK;
  if (T <= 65536) {
    CC_CHECK_CUDA(launch_pdl(k_row_map_1blk, dim3(1), dim3(1024), 0, s, rows, n_rows, T, map, err));
    return CC_OK;
  }
  CC_CHECK_CUDA(launch_pdl(k_fill_i32, dim3((T + 255) / 256), dim3(256), 0, s, map, T, -1));
  if (n_rows > 0) {
    CC_CHECK_CUDA(launch_pdl(k_ds_map, dim3((n_rows + 255) / 256), dim3(256), 0, s, rows, n_rows, T,
                              map, err));
  }
  return CC_OK;
}

cc_status launch_kv_slots_prefill(const int32_t* cu_seqlens, int n_seqs, int T,
                                  const int32_t* page_table, int max_pages, int page_size,
                                  int n_pages, int32_t* slots, int* err, cudaStream_t s,
                                  const int32_t* prefix) {
  if (T <= 0) return CC_OK;
  CC_CHECK_CUDA(launch_pdl(k_kv_slots_prefill, dim3((T + 255) / 256), dim3(256), 0, s, cu_seqlens,
                            n_seqs, T, page_table, max_pages, page_size, n_pages, slots, err,
                            prefix));
  return CC_OK;
}

cc_status launch_kv_slots_decode(const int32_t* seq_lens, int batch, const int32_t* page_table,
                                 int max_pages, int page_size, int n_pages, int32_t* slots,
                                 int32_t* n_keys, int* err, cudaStream_t s) {
  if (batch <= 0) return CC_OK;
  CC_CHECK_CUDA(launch_pdl(k_kv_slots_decode, dim3((batch + 127) / 128), dim3(128), 0, s, seq_lens,
                            batch, page_table, max_pages, page_size, n_pages, slots, n_keys, err));
  return CC_OK;
}

size_t q4_tiled_bytes(int rows, int K) {
  return (size_t)(rows / 128) * ((K / 64 + 1) / 2) * kQ4TileBlockBytes;
}

cc_status launch_q4_tile(const uint32_t* words, const uint16_t* scales, const uint16_t* biases,
                         int rows, int K, uint8_t* out, cudaStream_t s) {
  if (rows <= 0 || K <= 0) return CC_OK;
  const size_t n = q4_tiled_bytes(rows, K) / 4;
  const int grid = static_cast<int>(std::min<size_t>((n + 255) / 256, 8 * (size_t)num_sms()));
  CC_CHECK_CUDA(launch_pdl(k_q4_tile, dim3(grid), dim3(256), 0, s, words, scales, biases, rows, K,
                           reinterpret_cast<uint32_t*>(out)));
  return CC_OK;
}

}  // namespace cc

