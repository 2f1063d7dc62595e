// The float32 variant of the prefill path (fp32 weights and activations), on the CUDA
// cores. It serves fp32 checkpoints such as the single-layer fp32 workload; every step is
// the same as on the bf16 path (mlxcel issue "Cohere Compass / North-Micro-Vision",
// section "Text decoder forward"), without bf16 storage anywhere.
#include "kernels.h"
#include "ptx.cuh"

namespace cc {

namespace {

// C[M,N] = alpha * A[M,K] B[N,K]^T (+ C): 64 x 64 tiles, 16-deep K steps, 4 x 4 per thread.
__global__ void __launch_bounds__(256)
    k_gemm_f32(const float* __restrict__ A, int lda, const float* __restrict__ B, int ldb,
               float* __restrict__ C, int ldc, int M, int N, int K, float alpha, int accumulate) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 64 * 16; i += 256) {
      const int r = i / 16, kk = i % 16;
      const int gm = m0 + r, gn = n0 + r, gk = k0 + kk;
      As[kk][r] = (gm < M && gk < K) ? A[(size_t)gm * lda + gk] : 0.f;
      Bs[kk][r] = (gn < N && gk < K) ? B[(size_t)gn * ldb + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= N) continue;
      float* p = C + (size_t)gm * ldc + gn;
      *p = alpha * acc[i][j] + (accumulate ? *p : 0.f);
    }
  }
}

// Splits the fused projection output Y (columns q | k | v | SwiGLU blocks of 64 gate +
// 64 up) into rotated q, k, plain v and act = silu(gate) * up.
__global__ void k_qkv_mlp_f32(const float* __restrict__ Y, int ldy, int M, int q_cols,
                              int kv_cols, int d, int inter, const float2* __restrict__ rope,
                              float* __restrict__ q, float* __restrict__ k, float* __restrict__ v,
                              float* __restrict__ act, int ld_act) {
  const int heads_cols = q_cols + 2 * kv_cols;
  const int width = heads_cols + inter;
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long)M * width) return;
  const int row = static_cast<int>(idx / width), col = static_cast<int>(idx % width);
  const float* y = Y + (size_t)row * ldy;
  if (col < heads_cols) {
    const int half = d / 2;
    const int j = col % d;
    float val = y[col];
    const bool is_v = col >= q_cols + kv_cols;
    if (rope && !is_v) {
      const float2 cs = rope[(size_t)row * half + (j % half)];
      val = (j < half) ? y[col] * cs.x - y[col + half] * cs.y : y[col] * cs.x + y[col - half] * cs.y;
    }
    if (col < q_cols) q[(size_t)row * q_cols + col] = val;
    else if (!is_v) k[(size_t)row * kv_cols + (col - q_cols)] = val;
    else v[(size_t)row * kv_cols + (col - q_cols - kv_cols)] = val;
  } else {
    const int i = col - heads_cols;
    const int blk = i / 64, w = i % 64;
    const float g = y[heads_cols + blk * 128 + w], u = y[heads_cols + blk * 128 + 64 + w];
    act[(size_t)row * ld_act + i] = g / (1.0f + expf(-g)) * u;
  }
}

// One warp per (query, head): scores of the visible keys 32 at a time with an online
// max/sum, then a second pass accumulating p * v (lanes over the head dims).
__global__ void k_attn_f32(const float* __restrict__ q, const float* __restrict__ k,
                           const float* __restrict__ v, float* __restrict__ out, int ld_out,
                           const int32_t* __restrict__ cu, int n_seqs, int T, int n_q, int n_kv,
                           int d, int window, float scale) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= T * n_q) return;
  const int t = gw / n_q, h = gw % n_q;
  const int g = h / (n_q / n_kv);
  int s = 0;
  while (s + 1 < n_seqs && cu[s + 1] <= t) ++s;
  const int start = cu[s];
  const int i = t - start;
  const int j0 = window > 0 ? max(0, i - window + 1) : 0;
  const float* qr = q + (size_t)t * n_q * d + (size_t)h * d;
  float m = -INFINITY, l = 0.f;
  for (int jb = j0; jb <= i; jb += 32) {
    const int j = jb + lane;
    float sc = -INFINITY;
    if (j <= i) {
      const float* kr = k + (size_t)(start + j) * n_kv * d + (size_t)g * d;
      float acc = 0.f;
      for (int e = 0; e < d; ++e) acc = fmaf(qr[e], kr[e], acc);
      sc = acc * scale;
    }
    float cm = sc;
    for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
    const float mn = fmaxf(m, cm);
    float p = (j <= i) ? expf(sc - mn) : 0.f;
    for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
    l = l * expf(m - mn) + p;
    m = mn;
  }
  for (int e0 = 0; e0 < d; e0 += 32) {
    const int e = e0 + lane;
    float acc = 0.f;
    for (int j = j0; j <= i; ++j) {
      const float* kr = k + (size_t)(start + j) * n_kv * d + (size_t)g * d;
      float dot = 0.f;
      for (int c = 0; c < d; ++c) dot = fmaf(qr[c], kr[c], dot);
      const float p = expf(dot * scale - m) / l;
      if (e < d) acc = fmaf(p, v[(size_t)(start + j) * n_kv * d + (size_t)g * d + e], acc);
    }
    if (e < d) out[(size_t)t * ld_out + (size_t)h * d + e] = acc;
  }
}

__global__ void k_ds_add_f32(float* __restrict__ h, int H, const int32_t* __restrict__ rows,
                             int n_rows, const float* __restrict__ ds) {
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long)n_rows * H) return;
  const int r = static_cast<int>(idx / H), c = static_cast<int>(idx % H);
  h[(size_t)rows[r] * H + c] += ds[idx];
}

}  // namespace

cc_status launch_gemm_f32(const float* a, int lda, const float* b, int ldb, float* c, int ldc,
                          int M, int N, int K, float alpha, int accumulate, cudaStream_t s) {
  if (M <= 0 || N <= 0) return CC_OK;
  dim3 grid((N + 63) / 64, (M + 63) / 64);
  k_gemm_f32<<<grid, 256, 0, s>>>(a, lda, b, ldb, c, ldc, M, N, K, alpha, accumulate);
  CC_CHECK_CUDA(cudaGetLastError());
  return CC_OK;
}

cc_status launch_qkv_mlp_f32(const float* y, int ldy, int M, int q_cols, int kv_cols,
                             int head_dim, int inter, const float2* rope, float* q, float* k,
                             float* v, float* act, int ld_act, cudaStream_t s) {
  const long n = (long)M * (q_cols + 2 * kv_cols + inter);
  if (n <= 0) return CC_OK;
  k_qkv_mlp_f32<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(
      y, ldy, M, q_cols, kv_cols, head_dim, inter, rope, q, k, v, act, ld_act);
  CC_CHECK_CUDA(cudaGetLastError());
  return CC_OK;
}

cc_status launch_attn_f32(const float* q, const float* k, const float* v, float* out,
                          int ld_out, const int32_t* cu_seqlens, int n_seqs, int T, int n_q,
                          int n_kv, int head_dim, int window, cudaStream_t s) {
  const long warps = (long)T * n_q;
  if (warps <= 0) return CC_OK;
  k_attn_f32<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, s>>>(
      q, k, v, out, ld_out, cu_seqlens, n_seqs, T, n_q, n_kv, head_dim, window,
      1.0f / sqrtf(static_cast<float>(head_dim)));
  CC_CHECK_CUDA(cudaGetLastError());
  return CC_OK;
}

cc_status launch_ds_add_f32(float* h, int H, const int32_t* rows, int n_rows, const float* ds,
                            cudaStream_t s) {
  const long n = (long)n_rows * H;
  if (n <= 0) return CC_OK;
  k_ds_add_f32<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(h, H, rows, n_rows, ds);
  CC_CHECK_CUDA(cudaGetLastError());
  return CC_OK;
}

}  // namespace cc
