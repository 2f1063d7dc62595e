// Persistent, warp-specialised bf16 GEMM on the 5th-generation tensor cores (tcgen05).
//
//   C[M, N] = A[M, K] @ B[N, K]^T      A: activations (K-major), B: weights (K-major)
//
// One CTA per SM walks the (m-tile, n-tile, k-split) units of the problem. Per CTA:
//   warp 0      TMA producer: 128 x 64 A tile and BN x 64 B tile per stage, 128-byte swizzle
//   warp 1      MMA issuer: 4 x tcgen05.mma (M=128, N=BN, K=16) per stage into TMEM; owns
//               the TMEM allocation (two accumulators of BN fp32 columns)
//   warps 2..5  epilogue: each reads its 32-lane quarter of the accumulator with
//               tcgen05.ld (one output row per thread) while the MMA warp already fills
//               the other accumulator.
// Epilogues fuse the work that follows each projection of the parallel block (mlxcel
// issue "Cohere Compass / North-Micro-Vision", section "Text decoder forward"):
//   EPI_QKV_MLP  q/k rotation by the interleaved MRoPE table (split rotate-half), q, k, v
//                stored bf16 (k, v also into the paged cache), SwiGLU silu(g) * u -> bf16
//   EPI_RESID    h += o_proj(attn) + down_proj(act) (one GEMM over K = n_q d + I), plus
//                the deepstack row add after the first layers
//   EPI_F32      alpha * acc (+ c): plain GEMM and the tied head's logit_scale footer.
#include "kernels.h"
#include "ptx.cuh"

namespace cc {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;

template <int BN>
struct GemmCfg {
  static constexpr int kStages = (BN == 256) ? 4 : 6;
  static constexpr uint32_t kABytes = kBM * kBK * 2;
  static constexpr uint32_t kBBytes = BN * kBK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;
  static constexpr size_t kSmem = 1024 + kStages * kStageBytes + 256;
};

struct Unit {
  int mt, nt, kb0, kb1;
};

__device__ __forceinline__ Unit decode_unit(int u, int m_tiles, int n_tiles, int splits, int kbt) {
  Unit r;
  const int per_split = m_tiles * n_tiles;
  const int sp = u / per_split;
  const int rem = u - sp * per_split;
  r.mt = rem % m_tiles;  // m fastest: CTAs running together share the weight tile
  r.nt = rem / m_tiles;
  r.kb0 = (kbt * sp) / splits;
  r.kb1 = (kbt * (sp + 1)) / splits;
  return r;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

// Stores 32 consecutive fp32 values of one row as bf16 (64 bytes).
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v) {
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    st_global_v4(dst + i, pack_bf16x2(v[i], v[i + 1]), pack_bf16x2(v[i + 2], v[i + 3]),
                 pack_bf16x2(v[i + 4], v[i + 5]), pack_bf16x2(v[i + 6], v[i + 7]));
  }
}

// One 128-column head chunk (q, k or v) of the fused projection epilogue.
__device__ __forceinline__ void epi_head(uint32_t t_chunk, int row, bool row_ok, bool rotate,
                                         const float2* rope, __nv_bfloat16* dst,
                                         __nv_bfloat16* dst_pool) {
  float lo[32], hi[32];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    tmem_ld32(t_chunk + 32 * half, lo);
    tmem_ld32(t_chunk + 64 + 32 * half, hi);
    if (rotate && row_ok) {
      // y[j] = x[j] cos - x[j+64] sin ; y[j+64] = x[j+64] cos + x[j] sin  (j < 64)
      const float4* cs = reinterpret_cast<const float4*>(rope + (size_t)row * 64 + 32 * half);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float4 c2 = __ldg(cs + j / 2);
        float a = lo[j], b = hi[j];
        lo[j] = a * c2.x - b * c2.y;
        hi[j] = b * c2.x + a * c2.y;
        a = lo[j + 1];
        b = hi[j + 1];
        lo[j + 1] = a * c2.z - b * c2.w;
        hi[j + 1] = b * c2.z + a * c2.w;
      }
    }
    if (row_ok) {
      if (dst) {
        store_bf16x32(dst + 32 * half, lo);
        store_bf16x32(dst + 64 + 32 * half, hi);
      }
      if (dst_pool) {
        store_bf16x32(dst_pool + 32 * half, lo);
        store_bf16x32(dst_pool + 64 + 32 * half, hi);
      }
    }
  }
}

template <int BN, int EPI>
__device__ __forceinline__ void epilogue_tile(uint32_t t_row, int row, int n0, int M, int kb0,
                                              int splits, const EpiParams& ep) {
  const bool row_ok = row < M;
  if constexpr (EPI == EPI_F32 || EPI == EPI_RESID) {
    const bool additive = (EPI == EPI_RESID) || ep.accumulate;
    const __nv_bfloat16* ds_row = nullptr;
    if (EPI == EPI_RESID && ep.ds_map && row_ok && kb0 == 0) {
      const int r = ep.ds_map[row];
      if (r >= 0) ds_row = ep.ds + (size_t)r * ep.ldc;
    }
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      float v[32];
      tmem_ld32(t_row + c, v);
      if (!row_ok) continue;
      float* dst = ep.c + (size_t)row * ep.ldc + n0 + c;
      if (EPI == EPI_F32) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= ep.alpha;
      }
      if (ds_row) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const __nv_bfloat162 d2 =
              *reinterpret_cast<const __nv_bfloat162*>(ds_row + n0 + c + i);
          v[i] += __bfloat162float(d2.x);
          v[i + 1] += __bfloat162float(d2.y);
        }
      }
      if (splits > 1) {
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + i), "f"(v[i]),
                       "f"(v[i + 1]), "f"(v[i + 2]), "f"(v[i + 3])
                       : "memory");
      } else {
        float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float4 o = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          if (additive) {
            const float4 p = d4[i];
            o.x += p.x;
            o.y += p.y;
            o.z += p.z;
            o.w += p.w;
          }
          d4[i] = o;
        }
      }
    }
  } else {  // EPI_QKV_MLP
    const int mlp0 = ep.q_cols + 2 * ep.kv_cols;
#pragma unroll 1
    for (int cc = 0; cc < BN; cc += 128) {
      const int col0 = n0 + cc;
      const uint32_t t_chunk = t_row + cc;
      if (col0 < mlp0) {
        __nv_bfloat16* dst = nullptr;
        __nv_bfloat16* dst_pool = nullptr;
        bool rotate = ep.rope != nullptr;
        int slot = -1;
        if (col0 >= ep.q_cols && ep.kv_slot && row_ok) slot = ep.kv_slot[row];
        if (col0 < ep.q_cols) {
          dst = ep.q_out + (size_t)row * ep.ld_q + col0;
        } else {
          const bool is_k = col0 < ep.q_cols + ep.kv_cols;
          const int off = col0 - ep.q_cols - (is_k ? 0 : ep.kv_cols);
          const int kvh = off >> 7;
          __nv_bfloat16* base = is_k ? ep.k_out : ep.v_out;
          __nv_bfloat16* pool = is_k ? ep.k_pool : ep.v_pool;
          if (base) dst = base + (size_t)row * ep.ld_kv + off;
          if (pool && slot >= 0) {
            const int page = slot / ep.page_size, po = slot - page * ep.page_size;
            dst_pool = pool + (((size_t)page * ep.n_kv + kvh) * ep.page_size + po) * 128;
          }
          rotate = rotate && is_k;
        }
        epi_head(t_chunk, row, row_ok, rotate, ep.rope, dst, dst_pool);
      } else {
        const int blk = (col0 - mlp0) >> 7;  // 64 intermediate columns per block
        __nv_bfloat16* dst = ep.act_out + (size_t)row * ep.ld_act + blk * 64;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float g[32], u[32];
          tmem_ld32(t_chunk + 32 * half, g);
          tmem_ld32(t_chunk + 64 + 32 * half, u);
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 32; ++i) g[i] = silu_f(g[i]) * u[i];
            store_bf16x32(dst + 32 * half, g);
          }
        }
      }
    }
  }
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
           int M, int N, int K, int splits, const EpiParams ep, int* err) {
  using C = GemmCfg<BN>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * C::kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + S * C::kBBytes);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + S);
  const uint32_t tfull0 = smem_u32(bars + 2 * S);
  const uint32_t tempty0 = smem_u32(bars + 2 * S + 2);
  const uint32_t drain = smem_u32(bars + 2 * S + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  int* consumed_slot = reinterpret_cast<int*>(bars + 2 * S + 6);

  pdl_trigger();
  const int warp = warp_id(), lane = lane_id();
  const int m_tiles = (M + kBM - 1) / kBM;
  const int n_tiles = N / BN;
  const int kbt = K / kBK;
  const int units = m_tiles * n_tiles * splits;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 128);
    }
    mbar_init(drain, 1);
    *consumed_slot = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();   // the previous kernel's outputs (A, the residual) are complete from here on

  int issued = 0;  // producer: loads issued
  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit t = decode_unit(u, m_tiles, n_tiles, splits, kbt);
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, err)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * stage;
          mbar_expect_tx(fb, C::kStageBytes);
          tma_load_2d(smem_u32(sA + stage * C::kABytes), &tm_a, fb, kb * kBK, t.mt * kBM);
          tma_load_2d(smem_u32(sB + stage * C::kBBytes), &tm_b, fb, kb * kBK, t.nt * BN);
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16(kBM, BN, 0);
      int stage = 0;
      uint32_t phase = 0;
      int iter = 0, consumed = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++iter) {
        const Unit t = decode_unit(u, m_tiles, n_tiles, splits, kbt);
        const int acc = iter & 1;
        if (!mbar_wait(tempty0 + 8 * acc, ((iter >> 1) & 1) ^ 1, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, err)) {
            ok = false;
            break;
          }
          ++consumed;
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * C::kABytes);
          const uint32_t b0 = smem_u32(sB + stage * C::kBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            tc_mma(d_tmem, desc_kmajor_sw128(a0 + 32 * k), desc_kmajor_sw128(b0 + 32 * k), kIdesc,
                   (kb > t.kb0 || k > 0) ? 1u : 0u);
          }
          tc_commit(empty0 + 8 * stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(tfull0 + 8 * acc);
      }
      // every MMA issued by this thread has completed before TMEM is released
      tc_commit(drain);
      mbar_wait(drain, 0, nullptr);
      *consumed_slot = consumed;
    }
  } else {
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    int iter = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++iter) {
      const Unit t = decode_unit(u, m_tiles, n_tiles, splits, kbt);
      const int acc = iter & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, (iter >> 1) & 1, err))) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + acc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
      const int row = t.mt * kBM + quarter * 32 + lane;
      epilogue_tile<BN, EPI>(t_row, row, t.nt * BN, M, t.kb0, splits, ep);
      tc_fence_before();
      mbar_arrive(tempty0 + 8 * acc);
    }
  }
  __syncthreads();
  if (warp == 0 && lane == 0) {
    // a failed launch may leave loads in flight: wait (bounded) until they have landed
    for (int i = *consumed_slot; i < issued; ++i)
      mbar_wait(full0 + 8 * (i % S), (i / S) & 1, nullptr);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int BN, int EPI>
cc_status launch_t(const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K, int splits,
                   const EpiParams& ep, int* err, cudaStream_t s) {
  using C = GemmCfg<BN>;
  static bool attr_set = false;
  auto kern = k_gemm<BN, EPI>;
  if (!attr_set) {
    CC_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::kSmem)));
    attr_set = true;
  }
  const int m_tiles = (M + kBM - 1) / kBM;
  const int units = m_tiles * (N / BN) * splits;
  const int grid = units < num_sms() ? units : num_sms();
  CC_CHECK_CUDA(launch_pdl(kern, dim3(grid), dim3(kThreads), C::kSmem, s, ta, tb, M, N, K, splits,
                          ep, err));
  return CC_OK;
}

}  // namespace

// Tile shape and K splitting. With one row tile (M <= 128: decode steps, the head on a few
// rows) the GEMM streams its weights from HBM, so the choice maximises the number of CTAs
// reading them: 128-wide tiles and, for additive epilogues, K splits up to one CTA per SM.
// With several row tiles it is tensor bound and the 128 x 256 tile (the one whose operand
// traffic fits shared-memory bandwidth best) is kept unless it leaves most SMs idle.
void gemm_choose(int M, int N, int K, int epi, int* bn, int* splits) {
  const int sms = num_sms();
  const int m_tiles = (M + kBM - 1) / kBM;
  const int kbt = K / kBK;
  int b = (N % 256 == 0) ? 256 : 128;
  if (b == 256 && m_tiles * (N / 256) * 2 < sms) b = 128;
  if (b == 256 && m_tiles == 1 && (N / 256) < sms) b = 128;
  int sp = 1;
  const bool additive = (epi == EPI_RESID) || (epi == EPI_F32);
  if (additive && m_tiles == 1) {
    const int units = N / b;
    while (units * (sp + 1) <= sms && kbt / (sp + 1) >= 4) ++sp;
  }
  *bn = b;
  *splits = sp;
}

cc_status launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K, int bn,
                      int splits, int epi, const EpiParams& ep, int* err, cudaStream_t s) {
  if (M <= 0) return CC_OK;
  if (K % kBK != 0 || N % bn != 0 || splits < 1 || splits > K / kBK)
    return CC_ERR_INVALID_ARG;
  if (bn == 256) {
    switch (epi) {
      case EPI_F32: return launch_t<256, EPI_F32>(ta, tb, M, N, K, splits, ep, err, s);
      case EPI_RESID: return launch_t<256, EPI_RESID>(ta, tb, M, N, K, splits, ep, err, s);
      case EPI_QKV_MLP: return launch_t<256, EPI_QKV_MLP>(ta, tb, M, N, K, 1, ep, err, s);
    }
  } else if (bn == 128) {
    switch (epi) {
      case EPI_F32: return launch_t<128, EPI_F32>(ta, tb, M, N, K, splits, ep, err, s);
      case EPI_RESID: return launch_t<128, EPI_RESID>(ta, tb, M, N, K, splits, ep, err, s);
      case EPI_QKV_MLP: return launch_t<128, EPI_QKV_MLP>(ta, tb, M, N, K, 1, ep, err, s);
    }
  }
  return CC_ERR_INVALID_ARG;
}

}  // namespace cc
