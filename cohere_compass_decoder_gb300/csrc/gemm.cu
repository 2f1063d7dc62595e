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
//   EPI_RESID_LN EPI_RESID followed by the next layer's LayerNorm of the updated rows
//                (units in row-block order; a half-full last round runs as tile halves)
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
  int n0, nw;   // first output column and width (decode_item)
};

// Unit u of a launch. m fastest (the default): CTAs running together share the weight tile.
// n fastest (n_fast): the N / BN tiles of one row block are consecutive units, so that they
// run at the same time on distinct CTAs (the residual + LayerNorm epilogue needs that).
__device__ __forceinline__ Unit decode_unit(int u, int m_tiles, int n_tiles, int splits, int kbt,
                                            bool n_fast = false) {
  Unit r;
  const int per_split = m_tiles * n_tiles;
  const int sp = u / per_split;
  const int rem = u - sp * per_split;
  if (n_fast) {
    r.nt = rem % n_tiles;
    r.mt = rem / n_tiles;
  } else {
    r.mt = rem % m_tiles;
    r.nt = rem / m_tiles;
  }
  r.kb0 = (kbt * sp) / splits;
  r.kb1 = (kbt * (sp + 1)) / splits;
  return r;
}

// Work item i of a k_gemm launch. Items before `tail0` are the units of decode_unit, BN
// columns wide. From `tail0` on (only the residual + LayerNorm launch, and only when its last
// round of units would be at most half full) every remaining BN-wide tile is two items of BN/2
// columns with the whole K loop, taken by distinct CTAs, so that the last round costs half a
// tile. tail0 is a whole number of row blocks; the halves of a row block are consecutive.
template <int BN>
__device__ __forceinline__ Unit decode_item(int i, int m_tiles, int n_tiles, int splits, int kbt,
                                            bool n_fast, int tail0) {
  Unit r;
  if (i < tail0) {
    r = decode_unit(i, m_tiles, n_tiles, splits, kbt, n_fast);
    r.n0 = r.nt * BN;
    r.nw = BN;
  } else {
    const int j = i - tail0, per_block = 2 * n_tiles;
    r.mt = tail0 / n_tiles + j / per_block;
    r.nt = -1;
    r.n0 = (j % per_block) * (BN / 2);
    r.nw = BN / 2;
    r.kb0 = 0;
    r.kb1 = kbt;
  }
  return r;
}

// The four epilogue warps (128 threads) synchronise at named barrier 1; __syncthreads uses 0.
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// The four epilogue warps agree on a predicate (AND) at barrier 1, so that all of them leave
// or stay in the unit loop together and the exchange barriers stay matched.
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float2 ld_cg_f2(const float2* p) {
  float2 v;
  asm volatile("ld.global.cg.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
  return v;
}

// Waits (bounded) until *cnt reaches `target`: the other output tiles of a row block, which
// run at the same time on resident CTAs of this launch, count themselves there after storing.
__device__ __forceinline__ bool wait_count(const int32_t* cnt, int target, int* err) {
  const long long t0 = clock64();
  for (uint32_t n = 0;; ++n) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v >= target) return true;
    if ((n & 63u) == 63u) {
      if (err && *reinterpret_cast<volatile int*>(err) != 0) return false;
      if (clock64() - t0 > kWaitTimeoutCycles) {
        set_error(err, CC_DEV_TIMEOUT);
        return false;
      }
    }
    __nanosleep(32);
  }
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

// Loads 32 consecutive fp32 values (128 bytes) of one row.
__device__ __forceinline__ void ld_f32x32(const float* src, float4* v) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = s4[i];
}

// EPI_RESID_LN: the residual update of EPI_RESID followed by the next layer's LayerNorm of
// the updated rows (mlxcel issue "Cohere Compass / North-Micro-Vision", "Text decoder
// forward": a = LayerNorm(h), weight only, biased variance, eps inside the root, statistics
// in f32). The tile covers columns [n0, n0 + nw) of its row block, nw = BN or BN / 2 (a tail
// half). Pass 1 stores h += acc (+ deepstack), keeps the updated h in the tile's own TMEM
// columns (the accumulator is not released before pass 2 ends) and, per 128-column slot of
// the row, stores the slot's (mean, M2) (Chan's update per 32-column chunk); the residual of
// the next chunk is loaded while the current one is processed. The tile adds its slot count
// to the row block's counter and waits (bounded) for the block's other tiles, which run at
// the same time on other CTAs, until all N / 128 slots are in. Pass 2 merges the slots (equal
// counts: mean = the average of the means, M2 = sum M2_i + 128 sum (mean_i - mean)^2) and
// stores bf16((h - mean) * rstd * gamma) from the h held in TMEM. Returns false when the wait
// gave up (every epilogue thread gets the same answer).
template <int BN>
__device__ __forceinline__ bool epilogue_resid_ln(uint32_t t_row, int row, int mt, int n0, int nw,
                                                  int n_slots, int M, const EpiParams& ep,
                                                  int* err, volatile int* flag) {
  const bool row_ok = row < M;
  const __nv_bfloat16* ds_row = nullptr;
  if (ep.ds_map && row_ok) {
    const int r = ep.ds_map[row];
    if (r >= 0) ds_row = ep.ds + (size_t)r * ep.ldc;
  }
  float* hrow = ep.c + (size_t)row * ep.ldc + n0;
  float2* slots = ep.ln_part + (size_t)row * n_slots + (n0 >> 7);
  float mean = 0.f, m2 = 0.f;
  float4 hn[8];
  if (row_ok) ld_f32x32(hrow, hn);
#pragma unroll 1
  for (int c = 0; c < nw; c += 32) {
    float4 hc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) hc[i] = hn[i];
    if (row_ok && c + 32 < nw) ld_f32x32(hrow + c + 32, hn);
    float v[32];
    tmem_ld32(t_row + c, v);
    if (ds_row) {
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const __nv_bfloat162 d2 = *reinterpret_cast<const __nv_bfloat162*>(ds_row + n0 + c + i);
        v[i] += __bfloat162float(d2.x);
        v[i + 1] += __bfloat162float(d2.y);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[4 * i] += hc[i].x;
      v[4 * i + 1] += hc[i].y;
      v[4 * i + 2] += hc[i].z;
      v[4 * i + 3] += hc[i].w;
    }
    tmem_st32(t_row + c, v);
    if (!row_ok) continue;
    float4* d4 = reinterpret_cast<float4*>(hrow + c);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) sum += v[i];
    const float mc = sum * (1.0f / 32.0f);
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float d = v[i] - mc;
      q += d * d;
    }
    const float na = static_cast<float>(c & 127), tot = na + 32.0f;
    const float delta = mc - mean;
    mean += delta * (32.0f / tot);
    m2 += q + delta * delta * (na * 32.0f / tot);
    if ((c & 127) == 96) {   // the slot's 128 columns are in
      slots[c >> 7] = make_float2(mean, m2);
      mean = 0.f;
      m2 = 0.f;
    }
  }
  tmem_st_wait();
  __threadfence();
  epi_bar();
  if (threadIdx.x == 64) {   // the first epilogue thread counts the tile's slots and waits
    int32_t* cnt = ep.ln_cnt + mt;
    atomicAdd(cnt, nw >> 7);
    *flag = wait_count(cnt, n_slots, err) ? 1 : 0;
  }
  epi_bar();
  if (*flag == 0) return false;
  float mu = 0.f, rstd = 0.f;
  if (row_ok) {
    const float2* part = ep.ln_part + (size_t)row * n_slots;
    float sm = 0.f;
#pragma unroll 1
    for (int i = 0; i < n_slots; ++i) sm += ld_cg_f2(part + i).x;
    mu = sm / static_cast<float>(n_slots);
    float q = 0.f;
#pragma unroll 1
    for (int i = 0; i < n_slots; ++i) {
      const float2 pm = ld_cg_f2(part + i);
      const float d = pm.x - mu;
      q += pm.y + 128.0f * d * d;
    }
    rstd = rsqrtf(q / static_cast<float>(n_slots * 128) + ep.ln_eps);
  }
  __nv_bfloat16* dst = ep.ln_out + (size_t)row * ep.ldc + n0;
  const __nv_bfloat16* gam = ep.ln_gamma + n0;
#pragma unroll 1
  for (int c = 0; c < nw; c += 32) {
    float x[32];
    tmem_ld32(t_row + c, x);
    if (!row_ok) continue;
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      const uint4 graw = __ldg(reinterpret_cast<const uint4*>(gam + c + i));
      const float2 g0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&graw.x));
      const float2 g1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&graw.y));
      const float2 g2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&graw.z));
      const float2 g3 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&graw.w));
      st_global_v4(dst + c + i,
                   pack_bf16x2((x[i] - mu) * rstd * g0.x, (x[i + 1] - mu) * rstd * g0.y),
                   pack_bf16x2((x[i + 2] - mu) * rstd * g1.x, (x[i + 3] - mu) * rstd * g1.y),
                   pack_bf16x2((x[i + 4] - mu) * rstd * g2.x, (x[i + 5] - mu) * rstd * g2.y),
                   pack_bf16x2((x[i + 6] - mu) * rstd * g3.x, (x[i + 7] - mu) * rstd * g3.y));
    }
  }
  return true;
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
           const __grid_constant__ CUtensorMap tm_b_half, int M, int N, int K, int splits,
           int tail0, const EpiParams ep, int* err) {
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
  const uint32_t never = smem_u32(bars + 2 * S + 7);   // test hook: nothing arrives on it
  volatile int* ln_flag = reinterpret_cast<volatile int*>(bars + 2 * S + 8);
  constexpr bool kNFast = EPI == EPI_RESID_LN;
  // tail halves (decode_item) only in the 256-wide residual + LayerNorm launch
  constexpr bool kHalves = EPI == EPI_RESID_LN && BN == 256;

  pdl_trigger();
  const int warp = warp_id(), lane = lane_id();
  const int m_tiles = (M + kBM - 1) / kBM;
  const int n_tiles = N / BN;
  const int kbt = K / kBK;
  const int units = m_tiles * n_tiles * splits;
  if (!kHalves) tail0 = units;
  const int items = tail0 + 2 * (units - tail0);

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
    mbar_init(never, 1);
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
    if (kHalves && tail0 < units) tma_prefetch_desc(&tm_b_half);
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
      for (int u = blockIdx.x; u < items && ok; u += gridDim.x) {
        const Unit t = decode_item<BN>(u, m_tiles, n_tiles, splits, kbt, kNFast, tail0);
        const bool half = kHalves && t.nw != BN;
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, err)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * stage;
          mbar_expect_tx(fb, half ? C::kABytes + C::kBBytes / 2 : C::kStageBytes);
          tma_load_2d(smem_u32(sA + stage * C::kABytes), &tm_a, fb, kb * kBK, t.mt * kBM);
          tma_load_2d(smem_u32(sB + stage * C::kBBytes), half ? &tm_b_half : &tm_b, fb, kb * kBK,
                      t.n0);
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
      constexpr uint32_t kIdescHalf = idesc_bf16(kBM, BN / 2, 0);
      int stage = 0;
      uint32_t phase = 0;
      int iter = 0, consumed = 0;
      bool ok = true;
      if (ep.test_stall) ok = mbar_wait(never, 0, err, kTestStallCycles);
      for (int u = blockIdx.x; u < items && ok; u += gridDim.x, ++iter) {
        const Unit t = decode_item<BN>(u, m_tiles, n_tiles, splits, kbt, kNFast, tail0);
        const uint32_t idesc = (kHalves && t.nw != BN) ? kIdescHalf : kIdesc;
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
            tc_mma(d_tmem, desc_kmajor_sw128(a0 + 32 * k), desc_kmajor_sw128(b0 + 32 * k), idesc,
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
    for (int u = blockIdx.x; u < items; u += gridDim.x, ++iter) {
      const Unit t = decode_item<BN>(u, m_tiles, n_tiles, splits, kbt, kNFast, tail0);
      const int acc = iter & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, (iter >> 1) & 1, err))) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + acc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
      const int row = t.mt * kBM + quarter * 32 + lane;
      if constexpr (EPI == EPI_RESID_LN) {
        if (!epilogue_resid_ln<BN>(t_row, row, t.mt, t.n0, t.nw, N >> 7, M, ep, err, ln_flag))
          break;
      } else {
        epilogue_tile<BN, EPI>(t_row, row, t.n0, M, t.kb0, splits, ep);
      }
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
cc_status launch_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap* tb_half, int M,
                   int N, int K, int splits, const EpiParams& ep, int* err, cudaStream_t s) {
  using C = GemmCfg<BN>;
  static std::atomic<bool> smem_set{false};
  auto kern = k_gemm<BN, EPI>;
  CC_CHECK_CUDA(allow_dynamic_smem(kern, C::kSmem, smem_set));
  const int m_tiles = (M + kBM - 1) / kBM;
  const int units = m_tiles * (N / BN) * splits;
  int grid = units < num_sms() ? units : num_sms();
  int tail0 = units;
  if (EPI == EPI_RESID_LN) {
    // the N / BN tiles of a row block are consecutive units: with the grid a multiple of
    // N / BN they run in the same round, each on its own CTA (one resident CTA per SM)
    const int nt = N / BN;
    if (nt > num_sms() || splits != 1) return CC_ERR_UNSUPPORTED;
    grid = std::min(units, (num_sms() / nt) * nt);
    // a last round at most half full runs as 128-column halves of its tiles (decode_item)
    const int rounds = units / grid, rem = units - rounds * grid;
    if (BN == 256 && tb_half && rem > 0 && 2 * rem <= grid) tail0 = rounds * grid;
  }
  CC_CHECK_CUDA(launch_pdl(kern, dim3(grid), dim3(kThreads), C::kSmem, s, ta, tb,
                          tb_half ? *tb_half : tb, M, N, K, splits, tail0, ep, err));
  return CC_OK;
}

// ------------------------------------------------------------------ 4-bit affine weights
// C[M, N] (epilogue) = X[M, K] @ W[N, K]^T with W[n, k] = scale * q + bias per group of 64
// along K (the mlx conversion's affine 4-bit weights, Compass issue "Config (config.json)"),
// for decode-size M <= 128. Weight-stationary: each unit is 128 weight rows (the MMA's M side)
// against all M tokens (its N side, BT = M rounded up to 16), so the tensor work scales with
// the batch, and the weights stream from HBM at a quarter of their bf16 size, pre-tiled
// (launch_q4_tile): the packed words and (scale, bias) words of 128 rows x 128 K are one
// contiguous 9 KB block. 24 warps:
//   warp 0       weight blocks: one bulk copy per block into a 12-stage ring
//   warp 2       token tiles X (bf16, 128-byte swizzle): both 64-K halves of a block per stage
//   warps 1, 3   MMA, two issuing threads (one when BT > 64) taking alternate blocks into
//                separate partial accumulators: per block 8 x tcgen05.mma (M=128, N=BT, K=16) with the
//                dequantised W read from tensor memory (A operand) and X from shared memory.
//                Each K=16 instruction costs ~96 cycles for any N up to 128 and a barrier
//                wait a few hundred, so one issuer would leave the tensor core idle while it
//                waits. The token ring is waited on only here, in order per thread: its
//                stages may be fewer than the groups, so an out-of-order waiter could mistake
//                an older phase's parity for its own.
//   warps 4..7   epilogue: TMEM lane = weight row, column = token
//   warps 8..23  dequantisation, four groups of four warps (one per TMEM lane quarter); group
//                g takes every fourth weight block, so four blocks are in flight. Thread r of
//                a group owns row r: each 32-bit word gives four bf16x2 pairs (the nibble
//                pair goes into the mantissas of 128.0: 0x4300 | q is 128 + q in bf16; 128 is
//                subtracted exactly and fma.rn.bf16x2(scale, q, bias) rounds scale * q + bias
//                once), 32 columns per 64-K half stored to the group's TMEM slot, then the
//                group marks the block ready.
// TMEM: accumulators in columns [0, 256): two unit buffers x two partials of 64 columns when
// BT <= 64 (two MMA issuers), else two unit buffers of 128 (one issuer); W slots (group g,
// half h) at 256 + 32 (2 g + h).
constexpr int kQ4Threads = 768;
constexpr int kQ4Rows = 128;                          // weight rows per unit
constexpr int kQ4QStages = 12;                        // weight blocks: 128 K per stage
constexpr int kQ4Groups = 4;                          // dequantisation warp groups
constexpr int kQ4XMaxStages = 8;                      // token tiles: 128 K per stage
constexpr int kQ4Chunk = 16;                          // epilogue tokens per TMEM load
constexpr uint32_t kQ4QWords = kQ4Rows * 64;          // 8 KB: 128 rows x 64 bytes
constexpr uint32_t kQ4QBytes = kQ4QWords + 2 * kQ4Rows * 4;   // + two groups' (scale, bias)
static_assert(kQ4QBytes == kQ4TileBlockBytes, "tiled weight block");
constexpr uint32_t kQ4XRing = 80 * 1024;              // token ring: 80 KB / (BT * 256) stages
constexpr uint32_t kQ4ExBytes = kQ4Chunk * kQ4Rows * 4;
constexpr uint32_t kQ4OffX = 0;
constexpr uint32_t kQ4OffQ = kQ4OffX + kQ4XRing;
constexpr uint32_t kQ4OffEx = kQ4OffQ + kQ4QStages * kQ4QBytes;
constexpr uint32_t kQ4OffBar = kQ4OffEx + kQ4ExBytes;
constexpr uint32_t kQ4Bars = 2 * kQ4QStages + 2 * kQ4Groups + 2 * kQ4XMaxStages + 7;
constexpr size_t kQ4Smem = 1024 + kQ4OffBar + kQ4Bars * 8 + 64;
static_assert(kQ4Smem <= 232448, "shared memory of the 4-bit GEMM");

__device__ __forceinline__ uint32_t bf2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// four packed bf16x2 words (values 8 w' .. 8 w' + 7 of a row) from one word of nibbles
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t s2, uint32_t b2, uint32_t* o) {
  const uint32_t w4 = w >> 4;
  const uint32_t kMagic = 0x43004300u;              // (128, 128) in bf16
  const uint32_t kOne = 0x3F803F80u;                // (1, 1)
  const uint32_t kNeg128 = 0xC300C300u;             // (-128, -128)
  uint32_t x[4];
  x[0] = __byte_perm(w, w4, 0x4400);                // nibbles 0 (byte 0) and 1 (byte 2)
  x[1] = __byte_perm(w, w4, 0x5511);                // nibbles 2, 3
  x[2] = __byte_perm(w, w4, 0x6622);                // nibbles 4, 5
  x[3] = __byte_perm(w, w4, 0x7733);                // nibbles 6, 7
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t q128 = (x[j] & 0x000F000Fu) | kMagic;   // 128 + q, exact
    const uint32_t q = bf2_fma(q128, kOne, kNeg128);        // q, exact
    o[j] = bf2_fma(s2, q, b2);                              // round(scale * q + bias)
  }
}

// Epilogue of one chunk of kQ4Chunk tokens: v[i] = D[row n][token c0 + i].
template <int EPI>
__device__ __forceinline__ void q4_epilogue_chunk(const float* v, int n, int n0, int c0, int M,
                                                  int kb0, int splits, const EpiParams& ep,
                                                  float* ex) {
  constexpr int CH = kQ4Chunk;
  if constexpr (EPI == EPI_F32 || EPI == EPI_RESID) {
    const bool additive = (EPI == EPI_RESID) || ep.accumulate;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int m = c0 + i;
      if (m >= M) continue;
      float x = (EPI == EPI_F32) ? v[i] * ep.alpha : v[i];
      if (EPI == EPI_RESID && ep.ds_map && kb0 == 0) {
        const int r = ep.ds_map[m];
        if (r >= 0) x += __bfloat162float(ep.ds[(size_t)r * ep.ldc + n0 + n]);
      }
      float* dst = ep.c + (size_t)m * ep.ldc + n0 + n;
      if (splits > 1)
        asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst), "f"(x) : "memory");
      else
        *dst = additive ? *dst + x : x;
    }
  } else {
    // the partner row (n ^ 64): the other half of a rotation pair, or the up row of a gate
    epi_bar();                       // the previous chunk's reads are done
#pragma unroll
    for (int i = 0; i < CH; ++i) ex[i * kQ4Rows + n] = v[i];
    epi_bar();
    const int mlp0 = ep.q_cols + 2 * ep.kv_cols;
    const int p = n ^ 64;
    if (n0 < mlp0) {
      __nv_bfloat16* base = nullptr;
      __nv_bfloat16* pool = nullptr;
      int col = n0 + n, kvh = 0, ld = ep.ld_q;
      bool rotate = ep.rope != nullptr;
      if (n0 < ep.q_cols) {
        base = ep.q_out;
      } else {
        const bool is_k = n0 < ep.q_cols + ep.kv_cols;
        const int off = n0 - ep.q_cols - (is_k ? 0 : ep.kv_cols);
        kvh = off >> 7;
        col = off + n;
        ld = ep.ld_kv;
        base = is_k ? ep.k_out : ep.v_out;
        pool = is_k ? ep.k_pool : ep.v_pool;
        rotate = rotate && is_k;
      }
      const int j = n & 63;
      const bool to_pool = pool && ep.kv_slot;
      // per 8 tokens: every load first (cos / sin, cache slots), then the stores, so that
      // the loads' latency is paid once per 8 tokens, not once per token behind the stores
      constexpr int SB = 8;
#pragma unroll
      for (int i0 = 0; i0 < CH; i0 += SB) {
        float2 cs[SB];
        int slot[SB];
#pragma unroll
        for (int i = 0; i < SB; ++i) {
          const int m = c0 + i0 + i;
          cs[i] = (rotate && m < M) ? __ldg(ep.rope + (size_t)m * 64 + j) : make_float2(1.f, 0.f);
          slot[i] = (to_pool && m < M) ? __ldg(ep.kv_slot + m) : -1;
        }
#pragma unroll
        for (int i = 0; i < SB; ++i) {
          const int m = c0 + i0 + i;
          if (m >= M) continue;
          float y = v[i0 + i];
          if (rotate) {
            // y[j] = x[j] cos - x[j+64] sin ; y[j+64] = x[j+64] cos + x[j] sin  (j < 64)
            const float xp = ex[(i0 + i) * kQ4Rows + p];
            y = n < 64 ? y * cs[i].x - xp * cs[i].y : y * cs[i].x + xp * cs[i].y;
          }
          const __nv_bfloat16 yb = __float2bfloat16_rn(y);
          if (base) base[(size_t)m * ld + col] = yb;
          if (slot[i] >= 0) {
            const int page = slot[i] / ep.page_size, po = slot[i] - page * ep.page_size;
            pool[(((size_t)page * ep.n_kv + kvh) * ep.page_size + po) * 128 + n] = yb;
          }
        }
      }
    } else if (n < 64) {
      const int blk = (n0 - mlp0) >> 7;  // 64 intermediate columns per block
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int m = c0 + i;
        if (m >= M) continue;
        const float u = ex[i * kQ4Rows + p];
        ep.act_out[(size_t)m * ep.ld_act + blk * 64 + n] = __float2bfloat16_rn(silu_f(v[i]) * u);
      }
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(kQ4Threads, 1)
    k_gemm_q4(const __grid_constant__ CUtensorMap tm_x, const uint8_t* __restrict__ wt, int M,
              int BT, int N, int K, int splits, const EpiParams ep, int* err) {
  constexpr int QS = kQ4QStages;
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kQ4OffBar);
  const uint32_t qfull0 = smem_u32(bars);                      // [QS] block landed (tx)
  const uint32_t qempty0 = qfull0 + 8 * QS;                    // [QS] read by its group
  const uint32_t ready0 = qempty0 + 8 * QS;                    // [4] group's block ready
  const uint32_t wfree0 = ready0 + 8 * kQ4Groups;              // [4] group's slots read
  const uint32_t xfull0 = wfree0 + 8 * kQ4Groups;              // [8] token tiles landed (tx)
  const uint32_t xempty0 = xfull0 + 8 * kQ4XMaxStages;         // [8] read by the MMAs
  const uint32_t tfull0 = xempty0 + 8 * kQ4XMaxStages;         // [2 acc x 2 partials]
  const uint32_t tempty0 = tfull0 + 32;                        // [2]
  const uint32_t drain = tempty0 + 16;                         // both MMA threads
  uint32_t* slots = reinterpret_cast<uint32_t*>(bars + kQ4Bars);  // tmem, q / x consumed
  float* ex = reinterpret_cast<float*>(smem + kQ4OffEx);

  const int warp = warp_id(), lane = lane_id();
  const int n_tiles = N / kQ4Rows;
  const int kbt = K / kBK;
  const int kqt = (kbt + 1) / 2;                   // 128-K blocks (the last may be half)
  const int units = n_tiles * splits;
  const uint32_t x_half = static_cast<uint32_t>(BT) * 128;   // one 64-K token tile
  const uint32_t x_bytes = 2 * x_half;
  int XS = static_cast<int>(kQ4XRing / x_bytes);
  if (XS > kQ4XMaxStages) XS = kQ4XMaxStages;
  // MMA issuers (partials): two while two unit buffers of two partials fit the 256
  // accumulator columns (BT <= 64), else one; with two, the token ring's stage count is
  // even so that each stage has one in-order consumer
  const int npart = BT <= 64 ? 2 : 1;
  const uint32_t acc_cols = BT <= 64 ? 64u : 128u;
  if (npart == 2) XS &= ~1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < QS; ++i) {
      mbar_init(qfull0 + 8 * i, 1);
      mbar_init(qempty0 + 8 * i, 4);
    }
    for (int i = 0; i < kQ4Groups; ++i) {
      mbar_init(ready0 + 8 * i, 4);
      mbar_init(wfree0 + 8 * i, 1);
    }
    for (int i = 0; i < kQ4XMaxStages; ++i) {
      mbar_init(xfull0 + 8 * i, 1);
      mbar_init(xempty0 + 8 * i, 1);
    }
    for (int a = 0; a < 4; ++a) mbar_init(tfull0 + 8 * a, 1);
    for (int a = 0; a < 2; ++a) mbar_init(tempty0 + 8 * a, 128);
    mbar_init(drain, 2);
    slots[1] = 0;
    slots[2] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(slots), 512);   // accumulators (2 x 128) + W slots (8 x 32)
    tmem_relinquish();
  }
  if (warp == 2 && lane == 0) tma_prefetch_desc(&tm_x);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = slots[0];
  pdl_wait();

  int issued = 0;
  if (warp == 0) {
    // ------------------------------------------------------------ weight blocks
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit t = decode_unit(u, 1, n_tiles, splits, kqt);
        const uint8_t* src = wt + ((size_t)t.nt * kqt + t.kb0) * kQ4QBytes;
        for (int j = t.kb0; j < t.kb1; ++j, src += kQ4QBytes) {
          if (!(ok = mbar_wait(qempty0 + 8 * stage, phase ^ 1, err))) break;
          const uint32_t fb = qfull0 + 8 * stage;
          mbar_expect_tx(fb, kQ4QBytes);
          bulk_load(sbase + kQ4OffQ + stage * kQ4QBytes, src, kQ4QBytes, fb);
          ++issued;
          if (++stage == QS) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ token tiles
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit t = decode_unit(u, 1, n_tiles, splits, kqt);
        for (int j = t.kb0; j < t.kb1; ++j) {
          const int nkb = (2 * j + 1 < kbt) ? 2 : 1;
          if (!(ok = mbar_wait(xempty0 + 8 * stage, phase ^ 1, err))) break;
          const uint32_t fb = xfull0 + 8 * stage;
          mbar_expect_tx(fb, x_half * nkb);
          for (int h = 0; h < nkb; ++h)
            tma_load_2d(sbase + kQ4OffX + stage * x_bytes + h * x_half, &tm_x, fb,
                        (2 * j + h) * kBK, 0);
          ++issued;
          if (++stage == XS) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA (two issuers)
    // Thread p (warp 1: p = 0, warp 3: p = 1) takes the blocks with seq % 2 == p into its
    // own partial accumulator, so one thread's MMAs run while the other waits. With the
    // token ring's stage count even, each stage (and each group) has one in-order consumer.
    const int p = warp >> 1;
    if (lane == 0 && p < npart) {
      const uint32_t idesc = idesc_bf16(kQ4Rows, static_cast<uint32_t>(BT), 0);
      int xs = p;
      uint32_t xph = 0;
      int iter = 0, consumed = 0, seq = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++iter) {
        const Unit t = decode_unit(u, 1, n_tiles, splits, kqt);
        const int acc = iter & 1;
        if (!(ok = mbar_wait(tempty0 + 8 * acc, ((iter >> 1) & 1) ^ 1, err))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (acc * npart + p) * acc_cols;
        bool first = true;
        for (int j = t.kb0; j < t.kb1 && ok; ++j, ++seq) {
          if (seq % npart != p) continue;
          const int nkb = (2 * j + 1 < kbt) ? 2 : 1;
          const int g = seq % kQ4Groups;
          // the block's token tiles have landed, and the group's W halves are in TMEM
          if (!(ok = mbar_wait(xfull0 + 8 * xs, xph, err))) break;
          ++consumed;
          if (!(ok = mbar_wait(ready0 + 8 * g, (seq / kQ4Groups) & 1, err))) break;
          tc_fence_after();
          for (int h = 0; h < nkb; ++h) {
            const uint32_t a0 = tmem_base + 256 + 32 * (2 * g + h);
            const uint32_t x0 = sbase + kQ4OffX + xs * x_bytes + h * x_half;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              tc_mma_ts(d_tmem, a0 + 8 * k, desc_kmajor_sw128(x0 + 32 * k), idesc,
                        (!first || h > 0 || k > 0) ? 1u : 0u);
          }
          first = false;
          tc_commit(xempty0 + 8 * xs);
          tc_commit(wfree0 + 8 * g);
          xs += npart;                   // this thread's stages: p, p + npart, ...
          if (xs >= XS) {
            xs -= XS;
            xph ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(tfull0 + 8 * (2 * acc + p));
      }
      tc_commit(drain);
      mbar_wait(drain, 0, nullptr);
      atomicAdd(&slots[2], static_cast<uint32_t>(consumed));
    }
    if (lane == 0 && p >= npart) mbar_arrive(drain);   // the idle issuer's share
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int n = quarter * 32 + lane;               // weight row within the unit
    int iter = 0, seq = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++iter) {
      const Unit t = decode_unit(u, 1, n_tiles, splits, kqt);
      const int acc = iter & 1;
      const uint32_t par = (iter >> 1) & 1;
      // partial p holds data when the unit has a block with seq % npart == p
      const int nb = t.kb1 - t.kb0;
      const bool has[2] = {npart == 1 || (seq & 1) == 0 || nb >= 2,
                           npart == 2 && ((seq & 1) == 1 || nb >= 2)};
      seq += nb;
      bool got = mbar_wait(tfull0 + 8 * (2 * acc), par, err);
      if (npart == 2) got = got && mbar_wait(tfull0 + 8 * (2 * acc + 1), par, err);
      if (!epi_all(got)) break;
      tc_fence_after();
      const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
      const uint32_t t0 = tmem_base + lane_off + (acc * npart) * acc_cols;
      const uint32_t t1 = t0 + acc_cols;
      for (int c0 = 0; c0 < M; c0 += kQ4Chunk) {
        float v[kQ4Chunk], w[kQ4Chunk];
        tmem_ld16((has[0] ? t0 : t1) + c0, v);
        if (has[0] && has[1]) {
          tmem_ld16(t1 + c0, w);
#pragma unroll
          for (int i = 0; i < kQ4Chunk; ++i) v[i] += w[i];
        }
        q4_epilogue_chunk<EPI>(v, n, t.nt * kQ4Rows, c0, M, t.kb0, splits, ep, ex);
      }
      tc_fence_before();
      mbar_arrive(tempty0 + 8 * acc);
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dequantisation
    const int grp = (warp - 8) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;             // row of the unit = TMEM lane
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + 256;
    int seq = 0, qconsumed = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const Unit t = decode_unit(u, 1, n_tiles, splits, kqt);
      for (int j = t.kb0; j < t.kb1; ++j, ++seq) {
        if (seq % kQ4Groups != grp) continue;
        const int nkb = (2 * j + 1 < kbt) ? 2 : 1;
        const int qs = seq % QS;
        const uint32_t use = (seq / kQ4Groups) & 1;   // parity of this group's use
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(qfull0 + 8 * qs, (seq / QS) & 1, err))))
          break;
        // chunk-major block: the 16-byte chunk c of row r at (c * 128 + r) * 16
        const uint32_t qst = sbase + kQ4OffQ + qs * kQ4QBytes;
        uint32_t wd[16], sbv[2];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(wd[4 * c]), "=r"(wd[4 * c + 1]), "=r"(wd[4 * c + 2]),
                         "=r"(wd[4 * c + 3])
                       : "r"(qst + (c * kQ4Rows + r) * 16));
#pragma unroll
        for (int h = 0; h < 2; ++h)
          asm volatile("ld.shared.b32 %0, [%1];"
                       : "=r"(sbv[h])
                       : "r"(qst + kQ4QWords + (h * kQ4Rows + r) * 4));
        __syncwarp();
        if (lane == 0) mbar_arrive(qempty0 + 8 * qs);
        ++qconsumed;
        // the MMAs of this group's previous block have read its TMEM slots
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(wfree0 + 8 * grp, use ^ 1, err)))) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h >= nkb) break;
          const uint32_t s2 = __byte_perm(sbv[h], 0, 0x1010);   // (scale, scale)
          const uint32_t b2 = __byte_perm(sbv[h], 0, 0x3232);   // (bias, bias)
          uint32_t o[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) dequant_word(wd[8 * h + c], s2, b2, o + 4 * c);
          tmem_st32u(t_lane + 32 * (2 * grp + h), o);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ready0 + 8 * grp);
      }
    }
    if (lane == 0 && quarter == 0) atomicAdd(&slots[1], static_cast<uint32_t>(qconsumed));
  }
  __syncthreads();
  if (warp == 0 && lane == 0) {
    // a failed launch may leave loads in flight: wait (bounded) until they have landed
    for (int i = static_cast<int>(slots[1]); i < issued; ++i)
      mbar_wait(qfull0 + 8 * (i % QS), (i / QS) & 1, nullptr);
  }
  if (warp == 2 && lane == 0) {
    for (int i = static_cast<int>(slots[2]); i < issued; ++i)
      mbar_wait(xfull0 + 8 * (i % XS), (i / XS) & 1, nullptr);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int EPI>
cc_status launch_q4_t(const CUtensorMap& tx, const uint8_t* wt, int M, int BT, int N, int K,
                      int splits, const EpiParams& ep, int* err, cudaStream_t s) {
  static std::atomic<bool> smem_set{false};
  auto kern = k_gemm_q4<EPI>;
  CC_CHECK_CUDA(allow_dynamic_smem(kern, kQ4Smem, smem_set));
  const int units = (N / kQ4Rows) * splits;
  const int grid = units < num_sms() ? units : num_sms();
  CC_CHECK_CUDA(launch_pdl(kern, dim3(grid), dim3(kQ4Threads), kQ4Smem, s, tx, wt, M, BT, N, K,
                          splits, ep, err));
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

// The fused residual + LayerNorm epilogue replaces the plain residual one wherever that one
// would run unsplit (several row tiles); a single row tile keeps its K splits (decode).
bool gemm_resid_ln_ok(int M, int N, int K) {
  int bn, splits;
  gemm_choose(M, N, K, EPI_RESID, &bn, &splits);
  return M > 0 && splits == 1 && N % bn == 0 && N / bn <= num_sms();
}

static std::atomic<int> g_test_stall_next{0};

void test_stall_next_gemm() { g_test_stall_next.store(1); }

cc_status launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K, int bn,
                      int splits, int epi, const EpiParams& ep_in, int* err, cudaStream_t s,
                      const CUtensorMap* tb_half) {
  if (M <= 0) return CC_OK;
  if (K % kBK != 0 || N % bn != 0 || splits < 1 || splits > K / kBK)
    return CC_ERR_INVALID_ARG;
  EpiParams ep = ep_in;
  if (g_test_stall_next.load(std::memory_order_relaxed) && g_test_stall_next.exchange(0))
    ep.test_stall = 1;
  if (bn == 256) {
    switch (epi) {
      case EPI_F32:
        return launch_t<256, EPI_F32>(ta, tb, tb_half, M, N, K, splits, ep, err, s);
      case EPI_RESID:
        return launch_t<256, EPI_RESID>(ta, tb, tb_half, M, N, K, splits, ep, err, s);
      case EPI_QKV_MLP:
        return launch_t<256, EPI_QKV_MLP>(ta, tb, tb_half, M, N, K, 1, ep, err, s);
      case EPI_RESID_LN:
        return launch_t<256, EPI_RESID_LN>(ta, tb, tb_half, M, N, K, splits, ep, err, s);
    }
  } else if (bn == 128) {
    switch (epi) {
      case EPI_F32:
        return launch_t<128, EPI_F32>(ta, tb, tb_half, M, N, K, splits, ep, err, s);
      case EPI_RESID:
        return launch_t<128, EPI_RESID>(ta, tb, tb_half, M, N, K, splits, ep, err, s);
      case EPI_QKV_MLP:
        return launch_t<128, EPI_QKV_MLP>(ta, tb, tb_half, M, N, K, 1, ep, err, s);
      case EPI_RESID_LN:
        return launch_t<128, EPI_RESID_LN>(ta, tb, tb_half, M, N, K, splits, ep, err, s);
    }
  }
  return CC_ERR_INVALID_ARG;
}

int gemm_q4_token_tile(int M) { return M <= 16 ? 16 : (M + 15) / 16 * 16; }

cc_status launch_gemm_q4(const CUtensorMap& tx, const void* w_tiled, int M, int N, int K,
                         int epi, const EpiParams& ep, int* err, cudaStream_t s) {
  if (M <= 0) return CC_OK;
  if (M > 128 || N % kQ4Rows != 0 || K % kBK != 0 || !w_tiled ||
      (reinterpret_cast<uintptr_t>(w_tiled) & 15) != 0)
    return CC_ERR_INVALID_ARG;
  const uint8_t* wt = static_cast<const uint8_t*>(w_tiled);
  const int BT = gemm_q4_token_tile(M);
  // K splits only for additive epilogues (the f32 one when it accumulates into C), up to one
  // unit per SM
  int sp = 1;
  const int kqt = (K / kBK + 1) / 2;   // 128-K blocks
  if (epi == EPI_RESID || (epi == EPI_F32 && ep.accumulate)) {
    const int tiles = N / kQ4Rows;
    while (tiles * (sp + 1) <= num_sms() && kqt / (sp + 1) >= 2) ++sp;
  }
  switch (epi) {
    case EPI_F32: return launch_q4_t<EPI_F32>(tx, wt, M, BT, N, K, sp, ep, err, s);
    case EPI_RESID: return launch_q4_t<EPI_RESID>(tx, wt, M, BT, N, K, sp, ep, err, s);
    case EPI_QKV_MLP: return launch_q4_t<EPI_QKV_MLP>(tx, wt, M, BT, N, K, 1, ep, err, s);
  }
  return CC_ERR_INVALID_ARG;
}

}  // namespace cc
