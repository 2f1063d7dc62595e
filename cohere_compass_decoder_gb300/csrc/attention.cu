// Prefill attention on the tcgen05 tensor cores: causal or sliding-window, grouped-query,
// over packed sequences (cu_seqlens), head_dim 128.
//
// Definition (mlxcel issue "Cohere Compass / North-Micro-Vision", section "Text decoder
// forward", attention of layer i): O_i = sum_j softmax_j(q_i . k_j * d^-0.5) v_j over the
// keys j of the same sequence with j <= i (full layers) and additionally i - j < window
// (sliding layers: "causal restricted to the last 4096 keys"). Query head h reads KV head
// h / (n_q / n_kv).
//
// One CTA per (128-query tile, pair of query heads that read the same KV head; one head
// when n_q / n_kv is odd), 10 warps:
//   warp 0      TMA: the Q tiles once, then K and V tiles of 128 keys x 128 dims (two
//               64-column boxes, 128-byte swizzle) into 3-stage (K) and 2-stage (V) rings;
//               each K/V tile feeds both heads
//   warp 1      MMA: S_h = Q_h K^T (M=128, N=128) into the head's TMEM score region, and
//               O_h += P_h V with P_h read from tensor memory (M=128, N=128, V MN-major)
//   warps 2..5  softmax of head 0, warps 6..9 softmax of head 1: one query row per thread,
//               log2 domain; P is written as bf16 over the consumed scores (tcgen05.st), so
//               neither P nor a proxy fence touches shared memory, and the only shared-
//               memory operands of the MMAs are Q, K and V.
// Per tile the tensor cores run P V and the next scores of one head while the other head's
// softmax works. A group moves its running max (and rescales its O in TMEM) only when the
// max grows by more than 2^8; the stale max is used consistently for numerator and
// denominator, so the result is unchanged. The exponentials run two per MUFU operation
// (ex2.approx on packed bf16 pairs): the argument s * d^-0.5 * log2(e) - m is rounded to
// bf16 first and the result is the bf16 P the P V MMA consumes anyway; the row sums add
// exactly those bf16 values. Key tiles wholly outside the causal/window band are never
// loaded.
#include "kernels.h"
#include "ptx.cuh"

namespace cc {

namespace {

constexpr int kThreads = 320;
constexpr int kKeys = 128;                             // keys per tile
constexpr int kKStages = 3, kVStages = 2;
constexpr uint32_t kTile = 128 * 128 * 2;              // 32 KB: 128 rows x 128 dims
constexpr uint32_t kHalf = 128 * 64 * 2;               // one 64-dim box column: 16 KB
constexpr uint32_t kOffQ = 0;                          // 2 heads
constexpr uint32_t kOffK = kOffQ + 2 * kTile;
constexpr uint32_t kOffV = kOffK + kKStages * kTile;
constexpr uint32_t kOffBar = kOffV + kVStages * kTile;
constexpr size_t kSmem = 1024 + kOffBar + 256;
constexpr uint32_t kTmemCols = 512;  // head h: scores / P at 256 h, output at 256 h + 128
constexpr uint32_t kIdescS = idesc_bf16(128, kKeys, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, 1);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;          // log2 units

enum {
  B_Q = 0,
  B_KFULL = 1, B_KEMPTY = B_KFULL + kKStages, B_VFULL = B_KEMPTY + kKStages,
  B_VEMPTY = B_VFULL + kVStages,
  B_SFULL = B_VEMPTY + kVStages,  // [head]: scores of the head's current tile ready
  B_PFULL = B_SFULL + 2,          // [head], 128 arrivals: P of the head's current tile in TMEM
  B_ODONE = B_PFULL + 2,          // [head]: P V of the head's tiles
  B_DRAIN = B_ODONE + 2,
  B_COUNT = B_DRAIN + 1
};

__device__ __forceinline__ float ex2_mufu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


// 2^x of two bf16 values packed in one register (low half first), bf16 results.
__device__ __forceinline__ uint32_t ex2_bf16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_attn_prefill(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out,
                   int ld_out, const AttnTile* __restrict__ tiles, const int32_t* n_tiles_p,
                   int n_q, int n_kv, int window, float scale_log2, int* err) {
  if (static_cast<int>(blockIdx.x) >= *n_tiles_p) return;
  const AttnTile tile = tiles[blockIdx.x];
  const int G = n_q / n_kv;
  const bool paired = (G & 1) == 0;                    // two heads share this KV head
  const int nh = paired ? 2 : 1;
  const int head0 = paired ? 2 * blockIdx.y : blockIdx.y;
  const int kvh = head0 / G;
  const int q0 = tile.q0;
  const int q_last = min(q0 + 127, tile.seq_len - 1);
  const int kt_hi = q_last / kKeys;
  const int kt_lo = window > 0 ? max(0, q0 - window + 1) / kKeys : 0;
  const int n = kt_hi - kt_lo + 1;                     // key tiles

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT);

  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q), 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(B_SFULL + h), 1);
      mbar_init(bar(B_PFULL + h), 128);
      mbar_init(bar(B_ODONE + h), 1);
    }
    mbar_init(bar(B_DRAIN), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int issued_k = 0, issued_v = 0;
  if (warp == 0) {
    if (lane == 0) {
      const int kx = kvh * 128;
      mbar_expect_tx(bar(B_Q), nh * kTile);
      for (int h = 0; h < nh; ++h) {
        const int qx = (head0 + h) * 128;
        tma_load_2d(sbase + kOffQ + h * kTile, &tm_q, bar(B_Q), qx, tile.seq_start + q0);
        tma_load_2d(sbase + kOffQ + h * kTile + kHalf, &tm_q, bar(B_Q), qx + 64,
                    tile.seq_start + q0);
      }
      // K runs up to three tiles ahead, V up to two
      int tk = 0, tv = 0;
      while ((tk < n || tv < n)) {
        if (tk < n && tk <= tv + 1) {
          const int st = tk % kKStages;
          if (!mbar_wait(bar(B_KEMPTY + st), ((tk / kKStages) & 1) ^ 1, err)) break;
          const int y = tile.seq_start + (kt_lo + tk) * kKeys;
          mbar_expect_tx(bar(B_KFULL + st), kTile);
          tma_load_2d(sbase + kOffK + st * kTile, &tm_k, bar(B_KFULL + st), kx, y);
          tma_load_2d(sbase + kOffK + st * kTile + kHalf, &tm_k, bar(B_KFULL + st), kx + 64, y);
          ++tk;
          ++issued_k;
        } else {
          const int st = tv % kVStages;
          if (!mbar_wait(bar(B_VEMPTY + st), ((tv / kVStages) & 1) ^ 1, err)) break;
          const int y = tile.seq_start + (kt_lo + tv) * kKeys;
          mbar_expect_tx(bar(B_VFULL + st), kTile);
          tma_load_2d(sbase + kOffV + st * kTile, &tm_v, bar(B_VFULL + st), kx, y);
          tma_load_2d(sbase + kOffV + st * kTile + kHalf, &tm_v, bar(B_VFULL + st), kx + 64, y);
          ++tv;
          ++issued_v;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = mbar_wait(bar(B_Q), 0, err);
      auto issue_s = [&](int h, int t) {
        const uint32_t kb = sbase + kOffK + (t % kKStages) * kTile;
        const uint32_t qb = sbase + kOffQ + h * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc_mma(tmem + 256 * h, desc_kmajor_sw128(qb + off), desc_kmajor_sw128(kb + off),
                 kIdescS, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(B_SFULL + h));
      };
      if (ok) ok = mbar_wait(bar(B_KFULL + 0), 0, err);
      if (ok) {
        tc_fence_after();
        for (int h = 0; h < nh; ++h) issue_s(h, 0);
        tc_commit(bar(B_KEMPTY + 0));
      }
      for (int t = 0; t < n && ok; ++t) {
        const bool next = t + 1 < n;
        for (int h = 0; h < nh && ok; ++h) {
          // P_h(t) is in TMEM: O_h += P_h V(t), then the head's next scores (same columns)
          if (!(ok = mbar_wait(bar(B_PFULL + h), t & 1, err))) break;
          if (h == 0 && !(ok = mbar_wait(bar(B_VFULL + t % kVStages), (t / kVStages) & 1, err)))
            break;
          if (h == 0 && next &&
              !(ok = mbar_wait(bar(B_KFULL + (t + 1) % kKStages), ((t + 1) / kKStages) & 1, err)))
            break;
          tc_fence_after();
          const uint32_t vb = sbase + kOffV + (t % kVStages) * kTile;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {   // 16 keys per MMA: 8 packed P columns
            tc_mma_ts(tmem + 256 * h + 128, tmem + 256 * h + 8 * kk,
                      desc_mnmajor_sw128(vb + kk * 2048, kHalf), kIdescPV,
                      (t > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar(B_ODONE + h));
          if (next) issue_s(h, t + 1);
        }
        if (!ok) break;
        tc_commit(bar(B_VEMPTY + t % kVStages));
        if (next) tc_commit(bar(B_KEMPTY + (t + 1) % kKStages));
      }
      tc_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- softmax groups
    const int grp = (warp - 2) >> 2;                 // head slot of this group
    const int quarter = warp & 3;                    // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;               // query row in the tile
    const int qi = q0 + r;                           // query index in its sequence
    // this warp's rows that lie inside the sequence (rows past its end are never stored)
    const int qw_lo = q0 + quarter * 32, qw_hi = min(qw_lo + 31, tile.seq_len - 1);
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + 256 * grp + lane_off;
    const uint32_t o_tmem = s_tmem + 128;
    float m = -INFINITY, l = 0.f;
    bool ok = grp < nh;
    for (int t = 0; t < n && ok; ++t) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_SFULL + grp), t & 1, err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int kbase = (kt_lo + t) * kKeys;
      // warp-uniform: every key of the tile visible to every row of this warp
      const bool full = (kbase + kKeys - 1 <= qw_lo) && (window <= 0 || qw_hi - kbase < window);
      float s[kKeys];
      tmem_ld128(s_tmem, s);
      if (!full) {
        const int hi_c = qi - kbase;                             // causal: c <= hi_c
        const int lo_c = window > 0 ? qi - window + 1 - kbase : -1;
#pragma unroll
        for (int c = 0; c < kKeys; ++c) s[c] = (c <= hi_c && c >= lo_c) ? s[c] : -INFINITY;
      }
      float a0 = max3(s[0], s[1], s[2]), a1 = max3(s[3], s[4], s[5]);
      float a2 = max3(s[6], s[7], s[8]), a3 = max3(s[9], s[10], s[11]);
#pragma unroll
      for (int c = 12; c < 124; c += 8) {
        a0 = max3(a0, s[c], s[c + 1]);
        a1 = max3(a1, s[c + 2], s[c + 3]);
        a2 = max3(a2, s[c + 4], s[c + 5]);
        a3 = max3(a3, s[c + 6], s[c + 7]);
      }
      a0 = max3(a0, s[124], s[125]);
      a1 = max3(a1, s[126], s[127]);
      const float mt = fmaxf(max3(a0, a1, a2), a3) * scale_log2;
      const bool need = mt > m + kRescaleThreshold;  // also true when m == -inf < mt
      const bool need_o = need && (m != -INFINITY);
      if (__any_sync(0xffffffffu, need_o)) {
        // O holds P V of tiles < t, all complete: the scores of tile t were issued after them
        const float f = need_o ? ex2_mufu(m - mt) : 1.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(o_tmem + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          tmem_st32(o_tmem + 32 * c, o);
        }
        if (need_o) l *= f;
      }
      if (need) m = mt;
      const float mu = (m == -INFINITY) ? 0.f : m;
      // P = 2^(s * scale_log2 - m) (masked scores are -inf and give 0), its row sum, bf16 P
      // packed two keys per column over the first 64 score columns
      const float2 sc2 = make_float2(scale_log2, scale_log2);
      const float2 nm2 = make_float2(-mu, -mu);
      float2 sum[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                       make_float2(0.f, 0.f)};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int c = 64 * half + 2 * j;
          const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), sc2, nm2);
          // two probabilities per MUFU operation, already the bf16 P the P V MMA reads
          const uint32_t p2 = ex2_bf16x2(pack_bf16x2(x.x, x.y));
          pk[j] = p2;
          sum[j & 3] = __fadd2_rn(sum[j & 3], make_float2(__uint_as_float(p2 << 16),
                                                          __uint_as_float(p2 & 0xFFFF0000u)));
        }
        tmem_st32u(s_tmem + 32 * half, pk);
      }
      l += ((sum[0].x + sum[0].y) + (sum[1].x + sum[1].y)) +
           ((sum[2].x + sum[2].y) + (sum[3].x + sum[3].y));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + grp));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(B_ODONE + grp), (n - 1) & 1, err));
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool row_ok = qi < tile.seq_len;
      __nv_bfloat16* dst = out + (size_t)(tile.seq_start + qi) * ld_out + (head0 + grp) * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld32(o_tmem + 32 * c, o);
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            st_global_v4(dst + 32 * c + i, pack_bf16x2(o[i] * inv, o[i + 1] * inv),
                         pack_bf16x2(o[i + 2] * inv, o[i + 3] * inv),
                         pack_bf16x2(o[i + 4] * inv, o[i + 5] * inv),
                         pack_bf16x2(o[i + 6] * inv, o[i + 7] * inv));
          }
        }
      }
    }
  }
  __syncthreads();
  if (warp == 0 && lane == 0) {
    // after a failed launch, let issued loads land before the CTA exits (bounded); only the
    // last loads of each ring can still be pending
    for (int t = max(0, issued_k - kKStages); t < issued_k; ++t)
      mbar_wait(bar(B_KFULL + t % kKStages), (t / kKStages) & 1, nullptr);
    for (int t = max(0, issued_v - kVStages); t < issued_v; ++t)
      mbar_wait(bar(B_VFULL + t % kVStages), (t / kVStages) & 1, nullptr);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One block lists the 128-query tiles of every sequence, ordered by the number of key
// tiles they visit (largest first, a counting sort) so that the longest CTAs start first.
// Dynamic shared memory: tile offsets of the sequences [n_seqs + 1], then the histogram.
__device__ __forceinline__ int tile_work(int q0, int L, int window) {
  const int hi = min(q0 + 127, L - 1) >> 7;
  const int lo = window > 0 ? max(0, q0 - window + 1) >> 7 : 0;
  return hi - lo + 1;
}

__global__ void __launch_bounds__(1024)
    k_attn_tiles(const int32_t* __restrict__ cu, int n_seqs, int window, int max_work,
                 AttnTile* __restrict__ tiles, int32_t* n_tiles) {
  extern __shared__ int sh[];
  int* toff = sh;                   // [n_seqs + 1]
  int* hist = sh + n_seqs + 1;      // [max_work + 1]
  for (int i = threadIdx.x; i <= max_work; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int s = 0; s < n_seqs; ++s) {
      toff[s] = acc;
      acc += max(0, cu[s + 1] - cu[s] + 127) >> 7;
    }
    toff[n_seqs] = acc;
  }
  __syncthreads();
  const int total = toff[n_seqs];
  auto locate = [&](int g, int* s_out, int* q0_out) {
    int lo = 0, hi = n_seqs;  // toff[lo] <= g < toff[lo + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (toff[mid] <= g) lo = mid; else hi = mid;
    }
    *s_out = lo;
    *q0_out = (g - toff[lo]) * 128;
  };
  for (int g = threadIdx.x; g < total; g += blockDim.x) {
    int s, q0;
    locate(g, &s, &q0);
    atomicAdd(&hist[min(tile_work(q0, cu[s + 1] - cu[s], window), max_work)], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // start slot of every work value, largest work first
    int acc = 0;
    for (int w = max_work; w >= 0; --w) {
      const int c = hist[w];
      hist[w] = acc;
      acc += c;
    }
    *n_tiles = total;
  }
  __syncthreads();
  for (int g = threadIdx.x; g < total; g += blockDim.x) {
    int s, q0;
    locate(g, &s, &q0);
    const int L = cu[s + 1] - cu[s];
    const int slot = atomicAdd(&hist[min(tile_work(q0, L, window), max_work)], 1);
    tiles[slot] = AttnTile{cu[s], L, q0, 0};
  }
}

}  // namespace

int attn_max_tiles(int tokens, int n_seqs) { return (tokens + 127) / 128 + n_seqs; }

cc_status launch_attn_tiles(const int32_t* cu_seqlens, int n_seqs, int tokens, int window,
                            AttnTile* tiles, int32_t* n_tiles, cudaStream_t s) {
  const int max_work = (tokens + 127) / 128 + 1;
  const size_t smem = (size_t)(n_seqs + 1 + max_work + 1) * sizeof(int);
  if (smem > 200 * 1024) return CC_ERR_UNSUPPORTED;
  if (smem > 48 * 1024)
    CC_CHECK_CUDA(cudaFuncSetAttribute(k_attn_tiles, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem)));
  k_attn_tiles<<<1, 1024, smem, s>>>(cu_seqlens, n_seqs, window, max_work, tiles, n_tiles);
  CC_CHECK_CUDA(cudaGetLastError());
  return CC_OK;
}

cc_status launch_attn_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              __nv_bfloat16* out, int ld_out, const AttnTile* tiles,
                              const int32_t* n_tiles, int max_tiles, int n_q, int n_kv,
                              int window, int* err, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    CC_CHECK_CUDA(cudaFuncSetAttribute(k_attn_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmem)));
    attr_set = true;
  }
  if (max_tiles <= 0) return CC_OK;
  if (n_kv <= 0 || n_q % n_kv != 0) return CC_ERR_INVALID_ARG;
  const float scale_log2 = (1.0f / sqrtf(128.0f)) * kLog2e;
  const bool paired = ((n_q / n_kv) & 1) == 0;
  dim3 grid(max_tiles, paired ? n_q / 2 : n_q);
  k_attn_prefill<<<grid, kThreads, kSmem, s>>>(tq, tk, tv, out, ld_out, tiles, n_tiles, n_q, n_kv,
                                               window, scale_log2, err);
  CC_CHECK_CUDA(cudaGetLastError());
  return CC_OK;
}

int attn_kv_box_rows() { return kKeys; }

}  // namespace cc
