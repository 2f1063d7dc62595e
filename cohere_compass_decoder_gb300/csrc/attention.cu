// Prefill attention on the tcgen05 tensor cores: causal or sliding-window, grouped-query,
// over packed sequences (cu_seqlens), head_dim 128.
//
// Definition (mlxcel issue "Cohere Compass / North-Micro-Vision", section "Text decoder
// forward", attention of layer i): O_i = sum_j softmax_j(q_i . k_j * d^-0.5) v_j over the
// keys j of the same sequence with j <= i (full layers) and additionally i - j < window
// (sliding layers: "causal restricted to the last 4096 keys"). Query head h reads KV head
// h / (n_q / n_kv).
//
// One CTA per (128-query tile, query head). Warps:
//   warp 0      TMA: the Q tile once, then K and V tiles (128 keys x 128 dims, two
//               64-column boxes each, 128-byte swizzle) into 2-stage rings
//   warp 1      MMA: S = Q K^T into one of two TMEM score buffers (M=128, N=128), then
//               O += P V into the TMEM output accumulator (V read MN-major)
//   warps 2..5  softmax, one query row per thread: masked scores from TMEM, online
//               max/sum in the log2 domain, P (bf16) into a swizzled shared buffer, and
//               the final O / l.
// The running max is only moved (and O rescaled in TMEM) when it grows by more than
// 2^8; otherwise the stale max is kept. Both numerator and denominator use the same max,
// so the result is unchanged; only the range of P (< 2^8) is affected.
// Key tiles wholly outside the causal/window band are never loaded.
#include "kernels.h"
#include "ptx.cuh"

namespace cc {

namespace {

constexpr int kThreads = 192;
constexpr uint32_t kTile = 128 * 128 * 2;  // one 128 x 128 bf16 tile = two 16 KB boxes
constexpr uint32_t kHalf = 128 * 64 * 2;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTile;          // 2 stages
constexpr uint32_t kOffV = kOffK + 2 * kTile;      // 2 stages
constexpr uint32_t kOffP = kOffV + 2 * kTile;      // 2 buffers
constexpr uint32_t kOffBar = kOffP + 2 * kTile;
constexpr size_t kSmem = 1024 + kOffBar + 256;
constexpr uint32_t kTmemCols = 512;                // S0 | S1 | O (| unused)
constexpr uint32_t kIdescS = idesc_bf16(128, 128, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, 1);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;          // log2 units

enum {
  B_Q = 0, B_KFULL = 1, B_KEMPTY = 3, B_VFULL = 5, B_VEMPTY = 7, B_SFULL = 9, B_PFULL = 11,
  B_ODONE = 13, B_DRAIN = 15, B_COUNT = 16
};

__global__ void __launch_bounds__(kThreads, 1)
    k_attn_prefill(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out,
                   int ld_out, const AttnTile* __restrict__ tiles, const int32_t* n_tiles_p,
                   int n_q, int n_kv, int window, float scale_log2, int* err) {
  if (static_cast<int>(blockIdx.x) >= *n_tiles_p) return;
  const AttnTile tile = tiles[blockIdx.x];
  const int head = blockIdx.y;
  const int kvh = head / (n_q / n_kv);
  const int q0 = tile.q0;
  const int q_last = min(q0 + 127, tile.seq_len - 1);
  const int kt_hi = q_last >> 7;
  const int kt_lo = window > 0 ? max(0, q0 - window + 1) >> 7 : 0;
  const int n = kt_hi - kt_lo + 1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT);

  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_KFULL + i), 1);
      mbar_init(bar(B_KEMPTY + i), 1);
      mbar_init(bar(B_VFULL + i), 1);
      mbar_init(bar(B_VEMPTY + i), 1);
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_PFULL + i), 128);
      mbar_init(bar(B_ODONE + i), 1);
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
  const uint32_t tmem_o = tmem + 256;

  int issued_k = 0, issued_v = 0;
  if (warp == 0) {
    if (lane == 0) {
      const int qx = head * 128, kx = kvh * 128;
      mbar_expect_tx(bar(B_Q), kTile);
      tma_load_2d(sbase + kOffQ, &tm_q, bar(B_Q), qx, tile.seq_start + q0);
      tma_load_2d(sbase + kOffQ + kHalf, &tm_q, bar(B_Q), qx + 64, tile.seq_start + q0);
      for (int t = 0; t < n; ++t) {
        const int st = t & 1;
        const uint32_t ph = ((t >> 1) & 1) ^ 1;
        const int y = tile.seq_start + (kt_lo + t) * 128;
        if (!mbar_wait(bar(B_KEMPTY + st), ph, err)) break;
        mbar_expect_tx(bar(B_KFULL + st), kTile);
        tma_load_2d(sbase + kOffK + st * kTile, &tm_k, bar(B_KFULL + st), kx, y);
        tma_load_2d(sbase + kOffK + st * kTile + kHalf, &tm_k, bar(B_KFULL + st), kx + 64, y);
        ++issued_k;
        if (!mbar_wait(bar(B_VEMPTY + st), ph, err)) break;
        mbar_expect_tx(bar(B_VFULL + st), kTile);
        tma_load_2d(sbase + kOffV + st * kTile, &tm_v, bar(B_VFULL + st), kx, y);
        tma_load_2d(sbase + kOffV + st * kTile + kHalf, &tm_v, bar(B_VFULL + st), kx + 64, y);
        ++issued_v;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = mbar_wait(bar(B_Q), 0, err);
      auto issue_s = [&](int t) -> bool {
        const int st = t & 1;
        if (!mbar_wait(bar(B_KFULL + st), (t >> 1) & 1, err)) return false;
        tc_fence_after();
        const uint32_t d = tmem + 128 * (t & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc_mma(d, desc_kmajor_sw128(sbase + kOffQ + off),
                 desc_kmajor_sw128(sbase + kOffK + st * kTile + off), kIdescS, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(B_KEMPTY + st));
        tc_commit(bar(B_SFULL + (t & 1)));
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && n > 1) ok = issue_s(1);
      for (int t = 0; t < n && ok; ++t) {
        const int b = t & 1;
        if (!mbar_wait(bar(B_PFULL + b), (t >> 1) & 1, err)) break;
        if (!mbar_wait(bar(B_VFULL + b), (t >> 1) & 1, err)) break;
        tc_fence_after();
        const uint32_t pbase = sbase + kOffP + b * kTile;
        const uint32_t vbase = sbase + kOffV + b * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t da = desc_kmajor_sw128(pbase + (kk >> 2) * kHalf + (kk & 3) * 32);
          const uint64_t db = desc_mnmajor_sw128(vbase + kk * 2048, kHalf);
          tc_mma(tmem_o, da, db, kIdescPV, (t > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(B_VEMPTY + b));
        tc_commit(bar(B_ODONE + b));
        if (t + 2 < n) ok = issue_s(t + 2);
      }
      tc_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row in the tile
    const int qi = q0 + r;              // query index in its sequence
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      const int b = t & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_SFULL + b), (t >> 1) & 1, err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + 128 * b + lane_off + 32 * c, s + 32 * c);
      const int kbase = (kt_lo + t) * 128;
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        const int kj = kbase + c;
        const bool vis = (kj <= qi) && (window <= 0 || qi - kj < window);
        s[c] = vis ? s[c] * scale_log2 : -INFINITY;
        mt = fmaxf(mt, s[c]);
      }
      const bool need = mt > m + kRescaleThreshold;  // also true when m == -inf < mt
      const bool need_o = need && (m != -INFINITY);
      if (__any_sync(0xffffffffu, need_o)) {
        // O holds P V of tiles < t: wait for the last of them, then rescale in TMEM
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bar(B_ODONE + ((t - 1) & 1)), ((t - 1) >> 1) & 1, err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float f = need_o ? exp2f(m - mt) : 1.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(tmem_o + lane_off + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          tmem_st32(tmem_o + lane_off + 32 * c, o);
        }
        tmem_st_wait();
        if (need_o) l *= f;
      }
      if (need) m = mt;
      const float mu = (m == -INFINITY) ? 0.f : m;
      float rs = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        const float p0 = exp2f(s[c] - mu), p1 = exp2f(s[c + 1] - mu);
        rs += p0 + p1;
        pk[c >> 1] = pack_bf16x2(p0, p1);
      }
      l += rs;
      if (t >= 2) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_ODONE + b), ((t - 2) >> 1) & 1, err))) {
          ok = false;
          break;
        }
      }
      // row r of P: keys 0..63 in box 0, 64..127 in box 1; 16-byte chunk c of a
      // 128-byte row sits at chunk position c ^ (r & 7) (128-byte swizzle)
      const uint32_t prow = sbase + kOffP + b * kTile + r * 128;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint32_t box = c >> 3, ch = (c & 7) ^ (r & 7);
        st_shared_v4(prow + box * kHalf + ch * 16, pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                     pk[4 * c + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + b));
    }
    if (ok) ok = __all_sync(0xffffffffu,
                            mbar_wait(bar(B_ODONE + ((n - 1) & 1)), ((n - 1) >> 1) & 1, err));
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool row_ok = qi < tile.seq_len;
      __nv_bfloat16* dst = out + (size_t)(tile.seq_start + qi) * ld_out + head * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld32(tmem_o + lane_off + 32 * c, o);
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
    // after a failed launch, let issued loads land before the CTA exits (bounded)
    // (only the last load of each stage can still be pending)
    for (int st = 0; st < 2; ++st) {
      if (issued_k > st) {
        const int t = issued_k - 1 - ((issued_k - 1 - st) & 1);
        mbar_wait(bar(B_KFULL + st), (t >> 1) & 1, nullptr);
      }
      if (issued_v > st) {
        const int t = issued_v - 1 - ((issued_v - 1 - st) & 1);
        mbar_wait(bar(B_VFULL + st), (t >> 1) & 1, nullptr);
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One thread: lists the 128-query tiles of every sequence, ordered by the number of key
// tiles they visit (largest first) so that the longest CTAs start first.
__global__ void k_attn_tiles(const int32_t* cu, int n_seqs, int window, AttnTile* tiles,
                             int32_t* n_tiles) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int total = 0, max_w = 0;
  for (int s = 0; s < n_seqs; ++s) {
    const int L = cu[s + 1] - cu[s];
    for (int q0 = 0; q0 < L; q0 += 128) {
      const int hi = min(q0 + 127, L - 1) >> 7;
      const int lo = window > 0 ? max(0, q0 - window + 1) >> 7 : 0;
      max_w = max(max_w, hi - lo + 1);
      ++total;
    }
  }
  int k = 0;
  for (int w = max_w; w >= 1; --w) {
    for (int s = 0; s < n_seqs; ++s) {
      const int L = cu[s + 1] - cu[s];
      for (int q0 = 0; q0 < L; q0 += 128) {
        const int hi = min(q0 + 127, L - 1) >> 7;
        const int lo = window > 0 ? max(0, q0 - window + 1) >> 7 : 0;
        if (hi - lo + 1 == w) tiles[k++] = AttnTile{cu[s], L, q0, 0};
      }
    }
  }
  *n_tiles = total;
}

}  // namespace

int attn_max_tiles(int tokens, int n_seqs) { return (tokens + 127) / 128 + n_seqs; }

cc_status launch_attn_tiles(const int32_t* cu_seqlens, int n_seqs, int window, AttnTile* tiles,
                            int32_t* n_tiles, cudaStream_t s) {
  k_attn_tiles<<<1, 32, 0, s>>>(cu_seqlens, n_seqs, window, tiles, n_tiles);
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
  const float scale_log2 = (1.0f / sqrtf(128.0f)) * kLog2e;
  dim3 grid(max_tiles, n_q);
  k_attn_prefill<<<grid, kThreads, kSmem, s>>>(tq, tk, tv, out, ld_out, tiles, n_tiles, n_q, n_kv,
                                               window, scale_log2, err);
  CC_CHECK_CUDA(cudaGetLastError());
  return CC_OK;
}

}  // namespace cc
