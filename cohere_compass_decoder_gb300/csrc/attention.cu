// Prefill attention on the tcgen05 tensor cores: causal or sliding-window, grouped-query,
// over packed sequences (cu_seqlens), head_dim 128.
//
// Definition (mlxcel issue "Cohere Compass / North-Micro-Vision", section "Text decoder
// forward", attention of layer i): O_i = sum_j softmax_j(q_i . k_j * d^-0.5) v_j over the
// keys j of the same sequence with j <= i (full layers) and additionally i - j < window
// (sliding layers: "causal restricted to the last 4096 keys"). Query head h reads KV head
// h / (n_q / n_kv).
//
// Work items: (128-query tile or a chunk of its key tiles, head group), where a head group is
// the pair of query heads that read the same KV head (a single head when n_q / n_kv is odd).
// A tile builder lists them heaviest first and cuts a query tile whose key range is long
// next to the launch's average work per SM into chunks, so that the longest item of a short
// causal sequence no longer sets the kernel's duration. One persistent CTA per SM takes
// items in that order from a global counter; 10 warps:
//   warp 0      scheduler and TMA: takes the next item, hands it to the other warps through
//               a 2-entry shared-memory queue, loads its Q tiles, then its K and V tiles of
//               128 keys x 128 dims (two 64-column boxes, 128-byte swizzle) into 3-stage (K)
//               and 2-stage (V) rings; each K/V tile feeds both heads
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
// A chunk of a split tile stores (max, sum, O) of each of its rows in fp32 and counts itself
// in the tile's arrival counter; the chunk that arrives last merges all partials in chunk
// order (the same arithmetic whichever chunk is last) and writes the bf16 rows.
#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"

namespace cc {

namespace {

constexpr int kThreads = 320;
constexpr int kKeys = 128;                             // keys per tile
constexpr int kKStages = 3, kVStages = 2;
constexpr int kMinChunk = 6;                           // key tiles: never split below this
constexpr int kMergeTiles = 6;                         // a merge costs about this many tiles
constexpr int kMaxChunks = 8;                          // chunks of one split query tile
constexpr int kCounterInts = 1 + kMaxChunks;           // arrival count, ready flags
constexpr uint32_t kTile = 128 * 128 * 2;              // 32 KB: 128 rows x 128 dims
constexpr uint32_t kHalf = 128 * 64 * 2;               // one 64-dim box column: 16 KB
constexpr uint32_t kOffQ = 0;                          // 2 heads
constexpr uint32_t kOffK = kOffQ + 2 * kTile;
constexpr uint32_t kOffV = kOffK + kKStages * kTile;
constexpr uint32_t kOffBar = kOffV + kVStages * kTile;
constexpr uint32_t kBarBytes = 256;                    // barriers, TMEM slot, item queue
constexpr size_t kSmem = kOffBar + kBarBytes;         // the dynamic base is 1024-aligned
constexpr uint32_t kTmemCols = 512;  // head h: scores / P at 256 h, output at 256 h + 128
constexpr uint32_t kIdescS = idesc_bf16(128, kKeys, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, 1);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;          // log2 units
constexpr int kSoftmaxWarps = 8;

enum {
  B_Q = 0,        // Q tiles of the current item loaded
  B_QEMPTY,       // the current item's last scores are done with Q
  B_KFULL, B_KEMPTY = B_KFULL + kKStages, B_VFULL = B_KEMPTY + kKStages,
  B_VEMPTY = B_VFULL + kVStages,
  B_SFULL = B_VEMPTY + kVStages,  // [head]: scores of the head's current tile ready
  B_PFULL = B_SFULL + 2,          // [head], 128 arrivals: P of the head's current tile in TMEM
  B_ODONE = B_PFULL + 2,          // [head]: P V of the head's tiles
  B_IFULL = B_ODONE + 2,          // [2]: item queue entry written
  B_IEMPTY = B_IFULL + 2,         // [2], 1 + 8 arrivals: entry read by the MMA and softmax warps
  B_DRAIN = B_IEMPTY + 2,
  B_COUNT = B_DRAIN + 1
};
// after the barriers: TMEM base (4 B), item queue (2 x 4 B), merge flag (4 B)
static_assert(8 * B_COUNT + 16 <= kBarBytes, "barrier area");

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

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Barrier over `threads` threads that also ANDs a predicate across them.
__device__ __forceinline__ bool bar_and(int id, int threads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

// Loads that bypass L1: the partials of other CTAs are read once, after their arrival count.
__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float2 ld_cg_f2(const float2* p) {
  float2 v;
  asm volatile("ld.global.cg.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits (bounded, like the barrier waits) until another CTA has set *flag; that CTA has
// already counted its arrival, so it is running and only stores before setting it.
__device__ __forceinline__ bool wait_flag(const int* flag, int* err) {
  const long long t0 = clock64();
  for (uint32_t n = 0;; ++n) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v != 0) return true;
    if ((n & 63u) == 63u) {
      if (*reinterpret_cast<volatile int*>(err) != 0) return false;
      if (clock64() - t0 > kWaitTimeoutCycles) {
        set_error(err, CC_DEV_TIMEOUT);
        return false;
      }
    }
    __nanosleep(64);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    k_attn_prefill(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out,
                   int ld_out, const AttnTile* __restrict__ tiles, const int32_t* n_tiles_p,
                   int n_q, int n_kv, int window, float scale_log2, AttnScratch sc, AttnPaged paged,
                   int* err) {
  pdl_trigger();
  const int G = n_q / n_kv;
  const bool paired = (G & 1) == 0;                    // two heads share this KV head
  const int nh = paired ? 2 : 1;
  const int groups = paired ? n_q / 2 : n_q;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  const uint32_t sbase = smem_u32(smem);
  // the 128-byte-swizzled tiles need a 1024-byte aligned base; the kernel keeps no slack for
  // realigning, so a misplaced base is reported instead of used
  if ((sbase & 1023u) != 0) {
    if (threadIdx.x == 0) set_error(err, CC_DEV_CHECK);
    return;
  }
  auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT);
  volatile int* queue = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * B_COUNT + 4);
  volatile int* merge_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * B_COUNT + 12);

  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q), 1);
    mbar_init(bar(B_QEMPTY), 1);
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
      mbar_init(bar(B_PFULL + h), 32 * kSoftmaxWarps / 2);
      mbar_init(bar(B_ODONE + h), 1);
      mbar_init(bar(B_IFULL + h), 1);
      mbar_init(bar(B_IEMPTY + h), 1 + kSoftmaxWarps);
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
  pdl_wait();   // q, k, v and the work list of the previous kernels are complete from here on
  const int n_items = *n_tiles_p * groups;

  int issued_k = 0, issued_v = 0;
  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ scheduler + TMA
      for (int j = 0;; ++j) {
        const int e = j & 1;
        if (!mbar_wait(bar(B_IEMPTY + e), ((j >> 1) & 1) ^ 1, err)) break;
        // the first item of every CTA is its index, later ones come from the counter
        int u = j == 0 ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(sc.sched, 1);
        if (u >= n_items) u = -1;
        queue[e] = u;
        mbar_arrive(bar(B_IFULL + e));
        if (u < 0) break;
        const AttnTile tile = tiles[u / groups];
        const int head0 = (u % groups) * nh;
        const int kx = (head0 / G) * 128;
        const int n = tile.kt1 - tile.kt0;
        // Q of this item once the previous item's last scores no longer read it
        if (!mbar_wait(bar(B_QEMPTY), (j & 1) ^ 1, err)) break;
        mbar_expect_tx(bar(B_Q), nh * kTile);
        for (int h = 0; h < nh; ++h) {
          const int qx = (head0 + h) * 128;
          tma_load_2d(sbase + kOffQ + h * kTile, &tm_q, bar(B_Q), qx, tile.seq_start + tile.q0);
          tma_load_2d(sbase + kOffQ + h * kTile + kHalf, &tm_q, bar(B_Q), qx + 64,
                      tile.seq_start + tile.q0);
        }
        // one 128-key tile of K or V: two 64-column boxes of the contiguous K/V, or, paged,
        // the tile's 8 pages of 16 keys gathered through the page table (a page past the
        // call's last key is never read by a query: page 0 stands in for it)
        const int32_t* pt_row =
            paged.pt ? paged.pt + (size_t)tile.seq * paged.max_pages : nullptr;
        const int key_end = tile.prefix + tile.seq_len;
        auto load_tile = [&](const CUtensorMap* tm, uint32_t dst, uint32_t fb, int kt) {
          if (!pt_row) {
            const int y = tile.seq_start + kt * kKeys;
            tma_load_2d(dst, tm, fb, kx, y);
            tma_load_2d(dst + kHalf, tm, fb, kx + 64, y);
            return;
          }
          int ids[kKeys / 16];
#pragma unroll
          for (int i = 0; i < kKeys / 16; ++i) {
            const int pg = kt * (kKeys / 16) + i;
            ids[i] = pg < paged.max_pages ? pt_row[pg] : -1;
          }
#pragma unroll
          for (int i = 0; i < kKeys / 16; ++i) {
            int id = ids[i];
            if (id < 0 || id >= paged.n_pages) {
              if ((kt * (kKeys / 16) + i) * 16 < key_end) set_error(err, CC_DEV_CHECK);
              id = 0;
            }
            const int y = (id * n_kv + head0 / G) * 16;
            tma_load_2d(dst + i * 2048, tm, fb, 0, y);
            tma_load_2d(dst + kHalf + i * 2048, tm, fb, 64, y);
          }
        };
        // K runs up to one tile ahead of V within the item
        bool ok = true;
        for (int a = 0, b = 0; a < n || b < n;) {
          if (a < n && a <= b + 1) {
            const int st = issued_k % kKStages;
            if (!(ok = mbar_wait(bar(B_KEMPTY + st), ((issued_k / kKStages) & 1) ^ 1, err))) break;
            mbar_expect_tx(bar(B_KFULL + st), kTile);
            load_tile(&tm_k, sbase + kOffK + st * kTile, bar(B_KFULL + st), tile.kt0 + a);
            ++a;
            ++issued_k;
          } else {
            const int st = issued_v % kVStages;
            if (!(ok = mbar_wait(bar(B_VEMPTY + st), ((issued_v / kVStages) & 1) ^ 1, err))) break;
            mbar_expect_tx(bar(B_VFULL + st), kTile);
            load_tile(&tm_v, sbase + kOffV + st * kTile, bar(B_VFULL + st), tile.kt0 + b);
            ++b;
            ++issued_v;
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA
      auto issue_s = [&](int h, int g) {   // scores of head h against K tile g (CTA count)
        const uint32_t kb = sbase + kOffK + (g % kKStages) * kTile;
        const uint32_t qb = sbase + kOffQ + h * kTile;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc_mma(tmem + 256 * h, desc_kmajor_sw128(qb + off), desc_kmajor_sw128(kb + off),
                 kIdescS, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(B_SFULL + h));
      };
      bool ok = true;
      int gt = 0;   // key tiles of this CTA's earlier items
      for (int j = 0; ok; ++j) {
        const int e = j & 1;
        if (!(ok = mbar_wait(bar(B_IFULL + e), (j >> 1) & 1, err))) break;
        const int u = queue[e];
        mbar_arrive(bar(B_IEMPTY + e));
        if (u < 0) break;
        const AttnTile tile = tiles[u / groups];
        const int n = tile.kt1 - tile.kt0;
        if (!(ok = mbar_wait(bar(B_Q), j & 1, err))) break;
        if (!(ok = mbar_wait(bar(B_KFULL + gt % kKStages), (gt / kKStages) & 1, err))) break;
        tc_fence_after();
        for (int h = 0; h < nh; ++h) issue_s(h, gt);
        tc_commit(bar(B_KEMPTY + gt % kKStages));
        if (n == 1) tc_commit(bar(B_QEMPTY));
        for (int t = 0; t < n && ok; ++t) {
          const int g = gt + t;
          const bool next = t + 1 < n;
          for (int h = 0; h < nh && ok; ++h) {
            // P_h(t) is in TMEM: O_h += P_h V(t), then the head's next scores (same columns)
            if (!(ok = mbar_wait(bar(B_PFULL + h), g & 1, err))) break;
            if (h == 0 && !(ok = mbar_wait(bar(B_VFULL + g % kVStages), (g / kVStages) & 1, err)))
              break;
            if (h == 0 && next &&
                !(ok = mbar_wait(bar(B_KFULL + (g + 1) % kKStages), ((g + 1) / kKStages) & 1, err)))
              break;
            tc_fence_after();
            const uint32_t vb = sbase + kOffV + (g % kVStages) * kTile;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {   // 16 keys per MMA: 8 packed P columns
              tc_mma_ts(tmem + 256 * h + 128, tmem + 256 * h + 8 * kk,
                        desc_mnmajor_sw128(vb + kk * 2048, kHalf), kIdescPV,
                        (t > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(bar(B_ODONE + h));
            if (next) issue_s(h, g + 1);
          }
          if (!ok) break;
          tc_commit(bar(B_VEMPTY + g % kVStages));
          if (next) tc_commit(bar(B_KEMPTY + (g + 1) % kKStages));
          if (t == n - 2) tc_commit(bar(B_QEMPTY));   // the item's last scores are issued
        }
        gt += n;
      }
      tc_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax, a group per head
    // Warps 2..5 take head 0 of the item and warps 6..9 head 1 (the second group idles when
    // the item has one head). Thread r of a group owns query row r (its TMEM lane) and all 128
    // keys of every score tile, so a row's maximum, P and sum need no exchange between warps,
    // and the two heads' softmax chains run side by side while the tensor cores alternate
    // between the heads' products.
    const int wg = (warp - 2) >> 2;                  // this group's head within the item
    const int quarter = warp & 3;                    // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;               // query row in the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + 256 * wg + lane_off;   // the head's scores, then its P
    const uint32_t o_tmem = s_tmem + 128;                  // the head's output
    // All eight softmax warps take every decision to stop together, at a barrier that ANDs
    // their status, so none waits at a barrier another left.
    constexpr int kSmThreads = 32 * kSoftmaxWarps;
    bool ok = true;
    int gt = 0;
    for (int j = 0; ok; ++j) {
      const int e = j & 1;
      if (!bar_and(2, kSmThreads, mbar_wait(bar(B_IFULL + e), (j >> 1) & 1, err))) break;
      const int u = queue[e];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_IEMPTY + e));
      if (u < 0) break;
      const AttnTile tile = tiles[u / groups];
      const int n = tile.kt1 - tile.kt0;
      const int head0 = (u % groups) * nh;
      const bool active = wg < nh;                   // group-uniform
      const int q0 = tile.q0;
      const int qi = q0 + r;                         // query row among the call's tokens
      const int qa = tile.prefix + qi;               // its position: the key index it sees up to
      // this warp's rows that lie inside the sequence (rows past its end are never stored)
      const int qw_lo = tile.prefix + q0 + quarter * 32;
      const int qw_hi = tile.prefix + min(q0 + quarter * 32 + 31, tile.seq_len - 1);
      float m = -INFINITY, l = 0.f;
      for (int t = 0; t < n && ok && active; ++t) {
        const int g = gt + t;
        const int kbase = (tile.kt0 + t) * kKeys;                // first key of the tile
        // warp-uniform: every key of the tile visible to every row of this warp
        const bool full = (kbase + kKeys - 1 <= qw_lo) && (window <= 0 || qw_hi - kbase < window);
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_SFULL + wg), g & 1, err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[128];
        tmem_ld128(s_tmem, s);
        if (!full) {
          const int hi_c = qa - kbase;                           // causal: c <= hi_c
          const int lo_c = window > 0 ? qa - window + 1 - kbase : -1;
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (c <= hi_c && c >= lo_c) ? s[c] : -INFINITY;
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
        const float f = need_o ? ex2_mufu(m - mt) : 1.f;   // rescale of the older terms
        if (need) m = mt;
        const float mu = (m == -INFINITY) ? 0.f : m;
        // P = 2^(s * scale_log2 - m) (masked scores are -inf and give 0), its row sum, bf16
        // P packed two keys per column over the consumed scores: keys 64 hh .. 64 hh + 63 go
        // to columns 32 hh .. 32 hh + 31
        const float2 sc2 = make_float2(scale_log2, scale_log2);
        const float2 nm2 = make_float2(-mu, -mu);
        float2 sum[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pk[32];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int c = 64 * hh + 2 * jj;
            const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), sc2, nm2);
            // two probabilities per MUFU operation, already the bf16 P the P V MMA reads
            const uint32_t p2 = ex2_bf16x2(pack_bf16x2(x.x, x.y));
            pk[jj] = p2;
            sum[jj & 3] = __fadd2_rn(sum[jj & 3], make_float2(__uint_as_float(p2 << 16),
                                                              __uint_as_float(p2 & 0xFFFF0000u)));
          }
          tmem_st32u(s_tmem + 32 * hh, pk);
        }
        if (__any_sync(0xffffffffu, need_o)) {
          // O holds P V of tiles < t, all complete (the scores of tile t were issued after
          // them); rescaled after P is stored, so that the scores are no longer live
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float o[32];
            tmem_ld32(o_tmem + 32 * c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= f;
            tmem_st32(o_tmem + 32 * c, o);
          }
        }
        l = l * f + (((sum[0].x + sum[0].y) + (sum[1].x + sum[1].y)) +
                     ((sum[2].x + sum[2].y) + (sum[3].x + sum[3].y)));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL + wg));
      }
      if (active && ok)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B_ODONE + wg), (gt + n - 1) & 1, err));
      gt += n;
      const bool row_ok = qi < tile.seq_len;
      if (tile.n_chunks == 1) {
        if (ok && active) {
          tc_fence_after();
          const float inv = l > 0.f ? 1.f / l : 0.f;
          __nv_bfloat16* dst = out + (size_t)(tile.seq_start + qi) * ld_out + (head0 + wg) * 128;
#pragma unroll 1
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
        ok = bar_and(1, kSmThreads, ok);
        continue;
      }
      // ---- a chunk of a split query tile. Chunks count their arrival first; every chunk
      // but the last stores (max, sum, O) and raises its ready flag, and the last one waits
      // for those flags, then merges in chunk order with its own O still in tensor memory.
      // Partial O of a (slot, head) is [32 dim quads][128 rows][4]: a warp's float4 accesses
      // at one quad cover 512 contiguous bytes.
      const size_t blk = (size_t)n_q * 128 * 128;    // floats between consecutive slots
      const size_t ml_stride = (size_t)n_q * 128;
      int* const cnt = sc.counters + ((size_t)tile.split * groups + u % groups) * kCounterInts;
      const int nc = tile.n_chunks;
      ok = bar_and(1, kSmThreads, ok);
      if (threadIdx.x == 64) *merge_flag = ok ? atomicAdd(cnt, 1) : -1;
      named_barrier_sync(1, kSmThreads);
      const int order = *merge_flag;
      if (order < 0) {
        ok = false;
        continue;
      }
      tc_fence_after();
      if (order != nc - 1) {
        if (active) {
          const size_t hs = (size_t)tile.slot0 * n_q + head0 + wg;
          float* po = sc.part_o + (hs * 128 * 128 + 4 * r) + (size_t)tile.chunk * blk;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float o[32];
            tmem_ld32(o_tmem + 32 * c, o);
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(po + (size_t)((32 * c + i) >> 2) * 512) =
                  make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
          }
          sc.part_ml[hs * 128 + r + (size_t)tile.chunk * ml_stride] = make_float2(m, l);
        }
        __threadfence();
        named_barrier_sync(1, kSmThreads);
        if (threadIdx.x == 64) st_release_gpu(cnt + 1 + tile.chunk, 1);
        ok = bar_and(1, kSmThreads, ok);
        continue;
      }
      // the last chunk: wait (bounded) for the other chunks' partials
      if (threadIdx.x == 64) {
        bool ready = true;
        for (int c = 0; c < nc && ready; ++c) {
          if (c == tile.chunk) continue;
          ready = wait_flag(cnt + 1 + c, err);
        }
        if (ready) {   // every flag seen: reset the tile's counters for the next launch
          for (int c = 0; c < nc; ++c) cnt[1 + c] = 0;
          cnt[0] = 0;
        }
        *merge_flag = ready;
      }
      named_barrier_sync(1, kSmThreads);
      const bool merged = *merge_flag != 0;
      if (merged && active) {
        __threadfence();
        // chunk order, whichever chunk arrives last: M = max m_c, L = sum 2^(m_c - M) l_c,
        // O = sum 2^(m_c - M) O_c, this chunk's terms taken from its registers and TMEM
        const size_t hs = (size_t)tile.slot0 * n_q + head0 + wg;
        const float2* ml0 = sc.part_ml + hs * 128 + r;
        const float* po0 = sc.part_o + (hs * 128 * 128 + 4 * r);
        float f[kMaxChunks], lc[kMaxChunks];
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
          float2 v = make_float2(-INFINITY, 0.f);
          if (c == tile.chunk) v = make_float2(m, l);
          else if (c < nc) v = ld_cg_f2(ml0 + c * ml_stride);
          f[c] = v.x;
          lc[c] = v.y;
          M = fmaxf(M, v.x);
        }
        float Lm = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
          f[c] = (f[c] == -INFINITY) ? 0.f : ex2_mufu(f[c] - M);
          Lm += f[c] * lc[c];
        }
        const float inv = Lm > 0.f ? 1.f / Lm : 0.f;
        __nv_bfloat16* dst = out + (size_t)(tile.seq_start + qi) * ld_out + (head0 + wg) * 128;
#pragma unroll 1
        for (int cb = 0; cb < 8; ++cb) {   // 16 dims per pass
          float own[16];
          tmem_ld16(o_tmem + 16 * cb, own);
          float acc[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll 1
          for (int c = 0; c < nc; ++c) {
            if (c == tile.chunk) {
#pragma unroll
              for (int i = 0; i < 16; ++i) acc[i] += f[c] * own[i];
            } else {
              const float* po = po0 + (size_t)c * blk + (size_t)(4 * cb) * 512;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float4 v = ld_cg_f4(po + k * 512);
                acc[4 * k] += f[c] * v.x;
                acc[4 * k + 1] += f[c] * v.y;
                acc[4 * k + 2] += f[c] * v.z;
                acc[4 * k + 3] += f[c] * v.w;
              }
            }
          }
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 16; i += 8) {
              st_global_v4(dst + 16 * cb + i, pack_bf16x2(acc[i] * inv, acc[i + 1] * inv),
                           pack_bf16x2(acc[i + 2] * inv, acc[i + 3] * inv),
                           pack_bf16x2(acc[i + 4] * inv, acc[i + 5] * inv),
                           pack_bf16x2(acc[i + 6] * inv, acc[i + 7] * inv));
            }
          }
        }
      }
      ok = bar_and(1, kSmThreads, ok && merged);
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

// Key tiles [lo, hi) visited by the 128-query tile at q0 of a sequence of L new tokens that
// continue P cached keys (positions P .. P + L - 1).
__device__ __forceinline__ void tile_keys(int q0, int L, int P, int window, int* lo, int* hi) {
  *hi = ((P + min(q0 + 127, L - 1)) >> 7) + 1;
  *lo = window > 0 ? max(0, P + q0 - window + 1) >> 7 : 0;
}

// One block lists the work items of every sequence, heaviest first (a counting sort on the
// number of key tiles), so that the persistent CTAs take the longest items first.
// A query tile with w > C + kMergeTiles key tiles, C = max(kMinChunk, ceil(total work *
// groups / sms)), is cut into ceil(w / C) (at most kMaxChunks) chunks of near-equal length:
// only a tile well above the average work per SM is worth a merge. With C at least that
// average, the split tiles number fewer than sms / groups and their chunks fewer than
// 2 sms / groups, which bounds the partial buffers.
// Dynamic shared memory: tile offsets of the sequences [n_seqs + 1], then the histogram.
struct TileLists {
  int window[2];
  AttnTile* tiles[2];
  int32_t* n_tiles[2];
};

__global__ void __launch_bounds__(1024)
    k_attn_tiles(const int32_t* __restrict__ cu, int n_seqs, int max_work, int groups, int sms,
                 TileLists lists, int32_t* zero, int n_zero, const int32_t* __restrict__ prefix) {
  pdl_trigger();
  pdl_wait();
  // block b builds list b; block 0 also clears the launches' counters
  const int window = lists.window[blockIdx.x];
  AttnTile* __restrict__ tiles = lists.tiles[blockIdx.x];
  int32_t* n_tiles = lists.n_tiles[blockIdx.x];
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_zero; i += blockDim.x) zero[i] = 0;
  extern __shared__ int sh[];
  int* toff = sh;                   // [n_seqs + 1]
  int* hist = sh + n_seqs + 1;      // [max_work + 1]
  __shared__ unsigned long long wsum;
  __shared__ int n_split, n_slots, chunk_cap;
  for (int i = threadIdx.x; i <= max_work; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int s = 0; s < n_seqs; ++s) {
      toff[s] = acc;
      acc += max(0, cu[s + 1] - cu[s] + 127) >> 7;
    }
    toff[n_seqs] = acc;
    wsum = 0ull;
    n_split = 0;
    n_slots = 0;
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
  unsigned long long mine = 0;
  for (int g = threadIdx.x; g < total; g += blockDim.x) {
    int s, q0, lo, hi;
    locate(g, &s, &q0);
    tile_keys(q0, cu[s + 1] - cu[s], prefix ? prefix[s] : 0, window, &lo, &hi);
    mine += hi - lo;
  }
  atomicAdd(&wsum, mine);
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long avg = (wsum * groups + sms - 1) / sms;
    chunk_cap = static_cast<int>(max(static_cast<unsigned long long>(kMinChunk), avg));
  }
  __syncthreads();
  const int C = chunk_cap;
  for (int g = threadIdx.x; g < total; g += blockDim.x) {
    int s, q0, lo, hi;
    locate(g, &s, &q0);
    tile_keys(q0, cu[s + 1] - cu[s], prefix ? prefix[s] : 0, window, &lo, &hi);
    const int w = hi - lo;
    const int nc = w > C + kMergeTiles ? min((w + C - 1) / C, kMaxChunks) : 1;
    for (int c = 0; c < nc; ++c)
      atomicAdd(&hist[min((c + 1) * w / nc - c * w / nc, max_work)], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // start slot of every work value, largest work first
    int acc = 0;
    for (int w = max_work; w >= 0; --w) {
      const int c = hist[w];
      hist[w] = acc;
      acc += c;
    }
    *n_tiles = acc;
  }
  __syncthreads();
  for (int g = threadIdx.x; g < total; g += blockDim.x) {
    int s, q0, lo, hi;
    locate(g, &s, &q0);
    const int L = cu[s + 1] - cu[s];
    const int P = prefix ? prefix[s] : 0;
    tile_keys(q0, L, P, window, &lo, &hi);
    const int w = hi - lo;
    const int nc = w > C + kMergeTiles ? min((w + C - 1) / C, kMaxChunks) : 1;
    int split = -1, slot0 = -1;
    if (nc > 1) {
      split = atomicAdd(&n_split, 1);
      slot0 = atomicAdd(&n_slots, nc);
    }
    for (int c = 0; c < nc; ++c) {
      const int k0 = lo + c * w / nc, k1 = lo + (c + 1) * w / nc;
      const int slot = atomicAdd(&hist[min(k1 - k0, max_work)], 1);
      AttnTile t;
      t.seq_start = cu[s];
      t.seq_len = L;
      t.q0 = q0;
      t.kt0 = k0;
      t.kt1 = k1;
      t.chunk = c;
      t.n_chunks = nc;
      t.slot0 = slot0;
      t.split = split;
      t.prefix = P;
      t.seq = s;
      t.pad = 0;
      tiles[slot] = t;
    }
  }
}

}  // namespace

int attn_groups(int n_q, int n_kv) {
  return (n_kv > 0 && ((n_q / n_kv) & 1) == 0) ? n_q / 2 : n_q;
}
int attn_split_slots(int groups) { return 2 * num_sms() / groups + 1; }
int attn_split_tiles(int groups) { return num_sms() / groups + 1; }
int attn_counter_ints(int groups) { return attn_split_tiles(groups) * groups * kCounterInts; }
size_t attn_part_ml_pairs(int n_q, int n_kv) {
  return (size_t)attn_split_slots(attn_groups(n_q, n_kv)) * n_q * 128;
}
size_t attn_part_o_floats(int n_q, int n_kv) { return attn_part_ml_pairs(n_q, n_kv) * 128; }

int attn_max_tiles(int tokens, int n_seqs) { return (tokens + 127) / 128 + n_seqs + 2 * num_sms(); }

cc_status launch_attn_tiles(const int32_t* cu_seqlens, int n_seqs, int tokens, int groups,
                            int window_a, AttnTile* tiles_a, int32_t* n_tiles_a, int window_b,
                            AttnTile* tiles_b, int32_t* n_tiles_b, int32_t* zero, int n_zero,
                            cudaStream_t s, const int32_t* prefix, int max_prefix) {
  // key tiles of a query tile: at most (longest prefix + tokens) / 128 + 2
  const int max_work = (max_prefix + tokens + 127) / 128 + 1;
  const size_t smem = (size_t)(n_seqs + 1 + max_work + 1) * sizeof(int);
  if (groups <= 0 || !tiles_a || !n_tiles_a || n_zero < 0) return CC_ERR_INVALID_ARG;
  if (smem > 200 * 1024) return CC_ERR_UNSUPPORTED;
  if (smem > 48 * 1024)
    CC_CHECK_CUDA(cudaFuncSetAttribute(k_attn_tiles, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem)));
  TileLists lists;
  lists.window[0] = window_a;
  lists.tiles[0] = tiles_a;
  lists.n_tiles[0] = n_tiles_a;
  lists.window[1] = window_b;
  lists.tiles[1] = tiles_b;
  lists.n_tiles[1] = n_tiles_b;
  const int blocks = tiles_b ? 2 : 1;
  CC_CHECK_CUDA(launch_pdl(k_attn_tiles, dim3(blocks), dim3(1024), smem, s, cu_seqlens, n_seqs,
                          max_work, groups, num_sms(), lists, zero, n_zero, prefix));
  return CC_OK;
}

cc_status launch_attn_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              __nv_bfloat16* out, int ld_out, const AttnTile* tiles,
                              const int32_t* n_tiles, int max_tiles, int n_q, int n_kv,
                              int window, const AttnScratch& sc, int* err, cudaStream_t s,
                              const AttnPaged& paged) {
  static std::atomic<bool> smem_set{false};
  CC_CHECK_CUDA(allow_dynamic_smem(k_attn_prefill, kSmem, smem_set));
  if (max_tiles <= 0) return CC_OK;
  if (n_kv <= 0 || n_q % n_kv != 0) return CC_ERR_INVALID_ARG;
  if (!sc.part_o || !sc.part_ml || !sc.counters || !sc.sched) return CC_ERR_INVALID_ARG;
  const float scale_log2 = (1.0f / sqrtf(128.0f)) * kLog2e;
  const long long items = (long long)max_tiles * attn_groups(n_q, n_kv);
  const int grid = static_cast<int>(std::min<long long>(items, num_sms()));
  CC_CHECK_CUDA(launch_pdl(k_attn_prefill, dim3(grid), dim3(kThreads), kSmem, s, tq, tk, tv, out,
                          ld_out, tiles, n_tiles, n_q, n_kv, window, scale_log2, sc, paged, err));
  return CC_OK;
}

int attn_kv_box_rows() { return kKeys; }

}  // namespace cc
