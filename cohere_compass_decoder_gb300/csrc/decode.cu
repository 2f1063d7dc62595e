// Decode attention over a paged KV cache on the tcgen05 tensor cores: one query token per
// sequence, split-KV.
//
// Definition: the new token of sequence b (query index n-1, n = n_keys[b]) attends over
// keys 0..n-1 of its cache (full layers) or over the last `window` of them (sliding
// layers), grouped-query, scale d^-0.5 (mlxcel issue "Cohere Compass /
// North-Micro-Vision", section "Text decoder forward"). The cache layout is this
// library's: pool [page][kv_head][16 tokens][128], so one page of one KV head is a 4 KB
// contiguous block.
//
// Kernel 1, one CTA per (split of up to 1024 keys, KV head, sequence), 6 warps, two passes:
//   warp 0      TMA: the G query heads of the KV head (one 16-row box), then the split's K
//               tiles and after them its V tiles (128 keys each: the 8 pages gathered
//               through the page table straight into 128-byte-swizzled tiles) through one
//               2-stage ring
//   warp 1      MMA: S^T_i = K_i Q^T for every tile i (M = 128 keys, N = 16 query rows of
//               which G are used) into its own 16 TMEM columns; then O^T += V_i^T P_i (V read
//               MN-major as the A operand, P_i = [16 x 128 keys] bf16 in shared memory)
//   warps 2..5  softmax, one key of every tile per thread: the split's per-head maximum
//               (shuffles, then the four warps through shared memory), p = 2^(s - max),
//               P tiles into shared memory, per-head sums.
// With one maximum per split there is no rescaling, and the CTA synchronises twice in all.
// Each K/V byte is read from HBM once for all G query heads; the CTA needs about 100 KB of
// shared memory, so two CTAs share an SM and cover each other's latencies.
// Kernel 2 merges the splits of each (sequence, head) and writes O as bf16.
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace cc {

namespace {

constexpr int kThreads = 192;
constexpr int kPage = 16;
constexpr int kTileKeys = 128;
constexpr int kPagesPerTile = kTileKeys / kPage;   // 8
constexpr int kTilesPerSplit = 8;                  // 1024 keys per CTA
constexpr int kPagesPerSplit = kPagesPerTile * kTilesPerSplit;
constexpr int kStages = 2;
constexpr int kQRows = 16;                         // MMA N (query heads, padded)
constexpr uint32_t kTile = kTileKeys * 128 * 2;    // 32 KB: 128 keys x 128 dims
constexpr uint32_t kHalf = kTileKeys * 64 * 2;     // one 64-dim box column: 16 KB
constexpr uint32_t kQBytes = kQRows * 128 * 2;     // 4 KB
constexpr uint32_t kPBytes = kQRows * kTileKeys * 2;   // 4 KB per tile
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffRing = 4096;                // 1024-aligned
constexpr uint32_t kOffP = kOffRing + kStages * kTile;
constexpr uint32_t kOffRed = kOffP + kTilesPerSplit * kPBytes;   // [4 warps][16] floats
constexpr uint32_t kOffPid = kOffRed + 4 * 16 * 4;              // the split's page ids
constexpr uint32_t kOffBar = kOffPid + kPagesPerSplit * 4;
constexpr size_t kSmem = 1024 + kOffBar + 256;
constexpr uint32_t kTmemCols = 256;                // S^T of 8 tiles (16 columns each) | O^T
constexpr uint32_t kTmemO = 16 * kTilesPerSplit;
constexpr uint32_t kIdescS = idesc_bf16(128, kQRows, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, kQRows, 0) | (1u << 15);   // A MN-major
constexpr float kLog2e = 1.4426950408889634f;

enum {
  B_Q = 0, B_FULL = 1, B_EMPTY = 1 + kStages, B_SFULL = 1 + 2 * kStages, B_PFULL = B_SFULL + 1,
  B_ODONE = B_PFULL + 1, B_DRAIN = B_ODONE + 1, B_COUNT = B_DRAIN + 1
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Barrier over `threads` threads that also ANDs a predicate across them: the softmax warps
// take every give-up decision together, so none waits at a barrier the others left.
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

// Page id of page index p of sequence row `pt`, or -1 when the entry lies outside the table
// or names no page of the pool.
__device__ __forceinline__ int page_id(const int32_t* pt, int p, int max_pages, int n_pages) {
  if (p < 0 || p >= max_pages) return -1;
  const int id = pt[p];
  return (id >= 0 && id < n_pages) ? id : -1;
}

template <int G>
__global__ void __launch_bounds__(kThreads, 2)
    k_attn_decode(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, int n_pages,
                  const int32_t* __restrict__ page_table, int max_pages,
                  const int32_t* __restrict__ n_keys, int n_kv, int window, int splits,
                  float scale_log2, float* __restrict__ part_o, float* __restrict__ part_ml,
                  int* err) {
  pdl_trigger();
  pdl_wait();
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int n_q = n_kv * G;
  const int n = n_keys[b];
  const int lo = window > 0 ? max(0, n - window) : 0;
  const int t_first = lo / kTileKeys, t_last = (n - 1) / kTileKeys;   // key tiles in view
  const int st0 = t_first + split * kTilesPerSplit;
  const int nt = n <= 0 ? 0 : min(t_last, st0 + kTilesPerSplit - 1) - st0 + 1;
  const size_t part_base = ((size_t)b * n_q + (size_t)g * G) * splits + split;
  if (nt <= 0) {  // nothing to attend in this split
    if (threadIdx.x < G) {
      part_ml[(part_base + (size_t)threadIdx.x * splits) * 2 + 0] = -INFINITY;
      part_ml[(part_base + (size_t)threadIdx.x * splits) * 2 + 1] = 0.f;
    }
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  int* pid = reinterpret_cast<int*>(smem + kOffPid);
  const int32_t* pt = page_table + (size_t)b * max_pages;

  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
    }
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_PFULL), 128);
    mbar_init(bar(B_ODONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // the split's page ids, read once: the producer's gathers and the masks use this copy
  if (threadIdx.x < kPagesPerSplit)
    pid[threadIdx.x] = page_id(pt, st0 * kPagesPerTile + threadIdx.x, max_pages, n_pages);
  // P rows G..15 are padding: zero them in every tile buffer
  if (G < kQRows) {
    for (int i = threadIdx.x; i < kTilesPerSplit * kPBytes / 16; i += kThreads) {
      const uint32_t off = i * 16;
      const int row = (off % 2048) / 128;   // 16 rows of 128 B per 2 KB box
      if (row >= G) st_shared_v4(sbase + kOffP + off, 0u, 0u, 0u, 0u);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int issued = 0;
  if (warp == 0) {
    if (lane == 0) {
      mbar_expect_tx(bar(B_Q), kQBytes);
      tma_load_2d(sbase + kOffQ, &tm_q, bar(B_Q), 0, b * n_q + g * G);
      tma_load_2d(sbase + kOffQ + kQBytes / 2, &tm_q, bar(B_Q), 64, b * n_q + g * G);
      // ring slot j: K tile j for j < nt, then V tile j - nt
      for (int j = 0; j < 2 * nt; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(bar(B_EMPTY + s), ((j / kStages) & 1) ^ 1, err)) break;
        mbar_expect_tx(bar(B_FULL + s), kTile);
        const bool is_v = j >= nt;
        const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
        const int p0 = (is_v ? j - nt : j) * kPagesPerTile;
#pragma unroll
        for (int p = 0; p < kPagesPerTile; ++p) {
          const int id = max(pid[p0 + p], 0);   // keys of an invalid page are masked below
          const int y = (id * n_kv + g) * kPage;
          const uint32_t dst = sbase + kOffRing + s * kTile + p * (kPage * 128);
          tma_load_2d(dst, tm, bar(B_FULL + s), 0, y);
          tma_load_2d(dst + kHalf, tm, bar(B_FULL + s), 64, y);
        }
        ++issued;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = mbar_wait(bar(B_Q), 0, err);
      for (int j = 0; j < 2 * nt && ok; ++j) {
        const int s = j % kStages;
        if (j == nt) {   // every score tile done: wait for the softmax's P tiles
          tc_commit(bar(B_SFULL));
          if (!(ok = mbar_wait(bar(B_PFULL), 0, err))) break;
        }
        if (!(ok = mbar_wait(bar(B_FULL + s), (j / kStages) & 1, err))) break;
        tc_fence_after();
        const uint32_t tb = sbase + kOffRing + s * kTile;
        if (j < nt) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            const uint32_t qoff = (kk >> 2) * (kQBytes / 2) + (kk & 3) * 32;
            tc_mma(tmem + 16 * j, desc_kmajor_sw128(tb + off),
                   desc_kmajor_sw128(sbase + kOffQ + qoff), kIdescS, kk > 0 ? 1u : 0u);
          }
        } else {
          const int i = j - nt;
          const uint32_t pb = sbase + kOffP + i * kPBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {   // 16 keys per MMA
            tc_mma(tmem + kTmemO, desc_mnmajor_sw128(tb + kk * 2048, kHalf),
                   desc_kmajor_sw128(pb + (kk >> 2) * (kPBytes / 2) + (kk & 3) * 32), kIdescPV,
                   (i > 0 || kk > 0) ? 1u : 0u);
          }
        }
        tc_commit(bar(B_EMPTY + s));
      }
      if (ok) tc_commit(bar(B_ODONE));
      tc_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- softmax, key per thread
    const int quarter = warp & 3;
    const int t = quarter * 32 + lane;                  // key of every tile, TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = bar_and(2, 128, mbar_wait(bar(B_SFULL), 0, err));
    float m[G], lsum[G];
    float s[kTilesPerSplit][G];
    if (ok) {
      tc_fence_after();
      bool bad_page = false;
#pragma unroll
      for (int i = 0; i < kTilesPerSplit; ++i) {
        if (i < nt) {
          float v[16];
          tmem_ld16(tmem + 16 * i + lane_off, v);
          const int kj = (st0 + i) * kTileKeys + t;
          bool vis = kj >= lo && kj < n;
          if (vis && pid[i * kPagesPerTile + t / kPage] < 0) {
            bad_page = true;
            vis = false;
          }
#pragma unroll
          for (int hh = 0; hh < G; ++hh) s[i][hh] = vis ? v[hh] * scale_log2 : -INFINITY;
        } else {
#pragma unroll
          for (int hh = 0; hh < G; ++hh) s[i][hh] = -INFINITY;
        }
      }
      if (bad_page) set_error(err, CC_DEV_CHECK);
      // the split's maximum of every head
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float x = s[0][hh];
#pragma unroll
        for (int i = 1; i < kTilesPerSplit; ++i) x = fmaxf(x, s[i][hh]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
        if (lane == 0) red[quarter * 16 + hh] = x;
      }
    }
    named_barrier_sync(1, 128);
    if (ok) {
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float mx = fmaxf(fmaxf(red[hh], red[16 + hh]), fmaxf(red[32 + hh], red[48 + hh]));
        m[hh] = mx;
        lsum[hh] = 0.f;
      }
      // P tiles: row hh (head), key t of the 128-byte-swizzled [16 x 128] bf16 buffer
      const int ch = (t & 63) >> 3;
#pragma unroll
      for (int i = 0; i < kTilesPerSplit; ++i) {
        if (i >= nt) break;
        const uint32_t pb = sbase + kOffP + i * kPBytes + (t >> 6) * (kPBytes / 2);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float p = ex2f(s[i][hh] - (m[hh] == -INFINITY ? 0.f : m[hh]));
          lsum[hh] += p;
          const uint32_t addr = pb + hh * 128 + ((ch ^ (hh & 7)) << 4) + ((t & 7) << 1);
          const __nv_bfloat16 pv = __float2bfloat16_rn(p);
          asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr),
                       "h"(*reinterpret_cast<const unsigned short*>(&pv))
                       : "memory");
        }
      }
      fence_proxy_async_smem();
    }
    mbar_arrive(bar(B_PFULL));
    named_barrier_sync(1, 128);   // every thread has read the maxima from `red`
    if (ok) {
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float x = lsum[hh];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) red[quarter * 16 + hh] = x;
      }
    }
    named_barrier_sync(1, 128);
    if (ok) ok = bar_and(2, 128, mbar_wait(bar(B_ODONE), 0, err));
    if (ok) {
      tc_fence_after();
      float o[16];
      tmem_ld16(tmem + kTmemO + lane_off, o);   // lane t holds dim t of every head
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const size_t pb2 = part_base + (size_t)hh * splits;
        part_o[pb2 * 128 + t] = o[hh];
        if (t == 0) {
          part_ml[pb2 * 2 + 0] = m[hh];
          part_ml[pb2 * 2 + 1] = red[hh] + red[16 + hh] + red[32 + hh] + red[48 + hh];
        }
      }
    } else if (t == 0) {
      // a bounded wait gave up: the split counts as empty, so that the combine never merges
      // a partial that an earlier launch left in the scratch
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const size_t pb2 = part_base + (size_t)hh * splits;
        part_ml[pb2 * 2 + 0] = -INFINITY;
        part_ml[pb2 * 2 + 1] = 0.f;
      }
    }
  }
  __syncthreads();
  if (warp == 0 && lane == 0) {
    // a failed launch may leave loads in flight: let them land (bounded)
    for (int j = max(0, issued - kStages); j < issued; ++j)
      mbar_wait(bar(B_FULL + (j % kStages)), (j / kStages) & 1, nullptr);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

__global__ void __launch_bounds__(128)
    k_decode_combine(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                     int splits, int n_q, __nv_bfloat16* __restrict__ out, int ld_out) {
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const size_t base = ((size_t)b * n_q + h) * splits;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part_ml[(base + s) * 2]);
  float O = 0.f, Lsum = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const float ms = part_ml[(base + s) * 2];
      if (ms == -INFINITY) continue;
      const float f = exp2f(ms - M);
      O += f * part_o[(base + s) * 128 + d];
      Lsum += f * part_ml[(base + s) * 2 + 1];
    }
  }
  out[(size_t)b * ld_out + (size_t)h * 128 + d] = __float2bfloat16_rn(Lsum > 0.f ? O / Lsum : 0.f);
}


template <int G>
cc_status launch_dec(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     int n_pages, const int32_t* pt, int max_pages, const int32_t* n_keys,
                     int batch, int n_kv, int window, int splits, DecodeScratch scr, int* err,
                     cudaStream_t s) {
  static std::atomic<bool> smem_set{false};
  CC_CHECK_CUDA(allow_dynamic_smem(k_attn_decode<G>, kSmem, smem_set));
  const float sl2 = (1.0f / sqrtf(128.0f)) * kLog2e;
  dim3 grid(splits, n_kv, batch);
  CC_CHECK_CUDA(launch_pdl(k_attn_decode<G>, grid, dim3(kThreads), kSmem, s, tq, tk, tv, n_pages, pt,
                          max_pages, n_keys, n_kv, window, splits, sl2, scr.part_o, scr.part_ml,
                          err));
  return CC_OK;
}

}  // namespace

int decode_splits(int max_pages) { return (max_pages + kPagesPerSplit - 1) / kPagesPerSplit; }

size_t decode_scratch_floats(int batch, int n_q, int max_pages) {
  return (size_t)batch * n_q * decode_splits(max_pages) * (128 + 2);
}

cc_status launch_attn_decode(const __nv_bfloat16* q, int ld_q, const __nv_bfloat16* k_pool,
                             const __nv_bfloat16* v_pool, int n_pages, const int32_t* page_table,
                             int max_pages, const int32_t* n_keys, int batch, int n_q, int n_kv,
                             int page_size, int window, DecodeScratch scr, __nv_bfloat16* out,
                             int ld_out, int* err, cudaStream_t s) {
  if (batch <= 0) return CC_OK;
  if (page_size != kPage || n_q % n_kv != 0 || ld_q != n_q * 128) return CC_ERR_UNSUPPORTED;
  const int G = n_q / n_kv;
  CUtensorMap tq, tk, tv;
  const uint64_t pool_rows = (uint64_t)n_pages * n_kv * kPage;
  if (!make_tmap_bf16_2d(&tq, q, (uint64_t)batch * n_q, 128, 128, kQRows, 64) ||
      !make_tmap_bf16_2d(&tk, k_pool, pool_rows, 128, 128, kPage, 64) ||
      !make_tmap_bf16_2d(&tv, v_pool, pool_rows, 128, 128, kPage, 64))
    return CC_ERR_INVALID_ARG;
  const int splits = decode_splits(max_pages);
  cc_status st;
  switch (G) {
    case 1: st = launch_dec<1>(tq, tk, tv, n_pages, page_table, max_pages, n_keys, batch, n_kv,
                               window, splits, scr, err, s); break;
    case 2: st = launch_dec<2>(tq, tk, tv, n_pages, page_table, max_pages, n_keys, batch, n_kv,
                               window, splits, scr, err, s); break;
    case 4: st = launch_dec<4>(tq, tk, tv, n_pages, page_table, max_pages, n_keys, batch, n_kv,
                               window, splits, scr, err, s); break;
    case 8: st = launch_dec<8>(tq, tk, tv, n_pages, page_table, max_pages, n_keys, batch, n_kv,
                               window, splits, scr, err, s); break;
    case 16: st = launch_dec<16>(tq, tk, tv, n_pages, page_table, max_pages, n_keys, batch, n_kv,
                                 window, splits, scr, err, s); break;
    default: return CC_ERR_UNSUPPORTED;
  }
  if (st != CC_OK) return st;
  CC_CHECK_CUDA(launch_pdl(k_decode_combine, dim3(n_q, batch), dim3(128), 0, s, scr.part_o,
                          scr.part_ml, splits, n_q, out, ld_out));
  CC_CHECK_CUDA(cudaGetLastError());
  return CC_OK;
}

// ------------------------------------------------------------ no-allocation variant
// Fixed split-KV scratch for callers that cannot allocate: 4 Mi floats (16 MiB) per GPU.
// Every split of a call either writes its partial (max, sum, O) or marks itself empty
// (max = -inf): when it has no keys in view, and when one of its bounded waits gave up (the
// launch then also reports CC_ERR_TIMEOUT through err_flag, when one is given). The combine
// reads only the splits of the current call, so nothing needs clearing between calls.
constexpr size_t kNoAllocScratchFloats = size_t(1) << 22;
constexpr int kNoAllocMaxDevices = 64;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

// Device address of g_noalloc_scratch on the current device, looked up once per device.
static cc_status noalloc_scratch(float** out) {
  static std::mutex mu;
  static float* addr[kNoAllocMaxDevices] = {};
  int dev = 0;
  CC_CHECK_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return CC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      last_cuda_error() = e;
      return CC_ERR_CUDA;
    }
    addr[dev] = static_cast<float*>(p);
  }
  *out = addr[dev];
  return CC_OK;
}

}  // namespace cc

extern "C" cc_status cc_op_attention_decode_noalloc(const void* q, const void* k_pool,
                                                    const void* v_pool, int32_t n_pages,
                                                    const int32_t* page_table, int32_t max_pages,
                                                    const int32_t* n_keys, int32_t batch,
                                                    int32_t n_q, int32_t n_kv, int32_t page_size,
                                                    int32_t window, void* out, int32_t ld_out,
                                                    int32_t* err_flag, void* stream) {
  using namespace cc;
  if (batch < 0 || n_q <= 0 || n_kv <= 0 || n_q % n_kv || max_pages <= 0 || window < 0 ||
      page_size <= 0 || ld_out < n_q * 128 || n_pages <= 0)
    return CC_ERR_INVALID_ARG;
  if (batch == 0) return CC_OK;
  if (!q || !k_pool || !v_pool || !page_table || !n_keys || !out) return CC_ERR_INVALID_ARG;
  if (decode_scratch_floats(batch, n_q, max_pages) > kNoAllocScratchFloats)
    return CC_ERR_INVALID_ARG;
  float* scratch = nullptr;
  CC_CHECK_STATUS(noalloc_scratch(&scratch));
  DecodeScratch scr;
  scr.part_o = scratch;
  scr.part_ml = scratch + (size_t)batch * n_q * decode_splits(max_pages) * 128;
  return launch_attn_decode(static_cast<const __nv_bfloat16*>(q), n_q * 128,
                            static_cast<const __nv_bfloat16*>(k_pool),
                            static_cast<const __nv_bfloat16*>(v_pool), n_pages, page_table,
                            max_pages, n_keys, batch, n_q, n_kv, page_size, window, scr,
                            static_cast<__nv_bfloat16*>(out), ld_out, err_flag,
                            static_cast<cudaStream_t>(stream));
}
