// Decode attention over a paged KV cache: one query token per sequence, split-KV.
//
// Definition: the new token of sequence b (query index n-1, n = n_keys[b]) attends over
// keys 0..n-1 of its cache (full layers) or over the last `window` of them (sliding
// layers), grouped-query, scale d^-0.5 (mlxcel issue "Cohere Compass /
// North-Micro-Vision", section "Text decoder forward"; the cache layout is this
// library's: pool [page][kv_head][16 tokens][128], so one page of one KV head is a 4 KB
// contiguous block).
//
// Kernel 1 (grid: key splits x KV heads x batch, 4 warps): every warp streams its pages
// (4 KB of K and 4 KB of V each) with cp.async.bulk into a private 3-slot shared ring, so
// about 200 KB per SM are in flight. The G = n_q / n_kv query heads that share the KV head
// are handled together: per step 8 lanes take one key (16 of its 128 dims each, 16-byte
// shared loads that do not conflict), so each K/V byte is read from HBM once for all G
// heads. Online softmax per head in the log2 domain; the warps' partial results merge in
// shared memory and the split's (max, sum, unnormalised O) goes to scratch.
// Kernel 2 merges the splits of each (sequence, head) and writes O as bf16.
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace cc {

namespace {

constexpr int kWarps = 4;
constexpr int kSlots = 3;
constexpr int kPage = 16;
constexpr uint32_t kPageBytes = kPage * 128 * 2;       // 4 KB per page and head
constexpr uint32_t kSlotBytes = 2 * kPageBytes;        // K and V
constexpr int kPagesPerSplit = 16;
constexpr float kLog2e = 1.4426950408889634f;

template <int G>
struct DecSmem {
  static constexpr uint32_t kRing = kWarps * kSlots * kSlotBytes;      // 96 KB
  static constexpr uint32_t kMerge = kWarps * G * 128 * 4;             // per-warp O
  static constexpr uint32_t kML = kWarps * G * 2 * 4;
  static constexpr uint32_t kBars = kWarps * kSlots * 8;
  static constexpr size_t kTotal = 128 + kRing + kMerge + kML + kBars;
};

__device__ __forceinline__ void unpack8(uint4 raw, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

template <int G>
__global__ void __launch_bounds__(kWarps * 32)
    k_attn_decode(const __nv_bfloat16* __restrict__ q, int ld_q,
                  const __nv_bfloat16* __restrict__ kpool, const __nv_bfloat16* __restrict__ vpool,
                  int n_pages, const int32_t* __restrict__ page_table, int max_pages,
                  const int32_t* __restrict__ n_keys, int n_kv, int window, int splits,
                  float scale_log2, float* __restrict__ part_o, float* __restrict__ part_ml,
                  int* err) {
  using L = DecSmem<G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  uint8_t* ring = smem;
  float* wo = reinterpret_cast<float*>(smem + L::kRing);             // [warp][G][128]
  float* wml = reinterpret_cast<float*>(smem + L::kRing + L::kMerge);  // [warp][G][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kRing + L::kMerge + L::kML);

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int n_q = n_kv * G;
  const int warp = warp_id(), lane = lane_id();
  const int n = n_keys[b];
  const int lo = window > 0 ? max(0, n - window) : 0;
  const int p_first = lo / kPage, p_last = (n - 1) / kPage;
  const int sp0 = p_first + split * kPagesPerSplit;
  const int sp1 = min(p_last, sp0 + kPagesPerSplit - 1);
  const size_t part_base = ((size_t)b * n_q + (size_t)g * G) * splits + split;

  if (n <= 0 || sp0 > sp1) {  // nothing to attend in this split
    if (threadIdx.x < G) {
      part_ml[(part_base + (size_t)threadIdx.x * splits) * 2 + 0] = -INFINITY;
      part_ml[(part_base + (size_t)threadIdx.x * splits) * 2 + 1] = 0.f;
    }
    return;
  }

  // pages of this warp: sp0 + warp + kWarps * i, i < cnt
  const int cnt = (sp1 - sp0 - warp) >= 0 ? (sp1 - sp0 - warp) / kWarps + 1 : 0;
  const uint32_t ring_w = smem_u32(ring) + warp * kSlots * kSlotBytes;
  const uint32_t bar_w = smem_u32(bars) + warp * kSlots * 8;
  const int32_t* pt = page_table + (size_t)b * max_pages;

  // page id of this warp's i-th page; an id outside the pool is reported and replaced by
  // page 0 (its keys are masked) so that the ring's phase accounting stays regular
  auto page_of = [&](int i, bool* valid) -> int {
    const int p = sp0 + warp + kWarps * i;
    const int id = pt[p];
    *valid = id >= 0 && id < n_pages;
    return *valid ? id : 0;
  };
  int issued = 0;
  auto issue = [&](int i) {
    bool valid;
    const int id = page_of(i, &valid);
    if (!valid) set_error(err, CC_DEV_CHECK);
    const int slot = i % kSlots;
    const uint32_t bar = bar_w + 8 * slot;
    const size_t off = ((size_t)id * n_kv + g) * (kPage * 128);
    mbar_expect_tx(bar, kSlotBytes);
    bulk_load(ring_w + slot * kSlotBytes, kpool + off, kPageBytes, bar);
    bulk_load(ring_w + slot * kSlotBytes + kPageBytes, vpool + off, kPageBytes, bar);
    ++issued;
  };

  if (lane == 0) {
    for (int s = 0; s < kSlots; ++s) mbar_init(bar_w + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (lane == 0) {
    for (int i = 0; i < kSlots && i < cnt; ++i) issue(i);
  }

  // this lane's 16 dims: [8*(lane%8), +8) and [64 + 8*(lane%8), +8); its key in a step of 4
  const int sub = lane & 7, kg = lane >> 3;
  float qf[G][16];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const __nv_bfloat16* qp = q + (size_t)b * ld_q + (size_t)(g * G + h) * 128;
    unpack8(*reinterpret_cast<const uint4*>(qp + 8 * sub), qf[h]);
    unpack8(*reinterpret_cast<const uint4*>(qp + 64 + 8 * sub), qf[h] + 8);
  }
  float m[G], l[G], o[G][16];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) o[h][e] = 0.f;
  }

  bool ok = true;
  for (int i = 0; i < cnt && ok; ++i) {
    const int slot = i % kSlots;
    const int page_pos = sp0 + warp + kWarps * i;  // page index within the sequence
    bool valid;
    page_of(i, &valid);
    {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_w + 8 * slot, (i / kSlots) & 1, err));
      if (!ok) break;
      const uint32_t ks = ring_w + slot * kSlotBytes;
      const uint32_t vs = ks + kPageBytes;
      float sc[4][G];
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const int key = st * 4 + kg;
        uint4 r0, r1;
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r0.x), "=r"(r0.y), "=r"(r0.z), "=r"(r0.w)
                     : "r"(ks + key * 256 + sub * 16));
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r1.x), "=r"(r1.y), "=r"(r1.z), "=r"(r1.w)
                     : "r"(ks + key * 256 + 128 + sub * 16));
        float kf[16];
        unpack8(r0, kf);
        unpack8(r1, kf + 8);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float d = 0.f;
#pragma unroll
          for (int e = 0; e < 16; ++e) d = fmaf(qf[h][e], kf[e], d);
          d += __shfl_xor_sync(0xffffffffu, d, 1);
          d += __shfl_xor_sync(0xffffffffu, d, 2);
          d += __shfl_xor_sync(0xffffffffu, d, 4);
          const int kj = page_pos * kPage + key;
          sc[st][h] = (valid && kj >= lo && kj < n) ? d * scale_log2 : -INFINITY;
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float pm = fmaxf(fmaxf(sc[0][h], sc[1][h]), fmaxf(sc[2][h], sc[3][h]));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
        const float mn = fmaxf(m[h], pm);
        const float f = (m[h] == -INFINITY) ? 0.f : exp2f(m[h] - mn);
        const float mu = (mn == -INFINITY) ? 0.f : mn;
        l[h] *= f;
#pragma unroll
        for (int e = 0; e < 16; ++e) o[h][e] *= f;
        m[h] = mn;
#pragma unroll
        for (int st = 0; st < 4; ++st) sc[st][h] = exp2f(sc[st][h] - mu);
      }
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const int key = st * 4 + kg;
        uint4 r0, r1;
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r0.x), "=r"(r0.y), "=r"(r0.z), "=r"(r0.w)
                     : "r"(vs + key * 256 + sub * 16));
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r1.x), "=r"(r1.y), "=r"(r1.z), "=r"(r1.w)
                     : "r"(vs + key * 256 + 128 + sub * 16));
        float vf[16];
        unpack8(r0, vf);
        unpack8(r1, vf + 8);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float p = sc[st][h];
          l[h] += p;
#pragma unroll
          for (int e = 0; e < 16; ++e) o[h][e] = fmaf(p, vf[e], o[h][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0 && i + kSlots < cnt) issue(i + kSlots);
  }

  // the four key groups of the warp hold disjoint keys: sum them
#pragma unroll
  for (int h = 0; h < G; ++h) {
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 8);
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 16);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      o[h][e] += __shfl_xor_sync(0xffffffffu, o[h][e], 8);
      o[h][e] += __shfl_xor_sync(0xffffffffu, o[h][e], 16);
    }
  }
  if (lane < 8) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float* dst = wo + ((size_t)warp * G + h) * 128;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        dst[8 * sub + e] = o[h][e];
        dst[64 + 8 * sub + e] = o[h][8 + e];
      }
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      wml[(warp * G + h) * 2 + 0] = m[h];
      wml[(warp * G + h) * 2 + 1] = l[h];
    }
  }
  // drain: a slot issued but not consumed (only after a failed wait) must land first
  if (lane == 0 && !ok) {
    for (int i = max(0, issued - kSlots); i < issued; ++i)
      mbar_wait(bar_w + 8 * (i % kSlots), (i / kSlots) & 1, nullptr);
  }
  __syncthreads();
  // merge the warps: thread t owns dim t of every head
  const int d = threadIdx.x;
#pragma unroll 1
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wml[(w * G + h) * 2]);
    float O = 0.f, Lsum = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kWarps; ++w) {
        const float mw = wml[(w * G + h) * 2];
        if (mw == -INFINITY) continue;
        const float f = exp2f(mw - M);
        O += f * wo[((size_t)w * G + h) * 128 + d];
        Lsum += f * wml[(w * G + h) * 2 + 1];
      }
    }
    const size_t pb = part_base + (size_t)h * splits;
    part_o[pb * 128 + d] = O;
    if (d == 0) {
      part_ml[pb * 2 + 0] = M;
      part_ml[pb * 2 + 1] = Lsum;
    }
  }
}

__global__ void __launch_bounds__(128)
    k_decode_combine(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                     int splits, int n_q, __nv_bfloat16* __restrict__ out, int ld_out) {
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
cc_status launch_dec(const __nv_bfloat16* q, int ld_q, const __nv_bfloat16* kp,
                     const __nv_bfloat16* vp, int n_pages, const int32_t* pt, int max_pages,
                     const int32_t* n_keys, int batch, int n_kv, int window, int splits,
                     DecodeScratch scr, int* err, cudaStream_t s) {
  using L = DecSmem<G>;
  static bool attr_set = false;
  if (!attr_set) {
    CC_CHECK_CUDA(cudaFuncSetAttribute(k_attn_decode<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(L::kTotal)));
    attr_set = true;
  }
  const float sl2 = (1.0f / sqrtf(128.0f)) * kLog2e;
  dim3 grid(splits, n_kv, batch);
  k_attn_decode<G><<<grid, kWarps * 32, L::kTotal, s>>>(q, ld_q, kp, vp, n_pages, pt, max_pages,
                                                        n_keys, n_kv, window, splits, sl2,
                                                        scr.part_o, scr.part_ml, err);
  CC_CHECK_CUDA(cudaGetLastError());
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
  if (page_size != kPage || n_q % n_kv != 0) return CC_ERR_UNSUPPORTED;
  const int splits = decode_splits(max_pages);
  const int G = n_q / n_kv;
  cc_status st;
  switch (G) {
    case 1: st = launch_dec<1>(q, ld_q, k_pool, v_pool, n_pages, page_table, max_pages, n_keys,
                               batch, n_kv, window, splits, scr, err, s); break;
    case 2: st = launch_dec<2>(q, ld_q, k_pool, v_pool, n_pages, page_table, max_pages, n_keys,
                               batch, n_kv, window, splits, scr, err, s); break;
    case 4: st = launch_dec<4>(q, ld_q, k_pool, v_pool, n_pages, page_table, max_pages, n_keys,
                               batch, n_kv, window, splits, scr, err, s); break;
    case 8: st = launch_dec<8>(q, ld_q, k_pool, v_pool, n_pages, page_table, max_pages, n_keys,
                               batch, n_kv, window, splits, scr, err, s); break;
    default: return CC_ERR_UNSUPPORTED;
  }
  if (st != CC_OK) return st;
  k_decode_combine<<<dim3(n_q, batch), 128, 0, s>>>(scr.part_o, scr.part_ml, splits, n_q, out,
                                                     ld_out);
  CC_CHECK_CUDA(cudaGetLastError());
  return CC_OK;
}

// ------------------------------------------------------------ no-allocation variant
// Fixed split-KV scratch for callers that cannot allocate: 4 Mi floats (16 MiB) per GPU.
// Every split either writes its partial (max, sum, O) or marks itself empty (max = -inf),
// and the combine reads only the splits of the current call, so nothing needs clearing.
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
