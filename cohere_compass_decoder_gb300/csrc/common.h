// Shared constants and host helpers of the cc library (device-independent parts).
#pragma once

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/cc.h"

namespace cc {

// Device error codes written to the sticky error flag (same values as cc_status).
enum : int { CC_DEV_TIMEOUT = CC_ERR_TIMEOUT, CC_DEV_CHECK = CC_ERR_DEVICE_CHECK };

// A bounded inter-warp wait gives up after this many SM clock cycles counted with clock64()
// (about 1.9 s at the GB300's 2.07 GHz maximum clock, 2.7 s at 1.485 GHz; no launch here
// runs for seconds).
constexpr long long kWaitTimeoutCycles = 4000000000ll;
// The test hook's wait (cc_test_stall_next_gemm) gives up after this many cycles.
constexpr long long kTestStallCycles = 100000000ll;

constexpr int kNumSMsFallback = 152;

// ------------------------------------------------------------------ host helpers
#define CC_CHECK_CUDA(expr)                                                        \
  do {                                                                             \
    cudaError_t e_ = (expr);                                                       \
    if (e_ != cudaSuccess) {                                                       \
      cc::last_cuda_error() = e_;                                                  \
      return CC_ERR_CUDA;                                                          \
    }                                                                              \
  } while (0)

#define CC_CHECK_STATUS(expr)                                                      \
  do {                                                                             \
    cc_status s_ = (expr);                                                         \
    if (s_ != CC_OK) return s_;                                                    \
  } while (0)

cudaError_t& last_cuda_error();

// Number of SMs of the current device (cached per process).
int num_sms();

// 2-D bf16 tensor map for TMA: a [rows, cols] row-major matrix with leading dimension
// `ld` elements, boxes of box_cols x box_rows, 128-byte swizzle when box_cols*2 == 128.
// Zero fill out of bounds. Returns false on failure (bad alignment or driver error).
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint64_t ld, uint32_t box_rows, uint32_t box_cols);
// Launches a kernel of the path with programmatic stream serialization: its CTAs may start
// (barrier set-up, tensor-memory allocation) while the previous kernel on the stream
// finishes; every kernel waits (griddepcontrol.wait) before it touches global memory and
// lets its successor launch (griddepcontrol.launch_dependents) as soon as it starts.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raises a kernel's dynamic shared-memory limit to `bytes` on its first launch in the process
// (the library drives one device per process). Safe from several host threads: concurrent
// first launches may both set the attribute, which is idempotent.
template <typename... KArgs>
cudaError_t allow_dynamic_smem(void (*kernel)(KArgs...), size_t bytes, std::atomic<bool>& done) {
  if (done.load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(bytes));
  if (e == cudaSuccess) done.store(true, std::memory_order_release);
  return e;
}

}  // namespace cc
