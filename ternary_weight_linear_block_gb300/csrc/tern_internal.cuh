// Internal helpers shared by the kernels of libtern (device side and launch side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/tern.h"

namespace tern {

constexpr int kHBlock = 1024;   // Hadamard block width
constexpr int kGroup = 128;     // elements per scale group
constexpr int kMaxK = 65536;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t pad16(int64_t n) { return (n + 15) / 16 * 16; }

// Whether the calling thread's current device is an sm_103 GPU (cached per
// device).
bool device_supported();

// Per-device set-up (a kernel's shared-memory limit is an attribute of the
// kernel on the current device): runs set_up() until it first succeeds on
// the calling thread's current device, one bit of `done` per device (0-63).
// Concurrent first calls may both run it, so set_up must be idempotent.
template <class F>
cudaError_t once_per_device(std::atomic<unsigned long long>& done, F&& set_up) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const unsigned long long bit = 1ull << dev;
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = set_up();
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Programmatic dependent launch: every kernel waits for its predecessor
// grid before touching data a previous kernel may have written, and lets its
// successor launch early so the successor's independent prologue overlaps.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                   Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same in clusters of `cx` CTAs along x (grid.x a multiple of cx).
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t st, unsigned cx, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cx;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// How many clusters of `cx` CTAs of this kernel fit on the device at once
// (0 if the query fails).
template <typename... KArgs>
int max_active_clusters(void (*kernel)(KArgs...), dim3 block, size_t smem, unsigned cx) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cx);
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cx;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kernel), &cfg) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// Launchers (one per translation unit); they assume validated arguments.
cudaError_t launch_fwht(const uint16_t* x, int64_t M, int64_t K, const int8_t* sign, int mode,
                        void* out, float* out_scale, cudaStream_t st);
cudaError_t launch_fwht_shard(const uint16_t* x, int64_t M, int64_t Kr, int lead, int trail,
                              const int8_t* sign, float* xr, float* h_lead, float* h_trail,
                              cudaStream_t st);
cudaError_t launch_fwht_combine(const float* h_first, const float* h_second, int64_t M, int part,
                                float* xr, int64_t Kp, int64_t blk, cudaStream_t st);
cudaError_t launch_quant_rotated(const float* xr, int64_t M, int64_t K, int mode, void* out,
                                 float* out_scale, cudaStream_t st);
cudaError_t launch_pack(const int8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
                        uint8_t* packed, int8_t* q, float* rscale, int8_t* w_int8,
                        cudaStream_t st);
cudaError_t launch_widen_int8(const int8_t* src, int64_t count, uint16_t* dst, cudaStream_t st);
size_t gemv_packed_bytes(int64_t N, int64_t K);
size_t gemv_workspace_bytes(int64_t M, int64_t N, int64_t K);
bool gemv_needs_fixup(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemv(const uint8_t* packed, const uint16_t* xh, const float* xs, int64_t M,
                        int64_t N, int64_t K, uint16_t* y, void* ws, cudaStream_t st);
cudaError_t launch_linear_decode(const uint16_t* x, const int8_t* sign, const uint8_t* packed,
                                 int64_t M, int64_t N, int64_t K, uint16_t* y, void* ws,
                                 cudaStream_t st);
struct DensePlan {
  int S;      // slices per split tile (1: nothing split)
  int full;   // tiles computed whole, before the split ones
};
DensePlan dense_plan(int64_t M, int64_t N, int64_t K);
int dense_splits(int64_t M, int64_t N, int64_t K);
size_t gemm_dense_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm(const uint16_t* xq, const float* tscale, const uint16_t* w_q,
                        const float* rscale, int64_t M, int64_t N, int64_t K, uint16_t* y,
                        int32_t* acc, void* ws, size_t ws_bytes, cudaStream_t st);
cudaError_t launch_gemm_f16(const uint16_t* xh, const float* xs, const uint16_t* w_h, int64_t M,
                            int64_t N, int64_t K, uint16_t* y, void* ws, size_t ws_bytes,
                            cudaStream_t st);
cudaError_t launch_expand_fp16(const int8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
                               uint16_t* w_h, cudaStream_t st);
size_t gemm_packed_workspace_bytes(int64_t M, int64_t N, int64_t K);
int packed_splits(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_packed(const uint16_t* xq, const float* tscale, const uint8_t* packed,
                               const int8_t* q, const float* rscale, int64_t M, int64_t N,
                               int64_t K, uint16_t* y, int32_t* acc, void* ws, cudaStream_t st);
// Read and clear the device error word of the GEMV / GEMM translation unit.
cudaError_t gemv_read_clear_error(unsigned int* err);
cudaError_t gemm_read_clear_error(unsigned int* err);
cudaError_t launch_wait_selftest(uint32_t polls, cudaStream_t st);

}  // namespace tern
