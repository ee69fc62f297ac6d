// tern_gemv_decode_noalloc: the decode GEMV with its scratch memory in a
// fixed, file-scope device array instead of a caller-provided workspace.
//
// Who needs it: an application that embeds this layer and owns all of its
// device memory through its own pool (and hands the layer only its input and
// output buffers) cannot let the library take a separate workspace, and a
// decode loop that must never stall cannot call cudaMalloc, which may
// synchronise the whole device.  This entry point allocates nothing: the
// GEMV's partial sums (row blocks shared by several CTAs) live in
// g_noalloc_scratch, a static device array of TERN_NOALLOC_SCRATCH_BYTES that
// every GPU loading the library keeps until the process exits.
//
// The first call on a device (with that device current) looks up the array's
// device address with cudaGetSymbolAddress and caches it per device; that
// first call should come before any stream capture.  Every later call made
// outside a stream capture looks the address up again and refreshes the
// cache, so a device reset (which reloads the module at a new address) is
// picked up by the next uncaptured call; a call inside a capture uses the
// cached address.  All calls share the one
// array and it keeps the last call's contents, so each call zero-fills the
// part it uses on its stream before the kernel (a call that gave up waiting
// may have left published words set); calls that overlap on the GPU (for example
// on two streams) race on the array.
#include "tern_internal.cuh"

namespace tern {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TERN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
// Per device: the device address of g_noalloc_scratch.  Concurrent first
// calls store the same value.
std::atomic<void*> g_scratch_addr[kMaxDevices];

cudaError_t scratch_address(int dev, cudaStream_t st, void** out) {
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    (void)cudaGetLastError();          // e.g. the legacy stream during a global capture
    cs = cudaStreamCaptureStatusActive;
  }
  if (p == nullptr || cs == cudaStreamCaptureStatusNone) {
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace tern

extern "C" tern_status tern_gemv_decode_noalloc(const uint8_t* packed, const uint16_t* xh,
                                                const float* xs, int64_t M, int64_t N, int64_t K,
                                                uint16_t* y, void* stream) {
  using namespace tern;
  if (M < 0 || N < 0 || K < 0) return TERN_ERR_INVALID_ARG;
  if (K == 0 || K % kHBlock != 0 || K > kMaxK || M > 16) return TERN_ERR_SHAPE;
  if (N > (int64_t(1) << 30) / (K / 16)) return TERN_ERR_SHAPE;
  if (M == 0 || N == 0) return TERN_OK;
  if (packed == nullptr || xh == nullptr || xs == nullptr || y == nullptr)
    return TERN_ERR_INVALID_ARG;
  if (!aligned16(packed) || !aligned16(xh) || !aligned16(xs) || !aligned16(y))
    return TERN_ERR_ALIGN;
  if (gemv_workspace_bytes(M, N, K) > TERN_NOALLOC_SCRATCH_BYTES) return TERN_ERR_WORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices || !device_supported())
    return TERN_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  if (scratch_address(dev, st, &scratch) != cudaSuccess) return TERN_ERR_CUDA;
  if (cudaMemsetAsync(scratch, 0, gemv_workspace_bytes(M, N, K), st) != cudaSuccess)
    return TERN_ERR_CUDA;
  return launch_gemv(packed, xh, xs, M, N, K, y, scratch, st) == cudaSuccess ? TERN_OK
                                                                           : TERN_ERR_CUDA;
}
