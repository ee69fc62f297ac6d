// extern "C" entry points of libtern: argument validation, then the
// launchers of the kernel translation units.  The contract of every entry
// point is stated in include/tern.h.
#include <cstdio>

#include "tern_internal.cuh"

namespace tern {
namespace {
constexpr int kMaxDevices = 64;
// Per device: 0 unknown, 1 sm_103, -1 other.  Concurrent first calls store
// the same value.
std::atomic<int> g_dev_ok[kMaxDevices];
}  // namespace

bool device_supported() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return false;
  if (dev < kMaxDevices) {
    const int known = g_dev_ok[dev].load(std::memory_order_acquire);
    if (known != 0) return known > 0;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return false;
  const bool ok = (major == 10 && minor == 3);
  if (dev < kMaxDevices) g_dev_ok[dev].store(ok ? 1 : -1, std::memory_order_release);
  return ok;
}
}  // namespace tern

using namespace tern;

namespace {

tern_status from_cuda(cudaError_t e) { return e == cudaSuccess ? TERN_OK : TERN_ERR_CUDA; }

bool k_ok(int64_t K, int64_t kmax) { return K > 0 && K % kHBlock == 0 && K <= kmax; }

// Workspace of tern_gemv_decode_f32: the GEMV's partial sums (zero between
// calls), then the decode operand formed from xr (fp16 [M][K], records
// [G][48]), each part 256-byte aligned.
size_t align256(size_t b) { return (b + 255) / 256 * 256; }
size_t gemv_f32_xh_offset(int64_t M, int64_t N, int64_t K) {
  return align256(gemv_workspace_bytes(M, N, K));
}
size_t gemv_f32_aux_offset(int64_t M, int64_t N, int64_t K) {
  return gemv_f32_xh_offset(M, N, K) + align256(static_cast<size_t>(M) * K * 2);
}
size_t gemv_f32_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return gemv_f32_aux_offset(M, N, K) + static_cast<size_t>(K / kGroup) * 192;
}
// Workspace of tern_gemm_prefill_int8: the fp16-held xq, the fp16-held
// weight, then the K-split pieces of the GEMM, each part 256-byte aligned.
size_t gemm_int8_w_offset(int64_t M, int64_t N, int64_t K) {
  return align256(static_cast<size_t>(M) * K * 2);
}
size_t gemm_int8_split_offset(int64_t M, int64_t N, int64_t K) {
  return gemm_int8_w_offset(M, N, K) + align256(static_cast<size_t>(N) * K * 2);
}
size_t gemm_int8_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return gemm_int8_split_offset(M, N, K) + gemm_dense_workspace_bytes(M, N, K);
}

}  // namespace

extern "C" {

const char* tern_status_str(int status) {
  switch (status) {
    case TERN_OK: return "TERN_OK";
    case TERN_ERR_INVALID_ARG: return "TERN_ERR_INVALID_ARG";
    case TERN_ERR_SHAPE: return "TERN_ERR_SHAPE";
    case TERN_ERR_ALIGN: return "TERN_ERR_ALIGN";
    case TERN_ERR_UNSUPPORTED: return "TERN_ERR_UNSUPPORTED";
    case TERN_ERR_CUDA: return "TERN_ERR_CUDA";
    case TERN_ERR_WORKSPACE: return "TERN_ERR_WORKSPACE";
    case TERN_ERR_TIMEOUT: return "TERN_ERR_TIMEOUT";
    default: return "TERN_ERR_UNKNOWN";
  }
}

int tern_version(void) { return 100; }

size_t tern_packed_bytes(int64_t N, int64_t K) {
  if (N < 0 || K < 0 || K % kGroup != 0) return 0;
  return gemv_packed_bytes(N, K);
}

size_t tern_workspace_bytes(int op, int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  if (op == TERN_OP_GEMV) return gemv_workspace_bytes(M, N, K);
  if (op == TERN_OP_GEMV_F32) return M <= 16 ? gemv_f32_workspace_bytes(M, N, K) : 0;
  if (op == TERN_OP_GEMM_INT8) return gemm_int8_workspace_bytes(M, N, K);
  if (op == TERN_OP_GEMM_PACKED) return gemm_packed_workspace_bytes(M, N, K);
  if (op == TERN_OP_GEMM) return gemm_dense_workspace_bytes(M, N, K);
  return 0;
}

int tern_host_accessible(const void* host) {
  if (host == nullptr) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (a.type == cudaMemoryTypeHost) return a.devicePointer == host ? 1 : 0;
  if (a.type == cudaMemoryTypeUnregistered) {
    // pageable memory: only where the GPU uses the host's page tables
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrPageableMemoryAccessUsesHostPageTables, dev) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return v ? 1 : 0;
  }
  return 0;
}

int tern_kernel_launches(int op, int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  if (op == TERN_OP_GEMV) return gemv_needs_fixup(M, N, K) ? 2 : 1;
  if (op == TERN_OP_GEMV_F32) return gemv_needs_fixup(M, N, K) ? 3 : 2;
  if (op == TERN_OP_GEMM) return dense_splits(M, N, K) > 1 ? 2 : 1;
  if (op == TERN_OP_GEMM_INT8) return dense_splits(M, N, K) > 1 ? 4 : 3;
  if (op == TERN_OP_GEMM_PACKED) return packed_splits(M, N, K) > 1 ? 2 : 1;
  return 0;
}

tern_status tern_workspace_init(void* ws, size_t bytes, void* stream) {
  if (bytes == 0) return TERN_OK;
  if (ws == nullptr) return TERN_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(ws, 0, bytes, static_cast<cudaStream_t>(stream)));
}

tern_status tern_pack(const int8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
                      uint8_t* packed, int8_t* q, float* rscale, int8_t* w_q, void* stream) {
  if (N < 0 || K < 0) return TERN_ERR_INVALID_ARG;
  if (!k_ok(K, kMaxK)) return TERN_ERR_SHAPE;
  if ((q == nullptr) != (rscale == nullptr)) return TERN_ERR_INVALID_ARG;
  if (w_q != nullptr && q == nullptr) return TERN_ERR_INVALID_ARG;
  if (N == 0) return TERN_OK;
  if (codes == nullptr || scales == nullptr) return TERN_ERR_INVALID_ARG;
  if (packed == nullptr && q == nullptr) return TERN_OK;
  if (!aligned16(codes) || !aligned16(scales) || (packed && !aligned16(packed)) ||
      (q && !aligned16(q)) || (rscale && !aligned16(rscale)) || (w_q && !aligned16(w_q)))
    return TERN_ERR_ALIGN;
  if (N > (int64_t(1) << 30) / (K / 16)) return TERN_ERR_SHAPE;  // keeps int32 row math safe
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(launch_pack(codes, scales, N, K, packed, q, rscale, w_q,
                               static_cast<cudaStream_t>(stream)));
}

tern_status tern_widen_int8(const int8_t* src, int64_t rows, int64_t cols, uint16_t* dst,
                            void* stream) {
  if (rows < 0 || cols < 0) return TERN_ERR_INVALID_ARG;
  if (cols % 16 != 0 || (rows > 0 && cols > (int64_t(1) << 40) / rows)) return TERN_ERR_SHAPE;
  if (rows == 0 || cols == 0) return TERN_OK;
  if (src == nullptr || dst == nullptr) return TERN_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(launch_widen_int8(src, rows * cols, dst, static_cast<cudaStream_t>(stream)));
}

tern_status tern_fwht_quant(const uint16_t* x, int64_t M, int64_t K, const int8_t* sign,
                            int mode, void* out, float* out_scale, void* stream) {
  if (M < 0 || K < 0) return TERN_ERR_INVALID_ARG;
  if (mode != TERN_FWHT_F32 && mode != TERN_FWHT_DECODE && mode != TERN_FWHT_I8 &&
      mode != TERN_FWHT_F16 && mode != TERN_FWHT_I8H)
    return TERN_ERR_INVALID_ARG;
  if (!k_ok(K, (mode == TERN_FWHT_I8 || mode == TERN_FWHT_I8H) ? 32768 : kMaxK))
    return TERN_ERR_SHAPE;
  if (M > (int64_t(1) << 31) / K) return TERN_ERR_SHAPE;
  if (mode == TERN_FWHT_DECODE && M > 16) return TERN_ERR_SHAPE;
  if (M == 0) return TERN_OK;
  if (x == nullptr || out == nullptr) return TERN_ERR_INVALID_ARG;
  if (mode != TERN_FWHT_F32 && out_scale == nullptr) return TERN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || (mode != TERN_FWHT_F32 && !aligned16(out_scale)))
    return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(
      launch_fwht(x, M, K, sign, mode, out, out_scale, static_cast<cudaStream_t>(stream)));
}

tern_status tern_fwht_shard(const uint16_t* x, int64_t M, int64_t Kr, int lead, int trail,
                            const int8_t* sign, float* xr, float* h_lead, float* h_trail,
                            void* stream) {
  if (M < 0 || Kr < 0 || (lead != 0 && lead != 1) || (trail != 0 && trail != 1))
    return TERN_ERR_INVALID_ARG;
  const int64_t whole = Kr - 512 * (lead + trail);
  const int64_t Kp = Kr + 512 * (lead + trail);
  if (whole < 0 || whole % kHBlock != 0 || Kp == 0 || Kp > kMaxK) return TERN_ERR_SHAPE;
  if (M > (int64_t(1) << 31) / Kp) return TERN_ERR_SHAPE;
  if (M == 0) return TERN_OK;
  if (x == nullptr || (whole > 0 && xr == nullptr) || (lead && h_lead == nullptr) ||
      (trail && h_trail == nullptr))
    return TERN_ERR_INVALID_ARG;
  if (!aligned16(x) || (xr && !aligned16(xr)) || (h_lead && !aligned16(h_lead)) ||
      (h_trail && !aligned16(h_trail)))
    return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(launch_fwht_shard(x, M, Kr, lead, trail, sign, xr, h_lead, h_trail,
                                     static_cast<cudaStream_t>(stream)));
}

tern_status tern_fwht_combine(const float* h_first, const float* h_second, int64_t M, int part,
                              float* xr, int64_t Kp, int64_t blk, void* stream) {
  if (M < 0 || Kp < 0 || blk < 0 || (part != 0 && part != 1)) return TERN_ERR_INVALID_ARG;
  if (Kp == 0 || Kp % kHBlock != 0 || Kp > kMaxK || blk >= Kp / kHBlock) return TERN_ERR_SHAPE;
  if (M > (int64_t(1) << 31) / Kp) return TERN_ERR_SHAPE;
  if (M == 0) return TERN_OK;
  if (h_first == nullptr || h_second == nullptr || xr == nullptr) return TERN_ERR_INVALID_ARG;
  if (!aligned16(h_first) || !aligned16(h_second) || !aligned16(xr)) return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(launch_fwht_combine(h_first, h_second, M, part, xr, Kp, blk,
                                       static_cast<cudaStream_t>(stream)));
}

tern_status tern_quant_rotated(const float* xr, int64_t M, int64_t K, int mode, void* out,
                               float* out_scale, void* stream) {
  if (M < 0 || K < 0) return TERN_ERR_INVALID_ARG;
  if (mode != TERN_FWHT_DECODE && mode != TERN_FWHT_I8 && mode != TERN_FWHT_F16 &&
      mode != TERN_FWHT_I8H)
    return TERN_ERR_INVALID_ARG;
  if (!k_ok(K, kMaxK)) return TERN_ERR_SHAPE;
  if (M > (int64_t(1) << 31) / K) return TERN_ERR_SHAPE;
  if (mode == TERN_FWHT_DECODE && M > 16) return TERN_ERR_SHAPE;
  if (M == 0) return TERN_OK;
  if (xr == nullptr || out == nullptr || out_scale == nullptr) return TERN_ERR_INVALID_ARG;
  if (!aligned16(xr) || !aligned16(out) || !aligned16(out_scale)) return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(launch_quant_rotated(xr, M, K, mode, out, out_scale,
                                        static_cast<cudaStream_t>(stream)));
}

tern_status tern_gemv_decode(const uint8_t* packed, const uint16_t* xh, const float* xs,
                             int64_t M, int64_t N, int64_t K, uint16_t* y, void* ws,
                             size_t ws_bytes, void* stream) {
  if (M < 0 || N < 0 || K < 0) return TERN_ERR_INVALID_ARG;
  if (!k_ok(K, kMaxK)) return TERN_ERR_SHAPE;
  if (M > 16) return TERN_ERR_SHAPE;
  if (N > (int64_t(1) << 30) / (K / 16)) return TERN_ERR_SHAPE;
  if (M == 0 || N == 0) return TERN_OK;
  if (packed == nullptr || xh == nullptr || xs == nullptr || y == nullptr)
    return TERN_ERR_INVALID_ARG;
  if (!aligned16(packed) || !aligned16(xh) || !aligned16(xs) || !aligned16(y))
    return TERN_ERR_ALIGN;
  const size_t need = gemv_workspace_bytes(M, N, K);
  if (ws == nullptr || ws_bytes < need) return TERN_ERR_WORKSPACE;
  if (!aligned16(ws)) return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(launch_gemv(packed, xh, xs, M, N, K, y, ws, static_cast<cudaStream_t>(stream)));
}

tern_status tern_gemv_decode_f32(const uint8_t* packed, const float* xr, int64_t M, int64_t N,
                                 int64_t K, uint16_t* y, void* ws, size_t ws_bytes,
                                 void* stream) {
  if (M < 0 || N < 0 || K < 0) return TERN_ERR_INVALID_ARG;
  if (!k_ok(K, kMaxK)) return TERN_ERR_SHAPE;
  if (M > 16) return TERN_ERR_SHAPE;
  if (N > (int64_t(1) << 30) / (K / 16)) return TERN_ERR_SHAPE;
  if (M == 0 || N == 0) return TERN_OK;
  if (packed == nullptr || xr == nullptr || y == nullptr) return TERN_ERR_INVALID_ARG;
  if (!aligned16(packed) || !aligned16(xr) || !aligned16(y)) return TERN_ERR_ALIGN;
  if (ws == nullptr || ws_bytes < gemv_f32_workspace_bytes(M, N, K)) return TERN_ERR_WORKSPACE;
  if (!aligned16(ws)) return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint16_t* xh = reinterpret_cast<uint16_t*>(base + gemv_f32_xh_offset(M, N, K));
  float* aux = reinterpret_cast<float*>(base + gemv_f32_aux_offset(M, N, K));
  const cudaError_t e = launch_quant_rotated(xr, M, K, TERN_FWHT_DECODE, xh, aux, st);
  if (e != cudaSuccess) return TERN_ERR_CUDA;
  return from_cuda(launch_gemv(packed, xh, aux, M, N, K, y, ws, st));
}

tern_status tern_linear_decode(const uint16_t* x, const int8_t* sign, const uint8_t* packed,
                               int64_t M, int64_t N, int64_t K, uint16_t* y, void* ws,
                               size_t ws_bytes, void* stream) {
  if (M < 0 || N < 0 || K < 0) return TERN_ERR_INVALID_ARG;
  if (!k_ok(K, kMaxK)) return TERN_ERR_SHAPE;
  if (M > 16) return TERN_ERR_SHAPE;
  if (N > (int64_t(1) << 30) / (K / 16)) return TERN_ERR_SHAPE;
  if (M == 0 || N == 0) return TERN_OK;
  if (x == nullptr || packed == nullptr || y == nullptr) return TERN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(packed) || !aligned16(y)) return TERN_ERR_ALIGN;
  const size_t need = gemv_workspace_bytes(M, N, K);
  if (ws == nullptr || ws_bytes < need) return TERN_ERR_WORKSPACE;
  if (!aligned16(ws)) return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(
      launch_linear_decode(x, sign, packed, M, N, K, y, ws, static_cast<cudaStream_t>(stream)));
}

namespace {
tern_status gemm_int8_shape(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return TERN_ERR_INVALID_ARG;
  if (!k_ok(K, kMaxK)) return TERN_ERR_SHAPE;
  if (N % 16 != 0) return TERN_ERR_SHAPE;
  if (M > (int64_t(1) << 24) || N > (int64_t(1) << 24)) return TERN_ERR_SHAPE;
  if ((M + 127) / 128 * ((N + 255) / 256) >= (int64_t(1) << 31)) return TERN_ERR_SHAPE;  // tile count
  return TERN_OK;
}
}  // namespace

tern_status tern_gemm_prefill_int8h(const uint16_t* xq, const float* tscale, const uint16_t* w_q,
                                    const float* rscale, int64_t M, int64_t N, int64_t K,
                                    uint16_t* y, int32_t* acc, void* ws, size_t ws_bytes,
                                    void* stream) {
  const tern_status sh = gemm_int8_shape(M, N, K);
  if (sh != TERN_OK) return sh;
  if (M == 0 || N == 0) return TERN_OK;
  if (xq == nullptr || tscale == nullptr || w_q == nullptr || rscale == nullptr || y == nullptr)
    return TERN_ERR_INVALID_ARG;
  if (!aligned16(xq) || !aligned16(tscale) || !aligned16(w_q) || !aligned16(rscale) ||
      !aligned16(y) || (acc && !aligned16(acc)) || (ws && !aligned16(ws)))
    return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(launch_gemm(xq, tscale, w_q, rscale, M, N, K, y, acc, ws, ws_bytes,
                               static_cast<cudaStream_t>(stream)));
}

tern_status tern_gemm_prefill_int8(const int8_t* xq, const float* tscale, const int8_t* w_int8,
                                   const float* rscale, int64_t M, int64_t N, int64_t K,
                                   uint16_t* y, int32_t* acc, void* ws, size_t ws_bytes,
                                   void* stream) {
  const tern_status sh = gemm_int8_shape(M, N, K);
  if (sh != TERN_OK) return sh;
  if (M == 0 || N == 0) return TERN_OK;
  if (xq == nullptr || tscale == nullptr || w_int8 == nullptr || rscale == nullptr ||
      y == nullptr)
    return TERN_ERR_INVALID_ARG;
  if (!aligned16(xq) || !aligned16(tscale) || !aligned16(w_int8) || !aligned16(rscale) ||
      !aligned16(y) || (acc && !aligned16(acc)))
    return TERN_ERR_ALIGN;
  if (ws == nullptr || ws_bytes < gemm_int8_workspace_bytes(M, N, K)) return TERN_ERR_WORKSPACE;
  if (!aligned16(ws)) return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint16_t* xh = reinterpret_cast<uint16_t*>(base);
  uint16_t* wh = reinterpret_cast<uint16_t*>(base + gemm_int8_w_offset(M, N, K));
  const size_t split_off = gemm_int8_split_offset(M, N, K);
  cudaError_t e = launch_widen_int8(xq, M * K, xh, st);
  if (e == cudaSuccess) e = launch_widen_int8(w_int8, N * K, wh, st);
  if (e != cudaSuccess) return TERN_ERR_CUDA;
  return from_cuda(launch_gemm(xh, tscale, wh, rscale, M, N, K, y, acc, base + split_off,
                               ws_bytes - split_off, st));
}

tern_status tern_gemm_prefill_packed(const uint16_t* xq, const float* tscale,
                                     const uint8_t* packed, const int8_t* q, const float* rscale,
                                     int64_t M, int64_t N, int64_t K, uint16_t* y, int32_t* acc,
                                     void* ws, size_t ws_bytes, void* stream) {
  if (M < 0 || N < 0 || K < 0) return TERN_ERR_INVALID_ARG;
  if (!k_ok(K, kMaxK)) return TERN_ERR_SHAPE;
  if (M > (int64_t(1) << 24) || N > (int64_t(1) << 24)) return TERN_ERR_SHAPE;
  if (N % 16 != 0) return TERN_ERR_SHAPE;
  if ((M + 127) / 128 * ((N + 255) / 256) >= (int64_t(1) << 31)) return TERN_ERR_SHAPE;  // tile count
  if (M == 0 || N == 0) return TERN_OK;
  if (xq == nullptr || tscale == nullptr || packed == nullptr || q == nullptr ||
      rscale == nullptr || y == nullptr)
    return TERN_ERR_INVALID_ARG;
  if (!aligned16(xq) || !aligned16(tscale) || !aligned16(packed) || !aligned16(q) ||
      !aligned16(rscale) || !aligned16(y) || (acc && !aligned16(acc)))
    return TERN_ERR_ALIGN;
  if (gemm_packed_workspace_bytes(M, N, K) > 0 &&
      (ws == nullptr || ws_bytes < gemm_packed_workspace_bytes(M, N, K)))
    return TERN_ERR_WORKSPACE;
  if (ws != nullptr && !aligned16(ws)) return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(launch_gemm_packed(xq, tscale, packed, q, rscale, M, N, K, y, acc, ws,
                                      static_cast<cudaStream_t>(stream)));
}

tern_status tern_expand_fp16(const int8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
                             uint16_t* w_h, void* stream) {
  if (N < 0 || K < 0) return TERN_ERR_INVALID_ARG;
  if (!k_ok(K, kMaxK)) return TERN_ERR_SHAPE;
  if (N > (int64_t(1) << 34) / K) return TERN_ERR_SHAPE;
  if (N == 0) return TERN_OK;
  if (codes == nullptr || scales == nullptr || w_h == nullptr) return TERN_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(w_h)) return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(launch_expand_fp16(codes, scales, N, K, w_h, static_cast<cudaStream_t>(stream)));
}

tern_status tern_gemm_prefill_fp16(const uint16_t* xh, const float* xs, const uint16_t* w_h,
                                   int64_t M, int64_t N, int64_t K, uint16_t* y, void* ws,
                                   size_t ws_bytes, void* stream) {
  if (M < 0 || N < 0 || K < 0) return TERN_ERR_INVALID_ARG;
  if (!k_ok(K, kMaxK)) return TERN_ERR_SHAPE;
  if (N % 16 != 0) return TERN_ERR_SHAPE;
  if (M > (int64_t(1) << 24) || N > (int64_t(1) << 24)) return TERN_ERR_SHAPE;
  if ((M + 127) / 128 * ((N + 255) / 256) >= (int64_t(1) << 31)) return TERN_ERR_SHAPE;
  if (M == 0 || N == 0) return TERN_OK;
  if (xh == nullptr || xs == nullptr || w_h == nullptr || y == nullptr) return TERN_ERR_INVALID_ARG;
  if (!aligned16(xh) || !aligned16(xs) || !aligned16(w_h) || !aligned16(y) ||
      (ws && !aligned16(ws)))
    return TERN_ERR_ALIGN;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(launch_gemm_f16(xh, xs, w_h, M, N, K, y, ws, ws_bytes,
                                   static_cast<cudaStream_t>(stream)));
}

tern_status tern_selftest_wait(uint32_t polls, void* stream) {
  if (polls == 0 || polls > TERN_SELFTEST_MAX_POLLS) return TERN_ERR_INVALID_ARG;
  if (!device_supported()) return TERN_ERR_UNSUPPORTED;
  return from_cuda(launch_wait_selftest(polls, static_cast<cudaStream_t>(stream)));
}

tern_status tern_check(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return TERN_ERR_CUDA;
  unsigned int err_gemm = 0, err_gemv = 0;
  if (gemm_read_clear_error(&err_gemm) != cudaSuccess) return TERN_ERR_CUDA;
  if (gemv_read_clear_error(&err_gemv) != cudaSuccess) return TERN_ERR_CUDA;
  return (err_gemm | err_gemv) ? TERN_ERR_TIMEOUT : TERN_OK;
}

}  // extern "C"
