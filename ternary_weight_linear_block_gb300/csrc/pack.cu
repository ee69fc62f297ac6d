// Load-time weight conversion: packing of the 2-bit codes and their group
// scales into the decode GEMV's units, and the scale decomposition of the
// int8 path.
//
// Page "RTX 5070 x2 ... Ternary-Bonsai-2-27B on vLLM TP=2": section "前提"
// (codes in {-1,0,+1} at 2 bits, one scale per 128 elements of a row) and
// section 4 (q[n,g] = round(127 s[n,g] / smax[n]); W_int8[n,k] =
// code[n,k] q[n,k/128] fits int8 exactly).  Expanding the weights to int8
// once here, instead of on every prefill step, removes the run-time weight
// expansion that section 6 measures at 31 of 83 ms of ternary-linear time;
// widen_kernel holds int8 values in fp16 for the tensor cores' f16 kind.
// The packed unit format is defined in include/tern.h.
#include <cuda_fp16.h>

#include "tern_internal.cuh"

namespace tern {
namespace {

// The 2-bit field of a code: u = code + 1 (-1 -> 0, 0 -> 1, +1 -> 2).
__device__ __forceinline__ uint32_t field_of(int8_t c) {
  return static_cast<uint32_t>(static_cast<int>(c) + 1) & 3u;
}

constexpr int kUnitRows = 512;
constexpr int kUnitWords = 4352;       // 17408-byte unit: 4096 code words + 256 scale words

// One thread per 32-bit word of the packed units (codes and scales).
// The decode kernels (tern_gemv_decode, tern_linear_decode) start streaming
// the packed units before their programmatic launch wait, so a kernel that
// runs at the same time as them must not write the units.  This kernel
// therefore lets no later kernel start early (the stream's next kernel
// launches when this one has finished) and makes its stores visible to the
// whole GPU before its threads exit.
__global__ void pack_units_kernel(const int8_t* __restrict__ codes,
                                  const uint16_t* __restrict__ scales, int N, int K,
                                  uint32_t* __restrict__ packed, long n_words) {
  pdl_wait();
  const int G = K / kGroup;
  for (long wi = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; wi < n_words;
       wi += static_cast<long>(gridDim.x) * blockDim.x) {
    const long unit = wi / kUnitWords;
    const int w = static_cast<int>(wi % kUnitWords);
    const long rb = unit / G;
    const int g = static_cast<int>(unit % G);
    uint32_t out = 0;
    if (w < 4096) {
      // tile t, slot L = 4 r + c, word p (register p of the tile's A fragment)
      const int t = w >> 7, lane = (w >> 2) & 31, p = w & 3;
      const int r = lane >> 2, c = lane & 3;
      const long row = rb * kUnitRows + 16 * t + r + 8 * (p & 1);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        // field j: k16 step j; rows past N hold zero codes (u = 1)
        const int k = kGroup * g + 16 * j + 2 * c + 8 * (p >> 1);
        const uint32_t u0 = row < N ? field_of(codes[row * K + k]) : 1u;
        const uint32_t u1 = row < N ? field_of(codes[row * K + k + 1]) : 1u;
        out |= (u0 << (2 * j)) | (u1 << (16 + 2 * j));
      }
    } else {
      const int j = w - 4096;          // tile t = j / 8, pair gq = j % 8
      const int t = j >> 3, gq = j & 7;
      const long r0 = rb * kUnitRows + 16 * t + gq, r1 = r0 + 8;
      const uint32_t lo = r0 < N ? scales[r0 * G + g] : 0u;
      const uint32_t hi = r1 < N ? scales[r1 * G + g] : 0u;
      out = lo | (hi << 16);
    }
    packed[wi] = out;
  }
  __threadfence();
}

// One warp per row: smax, q, rscale.
__global__ void scale_decomp_kernel(const uint16_t* __restrict__ scales, int N, int G,
                                    int8_t* __restrict__ q, float* __restrict__ rscale) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long row = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= N) return;
  const __half* s = reinterpret_cast<const __half*>(scales) + row * G;
  float smax = 0.f;
  for (int g = lane; g < G; g += 32) smax = fmaxf(smax, fabsf(__half2float(s[g])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
  for (int g = lane; g < G; g += 32) {
    float v = 0.f;
    if (smax > 0.f) v = rintf(__fdiv_rn(__fmul_rn(127.0f, __half2float(s[g])), smax));
    q[row * G + g] = static_cast<int8_t>(static_cast<int>(v));
  }
  if (lane == 0) rscale[row] = smax > 0.f ? __fdiv_rn(smax, 127.0f) : 0.f;
}

// One thread per 8 consecutive elements of a row: W_int8 = code * q, exact in
// int8 (|code q| <= 127).
__global__ void w8_kernel(const int8_t* __restrict__ codes, const int8_t* __restrict__ q, int N,
                          int K, int8_t* __restrict__ w8, long n_vec) {
  pdl_wait();
  pdl_launch_dependents();
  const int G = K / kGroup;
  for (long vi = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; vi < n_vec;
       vi += static_cast<long>(gridDim.x) * blockDim.x) {
    const long e0 = vi * 8;
    const long row = e0 / K;
    const int k = static_cast<int>(e0 % K);
    const int qq = q[row * G + k / kGroup];
    const uint2 cw = *reinterpret_cast<const uint2*>(codes + e0);
    const int8_t* cb = reinterpret_cast<const int8_t*>(&cw);
    int8_t v[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) v[t] = static_cast<int8_t>(cb[t] * qq);
    *reinterpret_cast<uint2*>(w8 + e0) = *reinterpret_cast<const uint2*>(v);
  }
}

// One thread per 8 consecutive int8 values: the same integers held in fp16
// (exact), the operand format of the tensor-core GEMM.
__global__ void widen_kernel(const int8_t* __restrict__ src, __half* __restrict__ dst, long n_vec) {
  pdl_wait();
  pdl_launch_dependents();
  for (long vi = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; vi < n_vec;
       vi += static_cast<long>(gridDim.x) * blockDim.x) {
    const uint2 cw = *reinterpret_cast<const uint2*>(src + vi * 8);
    const int8_t* cb = reinterpret_cast<const int8_t*>(&cw);
    uint32_t w[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      __half2 h = __floats2half2_rn(static_cast<float>(cb[2 * t]), static_cast<float>(cb[2 * t + 1]));
      w[t] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(dst + vi * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// One thread per 8 consecutive elements of a row: w_h = code * s, the fp16
// weight of the fp16 prefill path (exact: a code is -1, 0 or +1).
__global__ void wh_kernel(const int8_t* __restrict__ codes, const __half* __restrict__ scales,
                          int N, int K, __half* __restrict__ wh, long n_vec) {
  pdl_wait();
  pdl_launch_dependents();
  const int G = K / kGroup;
  for (long vi = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; vi < n_vec;
       vi += static_cast<long>(gridDim.x) * blockDim.x) {
    const long e0 = vi * 8;
    const long row = e0 / K;
    const int k = static_cast<int>(e0 % K);
    const __half sc = scales[row * G + k / kGroup];
    const __half nsc = __hneg(sc);
    const uint2 cw = *reinterpret_cast<const uint2*>(codes + e0);
    const int8_t* cb = reinterpret_cast<const int8_t*>(&cw);
    __half v[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) v[t] = cb[t] > 0 ? sc : (cb[t] < 0 ? nsc : __float2half_rn(0.f));
    *reinterpret_cast<uint4*>(wh + e0) = *reinterpret_cast<const uint4*>(v);
  }
}

unsigned grid_for(long items, int threads) {
  long b = (items + threads - 1) / threads;
  if (b > 152L * 32) b = 152L * 32;
  return static_cast<unsigned>(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_expand_fp16(const int8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
                               uint16_t* w_h, cudaStream_t st) {
  const long n_vec = N * K / 8;
  return launch(wh_kernel, dim3(grid_for(n_vec, 256)), dim3(256), 0, st, codes,
                reinterpret_cast<const __half*>(scales), static_cast<int>(N), static_cast<int>(K),
                reinterpret_cast<__half*>(w_h), n_vec);
}

cudaError_t launch_widen_int8(const int8_t* src, int64_t count, uint16_t* dst, cudaStream_t st) {
  const long n_vec = count / 8;
  return launch(widen_kernel, dim3(grid_for(n_vec, 256)), dim3(256), 0, st, src,
                reinterpret_cast<__half*>(dst), n_vec);
}

cudaError_t launch_pack(const int8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
                        uint8_t* packed, int8_t* q, float* rscale, int8_t* w_int8,
                        cudaStream_t st) {
  const int n = static_cast<int>(N), k = static_cast<int>(K), G = static_cast<int>(K / kGroup);
  cudaError_t e = cudaSuccess;
  if (packed != nullptr) {
    const long n_words = (N + kUnitRows - 1) / kUnitRows * G * kUnitWords;
    e = launch(pack_units_kernel, dim3(grid_for(n_words, 256)), dim3(256), 0, st, codes, scales, n,
               k, reinterpret_cast<uint32_t*>(packed), n_words);
    if (e != cudaSuccess) return e;
  }
  if (q != nullptr) {
    e = launch(scale_decomp_kernel, dim3(static_cast<unsigned>((N + 7) / 8)), dim3(256), 0, st,
               scales, n, G, q, rscale);
    if (e != cudaSuccess) return e;
    if (w_int8 != nullptr) {
      const long n_vec = N * K / 8;
      e = launch(w8_kernel, dim3(grid_for(n_vec, 256)), dim3(256), 0, st, codes,
                 static_cast<const int8_t*>(q), n, k, w_int8, n_vec);
    }
  }
  return e;
}

}  // namespace tern
