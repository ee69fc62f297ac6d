// Block Hadamard rotation of the activations and its three output forms.
//
// Page "RTX 5070 x2 ... Ternary-Bonsai-2-27B on vLLM TP=2": section "前提"
// (block-wise Hadamard rotation on the input side) and section 1 (Sylvester
// structure, split identity H1024[a;b] = [H512 a + H512 b ; H512 a - H512 b]
// as the last butterfly stage); section 4 (per-token int8 quantisation after
// the rotation).  The butterfly routines and the decode operand's scaling are
// in fwht_dev.cuh.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fwht_dev.cuh"
#include "tern_internal.cuh"

namespace tern {
namespace {

using namespace fwht;

// Modes F32 and DECODE: one warp per (token, block).
template <int MODE>
__global__ void __launch_bounds__(128) fwht_block_kernel(const uint16_t* __restrict__ x, int M,
                                                         int K, const int8_t* __restrict__ sign,
                                                         void* __restrict__ out,
                                                         float* __restrict__ out_scale) {
  const int lane = threadIdx.x & 31;
  const int B = K / kHBlock;
  const long wid = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  pdl_launch_dependents();
  pdl_wait();
  if (wid >= static_cast<long>(M) * B) return;
  const int m = static_cast<int>(wid / B);
  const int b = static_cast<int>(wid % B);
  float v[4][8];
  load_block(x + static_cast<long>(m) * K + static_cast<long>(b) * kHBlock,
             sign ? sign + static_cast<long>(b) * kHBlock : nullptr, lane, v);
  fwht_1024(v, lane);
  if (MODE == TERN_FWHT_F32) {
    float* o = static_cast<float*>(out) + static_cast<long>(m) * K + static_cast<long>(b) * kHBlock;
#pragma unroll
    for (int ih = 0; ih < 4; ++ih) {
      float4* p = reinterpret_cast<float4*>(o + ih * 256 + lane * 8);
      p[0] = make_float4(v[ih][0], v[ih][1], v[ih][2], v[ih][3]);
      p[1] = make_float4(v[ih][4], v[ih][5], v[ih][6], v[ih][7]);
    }
  } else {
    float f, finv;
    decode_factor(v, f, finv);
    __half* o = static_cast<__half*>(out) + static_cast<long>(m) * K + static_cast<long>(b) * kHBlock;
#pragma unroll
    for (int ih = 0; ih < 4; ++ih)
      *reinterpret_cast<uint4*>(o + ih * 256 + lane * 8) = decode_pack8(v, ih, f);
    if (lane == 0) out_scale[static_cast<long>(m) * B + b] = finv;
  }
}

// Mode I8: one CTA (8 warps) per token; the rotated token is kept in shared
// memory until its absmax is known.
__global__ void __launch_bounds__(256) fwht_i8_kernel(const uint16_t* __restrict__ x, int M, int K,
                                                      const int8_t* __restrict__ sign,
                                                      __half* __restrict__ xq,
                                                      float* __restrict__ tscale) {
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);
  __shared__ float red[8];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int m = blockIdx.x;
  const int B = K / kHBlock;
  pdl_launch_dependents();
  pdl_wait();
  const uint16_t* xm = x + static_cast<long>(m) * K;
  float amax = 0.f;
  for (int b = warp; b < B; b += 8) {
    float v[4][8];
    load_block(xm + static_cast<long>(b) * kHBlock, sign ? sign + static_cast<long>(b) * kHBlock : nullptr,
               lane, v);
    fwht_1024(v, lane);
#pragma unroll
    for (int ih = 0; ih < 4; ++ih) {
      float4* p = reinterpret_cast<float4*>(xs + b * kHBlock + ih * 256 + lane * 8);
      p[0] = make_float4(v[ih][0], v[ih][1], v[ih][2], v[ih][3]);
      p[1] = make_float4(v[ih][4], v[ih][5], v[ih][6], v[ih][7]);
#pragma unroll
      for (int il = 0; il < 8; ++il) amax = fmaxf(amax, fabsf(v[ih][il]));
    }
  }
  amax = warp_max(amax);
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  float a = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) a = fmaxf(a, red[w]);
  const float ts = __fdiv_rn(a, 127.0f);
  const bool nz = ts > 0.f;
  if (threadIdx.x == 0) tscale[m] = nz ? ts : 0.f;
  __half* om = xq + static_cast<long>(m) * K;
  for (int i = threadIdx.x * 8; i < K; i += 256 * 8) {
    const float4 p0 = reinterpret_cast<const float4*>(xs + i)[0];
    const float4 p1 = reinterpret_cast<const float4*>(xs + i)[1];
    float vv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    uint32_t w[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      float q0 = 0.f, q1 = 0.f;
      if (nz) {
        q0 = fminf(fmaxf(rintf(__fdiv_rn(vv[2 * t], ts)), -127.f), 127.f);
        q1 = fminf(fmaxf(rintf(__fdiv_rn(vv[2 * t + 1], ts)), -127.f), 127.f);
      }
      __half2 h2 = __floats2half2_rn(q0, q1);   // integers in [-127,127]: exact
      w[t] = *reinterpret_cast<uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(om + i) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_fwht(const uint16_t* x, int64_t M, int64_t K, const int8_t* sign, int mode,
                        void* out, float* out_scale, cudaStream_t st) {
  const int m = static_cast<int>(M), k = static_cast<int>(K);
  if (mode == TERN_FWHT_I8) {
    const size_t smem = static_cast<size_t>(K) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(fwht_i8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch(fwht_i8_kernel, dim3(m), dim3(256), smem, st, x, m, k, sign,
                  static_cast<__half*>(out), out_scale);
  }
  const long warps = M * (K / kHBlock);
  const dim3 grid(static_cast<unsigned>((warps + 3) / 4));
  if (mode == TERN_FWHT_F32)
    return launch(fwht_block_kernel<TERN_FWHT_F32>, grid, dim3(128), 0, st, x, m, k, sign, out,
                  out_scale);
  return launch(fwht_block_kernel<TERN_FWHT_DECODE>, grid, dim3(128), 0, st, x, m, k, sign, out,
                out_scale);
}

}  // namespace tern
