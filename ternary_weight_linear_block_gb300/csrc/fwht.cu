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

// Modes F32, F16 and DECODE: one warp per (token, block).
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
  } else if (MODE == TERN_FWHT_F16) {
    float f, finv;
    f16_factor(v, f, finv);
    __half* o = static_cast<__half*>(out) + static_cast<long>(m) * K + static_cast<long>(b) * kHBlock;
#pragma unroll
    for (int ih = 0; ih < 4; ++ih)
      *reinterpret_cast<uint4*>(o + ih * 256 + lane * 8) = f16_pack8(v, ih, f);
    if (lane == 0) out_scale[static_cast<long>(m) * B + b] = finv;
  } else {
    decode_store(v, lane, m, b, M, K, static_cast<__half*>(out), out_scale);
  }
}

// Mode I8 (K <= 32768): one CTA per token with one warp per 1024-block.
// Each warp keeps its rotated block in registers while the CTA reduces the
// token's absmax, then quantises and writes its own block: no shared-memory
// copy of the token, and every warp loads at once.  Launch bounds: up to 18
// blocks (K <= 18432) two CTAs per SM (registers capped at 56), else one.
// The quantised values of 8 consecutive elements: int8 (TERN_FWHT_I8), or the
// same integers held in fp16 (TERN_FWHT_I8H, the tensor cores' operand).
__device__ __forceinline__ void store_q8(int8_t* p, const float (&q)[8]) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int t = 0; t < 8; ++t)
    w[t >> 2] |= (static_cast<uint32_t>(static_cast<int>(q[t])) & 0xffu) << (8 * (t & 3));
  *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
}
__device__ __forceinline__ void store_q8(__half* p, const float (&q)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    __half2 h2 = __floats2half2_rn(q[2 * t], q[2 * t + 1]);   // integers in [-127,127]: exact
    w[t] = *reinterpret_cast<uint32_t*>(&h2);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store_q4(int8_t* p, const float (&q)[4]) {
  uint32_t w = 0u;
#pragma unroll
  for (int t = 0; t < 4; ++t) w |= (static_cast<uint32_t>(static_cast<int>(q[t])) & 0xffu) << (8 * t);
  *reinterpret_cast<uint32_t*>(p) = w;
}
__device__ __forceinline__ void store_q4(__half* p, const float (&q)[4]) {
  __half2 a = __floats2half2_rn(q[0], q[1]), b = __floats2half2_rn(q[2], q[3]);
  *reinterpret_cast<uint2*>(p) =
      make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
}

template <int MAX_THREADS, int MIN_CTAS, typename OutT>
__global__ void __launch_bounds__(MAX_THREADS, MIN_CTAS)
    fwht_i8_reg_kernel(const uint16_t* __restrict__ x, int M, int K,
                       const int8_t* __restrict__ sign, OutT* __restrict__ xq,
                       float* __restrict__ tscale) {
  __shared__ float red[32];
  const int lane = threadIdx.x & 31;
  const int b = threadIdx.x >> 5;   // the warp's block
  const int nb = blockDim.x >> 5;   // = K / 1024
  const int m = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  float v[4][8];
  load_block(x + static_cast<long>(m) * K + static_cast<long>(b) * kHBlock,
             sign ? sign + static_cast<long>(b) * kHBlock : nullptr, lane, v);
  fwht_1024(v, lane);
  float amax = 0.f;
#pragma unroll
  for (int ih = 0; ih < 4; ++ih)
#pragma unroll
    for (int il = 0; il < 8; ++il) amax = fmaxf(amax, fabsf(v[ih][il]));
  amax = warp_max(amax);
  if (lane == 0) red[b] = amax;
  __syncthreads();
  float a = red[0];
  for (int w = 1; w < nb; ++w) a = fmaxf(a, red[w]);
  const float ts = __fdiv_rn(a, 127.0f);
  const bool nz = ts > 0.f;
  if (threadIdx.x == 0) tscale[m] = nz ? ts : 0.f;
  OutT* ob = xq + static_cast<long>(m) * K + static_cast<long>(b) * kHBlock;
  // The code of an element is rint(v / ts) with the quotient correctly
  // rounded.  The product p = v * (1 / ts), each factor rounded once, lies
  // within |v / ts| * 2^-23 <= 127.5 * 2^-23 < 2^-16 of the exact quotient
  // (|v| <= a = 127 ts up to rounding), and the rounded quotient within
  // 2^-18 of it.  So where p is farther than 2^-15 from every half-integer,
  // rint(p) is the code; a chunk where some lane's element comes nearer
  // (a tie or next to one) takes the division.  A token whose reciprocal
  // scale overflows (subnormal ts) takes the division everywhere.
  const float r = __fdiv_rn(1.0f, ts);
  const bool fast = nz && r <= 3.0e38f;
#pragma unroll
  for (int ih = 0; ih < 4; ++ih) {
    float qv[8];
    bool near = !fast;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const float pv = __fmul_rn(v[ih][t], r);
      qv[t] = rintf(pv);
      near = near || __fsub_rn(0.5f, fabsf(__fsub_rn(pv, qv[t]))) < 0x1p-15f;
    }
    if (__any_sync(0xffffffffu, near)) {
#pragma unroll
      for (int t = 0; t < 8; ++t) qv[t] = nz ? rintf(__fdiv_rn(v[ih][t], ts)) : 0.f;
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) qv[t] = fminf(fmaxf(qv[t], -127.f), 127.f);
    store_q8(ob + ih * 256 + lane * 8, qv);
  }
}

// ---------------------------------------------------------------------------
// K-split tensor parallelism (page section 1): a rank's shard of the input
// columns may start and/or end in the middle of a 1024-block.  The shard's
// whole blocks are rotated as usual (fp32, written to their place in the
// rank's padded layout: [lead block] [whole blocks] [trail block]); each half
// block gets the unnormalised H512 of its 512 values, which the ranks then
// exchange.

// One warp per (token, task): task 0 is the leading half (if any), the last
// task the trailing half (if any), the others the whole blocks.
__global__ void __launch_bounds__(128) fwht_shard_kernel(
    const uint16_t* __restrict__ x, int M, int Kr, int lead, int trail,
    const int8_t* __restrict__ sign, float* __restrict__ xr, int Kp, float* __restrict__ h_lead,
    float* __restrict__ h_trail) {
  const int lane = threadIdx.x & 31;
  const int nb = (Kr - 512 * (lead + trail)) / kHBlock;
  const int T = nb + lead + trail;
  const long wid = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  pdl_launch_dependents();
  pdl_wait();
  if (wid >= static_cast<long>(M) * T) return;
  const int m = static_cast<int>(wid / T);
  const int t = static_cast<int>(wid % T);
  const uint16_t* xm = x + static_cast<long>(m) * Kr;
  const bool is_lead = lead && t == 0;
  const bool is_trail = trail && t == T - 1;
  if (is_lead || is_trail) {
    const int off = is_lead ? 0 : Kr - 512;
    float v[2][8];
    load_half(xm + off, sign ? sign + off : nullptr, lane, v);
    fwht_512_unscaled(v, lane);
    float* o = (is_lead ? h_lead : h_trail) + static_cast<long>(m) * 512;
#pragma unroll
    for (int ih = 0; ih < 2; ++ih) {
      float4* p = reinterpret_cast<float4*>(o + ih * 256 + lane * 8);
      p[0] = make_float4(v[ih][0], v[ih][1], v[ih][2], v[ih][3]);
      p[1] = make_float4(v[ih][4], v[ih][5], v[ih][6], v[ih][7]);
    }
    return;
  }
  const int j = t - lead;
  const int off = 512 * lead + j * kHBlock;
  float v[4][8];
  load_block(xm + off, sign ? sign + off : nullptr, lane, v);
  fwht_1024(v, lane);
  float* o = xr + static_cast<long>(m) * Kp + static_cast<long>(lead + j) * kHBlock;
#pragma unroll
  for (int ih = 0; ih < 4; ++ih) {
    float4* p = reinterpret_cast<float4*>(o + ih * 256 + lane * 8);
    p[0] = make_float4(v[ih][0], v[ih][1], v[ih][2], v[ih][3]);
    p[1] = make_float4(v[ih][4], v[ih][5], v[ih][6], v[ih][7]);
  }
}

// The exchanged halves of one split block -> this rank's half of the rotated
// block: the stride-512 butterfly (first half: a + b, second half: a - b),
// then * 1/32, written to padded block `blk`; the block's other 512 entries
// (the peer's half) are set to 0.  One thread per 4 values of a token.
__global__ void __launch_bounds__(256) fwht_combine_kernel(
    const float* __restrict__ h_first, const float* __restrict__ h_second, int M, int part,
    float* __restrict__ xr, int Kp, int blk) {
  const long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;   // (m, quad)
  pdl_launch_dependents();
  pdl_wait();
  if (i >= static_cast<long>(M) * 128) return;
  const long m = i / 128;
  const int qd = static_cast<int>(i % 128);
  const float4 a = reinterpret_cast<const float4*>(h_first + m * 512)[qd];
  const float4 b = reinterpret_cast<const float4*>(h_second + m * 512)[qd];
  float4 r;
  if (part == 0) {
    r = make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z),
                    __fadd_rn(a.w, b.w));
  } else {
    r = make_float4(__fsub_rn(a.x, b.x), __fsub_rn(a.y, b.y), __fsub_rn(a.z, b.z),
                    __fsub_rn(a.w, b.w));
  }
  r = make_float4(__fmul_rn(r.x, 0.03125f), __fmul_rn(r.y, 0.03125f), __fmul_rn(r.z, 0.03125f),
                  __fmul_rn(r.w, 0.03125f));
  float* o = xr + m * Kp + static_cast<long>(blk) * kHBlock;
  reinterpret_cast<float4*>(o)[qd] = r;
  reinterpret_cast<float4*>(o + 512)[qd] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Already rotated fp32 activations -> the GEMV's decode operand (DECODE) or
// the fp16 operand (F16), with the rotation kernel's arithmetic; one warp per
// (token, block).
template <int MODE>
__global__ void __launch_bounds__(128) quant_block_kernel(const float* __restrict__ xr, int M,
                                                          int K, __half* __restrict__ out,
                                                          float* __restrict__ out_scale) {
  const int lane = threadIdx.x & 31;
  const int B = K / kHBlock;
  const long wid = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  pdl_launch_dependents();
  pdl_wait();
  if (wid >= static_cast<long>(M) * B) return;
  const int m = static_cast<int>(wid / B);
  const int b = static_cast<int>(wid % B);
  const float* src = xr + static_cast<long>(m) * K + static_cast<long>(b) * kHBlock;
  float v[4][8];
#pragma unroll
  for (int ih = 0; ih < 4; ++ih) {
    const float4 p0 = reinterpret_cast<const float4*>(src + ih * 256 + lane * 8)[0];
    const float4 p1 = reinterpret_cast<const float4*>(src + ih * 256 + lane * 8)[1];
    v[ih][0] = p0.x; v[ih][1] = p0.y; v[ih][2] = p0.z; v[ih][3] = p0.w;
    v[ih][4] = p1.x; v[ih][5] = p1.y; v[ih][6] = p1.z; v[ih][7] = p1.w;
  }
  if (MODE == TERN_FWHT_DECODE) {
    decode_store(v, lane, m, b, M, K, out, out_scale);
    return;
  }
  float f, finv;
  f16_factor(v, f, finv);
  __half* o = out + static_cast<long>(m) * K + static_cast<long>(b) * kHBlock;
#pragma unroll
  for (int ih = 0; ih < 4; ++ih)
    *reinterpret_cast<uint4*>(o + ih * 256 + lane * 8) = f16_pack8(v, ih, f);
  if (lane == 0) out_scale[static_cast<long>(m) * B + b] = finv;
}

// Per-token int8 quantisation of already rotated fp32 activations (the
// arithmetic of fwht_i8_reg_kernel); one CTA per token, two passes over the row.
template <typename OutT>
__global__ void __launch_bounds__(256) quant_i8_kernel(const float* __restrict__ xr, int M, int K,
                                                       OutT* __restrict__ xq,
                                                       float* __restrict__ tscale) {
  __shared__ float red[8];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int m = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  const float* xm = xr + static_cast<long>(m) * K;
  float amax = 0.f;
  for (int i = threadIdx.x * 4; i < K; i += 256 * 4) {
    const float4 p = reinterpret_cast<const float4*>(xm + i)[0];
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(p.x), fabsf(p.y)), fmaxf(fabsf(p.z), fabsf(p.w))));
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
  OutT* om = xq + static_cast<long>(m) * K;
  for (int i = threadIdx.x * 4; i < K; i += 256 * 4) {
    const float4 p = reinterpret_cast<const float4*>(xm + i)[0];
    const float vv[4] = {p.x, p.y, p.z, p.w};
    float qv[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
      qv[t] = nz ? fminf(fmaxf(rintf(__fdiv_rn(vv[t], ts)), -127.f), 127.f) : 0.f;
    store_q4(om + i, qv);
  }
}

}  // namespace

cudaError_t launch_fwht_shard(const uint16_t* x, int64_t M, int64_t Kr, int lead, int trail,
                              const int8_t* sign, float* xr, float* h_lead, float* h_trail,
                              cudaStream_t st) {
  const int64_t Kp = Kr + 512 * (lead + trail);
  const long warps = M * ((Kr - 512 * (lead + trail)) / kHBlock + lead + trail);
  return launch(fwht_shard_kernel, dim3(static_cast<unsigned>((warps + 3) / 4)), dim3(128), 0, st,
                x, static_cast<int>(M), static_cast<int>(Kr), lead, trail, sign, xr,
                static_cast<int>(Kp), h_lead, h_trail);
}

cudaError_t launch_fwht_combine(const float* h_first, const float* h_second, int64_t M, int part,
                                float* xr, int64_t Kp, int64_t blk, cudaStream_t st) {
  const long threads = M * 128;
  return launch(fwht_combine_kernel, dim3(static_cast<unsigned>((threads + 255) / 256)), dim3(256),
                0, st, h_first, h_second, static_cast<int>(M), part, xr, static_cast<int>(Kp),
                static_cast<int>(blk));
}

cudaError_t launch_quant_rotated(const float* xr, int64_t M, int64_t K, int mode, void* out,
                                 float* out_scale, cudaStream_t st) {
  if (mode == TERN_FWHT_I8)
    return launch(quant_i8_kernel<int8_t>, dim3(static_cast<unsigned>(M)), dim3(256), 0, st, xr,
                  static_cast<int>(M), static_cast<int>(K), static_cast<int8_t*>(out), out_scale);
  if (mode == TERN_FWHT_I8H)
    return launch(quant_i8_kernel<__half>, dim3(static_cast<unsigned>(M)), dim3(256), 0, st, xr,
                  static_cast<int>(M), static_cast<int>(K), static_cast<__half*>(out), out_scale);
  const long warps = M * (K / kHBlock);
  const dim3 grid(static_cast<unsigned>((warps + 3) / 4));
  if (mode == TERN_FWHT_DECODE)
    return launch(quant_block_kernel<TERN_FWHT_DECODE>, grid, dim3(128), 0, st, xr,
                  static_cast<int>(M), static_cast<int>(K), static_cast<__half*>(out), out_scale);
  return launch(quant_block_kernel<TERN_FWHT_F16>, grid, dim3(128), 0, st, xr,
                static_cast<int>(M), static_cast<int>(K), static_cast<__half*>(out), out_scale);
}

cudaError_t launch_fwht(const uint16_t* x, int64_t M, int64_t K, const int8_t* sign, int mode,
                        void* out, float* out_scale, cudaStream_t st) {
  const int m = static_cast<int>(M), k = static_cast<int>(K);
  if (mode == TERN_FWHT_I8 || mode == TERN_FWHT_I8H) {
    // the entry point admits K <= 32768 in these modes: at most 32 warps
    const unsigned threads = static_cast<unsigned>(32 * (K / kHBlock));
    const bool small = K <= 18 * kHBlock;
    if (mode == TERN_FWHT_I8)
      return small ? launch(fwht_i8_reg_kernel<576, 2, int8_t>, dim3(m), dim3(threads), 0, st, x,
                            m, k, sign, static_cast<int8_t*>(out), out_scale)
                   : launch(fwht_i8_reg_kernel<1024, 1, int8_t>, dim3(m), dim3(threads), 0, st,
                            x, m, k, sign, static_cast<int8_t*>(out), out_scale);
    return small ? launch(fwht_i8_reg_kernel<576, 2, __half>, dim3(m), dim3(threads), 0, st, x, m,
                          k, sign, static_cast<__half*>(out), out_scale)
                 : launch(fwht_i8_reg_kernel<1024, 1, __half>, dim3(m), dim3(threads), 0, st, x,
                          m, k, sign, static_cast<__half*>(out), out_scale);
  }
  const long warps = M * (K / kHBlock);
  const dim3 grid(static_cast<unsigned>((warps + 3) / 4));
  if (mode == TERN_FWHT_F32)
    return launch(fwht_block_kernel<TERN_FWHT_F32>, grid, dim3(128), 0, st, x, m, k, sign, out,
                  out_scale);
  if (mode == TERN_FWHT_F16)
    return launch(fwht_block_kernel<TERN_FWHT_F16>, grid, dim3(128), 0, st, x, m, k, sign, out,
                  out_scale);
  return launch(fwht_block_kernel<TERN_FWHT_DECODE>, grid, dim3(128), 0, st, x, m, k, sign, out,
                out_scale);
}

}  // namespace tern
