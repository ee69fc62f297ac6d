// Device routines of the block Hadamard rotation, shared by the rotation
// kernels (fwht.cu) and the fused rotate + decode GEMV (gemv.cu), so that both
// produce bit-identical operands.
//
// Page "RTX 5070 x2 ... Ternary-Bonsai-2-27B on vLLM TP=2": section "前提"
// (block-wise Hadamard rotation on the input side) and section 1 (Sylvester
// structure, split identity H1024[a;b] = [H512 a + H512 b ; H512 a - H512 b]
// as the last butterfly stage).
//
// One warp transforms one 1024-block of one token.  Lane l holds the 32
// elements with index  ih*256 + l*8 + il  (ih = 0..3, il = 0..7): index bits
// 0-2 are the register index il, bits 3-7 the lane, bits 8-9 the register
// index ih.  Stage s (stride 2^s) therefore runs inside a thread for
// s = 0,1,2,8,9 and across lanes (shuffle xor 2^(s-3)) for s = 3..7.  The
// stages run in the order s = 0..9 so the fp32 rounding is that of the
// canonical transform with the stride-512 split identity last.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace tern {
namespace fwht {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void load_block(const uint16_t* __restrict__ xb,
                                           const int8_t* __restrict__ sb, int lane,
                                           float (&v)[4][8]) {
#pragma unroll
  for (int ih = 0; ih < 4; ++ih) {
    uint4 raw = __ldg(reinterpret_cast<const uint4*>(xb + ih * 256 + lane * 8));
    uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v[ih][2 * q] = __uint_as_float(w[q] << 16);           // bf16 -> fp32 is exact
      v[ih][2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
    }
    if (sb != nullptr) {
#pragma unroll
      for (int il = 0; il < 8; ++il) {
        float s = static_cast<float>(__ldg(sb + ih * 256 + lane * 8 + il));
        v[ih][il] = v[ih][il] * s;
      }
    }
  }
}

// In-register butterfly between registers a (lower index) and b.
__device__ __forceinline__ void bfly(float& a, float& b) {
  float s = __fadd_rn(a, b);
  float d = __fsub_rn(a, b);
  a = s;
  b = d;
}

__device__ __forceinline__ void fwht_1024(float (&v)[4][8], int lane) {
  // stages 0, 1, 2: within the 8 registers of one ih
#pragma unroll
  for (int s = 0; s < 3; ++s) {
    const int h = 1 << s;
#pragma unroll
    for (int ih = 0; ih < 4; ++ih)
#pragma unroll
      for (int il = 0; il < 8; ++il)
        if ((il & h) == 0) bfly(v[ih][il], v[ih][il + h]);
  }
  // stages 3..7: across lanes
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int lm = 1 << s;
    // lower lane: u + v (own + partner); upper lane: u - v (partner - own),
    // both as one fma with the lane's sign (a product by +-1 is exact and
    // the fma rounds once: the same result, signed zeros included)
    const float sg = (lane & lm) != 0 ? -1.f : 1.f;
#pragma unroll
    for (int ih = 0; ih < 4; ++ih)
#pragma unroll
      for (int il = 0; il < 8; ++il) {
        const float p = __shfl_xor_sync(kFull, v[ih][il], lm);
        v[ih][il] = __fmaf_rn(v[ih][il], sg, p);
      }
  }
  // stages 8, 9: across the 4 register groups
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int h = 1 << s;
#pragma unroll
    for (int ih = 0; ih < 4; ++ih)
      if ((ih & h) == 0)
#pragma unroll
        for (int il = 0; il < 8; ++il) bfly(v[ih][il], v[ih + h][il]);
  }
#pragma unroll
  for (int ih = 0; ih < 4; ++ih)
#pragma unroll
    for (int il = 0; il < 8; ++il) v[ih][il] = __fmul_rn(v[ih][il], 0.03125f);
}

// The 512-element half of a block (page section 1: each rank of a K split
// that cuts a block in the middle transforms its own half): lane l holds the
// 16 elements ih*256 + l*8 + il (ih = 0..1, il = 0..7), loaded like
// load_block.
__device__ __forceinline__ void load_half(const uint16_t* __restrict__ xb,
                                          const int8_t* __restrict__ sb, int lane,
                                          float (&v)[2][8]) {
#pragma unroll
  for (int ih = 0; ih < 2; ++ih) {
    uint4 raw = __ldg(reinterpret_cast<const uint4*>(xb + ih * 256 + lane * 8));
    uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v[ih][2 * q] = __uint_as_float(w[q] << 16);
      v[ih][2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
    }
    if (sb != nullptr) {
#pragma unroll
      for (int il = 0; il < 8; ++il) {
        float s = static_cast<float>(__ldg(sb + ih * 256 + lane * 8 + il));
        v[ih][il] = v[ih][il] * s;
      }
    }
  }
}

// Unnormalised H512 of a half block: the stages with stride 1 .. 256 of the
// canonical transform, in the same order and fp32 operations as the first
// nine stages of fwht_1024, so that the stride-512 stage applied to two
// halves afterwards (sum for the first half, difference for the second,
// then * 1/32) reproduces fwht_1024 bit for bit.
__device__ __forceinline__ void fwht_512_unscaled(float (&v)[2][8], int lane) {
#pragma unroll
  for (int s = 0; s < 3; ++s) {
    const int h = 1 << s;
#pragma unroll
    for (int ih = 0; ih < 2; ++ih)
#pragma unroll
      for (int il = 0; il < 8; ++il)
        if ((il & h) == 0) bfly(v[ih][il], v[ih][il + h]);
  }
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int lm = 1 << s;
    const float sg = (lane & lm) != 0 ? -1.f : 1.f;   // as in fwht_1024
#pragma unroll
    for (int ih = 0; ih < 2; ++ih)
#pragma unroll
      for (int il = 0; il < 8; ++il) {
        const float p = __shfl_xor_sync(kFull, v[ih][il], lm);
        v[ih][il] = __fmaf_rn(v[ih][il], sg, p);
      }
  }
#pragma unroll
  for (int il = 0; il < 8; ++il) bfly(v[0][il], v[1][il]);
}

__device__ __forceinline__ float warp_max(float a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(kFull, a, o));
  return a;
}


// fp16 operand of one rotated block (the fp16 prefill variant's operand):
// the power-of-two factor F with max|xr * F| in [2^14, 2^15)
// (F = 2^min(14 - E, 126), E the exponent of the block's absmax), returned
// with its exact inverse; xr * F rounds to fp16.
__device__ __forceinline__ int block_shift(const float (&v)[4][8]) {
  float amax = 0.f;
#pragma unroll
  for (int ih = 0; ih < 4; ++ih)
#pragma unroll
    for (int il = 0; il < 8; ++il) amax = fmaxf(amax, fabsf(v[ih][il]));
  amax = warp_max(amax);
  const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127;
  return min(14 - e, 126);                         // >= -114
}
__device__ __forceinline__ float pow2f(int e) {    // 2^e for -126 <= e <= 127
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}
__device__ __forceinline__ void f16_factor(const float (&v)[4][8], float& f, float& finv) {
  const int sh = block_shift(v);
  f = pow2f(sh);
  finv = pow2f(-sh);
}

// fp16 (xr * f) of the 8 elements ih*256 + lane*8 + 0..7, packed as a uint4.
__device__ __forceinline__ uint4 f16_pack8(const float (&v)[4][8], int ih, float f) {
  uint32_t w[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    __half2 h2 = __floats2half2_rn(__fmul_rn(v[ih][2 * t], f), __fmul_rn(v[ih][2 * t + 1], f));
    w[t] = *reinterpret_cast<uint32_t*>(&h2);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------- decode operand
// The decode GEMV's operand (include/tern.h, TERN_FWHT_DECODE).  Lane l's 8
// elements ih*256 + l*8 + 0..7 lie in 128-group 2 ih + l / 16 of the block and
// in its k16 step j = (l % 16) / 2, whose packed field carries the power of
// four e(j) = j (j < 6) or j - 6.  The operand is fp16(xr * 2^(sh - 2e)); the
// group offset is the fp32 sum of fp16 value * 2^(2e - 24): each lane's 8
// terms left to right, then the 16 lanes of the group by a butterfly
// (xor 1, 2, 4, 8); the block's fold factor is 2^(12 - sh).
__device__ __forceinline__ int lane_step_exp(int lane) {
  const int j = (lane & 15) >> 1;
  return j < 6 ? j : j - 6;
}

// The fp16 operand of the lane's 8 elements of register group ih (packed as a
// uint4) and the lane's partial sum of the group offset.
__device__ __forceinline__ uint4 decode_pack8(const float (&v)[4][8], int ih, int sh, int e,
                                              float& part) {
  const float f = pow2f(sh - 2 * e);               // >= 2^-124: a normal float
  const float back = pow2f(2 * e - 24);
  uint32_t w[4];
  float acc = 0.f;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    __half2 h2 = __floats2half2_rn(__fmul_rn(v[ih][2 * t], f), __fmul_rn(v[ih][2 * t + 1], f));
    const float2 r = __half22float2(h2);
    acc = t == 0 ? __fmul_rn(r.x, back) : __fadd_rn(acc, __fmul_rn(r.x, back));
    acc = __fadd_rn(acc, __fmul_rn(r.y, back));
    w[t] = *reinterpret_cast<uint32_t*>(&h2);
  }
  part = acc;
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The group offset from the lanes' partial sums (every lane of the 16-lane
// half gets the same value).
__device__ __forceinline__ float group_offset(float part) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) part = __fadd_rn(part, __shfl_xor_sync(kFull, part, o));
  return part;
}

// Rotated block (token m, block b) -> the decode operand in global memory:
// xh [M][K] fp16 and the 48-float group records aux [G][48]: the negated
// offsets as the tensor core's accumulator quads (0 - X of tokens 2i and
// 2i + 1 at [g][4i], [g][4i + 1] and again at [g][4i + 2], [g][4i + 3]) and
// the block's fold factor of token m at [g][32 + m].  The warp of token 0
// also writes the zeros of tokens M..15 in the block's 8 records.
__device__ __forceinline__ void decode_store(const float (&v)[4][8], int lane, int m, int b,
                                             int M, int K, __half* __restrict__ out,
                                             float* __restrict__ aux) {
  const int sh = block_shift(v);
  const int e = lane_step_exp(lane);
  __half* o = out + static_cast<long>(m) * K + static_cast<long>(b) * 1024;
  float* ab = aux + static_cast<long>(b) * 8 * 48;
  const int qi = 4 * (m >> 1) + (m & 1);
#pragma unroll
  for (int ih = 0; ih < 4; ++ih) {
    float part;
    *reinterpret_cast<uint4*>(o + ih * 256 + lane * 8) = decode_pack8(v, ih, sh, e, part);
    const float x = __fsub_rn(0.f, group_offset(part));
    if ((lane & 15) == 0) {
      float* rec = ab + (2 * ih + (lane >> 4)) * 48;
      rec[qi] = x;
      rec[qi + 2] = x;
      rec[32 + m] = pow2f(12 - sh);
    }
  }
  if (m == 0)
    for (int i = lane; i < 8 * 16; i += 32) {
      const int t = i & 15;
      if (t >= M) {
        float* rec = ab + (i >> 4) * 48;
        const int q = 4 * (t >> 1) + (t & 1);
        rec[q] = 0.f;
        rec[q + 2] = 0.f;
        rec[32 + t] = 0.f;
      }
    }
}

}  // namespace fwht
}  // namespace tern
