// Decode GEMV for M <= 16 tokens over 2-bit ternary weights.
//
// Page "RTX 5070 x2 ... Ternary-Bonsai-2-27B on vLLM TP=2", section "前提":
// y[m,n] = sum_g s[n,g] sum_{k in g} code[n,k] xr[m,k] with codes in
// {-1,0,+1} at 2 bits and one fp16 scale per 128 elements of a row; xr is
// the block-Hadamard-rotated activation.  Section 5 records that an int8
// (dp4a) decode kernel added error and gained only 2% end to end, so the
// activations stay in fp16 here.
//
// Design (GB300):
// * Each weight byte is read once for all M tokens: tokens are the n side of
//   m16n8k16 tensor-core MMAs (one n8 tile for M <= 8, two for M <= 16), the
//   weight rows are the m side.
// * The packed format is laid out so that one 16-byte load per lane carries
//   the A fragments of 8 MMAs (16 rows x 128 k), and two register
//   instructions (shift, and) turn a 32-bit word into an fp16 pair 2*code.
// * Per 128-wide group, the raw code products accumulate in a fresh fp32
//   MMA accumulator; the group scale (times 1/2 for the 2*code reading, times
//   the per-block power of two of the fp16 operand) is applied with one FMA.
// * Work is split stream-K style: the units (256-row block, group) are cut
//   into equal contiguous ranges, one per persistent CTA (two per SM).  A row
//   block finished by one CTA is written directly; otherwise each
//   contributing CTA stores its partial in a slot of the workspace and the
//   last one to arrive (atomic counter, no waiting) sums the slots in fixed
//   order, writes bf16 and resets the counter.
// * The weights do not depend on the previous kernel, so each CTA issues its
//   first weight loads before waiting on the programmatic launch dependency.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tern_internal.cuh"

namespace tern {
namespace {

constexpr int kWarps = 8;           // warps per CTA
constexpr int kTW = 2;              // 16-row tiles per warp
constexpr int kRB = kWarps * kTW * 16;  // rows per row block (256)
constexpr int kPF = 3;              // units of weights in flight per warp
constexpr int kCtasPerSm = 2;

struct GemvPlan {
  int U;         // units = row blocks * G
  int C;         // CTAs
  int RBn;       // row blocks
  int S;         // partial slots per row block
};

__host__ __device__ inline long unit_begin(long c, long U, long C) { return c * U / C; }
// CTA owning unit u
__host__ __device__ inline long owner_of(long u, long U, long C) { return ((u + 1) * C - 1) / U; }

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1, bool zero_c) {
  if (zero_c) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

template <int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[kTW][NT][4]) {
#pragma unroll
  for (int tt = 0; tt < kTW; ++tt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[tt][nt][i] = 0.f;
}

// Weights of one unit for one warp: codes of its 16-row tiles and their scales.
struct Slot {
  uint4 c[kTW];
  uint32_t s[kTW];
};

template <int NT>
__global__ void __launch_bounds__(kWarps * 32, kCtasPerSm)
    gemv_decode_kernel(const uint4* __restrict__ packed, const uint32_t* __restrict__ sp,
                       const uint4* __restrict__ xh, const float* __restrict__ xs, int M, int N,
                       int K, __nv_bfloat16* __restrict__ y, unsigned int* __restrict__ counters,
                       float* __restrict__ partials, int U, int S) {
  // Activation fragments are prefetched one unit ahead when registers allow.
  constexpr bool kXPrefetch = (NT == 1);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int G = K / kGroup;
  const int B = K / kHBlock;
  const int n_tiles = (N + 15) / 16;
  const int C = gridDim.x;
  const int c = blockIdx.x;
  const int u0 = static_cast<int>(unit_begin(c, U, C));
  const int u1 = static_cast<int>(unit_begin(c + 1, U, C));
  const int r = lane >> 2;   // fragment row group
  const int cq = lane & 3;   // fragment column pair
  const int tile_in_rb = warp * kTW;

  __shared__ int s_last;

  // ---- weight prefetch cursor (rows of the warp, group) -------------------
  int pf_u = u0, pf_rb = u0 / G, pf_g = u0 % G;
  auto load_slot = [&](Slot& sl) {
#pragma unroll
    for (int tt = 0; tt < kTW; ++tt) {
      const int tile = pf_rb * (kRB / 16) + tile_in_rb + tt;
      if (tile < n_tiles) {
        const long chunk = static_cast<long>(tile) * G + pf_g;
        sl.c[tt] = ldg_stream(packed + chunk * 32 + lane);
        sl.s[tt] = __ldg(sp + chunk * 8 + r);
      } else {
        sl.c[tt] = make_uint4(0, 0, 0, 0);
        sl.s[tt] = 0u;
      }
    }
    ++pf_u;
    if (++pf_g == G) {
      pf_g = 0;
      ++pf_rb;
    }
  };

  Slot ring[kPF];
#pragma unroll
  for (int s = 0; s < kPF; ++s)
    if (pf_u < u1) load_slot(ring[s]);

  pdl_wait();
  pdl_launch_dependents();

  auto load_x = [&](int gg, uint4 (&xo)[4][NT], float (&xso)[NT][2]) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tok = nt * 8 + r;
        xo[ch][nt] = tok < M ? __ldg(xh + ((static_cast<long>(gg) * 4 + ch) * M + tok) * 4 + cq)
                             : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int tok = nt * 8 + 2 * cq + h;
        xso[nt][h] = tok < M ? __ldg(xs + static_cast<long>(tok) * B + (gg >> 3)) : 0.f;
      }
  };

  float acc[kTW][NT][4];
  zero_acc<NT>(acc);

  auto flush = [&](int rb, int ga, int gb) {
    if (ga == 0 && gb == G) {   // the whole row block is ours: write y directly
#pragma unroll
      for (int tt = 0; tt < kTW; ++tt) {
        const int row0 = (rb * (kRB / 16) + tile_in_rb + tt) * 16 + r;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = row0 + 8 * (i >> 1);
            const int tok = nt * 8 + 2 * cq + (i & 1);
            if (row < N && tok < M)
              y[static_cast<long>(tok) * N + row] = __float2bfloat16_rn(acc[tt][nt][i]);
          }
      }
      return;
    }
    // a piece of the row block: store it in our slot, last arriver reduces
    const long first = owner_of(static_cast<long>(rb) * G, U, C);
    const long last_owner = owner_of(static_cast<long>(rb) * G + G - 1, U, C);
    const long slot = c - first;
    float* base = partials + (static_cast<long>(rb) * S + slot) * static_cast<long>(M) * kRB;
#pragma unroll
    for (int tt = 0; tt < kTW; ++tt) {
      const int rowin0 = (tile_in_rb + tt) * 16 + r;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rowin = rowin0 + 8 * (i >> 1);
          const int tok = nt * 8 + 2 * cq + (i & 1);
          if (tok < M) __stcg(base + static_cast<long>(tok) * kRB + rowin, acc[tt][nt][i]);
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned add = static_cast<unsigned>(gb - ga);
      const unsigned old = atomicAdd(counters + rb, add);
      s_last = (old + add == static_cast<unsigned>(G)) ? 1 : 0;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      const long nslots = last_owner - first + 1;
#pragma unroll
      for (int tt = 0; tt < kTW; ++tt) {
        const int rowin0 = (tile_in_rb + tt) * 16 + r;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int rowin = rowin0 + 8 * (i >> 1);
            const int tok = nt * 8 + 2 * cq + (i & 1);
            const int row = rb * kRB + rowin;
            if (tok < M && row < N) {
              float sum = 0.f;
              for (long sl = 0; sl < nslots; ++sl)
                sum += __ldcg(partials + ((static_cast<long>(rb) * S + sl) * M + tok) * kRB + rowin);
              y[static_cast<long>(tok) * N + row] = __float2bfloat16_rn(sum);
            }
          }
      }
      if (threadIdx.x == 0) counters[rb] = 0u;
    }
    __syncthreads();
  };

  int rb = u0 / G, g = u0 % G;
  int seg_g0 = g;   // first group of the current row-block segment
  uint4 xv[4][NT];
  float xsv[NT][2];
  if (kXPrefetch && u0 < u1) load_x(g, xv, xsv);

  for (int ub = u0; ub < u1; ub += kPF) {
#pragma unroll
    for (int s = 0; s < kPF; ++s) {
      const int u = ub + s;
      if (u < u1) {
        int nrb = rb, ng = g + 1;
        if (ng == G) {
          ng = 0;
          ++nrb;
        }
        uint4 xn[4][NT];
        float xsn[NT][2];
        if (kXPrefetch) {
          if (u + 1 < u1) load_x(ng, xn, xsn);
        } else {
          load_x(g, xv, xsv);
        }
#pragma unroll
        for (int tt = 0; tt < kTW; ++tt) {
          uint32_t s2 = ring[s].s[tt];
          const float2 f2 = __half22float2(*reinterpret_cast<__half2*>(&s2));
          const float sr = f2.x * 0.5f, sr8 = f2.y * 0.5f;   // 1/2 undoes the 2*code reading
          const uint32_t w4[4] = {ring[s].c[tt].x, ring[s].c[tt].y, ring[s].c[tt].z,
                                  ring[s].c[tt].w};
          float d[NT][4];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t w = w4[j >> 1];
            const int e0 = (j & 1) * 4;
            uint32_t a[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) a[p] = (w << (14 - 2 * (e0 + p))) & 0xC000C000u;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint4 xq = xv[j >> 1][nt];
              mma16816(d[nt], a, (j & 1) ? xq.z : xq.x, (j & 1) ? xq.w : xq.y, j == 0);
            }
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            acc[tt][nt][0] = fmaf(d[nt][0], sr * xsv[nt][0], acc[tt][nt][0]);
            acc[tt][nt][1] = fmaf(d[nt][1], sr * xsv[nt][1], acc[tt][nt][1]);
            acc[tt][nt][2] = fmaf(d[nt][2], sr8 * xsv[nt][0], acc[tt][nt][2]);
            acc[tt][nt][3] = fmaf(d[nt][3], sr8 * xsv[nt][1], acc[tt][nt][3]);
          }
        }
        if (pf_u < u1) load_slot(ring[s]);
        if (u + 1 == u1 || nrb != rb) {
          flush(rb, seg_g0, g + 1);
          zero_acc<NT>(acc);
          seg_g0 = 0;
        }
        rb = nrb;
        g = ng;
        if (kXPrefetch) {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) xv[ch][nt] = xn[ch][nt];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            xsv[nt][0] = xsn[nt][0];
            xsv[nt][1] = xsn[nt][1];
          }
        }
      }
    }
  }
}

GemvPlan make_plan(int64_t M, int64_t N, int64_t K, int sms) {
  GemvPlan p;
  const long G = K / kGroup;
  p.RBn = static_cast<int>((N + kRB - 1) / kRB);
  p.U = static_cast<int>(p.RBn * G);
  const long cmax = static_cast<long>(sms) * kCtasPerSm;
  p.C = static_cast<int>(p.U < cmax ? p.U : cmax);
  // slots: the most CTAs that touch one row block
  long s = 1;
  for (long rb = 0; rb < p.RBn; ++rb) {
    const long a = owner_of(rb * G, p.U, p.C), b = owner_of(rb * G + G - 1, p.U, p.C);
    if (b - a + 1 > s) s = b - a + 1;
  }
  p.S = static_cast<int>(s);
  (void)M;
  return p;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 152;
  return n;
}

}  // namespace

// Workspace: [RBn] counters (padded to 256 B), then partials [RBn][S][M][256] fp32.
size_t gemv_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const GemvPlan p = make_plan(M, N, K, sm_count());
  const size_t cnt = (static_cast<size_t>(p.RBn) * 4 + 255) / 256 * 256;
  return cnt + static_cast<size_t>(p.RBn) * p.S * M * kRB * sizeof(float);
}

cudaError_t launch_gemv(const uint8_t* packed, const uint16_t* scales_packed, const uint16_t* xh,
                        const float* xs, int64_t M, int64_t N, int64_t K, uint16_t* y, void* ws,
                        cudaStream_t st) {
  const GemvPlan p = make_plan(M, N, K, sm_count());
  const size_t cnt = (static_cast<size_t>(p.RBn) * 4 + 255) / 256 * 256;
  unsigned int* counters = static_cast<unsigned int*>(ws);
  float* partials = reinterpret_cast<float*>(static_cast<char*>(ws) + cnt);
  const auto* pk = reinterpret_cast<const uint4*>(packed);
  const auto* spk = reinterpret_cast<const uint32_t*>(scales_packed);
  const auto* xv = reinterpret_cast<const uint4*>(xh);
  auto* yy = reinterpret_cast<__nv_bfloat16*>(y);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  if (M <= 8)
    return launch(gemv_decode_kernel<1>, dim3(p.C), dim3(kWarps * 32), 0, st, pk, spk, xv, xs, m,
                  n, k, yy, counters, partials, p.U, p.S);
  return launch(gemv_decode_kernel<2>, dim3(p.C), dim3(kWarps * 32), 0, st, pk, spk, xv, xs, m, n,
                k, yy, counters, partials, p.U, p.S);
}

}  // namespace tern
