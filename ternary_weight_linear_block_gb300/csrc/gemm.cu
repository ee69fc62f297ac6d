// The int8 prefill GEMMs with per-row and per-token rescale: gemm_i8_kernel
// on the expanded weight (below) and gemm_packed_kernel straight from the
// decode's 2-bit packed weights (further down), with bit-identical results.
//
// Page "RTX 5070 x2 ... Ternary-Bonsai-2-27B on vLLM TP=2", section 4
// ("prefill の線形層を int8 GEMM に"): with q[n,g] = round(127 s[n,g]/smax[n])
// the weight W_int8[n,k] = code[n,k] q[n,k/128] is an exact int8 matrix, the
// rotated activations are quantised per token to int8, one int8 GEMM gives
// acc[m,n] (int32), and y = acc * tscale[m] * rscale[n].
//
// GB300 design.  sm_103a has no tcgen05 int8 MMA kind (ptxas rejects
// kind::i8 for sm_103a) and the legacy int8 mma.sync runs at a quarter of the
// fp16 rate, so the product runs on the fp16 tensor path: every integer in
// [-127, 127] is exact in fp16 and every product (|.| <= 16129) is exact in
// the fp32 accumulator.  A sum of 1024 such products stays below
// 1024 * 127^2 < 2^24, so the fp32 accumulator of one 1024-wide K chunk holds
// the exact integer; the epilogue converts each chunk to int32 and adds
// chunks in int32.  acc is therefore bit-exact.
//
// Kernel: persistent CTAs (one per SM), tile 128 tokens x 256 weight rows,
// 64-wide K stages, 4-stage TMA ring (128-byte swizzle), tcgen05.mma
// (cta_group::1, kind::f16, M=128 N=256 K=16) accumulating one K chunk in a
// TMEM buffer; two TMEM buffers alternate so the MMA of chunk c+1 overlaps
// the epilogue draining chunk c.  Warp roles: 0 TMA producer, 1 MMA issuer,
// 2 TMEM allocator, 4-11 epilogue (two warpgroups, 128 columns each).
#include <cuda.h>
#include <cuda_bf16.h>

#include <type_traits>

#include "sm100_ptx.cuh"
#include "tern_internal.cuh"

namespace tern {

__device__ unsigned int g_gemm_error;

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int KCHUNK = 1024;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 384;
constexpr int TMEM_COLS = 512;
// Polls of a bounded barrier wait before it gives up: a poll that finds the
// phase incomplete suspends for about 3.8 us on GB300 (measured with
// tern_selftest_wait), so 2^18 polls give up after about one second; a
// wait of the working kernel lasts microseconds.
constexpr uint32_t WAIT_LIMIT = 1u << 18;
constexpr uint32_t IDESC = ptx::idesc_f16_f32(BM, BN);
// a CTA pair's MMA: 256 rows (128 per CTA) x 256 columns
constexpr uint32_t IDESC_PAIR = ptx::idesc_f16_f32(256, 256);
constexpr size_t SMEM_BYTES = static_cast<size_t>(STAGES) * STAGE_BYTES + 1024 + 256;
// a CTA pair's stage: 128 tokens and 128 weight rows (32 KB), six of them in
// the single CTA's four-stage area
constexpr int PAIR_STAGES = 6;
static_assert(PAIR_STAGES * (A_BYTES + B_BYTES / 2) <= STAGES * STAGE_BYTES, "pair stages fit");

enum : unsigned int {
  ERR_PRODUCER = 1u, ERR_MMA = 2u, ERR_EPILOGUE = 4u, ERR_DRAIN = 8u, ERR_EXPAND = 16u,
  ERR_SELFTEST = 32u
};

__device__ __forceinline__ void fail(volatile int* abort_flag, unsigned int code) {
  *abort_flag = 1;
  atomicOr(&g_gemm_error, code);
}

// The kernel body of both tensor-core GEMMs on an fp16 [N][K] weight.  FP =
// false: the int8 path (integer values, exact chunk sums, per-row and
// per-token rescale).  FP = true: the fp16 path, whose activations are the
// decode operand (fp16 with one power-of-two factor per token and 1024-block):
// each 1024-chunk of K is one rotation block, so the epilogue multiplies the
// chunk's fp32 sum by the token's block factor (`tscale` holds xs [M][K/1024])
// and adds the chunks in fp32; `rscale` and `acc_out` are unused.
// SPLIT: the tiles after the first `full_arg` (all tiles, or those of the
// last, partial wave) have their K range cut in S slices of whole
// 1024-chunks (units of work = (tile, slice)); a slice stores its partial
// sums (int32 or fp32) in its own [128][256] piece of `part`, and a second
// kernel adds each tile's pieces in slice order and finishes the output.
//
// PAIR (M > 128): clusters of two CTAs share each 256-token x 256-weight-row
// tile (tcgen05 cta_group::2).  Each CTA loads its own 128 tokens and 128
// weight rows (32 KB a stage, six stages), warp 3 relays "stage s landed" to
// the even CTA's pfull[s], and the even CTA issues 256 x 256 x 16 MMAs whose
// commits arrive (multicast) on both CTAs' barriers; each CTA's epilogue
// drains its 128 token rows (all 256 weight columns) and releases the
// accumulator buffer on the even CTA's dempty.  Per SM this halves the
// weight copies into shared memory and the tensor cores' reads of them, and
// shared-memory bandwidth (operand copies in, operand reads out) bounds the
// single-CTA tile.
template <bool FP, bool SPLIT, bool PAIR>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                          const float* __restrict__ tscale,
                                          const float* __restrict__ rscale, int M, int N, int K,
                                          __nv_bfloat16* __restrict__ y,
                                          int32_t* __restrict__ acc_out, int S_arg,
                                          int full_arg, void* __restrict__ part) {
  const int S = SPLIT ? S_arg : 1;
  constexpr int NST = PAIR ? PAIR_STAGES : STAGES;
  constexpr int TM = PAIR ? 2 * BM : BM;              // token rows of a tile
  constexpr int BB = PAIR ? B_BYTES / 2 : B_BYTES;    // this CTA's weight rows, one stage
  constexpr int WROWS_CTA = PAIR ? BN / 2 : BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + NST * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NST * (A_BYTES + BB));
  uint64_t* empty = full + NST;
  uint64_t* dfull = empty + NST;
  uint64_t* dempty = dfull + 2;
  uint64_t* done = dempty + 2;
  uint64_t* pfull = done + 1;   // (pairs) both CTAs' stage landed, in the even CTA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pfull + NST);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = PAIR ? static_cast<int>(ptx::cluster_ctarank()) : 0;
  const int team = PAIR ? static_cast<int>(ptx::cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int teams = PAIR ? static_cast<int>(ptx::cluster_count_x()) : static_cast<int>(gridDim.x);
  const int m_blocks = (M + TM - 1) / TM;
  const int n_blocks = (N + BN - 1) / BN;
  const int tiles = m_blocks * n_blocks;
  const int chunks = K / KCHUNK;
  // units: the first n_whole tiles whole, then every later tile in S slices
  const int n_whole = SPLIT ? full_arg : tiles;
  const int units = n_whole + (tiles - n_whole) * S;
  constexpr int kStagesPerChunk = KCHUNK / BK;
  // tile and chunk range [c0, c1) of unit u; piece = its slice index among
  // all slices (-1 for a whole tile)
  auto unit_of = [&](int u, int& tile, int& c0, int& c1, int& piece) {
    if (!SPLIT || u < n_whole) {
      tile = u;
      c0 = 0;
      c1 = chunks;
      piece = -1;
    } else {
      const int v = u - n_whole;
      const int sl = v % S;
      tile = n_whole + v / S;
      c0 = sl * chunks / S;
      c1 = (sl + 1) * chunks / S;
      piece = v;
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
      ptx::mbar_init(&pfull[s], 2);   // (pairs) one relay arrival per CTA
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&dfull[b], 1);
      ptx::mbar_init(&dempty[b], PAIR ? 16 : 8);   // one arrival per epilogue warp (of both CTAs)
    }
    ptx::mbar_init(done, 1);
    *abort_flag = 0;
    ptx::mbar_fence_init();
  }
  if (warp == 2) {
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(tmem_slot, TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(tmem_slot, TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) ptx::cluster_sync();   // both CTAs' barriers exist before any remote arrival
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_wait();   // xq / tscale come from the previous kernel
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int s = 0;
      uint32_t phase = 0;
      long issued = 0;
      bool ok = true;
      for (int u = team; u < units && ok; u += teams) {
        int tile, c0, c1, piece;
        unit_of(u, tile, c0, c1, piece);
        const int n_blk = tile / m_blocks, m_blk = tile % m_blocks;
        const int ks1 = c1 * kStagesPerChunk;
        for (int ks = c0 * kStagesPerChunk; ks < ks1; ++ks) {
          if (!ptx::mbar_wait(&empty[s], phase ^ 1u, abort_flag, WAIT_LIMIT)) {
            if (!*abort_flag) fail(abort_flag, ERR_PRODUCER);
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[s], A_BYTES + BB);
          ptx::tma_load_2d(sA + s * A_BYTES, &tmA, &full[s], ks * BK, m_blk * TM + rank * BM);
          ptx::tma_load_2d(sB + s * BB, &tmB, &full[s], ks * BK, n_blk * BN + rank * WROWS_CTA);
          ++issued;
          if (++s == NST) {
            s = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let the copies still in flight land before the CTA exits
        long back = issued < NST ? issued : NST;
        int ss = s;
        uint32_t ph = phase;
        for (long i = 0; i < back; ++i) {
          if (--ss < 0) {
            ss = NST - 1;
            ph ^= 1u;
          }
          if (!ptx::mbar_wait_bounded(&full[ss], ph, WAIT_LIMIT)) atomicOr(&g_gemm_error, ERR_DRAIN);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (one thread; in a pair, the even CTA's, for both)
      int s = 0;
      uint32_t phase = 0;
      uint32_t cc = 0;   // chunk counter across tiles
      bool ok = true;
      for (int u = team; u < units && ok; u += teams) {
        int tile, c0, c1, piece;
        unit_of(u, tile, c0, c1, piece);
        for (int c = c0; c < c1 && ok; ++c, ++cc) {
          const uint32_t buf = cc & 1u, dph = (cc >> 1) & 1u;
          if (!ptx::mbar_wait(&dempty[buf], dph ^ 1u, abort_flag, WAIT_LIMIT)) {
            if (!*abort_flag) fail(abort_flag, ERR_MMA);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem + buf * BN;
          for (int j = 0; j < kStagesPerChunk; ++j) {
            // (pairs: the even CTA waits until both CTAs' stage has landed)
            if (!ptx::mbar_wait(PAIR ? &pfull[s] : &full[s], phase, abort_flag, WAIT_LIMIT)) {
              if (!*abort_flag) fail(abort_flag, ERR_MMA);
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t a0 = ptx::sw128_kmajor_desc(ptx::smem_u32(sA + s * A_BYTES));
            const uint64_t b0 = ptx::sw128_kmajor_desc(ptx::smem_u32(sB + s * BB));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              if constexpr (PAIR)
                ptx::mma_f16_ss_pair(d_tmem, a0 + 2u * kk, b0 + 2u * kk, IDESC_PAIR,
                                     (j > 0 || kk > 0) ? 1u : 0u);
              else
                ptx::mma_f16_ss(d_tmem, a0 + 2u * kk, b0 + 2u * kk, IDESC,
                                (j > 0 || kk > 0) ? 1u : 0u);
            }
            if constexpr (PAIR)
              ptx::mma_commit_pair(&empty[s], 0x3);
            else
              ptx::mma_commit(&empty[s]);
            if (++s == NST) {
              s = 0;
              phase ^= 1u;
            }
          }
          if (ok) {
            if constexpr (PAIR)
              ptx::mma_commit_pair(&dfull[buf], 0x3);
            else
              ptx::mma_commit(&dfull[buf]);
          }
        }
      }
      // every MMA issued by this thread has completed once `done` fires
      if constexpr (PAIR)
        ptx::mma_commit_pair(done, 0x3);
      else
        ptx::mma_commit(done);
      if (!ptx::mbar_wait_bounded(done, 0, WAIT_LIMIT)) atomicOr(&g_gemm_error, ERR_DRAIN);
    }
    __syncwarp();
  } else if (warp == 3) {
    if (PAIR && lane == 0) {
      // ---------------- relay (pairs): once this CTA's stage has landed, one
      // arrival on the even CTA's pfull[s]
      int s = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint32_t pf = ptx::mapa_shared(pfull, 0);
      for (int u = team; u < units && ok; u += teams) {
        int tile, c0, c1, piece;
        unit_of(u, tile, c0, c1, piece);
        for (int j = 0; j < (c1 - c0) * kStagesPerChunk; ++j) {
          if (!ptx::mbar_wait(&full[s], phase, abort_flag, WAIT_LIMIT)) {
            if (!*abort_flag) fail(abort_flag, ERR_MMA);
            ok = false;
            break;
          }
          ptx::mbar_arrive_cluster(pf + 8u * static_cast<uint32_t>(s));
          if (++s == NST) {
            s = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- epilogue: warpgroup wg owns columns [128 wg, 128 wg + 128)
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;   // TMEM lane quarter accessible to this warp
    uint32_t cc = 0;
    bool ok = true;
    for (int u = team; u < units && ok; u += teams) {
      int tile, c0, c1, piece;
      unit_of(u, tile, c0, c1, piece);
      const int n_blk = tile / m_blocks, m_blk = tile % m_blocks;
      const int row = m_blk * TM + rank * BM + 32 * q + lane;
      typename std::conditional<FP, float, int32_t>::type sums[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) sums[i] = 0;
      for (int c = c0; c < c1; ++c, ++cc) {
        const uint32_t buf = cc & 1u, dph = (cc >> 1) & 1u;
        if (!ptx::mbar_wait_warp(&dfull[buf], dph, abort_flag, WAIT_LIMIT)) {
          if (!*abort_flag) fail(abort_flag, ERR_EPILOGUE);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        float f = 0.f;   // the token's factor of rotation block c (fp16 path)
        if (FP && row < M) f = __ldg(tscale + static_cast<long>(row) * chunks + c);
#pragma unroll
        for (int piece = 0; piece < 4; ++piece) {
          uint32_t v[32];
          const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * BN +
                                 wg * 128 + piece * 32;
          ptx::tmem_ld_32x32b_x32(taddr, v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if constexpr (FP)
              sums[piece * 32 + i] = __fadd_rn(sums[piece * 32 + i],
                                               __fmul_rn(__uint_as_float(v[i]), f));
            else
              sums[piece * 32 + i] += __float2int_rn(__uint_as_float(v[i]));   // exact integers
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            ptx::mbar_arrive_cluster(ptx::mapa_shared(&dempty[buf], 0));
          else
            ptx::mbar_arrive(&dempty[buf]);
        }
      }
      if (!ok) break;
      if (SPLIT && piece >= 0) {
        // one slice of a split tile: its partial sums into the slice's
        // [TM][256] piece of `part` (this CTA's rows of it); the finishing
        // kernel adds the pieces
        if (row < M) {
          const int n0 = n_blk * BN + wg * 128;
          auto* prow = static_cast<typename std::conditional<FP, float, int32_t>::type*>(part) +
                       (static_cast<long>(piece) * TM + rank * BM + 32 * q + lane) * BN +
                       wg * 128;
#pragma unroll
          for (int j = 0; j < 128; j += 8)
            if (n0 + j < N) {
              if constexpr (FP) {
                float4* pp = reinterpret_cast<float4*>(prow + j);
                pp[0] = make_float4(sums[j], sums[j + 1], sums[j + 2], sums[j + 3]);
                pp[1] = make_float4(sums[j + 4], sums[j + 5], sums[j + 6], sums[j + 7]);
              } else {
                int4* pp = reinterpret_cast<int4*>(prow + j);
                pp[0] = make_int4(sums[j], sums[j + 1], sums[j + 2], sums[j + 3]);
                pp[1] = make_int4(sums[j + 4], sums[j + 5], sums[j + 6], sums[j + 7]);
              }
            }
        }
        continue;
      }
      if (FP && row < M) {
        const int n0 = n_blk * BN + wg * 128;
        __nv_bfloat16* yrow = y + static_cast<long>(row) * N;
#pragma unroll
        for (int j = 0; j < 128; j += 8) {
          const int n = n0 + j;
          if (n < N) {
            uint32_t packed[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              __nv_bfloat162 h = __floats2bfloat162_rn(static_cast<float>(sums[j + 2 * t]),
                                                       static_cast<float>(sums[j + 2 * t + 1]));
              packed[t] = *reinterpret_cast<uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(yrow + n) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          }
        }
      }
      if (!FP && row < M) {
        const float ts = tscale[row];
        const int n0 = n_blk * BN + wg * 128;
        __nv_bfloat16* yrow = y + static_cast<long>(row) * N;
#pragma unroll
        for (int j = 0; j < 128; j += 8) {
          const int n = n0 + j;
          if (n < N) {
            const float4 r0 = __ldg(reinterpret_cast<const float4*>(rscale + n));
            const float4 r1 = __ldg(reinterpret_cast<const float4*>(rscale + n + 4));
            const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
            uint32_t packed[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const float f0 = __fmul_rn(
                  __fmul_rn(__int2float_rn(static_cast<int>(sums[j + 2 * t])), ts), rr[2 * t]);
              const float f1 = __fmul_rn(
                  __fmul_rn(__int2float_rn(static_cast<int>(sums[j + 2 * t + 1])), ts),
                  rr[2 * t + 1]);
              __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
              packed[t] = *reinterpret_cast<uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(yrow + n) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            if (acc_out != nullptr) {
              int4* ap = reinterpret_cast<int4*>(acc_out + static_cast<long>(row) * N + n);
              ap[0] = make_int4(static_cast<int>(sums[j]), static_cast<int>(sums[j + 1]),
                                static_cast<int>(sums[j + 2]), static_cast<int>(sums[j + 3]));
              ap[1] = make_int4(static_cast<int>(sums[j + 4]), static_cast<int>(sums[j + 5]),
                                static_cast<int>(sums[j + 6]), static_cast<int>(sums[j + 7]));
            }
          }
        }
      }
    }
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) {
    // the even CTA's MMAs (which read this CTA's shared memory and write its
    // tensor memory) are done, and both epilogues have read their rows
    ptx::cluster_sync();
    if (warp == 2) {
      ptx::tc_fence_after();
      ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
    }
  } else if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// SPLIT = false: one unit per tile (no slice arithmetic in the loops);
// SPLIT = true: S K slices per tile, partial sums to `part`.
template <bool SPLIT, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_i8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const float* __restrict__ tscale, const float* __restrict__ rscale, int M,
                   int N, int K, __nv_bfloat16* __restrict__ y, int32_t* __restrict__ acc_out,
                   int S, int full, int32_t* __restrict__ part) {
  gemm_body<false, SPLIT, PAIR>(tmA, tmB, tscale, rscale, M, N, K, y, acc_out, S, full, part);
}

template <bool SPLIT, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_f16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const float* __restrict__ xs, int M, int N, int K,
                    __nv_bfloat16* __restrict__ y, int S, int full, float* __restrict__ part) {
  gemm_body<true, SPLIT, PAIR>(tmA, tmB, xs, nullptr, M, N, K, y, nullptr, S, full, part);
}

// After a split GEMM: for every split tile (tiles full .. tiles-1), add its
// S pieces in slice order and finish the output -- int8 path: the exact sum,
// rescaled (and stored to acc when given); fp16 path: bf16 of the fp32 sum.
// One thread per 8 outputs of a tile row.
template <bool FP>
__global__ void __launch_bounds__(256)
    split_finalize_kernel(const void* __restrict__ part, int S, int full, int n_split,
                          int m_blocks, int tm, int M, int N, const float* __restrict__ tscale,
                          const float* __restrict__ rscale, __nv_bfloat16* __restrict__ y,
                          int32_t* __restrict__ acc_out) {
  pdl_launch_dependents();
  const long i = static_cast<long>(blockIdx.x) * 256 + threadIdx.x;
  constexpr int PER_ROW = BN / 8;
  const long st = i / (static_cast<long>(tm) * PER_ROW);   // tiles of tm token rows
  const int r = static_cast<int>((i / PER_ROW) % tm);
  const int c8 = static_cast<int>(i % PER_ROW);
  pdl_wait();   // the GEMM's pieces
  if (st >= n_split) return;
  const int tile = full + static_cast<int>(st);
  const int n_blk = tile / m_blocks, m_blk = tile % m_blocks;
  const long row = static_cast<long>(m_blk) * tm + r;
  const int n = n_blk * BN + c8 * 8;
  if (row >= M || n >= N) return;
  typename std::conditional<FP, float, int>::type a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  // four slices' loads in flight before their adds (in slice order)
  for (int sl0 = 0; sl0 < S; sl0 += 4) {
    int4 v[4][2];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (sl0 + u < S) {
        const int4* p = static_cast<const int4*>(part) +
                        (((st * S + sl0 + u) * tm + r) * BN + c8 * 8) / 4;
        v[u][0] = __ldcs(p);
        v[u][1] = __ldcs(p + 1);
      }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (sl0 + u < S) {
        const int w[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w,
                          v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if constexpr (FP)
            a[i] = __fadd_rn(a[i], __int_as_float(w[i]));
          else
            a[i] += w[i];
        }
      }
  }
  uint32_t out[4];
  if constexpr (FP) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      __nv_bfloat162 h = __floats2bfloat162_rn(a[2 * t], a[2 * t + 1]);
      out[t] = *reinterpret_cast<uint32_t*>(&h);
    }
  } else {
    const float4 r0 = __ldg(reinterpret_cast<const float4*>(rscale + n));
    const float4 r1 = __ldg(reinterpret_cast<const float4*>(rscale + n + 4));
    const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    const float ts = tscale[row];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float f0 = __fmul_rn(__fmul_rn(__int2float_rn(a[2 * t]), ts), rr[2 * t]);
      const float f1 = __fmul_rn(__fmul_rn(__int2float_rn(a[2 * t + 1]), ts), rr[2 * t + 1]);
      __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
      out[t] = *reinterpret_cast<uint32_t*>(&h);
    }
    if (acc_out != nullptr) {
      int4* ap = reinterpret_cast<int4*>(acc_out + row * N + n);
      ap[0] = make_int4(a[0], a[1], a[2], a[3]);
      ap[1] = make_int4(a[4], a[5], a[6], a[7]);
    }
  }
  *reinterpret_cast<uint4*>(y + row * N + n) = make_uint4(out[0], out[1], out[2], out[3]);
}


// ---------------------------------------------------------------------------
// The same int8 GEMM straight from the decode's 2-bit packed weights: no
// W_int8 is held in memory (section 6 of the page measured the run-time
// 2-bit -> int8 expansion as 31 of 83 ms per step; here it runs in shared
// memory, beside the tensor cores).
//
// Tile: 128 tokens (MMA M) x 256 weight rows (MMA N: half of a 512-row unit
// of the packed format), 64-wide K stages -- the instruction shape of the
// kernel above, since a tcgen05.mma costs about the same time at any N up to
// 256.  Per 128-wide group the producer bulk-copies the 8 KB of codes of the
// tile's 256 rows into a code ring and TMA-loads the tokens; four expansion
// warps turn the codes into the exact int8 weight values code * q[n, g],
// held in fp16 and written in the 128-byte-swizzled K-major layout the MMA
// reads (a field masked in place reads u * 4^e * 2^-24, u = code + 1; times
// 2^(15 - 2e), then fma with 512 q and -q, gives code * q; all exact).  MMA,
// per-1024 chunk int32 conversion and epilogue are those of the kernel above.
// Warp roles: 0 producer, 1 MMA issuer, 2 TMEM allocator, 3 relay (pairs;
// else idle), 4-11 epilogue, 12-15 expansion.
//
// Two tile orientations (template WM).  WM = false: tokens on the MMA's M
// side (128 per tile) and weight rows on its N side (256), for M <= 128
// (one token block).  WM = true, for larger M: 128 weight rows on the M side
// and 256 tokens on the N side, so each expanded weight value feeds 256
// tokens instead of 128 -- half the expansion work and half the shared-
// memory writes per MMA -- while the MMA shape, the stage size (A 16 KB, B
// 32 KB) and the TMEM buffers stay the same; the accumulator's lanes are
// then weight rows and its columns tokens.
//
// WM = true runs in CTA pairs (PAIR, clusters of two, tcgen05 cta_group::2):
// a pair tile is 256 weight rows x 256 tokens, each CTA expanding its own 128
// weight rows and loading its own 128 tokens, and the even CTA issuing one
// 256 x 256 x 16 MMA per k16 step that reads both CTAs' shared memory and
// writes both CTAs' tensor memory (each CTA's 128 rows, all 256 token
// columns).  The tensor cores' operand reads and the token copies per SM are
// then two thirds of a single CTA's for the same work, which matters because
// shared-memory bandwidth, not the tensor pipe, bounds the single-CTA kernel:
// per SM and 64-k stage it carries the 48 KB the MMA reads, the 32 KB of
// tokens TMA writes, the expansion's 16 KB of stores and the codes.  Each
// CTA's warp 3 relays "stage s holds my tokens and expanded weights" to the
// even CTA's pfull[s]; the MMA commits arrive (multicast) on both CTAs'
// stage-free and accumulator-full barriers; both CTAs' epilogue warps
// release an accumulator buffer on the even CTA's dempty.  (The even CTA's
// issuer waiting on its own stage's barriers directly, beside the odd CTA's
// relay, measured slower: 480 -> 547 us at gate/up M = 2048.)  The 512 threads launch with 128 registers each;
// the epilogue's 128 int32 sums per thread need more, so the warpgroups
// re-split the block's registers with setmaxnreg (control 48, epilogue 168,
// expansion 120 per thread); the launcher refuses to launch unless the kernel
// was built with exactly 128 registers per thread, so the split always fits.
constexpr int PBN = 256;                 // weight rows per tile (WM = false)
constexpr int PUNIT_BYTES = 17408;       // one 512-row x 128-k unit of the packed format
constexpr int PCODE_BYTES = 8192;        // code ring slot: the codes of up to 256 rows of a unit
// tokens and weight rows per tile, and the bytes of a tile's codes per group
template <bool WM> constexpr int p_tok() { return WM ? 256 : BM; }
template <bool WM> constexpr int p_wrows() { return WM ? 128 : PBN; }
template <bool WM> constexpr int p_code_bytes() { return p_wrows<WM>() * 32; }
constexpr int PSTAGES = 4;
constexpr int PCSTAGES = 4;
constexpr int PA_BYTES = BM * BK * 2;    // tokens
constexpr int PB_BYTES = PBN * BK * 2;   // expanded weights
constexpr int PSTAGE_BYTES = PA_BYTES + PB_BYTES;
constexpr int PSTAGES_PAIR = 6;
constexpr int PSTAGE_BYTES_PAIR = PA_BYTES + PB_BYTES / 2;   // 128 weight rows + 128 tokens
constexpr int P_THREADS = 512;
constexpr int P_LAUNCH_REGS = 128;
constexpr int P_REGS_CONTROL = 48, P_REGS_EPILOGUE = 168, P_REGS_EXPAND = 120;
constexpr size_t PSMEM_BYTES =
    static_cast<size_t>(PSTAGES) * PSTAGE_BYTES + PCSTAGES * PCODE_BYTES + 1024 + 512;
static_assert(PSMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(PSTAGE_BYTES % 1024 == 0 && PA_BYTES % 1024 == 0, "stage alignment");
static_assert(PSTAGES_PAIR * PSTAGE_BYTES_PAIR <= PSTAGES * PSTAGE_BYTES,
              "pair stages fit the single-CTA stage area");
static_assert(128 * P_REGS_CONTROL + 256 * P_REGS_EPILOGUE + 128 * P_REGS_EXPAND <=
                  P_THREADS * P_LAUNCH_REGS,
              "register split exceeds the block's launch allocation");

template <int R>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}

template <bool WM, bool PAIR>
__global__ void __launch_bounds__(P_THREADS, 1)
    gemm_packed_kernel(const __grid_constant__ CUtensorMap tmA, const uint8_t* __restrict__ packed,
                       const int8_t* __restrict__ q, const float* __restrict__ tscale,
                       const float* __restrict__ rscale, int M, int N, int K,
                       __nv_bfloat16* __restrict__ y, int32_t* __restrict__ acc_out, int S,
                       int full, int32_t* __restrict__ part) {
  // a pair's stage holds 128 tokens (16 KB) instead of 256, so six stages
  // fit where a single CTA has four
  constexpr int NST = PAIR ? PSTAGES_PAIR : PSTAGES;
  constexpr int SGB = PAIR ? PSTAGE_BYTES_PAIR : PSTAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* scode = smem + NST * SGB;
  uint64_t* afull = reinterpret_cast<uint64_t*>(scode + PCSTAGES * PCODE_BYTES);
  uint64_t* wfull = afull + NST;
  uint64_t* empty = wfull + NST;
  uint64_t* cfull = empty + NST;
  uint64_t* cempty = cfull + PCSTAGES;
  uint64_t* dfull = cempty + PCSTAGES;
  uint64_t* dempty = dfull + 2;
  uint64_t* done = dempty + 2;
  uint64_t* pfull = done + 1;   // (pairs) both CTAs' stage ready, in the even CTA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pfull + NST);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  static_assert(!PAIR || WM, "CTA pairs split 256 weight rows x 256 tokens");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int TOK = p_tok<WM>(), WROWS = p_wrows<WM>(), CODE_BYTES = p_code_bytes<WM>();
  // In a pair, each CTA loads half of the tile's tokens (the MMA's N side) and
  // expands its own 128 weight rows (half of the M side).
  constexpr int TOK_CTA = PAIR ? TOK / 2 : TOK;
  constexpr int CTAS = PAIR ? 2 : 1;
  const int rank = PAIR ? static_cast<int>(ptx::cluster_ctarank()) : 0;
  const int team = PAIR ? static_cast<int>(ptx::cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int teams = PAIR ? static_cast<int>(ptx::cluster_count_x()) : static_cast<int>(gridDim.x);
  // stage layout: MMA operand A (16 KB) at offset 0, B (32 KB) after it; the
  // tokens are A for WM = false and B for WM = true
  constexpr uint32_t TOK_OFF = WM ? PA_BYTES : 0, W_OFF = WM ? 0 : PA_BYTES;
  constexpr uint32_t TOK_BYTES = TOK_CTA * BK * 2;
  const int G = K / kGroup;
  // stage s free again (in a pair, the even CTA's MMA commit completes it;
  // the ring keeps these waits off the critical path, so they suspend)
  auto empty_wait = [&](uint64_t* bar, uint32_t parity) {
    return ptx::mbar_wait(bar, parity, abort_flag, WAIT_LIMIT);
  };
  const int m_blocks = (M + TOK - 1) / TOK;   // token blocks (fastest in the tile order)
  const int tiles = m_blocks * ((N + CTAS * WROWS - 1) / (CTAS * WROWS));
  // units: the first `full` tiles whole, then every later tile in S K
  // slices of whole 128-groups (S = 1: all whole)
  const int units = full + (tiles - full) * S;
  // the tile and the group range [g0, g1) of a unit; the MMA accumulates it
  // in pieces that end at every 1024-chunk boundary (and at g1), so each
  // fp32 partial stays exact
  auto unit_of = [&](int u, int& tile, int& g0, int& g1) {
    if (u < full) {
      tile = u;
      g0 = 0;
      g1 = G;
    } else {
      const int v = u - full;
      tile = full + v / S;
      const int sl = v % S;
      g0 = sl * G / S;
      g1 = (sl + 1) * G / S;
    }
  };
  auto piece_end = [&](int gp, int g1) {
    const int e = (gp / 8 + 1) * 8;
    return e < g1 ? e : g1;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      ptx::mbar_init(&afull[s], 1);
      ptx::mbar_init(&wfull[s], 4);   // one arrival per expansion warp
      ptx::mbar_init(&empty[s], 1);
    }
    for (int c = 0; c < PCSTAGES; ++c) {
      ptx::mbar_init(&cfull[c], 1);
      ptx::mbar_init(&cempty[c], 4);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&dfull[b], 1);
      ptx::mbar_init(&dempty[b], 8 * CTAS);   // one arrival per epilogue warp (of both CTAs)
    }
    ptx::mbar_init(done, 1);
    for (int s = 0; s < NST; ++s) ptx::mbar_init(&pfull[s], 2);   // one relay per CTA
    *abort_flag = 0;
    ptx::mbar_fence_init();
  }
  if (warp == 2) {
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(tmem_slot, TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(tmem_slot, TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) ptx::prefetch_tmap(&tmA);
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) ptx::cluster_sync();   // both CTAs' barriers exist before any remote arrival
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_wait();   // xq / tscale come from the previous kernel
  pdl_launch_dependents();

  if (warp < 4) {
    regs_dec<P_REGS_CONTROL>();
    if (warp == 0 && lane == 0) {
      // ---------------- producer: code groups (bulk) and token stages (TMA)
      int s = 0, c = 0;
      uint32_t ph = 0, cph = 0;
      long a_issued = 0, c_issued = 0;
      bool ok = true;
      for (int u = team; u < units && ok; u += teams) {
        int tile, g0, g1;
        unit_of(u, tile, g0, g1);
        const int n_blk = (tile / m_blocks) * CTAS + rank, m_blk = tile % m_blocks;
        constexpr int PER_UNIT = 512 / WROWS;   // weight blocks per 512-row unit
        const uint8_t* wsrc = packed + static_cast<size_t>(n_blk / PER_UNIT) * G * PUNIT_BYTES +
                              (n_blk % PER_UNIT) * CODE_BYTES;
        for (int g = g0; g < g1 && ok; ++g) {
          if (!ptx::mbar_wait(&cempty[c], cph ^ 1u, abort_flag, WAIT_LIMIT)) {
            if (!*abort_flag) fail(abort_flag, ERR_PRODUCER);
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&cfull[c], CODE_BYTES);
          ptx::bulk_load(scode + c * PCODE_BYTES, wsrc + static_cast<size_t>(g) * PUNIT_BYTES,
                         CODE_BYTES, &cfull[c]);
          ++c_issued;
          if (++c == PCSTAGES) {
            c = 0;
            cph ^= 1u;
          }
          for (int h = 0; h < 2; ++h) {
            if (!empty_wait(&empty[s], ph ^ 1u)) {
              if (!*abort_flag) fail(abort_flag, ERR_PRODUCER);
              ok = false;
              break;
            }
            ptx::mbar_arrive_expect_tx(&afull[s], TOK_BYTES);
            ptx::tma_load_2d(smem + s * SGB + TOK_OFF, &tmA, &afull[s],
                             g * kGroup + h * BK, m_blk * TOK + rank * TOK_CTA);
            ++a_issued;
            if (++s == NST) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // let the copies still in flight land before the CTA exits
        long back = a_issued < NST ? a_issued : NST;
        for (long i = 0; i < back; ++i) {
          if (--s < 0) {
            s = NST - 1;
            ph ^= 1u;
          }
          if (!ptx::mbar_wait_bounded(&afull[s], ph, WAIT_LIMIT)) atomicOr(&g_gemm_error, ERR_DRAIN);
        }
        back = c_issued < PCSTAGES ? c_issued : PCSTAGES;
        for (long i = 0; i < back; ++i) {
          if (--c < 0) {
            c = PCSTAGES - 1;
            cph ^= 1u;
          }
          if (!ptx::mbar_wait_bounded(&cfull[c], cph, WAIT_LIMIT)) atomicOr(&g_gemm_error, ERR_DRAIN);
        }
      }
    } else if (warp == 1 && lane == 0 && rank == 0) {
      // ---------------- MMA issuer (one thread; in a pair, the even CTA's, for
      // both: 256 x 256 x 16 MMAs whose commits arrive in both CTAs)
      int s = 0;
      uint32_t ph = 0;
      uint32_t cc = 0;
      bool ok = true;
      for (int u = team; u < units && ok; u += teams) {
        int tile, g0, g1;
        unit_of(u, tile, g0, g1);
        for (int gp = g0; gp < g1 && ok; gp = piece_end(gp, g1), ++cc) {
          const uint32_t buf = cc & 1u, dph = (cc >> 1) & 1u;
          if (!ptx::mbar_wait(&dempty[buf], dph ^ 1u, abort_flag, WAIT_LIMIT)) {
            if (!*abort_flag) fail(abort_flag, ERR_MMA);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem + buf * BN;
          const int n_stages = 2 * (piece_end(gp, g1) - gp);
          for (int j = 0; j < n_stages; ++j) {
            const bool ready =
                PAIR ? ptx::mbar_wait(&pfull[s], ph, abort_flag, WAIT_LIMIT)
                     : (ptx::mbar_wait(&afull[s], ph, abort_flag, WAIT_LIMIT) &&
                        ptx::mbar_wait(&wfull[s], ph, abort_flag, WAIT_LIMIT));
            if (!ready) {
              if (!*abort_flag) fail(abort_flag, ERR_MMA);
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t a0 = ptx::sw128_kmajor_desc(ptx::smem_u32(smem + s * SGB));
            const uint64_t b0 =
                ptx::sw128_kmajor_desc(ptx::smem_u32(smem + s * SGB + PA_BYTES));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              if constexpr (PAIR)
                ptx::mma_f16_ss_pair(d_tmem, a0 + 2u * kk, b0 + 2u * kk, IDESC_PAIR,
                                     (j > 0 || kk > 0) ? 1u : 0u);
              else
                ptx::mma_f16_ss(d_tmem, a0 + 2u * kk, b0 + 2u * kk, IDESC,
                                (j > 0 || kk > 0) ? 1u : 0u);
            }
            if constexpr (PAIR)
              ptx::mma_commit_pair(&empty[s], 0x3);
            else
              ptx::mma_commit(&empty[s]);
            if (++s == NST) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (ok) {
            if constexpr (PAIR)
              ptx::mma_commit_pair(&dfull[buf], 0x3);
            else
              ptx::mma_commit(&dfull[buf]);
          }
        }
      }
      if constexpr (PAIR)
        ptx::mma_commit_pair(done, 0x3);
      else
        ptx::mma_commit(done);
      if (!ptx::mbar_wait_bounded(done, 0, WAIT_LIMIT)) atomicOr(&g_gemm_error, ERR_DRAIN);
    } else if (PAIR && warp == 3 && lane == 0) {
      // ---------------- relay (pairs): once this CTA's stage holds its tokens
      // and its expanded weights, one arrival on the even CTA's pfull[s]
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      const uint32_t pf = ptx::mapa_shared(pfull, 0);
      for (int u = team; u < units && ok; u += teams) {
        int tile, g0, g1;
        unit_of(u, tile, g0, g1);
        for (int j = 0; j < 2 * (g1 - g0); ++j) {
          if (!ptx::mbar_wait(&afull[s], ph, abort_flag, WAIT_LIMIT) ||
              !ptx::mbar_wait(&wfull[s], ph, abort_flag, WAIT_LIMIT)) {
            if (!*abort_flag) fail(abort_flag, ERR_MMA);
            ok = false;
            break;
          }
          ptx::mbar_arrive_cluster(pf + 8u * static_cast<uint32_t>(s));
          if (++s == NST) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp < 12) {
    regs_inc<P_REGS_EPILOGUE>();
    // ---------------- epilogue: warpgroup wg owns columns [128 wg, 128 wg + 128)
    const int wg = (warp - 4) >> 2;
    const int qd = warp & 3;   // TMEM lane quarter accessible to this warp
    uint32_t cc = 0;
    bool ok = true;
    for (int u = team; u < units && ok; u += teams) {
      int tile, g0, g1;
      unit_of(u, tile, g0, g1);
      const int n_blk = (tile / m_blocks) * CTAS + rank, m_blk = tile % m_blocks;
      int32_t sums[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) sums[i] = 0;
      for (int gp = g0; gp < g1; gp = piece_end(gp, g1), ++cc) {
        const uint32_t buf = cc & 1u, dph = (cc >> 1) & 1u;
        const bool full = ptx::mbar_wait_warp(&dfull[buf], dph, abort_flag, WAIT_LIMIT);
        if (!full) {
          if (!*abort_flag) fail(abort_flag, ERR_EPILOGUE);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int piece = 0; piece < 4; ++piece) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * qd) << 16) + buf * BN +
                                      wg * 128 + piece * 32,
                                  v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            sums[piece * 32 + i] += __float2int_rn(__uint_as_float(v[i]));   // exact integers
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            ptx::mbar_arrive_cluster(ptx::mapa_shared(&dempty[buf], 0));
          else
            ptx::mbar_arrive(&dempty[buf]);
        }
      }
      if (!ok) break;
      if constexpr (WM) {
        // lanes are weight rows, columns tokens: per token, the warp's 32
        // lanes write 32 consecutive outputs of y (or of the slice's plane)
        const int n = n_blk * WROWS + 32 * qd + lane;
        const int t0 = m_blk * TOK + wg * 128;
        if (n < N) {
          if (u >= full) {
            // one K slice of a split tile: its exact partial sums go to the
            // slice's piece [256 tokens][256 weight rows] of `part` (this
            // CTA's 128 rows), which the finishing kernel adds
            int32_t* pcol = part + (static_cast<long>(u - full) * TOK + wg * 128) * (CTAS * WROWS) +
                            rank * WROWS + 32 * qd + lane;
#pragma unroll
            for (int j = 0; j < 128; ++j) pcol[j * (CTAS * WROWS)] = sums[j];
          } else {
            const float rs = rscale[n];
#pragma unroll
            for (int j = 0; j < 128; ++j) {
              const int t = t0 + j;
              if (t < M) {
                const float f =
                    __fmul_rn(__fmul_rn(__int2float_rn(sums[j]), __ldg(tscale + t)), rs);
                y[static_cast<long>(t) * N + n] = __float2bfloat16_rn(f);
                if (acc_out != nullptr) acc_out[static_cast<long>(t) * N + n] = sums[j];
              }
            }
          }
        }
        continue;
      }
      const int row = m_blk * BM + 32 * qd + lane;
      if (u >= full) {
        // one K slice of the tile: store its exact partial sums in the
        // slice's plane of the workspace; the rescale kernel adds the planes
        if (row < M) {
          const int n0 = n_blk * PBN + wg * 128;
          int32_t* prow = part + (static_cast<long>(u % S) * M + row) * N + n0;
#pragma unroll
          for (int j = 0; j < 128; j += 8)
            if (n0 + j < N) {
              int4* pp = reinterpret_cast<int4*>(prow + j);
              pp[0] = make_int4(sums[j], sums[j + 1], sums[j + 2], sums[j + 3]);
              pp[1] = make_int4(sums[j + 4], sums[j + 5], sums[j + 6], sums[j + 7]);
            }
        }
        continue;
      }
      if (row < M) {
        const float ts = tscale[row];
        const int n0 = n_blk * PBN + wg * 128;
        __nv_bfloat16* yrow = y + static_cast<long>(row) * N;
#pragma unroll
        for (int j = 0; j < 128; j += 8) {
          const int n = n0 + j;
          if (n < N) {
            const float4 r0 = __ldg(reinterpret_cast<const float4*>(rscale + n));
            const float4 r1 = __ldg(reinterpret_cast<const float4*>(rscale + n + 4));
            const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
            uint32_t packed_y[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const float f0 = __fmul_rn(__fmul_rn(__int2float_rn(sums[j + 2 * t]), ts), rr[2 * t]);
              const float f1 =
                  __fmul_rn(__fmul_rn(__int2float_rn(sums[j + 2 * t + 1]), ts), rr[2 * t + 1]);
              __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
              packed_y[t] = *reinterpret_cast<uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(yrow + n) =
                make_uint4(packed_y[0], packed_y[1], packed_y[2], packed_y[3]);
            if (acc_out != nullptr) {
              int4* ap = reinterpret_cast<int4*>(acc_out + static_cast<long>(row) * N + n);
              ap[0] = make_int4(sums[j], sums[j + 1], sums[j + 2], sums[j + 3]);
              ap[1] = make_int4(sums[j + 4], sums[j + 5], sums[j + 6], sums[j + 7]);
            }
          }
        }
      }
    }
    __syncwarp();
  } else {
    regs_dec<P_REGS_EXPAND>();
    // ---------------- expansion: warp xw owns tiles xw + 4 u (u = 0..3) of the
    // 16 16-row tiles of the half unit; lane = slot L = 4 r + c of the packed
    // format
    const int xw = warp - 12;
    const int r = lane >> 2;
    constexpr int UPW = WROWS / 64;   // tiles of 16 rows per expansion warp
    // The expanded values of a k16 step leave in one stmatrix.x4: register p
    // (row parity p % 2, 8-column half p / 2) is matrix p, whose 16-byte rows
    // lanes 8 p .. 8 p + 7 address.  This lane addresses row 16 xw + ri +
    // 8 (mi % 2) of its tile, 8-column half mi / 2 (u adds 64 rows).
    const int mi = lane >> 3, ri = lane & 7;
    const uint32_t row_off = static_cast<uint32_t>(W_OFF + (16 * xw + ri + 8 * (mi & 1)) * 128);
    uint32_t xo[4];   // the step jl's 16-byte chunk 2 jl + mi / 2 in the 128-byte swizzle
#pragma unroll
    for (int jl = 0; jl < 4; ++jl) xo[jl] = static_cast<uint32_t>(((2 * jl + (mi >> 1)) ^ ri) << 4);
    const uint32_t smem_base = ptx::smem_u32(smem);
    int s = 0, c = 0;
    uint32_t ph = 0, cph = 0;
    bool ok = true;
    for (int unit = team; unit < units && ok; unit += teams) {
      int tile, g0, g1;
      unit_of(unit, tile, g0, g1);
      const int n_blk = (tile / m_blocks) * CTAS + rank;
      // q of the thread's 2 UPW rows (slots u, row parities par); rows past N read row 0
      const int8_t* qp[UPW][2];
      bool qv_ok[UPW][2];
#pragma unroll
      for (int u = 0; u < UPW; ++u)
#pragma unroll
        for (int par = 0; par < 2; ++par) {
          const int n = n_blk * WROWS + 16 * (xw + 4 * u) + r + 8 * par;
          qv_ok[u][par] = n < N;
          qp[u][par] = q + static_cast<long>(n < N ? n : 0) * G;
        }
      for (int g = g0; g < g1 && ok; ++g) {
        int qv[UPW][2];
#pragma unroll
        for (int u = 0; u < UPW; ++u)
#pragma unroll
          for (int par = 0; par < 2; ++par)
            qv[u][par] = qv_ok[u][par] ? static_cast<int>(__ldg(qp[u][par] + g)) : 0;
        if (!ptx::mbar_wait(&cfull[c], cph, abort_flag, WAIT_LIMIT)) {
          if (!*abort_flag) fail(abort_flag, ERR_EXPAND);
          ok = false;
          break;
        }
        uint4 wv[UPW];
#pragma unroll
        for (int u = 0; u < UPW; ++u)
          wv[u] = *reinterpret_cast<const uint4*>(scode + c * PCODE_BYTES + 512 * (xw + 4 * u) +
                                                  16 * lane);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&cempty[c]);
        if (++c == PCSTAGES) {
          c = 0;
          cph ^= 1u;
        }
        // code * q from the field u = code + 1 read as u * 4^e * 2^-24 (one
        // AND): times 2^(15 - 2e) it is u * 2^-9, and fma(u * 2^-9, 512 q, -q)
        // = (u - 1) q; every step exact in fp16 (512 q <= 65024)
        uint32_t q512[UPW][2], qneg[UPW][2];
#pragma unroll
        for (int u = 0; u < UPW; ++u)
#pragma unroll
          for (int par = 0; par < 2; ++par) {
            __half2 a2 = __half2half2(__float2half_rn(512.0f * static_cast<float>(qv[u][par])));
            __half2 b2 = __half2half2(__float2half_rn(-static_cast<float>(qv[u][par])));
            q512[u][par] = *reinterpret_cast<uint32_t*>(&a2);
            qneg[u][par] = *reinterpret_cast<uint32_t*>(&b2);
          }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!empty_wait(&empty[s], ph ^ 1u)) {
            if (!*abort_flag) fail(abort_flag, ERR_EXPAND);
            ok = false;
            break;
          }
          const uint32_t base = smem_base + s * SGB + row_off;
          // this stage holds k16 steps j = 4h .. 4h + 3 of the group; word p is
          // register p (row parity p % 2, 8-column half p / 2)
#pragma unroll
          for (int jl = 0; jl < 4; ++jl) {
            const int j = 4 * h + jl;
            const int e = j < 6 ? j : j - 6;
            const uint32_t mask = 0x00030003u << (2 * e);
            const uint32_t mul = 0x00010001u * static_cast<uint32_t>((30 - 2 * e) << 10);   // 2^(15-2e)
#pragma unroll
            for (int u = 0; u < UPW; ++u) {
              const uint32_t w4[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
              uint32_t v[4];
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                const uint32_t f = (j < 6 ? w4[p] : w4[p] >> 12) & mask;
                v[p] = ptx::fma_f16x2(ptx::mul_f16x2(f, mul), q512[u][p & 1], qneg[u][p & 1]);
              }
              ptx::stsm_x4(base + xo[jl] + 8192u * u, v[0], v[1], v[2], v[3]);
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&wfull[s]);
          if (++s == NST) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) {
    // the even CTA's MMAs (which read this CTA's shared memory and write its
    // tensor memory) are done, and both epilogues have read their columns
    ptx::cluster_sync();
    if (warp == 2) {
      ptx::tc_fence_after();
      ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
    }
  } else if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// After a split-K packed GEMM: acc = the sum of the S slices' exact partial
// sums (int32, any order gives the same integer), then y = bf16_rn((acc *
// tscale[m]) * rscale[n]) with the epilogue's arithmetic; one thread per 8
// outputs of a row (N % 16 == 0).
constexpr int FIN_THREADS = 256;
__global__ void __launch_bounds__(FIN_THREADS)
    packed_finalize_kernel(const int32_t* __restrict__ part, int S,
                           const float* __restrict__ tscale, const float* __restrict__ rscale,
                           int M, int N, __nv_bfloat16* __restrict__ y,
                           int32_t* __restrict__ acc_out) {
  pdl_launch_dependents();
  const long i = static_cast<long>(blockIdx.x) * FIN_THREADS + threadIdx.x;
  const long per_row = N / 8;
  const long row = i / per_row;
  const int n = static_cast<int>(i % per_row) * 8;
  pdl_wait();   // the GEMM's partial sums
  if (row >= M) return;
  int aa[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int sl0 = 0; sl0 < S; sl0 += 4) {   // four planes' loads in flight
    int4 v[4][2];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (sl0 + u < S) {
        const int4* p = reinterpret_cast<const int4*>(
            part + (static_cast<long>(sl0 + u) * M + row) * N + n);
        v[u][0] = __ldcs(p);
        v[u][1] = __ldcs(p + 1);
      }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (sl0 + u < S) {
        aa[0] += v[u][0].x; aa[1] += v[u][0].y; aa[2] += v[u][0].z; aa[3] += v[u][0].w;
        aa[4] += v[u][1].x; aa[5] += v[u][1].y; aa[6] += v[u][1].z; aa[7] += v[u][1].w;
      }
  }
  const float4 r0 = __ldg(reinterpret_cast<const float4*>(rscale + n));
  const float4 r1 = __ldg(reinterpret_cast<const float4*>(rscale + n + 4));
  const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
  const float ts = tscale[row];
  uint32_t out[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float f0 = __fmul_rn(__fmul_rn(__int2float_rn(aa[2 * t]), ts), rr[2 * t]);
    const float f1 = __fmul_rn(__fmul_rn(__int2float_rn(aa[2 * t + 1]), ts), rr[2 * t + 1]);
    __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
    out[t] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(y + row * N + n) = make_uint4(out[0], out[1], out[2], out[3]);
  if (acc_out != nullptr) {
    int4* ap = reinterpret_cast<int4*>(acc_out + row * N + n);
    ap[0] = make_int4(aa[0], aa[1], aa[2], aa[3]);
    ap[1] = make_int4(aa[4], aa[5], aa[6], aa[7]);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (f == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<EncodeTiledFn>(p);
      fn.store(f, std::memory_order_release);
    }
  }
  return f;
}

// 2-D map over a row-major fp16 [rows][K] matrix, boxes of 64 K x box_rows rows.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 152;
  return n;
}

// Token rows of a dense GEMM tile: 128 for one CTA, 256 for a CTA pair
// (above one 128-token block).
long dense_tile_rows(int64_t M) { return M > BM ? 2 * BM : BM; }

}  // namespace

// How the expanded-weight GEMMs cut their work: the first `full` tiles whole,
// the others (the last, partial wave, or all tiles) in S slices of whole
// 1024-chunks.  The plan with the least estimated time wins: waves of units
// x chunks per unit x one tile-chunk (measured on GB300: ~5.9 us for a
// CTA's 128 x 256 tile, ~5.2 us for a pair's 256 x 256), plus writing and
// reading the partial pieces and a launch for the finishing kernel; a split
// has to win by 1 %.  (Gate/up at M = 2048, 1088 pair tiles on 76 pairs:
// the last wave's 24 tiles in 3 slices, 387 -> 380 us.)
DensePlan dense_plan(int64_t M, int64_t N, int64_t K) {
  // a team is one SM's CTA, or (M > 128) a CTA pair with twice the tile
  const long tm = dense_tile_rows(M);
  const long tiles = ((M + tm - 1) / tm) * ((N + BN - 1) / BN);
  const long sms = tm == BM ? sm_count() : sm_count() / 2;
  const long chunks = K / KCHUNK;
  const double t_chunk = tm == BM ? 5.9e-6 : 5.2e-6, bw = 6.0e12, t_launch = 3e-6;
  const double piece_bytes = static_cast<double>(tm) * BN * 4;
  auto cost = [&](long full, long S) {
    const long split = tiles - full;
    const long per_cta_whole = (full + sms - 1) / sms;
    const long per_cta_split = (split * S + sms - 1) / sms;
    double t = (static_cast<double>(per_cta_whole) * chunks +
                static_cast<double>(per_cta_split) * ((chunks + S - 1) / S)) * t_chunk;
    if (S > 1) t += (2.0 * split * S * piece_bytes + 2.0 * split * tm * BN) / bw + t_launch;
    return t;
  };
  DensePlan best{1, static_cast<int>(tiles)};
  double best_t = cost(tiles, 1);
  auto consider = [&](long full, long S) {
    if (S < 2 || S > chunks || full >= tiles) return;
    const double t = cost(full, S);
    if (t < 0.99 * best_t) {
      best_t = t;
      best = DensePlan{static_cast<int>(S), static_cast<int>(full)};
    }
  };
  for (long S = 2; S <= chunks && S <= 32; ++S) consider(0, S);      // every tile split
  const long full = tiles / sms * sms;                                 // whole waves kept whole
  if (full > 0 && full < tiles) {
    const long tail = tiles - full;
    for (long S = 2; S <= chunks && S <= 32; ++S) consider(full, S);   // the last wave split
    (void)tail;
  }
  return best;
}

size_t gemm_dense_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const DensePlan p = dense_plan(M, N, K);
  if (p.S == 1) return 0;
  const long tm = dense_tile_rows(M);
  const long tiles = ((M + tm - 1) / tm) * ((N + BN - 1) / BN);
  return static_cast<size_t>(tiles - p.full) * p.S * tm * BN * 4;
}

int dense_splits(int64_t M, int64_t N, int64_t K) { return dense_plan(M, N, K).S; }

namespace {
// The plan to use: dense_plan's when the caller gave a large enough
// workspace, else everything whole.
DensePlan usable_plan(int64_t M, int64_t N, int64_t K, const void* ws, size_t ws_bytes) {
  const DensePlan p = dense_plan(M, N, K);
  const long tm = dense_tile_rows(M);
  const long tiles = ((M + tm - 1) / tm) * ((N + BN - 1) / BN);
  if (p.S > 1 && (ws == nullptr || ws_bytes < gemm_dense_workspace_bytes(M, N, K)))
    return DensePlan{1, static_cast<int>(tiles)};
  return p;
}

template <bool FP>
cudaError_t launch_split_finalize(const void* part, const DensePlan& p, int64_t M, int64_t N,
                                  const float* tscale, const float* rscale, uint16_t* y,
                                  int32_t* acc, cudaStream_t st) {
  const long tm = dense_tile_rows(M);
  const long m_blocks = (M + tm - 1) / tm;
  const long tiles = m_blocks * ((N + BN - 1) / BN);
  const long n_split = tiles - p.full;
  const long threads = n_split * tm * (BN / 8);
  return launch(split_finalize_kernel<FP>, dim3(static_cast<unsigned>((threads + 255) / 256)),
                dim3(256), 0, st, part, p.S, p.full, static_cast<int>(n_split),
                static_cast<int>(m_blocks), static_cast<int>(tm), static_cast<int>(M),
                static_cast<int>(N), tscale, rscale, reinterpret_cast<__nv_bfloat16*>(y), acc);
}

// Launch one of a dense GEMM's four kernels (split or not, pair or not):
// pairs run as clusters of two, as many as fit on the device at once.
template <typename Kern, typename... Args>
cudaError_t launch_dense(Kern kern, bool pair, long units, cudaStream_t st, Args... args) {
  if (!pair) {
    const int grid = static_cast<int>(units < sm_count() ? units : sm_count());
    return launch(kern, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, st, args...);
  }
  // the number of pairs that fit, queried once per kernel
  static std::atomic<const void*> keys[4];
  static std::atomic<int> vals[4];
  const void* key = reinterpret_cast<const void*>(kern);
  int pairs = 0;
  for (int i = 0; i < 4 && pairs == 0; ++i)
    if (keys[i].load(std::memory_order_acquire) == key) pairs = vals[i].load(std::memory_order_acquire);
  if (pairs == 0) {
    pairs = max_active_clusters(kern, dim3(NUM_THREADS), SMEM_BYTES, 2);
    if (pairs <= 0) return cudaErrorNotSupported;
    for (int i = 0; i < 4; ++i) {
      const void* expect = nullptr;
      if (keys[i].load(std::memory_order_acquire) == key) break;
      if (vals[i].load(std::memory_order_acquire) == 0) {
        vals[i].store(pairs, std::memory_order_release);
        if (keys[i].compare_exchange_strong(expect, key)) break;
      }
    }
  }
  const long teams = units < pairs ? units : pairs;
  return launch_cluster(kern, dim3(static_cast<unsigned>(2 * teams)), dim3(NUM_THREADS),
                        SMEM_BYTES, st, 2u, args...);
}
}  // namespace

cudaError_t launch_gemm(const uint16_t* xq, const float* tscale, const uint16_t* w_q,
                        const float* rscale, int64_t M, int64_t N, int64_t K, uint16_t* y,
                        int32_t* acc, void* ws, size_t ws_bytes, cudaStream_t st) {
  const bool pair = dense_tile_rows(M) > BM;
  CUtensorMap ta, tb;   // token boxes of 128 rows; weight boxes of 256 rows (128 in a pair)
  if (!make_map(&ta, xq, M, K, BM) || !make_map(&tb, w_q, N, K, pair ? BN / 2 : BN))
    return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t ea = once_per_device(attr_done, [] {
    for (auto* kern : {gemm_i8_kernel<false, false>, gemm_i8_kernel<true, false>,
                       gemm_i8_kernel<false, true>, gemm_i8_kernel<true, true>}) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(SMEM_BYTES));
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  });
  if (ea != cudaSuccess) return ea;
  const DensePlan p = usable_plan(M, N, K, ws, ws_bytes);
  int32_t* part = p.S > 1 ? static_cast<int32_t*>(ws) : nullptr;
  const long tm = dense_tile_rows(M);
  const long tiles = ((M + tm - 1) / tm) * ((N + BN - 1) / BN);
  const long units = p.full + (tiles - p.full) * p.S;
  auto* kern = p.S > 1 ? (pair ? gemm_i8_kernel<true, true> : gemm_i8_kernel<true, false>)
                       : (pair ? gemm_i8_kernel<false, true> : gemm_i8_kernel<false, false>);
  cudaError_t e = launch_dense(kern, pair, units, st, ta, tb, tscale, rscale, static_cast<int>(M),
                               static_cast<int>(N), static_cast<int>(K),
                               reinterpret_cast<__nv_bfloat16*>(y), acc, p.S, p.full, part);
  if (e != cudaSuccess || p.S == 1) return e;
  return launch_split_finalize<false>(part, p, M, N, tscale, rscale, y, acc, st);
}

namespace {
// Tile orientation of the packed GEMM: weight rows on the MMA's M side
// (256-token tiles, run by CTA pairs) above one 128-token block.
bool packed_wm(int64_t M) { return M > BM; }

// Tiles: 128 tokens x 256 weight rows per CTA, or 256 weight rows x 256
// tokens per CTA pair; a "team" is one CTA or one pair.
long packed_tiles(int64_t M, int64_t N) {
  return packed_wm(M) ? ((M + 255) / 256) * ((N + 255) / 256)
                      : ((M + BM - 1) / BM) * ((N + PBN - 1) / PBN);
}
long packed_teams(int64_t M) { return packed_wm(M) ? sm_count() / 2 : sm_count(); }
}  // namespace

namespace {
struct PackedPlan {
  int S;      // K slices per split tile (1: nothing split)
  int full;   // tiles computed whole, before the split ones
};

// How the packed GEMM cuts its work.  Up to 128 tokens (one CTA per tile):
// whole tiles when they fill most of the GPU, else every tile in as many K
// slices of whole 128-groups as keep one unit per CTA (partial sums in S
// planes [M][N]).  CTA pairs: like the expanded GEMMs, the whole waves of
// tiles whole and the tiles of the last, partial wave (all tiles when there
// are fewer than pairs) in S slices, if the estimate is at least 1 % shorter:
// waves x 128-groups per unit x one tile-group (~0.80 us measured), plus
// the pieces' traffic and the finishing kernel's launch.
PackedPlan packed_plan(int64_t M, int64_t N, int64_t K) {
  const long tiles = packed_tiles(M, N);
  const long teams = packed_teams(M);
  const long groups = K / kGroup;
  if (!packed_wm(M)) {
    if (4 * tiles >= 3 * teams) return PackedPlan{1, static_cast<int>(tiles)};
    const long want = teams / tiles;
    return PackedPlan{static_cast<int>(want < groups ? want : groups), 0};
  }
  const double t_group = 0.80e-6, bw = 6.0e12, t_launch = 3e-6;
  const double piece_bytes = 256.0 * 256 * 4;
  const long full = tiles / teams * teams, rest = tiles - full;
  const double whole = static_cast<double>((tiles + teams - 1) / teams * groups) * t_group;
  PackedPlan best{1, static_cast<int>(tiles)};
  double best_t = whole;
  for (long S = 2; rest > 0 && S <= groups && S <= 64; ++S) {
    const long rounds = (rest * S + teams - 1) / teams;
    const double t = static_cast<double>(full / teams * groups + rounds * ((groups + S - 1) / S)) *
                         t_group +
                     (2.0 * rest * S * piece_bytes + 2.0 * rest * 256 * 256) / bw + t_launch;
    if (t < 0.99 * whole && t < best_t) {
      best_t = t;
      best = PackedPlan{static_cast<int>(S), static_cast<int>(full)};
    }
  }
  return best;
}
}  // namespace

int packed_splits(int64_t M, int64_t N, int64_t K) { return packed_plan(M, N, K).S; }

size_t gemm_packed_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const PackedPlan p = packed_plan(M, N, K);
  if (p.S == 1) return 0;
  if (!packed_wm(M)) return static_cast<size_t>(p.S) * M * N * sizeof(int32_t);
  return static_cast<size_t>(packed_tiles(M, N) - p.full) * p.S * 256 * 256 * sizeof(int32_t);
}

cudaError_t launch_gemm_packed(const uint16_t* xq, const float* tscale, const uint8_t* packed,
                               const int8_t* q, const float* rscale, int64_t M, int64_t N,
                               int64_t K, uint16_t* y, int32_t* acc, void* ws, cudaStream_t st) {
  // 0 unknown, 1 both orientations built with the launch allocation the
  // register split needs, -1 not
  static std::atomic<int> regs_ok{0};
  if (regs_ok.load(std::memory_order_acquire) == 0) {
    int ok = 1;
    for (auto* kern : {gemm_packed_kernel<false, false>, gemm_packed_kernel<true, true>}) {
      cudaFuncAttributes fa;
      cudaError_t e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != P_LAUNCH_REGS) ok = -1;
    }
    regs_ok.store(ok, std::memory_order_release);
  }
  // never launch a register split that may not fit the block's allocation
  if (regs_ok.load(std::memory_order_acquire) < 0) return cudaErrorNotSupported;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t ea = once_per_device(attr_done, [] {
    for (auto* kern : {gemm_packed_kernel<false, false>, gemm_packed_kernel<true, true>}) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(PSMEM_BYTES));
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  });
  if (ea != cudaSuccess) return ea;
  const bool wm = packed_wm(M);
  CUtensorMap ta;   // token boxes: 64 k x (128 tokens, one CTA's half of a pair tile)
  if (!make_map(&ta, xq, M, K, BM)) return cudaErrorInvalidValue;
  const PackedPlan p = packed_plan(M, N, K);
  const int S = p.S;
  int32_t* part = S > 1 ? static_cast<int32_t*>(ws) : nullptr;
  const long tiles = packed_tiles(M, N);
  const long units = p.full + (tiles - p.full) * S;
  cudaError_t e;
  if (wm) {
    // one CTA pair per team, as many as fit on the device at once
    static std::atomic<long> pairs_cached{0};
    long pairs = pairs_cached.load(std::memory_order_acquire);
    if (pairs == 0) {
      pairs = max_active_clusters(gemm_packed_kernel<true, true>, dim3(P_THREADS), PSMEM_BYTES, 2);
      if (pairs <= 0) return cudaErrorNotSupported;
      pairs_cached.store(pairs, std::memory_order_release);
    }
    const long teams = units < pairs ? units : pairs;
    e = launch_cluster(gemm_packed_kernel<true, true>, dim3(static_cast<unsigned>(2 * teams)),
                       dim3(P_THREADS), PSMEM_BYTES, st, 2u, ta, packed, q, tscale, rscale,
                       static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                       reinterpret_cast<__nv_bfloat16*>(y), acc, S, p.full, part);
  } else {
    const int grid = static_cast<int>(units < sm_count() ? units : sm_count());
    e = launch(gemm_packed_kernel<false, false>, dim3(grid), dim3(P_THREADS), PSMEM_BYTES, st, ta,
               packed, q, tscale, rscale, static_cast<int>(M), static_cast<int>(N),
               static_cast<int>(K), reinterpret_cast<__nv_bfloat16*>(y), acc, S, p.full, part);
  }
  if (e != cudaSuccess || S == 1) return e;
  if (wm) {
    // the split tiles' pieces, [256 tokens][256 weight rows] each: the
    // expanded GEMMs' finishing kernel (same tile order and epilogue)
    const long m_blocks = (M + 255) / 256;
    const long n_split = tiles - p.full;
    const long threads = n_split * 256 * (BN / 8);
    return launch(split_finalize_kernel<false>,
                  dim3(static_cast<unsigned>((threads + 255) / 256)), dim3(256), 0, st,
                  static_cast<const void*>(part), S, p.full, static_cast<int>(n_split),
                  static_cast<int>(m_blocks), 256, static_cast<int>(M), static_cast<int>(N),
                  tscale, rscale, reinterpret_cast<__nv_bfloat16*>(y), acc);
  }
  const long threads = M * N / 8;
  return launch(packed_finalize_kernel, dim3(static_cast<unsigned>((threads + FIN_THREADS - 1) /
                                                                   FIN_THREADS)),
                dim3(FIN_THREADS), 0, st, static_cast<const int32_t*>(part), S, tscale, rscale,
                static_cast<int>(M), static_cast<int>(N), reinterpret_cast<__nv_bfloat16*>(y),
                acc);
}

cudaError_t launch_gemm_f16(const uint16_t* xh, const float* xs, const uint16_t* w_h, int64_t M,
                            int64_t N, int64_t K, uint16_t* y, void* ws, size_t ws_bytes,
                            cudaStream_t st) {
  const bool pair = dense_tile_rows(M) > BM;
  CUtensorMap ta, tb;
  if (!make_map(&ta, xh, M, K, BM) || !make_map(&tb, w_h, N, K, pair ? BN / 2 : BN))
    return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t ea = once_per_device(attr_done, [] {
    for (auto* kern : {gemm_f16_kernel<false, false>, gemm_f16_kernel<true, false>,
                       gemm_f16_kernel<false, true>, gemm_f16_kernel<true, true>}) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(SMEM_BYTES));
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  });
  if (ea != cudaSuccess) return ea;
  const DensePlan p = usable_plan(M, N, K, ws, ws_bytes);
  float* part = p.S > 1 ? static_cast<float*>(ws) : nullptr;
  const long tm = dense_tile_rows(M);
  const long tiles = ((M + tm - 1) / tm) * ((N + BN - 1) / BN);
  const long units = p.full + (tiles - p.full) * p.S;
  auto* kern = p.S > 1 ? (pair ? gemm_f16_kernel<true, true> : gemm_f16_kernel<true, false>)
                       : (pair ? gemm_f16_kernel<false, true> : gemm_f16_kernel<false, false>);
  cudaError_t e = launch_dense(kern, pair, units, st, ta, tb, xs, static_cast<int>(M),
                               static_cast<int>(N), static_cast<int>(K),
                               reinterpret_cast<__nv_bfloat16*>(y), p.S, p.full, part);
  if (e != cudaSuccess || p.S == 1) return e;
  return launch_split_finalize<true>(part, p, M, N, nullptr, nullptr, y, nullptr, st);
}

namespace {
// Self-test of the bounded waits: one warp waits, with the kernels' own wait
// helper, on an mbarrier that nothing arrives on (parity 0 of a freshly
// initialised barrier), gives up after `polls` polls and records it in the
// error word tern_check() reads -- what a kernel whose copy never lands
// does.  It holds no tensor memory and has no copies in flight.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint32_t polls) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::mbar_fence_init();
  }
  __syncwarp();
  if (!ptx::mbar_wait_warp(&bar, 0, &abort_flag, polls) && threadIdx.x == 0)
    atomicOr(&g_gemm_error, ERR_SELFTEST);
}
}  // namespace

cudaError_t launch_wait_selftest(uint32_t polls, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(polls);
  return cudaGetLastError();
}

cudaError_t gemm_read_clear_error(unsigned int* err) {
  cudaError_t e = cudaMemcpyFromSymbol(err, g_gemm_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(unsigned int));
}

}  // namespace tern
