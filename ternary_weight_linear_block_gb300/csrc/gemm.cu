// The int8 prefill GEMM with per-row and per-token rescale.
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
constexpr uint32_t WAIT_LIMIT = 1u << 26;
constexpr uint32_t IDESC = ptx::idesc_f16_f32(BM, BN);
constexpr size_t SMEM_BYTES = static_cast<size_t>(STAGES) * STAGE_BYTES + 1024 + 256;

enum : unsigned int { ERR_PRODUCER = 1u, ERR_MMA = 2u, ERR_EPILOGUE = 4u, ERR_DRAIN = 8u };

__device__ __forceinline__ void fail(volatile int* abort_flag, unsigned int code) {
  *abort_flag = 1;
  atomicOr(&g_gemm_error, code);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_i8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const float* __restrict__ tscale, const float* __restrict__ rscale, int M,
                   int N, int K, __nv_bfloat16* __restrict__ y, int32_t* __restrict__ acc_out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* dfull = empty + STAGES;
  uint64_t* dempty = dfull + 2;
  uint64_t* done = dempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_blocks = (M + BM - 1) / BM;
  const int n_blocks = (N + BN - 1) / BN;
  const int tiles = m_blocks * n_blocks;
  const int kstages = K / BK;
  const int chunks = K / KCHUNK;
  constexpr int kStagesPerChunk = KCHUNK / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&dfull[b], 1);
      ptx::mbar_init(&dempty[b], 8);   // one arrival per epilogue warp
    }
    ptx::mbar_init(done, 1);
    *abort_flag = 0;
    ptx::mbar_fence_init();
  }
  if (warp == 2) {
    ptx::tmem_alloc(tmem_slot, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  ptx::tc_fence_before();
  __syncthreads();
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
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        const int n_blk = tile / m_blocks, m_blk = tile % m_blocks;
        for (int ks = 0; ks < kstages; ++ks) {
          if (!ptx::mbar_wait(&empty[s], phase ^ 1u, abort_flag, WAIT_LIMIT)) {
            if (!*abort_flag) fail(abort_flag, ERR_PRODUCER);
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
          ptx::tma_load_2d(sA + s * A_BYTES, &tmA, &full[s], ks * BK, m_blk * BM);
          ptx::tma_load_2d(sB + s * B_BYTES, &tmB, &full[s], ks * BK, n_blk * BN);
          ++issued;
          if (++s == STAGES) {
            s = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let the copies still in flight land before the CTA exits
        long back = issued < STAGES ? issued : STAGES;
        int ss = s;
        uint32_t ph = phase;
        for (long i = 0; i < back; ++i) {
          if (--ss < 0) {
            ss = STAGES - 1;
            ph ^= 1u;
          }
          if (!ptx::mbar_wait_bounded(&full[ss], ph, WAIT_LIMIT)) atomicOr(&g_gemm_error, ERR_DRAIN);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer (one thread)
      int s = 0;
      uint32_t phase = 0;
      uint32_t cc = 0;   // chunk counter across tiles
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        for (int c = 0; c < chunks && ok; ++c, ++cc) {
          const uint32_t buf = cc & 1u, dph = (cc >> 1) & 1u;
          if (!ptx::mbar_wait(&dempty[buf], dph ^ 1u, abort_flag, WAIT_LIMIT)) {
            if (!*abort_flag) fail(abort_flag, ERR_MMA);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem + buf * BN;
          for (int j = 0; j < kStagesPerChunk; ++j) {
            if (!ptx::mbar_wait(&full[s], phase, abort_flag, WAIT_LIMIT)) {
              if (!*abort_flag) fail(abort_flag, ERR_MMA);
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t a0 = ptx::sw128_kmajor_desc(ptx::smem_u32(sA + s * A_BYTES));
            const uint64_t b0 = ptx::sw128_kmajor_desc(ptx::smem_u32(sB + s * B_BYTES));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              ptx::mma_f16_ss(d_tmem, a0 + 2u * kk, b0 + 2u * kk, IDESC,
                              (j > 0 || kk > 0) ? 1u : 0u);
            ptx::mma_commit(&empty[s]);
            if (++s == STAGES) {
              s = 0;
              phase ^= 1u;
            }
          }
          if (ok) ptx::mma_commit(&dfull[buf]);
        }
      }
      // every MMA issued by this thread has completed once `done` fires
      ptx::mma_commit(done);
      if (!ptx::mbar_wait_bounded(done, 0, WAIT_LIMIT)) atomicOr(&g_gemm_error, ERR_DRAIN);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- epilogue: warpgroup wg owns columns [128 wg, 128 wg + 128)
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;   // TMEM lane quarter accessible to this warp
    uint32_t cc = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      const int n_blk = tile / m_blocks, m_blk = tile % m_blocks;
      int32_t sums[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) sums[i] = 0;
      for (int c = 0; c < chunks; ++c, ++cc) {
        const uint32_t buf = cc & 1u, dph = (cc >> 1) & 1u;
        if (!ptx::mbar_wait(&dfull[buf], dph, abort_flag, WAIT_LIMIT)) {
          if (!*abort_flag) fail(abort_flag, ERR_EPILOGUE);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int piece = 0; piece < 4; ++piece) {
          uint32_t v[32];
          const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * BN +
                                 wg * 128 + piece * 32;
          ptx::tmem_ld_32x32b_x32(taddr, v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            sums[piece * 32 + i] += __float2int_rn(__uint_as_float(v[i]));   // exact integers
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&dempty[buf]);
      }
      if (!ok) break;
      const int row = m_blk * BM + 32 * q + lane;
      if (row < M) {
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
              const float f0 = __fmul_rn(__fmul_rn(__int2float_rn(sums[j + 2 * t]), ts), rr[2 * t]);
              const float f1 =
                  __fmul_rn(__fmul_rn(__int2float_rn(sums[j + 2 * t + 1]), ts), rr[2 * t + 1]);
              __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
              packed[t] = *reinterpret_cast<uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(yrow + n) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
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
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
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

}  // namespace

cudaError_t launch_gemm(const uint16_t* xq, const float* tscale, const uint16_t* w_q,
                        const float* rscale, int64_t M, int64_t N, int64_t K, uint16_t* y,
                        int32_t* acc, cudaStream_t st) {
  CUtensorMap ta, tb;
  if (!make_map(&ta, xq, M, K, BM) || !make_map(&tb, w_q, N, K, BN)) return cudaErrorInvalidValue;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(gemm_i8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const long tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  return launch(gemm_i8_kernel, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, st, ta, tb, tscale,
                rscale, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                reinterpret_cast<__nv_bfloat16*>(y), acc);
}

cudaError_t gemm_read_clear_error(unsigned int* err) {
  cudaError_t e = cudaMemcpyFromSymbol(err, g_gemm_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(unsigned int));
}

}  // namespace tern
