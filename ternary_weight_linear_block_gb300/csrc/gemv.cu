// Decode GEMV for M <= 16 tokens over 2-bit ternary weights.
//
// Page "RTX 5070 x2 ... Ternary-Bonsai-2-27B on vLLM TP=2", section "前提":
// y[m,n] = sum_g s[n,g] sum_{k in g} code[n,k] xr[m,k], codes in {-1,0,+1}
// stored at 2 bits, one fp16 scale per 128 elements of a row, xr the
// block-Hadamard-rotated activation.  Section 5 records that an int8 (dp4a)
// decode kernel added error for a 2% end-to-end gain; here the activations
// stay in fp16 (a power of two per block and per k16 step, see
// tern_fwht_quant).
//
// GB300 design.  The layer is one stream of weight bytes; everything else is
// arranged so that stream runs at HBM speed with few instructions per byte:
// * unit = 512 weight rows x one 128-wide group: 16384 bytes of codes and
//   1024 bytes of scales, contiguous in the packed format, fetched by one
//   bulk copy (L2 evict-first) into a 4-stage shared-memory ring; the
//   activation tile of the group (16 token rows x 128 k, fp16) arrives by
//   TMA (128-byte swizzle) into the same stage, with the group's 192-byte
//   record (negated token offsets as accumulator quads, block fold
//   factors); token rows >= M are
//   zero-filled by TMA and cost no memory traffic.
// * each 32-bit word of the packed format is one register of an m16n8k16 A
//   fragment for all 8 k16 steps of the group: one AND (after a shift by 12
//   for steps 6 and 7) gives the fp16 pair u * 4^e * 2^-24, u = code + 1 (a
//   subnormal, or the two lowest exponent bits), exactly; the operand carries
//   4^-e, and each group's accumulator starts at minus the tokens' offset
//   (the group sum of what u = 1 would give), which leaves sum code * x.
//   Tokens are the n side of the MMA (one n8 tile for M <= 8, two for
//   M <= 16), so every weight byte is read once for all M tokens.
//   (On sm_103a the legacy fp8 mma.sync issues four FMA-pipe instructions
//   per MMA and tcgen05 costs ~100 cycles per MMA even at N = 16, so the
//   fp16 mma.sync pipe is the fastest tensor path at this shape.)
// * sixteen consumer warps each own 32 rows (2 tiles) of a unit: B fragments
//   come from ldmatrix, A fragments from the masked words; per group the
//   fp32 accumulators are scaled by the row's group scale, per 1024-block by
//   the block's fold factor, and the result by 2^12 before the bf16 rounding.
// * units are cut into equal contiguous ranges, one per persistent CTA
//   (stream-K).  A 512-row block finished by one CTA is written directly.  A
//   block shared by at most 4 CTAs at M <= 8 is summed by its first owner,
//   which in this order reaches it last, from 32-bit words the other owners
//   publish without fences or atomics (a nonzero word is a published value);
//   otherwise (more owners: small N, large K; or M > 8) the block's partial
//   sums go to a small fixup kernel, launched right after (programmatic
//   launch), which adds them in slot order across the whole GPU, so no
//   block's first owner reads many slots.  The segment's end
//   runs outside the per-unit loop, which keeps the hot loop's registers for
//   the hot loop.
// * the weight copies do not depend on the previous kernel, so the producer
//   issues the first ring of them before the programmatic launch wait, and
//   every CTA lets the next kernel launch as soon as it starts.
// * the producer is a warp of its own.  At M > 8 each group's sums are
//   scaled straight into the accumulators (group scale times the block's
//   power-of-two fold factor), so that the two token tiles fit the 544-thread
//   block's registers; at M <= 8 a block's group sums are folded once per
//   1024-block (see unit_math_direct).
// All barrier and tag waits are bounded; a wait that gives up sets an error
// word that tern_check() reports (the workspace must then be re-initialised).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <utility>

#include "fwht_dev.cuh"
#include "sm100_ptx.cuh"
#include "tern_internal.cuh"

namespace tern {

__device__ unsigned int g_gemv_error;

namespace {

constexpr int RB = 512;                         // weight rows per unit
constexpr int TILES = RB / 16;
constexpr int UNIT_CODE_BYTES = RB * 32;        // 512 rows x 128 codes x 2 bits
constexpr int UNIT_BYTES = UNIT_CODE_BYTES + TILES * 32;
constexpr int XTILE_BYTES = 16 * kGroup * 2;    // 16 token rows x 128 k, fp16 (two 64-k boxes)
constexpr int AUX_BYTES = 192;                  // the group's record: 8 offset quads, 16 fold factors
constexpr int AUX_OFF = XTILE_BYTES + UNIT_BYTES;
constexpr int STAGE_TX = XTILE_BYTES + UNIT_BYTES + AUX_BYTES;
constexpr int STAGE_BYTES = 24576;
// The decode operand's fold factors are 2^(12 - sh): the sums carry 2^-12.
constexpr float OUT_SCALE = 4096.f;
// Ring depth: measured on gate/up, down, qkv and o at M = 1-16, four stages
// beat three, five to nine (eight: 16.60 -> 16.41 us per gate/up launch at
// M = 4, down 12.61 -> 11.65 us at M = 1).
constexpr int STAGES = 4;
constexpr int CONSUMERS = 16;                   // consumer warps
constexpr int TPW = TILES / CONSUMERS;          // tiles per consumer warp (2)
constexpr int NUM_THREADS = 32 * (1 + CONSUMERS);   // a producer warp + the consumers
// Both token widths run a producer warp and the 16 consumer warps (544
// threads; the per-SMSP register file holds such a block to 96 registers per
// thread).  At M > 8 the two n8 token tiles' accumulators fit that only
// without the per-block sums (see unit_math_direct).
// Polls of a bounded barrier wait before it gives up: a poll that finds the
// phase incomplete suspends for about 3.8 us on GB300 (measured with
// tern_selftest_wait), so 2^18 polls give up after about one second; a
// wait of the working kernel lasts microseconds.
constexpr uint32_t WAIT_LIMIT = 1u << 18;
// Tries of the tagged-word wait (a load round trip and a 32 ns sleep each:
// about 50 ms in all).  A first owner polls only at its range's end, when
// its own loop is done; the short sleep keeps the detection of the last
// publication prompt (a 200 ns sleep measured 14.95 against 14.89 us per
// gate/up launch at M = 4).
constexpr uint32_t TAG_TRIES = 1u << 16;
constexpr size_t SMEM_BYTES = static_cast<size_t>(STAGES) * STAGE_BYTES + 1024 + 256;

static_assert(STAGE_TX <= STAGE_BYTES, "stage too small");
static_assert(AUX_OFF % 16 == 0, "bulk copy alignment");
static_assert(STAGE_BYTES % 1024 == 0 && XTILE_BYTES % 16 == 0, "stage alignment");

enum : unsigned int { ERR_PRODUCER = 1u, ERR_CONSUMER = 2u, ERR_DRAIN = 4u, ERR_REDUCE = 8u };

// Owners of a 512-row block summed inside the GEMV (M <= 8 only: with two n8
// tiles the first owner's share of the sums costs more than the fixup
// launch); blocks with more owners go through the fixup kernel.
template <int NT>
__host__ __device__ constexpr int tag_slots() { return NT == 1 ? 4 : 1; }

__host__ __device__ inline long unit_begin(long c, long U, long C) { return c * U / C; }
__host__ __device__ inline long owner_of(long u, long U, long C) { return ((u + 1) * C - 1) / U; }
// The same owner in 32-bit arithmetic for the kernels: the entry points keep
// N * K <= 2^34, so U <= 2^18 + 512 and (u + 1) * C stays far below 2^32.
__device__ __forceinline__ int owner32(int u, int U, int C) {
  return static_cast<int>((static_cast<unsigned>(u + 1) * static_cast<unsigned>(C) - 1u) /
                          static_cast<unsigned>(U));
}

__device__ __forceinline__ void fail(volatile int* abort_flag, unsigned int code) {
  *abort_flag = 1;
  atomicOr(&g_gemv_error, code);
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Shared-memory loads at 32-bit shared addresses (the stage contents arrive
// by the async proxy; the loads follow the barrier wait that covers them).
template <int OFF = 0>
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+%5];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a), "n"(OFF));
  return v;
}
// (a volatile load: each tile's accumulator quad is loaded into registers of
// its own, so the MMAs accumulate in place)
template <int OFF = 0>
__device__ __forceinline__ void lds_v4f(uint32_t a, float (&v)[4]) {
  asm volatile("ld.volatile.shared.v4.f32 {%0,%1,%2,%3}, [%4+%5];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
               : "r"(a), "n"(OFF));
}
template <int OFF = 0>
__device__ __forceinline__ float2 lds_v2f(uint32_t a) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2+%3];" : "=f"(v.x), "=f"(v.y) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF = 0>
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1+%2];" : "=r"(v) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF = 0>
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4+%5];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a), "n"(OFF));
}

// The loads of one unit for a warp's TPW tiles, at compile-time offsets from
// three per-lane base addresses: code slots (512 bytes apart), scale pairs
// (32 bytes apart) and, for each tile, the record's offset quad of n8 tile nt
// (64 bytes apart) as the tile's initial accumulators.
template <int NT, size_t... T>
__device__ __forceinline__ void load_tiles(uint32_t a_code, uint32_t a_sp, uint32_t a_rec,
                                           uint4 (&cv)[TPW], uint32_t (&sp)[TPW],
                                           float (&d)[TPW][NT][4], std::index_sequence<T...>) {
  ((cv[T] = lds_v4<512 * static_cast<int>(T)>(a_code)), ...);
  ((sp[T] = lds_u32<32 * static_cast<int>(T)>(a_sp)), ...);
  (lds_v4f<0>(a_rec, d[T][0]), ...);
  if constexpr (NT == 2) (lds_v4f<64>(a_rec, d[T][NT - 1]), ...);
}


__device__ __forceinline__ void st_word(unsigned int* p, unsigned int v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_word(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// A published partial sum: its fp32 bits, with +0.0 sent as -0.0, so that a
// word is nonzero exactly when it has been published (adding -0.0 instead
// of +0.0 changes at most the sign of a zero sum).
__device__ __forceinline__ unsigned int published(float v) {
  const unsigned int b = __float_as_uint(v);
  return b != 0u ? b : 0x80000000u;
}

// A segment [ga, gb) of row block rb ends.  A row block finished by one CTA
// is written directly.  A block shared by at most tag_slots CTAs is summed by
// its first owner, which in stream-K order finishes the block last: every
// other owner publishes its 32 rows per warp as 32-bit words in its slot
// (published(): never zero), with no fence and no atomic (each word is
// single-copy atomic, so a nonzero word is the whole value), and the first
// owner reads them, adds them in slot order, writes y and zeroes them.  A
// block with more owners would load its first owner with too many slots:
// there every owner stores its words and the fixup kernel adds them across
// the whole GPU after the GEMV, and zeroes them.  Between calls every word
// of the workspace is zero.  The first owner's wait needs its co-owners (the
// next CTAs in launch order) resident with it: the grid is at most one CTA
// per SM and one CTA fits an SM; where the GPU cannot hold the whole grid
// the bounded wait gives up and the call reports a timeout.
template <int NT>
__device__ __forceinline__ void end_segment(const float (&acc)[TPW][NT][4], int ga, int gb, int rb,
                                         int G, int U, int C, int S, int M, int N, int cw,
                                         int lane, __nv_bfloat16* __restrict__ y,
                                         unsigned int* __restrict__ partials,
                                         volatile int* abort_flag) {
  const int gq = lane >> 2, cq = lane & 3;
  constexpr int NV = TPW * NT * 4;
  if (ga == 0 && gb == G) {
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int tt = v / (NT * 4), nt = (v / 4) % NT, i = v % 4;
      const int row = rb * RB + 16 * (TPW * cw + tt) + gq + 8 * (i >> 1);
      const int tok = 8 * nt + 2 * cq + (i & 1);
      if (row < N && tok < M)
        y[static_cast<long>(tok) * N + row] =
            __float2bfloat16_rn(__fmul_rn(acc[tt][nt][i], OUT_SCALE));
    }
    return;
  }
  const int first = owner32(rb * G, U, C);
  const int slot = static_cast<int>(blockIdx.x) - first;
  const int nslots = owner32(rb * G + G - 1, U, C) - first + 1;
  if (NT == 2 || nslots > tag_slots<NT>()) {
    unsigned int* base = partials + (static_cast<long>(rb) * S + slot) * M * RB;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int tt = v / (NT * 4), nt = (v / 4) % NT, i = v % 4;
      const int rin = 16 * (TPW * cw + tt) + gq + 8 * (i >> 1);
      const int tok = 8 * nt + 2 * cq + (i & 1);
      if (tok < M) __stcg(base + tok * RB + rin, __float_as_uint(acc[tt][nt][i]));
    }
    return;
  }
  if (slot != 0) {
    unsigned int* base = partials + (static_cast<long>(rb) * S + slot) * M * RB;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int tt = v / (NT * 4), nt = (v / 4) % NT, i = v % 4;
      const int rin = 16 * (TPW * cw + tt) + gq + 8 * (i >> 1);
      const int tok = 8 * nt + 2 * cq + (i & 1);
      if (tok < M) st_word(base + tok * RB + rin, published(acc[tt][nt][i]));
    }
    return;
  }
  float sum[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) sum[v] = acc[v / (NT * 4)][(v / 4) % NT][v % 4];
  // the other slots in order, SB at a time: all words of a round are loaded
  // before any is checked, so slots published long ago cost one memory round
  // trip; a slot not yet complete is loaded again (bounded).  Measured with
  // 32-bit words: SB = 2 beats loading all three other slots at once at
  // every M (gate/up 14.56 -> 14.35 us at M = 4, 14.24 -> 13.81 at M = 1).
  constexpr int SB = 2;
  bool ok = true;
  for (int sl0 = 1; sl0 < nslots && ok; sl0 += SB) {
    unsigned int w[SB][NV];
    for (uint32_t tries = 0;; ++tries) {
      bool ready = true;
#pragma unroll
      for (int sb = 0; sb < SB; ++sb) {
        const unsigned int* base = partials + (static_cast<long>(rb) * S + sl0 + sb) * M * RB;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          const int tt = v / (NT * 4), nt = (v / 4) % NT, i = v % 4;
          const int rin = 16 * (TPW * cw + tt) + gq + 8 * (i >> 1);
          const int tok = 8 * nt + 2 * cq + (i & 1);
          w[sb][v] = (sl0 + sb < nslots && tok < M) ? ld_word(base + tok * RB + rin) : 1u;
        }
      }
#pragma unroll
      for (int sb = 0; sb < SB; ++sb)
#pragma unroll
        for (int v = 0; v < NV; ++v) ready = ready && w[sb][v] != 0u;
      if (__all_sync(0xffffffffu, ready)) break;
      if (tries >= TAG_TRIES || *abort_flag) {
        if (lane == 0) fail(abort_flag, ERR_REDUCE);
        ok = false;
        break;
      }
      __nanosleep(32);
    }
    if (!ok) break;
#pragma unroll
    for (int sb = 0; sb < SB; ++sb) {
      if (sl0 + sb >= nslots) continue;
#pragma unroll
      for (int v = 0; v < NV; ++v) sum[v] += __uint_as_float(w[sb][v]);
      unsigned int* base = partials + (static_cast<long>(rb) * S + sl0 + sb) * M * RB;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int tt = v / (NT * 4), nt = (v / 4) % NT, i = v % 4;
        const int rin = 16 * (TPW * cw + tt) + gq + 8 * (i >> 1);
        const int tok = 8 * nt + 2 * cq + (i & 1);
        if (tok < M) st_word(base + tok * RB + rin, 0u);
      }
    }
  }
  if (!ok) return;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int tt = v / (NT * 4), nt = (v / 4) % NT, i = v % 4;
    const int row = rb * RB + 16 * (TPW * cw + tt) + gq + 8 * (i >> 1);
    const int tok = 8 * nt + 2 * cq + (i & 1);
    if (row < N && tok < M)
      y[static_cast<long>(tok) * N + row] = __float2bfloat16_rn(__fmul_rn(sum[v], OUT_SCALE));
  }
}

// Fixup after the GEMV: y[tok][row] = bf16(2^12 x the sum of the slots of
// the row's block, in slot order) for every row of a block shared by more than
// tag_slots CTAs.
// One thread per (block, token, row), consecutive threads on consecutive rows
// (coalesced); the slot loads of a thread are independent.  The reduction is
// spread over the whole GPU instead of the blocks' owners.
constexpr int FIX_THREADS = 256;
// BATCH slots' loads go out before their adds (in slot order), so a row of
// S slots costs ceil(S / BATCH) memory round trips.  The launcher takes
// BATCH = 16 (52 registers) when some block has more than 8 owners and the
// grid has more CTAs than the GPU has SMs, and 8 (32 registers) otherwise.
// Measured on GB300, GEMV + fixup per call: with at most one fixup CTA per SM
// the 8-slot batch is faster even at 16 slots (down 17408->5120 at M = 1-7:
// 10.6-10.9 against 11.5-11.7 us); past one per SM the 16-slot batch is
// (qkv 5120->10240 at M = 4-8: 8.9-9.1 against 9.6-10.4 us; down and o at
// M = 8: 11.5 against 12.8 us, 7.9 against 8.7 us).  With 8 slots or fewer
// one 8-slot round covers them (gate/up at M = 16: 26.3 against 27.6 us).
template <int BATCH>
__global__ void __launch_bounds__(FIX_THREADS)
    fixup_kernel(unsigned int* __restrict__ partials, __nv_bfloat16* __restrict__ y, int M, int N,
                 int G, int U, int C, int S, int tag) {
  pdl_launch_dependents();
  const int t = static_cast<int>(blockIdx.x) * FIX_THREADS + threadIdx.x;
  const int rin = t % RB;
  const int tok = (t / RB) % M;
  const int rb = t / (RB * M);
  const int first = owner32(rb * G, U, C);
  const int nslots = owner32(rb * G + G - 1, U, C) - first + 1;
  const long row = static_cast<long>(rb) * RB + rin;
  pdl_wait();   // the GEMV's partial sums
  if (nslots <= tag || row >= N) return;
  unsigned int* p = partials + (static_cast<long>(rb) * S * M + tok) * RB + rin;
  const long stride = static_cast<long>(M) * RB;   // one slot
  float sum = 0.f;
  for (int sl = 0; sl < nslots; sl += BATCH) {
    unsigned int a[BATCH];
#pragma unroll
    for (int j = 0; j < BATCH; ++j)
      if (sl + j < nslots) a[j] = __ldcg(p + (sl + j) * stride);
#pragma unroll
    for (int j = 0; j < BATCH; ++j)
      if (sl + j < nslots) sum += __uint_as_float(a[j]);
  }
  // the workspace is zero again after the call (the words' values are in
  // registers by now, so the stores do not wait on the loads)
  for (int sl = 0; sl < nslots; ++sl) __stcg(p + sl * stride, 0u);
  y[static_cast<long>(tok) * N + row] = __float2bfloat16_rn(__fmul_rn(sum, OUT_SCALE));
}

// The MMAs of one unit for this warp's tiles: codes cv and the B fragments bf
// of the group's 8 k16 steps accumulate into d, which arrives holding the
// tokens' negated group offsets.  Word p of a tile's slot is A-fragment
// register p for every step j: one AND per register (steps 6 and 7 from the
// word shifted right by 12) gives the fp16 pair u * 4^e * 2^-24, u = code +
// 1; the operand carries 4^-e, and the offset start removes the "+1" of u.
template <int NT>
__device__ __forceinline__ void unit_mma(const uint4 (&cv)[TPW], const uint32_t (&bf)[NT][8][2],
                                         float (&d)[TPW][NT][4]) {
  uint32_t hi[TPW][4];
#pragma unroll
  for (int tt = 0; tt < TPW; ++tt) {
    hi[tt][0] = cv[tt].x >> 12;
    hi[tt][1] = cv[tt].y >> 12;
    hi[tt][2] = cv[tt].z >> 12;
    hi[tt][3] = cv[tt].w >> 12;
  }
  // k16 steps outer, tiles inner: the tiles' MMA chains alternate
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t mask = 0x00030003u << (2 * (j < 6 ? j : j - 6));
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt) {
      const uint32_t w4[4] = {cv[tt].x, cv[tt].y, cv[tt].z, cv[tt].w};
      uint32_t a[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) a[p] = (j < 6 ? w4[p] : hi[tt][p]) & mask;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_f16(d[tt][nt], a[0], a[1], a[2], a[3], bf[nt][j][0], bf[nt][j][1]);
    }
  }
}

// One unit at M <= 8: the group sums, scaled by the rows' group scales sp,
// are added to the 1024-block's sums bacc (folded into acc once per block).
template <int NT>
__device__ __forceinline__ void unit_math(const uint4 (&cv)[TPW], const uint32_t (&sp)[TPW],
                                          const uint32_t (&bf)[NT][8][2], float (&d)[TPW][NT][4],
                                          float (&bacc)[TPW][NT][4]) {
  unit_mma<NT>(cv, bf, d);
#pragma unroll
  for (int tt = 0; tt < TPW; ++tt) {
    uint32_t spv = sp[tt];
    const float2 s2 = __half22float2(*reinterpret_cast<__half2*>(&spv));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      bacc[tt][nt][0] = fmaf(d[tt][nt][0], s2.x, bacc[tt][nt][0]);
      bacc[tt][nt][1] = fmaf(d[tt][nt][1], s2.x, bacc[tt][nt][1]);
      bacc[tt][nt][2] = fmaf(d[tt][nt][2], s2.y, bacc[tt][nt][2]);
      bacc[tt][nt][3] = fmaf(d[tt][nt][3], s2.y, bacc[tt][nt][3]);
    }
  }
}

// One unit with the group sums scaled straight into acc: the scale of a
// row's group times the block's fold factor of a token (a power of two, so
// the product is exact).  The M > 8 kernels use it: without the per-block
// sums bacc the two token tiles' accumulators fit a 544-thread block's 96
// registers, which gives them a producer warp of their own (measured on
// GB300 against a producer thread inside consumer warp 0: gate/up at M = 16
// 26.3 -> 23.6 us, down 14.8 -> 13.9 us).  At M <= 8 the per-block fold
// stays: its extra multiply per group cost gate/up 0.6-1.2 us there.
template <int NT>
__device__ __forceinline__ void unit_math_direct(const uint4 (&cv)[TPW], const uint32_t (&sp)[TPW],
                                                 const uint32_t (&bf)[NT][8][2],
                                                 float (&d)[TPW][NT][4], const float (&f)[NT][2],
                                                 float (&acc)[TPW][NT][4]) {
  unit_mma<NT>(cv, bf, d);
#pragma unroll
  for (int tt = 0; tt < TPW; ++tt) {
    uint32_t spv = sp[tt];
    const float2 s2 = __half22float2(*reinterpret_cast<__half2*>(&spv));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      acc[tt][nt][0] = fmaf(d[tt][nt][0], s2.x * f[nt][0], acc[tt][nt][0]);
      acc[tt][nt][1] = fmaf(d[tt][nt][1], s2.x * f[nt][1], acc[tt][nt][1]);
      acc[tt][nt][2] = fmaf(d[tt][nt][2], s2.y * f[nt][0], acc[tt][nt][2]);
      acc[tt][nt][3] = fmaf(d[tt][nt][3], s2.y * f[nt][1], acc[tt][nt][3]);
    }
  }
}

// End of a 1024-block: acc += bacc * f (f the block's fold factor of the
// thread's two tokens per n8 tile).
template <int NT>
__device__ __forceinline__ void fold_block(float (&acc)[TPW][NT][4], float (&bacc)[TPW][NT][4],
                                           const float (&f)[NT][2]) {
#pragma unroll
  for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[tt][nt][q] = fmaf(bacc[tt][nt][q], f[nt][q & 1], acc[tt][nt][q]);
        bacc[tt][nt][q] = 0.f;
      }
}

template <int NT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tmX, const uint8_t* __restrict__ packed,
                const float* __restrict__ aux, int M, int N, int K, __nv_bfloat16* __restrict__ y,
                unsigned int* __restrict__ partials, int U, int S) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STAGES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = K / kGroup;
  const int C = gridDim.x;
  const int u0 = static_cast<int>(unit_begin(blockIdx.x, U, C));
  const int u1 = static_cast<int>(unit_begin(blockIdx.x + 1, U, C));
  const int n_units = u1 - u0;

  pdl_launch_dependents();   // the next kernel may start its own independent prologue
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], CONSUMERS);
    }
    *abort_flag = 0;
    ptx::mbar_fence_init();
  }
  __syncthreads();

  // Lane 0 of warp 0 produces: it issues the first STAGES units (the weights
  // before the programmatic launch wait, which they do not depend on, the
  // activation tiles after it), then refills each stage once every consumer
  // warp has released it.
  const uint64_t pol = ptx::l2_policy_evict_first();
  const int pre = n_units < STAGES ? n_units : STAGES;
  if (warp == 0) {
    // ------------------------------------------------ producer warp
    if (lane == 0) {
      ptx::prefetch_tmap(&tmX);
      for (int i = 0; i < pre; ++i) {
        ptx::mbar_arrive_expect_tx(&full[i], STAGE_TX);
        ptx::bulk_load_hint(smem + i * STAGE_BYTES + XTILE_BYTES,
                            packed + static_cast<size_t>(u0 + i) * UNIT_BYTES, UNIT_BYTES, &full[i],
                            pol);
      }
      pdl_wait();   // the activations are written by the previous kernel
      int g = u0 % G;
      int issued = pre;   // units whose weight copies are issued
      bool ok = true;
      for (int i = 0; i < n_units; ++i) {
        const int s = i % STAGES;
        uint8_t* st = smem + s * STAGE_BYTES;
        if (i >= STAGES) {
          const uint32_t ph = static_cast<uint32_t>(i / STAGES) & 1u;
          if (!ptx::mbar_wait(&empty[s], ph ^ 1u, abort_flag, WAIT_LIMIT)) {
            if (!*abort_flag) fail(abort_flag, ERR_PRODUCER);
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[s], STAGE_TX);
          ptx::bulk_load_hint(st + XTILE_BYTES, packed + static_cast<size_t>(u0 + i) * UNIT_BYTES,
                              UNIT_BYTES, &full[s], pol);
          ++issued;
        }
        ptx::tma_load_2d(st, &tmX, &full[s], g * kGroup, 0);
        ptx::tma_load_2d(st + XTILE_BYTES / 2, &tmX, &full[s], g * kGroup + 64, 0);
        ptx::bulk_load(st + AUX_OFF, aux + static_cast<size_t>(g) * 48, AUX_BYTES, &full[s]);
        if (++g == G) g = 0;
      }
      if (!ok) {
        // let every copy still in flight land before the CTA exits
        for (int i = issued - 1; i >= 0 && i >= issued - STAGES; --i) {
          const uint32_t ph = static_cast<uint32_t>(i / STAGES) & 1u;
          if (!ptx::mbar_wait_bounded(&full[i % STAGES], ph, WAIT_LIMIT))
            atomicOr(&g_gemv_error, ERR_DRAIN);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ consumers
    const int cw = warp - 1;   // owns tiles TPW*cw .. TPW*cw + TPW-1 of each unit
    const int gq = lane >> 2, cq = lane & 3;
    pdl_wait();   // y / ws may still be read by the previous kernel

    // Per-lane shared-memory offsets, fixed for the whole kernel.  ldmatrix
    // matrix mi = lane / 8 covers (k16 step j0 + mi / 2, 8-wide k half mi % 2),
    // token row 8 nt + lane % 8, in the 128-byte-swizzled activation tile.
    const int mi = lane >> 3, lrow = lane & 7;
    uint32_t bf_off[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = 2 * q + (mi >> 1);
        const int row = 8 * nt + lrow;
        const int chunk = 2 * (j & 3) + (mi & 1);
        bf_off[nt][q] = (j >> 2) * (XTILE_BYTES / 2) + row * 128 + ((chunk ^ (row & 7)) << 4);
      }
    // the warp's two tiles' code slots, their scale pairs, the record's
    // offset quads and fold factors of tokens 8 nt + 2 cq + {0, 1}
    const uint32_t code_off = XTILE_BYTES + 512 * (TPW * cw) + 16 * lane;
    const uint32_t sp_off = XTILE_BYTES + UNIT_CODE_BYTES + 32 * (TPW * cw) + 4 * gq;
    const uint32_t rec_off = AUX_OFF + 16 * cq;    // offset quads; fold factors at + 128 - 8 cq
    const uint32_t smem_base = ptx::smem_u32(smem);

    float acc[TPW][NT][4], bacc[TPW][NT][4];
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[tt][nt][i] = bacc[tt][nt][i] = 0.f;

    int rb = u0 / G, g = u0 % G, seg_g0 = g;
    int s = 0;               // ring stage of unit i
    uint32_t ph = 0;         // its phase

    // The CTA's units form segments, one per row block they touch; the hot
    // loop runs over the units of one segment and the segment's end (direct
    // write, publication or reduction) happens outside it.
    bool alive = true;
    for (int i = 0; alive && i < n_units;) {
      const int seg_len = (n_units - i < G - g) ? n_units - i : G - g;
      const int i_end = i + seg_len;
      for (; i < i_end; ++i) {
        if (!ptx::mbar_wait_warp(&full[s], ph, abort_flag, WAIT_LIMIT)) {
          if (!*abort_flag) fail(abort_flag, ERR_CONSUMER);
          alive = false;
          break;
        }
        const uint32_t st = smem_base + s * STAGE_BYTES;
        const uint32_t a_code = st + code_off, a_sp = st + sp_off, a_rec = st + rec_off;
        uint4 cv[TPW];
        uint32_t sp[TPW];
        float d[TPW][NT][4];       // each tile's accumulators start at the offset quad
        load_tiles<NT>(a_code, a_sp, a_rec, cv, sp, d, std::make_index_sequence<TPW>{});
        float fo[NT][2];
        {
          const float2 f2 = lds_v2f<0>(a_rec + 128 - 8 * cq);
          fo[0][0] = f2.x;
          fo[0][1] = f2.y;
        }
        if constexpr (NT == 2) {
          const float2 f2 = lds_v2f<32>(a_rec + 128 - 8 * cq);
          fo[NT - 1][0] = f2.x;
          fo[NT - 1][1] = f2.y;
        }
        // B fragments: bf[nt][j][0..1] for the 8 k16 steps of the group; the
        // steps 4..7 lie XTILE_BYTES / 2 after steps 0..3
        uint32_t bf[NT][8][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint32_t b0 = st + bf_off[nt][0], b1 = st + bf_off[nt][1];
          ldsm_x4<0>(b0, bf[nt][0][0], bf[nt][0][1], bf[nt][1][0], bf[nt][1][1]);
          ldsm_x4<0>(b1, bf[nt][2][0], bf[nt][2][1], bf[nt][3][0], bf[nt][3][1]);
          ldsm_x4<XTILE_BYTES / 2>(b0, bf[nt][4][0], bf[nt][4][1], bf[nt][5][0], bf[nt][5][1]);
          ldsm_x4<XTILE_BYTES / 2>(b1, bf[nt][6][0], bf[nt][6][1], bf[nt][7][0], bf[nt][7][1]);
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&empty[s]);
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
        if constexpr (NT == 1) {
          unit_math<NT>(cv, sp, bf, d, bacc);
          if ((g & 7) == 7 || i + 1 == i_end) fold_block<NT>(acc, bacc, fo);
        } else {
          unit_math_direct<NT>(cv, sp, bf, d, fo, acc);
        }
        ++g;
      }
      if (!alive) break;
      end_segment<NT>(acc, seg_g0, g, rb, G, U, C, S, M, N, cw, lane, y, partials, abort_flag);
#pragma unroll
      for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[tt][nt][q] = 0.f;
      seg_g0 = 0;
      g = 0;
      ++rb;
    }
    __syncwarp();
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Fused decode linear: rotation + quantisation to the decode operand + GEMV in
// one launch (the layer's decode path with tern_fwht_quant folded into the
// GEMV prologue).  Each CTA rotates only the 1024-blocks its units touch, from
// the bf16 input, with the same butterflies and scaling as the rotation
// kernel (fwht_dev.cuh), and keeps the resulting fp16 operand of its groups
// resident in shared memory (token rows padded by 16 bytes so ldmatrix reads
// hit distinct banks); the pipeline ring then carries weight units only.  A
// CTA whose groups do not fit the resident area processes them in chunks and
// rotates again for each chunk.  Results are bit-identical to
// tern_fwht_quant(TERN_FWHT_DECODE) followed by tern_gemv_decode.
constexpr int LSTAGES = 8;
constexpr int LX_BYTES = 76 * 1024;             // resident decode operand (a chunk of groups)
constexpr int LCHUNK_MAX = 64;                  // groups of one chunk at most
// one group record per chunk position, laid out like the rotation kernel's
// (negated offset quads of 16 tokens, then their block's fold factors)
constexpr int LREC_BYTES = LCHUNK_MAX * AUX_BYTES;
constexpr size_t LSMEM_BYTES = static_cast<size_t>(LSTAGES) * UNIT_BYTES + LX_BYTES + LREC_BYTES +
                               1024 + 256;
static_assert(LSMEM_BYTES <= 227 * 1024, "shared memory budget");

// Groups of one chunk: each 256 bytes per token row.
__host__ __device__ inline int chunk_groups(int M, int G) {
  int cu = (LX_BYTES / M - 16) / 256;
  if (cu > LCHUNK_MAX) cu = LCHUNK_MAX;
  return cu < G ? cu : G;
}

template <int NT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    linear_kernel(const uint16_t* __restrict__ x, const int8_t* __restrict__ sign,
                  const uint8_t* __restrict__ packed, int M, int N, int K,
                  __nv_bfloat16* __restrict__ y, unsigned int* __restrict__ partials, int U,
                  int S) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* xreg = smem + LSTAGES * UNIT_BYTES;
  float* rec_s = reinterpret_cast<float*>(xreg + LX_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(rec_s + LREC_BYTES / 4);
  uint64_t* empty = full + LSTAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + LSTAGES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = K / kGroup;
  const int B = K / kHBlock;
  const int C = gridDim.x;
  const int u0 = static_cast<int>(unit_begin(blockIdx.x, U, C));
  const int u1 = static_cast<int>(unit_begin(blockIdx.x + 1, U, C));
  const int n_units = u1 - u0;
  const int CU = chunk_groups(M, G);
  const int pitch = CU * 256 + 16;               // bytes per token row of the resident operand

  pdl_launch_dependents();   // the next kernel may start its own independent prologue
  if (threadIdx.x == 0) {
    for (int s = 0; s < LSTAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], CONSUMERS);
    }
    *abort_flag = 0;
    ptx::mbar_fence_init();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ producer: weights only,
      // which do not depend on the previous kernel
      const uint64_t pol = ptx::l2_policy_evict_first();
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < n_units; ++i) {
        const int s = i % LSTAGES;
        if (i >= LSTAGES) {
          const uint32_t ph = static_cast<uint32_t>(i / LSTAGES) & 1u;
          if (!ptx::mbar_wait(&empty[s], ph ^ 1u, abort_flag, WAIT_LIMIT)) {
            if (!*abort_flag) fail(abort_flag, ERR_PRODUCER);
            ok = false;
            break;
          }
        }
        ptx::mbar_arrive_expect_tx(&full[s], UNIT_BYTES);
        ptx::bulk_load_hint(smem + s * UNIT_BYTES, packed + static_cast<size_t>(u0 + i) * UNIT_BYTES,
                            UNIT_BYTES, &full[s], pol);
        ++issued;
      }
      if (!ok) {
        // let every copy still in flight land before the CTA exits
        for (int i = issued - 1; i >= 0 && i >= issued - LSTAGES; --i) {
          const uint32_t ph = static_cast<uint32_t>(i / LSTAGES) & 1u;
          if (!ptx::mbar_wait_bounded(&full[i % LSTAGES], ph, WAIT_LIMIT))
            atomicOr(&g_gemv_error, ERR_DRAIN);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ consumers
    const int cw = warp - 1;          // owns tiles TPW*cw .. TPW*cw + TPW-1 of each unit
    const int gq = lane >> 2, cq = lane & 3;
    pdl_wait();   // x is written by the previous kernel; y / ws may still be read by it

    // ldmatrix: matrix mi = lane / 8 covers (k16 step 2q + mi / 2, 8-wide k
    // half mi % 2) of token row 8 nt + lane % 8; rows >= M read row 0 (their
    // products land in output columns that are never stored).
    const int mi = lane >> 3;
    uint32_t bf_off[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tok = 8 * nt + (lane & 7);
      bf_off[nt] = (tok < M ? tok : 0) * pitch + 32 * (mi >> 1) + 16 * (mi & 1);
    }
    const uint32_t smem_base = ptx::smem_u32(smem);
    const uint32_t x_base = ptx::smem_u32(xreg);
    const uint32_t rec_base = ptx::smem_u32(rec_s);

    // Rotate the 1024-blocks holding the groups gs .. gs + ng - 1 (mod G) and
    // store those groups' decode operand at positions 0 .. ng - 1 and their
    // group records at the same positions (the arithmetic and the record
    // layout of the rotation kernel: the negated offsets as the tensor
    // core's accumulator quads, then the block's fold factor per token).
    auto build = [&](int gs, int ng) {
      for (int t = cw; t < M * B; t += CONSUMERS) {
        const int m = t / B, b = t - m * B;
        // the block is needed when one of its groups lies in the chunk
        bool need = false;
#pragma unroll
        for (int j = 0; j < 8; ++j) need = need || ((8 * b + j - gs + G) % G) < ng;
        if (!need) continue;
        float v[4][8];
        fwht::load_block(x + static_cast<long>(m) * K + static_cast<long>(b) * kHBlock,
                         sign ? sign + static_cast<long>(b) * kHBlock : nullptr, lane, v);
        fwht::fwht_1024(v, lane);
        const int sh = fwht::block_shift(v);
        const int e = fwht::lane_step_exp(lane);
        const float fold = fwht::pow2f(12 - sh);
        const int qi = 4 * (m >> 1) + (m & 1);
#pragma unroll
        for (int ih = 0; ih < 4; ++ih) {
          // lanes 0-15 hold group 2 ih of the block, lanes 16-31 group 2 ih + 1
          const int gg = 8 * b + 2 * ih + (lane >> 4);
          const int pos = (gg - gs + G) % G;
          float part;
          const uint4 w = fwht::decode_pack8(v, ih, sh, e, part);
          const float xoff = __fsub_rn(0.f, fwht::group_offset(part));
          if (pos < ng) {
            *reinterpret_cast<uint4*>(xreg + m * pitch + pos * 256 + (lane & 15) * 16) = w;
            if ((lane & 15) == 0) {
              float* rec = rec_s + pos * (AUX_BYTES / 4);
              rec[qi] = xoff;
              rec[qi + 2] = xoff;
              rec[32 + m] = fold;
            }
          }
        }
      }
    };

    // the records' entries of tokens M .. 15 stay zero (offsets and fold
    // factors), as in the rotation kernel's records
    for (int i = threadIdx.x - 32; i < LREC_BYTES / 4; i += 32 * CONSUMERS) rec_s[i] = 0.f;
    ptx::named_sync(1, 32 * CONSUMERS);

    // Per-lane shared-memory offsets, fixed for the whole kernel (as in the
    // GEMV): the warp's two tiles' code slots and scale pairs in a stage,
    // and the record's offset quads and fold factors of tokens 8 nt + 2 cq +
    // {0, 1}.
    const uint32_t code_off = 512 * (TPW * cw) + 16 * lane;
    const uint32_t sp_off = UNIT_CODE_BYTES + 32 * (TPW * cw) + 4 * gq;
    const uint32_t rec_off = 16 * cq;

    float acc[TPW][NT][4], bacc[TPW][NT][4];
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[tt][nt][i] = bacc[tt][nt][i] = 0.f;

    int rb = u0 / G, g = u0 % G, seg_g0 = g, gs = g;
    int s = 0;               // ring stage of unit i
    uint32_t ph = 0;         // its phase
    bool alive = true;
    int c_end = 0;
    for (int i = 0; alive && i < n_units;) {
      if (i == c_end) {
        // next chunk: every consumer is done with the resident operand
        if (i > 0) ptx::named_sync(1, 32 * CONSUMERS);
        gs = g;
        c_end = n_units - i < CU ? n_units : i + CU;
        build(gs, c_end - i);
        ptx::named_sync(1, 32 * CONSUMERS);
      }
      // units up to the end of the segment (row block) or of the chunk
      const int seg_stop = i + (G - g);
      const int stop = seg_stop < c_end ? seg_stop : c_end;
      for (; i < stop; ++i) {
        if (!ptx::mbar_wait_warp(&full[s], ph, abort_flag, WAIT_LIMIT)) {
          if (!*abort_flag) fail(abort_flag, ERR_CONSUMER);
          alive = false;
          break;
        }
        const uint32_t st = smem_base + s * UNIT_BYTES;
        const int pos = g >= gs ? g - gs : g + G - gs;
        const uint32_t a_rec = rec_base + pos * AUX_BYTES + rec_off;
        uint4 cv[TPW];
        uint32_t sp[TPW];
        float d[TPW][NT][4];       // each tile's accumulators start at the offset quad
        load_tiles<NT>(st + code_off, st + sp_off, a_rec, cv, sp, d,
                       std::make_index_sequence<TPW>{});
        float fo[NT][2];
        {
          const float2 f2 = lds_v2f<0>(a_rec + 128 - 8 * cq);
          fo[0][0] = f2.x;
          fo[0][1] = f2.y;
        }
        if constexpr (NT == 2) {
          const float2 f2 = lds_v2f<32>(a_rec + 128 - 8 * cq);
          fo[NT - 1][0] = f2.x;
          fo[NT - 1][1] = f2.y;
        }
        uint32_t bf[NT][8][2];
        const uint32_t xb = x_base + pos * 256;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            ldmatrix_x4(xb + bf_off[nt] + 64 * q, bf[nt][2 * q][0], bf[nt][2 * q][1],
                        bf[nt][2 * q + 1][0], bf[nt][2 * q + 1][1]);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&empty[s]);
        if (++s == LSTAGES) {
          s = 0;
          ph ^= 1u;
        }
        if constexpr (NT == 1) {
          unit_math<NT>(cv, sp, bf, d, bacc);
          if ((g & 7) == 7 || i + 1 == n_units) fold_block<NT>(acc, bacc, fo);
        } else {
          unit_math_direct<NT>(cv, sp, bf, d, fo, acc);
        }
        ++g;
      }
      if (!alive) break;
      if (g == G || i == n_units) {
        end_segment<NT>(acc, seg_g0, g, rb, G, U, C, S, M, N, cw, lane, y, partials, abort_flag);
#pragma unroll
        for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[tt][nt][q] = 0.f;
        seg_g0 = 0;
        if (g == G) {
          g = 0;
          ++rb;
        }
      }
    }
    // a consumer that stopped early still meets the others at their barriers
    if (!alive)
      for (int i = c_end; i < n_units; i += CU) {
        ptx::named_sync(1, 32 * CONSUMERS);
        ptx::named_sync(1, 32 * CONSUMERS);
      }
    __syncwarp();
  }
  __syncthreads();
}

struct GemvPlan {
  int U, C, RBn, S;
};

GemvPlan make_plan(int64_t N, int64_t K, int sms) {
  GemvPlan p;
  const long G = K / kGroup;
  p.RBn = static_cast<int>((N + RB - 1) / RB);
  p.U = static_cast<int>(p.RBn * G);
  p.C = p.U < sms ? p.U : sms;
  long s = 1;
  for (long rb = 0; rb < p.RBn; ++rb) {
    const long a = owner_of(rb * G, p.U, p.C), b = owner_of(rb * G + G - 1, p.U, p.C);
    if (b - a + 1 > s) s = b - a + 1;
  }
  p.S = static_cast<int>(s);
  return p;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 152;
  return n;
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

template <int NT>
cudaError_t launch_nt(const CUtensorMap& tm, const uint8_t* packed, const float* xs, int M, int N,
                      int K, __nv_bfloat16* y, unsigned int* partials,
                      const GemvPlan& p, cudaStream_t st) {
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t e = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(gemv_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(SMEM_BYTES));
  });
  if (e != cudaSuccess) return e;
  return launch(gemv_kernel<NT>, dim3(p.C), dim3(NUM_THREADS), SMEM_BYTES, st, tm, packed, xs, M,
                N, K, y, partials, p.U, p.S);
}

}  // namespace

size_t gemv_packed_bytes(int64_t N, int64_t K) {
  return static_cast<size_t>((N + RB - 1) / RB) * static_cast<size_t>(K / kGroup) * UNIT_BYTES;
}

// Workspace: 32-bit partial-sum words [RBn][S][M][512] of row blocks shared
// by several CTAs (nonzero once published); every call leaves them all 0.
size_t gemv_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const GemvPlan p = make_plan(N, K, sm_count());
  return static_cast<size_t>(p.RBn) * p.S * M * RB * sizeof(unsigned int);
}

// Whether a call at this shape ends with the fixup kernel: some row block is
// shared by more CTAs than the main kernel sums in place.
bool gemv_needs_fixup(int64_t M, int64_t N, int64_t K) {
  const GemvPlan p = make_plan(N, K, sm_count());
  return p.S > (M <= 8 ? tag_slots<1>() : tag_slots<2>());
}

// The fixup kernel over every (block, token, row), when some block is shared.
cudaError_t launch_fixup(const GemvPlan& p, unsigned int* partials, __nv_bfloat16* y, int M,
                         int N, int G, cudaStream_t st) {
  const int tag = M <= 8 ? tag_slots<1>() : tag_slots<2>();
  if (p.S <= tag) return cudaSuccess;
  const long threads = static_cast<long>(p.RBn) * M * RB;
  const dim3 grid(static_cast<unsigned>((threads + FIX_THREADS - 1) / FIX_THREADS));
  const bool wide = p.S > 8 && grid.x > static_cast<unsigned>(sm_count());
  auto* kern = wide ? fixup_kernel<16> : fixup_kernel<8>;
  return launch(kern, grid, dim3(FIX_THREADS), 0, st,
                partials, y, M, N, G, p.U, p.C, p.S, tag);
}

cudaError_t launch_gemv(const uint8_t* packed, const uint16_t* xh, const float* xs, int64_t M,
                        int64_t N, int64_t K, uint16_t* y, void* ws, cudaStream_t st) {
  const GemvPlan p = make_plan(N, K, sm_count());
  auto* partials = static_cast<unsigned int*>(ws);
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  // the fp16 activations [M][K]; boxes of 64 k x 16 token rows
  CUtensorMap tm;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {64, 16};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(xh), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  auto* yy = reinterpret_cast<__nv_bfloat16*>(y);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  const cudaError_t e = M <= 8 ? launch_nt<1>(tm, packed, xs, m, n, k, yy, partials, p, st)
                               : launch_nt<2>(tm, packed, xs, m, n, k, yy, partials, p, st);
  if (e != cudaSuccess) return e;
  return launch_fixup(p, partials, yy, m, n, static_cast<int>(K / kGroup), st);
}

namespace {
template <int NT>
cudaError_t launch_linear_nt(const uint16_t* x, const int8_t* sign, const uint8_t* packed, int M,
                             int N, int K, __nv_bfloat16* y, unsigned int* partials,
                             const GemvPlan& p, cudaStream_t st) {
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t e = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(linear_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(LSMEM_BYTES));
  });
  if (e != cudaSuccess) return e;
  return launch(linear_kernel<NT>, dim3(p.C), dim3(NUM_THREADS), LSMEM_BYTES, st, x, sign, packed,
                M, N, K, y, partials, p.U, p.S);
}
}  // namespace

cudaError_t launch_linear_decode(const uint16_t* x, const int8_t* sign, const uint8_t* packed,
                                 int64_t M, int64_t N, int64_t K, uint16_t* y, void* ws,
                                 cudaStream_t st) {
  const GemvPlan p = make_plan(N, K, sm_count());
  auto* partials = static_cast<unsigned int*>(ws);
  auto* yy = reinterpret_cast<__nv_bfloat16*>(y);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  const cudaError_t e = M <= 8 ? launch_linear_nt<1>(x, sign, packed, m, n, k, yy, partials, p, st)
                               : launch_linear_nt<2>(x, sign, packed, m, n, k, yy, partials, p, st);
  if (e != cudaSuccess) return e;
  return launch_fixup(p, partials, yy, m, n, static_cast<int>(K / kGroup), st);
}

cudaError_t gemv_read_clear_error(unsigned int* err) {
  cudaError_t e = cudaMemcpyFromSymbol(err, g_gemv_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(unsigned int));
}

}  // namespace tern
