/*
 * tern.h -- C ABI of the GB300 (sm_103a) ternary-weight linear layer.
 *
 * The layer (page "RTX 5070 x2 ... Ternary-Bonsai-2-27B on vLLM TP=2",
 * qiita.com/nakanokensetsu/items/ecc183fae033565af7cb):
 *   - weights are codes in {-1, 0, +1} stored at 2 bits, with one fp16 scale
 *     per 128 consecutive elements of each output row (section "前提");
 *   - a block-wise Sylvester Hadamard rotation of width 1024, normalised by
 *     1/sqrt(1024) = 1/32, is applied to the input activations (section
 *     "前提" and section 1, split identity H1024[a;b] = [H512 a + H512 b ;
 *     H512 a - H512 b]);
 *   - decode: y[m,n] = sum_k code[n,k] s[n,k/128] xr[m,k] for M <= 16 tokens;
 *   - prefill (section 4): q[n,g] = round(127 s[n,g] / smax[n]),
 *     W_int8[n,k] = code[n,k] q[n,k/128] (exactly int8), per-token int8
 *     activations after the rotation, one int8 GEMM with int32 accumulation,
 *     then a per-row and per-token rescale to bf16.
 *
 * Notation: M tokens, N output rows, K input width (a multiple of 1024),
 * G = K/128 scale groups, B = K/1024 Hadamard blocks, Np = N rounded up to a
 * multiple of 16.
 *
 * Conventions for every entry point:
 *   - all data pointers are DEVICE pointers unless stated (host memory the
 *     GPU can address directly counts, see tern_host_accessible); the caller
 *     allocates and owns every buffer; the library allocates nothing and
 *     keeps no state besides a per-translation-unit device error word;
 *   - fp16 and bf16 data are passed as uint16_t bit patterns;
 *   - every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and returns after enqueueing its kernels;
 *   - kernels use programmatic dependent launch: each waits for the kernel
 *     before it in the stream before it reads anything that kernel may have
 *     written, and lets the next kernel start early.  One exception: the
 *     decode kernels (tern_gemv_decode, tern_gemv_decode_noalloc,
 *     tern_linear_decode) stream the packed weights before that wait, so the
 *     packed weights must be complete when the kernel before them starts.
 *     tern_pack ensures this for its own output (its packing kernel lets no
 *     later kernel start before it has finished); a caller that writes
 *     packed weights with its own kernel must let that kernel finish first
 *     (no programmatic early launch of what follows it);
 *   - argument errors are detected on the host before anything is enqueued
 *     and nothing is written; launch errors are reported as TERN_ERR_CUDA;
 *   - M == 0 (or N == 0) is a valid no-op returning TERN_OK;
 *   - buffers must be 16-byte aligned unless stated; rows are dense
 *     (leading dimension = the row length);
 *   - the kernels require a compute capability 10.3 device (GB300); on any
 *     other device the calls return TERN_ERR_UNSUPPORTED.
 */
#ifndef TERN_H_
#define TERN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TERN_OK = 0,
  TERN_ERR_INVALID_ARG = 1, /* null pointer for a required buffer, bad mode, negative size */
  TERN_ERR_SHAPE = 2,       /* K not a multiple of 1024, M out of range, sizes too large */
  TERN_ERR_ALIGN = 3,       /* a buffer is not 16-byte aligned */
  TERN_ERR_UNSUPPORTED = 4, /* no sm_103 device current */
  TERN_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  TERN_ERR_WORKSPACE = 6,   /* workspace missing or smaller than tern_workspace_bytes() */
  TERN_ERR_TIMEOUT = 7      /* a bounded device-side wait gave up (see tern_check) */
} tern_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* tern_status_str(int status);

/* Library ABI version (major * 100 + minor). */
int tern_version(void);

/* ------------------------------------------------------------------------
 * Packed weight format (defined by this library; the page does not give one)
 *
 * 2-bit field: u = code + 1 (-1 -> 0b00, 0 -> 0b01, +1 -> 0b10; 0b11 is
 * never written).
 *
 * Rows are padded with zero codes and zero scales to Np512 = N rounded up to
 * a multiple of 512.  `packed` is a sequence of 17408-byte units, unit
 * (rb * G + g) for row block rb (rows 512 rb .. 512 rb + 511) and group g
 * (k = 128 g .. 128 g + 127).  A unit holds
 *   bytes [0, 16384):      codes, 32 tiles of 16 rows.  Tile t (rows
 *       512 rb + 16 t ..) starts at byte 512 t; slot L (0..31) of the tile,
 *       bytes 512 t + 16 L .. + 15, holds four little-endian 32-bit words
 *       w_0..w_3.  With r = L / 4, c = L % 4, word p and field j (0..7):
 *         bits 2j..2j+1 of w_p:      u(row, k),
 *         bits 16+2j..17+2j of w_p:  u(row, k + 1),
 *       with row = 512 rb + 16 t + r + 8 (p % 2),
 *            k   = 128 g + 16 j + 2 c + 8 (p / 2);
 *   bytes [16384, 17408):  fp16 scales: tile t at 16384 + 32 t holds 8 pairs
 *       (s[512 rb + 16 t + r][g], s[512 rb + 16 t + r + 8][g]), r = 0..7.
 * Word p is register p of the A fragment of a 16 x 16 tensor-core tile for
 * every k16 step j of the group: w_p & (0x00030003 << 2j) for j < 6, and
 * (w_p >> 12) & (0x00030003 << 2(j - 6)) for j = 6, 7, read as an fp16 pair,
 * is (u(row, k), u(row, k + 1)) * 4^e * 2^-24 with e = j (j < 6) or j - 6
 * (a subnormal for e <= 4; the two lowest exponent bits, 2^-14 and 2^-13,
 * for e = 5): one AND per register.
 * ---------------------------------------------------------------------- */

/* Bytes of `packed` for an N x K weight: ceil(N/512) * (K/128) * 17408. */
size_t tern_packed_bytes(int64_t N, int64_t K);

/*
 * tern_pack -- load-time conversion of one layer's weights (page section
 * "前提" for the format; section 4 for the scale decomposition).
 *
 *   codes   int8 [N][K], values in {-1,0,+1} (other values: undefined result)
 *   scales  fp16 [N][G]
 * outputs (any may be NULL; packed is the decode operand, q / rscale / w_q
 * the prefill operands):
 *   packed         uint8, tern_packed_bytes(N,K) bytes, format above
 *   q              int8 [N][G]: rint((127*s)/smax) in fp32, half to even,
 *                  smax[n] = max_g |s[n,g]|; a zero row gives q = 0
 *   rscale         fp32 [N]: smax/127 (0 for a zero row)
 *   w_int8         int8 [N][K]: the exact int8 weight code*q[n,k/128] (section 4:
 *                  it fits int8 exactly); needs q and rscale non-NULL.
 *                  q and rscale must be both NULL or both non-NULL.
 * Requirements: K % 1024 == 0, 1 <= K <= 65536, N >= 0.
 */
tern_status tern_pack(const int8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
                      uint8_t* packed, int8_t* q, float* rscale, int8_t* w_int8, void* stream);

/* tern_widen_int8 -- int8 [rows][cols] -> the same integers held in fp16
 * (exact), the operand format of the sm_103a tensor cores' f16 kind (the
 * chip has no tcgen05 int8 kind).  Used at load time for the fp16-held
 * weight of tern_gemm_prefill_int8h.  Requirements: cols % 16 == 0;
 * rows * cols < 2^40. */
tern_status tern_widen_int8(const int8_t* src, int64_t rows, int64_t cols, uint16_t* dst,
                            void* stream);

/* ------------------------------------------------------------------------
 * tern_fwht_quant -- block Hadamard rotation of the activations (page
 * section "前提", section 1) and, in TERN_FWHT_I8 mode, the per-token int8
 * quantisation of section 4.
 *
 * The rotation: per token and per 1024-block, butterfly stages with stride
 * 1, 2, 4, ..., 512 (in that order; the last one is the page's split
 * identity), each (u, v) -> (u + v, u - v) in fp32, then * (1/32).  If
 * `sign` (int8 [K] of +-1) is given, x is multiplied by it first (the
 * optional "rotation sign table"); NULL means all +1.
 *
 *   x      bf16 [M][K]
 *   mode   TERN_FWHT_F32:    out = float xr[M][K]; out_scale unused (may be NULL)
 *          TERN_FWHT_DECODE: the decode GEMV's operand, M <= 16.  With
 *                 sh[m,b] = min(14 - E, 126), E = (biased exponent field of
 *                 the fp32 value max_{k in block b} |xr[m,k]|) - 127 (so
 *                 2^sh puts the block's largest magnitude in [2^14, 2^15))
 *                 and, for column k in k16 step j = (k % 128) / 16,
 *                 e = j (j < 6) or j - 6 (the power of four the packed field
 *                 of that step carries):
 *                 out = fp16 [M][K], fp16_rn(xr[m,k] * 2^(sh - 2e));
 *                 out_scale = float aux[G][48], one 192-byte record per
 *                 128-group g.  With X[g,m] = the fp32 sum over k in g of
 *                 out[m,k] * 2^(2e - 24) (every term exact; the 8
 *                 consecutive columns 8q .. 8q + 7 left to right, then the
 *                 16 partial sums by a butterfly p[q] += p[q ^ s],
 *                 s = 1, 2, 4, 8) and 0 for m >= M: aux[g][4i .. 4i + 3] =
 *                 (0 - X[g,2i], 0 - X[g,2i+1], 0 - X[g,2i], 0 - X[g,2i+1])
 *                 for i = 0..7 (fp32; the tensor core's accumulator quad:
 *                 the fields hold code + 1, so each group sum starts at minus
 *                 the offset), aux[g][32 + m] = 2^(12 - sh) of the block
 *                 holding g (0 for m >= M), the block's fold factor
 *          TERN_FWHT_F16:    out = fp16 [M][K], the fp16 prefill variant's
 *                 operand: fp16_rn(xr[m,k] * 2^sh[m,b]); out_scale = float
 *                 [M][B] holding 2^-sh[m,b] (exact); any M
 *          TERN_FWHT_I8:     out = int8 xq [M][K]; out_scale = float tscale[M]:
 *                 a = max_k |xr[m,k]|, tscale = a/127 (fp32),
 *                 xq = clamp(rint(xr / tscale), -127, 127) (fp32 division,
 *                 half to even); a == 0 gives xq = 0 and tscale = 0.
 *          TERN_FWHT_I8H:    the same xq held in fp16 [M][K] (exact), the
 *                 operand of tern_gemm_prefill_int8h and _packed.
 * Requirements: K % 1024 == 0, K <= 65536 (K <= 32768 in the two int8 modes),
 * M >= 0 (M <= 16 in TERN_FWHT_DECODE mode); `sign` may be unaligned.
 * ---------------------------------------------------------------------- */
#define TERN_FWHT_F32 0
#define TERN_FWHT_DECODE 1
#define TERN_FWHT_I8 2
#define TERN_FWHT_F16 3
#define TERN_FWHT_I8H 4
tern_status tern_fwht_quant(const uint16_t* x, int64_t M, int64_t K, const int8_t* sign,
                            int mode, void* out, float* out_scale, void* stream);

/* ------------------------------------------------------------------------
 * K-split tensor parallelism (page section 1, "TP=2 への移植"): when a
 * row-parallel layer's input width is split over ranks, a shard boundary
 * may fall in the middle of a 1024-block (down 17408 over 2 ranks: 8704 =
 * 8.5 blocks).  Each rank transforms its own 512-element half with H512,
 * the ranks exchange those halves (an all-gather), and the rank holding the
 * first half takes their sum, the rank holding the second half their
 * difference (the split identity H1024[a;b] = [H512 a + H512 b ; H512 a -
 * H512 b], which is the last butterfly stage), times 1/32.  The rotated
 * values are then bit for bit those of the whole-width rotation.
 *
 * A rank's shard x: bf16 [M][Kr] (dense rows, Kr = 1024 nb + 512 (lead +
 * trail)): an optional leading half (the second half of a block shared with
 * the previous rank), nb whole blocks, an optional trailing half (the first
 * half of a block shared with the next rank).  Its padded layout, of width
 * Kp = 1024 (nb + lead + trail), is [lead block] [nb whole blocks] [trail
 * block]; in a padded half block the rank's 512 values come first and the
 * other 512 are zero (the rank's weights get 512 zero columns there, so the
 * GEMV and GEMM run unchanged on Kp).
 *
 * tern_fwht_shard -- the rank-local part: whole blocks rotated into
 *   xr (fp32 [M][Kp], at their padded positions; the half blocks' places are
 *   left for tern_fwht_combine), and the unnormalised H512 (canonical stages
 *   of stride 1 .. 256, fp32) of the leading / trailing half into
 *   h_lead / h_trail (fp32 [M][512]; NULL when that half is absent).
 *   sign: int8 [Kr] of +-1 for the shard's columns, or NULL.
 *   Requirements: lead, trail in {0,1}; Kr - 512 (lead + trail) a
 *   non-negative multiple of 1024; Kp <= 65536; M Kp < 2^31.
 * tern_fwht_combine -- one split block after the exchange: h_first is the
 *   H512 of the block's first half (from the rank that holds it), h_second
 *   of its second half; part 0 (this rank holds the first half) writes
 *   (h_first + h_second) / 32, part 1 writes (h_first - h_second) / 32, into
 *   xr[:, 1024 blk .. 1024 blk + 511] of the padded layout (width Kp), and
 *   zeros into xr[:, 1024 blk + 512 .. 1024 blk + 1023].
 * tern_quant_rotated -- quantise rotated fp32 activations xr [M][K]
 *   (K % 1024 == 0) exactly as tern_fwht_quant does after its rotation:
 *   mode TERN_FWHT_DECODE (the decode GEMV's operand, M <= 16),
 *   TERN_FWHT_F16 (fp16 + per-block factors), TERN_FWHT_I8 (int8 xq +
 *   per-token tscale) or TERN_FWHT_I8H (the same xq held in fp16).  After a K split each rank quantises its own padded
 *   shard (per-token int8 scales are the rank's own).
 * ---------------------------------------------------------------------- */
tern_status tern_fwht_shard(const uint16_t* x, int64_t M, int64_t Kr, int lead, int trail,
                            const int8_t* sign, float* xr, float* h_lead, float* h_trail,
                            void* stream);
tern_status tern_fwht_combine(const float* h_first, const float* h_second, int64_t M, int part,
                              float* xr, int64_t Kp, int64_t blk, void* stream);
tern_status tern_quant_rotated(const float* xr, int64_t M, int64_t K, int mode, void* out,
                               float* out_scale, void* stream);

/* ------------------------------------------------------------------------
 * tern_gemv_decode -- decode GEMV for 1 <= M <= 16 tokens:
 *     y[m,n] = bf16_rn( sum_g s[n,g] * sum_{k in g} code[n,k] * xr[m,k] )
 * computed from the packed weights and the TERN_FWHT_DECODE operand with fp16
 * tensor-core products (the field read u * 4^e * 2^-24 times the operand,
 * exact) and fp32 accumulation; each group's sum starts at minus its offset
 * (the fields hold code + 1), is scaled by the group's scale, each block's
 * sum by its fold factor, and the total by 2^12 before the bf16 rounding.
 * Every weight byte is read once for all M tokens.
 *
 *   packed                  from tern_pack (this layer's N, K)
 *   xh, xs                  from tern_fwht_quant(mode = TERN_FWHT_DECODE):
 *                           fp16 [M][K] and the float aux [K/128][48] records
 *   y                       bf16 [M][N]
 *   ws, ws_bytes            workspace of at least
 *                           tern_workspace_bytes(TERN_OP_GEMV, M, N, K) bytes,
 *                           16-byte aligned, ZERO-FILLED before its first use
 *                           (tern_workspace_init); every call leaves it
 *                           zero-filled again on completion (it holds the
 *                           partial sums of 512-row blocks that several CTAs
 *                           share).  Calls that share a workspace must not run
 *                           concurrently.
 * Requirements: 1 <= M <= 16 (M == 0 is a no-op), K % 1024 == 0, K <= 65536.
 * A call is the GEMV kernel and, when some 512-row block is shared by more
 * than four CTAs (M <= 8) or by several CTAs (M > 8), a fixup kernel that
 * adds those blocks' partial sums in slot order.  Device-side waits are
 * bounded; a wait that gives up makes the call's outputs undefined and is
 * reported by tern_check(); the workspace must then be zero-filled again
 * (tern_workspace_init) before its next use.
 * ---------------------------------------------------------------------- */
tern_status tern_gemv_decode(const uint8_t* packed, const uint16_t* xh, const float* xs,
                             int64_t M, int64_t N, int64_t K, uint16_t* y, void* ws,
                             size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * tern_gemv_decode_f32 -- the same decode GEMV from fp32 rotated activations:
 *     y[m,n] = bf16_rn( sum_g s[n,g] * sum_{k in g} code[n,k] * xr[m,k] )
 * Page "RTX 5070 x2 ... Ternary-Bonsai-2-27B on vLLM TP=2", section "前提".
 * The call first forms the decode operand from xr exactly as
 * tern_quant_rotated(TERN_FWHT_DECODE) does (into the workspace), then runs
 * tern_gemv_decode on it: results are bit-identical to those two calls.
 *
 *   packed                  from tern_pack (this layer's N, K)
 *   xr                      float [M][K], the rotated activations (for
 *                           example tern_fwht_quant(TERN_FWHT_F32) output)
 *   y                       bf16 [M][N]
 *   ws, ws_bytes            workspace of at least
 *                           tern_workspace_bytes(TERN_OP_GEMV_F32, M, N, K)
 *                           bytes, 16-byte aligned, zero-filled before its
 *                           first use (tern_workspace_init); its first
 *                           tern_workspace_bytes(TERN_OP_GEMV, M, N, K) bytes
 *                           are the GEMV's and are left zero-filled again by
 *                           every call, the rest holds the operand.
 * Requirements and errors as for tern_gemv_decode.
 * ---------------------------------------------------------------------- */
tern_status tern_gemv_decode_f32(const uint8_t* packed, const float* xr, int64_t M, int64_t N,
                                 int64_t K, uint16_t* y, void* ws, size_t ws_bytes,
                                 void* stream);

/* ------------------------------------------------------------------------
 * tern_linear_decode -- the layer's whole decode path in one launch:
 *     y = tern_gemv_decode(tern_fwht_quant(x, sign, TERN_FWHT_DECODE))
 * Page "RTX 5070 x2 ... Ternary-Bonsai-2-27B on vLLM TP=2", section "前提"
 * (input-side block rotation, then the ternary g128 product).  The rotation
 * is folded into the GEMV's prologue: each CTA rotates only the 1024-blocks
 * its share of the weights needs and keeps the fp16 operand on chip, so the
 * separate rotation launch and its [M][K] round trip through memory go away.
 * The result is bit-identical to the two calls.
 *
 *   x                       bf16 [M][K], 16-byte aligned
 *   sign                    optional +-1 per k (NULL = identity), as for
 *                           tern_fwht_quant; any alignment
 *   packed, M, N, K, y, ws, ws_bytes, stream: as for tern_gemv_decode (the
 *                           workspace size is tern_workspace_bytes(
 *                           TERN_OP_GEMV, M, N, K))
 * Requirements and errors as for tern_gemv_decode.
 * ---------------------------------------------------------------------- */
tern_status tern_linear_decode(const uint16_t* x, const int8_t* sign, const uint8_t* packed,
                               int64_t M, int64_t N, int64_t K, uint16_t* y, void* ws,
                               size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * tern_gemv_decode_noalloc -- the same decode GEMV as tern_gemv_decode, for
 * callers that cannot allocate device memory.  The page has no counterpart.
 *
 * An application that embeds this layer and owns every byte of device memory
 * through its own pool, handing the layer only its inputs and outputs, cannot
 * give it a separate workspace, and a decode loop that must never stall
 * cannot call cudaMalloc, which may synchronise the device.  This call takes
 * no workspace and allocates nothing: its scratch (the partial sums of row
 * blocks shared by several CTAs) lives in a static device array of
 * TERN_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library holds until the process exits.
 *
 *   packed, xh, xs, M, N, K, y, stream: as for tern_gemv_decode.
 * Returns TERN_ERR_WORKSPACE when tern_workspace_bytes(TERN_OP_GEMV, M, N, K)
 * exceeds TERN_NOALLOC_SCRATCH_BYTES (nothing is launched).  The first call
 * on a device, with that device current, looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture.  Later calls outside a stream capture look the address up
 * again (a device reset moves the array; a call inside a capture uses the
 * cached address, so capture no call after a reset before an uncaptured one
 * has run).  Every call shares the one array: each call zero-fills the part
 * it uses on its stream first (so a call that gave up waiting leaves nothing
 * behind), and calls that overlap on the GPU race on the array.
 * The limit, 24 MiB, covers every workload shape of the 27B model's linear
 * stack up to M = 16 (gate/up 5120 -> 34816 at M = 16 needs about 17 MiB on
 * a 152-SM GB300).
 * ---------------------------------------------------------------------- */
#define TERN_NOALLOC_SCRATCH_BYTES (24u << 20)
tern_status tern_gemv_decode_noalloc(const uint8_t* packed, const uint16_t* xh, const float* xs,
                                     int64_t M, int64_t N, int64_t K, uint16_t* y,
                                     void* stream);

/* ------------------------------------------------------------------------
 * tern_gemm_prefill_int8 -- the int8 prefill GEMM of page section 4:
 *     acc[m,n] = sum_k xq[m,k] * W_int8[n,k]            (exact int32)
 *     y[m,n]   = bf16_rn(((float)acc[m,n] * tscale[m]) * rscale[n])
 * on int8 operands.  sm_103a's tensor cores have no int8 kind, so the call
 * holds both operands' integers in fp16 in its workspace (exact), then runs
 * the tcgen05 GEMM of tern_gemm_prefill_int8h on them; the f16 kind
 * multiplies them exactly and the kernel keeps every fp32 partial sum below
 * 2^24 (1024-wide chunks, then int32), so acc is bit-exact.
 *
 *   xq      int8 [M][K] (TERN_FWHT_I8 output), tscale fp32 [M]
 *   w_int8  int8 [N][K] (tern_pack output),    rscale fp32 [N]
 *   y       bf16 [M][N]
 *   acc     int32 [M][N] or NULL
 *   ws      device workspace (any contents) of at least
 *           tern_workspace_bytes(TERN_OP_GEMM_INT8, M, N, K) bytes: the two
 *           fp16 operand copies, then the K-split pieces of
 *           tern_gemm_prefill_int8h.  It is required.
 * Requirements and errors as for tern_gemm_prefill_int8h (TERN_ERR_WORKSPACE
 * for a missing or small workspace).  A caller that keeps the fp16-held
 * weight (tern_widen_int8, twice the bytes) saves the weight's widening on
 * every call by calling tern_gemm_prefill_int8h directly.
 * ---------------------------------------------------------------------- */
tern_status tern_gemm_prefill_int8(const int8_t* xq, const float* tscale, const int8_t* w_int8,
                                   const float* rscale, int64_t M, int64_t N, int64_t K,
                                   uint16_t* y, int32_t* acc, void* ws, size_t ws_bytes,
                                   void* stream);

/* ------------------------------------------------------------------------
 * tern_gemm_prefill_int8h -- the same GEMM on the int8 integers held in fp16
 * (tcgen05.mma kind::f16, TMA-fed, TMEM accumulators, fused rescale).  Tiles
 * are 128 tokens x 256 weight rows per CTA up to M = 128; above, 256 tokens x
 * 256 weight rows per cluster of two CTAs sharing each MMA (cta_group::2):
 *
 *   xq      fp16 [M][K] holding xq (TERN_FWHT_I8H output), tscale fp32 [M]
 *   w_q     fp16 [N][K] holding W_int8 (tern_widen_int8 of tern_pack's
 *           w_int8), rscale fp32 [N]
 *   y       bf16 [M][N]
 *   acc     int32 [M][N] or NULL
 *   ws      optional device workspace (any contents) of
 *           tern_workspace_bytes(TERN_OP_GEMM, M, N, K) bytes.  With it, a
 *           call whose tiles fill the GPU unevenly splits K in slices of
 *           whole 1024-chunks -- in every tile, or only in the tiles of the
 *           last, partial wave, as a cost model picks: the slices' exact
 *           int32 partial sums go to one piece per tile and slice in ws
 *           ([128][256], or [256][256] for the pairs' tiles) and a second
 *           kernel adds them and rescales (same results bit for bit).  With
 *           NULL (or less) the call runs unsplit.  A split call leaves partial sums
 *           in ws: a buffer also used as a tern_gemv_decode workspace must
 *           be zero-filled again (tern_workspace_init) before that call.
 * Requirements: K % 1024 == 0, K <= 65536, M >= 0, N % 16 == 0, N >= 0.
 * Device-side waits are bounded; a wait that gives up makes the call's
 * outputs undefined and is reported by tern_check().
 * ---------------------------------------------------------------------- */
tern_status tern_gemm_prefill_int8h(const uint16_t* xq, const float* tscale, const uint16_t* w_q,
                                    const float* rscale, int64_t M, int64_t N, int64_t K,
                                    uint16_t* y, int32_t* acc, void* ws, size_t ws_bytes,
                                    void* stream);

/* ------------------------------------------------------------------------
 * tern_gemm_prefill_packed -- the same int8 prefill GEMM (page section 4)
 * read straight from the decode's 2-bit packed weights and q, with no
 * W_int8 in memory (page section 6 measured the run-time 2-bit -> int8
 * expansion; here it happens in shared memory beside the tensor cores):
 *     W_int8[n,k] = code[n,k] * q[n,k/128]     (formed on chip, never stored)
 *     acc[m,n]    = sum_k xq[m,k] * W_int8[n,k]  (exact int32)
 *     y[m,n]      = bf16_rn(((float)acc[m,n] * tscale[m]) * rscale[n])
 * Results are bit-identical to tern_gemm_prefill_int8 on the same layer.
 * Tiles: 128 tokens x 256 weight rows up to M = 128; above, 256 weight rows
 * x 256 tokens per cluster of two CTAs (cta_group::2; the weights on the
 * MMA's M side, each CTA expanding its 128 rows, so each expanded weight
 * serves 256 tokens).  The weights are read at 2 bits each (plus q) once
 * per token block, so mid-size M costs the packed bytes instead of the
 * 2-byte expanded weight.
 *
 *   xq      fp16 [M][K] holding xq (TERN_FWHT_I8H output), tscale fp32 [M]
 *   packed  tern_pack's `packed` output (tern_packed_bytes(N, K) bytes)
 *   q       int8 [N][G] and rscale fp32 [N] (tern_pack outputs)
 *   y       bf16 [M][N]
 *   acc     int32 [M][N] or NULL
 *   ws      device workspace of tern_workspace_bytes(TERN_OP_GEMM_PACKED,
 *           M, N, K) bytes (any contents; NULL when that is 0).  When the
 *           tiles fill the GPU unevenly, K ranges are split in S slices of
 *           whole 128-groups whose exact int32 partial sums a second kernel
 *           adds (integer sums: the same result in any order) before the
 *           rescale (tern_kernel_launches).  Up to 128 tokens, with too few
 *           tiles for the GPU, every tile is split and the slices' sums go
 *           to S planes [M][N] of ws; above, the whole waves of pair tiles
 *           stay whole and only the last, partial wave's tiles (all tiles
 *           when there are fewer than pairs) are split, one [256][256]
 *           piece per tile and slice in ws.  As for tern_gemm_prefill_int8,
 *           a split call leaves partial sums in ws.
 * Requirements: K % 1024 == 0, K <= 65536, N % 16 == 0, 0 <= M, N <= 2^24.
 * Device-side waits are bounded; a wait that gives up makes the call's
 * outputs undefined and is reported by tern_check().
 * ---------------------------------------------------------------------- */
tern_status tern_gemm_prefill_packed(const uint16_t* xq, const float* tscale,
                                     const uint8_t* packed, const int8_t* q, const float* rscale,
                                     int64_t M, int64_t N, int64_t K, uint16_t* y, int32_t* acc,
                                     void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * The fp16 prefill variant (compared with the int8 path of page section 4).
 * On sm_103a the int8 values of section 4 already run on the f16 tensor
 * kind (there is no tcgen05 int8 kind), so an fp16 GEMM costs the same MMA
 * time; it keeps the scales exact instead of rounding them to q, and the
 * activations at fp16 precision (TERN_FWHT_F16) instead of per-token int8.
 *
 * tern_expand_fp16 -- w_h fp16 [N][K] = code[n,k] * s[n, k/128] (exact).
 *   codes int8 [N][K], scales fp16 [N][G].  Requirements: K % 1024 == 0,
 *   K <= 65536, N * K < 2^34.
 * tern_gemm_prefill_fp16 --
 *     y[m,n] = bf16_rn( sum_b xs[m,b] * sum_{k in block b} xh[m,k] w_h[n,k] )
 *   with xh fp16 [M][K] and xs fp32 [M][K/1024] the fp16 operand of
 *   tern_fwht_quant(TERN_FWHT_F16) (any M), each block's sum accumulated
 *   in fp32 by the tensor cores and the blocks added in fp32 in order.
 *   y bf16 [M][N].  ws: optional workspace as for tern_gemm_prefill_int8
 *   (TERN_OP_GEMM); a split call adds fp32 slice sums in slice order, so
 *   its rounding differs from the unsplit order.  Requirements:
 *   K % 1024 == 0, K <= 65536, N % 16 == 0, 0 <= M, N <= 2^24.
 * ---------------------------------------------------------------------- */
tern_status tern_expand_fp16(const int8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
                             uint16_t* w_h, void* stream);
tern_status tern_gemm_prefill_fp16(const uint16_t* xh, const float* xs, const uint16_t* w_h,
                                   int64_t M, int64_t N, int64_t K, uint16_t* y, void* ws,
                                   size_t ws_bytes, void* stream);

/* Workspace sizing and initialisation. */
#define TERN_OP_GEMV 1
#define TERN_OP_GEMM 2
#define TERN_OP_GEMM_PACKED 3
#define TERN_OP_GEMV_F32 4
#define TERN_OP_GEMM_INT8 5
size_t tern_workspace_bytes(int op, int64_t M, int64_t N, int64_t K);
/* 1 if the GPU current on this thread can load and store `host` directly
 * at that same address -- a pinned host buffer mapped into the device's
 * address space, or any host memory on a system whose GPU walks the host
 * page tables (Grace-Blackwell, over NVLink-C2C) -- else 0.  Such a pointer
 * may be passed wherever these calls take a device pointer: the kernels
 * then read their input from, or write their output to, host memory without
 * a separate copy. */
int tern_host_accessible(const void* host);

/* Number of kernels one call launches at this shape on the current device
 * (0 for an empty call or an unknown op): for TERN_OP_GEMV the GEMV kernel,
 * plus the fixup kernel when a 512-row block is shared by more CTAs than the
 * GEMV sums in place (tern_gemv_decode, tern_linear_decode and
 * tern_gemv_decode_noalloc launch the same count); for TERN_OP_GEMV_F32 one
 * more (the operand's quantisation kernel); for TERN_OP_GEMM the
 * int8h (or fp16) GEMM, plus its finishing kernel when it is given the
 * workspace and splits K; for TERN_OP_GEMM_INT8 two more (the operands'
 * widening); for TERN_OP_GEMM_PACKED the GEMM, plus the
 * rescale kernel when its tiles are split along K.  Host-only; launch
 * counting for CUDA-graph sizing and profiling. */
int tern_kernel_launches(int op, int64_t M, int64_t N, int64_t K);
/* Zero-fill `bytes` of device memory at ws on `stream` (asynchronous). */
tern_status tern_workspace_init(void* ws, size_t bytes, void* stream);

/* Synchronise `stream`, then read and clear the device error words.
 * Returns TERN_ERR_TIMEOUT if a bounded device-side wait gave up since the
 * last check, TERN_ERR_CUDA on a sticky CUDA error, else TERN_OK. */
tern_status tern_check(void* stream);

/* Self-test of the failure path of the bounded device-side waits: launches
 * one warp on `stream` that waits, with the kernels' own wait helper, on a
 * barrier nothing ever completes, gives up after `polls` polls
 * (1 <= polls <= TERN_SELFTEST_MAX_POLLS) and records it in the error word,
 * so that the next tern_check() returns TERN_ERR_TIMEOUT (and clears it).
 * Nothing else is touched, no memory is faulted and the context stays
 * usable.  TERN_ERR_INVALID_ARG for polls out of range, TERN_ERR_UNSUPPORTED
 * without an sm_103 device. */
#define TERN_SELFTEST_MAX_POLLS (1u << 20)
tern_status tern_selftest_wait(uint32_t polls, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TERN_H_ */
