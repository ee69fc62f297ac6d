"""CPU oracle for the ternary-weight linear layer.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain reference that the
CUDA library is checked against.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it; the
product path never does.  It shares no code with the CUDA kernels.

Source of the method: the page "RTX 5070 x2 ... Ternary-Bonsai-2-27B on vLLM
TP=2" (qiita.com/nakanokensetsu/items/ecc183fae033565af7cb):

* "前提" (premises): weights are codes in {-1,0,+1} stored at 2 bits with one
  scale per 128 elements of a row, and a block-wise Hadamard rotation is
  applied on the input side;
* section 1 "TP=2 への移植": the rotation is a Sylvester Hadamard of block 1024
  with the split identity H1024[a;b] = [H512 a + H512 b ; H512 a - H512 b],
  which is the last butterfly stage of the kernel;
* section 4 "効いた高速化", int8 prefill: q[n,g] = round(127 s[n,g] / smax[n]),
  W_int8[n,k] = code[n,k] q[n,k/128] fits int8 exactly, activations are
  quantised to int8 per token after the rotation, one int8 GEMM, then a
  per-row and per-token rescale.

Two references live here:

O1 (exact, fp64)        rotate_f64 / dequant_f64 / linear_f64
O2 (int8 path, spec-exact fp32 operation sequence)
                        fwht_f32 / quant_tokens / decompose_scales /
                        w_int8 / acc_int8 / y_int8 / linear_int8
K split (section 1)     fwht_half_f32 / ksplit_combine / ksplit_rotate_f32

plus the 2-bit storage format (pack_weights / unpack_weights), the decode
GEMV's activation operand (decode_operand: fp16 with a power of two per block
and per k16 step, plus per-group offsets and per-block fold factors) and the
fp16 prefill variant's operand (f16_operand), which the pages leave open and
this library defines (see ``include/tern.h``).

Readings of the pages taken here (each is also listed in the design notes):
* natural (Sylvester) order H, not sequency order; normalised by 1/32 per block;
* the butterfly stages run with stride 1, 2, 4, ..., 512, so the stride-512
  stage (the printed split identity) is the last one;
* the optional "rotation sign table" is a +-1 vector applied to x before H;
* group index g = floor(k/128) within the row;
* smax[n] = max_g |s[n,g]|; q = rint((127*s)/smax) in fp32, left to right as
  printed, round half to even; rscale = smax/127; a zero row gives q = 0,
  rscale = 0;
* per-token symmetric absmax quantisation over the whole row of K:
  tscale = absmax/127, xq = clamp(rint(xr / tscale), -127, 127); a zero token
  gives xq = 0, tscale = 0;
* y = bf16_rn(((float)acc * tscale[m]) * rscale[n]), fp32 left to right.
"""

from __future__ import annotations

import numpy as np

HBLOCK = 1024          # Hadamard block width (the page's section 1)
GROUP = 128            # elements per scale group (the page's premises)
INV_SQRT_BLOCK = 1.0 / 32.0


# --------------------------------------------------------------------------
# Hadamard rotation
# --------------------------------------------------------------------------

def hadamard_dense(n: int) -> np.ndarray:
    """Natural-order Sylvester Hadamard matrix of size n (fp64, entries +-1).

    H_1 = [1];  H_2m = [[H_m, H_m], [H_m, -H_m]]  (the page's section 1: the
    recursive Sylvester structure behind the split identity).
    """
    if n < 1 or (n & (n - 1)) != 0:
        raise ValueError("n must be a power of two")
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


_H1024 = None


def _h1024() -> np.ndarray:
    global _H1024
    if _H1024 is None:
        _H1024 = hadamard_dense(HBLOCK)
    return _H1024


def rotate_f64(x, sign=None) -> np.ndarray:
    """O1 rotation: xr = (I_B kron H1024/32) (sign * x), exactly, in fp64.

    Computed as a dense matrix product per 1024-block (the page's premises and
    section 1), deliberately not as butterflies.
    x: [M, K] (any float dtype), K a multiple of 1024.  sign: None or [K] of +-1.
    """
    x = np.asarray(x, dtype=np.float64)
    m, k = x.shape
    if k % HBLOCK:
        raise ValueError("K must be a multiple of 1024")
    if sign is not None:
        x = x * np.asarray(sign, dtype=np.float64)[None, :]
    h = _h1024()
    out = np.empty_like(x)
    for b in range(k // HBLOCK):
        blk = x[:, b * HBLOCK:(b + 1) * HBLOCK]
        out[:, b * HBLOCK:(b + 1) * HBLOCK] = (blk @ h.T) * INV_SQRT_BLOCK
    return out


def fwht_f32(x, sign=None) -> np.ndarray:
    """O2 rotation: the canonical fast Walsh-Hadamard transform in fp32.

    Per 1024-block, butterfly stages with stride h = 1, 2, 4, ..., 512 in that
    order; each butterfly maps (u, v) -> (u + v, u - v) with u the lower index.
    The last stage (h = 512) is the split identity printed on the page,
    section 1.  Then every element is multiplied by 1/32 (exact).  Every
    operation is one correctly rounded fp32 add, subtract or multiply.
    x: [M, K]; bf16 inputs must be passed already widened to fp32 (exact).
    """
    x = np.asarray(x, dtype=np.float32)
    m, k = x.shape
    if k % HBLOCK:
        raise ValueError("K must be a multiple of 1024")
    if sign is not None:
        x = x * np.asarray(sign, dtype=np.float32)[None, :]
    v = x.reshape(m, k // HBLOCK, HBLOCK).copy()
    h = 1
    while h < HBLOCK:
        w = v.reshape(m, k // HBLOCK, HBLOCK // (2 * h), 2, h)
        lo = w[:, :, :, 0, :]
        hi = w[:, :, :, 1, :]
        s = lo + hi
        d = lo - hi
        v = np.stack([s, d], axis=3).reshape(m, k // HBLOCK, HBLOCK)
        h *= 2
    v = v * np.float32(INV_SQRT_BLOCK)
    return v.reshape(m, k).astype(np.float32)


# --------------------------------------------------------------------------
# K split over ranks with the half-block exchange (the page's section 1)
# --------------------------------------------------------------------------

HALF = HBLOCK // 2


def fwht_half_f32(x) -> np.ndarray:
    """Unnormalised H512 of each 512-element row in fp32: the butterfly
    stages of stride 1, 2, ..., 256 of the canonical order, i.e. what one rank
    computes on its half of a block that the K split cuts in the middle
    (the page's section 1).  x: [M, 512]."""
    v = np.asarray(x, dtype=np.float32).copy()
    m = v.shape[0]
    if v.shape[1] != HALF:
        raise ValueError("rows of 512 elements expected")
    h = 1
    while h < HALF:
        w = v.reshape(m, HALF // (2 * h), 2, h)
        lo = w[:, :, 0, :]
        hi = w[:, :, 1, :]
        v = np.stack([lo + hi, lo - hi], axis=2).reshape(m, HALF)
        h *= 2
    return v


def ksplit_combine(h_first, h_second, part) -> np.ndarray:
    """The exchange of the page's section 1: with a = H512 of a block's first
    half and b = H512 of its second half, H1024 [a; b] = [a + b ; a - b]; the
    rank that holds the first half keeps (a + b) / 32 (part 0), the rank that
    holds the second half keeps (a - b) / 32 (part 1).  fp32."""
    a = np.asarray(h_first, dtype=np.float32)
    b = np.asarray(h_second, dtype=np.float32)
    v = (a + b) if part == 0 else (a - b)
    return (v * np.float32(INV_SQRT_BLOCK)).astype(np.float32)


def ksplit_rotate_f32(x, world: int, sign=None):
    """Rotation of x [M, K] whose columns are split in `world` equal
    contiguous shards (K / world a multiple of 512), as the page's section 1
    runs it: each rank rotates its whole blocks itself (fwht_f32), a block cut
    in the middle is transformed half by half on its two ranks
    (fwht_half_f32), the halves are exchanged, and each rank combines them
    (ksplit_combine).  Returns the ranks' rotated columns, in order."""
    x = np.asarray(x, dtype=np.float32)
    if sign is not None:
        x = x * np.asarray(sign, dtype=np.float32)[None, :]
    m, k = x.shape
    if k % world or (k // world) % HALF:
        raise ValueError("each shard must be a whole number of half blocks")
    kr = k // world
    bounds = [(r * kr, (r + 1) * kr) for r in range(world)]
    # every rank's transform of each half block it holds (rank-local step)
    halves = {}
    for r, (k0, k1) in enumerate(bounds):
        if k0 % HBLOCK:
            halves[(r, "lead")] = fwht_half_f32(x[:, k0:k0 + HALF])
        if k1 % HBLOCK:
            halves[(r, "trail")] = fwht_half_f32(x[:, k1 - HALF:k1])
    out = []
    for r, (k0, k1) in enumerate(bounds):
        parts = []
        if k0 % HBLOCK:   # second half of a block shared with rank r - 1
            parts.append(ksplit_combine(halves[(r - 1, "trail")], halves[(r, "lead")], 1))
        a = k0 + (HALF if k0 % HBLOCK else 0)
        b = k1 - (HALF if k1 % HBLOCK else 0)
        if b > a:
            parts.append(fwht_f32(x[:, a:b]))
        if k1 % HBLOCK:   # first half of a block shared with rank r + 1
            parts.append(ksplit_combine(halves[(r, "trail")], halves[(r + 1, "lead")], 0))
        out.append(np.concatenate(parts, axis=1))
    return out


# --------------------------------------------------------------------------
# Weights: dequantisation (O1) and the scale decomposition (O2)
# --------------------------------------------------------------------------

def dequant_f64(codes, scales) -> np.ndarray:
    """O1 weight: W[n,k] = code[n,k] * s[n, k // 128] in fp64 (the page's premises)."""
    codes = np.asarray(codes)
    s = np.asarray(scales).astype(np.float64)
    return codes.astype(np.float64) * np.repeat(s, GROUP, axis=1)


def decompose_scales(scales):
    """Scale decomposition of the page's section 4 (int8 prefill).

    smax[n] = max_g |s[n,g]| (fp32, exact from fp16),
    q[n,g]  = rint((127 * s[n,g]) / smax[n]) with both operations in fp32,
              round half to even (127*s is exact in fp32 for fp16 s),
    rscale[n] = smax[n] / 127 (fp32).
    A row whose scales are all zero gets q = 0 and rscale = 0.
    Returns (q int8 [N,G], rscale fp32 [N], smax fp32 [N]).
    """
    s = np.asarray(scales).astype(np.float32)
    smax = np.max(np.abs(s), axis=1).astype(np.float32)
    q = np.zeros(s.shape, dtype=np.float32)
    nz = smax > 0
    num = (np.float32(127.0) * s[nz]).astype(np.float32)
    q[nz] = np.rint((num / smax[nz, None]).astype(np.float32))
    rscale = np.zeros_like(smax)
    rscale[nz] = (smax[nz] / np.float32(127.0)).astype(np.float32)
    if np.any(np.abs(q) > 127):
        raise AssertionError("|q| > 127")
    return q.astype(np.int8), rscale, smax


def w_int8(codes, q) -> np.ndarray:
    """W_int8[n,k] = code[n,k] * q[n, k // 128]  (the page's section 4).  int16 result."""
    codes = np.asarray(codes).astype(np.int16)
    qq = np.repeat(np.asarray(q).astype(np.int16), GROUP, axis=1)
    return codes * qq


# --------------------------------------------------------------------------
# Activations: per-token int8 quantisation (O2)
# --------------------------------------------------------------------------

def quant_tokens(xr):
    """Per-token symmetric int8 quantisation of the rotated activations.

    The page's section 4: activations are quantised to int8 per token after the
    Hadamard rotation.  a[m] = max_k |xr[m,k]| (fp32), tscale[m] = a[m]/127
    (fp32), xq = clamp(rint(xr / tscale), -127, 127) with the division and the
    rounding in fp32 (half to even).  A zero token gives xq = 0, tscale = 0.
    Returns (xq int8 [M,K], tscale fp32 [M]).
    """
    xr = np.asarray(xr, dtype=np.float32)
    a = np.max(np.abs(xr), axis=1).astype(np.float32) if xr.shape[1] else \
        np.zeros(xr.shape[0], np.float32)
    tscale = (a / np.float32(127.0)).astype(np.float32)
    xq = np.zeros(xr.shape, dtype=np.float32)
    nz = tscale > 0
    xq[nz] = np.rint((xr[nz] / tscale[nz, None]).astype(np.float32))
    xq = np.clip(xq, -127, 127)
    tscale = np.where(nz, tscale, np.float32(0)).astype(np.float32)
    return xq.astype(np.int8), tscale


# --------------------------------------------------------------------------
# The int8 GEMM and its rescale (O2)
# --------------------------------------------------------------------------

INT32_MAX = 2 ** 31 - 1


def acc_int8(xq, w) -> np.ndarray:
    """acc[m,n] = sum_k xq[m,k] * W_int8[n,k], exact.

    The products and all partial sums are integers of magnitude below 2^53,
    so an fp64 matrix product is exact in any summation order.  The result
    is checked to fit int32.  Returns int64 [M,N].
    """
    a = np.asarray(xq).astype(np.float64)
    b = np.asarray(w).astype(np.float64)
    k = a.shape[1]
    if k and 127.0 * 127.0 * k >= 2.0 ** 53:
        raise ValueError("K too large for exact fp64 accumulation")
    acc = a @ b.T
    acc_i = np.rint(acc).astype(np.int64)
    if np.any(np.abs(acc_i) > INT32_MAX):
        raise AssertionError("accumulator exceeds int32")
    return acc_i


def bf16_round(x32) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even).

    Returned as fp32 values that are exactly representable in bf16.  NaN is
    kept quiet; infinities pass through.
    """
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    u = x32.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) & 0xFFFF0000
    r = r.astype(np.uint32)
    nan = np.isnan(x32)
    r[nan] = 0x7FC00000
    return r.view(np.float32)


def bf16_bits(x32) -> np.ndarray:
    """bf16 bit patterns (uint16) of bf16_round(x32)."""
    return (bf16_round(x32).view(np.uint32) >> 16).astype(np.uint16)


def y_int8(acc, tscale, rscale) -> np.ndarray:
    """y[m,n] = bf16_rn(((float)acc[m,n] * tscale[m]) * rscale[n]).

    Every step is one fp32 operation (the int32 -> fp32 conversion rounds to
    nearest even), evaluated left to right.  Returns fp32 values on the bf16
    grid.
    """
    a = np.asarray(acc).astype(np.float32)
    t = np.asarray(tscale, dtype=np.float32)[:, None]
    r = np.asarray(rscale, dtype=np.float32)[None, :]
    y = ((a * t).astype(np.float32) * r).astype(np.float32)
    return bf16_round(y)


# --------------------------------------------------------------------------
# Whole layer, both references
# --------------------------------------------------------------------------

def linear_f64(x, codes, scales, sign=None) -> np.ndarray:
    """O1: y = (H_blk (sign*x)) W^T in fp64, W = code * s (the page's premises)."""
    return rotate_f64(x, sign) @ dequant_f64(codes, scales).T


def linear_int8(x, codes, scales, sign=None):
    """O2: the whole int8 prefill path of the page's section 4.

    Returns a dict with xr (fp32), xq, tscale, q, rscale, w (int16 holding the
    int8 weights), acc (int64) and y (fp32 on the bf16 grid).
    """
    xr = fwht_f32(np.asarray(x, dtype=np.float32), sign)
    xq, tscale = quant_tokens(xr)
    q, rscale, _ = decompose_scales(scales)
    w = w_int8(codes, q)
    acc = acc_int8(xq, w)
    y = y_int8(acc, tscale, rscale)
    return dict(xr=xr, xq=xq, tscale=tscale, q=q, rscale=rscale, w=w, acc=acc, y=y)


def rel_frobenius(y, yref) -> float:
    """||y - yref||_F / ||yref||_F in fp64 (0 when both are zero)."""
    y = np.asarray(y, dtype=np.float64)
    yref = np.asarray(yref, dtype=np.float64)
    den = np.linalg.norm(yref)
    num = np.linalg.norm(y - yref)
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return float(num / den)


# --------------------------------------------------------------------------
# 2-bit storage format (defined by this library; the pages leave it open)
# --------------------------------------------------------------------------
#
# A 2-bit field holds u = code + 1: -1 -> 0, 0 -> 1, +1 -> 2 (3 is never
# written).  Rows are padded with zero codes (u = 1) and zero scales to a
# multiple of 512.  The packed buffer is a sequence of 17408-byte units, unit
# rb * G + g for row block rb (512 rows) and group g (128 k), G = K / 128.
# In a unit:
#   bytes [0, 16384): 32 tiles of 16 rows, tile t at byte 512 t; slot L
#     (bytes 512 t + 16 L ..) holds four little-endian 32-bit words w_0..w_3;
#     with r = L // 4, c = L % 4, word p and field j (0..7):
#       bits 2j..2j+1 of w_p:     u(row, k)
#       bits 16+2j..17+2j of w_p: u(row, k + 1)
#     with row = 512 rb + 16 t + r + 8 (p % 2), k = 128 g + 16 j + 2 c + 8 (p // 2);
#   bytes [16384, 17408): fp16 scale pairs, tile t at 16384 + 32 t:
#     (s[512 rb + 16 t + r, g], s[512 rb + 16 t + r + 8, g]) for r = 0..7.
#
# Word p is register p of the A fragment of a 16 x 16 tensor-core tile for
# all 8 k16 steps j of the group: field j masked in place (j < 6), or field
# j of w_p >> 12 for j = 6, 7 (that is, field j - 6 of the shifted word),
# read as an fp16 pair, is u * 4^e(j) * 2^-24 with e(j) = j for j < 6 and
# j - 6 otherwise: a subnormal (e <= 4, the field inside the mantissa) or the
# two lowest exponent bits (e = 5: 0x0400 = 2^-14, 0x0800 = 2^-13).

UNIT_ROWS = 512
UNIT_BYTES = 17408


def step_exponent(j: int) -> int:
    """e(j): the power of four carried by the field of k16 step j."""
    return j if j < 6 else j - 6


def padded_rows(n: int) -> int:
    return (n + UNIT_ROWS - 1) // UNIT_ROWS * UNIT_ROWS


def pack_weights(codes, scales) -> np.ndarray:
    """Pack int8 codes [N,K] and fp16 scales [N,K/128] into the unit format."""
    codes = np.asarray(codes)
    n, k = codes.shape
    if k % GROUP:
        raise ValueError("K must be a multiple of 128")
    g_count = k // GROUP
    npad = padded_rows(n)
    full = np.zeros((npad, k), dtype=np.int64)
    full[:n] = codes
    sfull = np.zeros((npad, g_count), dtype=np.float16)
    sfull[:n] = np.asarray(scales, dtype=np.float16)
    rbs = npad // UNIT_ROWS
    # [rb, t, rh, r, g, j, kh, c, lohi]: row = 512 rb + 16 t + 8 rh + r,
    # k = 128 g + 16 j + 8 kh + 2 c + lohi
    u = (full + 1).astype(np.uint64).reshape(rbs, 32, 2, 8, g_count, 8, 2, 4, 2)
    words = np.zeros((rbs, g_count, 32, 8, 4, 4), dtype=np.uint64)     # rb, g, t, r, c, p
    for j in range(8):
        for kh in range(2):
            for rh in range(2):
                for lohi in range(2):
                    part = u[:, :, rh, :, :, j, kh, :, lohi]            # rb, t, r, g, c
                    words[..., 2 * kh + rh] |= part.transpose(0, 3, 1, 2, 4) << \
                        np.uint64(16 * lohi + 2 * j)
    code_bytes = words.astype("<u4").reshape(rbs, g_count, 4096).view(np.uint8)
    sc = sfull.reshape(rbs, 32, 2, 8, g_count).transpose(0, 4, 1, 3, 2)  # rb, g, t, r, rh
    scale_bytes = np.ascontiguousarray(sc).astype("<f2").view(np.uint8).reshape(rbs, g_count, 1024)
    out = np.concatenate([code_bytes, scale_bytes], axis=2)
    return out.reshape(-1).copy()


def unpack_weights(packed, n: int, k: int):
    """Inverse of pack_weights: returns (codes int8 [n,k], scales fp16 [n,k/128])."""
    g_count = k // GROUP
    npad = padded_rows(n)
    rbs = npad // UNIT_ROWS
    units = np.ascontiguousarray(packed, dtype=np.uint8).reshape(rbs, g_count, UNIT_BYTES)
    words = units[:, :, :16384].copy().view("<u4").reshape(rbs, g_count, 32, 8, 4, 4)
    words = words.astype(np.uint64)                                     # rb, g, t, r, c, p
    out = np.zeros((rbs, 32, 2, 8, g_count, 8, 2, 4, 2), dtype=np.int8)
    for j in range(8):
        for kh in range(2):
            for rh in range(2):
                for lohi in range(2):
                    fld = (words[..., 2 * kh + rh] >> np.uint64(16 * lohi + 2 * j)) & np.uint64(3)
                    out[:, :, rh, :, :, j, kh, :, lohi] = \
                        (fld.astype(np.int64) - 1).astype(np.int8).transpose(0, 2, 3, 1, 4)
    codes = out.reshape(npad, k)
    sc = units[:, :, 16384:].copy().view("<f2").reshape(rbs, g_count, 32, 8, 2)
    scales = sc.transpose(0, 2, 4, 3, 1).reshape(npad, g_count)
    return codes[:n], scales[:n].astype(np.float16)


# --------------------------------------------------------------------------
# Decode operand (the GEMV's activation format, defined in include/tern.h)
# --------------------------------------------------------------------------

def _block_shift(xr):
    """sh[m, b] = min(14 - E, 126), E = (biased exponent field of the fp32
    absmax of the block) - 127: 2^sh puts the block's largest magnitude in
    [2^14, 2^15)."""
    xr = np.asarray(xr, dtype=np.float32)
    m, k = xr.shape
    blocks = np.abs(xr).reshape(m, k // HBLOCK, HBLOCK).max(axis=2).astype(np.float32)
    e = ((blocks.view(np.uint32) >> 23) & 0xFF).astype(np.int64) - 127
    return np.minimum(14 - e, 126)


def f16_operand(xr):
    """fp16 copy of the rotated activations, one power-of-two factor per block
    (the fp16 prefill variant's operand).

    For token m and 1024-block b: F = 2^sh (_block_shift); values
    fp16_rn(xr * F) (the fp32 product is exact), natural [M, K] order.
    Returns (fp16 [M, K], inv [M, B] with inv = 1/F).
    """
    xr = np.asarray(xr, dtype=np.float32)
    m, k = xr.shape
    nb = k // HBLOCK
    sh = _block_shift(xr)
    f = np.ldexp(np.float32(1.0), sh).astype(np.float32)
    inv = np.ldexp(np.float32(1.0), -sh).astype(np.float32)
    scaled = (xr.reshape(m, nb, HBLOCK) * f[:, :, None]).astype(np.float32).reshape(m, k)
    return scaled.astype(np.float16), inv


def _k_exponents(k: int) -> np.ndarray:
    """e(j(k)) for every column k: the k16 step j = (k mod 128) // 16."""
    j = (np.arange(k) % GROUP) // 16
    return np.where(j < 6, j, j - 6)


def decode_operand(xr):
    """The decode GEMV's activation operand for M <= 16 tokens.

    For token m, 1024-block b (F = 2^sh, _block_shift) and column k of k16
    step j (e = e(j), see the packed format):
      xh[m, k] = fp16_rn(xr[m, k] * 2^(sh - 2e))      (the fp32 product is exact)
    and per 128-group g a 48-float record aux[g]:
      X[g, m] = the fp32 sum over k in g of xh[m, k] * 2^(2e - 24) (each term
                exact), added in this order: the eight consecutive columns
                8q .. 8q + 7 of the group left to right (q = 0..15), then the
                sixteen partial sums by a butterfly tree,
                p[q] <- p[q] + p[q ^ s] for s = 1, 2, 4, 8;
      aux[g][4 i .. 4 i + 3] = (-X[g, 2i], -X[g, 2i+1], -X[g, 2i], -X[g, 2i+1])
                for i = 0..7 (the tensor core's accumulator starts there),
                each computed as 0 - X in fp32 (+0 where X is 0);
      aux[g][32 + m] = 2^(12 - sh) of the block holding g;
      X and the fold factor are 0 for m >= M.
    A field read u * 4^e * 2^-24 times xh[m, k] is u * xh * 2^(2e - 24), so the
    tensor core's group sum minus X is sum_k code * xr * 2^(sh - 24) (up to
    rounding); times the block's 2^(12 - sh) that is 2^-12 sum_k code * xr.
    Returns (fp16 [M, K], float32 [G, 48]).
    """
    xr = np.asarray(xr, dtype=np.float32)
    m, k = xr.shape
    if m > 16:
        raise ValueError("the decode operand holds at most 16 tokens")
    g_count = k // GROUP
    sh = _block_shift(xr)                                             # [m, nb]
    e = _k_exponents(k)                                               # [k]
    shk = np.repeat(sh, HBLOCK, axis=1) - 2 * e[None, :]              # [m, k]
    xh = (xr * np.ldexp(np.float32(1.0), shk).astype(np.float32)).astype(np.float32)
    xh = xh.astype(np.float16)
    terms = (xh.astype(np.float32) * np.ldexp(np.float32(1.0), 2 * e - 24)
             .astype(np.float32)[None, :]).astype(np.float32)         # exact
    t = terms.reshape(m, g_count, 16, 8)
    p = t[..., 0].copy()
    for i in range(1, 8):
        p = (p + t[..., i]).astype(np.float32)
    idx = np.arange(16)
    for sft in (1, 2, 4, 8):
        p = (p + p[..., idx ^ sft]).astype(np.float32)
    x16 = np.zeros((g_count, 16), dtype=np.float32)
    x16[:, :m] = p[:, :, 0].T
    aux = np.zeros((g_count, 48), dtype=np.float32)
    pairs = x16.reshape(g_count, 8, 2)
    aux[:, :32] = -np.concatenate([pairs, pairs], axis=2).reshape(g_count, 32)
    aux[:, :32] += np.float32(0.0)                                    # 0 - X: -0 becomes +0
    fold = np.ldexp(np.float32(1.0), 12 - sh).astype(np.float32)      # [m, nb]
    aux[:, 32:32 + m] = np.repeat(fold, HBLOCK // GROUP, axis=1).T
    return xh, aux


def decode_offsets(aux):
    """The group offsets X[g, m] (16 tokens) of a decode operand record."""
    aux = np.asarray(aux, dtype=np.float32)
    return -aux[:, 0:32].reshape(-1, 8, 4)[:, :, :2].reshape(-1, 16)


def decode_folds(aux):
    """The fold factors [g, m] (16 tokens) of a decode operand record."""
    return np.asarray(aux, dtype=np.float32)[:, 32:48]
