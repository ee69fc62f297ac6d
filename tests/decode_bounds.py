"""Element-wise error bound of the decode path (test infrastructure).

The decode GEMV's accuracy bar is a relative Frobenius error over the whole
output.  A norm over thousands of outputs can hide a localised mistake (one
wrong 512-row block, a mis-scaled group, a lost partial sum), so the decode
tests also bound every compared element on its own:

    |y[m,n] - yref[m,n]| <= 2^-7 |yref[m,n]| + 2^-7 ||W[n,:] * xr[m,:]||_2
                            + 2^-18 sum_k |s[n,k/128] xr[m,k]|

with W[n,k] = code[n,k] s[n,k/128], xr the exact rotated activation and
W[n,:] * xr[m,:] the element-wise product.

Derivation.  The bf16 output rounding is at most half an ulp, 2^-8 relative
(the first term keeps a factor of two for the distance between |y| and
|yref|).  The decode operand rounds each rotated value to fp16 after an exact
power-of-two scaling: an error of at most 2^-11 |xr[m,k]| per element, zero
mean and independent across k, so their weighted sum has a standard deviation
of at most 2^-11 / sqrt(3) ||W[n] * xr[m]||; the second term is 27 of those
standard deviations (the worst case, all errors aligned, is the
Cauchy-Schwarz 2^-11 ||W[n]|| ||xr[m]||, far looser).  The packed fields hold
code + 1, so each group's tensor-core sum carries the sum of the activations
it multiplies, which the group offset (summed in fp32 by the rotation)
removes; the two sums round differently, by at most a few dozen fp32 ulps of
sum_{k in g} |xr[m,k]| per group, scaled by s[n,g]: the third term (64 ulps of
2^-24).  It is what remains for a row of zero codes, and for random weights it
is a few percent of the second term.  fp32 accumulation adds less.  A dropped, doubled or mis-scaled 128-group of a
row moves y[m,n] by about ||W[n,g] * xr[m,g]||, which for the workload widths
(K <= 17408, 40 to 136 groups) is 10 to 25 times the second term, so such a
slip fails the bound wherever it lands.
"""

from __future__ import annotations

import numpy as np

from oracle import tern_oracle as O


def check_elementwise(y, yref, codes, scales, x, sign=None, what=""):
    """Assert the element-wise bound on every element of y [M][R] against
    yref [M][R], where codes / scales hold the R compared rows and x is the
    bf16 activation as fp64 [M][K].  Returns the largest error / bound."""
    y = np.asarray(y, np.float64)
    yref = np.asarray(yref, np.float64)
    assert y.shape == yref.shape, (y.shape, yref.shape)
    xr = O.rotate_f64(x, sign)
    w = O.dequant_f64(codes, scales)
    prod_norm = np.sqrt((xr * xr) @ (w * w).T)                 # [M][R]
    s_abs = np.repeat(np.abs(np.asarray(scales, np.float64)), 128, axis=1)   # [R][K]
    offset_term = np.abs(xr) @ s_abs.T                           # [M][R]
    bound = 2.0 ** -7 * np.abs(yref) + 2.0 ** -7 * prod_norm + 2.0 ** -18 * offset_term
    err = np.abs(y - yref)
    bad = ~(err <= bound)
    if bad.any():
        m, r = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside the element-wise bound; "
            f"first at token {m}, compared row {r}: y={y[m, r]!r} yref={yref[m, r]!r} "
            f"err={err[m, r]:.3e} bound={bound[m, r]:.3e}")
    return float(np.max(err / np.maximum(bound, 1e-300)))


def block_sample_rows(n: int, seed: int, extra: int = 512, per_block: int = 2) -> np.ndarray:
    """A seeded sample of output rows: `extra` rows at random plus `per_block`
    rows of every 512-row block (the GEMV's unit of rows), sorted, unique."""
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(n, min(extra, n), replace=False).tolist())
    for b0 in range(0, n, 512):
        b1 = min(n, b0 + 512)
        rows.update(rng.choice(np.arange(b0, b1), min(per_block, b1 - b0),
                               replace=False).tolist())
    return np.array(sorted(rows))


def emulate_decode(codes, scales, x, sign=None):
    """The decode GEMV's arithmetic in fp64 from the oracle's pieces: the
    packed fields read as A fragments (u * 4^e * 2^-24), the decode operand as
    B, each group's sum minus its offset times the group scale, each block's
    sum times its fold factor, times 2^12, then the bf16 output rounding."""
    n, k = codes.shape
    packed = O.pack_weights(codes, scales)
    c2, s2 = O.unpack_weights(packed, n, k)
    xh, aux = O.decode_operand(O.fwht_f32(np.asarray(x, np.float32), sign))
    off, fold = O.decode_offsets(aux), O.decode_folds(aux)
    m = xh.shape[0]
    j = (np.arange(k) % 128) // 16
    e = np.where(j < 6, j, j - 6)
    a = (c2.astype(np.float64) + 1.0) * 4.0 ** e[None, :] * 2.0 ** -24
    y = np.zeros((m, n))
    for g in range(k // 128):
        cols = slice(128 * g, 128 * g + 128)
        d = xh[:, cols].astype(np.float64) @ a[:, cols].T - off[g, :m][:, None].astype(np.float64)
        y += (d * s2[:, g].astype(np.float64)[None, :]) * fold[g, :m][:, None]
    return O.bf16_round((y * 2.0 ** 12).astype(np.float32)).astype(np.float64)
