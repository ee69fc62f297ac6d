"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties an oracle function to a fact fixed by the pages or by the
mathematics: textbook matrices, closed forms, invariants, hand-computed
worked examples (tests/golden/), brute force on tiny inputs, and library
routines where a special case reduces to one.  A planted-mistake test shows
that the pins catch plausible errors.
"""

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import tern_oracle as O
from ternary_weight_linear_block_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


def _walsh_popcount(n):
    """Closed form of natural-order Hadamard: H[i,j] = (-1)^popcount(i & j)."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    bits = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    return np.where(bits % 2 == 0, 1.0, -1.0)


# ---------------------------------------------------------------- Hadamard

def test_h8_matches_textbook_golden():
    h8 = np.array([[float(v) for v in r.split()] for r in _rows("hadamard8_natural.txt")])
    assert np.array_equal(O.hadamard_dense(8), h8)


@pytest.mark.parametrize("n", [1, 2, 4, 16, 64, 1024])
def test_hadamard_closed_form_and_orthogonality(n):
    h = O.hadamard_dense(n)
    assert np.array_equal(h, _walsh_popcount(n))
    assert np.array_equal(h, h.T)
    assert np.array_equal(h @ h.T, n * np.eye(n))


def test_normalised_rotation_is_an_involution_and_orthonormal():
    # (H/32)(H/32) = I exactly in fp64 (entries +-1/32, sums of 1024 terms).
    h = O.hadamard_dense(1024) / 32.0
    assert np.array_equal(h @ h, np.eye(1024))
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 2048))
    xr = O.rotate_f64(x)
    assert np.allclose(O.rotate_f64(xr), x, rtol=0, atol=1e-12)
    assert np.allclose(np.linalg.norm(xr, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_split_identity_of_the_page():
    # H1024 [a; b] = [H512 a + H512 b ; H512 a - H512 b]   (the page's section 1)
    rng = np.random.default_rng(2)
    a = rng.integers(-50, 50, 512).astype(np.float64)
    b = rng.integers(-50, 50, 512).astype(np.float64)
    h512 = _walsh_popcount(512)
    lhs = O.rotate_f64(np.concatenate([a, b])[None, :])[0] * 32.0
    rhs = np.concatenate([h512 @ a + h512 @ b, h512 @ a - h512 @ b])
    assert np.array_equal(lhs, rhs)
    # negative control: swapping the halves (the swapped-rank mistake the
    # page's CPU mock detects) must not satisfy the identity
    bad = np.concatenate([h512 @ a - h512 @ b, h512 @ a + h512 @ b])
    assert O.rel_frobenius(bad, lhs) > 0.5


def test_fwht_f32_exact_on_integers_and_matches_closed_form():
    rng = np.random.default_rng(3)
    x = rng.integers(-1000, 1000, (4, 3072)).astype(np.float32)
    got = O.fwht_f32(x)
    ref = np.concatenate([x[:, b * 1024:(b + 1) * 1024].astype(np.float64)
                          @ _walsh_popcount(1024).T / 32.0 for b in range(3)], axis=1)
    assert np.array_equal(got.astype(np.float64), ref)


def test_fwht_f32_special_cases():
    k = 2048
    x = np.zeros((3, k), np.float32)
    x[0, :1024] = 3.0                     # constant block -> 32c at index 0
    x[1, 1024 + 37] = 1.0                 # one-hot -> column of H / 32
    x[2, 5] = -2.0
    y = O.fwht_f32(x)
    e0 = np.zeros(1024, np.float32)
    e0[0] = 96.0
    assert np.array_equal(y[0, :1024], e0) and not y[0, 1024:].any()
    col = _walsh_popcount(1024)[:, 37] / 32.0
    assert np.array_equal(y[1, 1024:].astype(np.float64), col) and not y[1, :1024].any()
    assert np.array_equal(y[2, :1024].astype(np.float64), -2.0 * _walsh_popcount(1024)[:, 5] / 32.0)


def test_fwht_f32_close_to_exact_on_random_and_sign_vector():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, 2048)).astype(np.float32)
    sign = rng.choice([-1.0, 1.0], 2048)
    got = O.fwht_f32(x, sign).astype(np.float64)
    ref = _walsh_popcount(1024)
    exact = np.concatenate([(x[:, b * 1024:(b + 1) * 1024] * sign[b * 1024:(b + 1) * 1024])
                            .astype(np.float64) @ ref.T / 32.0 for b in range(2)], axis=1)
    assert O.rel_frobenius(got, exact) < 1e-6
    assert O.rel_frobenius(O.rotate_f64(x, sign), exact) < 1e-14


def test_planted_mistakes_are_caught():
    """Mutants of the butterfly (sign swap, wrong stage set) fail the pins."""
    def fwht_mutant(x, swap_sign=False, skip_last=False):
        v = np.asarray(x, np.float32).reshape(x.shape[0], -1, 1024).copy()
        h = 1
        while h < 1024:
            if skip_last and h == 512:
                break
            w = v.reshape(v.shape[0], v.shape[1], 1024 // (2 * h), 2, h)
            lo, hi = w[:, :, :, 0, :], w[:, :, :, 1, :]
            d = (hi - lo) if swap_sign else (lo - hi)
            v = np.stack([lo + hi, d], axis=3).reshape(v.shape)
            h *= 2
        return (v * np.float32(1 / 32)).reshape(x.shape)

    rng = np.random.default_rng(5)
    x = rng.integers(-9, 9, (2, 1024)).astype(np.float32)
    exact = x.astype(np.float64) @ _walsh_popcount(1024).T / 32.0
    assert np.array_equal(O.fwht_f32(x).astype(np.float64), exact)
    for kw in ({"swap_sign": True}, {"skip_last": True}):
        assert not np.array_equal(fwht_mutant(x, **kw).astype(np.float64), exact)


# ---------------------------------------------------------------- scales

def test_scale_decomposition_golden():
    for r in _rows("scale_decomposition.txt"):
        s_txt, q_txt, smax_txt = [p.strip() for p in r.split("|")]
        s = np.array([[float(v) for v in s_txt.split()]], dtype=np.float16)
        q, rscale, smax = O.decompose_scales(s)
        assert q[0].tolist() == [int(v) for v in q_txt.split()]
        assert smax[0] == np.float32(np.float16(float(smax_txt)))
        assert rscale[0] == np.float32(smax[0] / np.float32(127.0))


def test_scale_decomposition_exact_rational_and_invariants():
    rng = np.random.default_rng(6)
    s = (0.02 * np.abs(rng.standard_normal((64, 40))) + 1e-3).astype(np.float16)
    s[3] = 0
    s[5, ::3] *= -1
    q, rscale, smax = O.decompose_scales(s)
    for n in range(s.shape[0]):
        sm = max(abs(Fraction(float(v))) for v in s[n])
        for g in range(s.shape[1]):
            if sm == 0:
                want = 0
            else:
                want = round(127 * Fraction(float(s[n, g])) / sm)   # exact, half to even
            assert q[n, g] == want
    assert np.all(np.abs(q.astype(int)) <= 127)
    nz = smax > 0
    am = np.argmax(np.abs(s.astype(np.float32)), axis=1)
    assert np.all(np.abs(q[np.arange(64), am][nz]) == 127)
    assert q[3].max() == 0 and rscale[3] == 0


def test_int8_weight_fits_and_approximates_dequant():
    d = I.make_layer(I.TINY, m=1, seed=0, n=64)
    q, rscale, _ = O.decompose_scales(d.scales)
    w = O.w_int8(d.codes, q)
    assert np.abs(w).max() <= 127                     # "fits int8 exactly"
    wd = O.dequant_f64(d.codes, d.scales)
    err = np.abs(w * rscale[:, None].astype(np.float64) - wd)
    assert np.all(err <= 0.5 * rscale[:, None] * (1 + 1e-6) + 1e-12)


# ---------------------------------------------------------------- activations

def test_token_quant_golden():
    for r in _rows("token_quant.txt"):
        x_txt, q_txt, t_txt = [p.strip() for p in r.split("|")]
        xr = np.array([[float(v) for v in x_txt.split()]], np.float32)
        xq, t = O.quant_tokens(xr)
        assert xq[0].tolist() == [int(v) for v in q_txt.split()]
        assert t[0] == np.float32(float(t_txt))


def test_token_quant_rational_and_invariants():
    rng = np.random.default_rng(7)
    xr = rng.standard_normal((16, 1024)).astype(np.float32)
    xr[4] = 0
    xq, t = O.quant_tokens(xr)
    assert np.all(np.abs(xq.astype(int)) <= 127)
    am = np.argmax(np.abs(xr), axis=1)
    for m in range(16):
        if m == 4:
            assert t[m] == 0 and not xq[m].any()
            continue
        assert abs(int(xq[m, am[m]])) == 127
        tm = Fraction(float(t[m]))
        for k in range(0, 1024, 7):
            exact = Fraction(float(xr[m, k])) / tm
            want = max(-127, min(127, round(exact)))
            if xq[m, k] != want:     # only a quotient rounded onto a tie may differ
                assert abs(abs(exact - int(exact)) - Fraction(1, 2)) < Fraction(1, 1 << 19)
    err = np.abs(xq.astype(np.float64) * t[:, None] - xr)
    assert np.all(err <= 0.5 * t[:, None] * (1 + 1e-5) + 1e-30)


# ---------------------------------------------------------------- int8 GEMM

def test_acc_int8_brute_force_tiny():
    rng = np.random.default_rng(8)
    xq = rng.integers(-127, 128, (3, 256)).astype(np.int8)
    w = rng.integers(-127, 128, (5, 256)).astype(np.int16)
    acc = O.acc_int8(xq, w)
    for m in range(3):
        for n in range(5):
            assert acc[m, n] == sum(int(a) * int(b) for a, b in zip(xq[m], w[n]))


def test_acc_int8_extreme_magnitude_exact():
    k = 17408
    xq = np.full((2, k), 127, np.int8)
    xq[1] = -127
    w = np.full((2, k), 127, np.int16)
    acc = O.acc_int8(xq, w)
    assert acc[0, 0] == 127 * 127 * k and acc[1, 1] == -127 * 127 * k
    assert 127 * 127 * k < 2 ** 31


def test_equal_scales_reduce_to_plain_integer_gemm():
    # all s equal -> q = 127 everywhere -> W_int8 = 127 * code: a textbook
    # integer matrix product, checked with pure Python loops
    rng = np.random.default_rng(9)
    codes = rng.integers(-1, 2, (4, 1024)).astype(np.int8)
    s = np.full((4, 8), 0.0137, np.float16)
    q, rscale, _ = O.decompose_scales(s)
    assert np.all(q == 127)
    xq = rng.integers(-127, 128, (2, 1024)).astype(np.int8)
    acc = O.acc_int8(xq, O.w_int8(codes, q))
    for m in range(2):
        for n in range(4):
            assert acc[m, n] == 127 * sum(int(a) * int(c) for a, c in zip(xq[m], codes[n]))


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(10)
    v = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 1e3,
                        np.array([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1e-40,
                                  3.0e38, -1.5, np.inf, -np.inf], np.float32)])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(O.bf16_round(v).view(np.uint32), ref.view(np.uint32))


def test_y_rescale_order_and_rounding():
    acc = np.array([[16777217, -3, 0]], np.int64)     # 2^24+1 rounds in the cast
    t = np.array([0.5], np.float32)
    r = np.array([2.0, 0.1, 7.0], np.float32)
    y = O.y_int8(acc, t, r)
    assert y[0, 0] == np.float32(16777216.0)
    assert y[0, 1] == O.bf16_round(np.array([np.float32(-1.5) * np.float32(0.1)]))[0]
    assert y[0, 2] == 0.0


# ---------------------------------------------------------------- whole layer

def test_linear_f64_two_formulations_agree():
    d = I.make_layer(I.TINY, m=8, seed=0)
    y1 = O.linear_f64(d.x, d.codes, d.scales)
    wh = O.dequant_f64(d.codes, d.scales) @ (O.hadamard_dense(1024) / 32.0)   # (W H) x
    y2 = d.x.astype(np.float64) @ wh.T
    assert O.rel_frobenius(y1, y2) < 1e-12


def test_linear_f64_special_cases():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((2, 2048))
    codes = np.zeros((6, 2048), np.int8)
    s = (np.abs(rng.standard_normal((6, 16))) * 0.02 + 1e-3).astype(np.float16)
    assert not O.linear_f64(x, codes, s).any()
    codes[1, 1500] = -1
    y = O.linear_f64(x, codes, s)
    xr = O.rotate_f64(x)
    assert np.allclose(y[:, 1], -float(s[1, 1500 // 128]) * xr[:, 1500], rtol=1e-15, atol=0)
    codes = rng.integers(-1, 2, (6, 2048)).astype(np.int8)
    s_eq = np.full((6, 16), 0.25, np.float16)
    y = O.linear_f64(x, codes, s_eq)
    assert np.allclose(y, 0.25 * (xr @ codes.T.astype(np.float64)), rtol=1e-13, atol=1e-13)


def test_int8_path_error_against_exact_tiny_config():
    # expected: activation quant + scale quant give about 1e-2 relative
    # error; the page reports 9.5e-3 per layer on real weights
    d = I.make_layer(I.TINY, m=8, seed=0)
    r = O.linear_int8(d.x, d.codes, d.scales)
    exact = O.linear_f64(d.x, d.codes, d.scales)
    e = O.rel_frobenius(r["y"], exact)
    assert 1e-3 < e < 2e-2


# ---------------------------------------------------------------- 2-bit format

def test_pack_format_golden():
    codes = np.zeros((512, 256), np.int8)
    expect = {}
    for r in _rows("packed_format.txt"):
        left, off, word = [p.strip() for p in r.split("|")]
        row, k, c = [int(v) for v in left.split()]
        codes[row, k] = c
        expect[int(off)] = int(word, 16)
    scales = np.zeros((512, 2), np.float16)
    scales[3, 1] = 0.5      # unit 1, tile 0, pair r = 3, low half
    scales[20, 0] = 0.25    # unit 0, tile 1, pair r = 4, low half
    p = O.pack_weights(codes, scales)
    assert p.size == 2 * 17408
    code_words = {}
    for unit in range(2):
        w = p[unit * 17408:unit * 17408 + 16384].view("<u4")
        code_words.update({unit * 17408 + 4 * i: int(v) for i, v in enumerate(w)
                           if v != 0x55555555})
    assert code_words == expect
    # scale pairs: s[3, 1] -> unit 1, tile 0, pair 3, low half; s[20, 0] -> tile 1, pair 4
    assert p[17408 + 16384 + 12:17408 + 16384 + 14].view("<f2")[0] == np.float16(0.5)
    assert p[16384 + 32 + 16:16384 + 32 + 18].view("<f2")[0] == np.float16(0.25)
    assert np.count_nonzero(p[16384:17408]) == 1 and np.count_nonzero(p[17408 + 16384:]) == 1


@pytest.mark.parametrize("n,k", [(512, 128), (40, 1024), (7, 256), (700, 2048)])
def test_pack_roundtrip(n, k):
    rng = np.random.default_rng(n * 7 + k)
    codes = rng.integers(-1, 2, (n, k)).astype(np.int8)
    s = rng.standard_normal((n, k // 128)).astype(np.float16)
    p = O.pack_weights(codes, s)
    assert p.size == O.padded_rows(n) // 512 * (k // 128) * 17408
    c2, s2 = O.unpack_weights(p, n, k)
    assert np.array_equal(c2, codes) and np.array_equal(s2, s)


def _f16(bits):
    return float(np.array([bits], np.uint16).view(np.float16)[0])


def test_pack_field_reading_is_the_a_fragment():
    """Field j of word p, masked in place (j < 6) or from the word shifted
    right by 12 (j = 6, 7), read as an fp16 pair, is (u(row, k), u(row, k+1))
    * 4^e(j) * 2^-24 with u = code + 1, row = 16 t + r + 8 (p % 2),
    k = 16 j + 2 c + 8 (p // 2): register p of the A fragment of a 16 x 16
    tensor-core tile for k16 step j.  The fp16 values are computed here from
    the IEEE encoding (subnormal: m * 2^-24; exponent field 1 or 2 with a zero
    mantissa: 2^-14, 2^-13), not from the oracle."""
    rng = np.random.default_rng(12)
    codes = rng.integers(-1, 2, (512, 128)).astype(np.int8)
    words = O.pack_weights(codes, np.zeros((512, 1), np.float16))[:16384].view("<u4")
    words = words.reshape(32, 32, 4)                 # tile, slot, word
    for t in range(0, 32, 7):
        for lane in range(32):
            r, c = lane // 4, lane % 4
            for p in range(4):
                w = int(words[t, lane, p])
                for j in range(8):
                    v = (w if j < 6 else w >> 12) & (0x00030003 << (2 * (j % 6)))
                    e = j if j < 6 else j - 6
                    row = 16 * t + r + 8 * (p % 2)
                    k = 16 * j + 2 * c + 8 * (p // 2)
                    for half, kk in ((v & 0xFFFF, k), (v >> 16, k + 1)):
                        u = codes[row, kk] + 1
                        assert _f16(half) == u * 4.0 ** e * 2.0 ** -24, (t, lane, p, j)
    # the two readings of field 5 use the exponent: 0x0400 = 2^-14, 0x0800 = 2^-13
    assert _f16(0x0400) == 2.0 ** -14 and _f16(0x0800) == 2.0 ** -13


# ---------------------------------------------------------------- decode operand

def _operand_case():
    rng = np.random.default_rng(13)
    xr = (rng.standard_normal((4, 2048)) * np.array([[1e-3], [1.0], [3e4], [2.0]])
          ).astype(np.float32)
    xr[1, 1024:] = 0.0                                  # an all-zero block
    xr[3, 5] = 900.0                                    # one large value
    return xr


def test_decode_operand_scaling_and_precision():
    xr = _operand_case()
    xh, aux = O.decode_operand(xr)
    k = xr.shape[1]
    j = (np.arange(k) % 128) // 16
    e = np.where(j < 6, j, j - 6)
    fold = O.decode_folds(aux)[::8, :4].T                # [m, block]: 2^(12 - sh)
    sh = 12 - np.log2(fold.astype(np.float64))
    assert np.all(sh == np.round(sh))
    shk = np.repeat(sh, 1024, axis=1) - 2 * e[None, :]
    # fp16 cast matches torch's (library) round-to-nearest-even cast of the exact product
    scaled = (xr.astype(np.float64) * 2.0 ** shk).astype(np.float32)
    ref = torch.from_numpy(scaled).to(torch.float16).numpy()
    assert np.array_equal(xh.view(np.uint16), ref.view(np.uint16))
    # undoing the per-step power of four, each nonzero block's largest magnitude
    # lands in [2^14, 2^15)
    xs = xh.astype(np.float64) * 4.0 ** e[None, :]
    bm = np.abs(xs).reshape(4, 2, 1024).max(axis=2)
    for m in range(4):
        for b in range(2):
            if np.abs(xr[m, b * 1024:(b + 1) * 1024]).max() > 0:
                assert 2 ** 14 <= bm[m, b] < 2 ** 15
    back = xh.astype(np.float64) * 2.0 ** (-shk)
    # fp16 relative rounding, plus half the subnormal spacing where xh is subnormal
    assert np.all(np.abs(back - xr) <= np.abs(xr) * 2.0 ** -11 + 2.0 ** (-25 - shk))


def test_decode_operand_group_offsets_exact_sum_and_padding():
    xr = _operand_case()
    xh, aux = O.decode_operand(xr)
    m, k = xr.shape
    assert aux.shape == (k // 128, 48) and aux.dtype == np.float32
    off, fold = O.decode_offsets(aux), O.decode_folds(aux)
    assert not off[:, m:].any() and not fold[:, m:].any()
    # the accumulator quads: (-X[2i], -X[2i+1], -X[2i], -X[2i+1]), +0 for a zero offset
    q = aux[:, :32].reshape(-1, 8, 4)
    assert np.array_equal(q[:, :, :2].view(np.uint32), q[:, :, 2:].view(np.uint32))
    assert not np.signbit(aux[:, :32][aux[:, :32] == 0]).any()
    j = (np.arange(k) % 128) // 16
    e = np.where(j < 6, j, j - 6)
    for mm in range(m):
        for g in range(k // 128):
            terms = [Fraction(float(xh[mm, kk])) * Fraction(2) ** int(2 * e[kk] - 24)
                     for kk in range(128 * g, 128 * g + 128)]
            exact = sum(terms)
            bound = sum(abs(t) for t in terms) * Fraction(8, 2 ** 24)
            assert abs(Fraction(float(off[g, mm])) - exact) <= bound, (mm, g)


def _emulated_gemv(packed, n, k, xh, aux, m):
    """The decode arithmetic read straight from the packed bytes and the
    operand, in fp64: y = 2^12 sum_b fold[b] sum_{g in b} s (sum_k A B - X)."""
    codes, scales = O.unpack_weights(packed, n, k)
    g_count = k // 128
    j = (np.arange(k) % 128) // 16
    e = np.where(j < 6, j, j - 6)
    a = (codes.astype(np.float64) + 1.0) * 4.0 ** e[None, :] * 2.0 ** -24     # A fragment values
    y = np.zeros((m, n))
    for g in range(g_count):
        cols = slice(128 * g, 128 * g + 128)
        d = xh[:, cols].astype(np.float64) @ a[:, cols].T - \
            O.decode_offsets(aux)[g, :m][:, None].astype(np.float64)
        y += (d * scales[:, g].astype(np.float64)[None, :]) * O.decode_folds(aux)[g, :m][:, None]
    return y * 2.0 ** 12


def test_decode_arithmetic_reproduces_the_layer():
    """The fields as A fragments, the operand as B, the group offsets and the
    fold factors together give the exact layer (fp64 emulation of the GEMV's
    arithmetic, no fp32 rounding) within the fp16 rounding of the operand; a
    wrong power of four for steps 6 and 7, or a missing offset, does not."""
    rng = np.random.default_rng(14)
    n, k, m = 64, 2048, 3
    codes = rng.integers(-1, 2, (n, k)).astype(np.int8)
    scales = (0.02 * np.abs(rng.standard_normal((n, k // 128))) + 1e-3).astype(np.float16)
    x = rng.standard_normal((m, k)).astype(np.float32)
    exact = O.linear_f64(x, codes, scales)
    packed = O.pack_weights(codes, scales)
    xh, aux = O.decode_operand(O.fwht_f32(x))
    y = _emulated_gemv(packed, n, k, xh, aux, m)
    assert O.rel_frobenius(y, exact) < 6e-4           # fp16 rounding of the operand: ~2.5e-4
    bad = aux.copy()
    bad[:, :32] = 0.0                                # offsets dropped
    assert O.rel_frobenius(_emulated_gemv(packed, n, k, xh, bad, m), exact) > 0.5
    wrong = xh.copy()                                # steps 6, 7 read with 4^6, 4^7
    cols = ((np.arange(k) % 128) // 16) >= 6
    wrong[:, cols] = (wrong[:, cols].astype(np.float32) / np.float32(4096)).astype(np.float16)
    assert O.rel_frobenius(_emulated_gemv(packed, n, k, wrong, aux, m), exact) > 0.1


def test_f16_operand_range_and_precision():
    xr = _operand_case()
    vals, inv = O.f16_operand(xr)
    # fp16 cast matches torch's (library) round-to-nearest-even cast
    f = (1.0 / inv).astype(np.float32)
    scaled = (xr.reshape(4, 2, 1024) * f[:, :, None]).reshape(4, 2048).astype(np.float32)
    ref = torch.from_numpy(scaled).to(torch.float16).numpy()
    assert np.array_equal(vals.view(np.uint16), ref.view(np.uint16))
    bm = np.abs(vals.astype(np.float32)).reshape(4, 2, 1024).max(axis=2)
    for m in range(4):
        for b in range(2):
            if np.abs(xr[m, b * 1024:(b + 1) * 1024]).max() > 0:
                assert 2 ** 14 <= bm[m, b] < 2 ** 15
    back = vals.astype(np.float64) * np.repeat(inv, 1024, axis=1)
    assert np.all(np.abs(back - xr) <= np.abs(xr) * 2.0 ** -11 + 1e-30)


# ---------------------------------------------------------------- K split (section 1)

def test_half_transform_is_dense_h512():
    """fwht_half_f32 is the unnormalised H512 (closed form, exact on integers)."""
    rng = np.random.default_rng(40)
    x = rng.integers(-50, 51, (3, 512)).astype(np.float32)
    ref = x.astype(np.float64) @ _walsh_popcount(512).T
    assert np.array_equal(O.fwht_half_f32(x).astype(np.float64), ref)


@pytest.mark.parametrize("k,world", [(17408, 2), (3072, 2), (4096, 4), (2048, 4), (5120, 2)])
def test_ksplit_rotation_equals_whole_width_rotation(k, world):
    """The half-block exchange reproduces the canonical whole-width rotation
    bit for bit (the stride-512 stage is the last one), with or without a
    sign vector, whether the shard boundaries cut blocks or not."""
    rng = np.random.default_rng(k + world)
    x = O.bf16_round(rng.standard_normal((3, k)).astype(np.float32))
    sign = np.where(rng.random(k) < 0.5, -1, 1).astype(np.int8)
    for sg in (None, sign):
        got = np.concatenate(O.ksplit_rotate_f32(x, world, sg), axis=1)
        ref = O.fwht_f32(x, sg)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    # and it matches the exact fp64 rotation to fp32 accuracy
    assert O.rel_frobenius(got, O.rotate_f64(x, sign)) < 1e-6


def test_ksplit_swapped_parts_is_caught():
    """Negative control (the page's section 1 checks that swapping the ranks'
    roles is detected): if the first-half rank takes the difference and the
    second-half rank the sum, the result is far from the rotation."""
    rng = np.random.default_rng(41)
    k = 17408
    x = rng.standard_normal((2, k)).astype(np.float32)
    half = k // 2
    a = O.fwht_half_f32(x[:, half - 512:half])
    b = O.fwht_half_f32(x[:, half:half + 512])
    ref = O.fwht_f32(x)[:, half - 512:half + 512]   # the split block, columns 8192 .. 9215
    good = np.concatenate([O.ksplit_combine(a, b, 0), O.ksplit_combine(a, b, 1)], axis=1)
    bad = np.concatenate([O.ksplit_combine(a, b, 1), O.ksplit_combine(a, b, 0)], axis=1)
    assert np.array_equal(good, ref)
    assert O.rel_frobenius(bad, ref) > 1.0


# ---------------------------------------------------------------- error metric

def _matrix(txt):
    return np.array([[float(v) for v in row.split()] for row in txt.split(";")])


def _rel_frobenius_golden():
    out = []
    for r in _rows("rel_frobenius.txt"):
        y_txt, ref_txt, sq_txt = [p.strip() for p in r.split("|")]
        out.append((_matrix(y_txt), _matrix(ref_txt), Fraction(sq_txt)))
    return out


def test_rel_frobenius_hand_computed_golden():
    """The metric every tolerance is stated in (relative Frobenius error over
    the whole output), against hand-computed rationals: the square of the
    returned value equals num^2 / den^2 to the last bits of fp64."""
    cases = _rel_frobenius_golden()
    assert len(cases) == 5
    for y, ref, sq in cases:
        got = O.rel_frobenius(y, ref)
        assert abs(Fraction(got) ** 2 - sq) <= Fraction(1, 2 ** 48) * max(sq, 1), (y, ref, got)
    # the first worked example: sqrt(10) / 5
    assert O.rel_frobenius([[3.0, 4.0]], [[0.0, 5.0]]) == pytest.approx(np.sqrt(10) / 5, rel=1e-15)


def test_rel_frobenius_invariants():
    rng = np.random.default_rng(11)
    ref = rng.standard_normal((4, 37))
    y = ref + 1e-3 * rng.standard_normal((4, 37))
    e = O.rel_frobenius(y, ref)
    # scale invariance, exact for powers of two
    assert O.rel_frobenius(8.0 * y, 8.0 * ref) == e
    # invariant under any permutation of the entries applied to both
    p = rng.permutation(y.size)
    assert O.rel_frobenius(y.ravel()[p], ref.ravel()[p]) == pytest.approx(e, rel=1e-14)
    # a whole-output metric: equals the root of the summed squared row errors
    num = sum(float(np.sum((y[i] - ref[i]) ** 2)) for i in range(4))
    den = sum(float(np.sum(ref[i] ** 2)) for i in range(4))
    assert e == pytest.approx(np.sqrt(num / den), rel=1e-14)
    # degenerate cases
    assert O.rel_frobenius(ref, ref) == 0.0
    assert O.rel_frobenius(np.zeros(3), np.zeros(3)) == 0.0
    assert O.rel_frobenius(np.ones(3), np.zeros(3)) == float("inf")
    assert O.rel_frobenius(np.zeros((2, 3)), ref[:2, :3]) == pytest.approx(1.0, rel=1e-15)


def test_rel_frobenius_planted_mistakes_are_caught():
    """Plausible slips in the metric (arguments swapped, the square root
    dropped, a max norm or a per-row mean in place of the whole-output norm,
    the denominator taken from the difference) each fail the golden."""
    def swapped(y, ref):
        y, ref = np.asarray(y, np.float64), np.asarray(ref, np.float64)
        return float(np.linalg.norm(y - ref) / np.linalg.norm(y))

    def no_sqrt(y, ref):
        y, ref = np.asarray(y, np.float64), np.asarray(ref, np.float64)
        return float(np.sum((y - ref) ** 2) / np.sum(ref ** 2))

    def max_norm(y, ref):
        y, ref = np.asarray(y, np.float64), np.asarray(ref, np.float64)
        return float(np.max(np.abs(y - ref)) / np.max(np.abs(ref)))

    def row_mean(y, ref):
        y, ref = np.atleast_2d(np.asarray(y, np.float64)), np.atleast_2d(np.asarray(ref, np.float64))
        return float(np.mean([np.linalg.norm(a - b) / np.linalg.norm(b) for a, b in zip(y, ref)]))

    def diff_denominator(y, ref):
        y, ref = np.asarray(y, np.float64), np.asarray(ref, np.float64)
        return float(np.linalg.norm(y - ref) / np.linalg.norm(y - ref + ref))

    cases = _rel_frobenius_golden()

    def passes(fn):
        return all(abs(Fraction(fn(y, ref)) ** 2 - sq) <= Fraction(1, 2 ** 40) * max(sq, 1)
                   for y, ref, sq in cases)

    assert passes(O.rel_frobenius)
    for mutant in (swapped, no_sqrt, max_norm, row_mean, diff_denominator):
        assert not passes(mutant), mutant.__name__
