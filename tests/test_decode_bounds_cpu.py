"""The element-wise decode bound (tests/decode_bounds.py) on the CPU.

An emulation of the decode arithmetic from the oracle's pieces (the packed
fields as tensor-core fragments, the decode operand with its group offsets
and fold factors, fp64 accumulation, bf16 output rounding) must pass the
bound on every element; the same emulation with a
planted localised mistake (one 128-group of one row dropped, one group's
scale doubled, one row block's output left at zero) must fail it, although
the first two stay far inside the whole-output 4e-3 Frobenius bar.
"""

import numpy as np
import pytest

from oracle import tern_oracle as O
from ternary_weight_linear_block_gb300 import inputs as I
from tests.decode_bounds import block_sample_rows, check_elementwise, emulate_decode


def _emulated_decode(x, codes, scales):
    return emulate_decode(codes, scales, x)


@pytest.mark.parametrize("k,n,m", [(5120, 256, 4), (17408, 128, 2)])
def test_bound_accepts_the_decode_arithmetic(k, n, m):
    codes = I.make_codes(3, n, k)
    scales = I.make_scales(3, n, k)
    _, x = I.make_activations(3, m, k, 0.001, 50.0)
    y = _emulated_decode(x, codes, scales)
    ref = O.linear_f64(x, codes, scales)
    ratio = check_elementwise(y, ref, codes, scales, x, what="emulated decode")
    assert ratio < 0.5
    assert O.rel_frobenius(y, ref) < 4e-3


def test_bound_rejects_localised_mistakes():
    k, n, m = 2048, 16384, 2          # enough rows that one group is lost in the norm
    codes = I.make_codes(4, n, k)
    scales = I.make_scales(4, n, k)
    _, x = I.make_activations(4, m, k, 0.001, 50.0)
    ref = O.linear_f64(x, codes, scales)
    xr = O.rotate_f64(x)
    w = O.dequant_f64(codes, scales)
    good = _emulated_decode(x, codes, scales)

    dropped = good.copy()              # row 77 loses group 13
    g = slice(13 * 128, 14 * 128)
    dropped[:, 77] -= xr[:, g] @ w[77, g]
    doubled = good.copy()              # row 200's group 11 counted with twice its scale
    g = slice(11 * 128, 12 * 128)
    doubled[:, 200] += xr[:, g] @ w[200, g]
    for bad in (dropped, doubled):
        assert O.rel_frobenius(bad, ref) < 4e-3        # invisible to the whole-output norm
        with pytest.raises(AssertionError, match="element-wise bound"):
            check_elementwise(bad, ref, codes, scales, x)
    zero_block = good.copy()
    zero_block[:, 0:16] = 0.0
    with pytest.raises(AssertionError, match="element-wise bound"):
        check_elementwise(zero_block, ref, codes, scales, x)


def test_block_sample_rows_touches_every_block_twice():
    for n in (34816, 5120, 10240, 1000):
        rows = block_sample_rows(n, seed=1)
        assert np.all(np.diff(rows) > 0) and rows[0] >= 0 and rows[-1] < n
        counts = np.bincount(rows // 512, minlength=(n + 511) // 512)
        assert counts.min() >= 2
