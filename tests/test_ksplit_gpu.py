"""K-split tensor parallelism (the page's section 1) through the library's
kernels, the ranks emulated in turn on one GPU (no rank waits on another:
each phase runs to completion before the next starts, and the exchange is a
list of the ranks' tensors).

Checks against the oracle: every rank's rotated columns (tern_fwht_shard +
tern_fwht_combine) equal the whole-width canonical rotation bit for bit; the
sum of the ranks' partial outputs matches the whole-width layer within the
decode (4e-3) and int8 (2e-2) tolerances; the rotation kernels agree with
the oracle's half-block steps.
"""

import numpy as np
import pytest
import torch

from oracle import tern_oracle as O
from ternary_weight_linear_block_gb300 import binding as B
from ternary_weight_linear_block_gb300 import inputs as I
from ternary_weight_linear_block_gb300 import tp as TP
from tests.gpu_helpers import bf16_to_f32, ensure_lib, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _emulate(k, n, m, world, mode, seed=60, sign=None, expand=True):
    codes = I.make_codes(seed, n, k)
    scales = I.make_scales(seed, n, k)
    bits, x = I.make_activations(seed, m, k, 0.001, 50.0)
    plans = [TP.ksplit_plan(k, world, r) for r in range(world)]
    lins, xs, locs = [], [], []
    for p in plans:
        cr = to_dev(np.ascontiguousarray(codes[:, p.k0:p.k1]))
        sr = to_dev(np.ascontiguousarray(scales[:, p.k0 // 128:p.k1 // 128]))
        lins.append(TP.KSplitLinear(p, cr, sr, decode=True, prefill=True, expand=expand))
        xs.append(to_dev_bf16(np.ascontiguousarray(bits[:, p.k0:p.k1])))
    sg = [None] * world if sign is None else [to_dev(sign[p.k0:p.k1]) for p in plans]
    for lin, xb, s in zip(lins, xs, sg):
        locs.append(TP.local_phase(lin, xb, s))
    h_all = [h for _, h in locs]
    ys = [TP.finish_phase(lin, xr, h_all, mode) for lin, (xr, _) in zip(lins, locs)]
    B.tern_check()
    rot = [np.concatenate([xr.cpu().numpy()[:, a:a + ln] for a, _, ln in p.padded_columns()],
                          axis=1) for p, (xr, _) in zip(plans, locs)]
    y = sum(bf16_to_f32(yy).astype(np.float64) for yy in ys)
    return codes, scales, x, np.concatenate(rot, axis=1), y, locs, plans


@pytest.mark.parametrize("k,world", [(17408, 2), (3072, 2), (6144, 4), (4096, 2)])
def test_rotation_bitwise_and_decode(k, world):
    codes, scales, x, rot, y, _, _ = _emulate(k, 256, 5, world, "decode")
    assert np.array_equal(rot.view(np.uint32), O.fwht_f32(x).view(np.uint32))
    assert O.rel_frobenius(y, O.linear_f64(x, codes, scales)) <= 4e-3


def test_half_transforms_match_oracle():
    k, world = 17408, 2
    codes, scales, x, rot, y, locs, plans = _emulate(k, 256, 4, world, "decode")
    h0 = locs[0][1].cpu().numpy()[1]      # rank 0: trailing half (first half of block 8)
    h1 = locs[1][1].cpu().numpy()[0]      # rank 1: leading half (second half of block 8)
    assert np.array_equal(h0, O.fwht_half_f32(x[:, 8192:8704]))
    assert np.array_equal(h1, O.fwht_half_f32(x[:, 8704:9216]))
    assert not locs[0][1][0].any() and not locs[1][1][1].any()   # absent halves stay zero


@pytest.mark.parametrize("expand,m", [(True, 40), (False, 40), (True, 200), (False, 200)])
def test_prefill_int8(expand, m):
    """Each rank's prefill on its padded shard; without the expanded weight at
    M = 200 the packed GEMM runs 256-token tiles, split along K."""
    k, world, n = 17408, 2, 512
    codes, scales, x, rot, y, _, _ = _emulate(k, n, m, world, "prefill", expand=expand)
    assert O.rel_frobenius(y, O.linear_f64(x, codes, scales)) <= 2e-2


def test_sign_vector():
    k, world = 17408, 2
    sign = np.where(np.random.default_rng(61).random(k) < 0.5, -1, 1).astype(np.int8)
    codes, scales, x, rot, y, _, _ = _emulate(k, 256, 3, world, "decode", sign=sign)
    assert np.array_equal(rot.view(np.uint32), O.fwht_f32(x, sign).view(np.uint32))
    assert O.rel_frobenius(y, O.linear_f64(x, codes, scales, sign)) <= 4e-3


def test_quant_rotated_matches_fwht_quant():
    """Quantising the rotated values separately gives the rotation kernel's
    own decode operand, fp16 operand and int8 output bit for bit."""
    m, k = 7, 5120
    bits, x = I.make_activations(62, m, k, 0.001, 50.0)
    xb = to_dev_bf16(bits)
    xr, _ = B.fwht(xb, B.TERN_FWHT_F32)
    for mode in (B.TERN_FWHT_DECODE, B.TERN_FWHT_F16, B.TERN_FWHT_I8, B.TERN_FWHT_I8H):
        out, sc = B.fwht(xb, mode)
        out2 = torch.empty_like(out)
        sc2 = torch.empty_like(sc)
        B.tern_quant_rotated(xr, m, k, mode, out2, sc2)
        B.tern_check()
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
        assert torch.equal(sc, sc2)


def test_argument_errors():
    st = B.lib().tern_fwht_shard
    assert st(None, 1, 8704, 0, 1, None, None, None, None, None) == 1      # null x
    x = torch.empty((1, 8704), dtype=torch.bfloat16, device="cuda")
    xr = torch.empty((1, 9216), dtype=torch.float32, device="cuda")
    assert st(x.data_ptr(), 1, 8704, 0, 0, None, xr.data_ptr(), None, None, None) == 2   # 8.5 blocks
    assert st(x.data_ptr(), 1, 8704, 0, 1, None, xr.data_ptr(), None, None, None) == 1   # no h_trail
    cb = B.lib().tern_fwht_combine
    h = torch.empty((1, 512), dtype=torch.float32, device="cuda")
    assert cb(h.data_ptr(), h.data_ptr(), 1, 2, xr.data_ptr(), 9216, 0, None) == 1      # bad part
    assert cb(h.data_ptr(), h.data_ptr(), 1, 0, xr.data_ptr(), 9216, 9, None) == 2      # no block 9
