"""GPU parity of the fp16 prefill variant (tern_expand_fp16 +
tern_gemm_prefill_fp16) against the oracle.

The variant multiplies the decode operand (fp16 rotated activations with one
power-of-two factor per token and block) by the exact fp16 weight code * s.
Its output must be within 4e-3 of the exact fp64 layer (the decode
tolerance), within 2e-3 of the same arithmetic done in fp64 on the same fp16
operands, and more accurate than the int8 path on the same inputs.
"""

import numpy as np
import pytest
import torch

from oracle import tern_oracle as O
from ternary_weight_linear_block_gb300 import binding as B
from ternary_weight_linear_block_gb300 import inputs as I
from tests.gpu_helpers import bf16_to_f32, ensure_lib, poison, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _operand_ref(x, codes, scales):
    """fp64 of the variant's arithmetic on its exact fp16 operands."""
    xh, inv = O.f16_operand(O.fwht_f32(x))
    m, k = xh.shape
    xe = (xh.astype(np.float64).reshape(m, k // 1024, 1024) *
          inv.astype(np.float64)[:, :, None]).reshape(m, k)
    return xe @ O.dequant_f64(codes, scales).T


def _run(codes, scales, bits, m):
    w_h = B.expand_fp16(to_dev(codes), to_dev(scales))
    y = poison(torch.empty((m, codes.shape[0]), dtype=torch.bfloat16, device="cuda"))
    B.prefill_fp16(w_h, to_dev_bf16(bits), y=y)
    B.tern_check()
    return w_h, bf16_to_f32(y)


def test_expand_is_exact():
    d = I.make_layer(I.TINY, 1, seed=3)
    w_h, _ = _run(d.codes, d.scales, d.x_bits, 1)
    ref = O.dequant_f64(d.codes, d.scales).astype(np.float16)
    assert np.array_equal(w_h.cpu().numpy().view(np.uint16), ref.view(np.uint16))


@pytest.mark.parametrize("m", [1, 8, 128, 200])
def test_tiny_layer(m):
    d = I.make_layer(I.TINY, m, seed=0)
    _, y = _run(d.codes, d.scales, d.x_bits, m)
    assert O.rel_frobenius(y, _operand_ref(d.x, d.codes, d.scales)) <= 2e-3
    assert O.rel_frobenius(y, O.linear_f64(d.x, d.codes, d.scales)) <= 4e-3


@pytest.mark.parametrize("m,n,k", [(300, 272, 2048), (129, 528, 3072), (257, 1040, 5120),
                                   (40, 256, 17408), (130, 16, 1024)])
def test_ragged_shapes(m, n, k):
    codes = I.make_codes(17, n, k)
    scales = I.make_scales(17, n, k)
    bits, x = I.make_activations(17, m, k, 0.001, 50.0)
    _, y = _run(codes, scales, bits, m)
    assert O.rel_frobenius(y, _operand_ref(x, codes, scales)) <= 2e-3
    assert O.rel_frobenius(y, O.linear_f64(x, codes, scales)) <= 4e-3


@pytest.mark.parametrize("layer,m", [(I.GATE_UP, 2048), (I.DOWN, 512)])
def test_full_size_sampled_and_more_accurate_than_int8(layer, m):
    d = I.make_layer(layer, m, seed=0)
    w_h = B.expand_fp16(to_dev(d.codes), to_dev(d.scales))
    x = to_dev_bf16(d.x_bits)
    y16 = B.prefill_fp16(w_h, x)
    lay = B.pack_layer(to_dev(d.codes), to_dev(d.scales), decode=False, prefill=True)
    y8 = B.prefill(lay, x)
    B.tern_check()
    rows = np.sort(np.random.default_rng(4).choice(layer.n, 192, replace=False))
    toks = np.sort(np.random.default_rng(5).choice(m, 96, replace=False))
    rt, tt = torch.from_numpy(rows).cuda(), torch.from_numpy(toks).cuda()
    exact = O.linear_f64(d.x[toks], d.codes[rows], d.scales[rows])
    e16 = O.rel_frobenius(bf16_to_f32(y16[tt][:, rt]), exact)
    e8 = O.rel_frobenius(bf16_to_f32(y8[tt][:, rt]), exact)
    assert e16 <= 4e-3
    assert e16 < e8 / 2
    assert np.isfinite(bf16_to_f32(y16)).all()


def test_zero_and_empty():
    m, n, k = 16, 256, 1024
    w_h = B.expand_fp16(to_dev(np.zeros((n, k), np.int8)), to_dev(np.zeros((n, 8), np.float16)))
    xh = to_dev(np.ones((m, k), np.float16))
    xs = to_dev(np.ones((m, 1), np.float32))
    y = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
    B.tern_gemm_prefill_fp16(xh, xs, w_h, m, n, k, y)
    B.tern_check()
    assert not bf16_to_f32(y).any()
    B.tern_gemm_prefill_fp16(xh, xs, w_h, 0, n, k, y)


@pytest.mark.parametrize("m,n,k", [(128, 5120, 17408), (2048, 5120, 17408)])
def test_split_k_within_rounding(m, n, k):
    """Split along K (workspace given; all tiles, or the last wave's), the fp32
    slice sums are added in slice order: the same output up to fp32 rounding."""
    assert B.tern_workspace_bytes(B.TERN_OP_GEMM, m, n, k) > 0
    codes = I.make_codes(24, n, k)
    scales = I.make_scales(24, n, k)
    bits, x = I.make_activations(24, m, k, 0.001, 50.0)
    w_h = B.expand_fp16(to_dev(codes), to_dev(scales))
    xh, xs = B.fwht(to_dev_bf16(bits), B.TERN_FWHT_F16)
    y0 = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
    y1 = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
    B.tern_gemm_prefill_fp16(xh, xs, w_h, m, n, k, y0)
    nb = B.tern_workspace_bytes(B.TERN_OP_GEMM, m, n, k)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    B.tern_gemm_prefill_fp16(xh, xs, w_h, m, n, k, y1, ws, nb)
    B.tern_check()
    a, b = bf16_to_f32(y0), bf16_to_f32(y1)
    assert O.rel_frobenius(b, a) <= 2e-3
    rows = np.sort(np.random.default_rng(7).choice(n, 128, replace=False))
    exact = O.linear_f64(x, codes[rows], scales[rows])
    assert O.rel_frobenius(b[:, rows], exact) <= 4e-3
