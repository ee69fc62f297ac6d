"""GPU parity of the int8 prefill path against the oracle.

acc (int32) must equal the integer oracle bit for bit; y must be within
2e-3 (relative Frobenius) of the CPU int8-path oracle and within 2e-2 of
the exact fp64 layer.
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


def _gemm_raw(xq, ts, w, rs, typed=False):
    """Call a GEMM entry point directly on integer operands: the fp16-held
    one (tern_gemm_prefill_int8h) or, with ``typed``, the int8-typed one
    (tern_gemm_prefill_int8, which needs its workspace)."""
    m, k = xq.shape
    n = w.shape[0]
    y = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
    acc = poison(torch.empty((m, n), dtype=torch.int32, device="cuda"))
    if typed:
        nb = B.tern_workspace_bytes(B.TERN_OP_GEMM_INT8, m, n, k)
        ws = poison(torch.empty(nb, dtype=torch.uint8, device="cuda"))
        B.tern_gemm_prefill_int8(to_dev(xq.astype(np.int8)), to_dev(ts), to_dev(w.astype(np.int8)),
                                 to_dev(rs), m, n, k, y, acc, ws, nb)
    else:
        B.tern_gemm_prefill_int8h(to_dev(xq.astype(np.float16)), to_dev(ts),
                                  to_dev(w.astype(np.float16)), to_dev(rs), m, n, k, y, acc)
    B.tern_check()
    return acc.cpu().numpy().astype(np.int64), bf16_to_f32(y)


def _prefill(codes, scales, bits, m, typed=False):
    """The layer's prefill through binding.prefill: on the fp16-held weight
    (I8H operand, tern_gemm_prefill_int8h) or, with ``typed``, on the int8
    weight (I8 operand, tern_gemm_prefill_int8)."""
    layer = B.pack_layer(to_dev(codes), to_dev(scales), decode=False, prefill=True,
                         expand=not typed, int8=typed)
    assert (layer.w_q is None) == typed and (layer.w_int8 is None) != typed
    y = poison(torch.empty((m, layer.n), dtype=torch.bfloat16, device="cuda"))
    acc = poison(torch.empty((m, layer.n), dtype=torch.int32, device="cuda"))
    B.prefill(layer, to_dev_bf16(bits), y=y, acc=acc, from_packed=False)
    B.tern_check()
    return acc, y


@pytest.mark.parametrize("typed", [False, True])
@pytest.mark.parametrize("m", [1, 8, 128, 200])
def test_tiny_layer(m, typed):
    d = I.make_layer(I.TINY, m, seed=0)
    acc, y = _prefill(d.codes, d.scales, d.x_bits, m, typed)
    r = O.linear_int8(d.x, d.codes, d.scales)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), r["acc"])
    yg = bf16_to_f32(y)
    assert O.rel_frobenius(yg, r["y"]) <= 2e-3
    assert np.array_equal(yg.view(np.uint32), r["y"].view(np.uint32))   # same fp32 steps
    assert O.rel_frobenius(yg, O.linear_f64(d.x, d.codes, d.scales)) <= 2e-2


@pytest.mark.parametrize("m,n,k", [(300, 272, 2048), (129, 528, 3072), (64, 256, 1024),
                                   (257, 1040, 5120), (130, 16, 1024), (384, 144, 2048)])
@pytest.mark.parametrize("typed", [False, True])
def test_ragged_shapes(m, n, k, typed):
    """Ragged M and N on both sides of the switch to CTA pairs (M > 128),
    including pair tiles whose odd CTA holds no valid weight row (N = 16)
    or only 16 of its 128 (N = 144)."""
    codes = I.make_codes(11, n, k)
    scales = I.make_scales(11, n, k)
    bits, x = I.make_activations(11, m, k, 0.01, 20.0)
    acc, y = _prefill(codes, scales, bits, m, typed)
    r = O.linear_int8(x, codes, scales)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), r["acc"])
    assert np.array_equal(bf16_to_f32(y).view(np.uint32), r["y"].view(np.uint32))


@pytest.mark.parametrize("typed", [False, True])
@pytest.mark.parametrize("k", [1024, 5120, 17408])
def test_extreme_magnitudes_exact(k, typed):
    """|acc| up to 127*127*K: every fp32 chunk sum is at its largest."""
    m, n = 130, 272
    rng = np.random.default_rng(k)
    xq = np.full((m, k), 127, np.int16)
    xq[1] = -127
    xq[2, ::2] = -127
    xq[3:] = rng.integers(-127, 128, (m - 3, k))
    w = np.full((n, k), 127, np.int16)
    w[5] = -127
    w[6, 1::3] = 0
    w[7:] = rng.integers(-127, 128, (n - 7, k))
    ts = np.full(m, 1e-3, np.float32)
    rs = np.full(n, 2e-3, np.float32)
    acc, y = _gemm_raw(xq, ts, w, rs, typed)
    ref = O.acc_int8(xq, w)
    assert acc[0, 0] == 127 * 127 * k
    assert np.array_equal(acc, ref)
    assert np.array_equal(y.view(np.uint32), O.y_int8(ref, ts, rs).view(np.uint32))


@pytest.mark.parametrize("layer,m,typed", [
    (I.GATE_UP, 512, False), (I.DOWN, 512, False), (I.GATE_UP, 2048, False),
    (I.DOWN, 2048, False), (I.QKV, 512, False), (I.QKV, 2048, False), (I.O_PROJ, 512, False),
    (I.O_PROJ, 2048, False), (I.GATE_UP, 2048, True), (I.DOWN, 2048, True)])
def test_full_size_sampled(layer, m, typed):
    """Full prefill shapes of the 64-layer stack, with the workspace the bench
    gives, so the K-split plans run where the cost model picks them (on 152
    SMs: qkv and down at M = 512, down, qkv and o at M = 2048); the oracle
    computes a seeded sample of rows."""
    d = I.make_layer(layer, m, seed=0)
    acc, y = _prefill(d.codes, d.scales, d.x_bits, m, typed)
    rows = np.sort(np.random.default_rng(2).choice(layer.n, 256, replace=False))
    toks = np.sort(np.random.default_rng(3).choice(m, min(m, 256), replace=False))
    r = O.linear_int8(d.x[toks], d.codes[rows], d.scales[rows])
    # per-token quantisation sees the whole token, so the token sample is exact
    rt = torch.from_numpy(rows).cuda()
    tt = torch.from_numpy(toks).cuda()
    acc_s = acc[tt][:, rt].cpu().numpy().astype(np.int64)
    y_s = bf16_to_f32(y[tt][:, rt])
    assert np.array_equal(acc_s, r["acc"])
    assert np.array_equal(y_s.view(np.uint32), r["y"].view(np.uint32))
    exact = O.linear_f64(d.x[toks], d.codes[rows], d.scales[rows])
    assert O.rel_frobenius(y_s, exact) <= 2e-2
    assert np.isfinite(bf16_to_f32(y)).all()


@pytest.mark.parametrize("typed", [False, True])
def test_zero_operands(typed):
    m, n, k = 40, 256, 1024
    acc, y = _gemm_raw(np.zeros((m, k), np.int16), np.zeros(m, np.float32),
                       np.zeros((n, k), np.int16), np.zeros(n, np.float32), typed)
    assert not acc.any() and not y.any()


@pytest.mark.parametrize("m,n,k", [(128, 5120, 17408), (40, 1024, 5120), (512, 5120, 17408),
                                   (2048, 5120, 17408), (512, 10240, 5120)])
def test_split_k_is_bit_identical(m, n, k):
    """With a workspace, calls whose tiles fill the GPU unevenly split K in
    slices of whole chunks -- every tile, or only the tiles of the last,
    partial wave (the last two shapes); the int32 partials are exact, so acc
    and y equal the unsplit call's bit for bit (and the integer oracle on a
    sample)."""
    assert B.tern_workspace_bytes(B.TERN_OP_GEMM, m, n, k) > 0
    codes = I.make_codes(23, n, k)
    scales = I.make_scales(23, n, k)
    bits, x = I.make_activations(23, m, k, 0.001, 50.0)
    layer = B.pack_layer(to_dev(codes), to_dev(scales), decode=False, prefill=True, int8=True)
    xq, ts = B.fwht(to_dev_bf16(bits), B.TERN_FWHT_I8H)
    outs = []
    for split in (False, True):
        y = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
        acc = poison(torch.empty((m, n), dtype=torch.int32, device="cuda"))
        nb = B.tern_workspace_bytes(B.TERN_OP_GEMM, m, n, k) if split else 0
        ws = torch.full((max(nb, 16),), 0x5A, dtype=torch.uint8, device="cuda")
        B.tern_gemm_prefill_int8h(xq, ts, layer.w_q, layer.rscale, m, n, k, y, acc,
                                  ws if split else None, nb)
        outs.append((acc, y))
    # the int8-typed call: its workspace holds both widened operands, then the split pieces
    xq8, ts8 = B.fwht(to_dev_bf16(bits), B.TERN_FWHT_I8)
    nb8 = B.tern_workspace_bytes(B.TERN_OP_GEMM_INT8, m, n, k)
    assert nb8 >= (m * k + n * k) * 2 + B.tern_workspace_bytes(B.TERN_OP_GEMM, m, n, k)
    ws8 = torch.full((nb8,), 0x5A, dtype=torch.uint8, device="cuda")
    y = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
    acc = poison(torch.empty((m, n), dtype=torch.int32, device="cuda"))
    B.tern_gemm_prefill_int8(xq8, ts8, layer.w_int8, layer.rscale, m, n, k, y, acc, ws8, nb8)
    outs.append((acc, y))
    B.tern_check()
    assert torch.equal(ts, ts8)
    for acc_i, y_i in outs[1:]:
        assert torch.equal(outs[0][0], acc_i)
        assert torch.equal(outs[0][1].view(torch.int16), y_i.view(torch.int16))
    rows = np.sort(np.random.default_rng(6).choice(n, 64, replace=False))
    r = O.linear_int8(x, codes[rows], scales[rows])
    assert np.array_equal(outs[1][0][:, torch.from_numpy(rows).cuda()].cpu().numpy()
                          .astype(np.int64), r["acc"])
