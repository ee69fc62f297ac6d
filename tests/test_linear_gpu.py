"""GPU parity of tern_linear_decode, the one-launch decode path (rotation
folded into the GEMV prologue): bit-identical to tern_fwht_quant(DECODE)
followed by tern_gemv_decode, and within the decode tolerance of the fp64
oracle."""

import numpy as np
import pytest
import torch

from oracle import tern_oracle as O
from ternary_weight_linear_block_gb300 import binding as B
from ternary_weight_linear_block_gb300 import inputs as I
from tests.decode_bounds import block_sample_rows, check_elementwise
from tests.gpu_helpers import bf16_to_f32, ensure_lib, poison, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

TOL = 4e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _layer(codes, scales):
    return B.pack_layer(to_dev(codes), to_dev(scales), decode=True, prefill=False)


def _both(layer, x, m, sign=None):
    """(fused, two-call) outputs as raw bf16 bits."""
    out = []
    for fused in (True, False):
        y = poison(torch.empty((m, layer.n), dtype=torch.bfloat16, device="cuda"))
        B.decode(layer, x, B.Workspace(), y=y, sign=sign, fused=fused)
        B.tern_check()
        out.append(y.cpu().view(torch.int16).numpy())
    return out


@pytest.mark.parametrize("n,k,m", [(256, 1024, 1), (256, 1024, 8), (100, 2048, 3), (272, 3072, 13),
                                   (4112, 4096, 5), (1040, 8192, 16), (10240, 5120, 4),
                                   (5120, 17408, 16), (34816, 5120, 1), (34816, 5120, 16)])
def test_bit_identical_to_two_calls(n, k, m):
    codes = I.make_codes(11, n, k)
    scales = I.make_scales(11, n, k)
    bits, _ = I.make_activations(11, m, k, 0.001, 50.0)
    f, u = _both(_layer(codes, scales), to_dev_bf16(bits), m)
    assert np.array_equal(f, u)


def test_bit_identical_with_sign_vector():
    n, k, m = 2048, 4096, 6
    codes = I.make_codes(12, n, k)
    scales = I.make_scales(12, n, k)
    bits, _ = I.make_activations(12, m, k, 0.01, 20.0)
    sign = torch.from_numpy(np.where(np.random.default_rng(5).random(k) < 0.5, -1, 1)
                            .astype(np.int8)).cuda()
    f, u = _both(_layer(codes, scales), to_dev_bf16(bits), m, sign=sign)
    assert np.array_equal(f, u)


@pytest.mark.parametrize("m", [16, 9])
def test_resident_operand_in_chunks(m):
    """More groups per CTA than the resident area holds at this M: the CTA
    rotates again for each chunk (40000 rows x 5120: 71 units per CTA)."""
    n, k = 40000, 5120
    codes = I.make_codes(13, n, k)
    scales = I.make_scales(13, n, k)
    bits, _ = I.make_activations(13, m, k, 0.001, 50.0)
    f, u = _both(_layer(codes, scales), to_dev_bf16(bits), m)
    assert np.array_equal(f, u)


@pytest.mark.parametrize("layer,m", [(I.TINY, 1), (I.TINY, 8), (I.GATE_UP, 1), (I.GATE_UP, 4),
                                     (I.DOWN, 16), (I.QKV, 8), (I.O_PROJ, 4)])
def test_against_oracle(layer, m):
    d = I.make_layer(layer, m, seed=0)
    lay = _layer(d.codes, d.scales)
    y = poison(torch.empty((m, lay.n), dtype=torch.bfloat16, device="cuda"))
    B.decode(lay, to_dev_bf16(d.x_bits), B.Workspace(), y=y, fused=True)
    B.tern_check()
    y = bf16_to_f32(y)
    rows = np.arange(lay.n) if lay.n <= 512 else block_sample_rows(lay.n, seed=2)
    ref = O.linear_f64(d.x, d.codes[rows], d.scales[rows])
    e = O.rel_frobenius(y[:, rows], ref)
    assert e <= TOL, e
    assert np.isfinite(y).all()
    check_elementwise(y[:, rows], ref, d.codes[rows], d.scales[rows], d.x,
                      what=f"fused {layer.name} M={m}")


def test_empty_and_repeat():
    d = I.make_layer(I.QKV, 4, seed=3)
    lay = _layer(d.codes, d.scales)
    x = to_dev_bf16(d.x_bits)
    ws = B.Workspace()
    assert B.tern_linear_decode(x, None, lay.packed, 0, lay.n, lay.k, x, None, 0) == B.TERN_OK
    y1 = B.decode(lay, x, ws, fused=True)
    y2 = B.decode(lay, x, ws, fused=True)
    B.tern_check()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("fused", [False, True])
def test_decode_graph_matches_decode(fused):
    """B.DecodeGraph (host in, graph replay, host out) returns exactly what
    B.decode returns, for two different inputs replayed through one graph."""
    d = I.make_layer(I.QKV, 4, seed=4)
    lay = _layer(d.codes, d.scales)
    plan = B.DecodeGraph(lay, 4, fused=fused)
    for seed in (5, 6):
        bits, _ = I.make_activations(seed, 4, lay.k, 0.001, 50.0)
        x = to_dev_bf16(bits)
        want = B.decode(lay, x, B.Workspace())
        got = plan.run(x.cpu())
        B.tern_check()
        assert torch.equal(got, want.cpu())


def test_decode_step_graph_matches_decode():
    """B.DecodeStepGraph: several (layer, M) decode forwards in one graph, each
    returning exactly what B.decode returns."""
    d1 = I.make_layer(I.QKV, 4, seed=7)
    d2 = I.make_layer(I.O_PROJ, 1, seed=8)
    l1 = _layer(d1.codes, d1.scales)
    l2 = _layer(d2.codes, d2.scales)
    plan = B.DecodeStepGraph([(l1, 1), (l1, 4), (l2, 1)])
    for seed in (9, 10):
        xs = []
        for i, (lay, m) in enumerate([(l1, 1), (l1, 4), (l2, 1)]):
            bits, _ = I.make_activations(seed + 10 * i, m, lay.k, 0.001, 50.0)
            xs.append(to_dev_bf16(bits))
            plan.x_host[i].copy_(xs[-1].cpu())
        got = plan.run()
        B.tern_check()
        for (lay, m), x, y in zip([(l1, 1), (l1, 4), (l2, 1)], xs, got):
            assert torch.equal(y, B.decode(lay, x, B.Workspace()).cpu())


@pytest.mark.parametrize("fused", [False, True])
def test_zero_copy_graph_matches_copies(fused):
    """Zero-copy (kernels read x from and write y to pinned host memory) and
    copying graphs return the same bits, at a fixup shape (M = 16) too."""
    d = I.make_layer(I.QKV, 16, seed=11)
    lay = _layer(d.codes, d.scales)
    entries = [(lay, 1), (lay, 16)]
    zc = B.DecodeStepGraph(entries, fused=fused, zero_copy=None)
    cp = B.DecodeStepGraph(entries, fused=fused, zero_copy=False)
    assert not cp.zero_copy
    for i, (_, m) in enumerate(entries):
        bits, _ = I.make_activations(12 + i, m, lay.k, 0.001, 50.0)
        x = to_dev_bf16(bits).cpu()
        zc.x_host[i].copy_(x)
        cp.x_host[i].copy_(x)
    a = zc.run()
    b = cp.run()
    B.tern_check()
    for ya, yb in zip(a, b):
        assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))
