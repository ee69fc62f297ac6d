"""GPU parity of the decode path (rotation + tern_gemv_decode) against the
fp64 oracle: relative Frobenius error <= 4e-3 on bf16 outputs, and every
compared element within the element-wise bound of tests/decode_bounds.py."""

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


def _decode(layer, bits, m, ws=None):
    ws = ws or B.Workspace()
    y = poison(torch.empty((m, layer.n), dtype=torch.bfloat16, device="cuda"))
    B.decode(layer, to_dev_bf16(bits), ws, y=y)   # rotation, then tern_gemv_decode
    B.tern_check()          # raises if a bounded device-side wait gave up
    return bf16_to_f32(y)


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8, 9, 12, 16])
def test_tiny_layer(m):
    d = I.make_layer(I.TINY, m, seed=0)
    y = _decode(_layer(d.codes, d.scales), d.x_bits, m)
    ref = O.linear_f64(d.x, d.codes, d.scales)
    assert np.isfinite(y).all()
    e = O.rel_frobenius(y, ref)
    assert e <= TOL, e
    assert e > 0   # an exact match against fp64 would be suspicious for bf16 outputs
    check_elementwise(y, ref, d.codes, d.scales, d.x, what=f"tiny M={m}")


@pytest.mark.parametrize("n,k,m", [(100, 2048, 3), (272, 3072, 13), (16, 1024, 1), (4112, 4096, 5),
                                   (1040, 8192, 16)])
def test_ragged_shapes(n, k, m):
    codes = I.make_codes(7, n, k)
    scales = I.make_scales(7, n, k)
    bits, x = I.make_activations(7, m, k, 0.01, 20.0)
    y = _decode(_layer(codes, scales), bits, m)
    ref = O.linear_f64(x, codes, scales)
    e = O.rel_frobenius(y, ref)
    assert e <= TOL, e
    check_elementwise(y, ref, codes, scales, x, what=f"{n}x{k} M={m}")


@pytest.mark.parametrize("layer,m", [(I.GATE_UP, 1), (I.GATE_UP, 4), (I.GATE_UP, 16), (I.DOWN, 1),
                                     (I.DOWN, 4), (I.DOWN, 8), (I.DOWN, 16), (I.QKV, 1),
                                     (I.QKV, 8), (I.QKV, 16), (I.O_PROJ, 4)])
def test_full_size_sampled_rows(layer, m):
    """Full workload shapes in the benchmarked launch; the oracle computes a
    seeded sample of output rows for all tokens: 512 at random plus two of
    every 512-row block (the GEMV's unit of rows, so every block, every
    block's owners and every owner's slot are looked at)."""
    d = I.make_layer(layer, m, seed=0)
    y = _decode(_layer(d.codes, d.scales), d.x_bits, m)
    rows = block_sample_rows(layer.n, seed=1)
    ref = O.linear_f64(d.x, d.codes[rows], d.scales[rows])
    e = O.rel_frobenius(y[:, rows], ref)
    assert e <= TOL, e
    assert np.isfinite(y).all()
    check_elementwise(y[:, rows], ref, d.codes[rows], d.scales[rows], d.x,
                      what=f"{layer.name} M={m}")


@pytest.mark.parametrize("layer,m", [(I.QKV, 4), (I.DOWN, 1), (I.DOWN, 16), (I.GATE_UP, 8)])
def test_repeat_calls_reuse_workspace(layer, m):
    """Repeated calls on one workspace give the same bits, in-kernel sums
    (gate/up at M <= 8) and fixup shapes alike: the shared blocks' slots are
    added in slot order, and every call leaves every word of the workspace
    zero (a nonzero word is a published partial sum), so the next call's
    first owners wait for fresh words."""
    d = I.make_layer(layer, m, seed=3)
    lay = _layer(d.codes, d.scales)
    ws = B.Workspace()
    ys = [_decode(lay, d.x_bits, m, ws) for _ in range(4)]
    for y in ys[1:]:
        assert np.array_equal(y.view(np.uint32), ys[0].view(np.uint32))
    words = ws.buf[:B.tern_workspace_bytes(B.TERN_OP_GEMV, m, layer.n, layer.k)]
    assert not words.any()


def test_special_weights():
    k, n, m = 2048, 64, 3
    bits, x = I.make_activations(9, m, k, 0.0, 1.0)
    scales = I.make_scales(9, n, k)
    codes = np.zeros((n, k), np.int8)
    y = _decode(_layer(codes, scales), bits, m)
    # all-zero codes: only the rounding left by the group offsets' cancellation
    check_elementwise(y, np.zeros((m, n)), codes, scales, x, what="zero codes")
    assert np.abs(y).max() < 1e-3 * np.abs(O.rotate_f64(x)).max()
    codes[5, 1300] = -1                     # a single nonzero code
    y = _decode(_layer(codes, scales), bits, m)
    ref = O.linear_f64(x, codes, scales)
    check_elementwise(y, ref, codes, scales, x, what="one code")
    xr = O.rotate_f64(x)
    want = -float(scales[5, 1300 // 128]) * xr[:, 1300]
    assert np.allclose(y[:, 5], want, rtol=2 ** -7, atol=1e-4)


def test_workspace_after_a_gemm_is_cleaned():
    """A Workspace a split GEMM used holds partial sums; nonzero words would
    pass for the GEMV's published partial sums.  Poison it that way through
    ``scratch`` (as a GEMM may leave it): the next decode through ``get``
    zero-fills it first, so the in-kernel reduction (one launch, row blocks
    shared by up to four CTAs at M = 1) matches a fresh workspace bit for
    bit."""
    n, k, m = 34816, 1024, 1
    assert B.tern_kernel_launches(B.TERN_OP_GEMV, m, n, k) == 1
    codes = I.make_codes(41, n, k)
    scales = I.make_scales(41, n, k)
    bits, x = I.make_activations(41, m, k, 0.001, 50.0)
    layer = _layer(codes, scales)
    want = _decode(layer, bits, m)
    ws = B.Workspace()
    buf = ws.scratch(B.tern_workspace_bytes(B.TERN_OP_GEMM, 512, 5120, 17408))
    buf.view(torch.int32).fill_(0x3F800000)               # 1.0f in every word
    got = _decode(layer, bits, m, ws)
    assert np.array_equal(got, want)
    rows = block_sample_rows(n, seed=2, extra=256)
    ref = O.linear_f64(x, codes[rows], scales[rows])
    assert O.rel_frobenius(got[:, rows], ref) <= TOL
    check_elementwise(got[:, rows], ref, codes[rows], scales[rows], x, what="after a GEMM")


def test_repack_in_place_then_decode_on_the_same_stream():
    """tern_pack rewrites a layer's packed units in place and the decode call
    follows on the same stream with no synchronisation in between.  The GEMV
    streams the weights before its programmatic launch wait, so it must still
    see the new weights: the packing kernel lets no later kernel start before
    it has finished."""
    n, k, m = I.GATE_UP.n, I.GATE_UP.k, 4
    g = torch.Generator(device="cuda")
    sets = []
    for s in range(2):
        g.manual_seed(500 + s)
        codes = (torch.randint(0, 3, (n, k), dtype=torch.int8, device="cuda", generator=g)
                 - 1).to(torch.int8)
        scales = (0.02 * torch.randn((n, k // 128), device="cuda", generator=g).abs()
                  + 1e-3).to(torch.float16)
        sets.append((codes, scales))
    x = to_dev_bf16(I.make_activations(501, m, k, I.GATE_UP.outlier_frac,
                                       I.GATE_UP.outlier_mult)[0])
    ws = B.Workspace()
    ref = []
    for codes, scales in sets:
        lay = B.pack_layer(codes, scales, decode=True, prefill=False)
        torch.cuda.synchronize()
        y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        B.decode(lay, x, ws, y=y)
        torch.cuda.synchronize()
        ref.append(y.clone())
    assert not torch.equal(ref[0], ref[1])
    shared = B.pack_layer(*sets[0], decode=True, prefill=False)
    ys = []
    for it in range(8):
        codes, scales = sets[it % 2]
        B.tern_pack(codes, scales, n, k, shared.packed, None, None, None)
        y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        B.decode(shared, x, ws, y=y)
        ys.append(y)
    B.tern_check()
    for it, y in enumerate(ys):
        assert torch.equal(y, ref[it % 2]), f"call {it} saw other weights"


@pytest.mark.parametrize("layer,m", [(I.TINY, 3), (I.QKV, 4), (I.DOWN, 16), (I.GATE_UP, 1)])
def test_f32_input_entry_point(layer, m):
    """tern_gemv_decode_f32 (fp32 rotated activations in, the operand formed
    in the workspace) is bit-identical to rotation -> tern_gemv_decode, and
    within the decode tolerance of the oracle."""
    d = I.make_layer(layer, m, seed=21)
    lay = _layer(d.codes, d.scales)
    x = to_dev_bf16(d.x_bits)
    want = bf16_to_f32(B.decode(lay, x, B.Workspace()))
    xr, _ = B.fwht(x, B.TERN_FWHT_F32)
    n, k = layer.n, layer.k
    ws = B.Workspace()
    for _ in range(2):                       # twice: the GEMV part is left zero-filled
        buf = ws.get(B.tern_workspace_bytes(B.TERN_OP_GEMV_F32, m, n, k))
        y = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
        B.tern_gemv_decode_f32(lay.packed, xr, m, n, k, y, buf, buf.numel())
        B.tern_check()
        got = bf16_to_f32(y)
        assert np.array_equal(got, want)
    rows = np.arange(n) if n <= 512 else block_sample_rows(n, seed=3, extra=128)
    ref = O.linear_f64(d.x, d.codes[rows], d.scales[rows])
    assert O.rel_frobenius(got[:, rows], ref) <= TOL
    check_elementwise(got[:, rows], ref, d.codes[rows], d.scales[rows], d.x, what="f32 entry")
