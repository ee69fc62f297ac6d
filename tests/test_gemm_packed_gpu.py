"""GPU parity of the int8 prefill GEMM read straight from the packed 2-bit
weights (tern_gemm_prefill_packed) against the oracle.

acc (int32) must equal the integer oracle bit for bit and y must equal the
oracle's fp32 rescale bit for bit, on ragged M (not a multiple of the
128-token tile) and N (not a multiple of the 256-row tile), and bit for bit
with the GEMM on the expanded weight.
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


def _layer(codes, scales, expand=False):
    return B.pack_layer(to_dev(codes), to_dev(scales), decode=True, prefill=True, expand=expand)


def _ws(m, n, k):
    nb = max(B.tern_workspace_bytes(B.TERN_OP_GEMM_PACKED, m, n, k), 16)
    return torch.empty(nb, dtype=torch.uint8, device="cuda"), nb


def _run(layer, bits, m):
    y = poison(torch.empty((m, layer.n), dtype=torch.bfloat16, device="cuda"))
    acc = poison(torch.empty((m, layer.n), dtype=torch.int32, device="cuda"))
    B.prefill(layer, to_dev_bf16(bits), y=y, acc=acc, from_packed=True)
    B.tern_check()
    return acc, y


@pytest.mark.parametrize("m", [1, 8, 32, 33, 64, 65, 128, 200])
def test_tiny_layer(m):
    d = I.make_layer(I.TINY, m, seed=0)
    acc, y = _run(_layer(d.codes, d.scales), d.x_bits, m)
    r = O.linear_int8(d.x, d.codes, d.scales)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), r["acc"])
    yg = bf16_to_f32(y)
    assert np.array_equal(yg.view(np.uint32), r["y"].view(np.uint32))
    assert O.rel_frobenius(yg, O.linear_f64(d.x, d.codes, d.scales)) <= 2e-2


@pytest.mark.parametrize("m,n,k", [(300, 272, 2048), (129, 528, 3072), (64, 112, 1024),
                                   (257, 1040, 5120), (31, 1008, 1024), (50, 784, 2048),
                                   (130, 16, 1024), (384, 144, 2048)])
def test_ragged_shapes(m, n, k):
    codes = I.make_codes(13, n, k)
    scales = I.make_scales(13, n, k)
    bits, x = I.make_activations(13, m, k, 0.01, 20.0)
    acc, y = _run(_layer(codes, scales), bits, m)
    r = O.linear_int8(x, codes, scales)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), r["acc"])
    assert np.array_equal(bf16_to_f32(y).view(np.uint32), r["y"].view(np.uint32))


@pytest.mark.parametrize("k", [1024, 5120, 17408])
def test_extreme_magnitudes_exact(k):
    """Every weight +-127 (equal scales give q = 127) against xq = +-127:
    each fp32 chunk sum is at its largest and acc reaches 127 * 127 * K."""
    m, n = 130, 304
    rng = np.random.default_rng(k)
    codes = np.ones((n, k), np.int8)
    codes[5] = -1
    codes[6, 1::3] = 0
    codes[7:] = rng.integers(-1, 2, (n - 7, k)).astype(np.int8)
    scales = np.full((n, k // 128), 0.0625, np.float16)
    lay = _layer(codes, scales)
    xq = np.full((m, k), 127, np.int16)
    xq[1] = -127
    xq[2, ::2] = -127
    xq[3:] = rng.integers(-127, 128, (m - 3, k))
    ts = np.full(m, 1e-3, np.float32)
    y = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
    acc = poison(torch.empty((m, n), dtype=torch.int32, device="cuda"))
    B.tern_gemm_prefill_packed(to_dev(xq.astype(np.float16)), to_dev(ts), lay.packed, lay.q,
                               lay.rscale, m, n, k, y, acc, *_ws(m, n, k))
    B.tern_check()
    assert np.all(lay.q.cpu().numpy() == 127)
    w = codes.astype(np.int64) * 127
    ref = O.acc_int8(xq, w)
    a = acc.cpu().numpy().astype(np.int64)
    assert a[0, 0] == 127 * 127 * k
    assert np.array_equal(a, ref)
    rs = lay.rscale.cpu().numpy()
    assert np.array_equal(bf16_to_f32(y).view(np.uint32), O.y_int8(ref, ts, rs).view(np.uint32))


@pytest.mark.parametrize("m", [16, 48, 96, 512])
def test_equals_expanded_gemm(m):
    """The packed path and the expanded-weight path agree bit for bit."""
    n, k = 2560, 5120
    codes = I.make_codes(21, n, k)
    scales = I.make_scales(21, n, k)
    bits, _ = I.make_activations(21, m, k, 0.001, 50.0)
    lay = _layer(codes, scales, expand=True)
    x = to_dev_bf16(bits)
    outs = []
    for fp in (False, True):
        y = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
        acc = poison(torch.empty((m, n), dtype=torch.int32, device="cuda"))
        B.prefill(lay, x, y=y, acc=acc, from_packed=fp)
        outs.append((acc.clone(), y.clone()))
    B.tern_check()
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))


@pytest.mark.parametrize("layer,m", [(I.GATE_UP, 2048), (I.DOWN, 512), (I.QKV, 64), (I.GATE_UP, 512),
                                     (I.DOWN, 2048), (I.QKV, 2048), (I.O_PROJ, 512), (I.O_PROJ, 128)])
def test_full_size_sampled(layer, m):
    """Full shapes, launched as the bench times them; the oracle computes a
    seeded sample of rows and tokens."""
    d = I.make_layer(layer, m, seed=0)
    acc, y = _run(_layer(d.codes, d.scales), d.x_bits, m)
    rows = np.sort(np.random.default_rng(2).choice(layer.n, 256, replace=False))
    toks = np.sort(np.random.default_rng(3).choice(m, min(m, 128), replace=False))
    r = O.linear_int8(d.x[toks], d.codes[rows], d.scales[rows])
    rt = torch.from_numpy(rows).cuda()
    tt = torch.from_numpy(toks).cuda()
    assert np.array_equal(acc[tt][:, rt].cpu().numpy().astype(np.int64), r["acc"])
    y_s = bf16_to_f32(y[tt][:, rt])
    assert np.array_equal(y_s.view(np.uint32), r["y"].view(np.uint32))
    assert np.isfinite(bf16_to_f32(y)).all()


@pytest.mark.parametrize("m,n,k", [(100, 512, 5120), (128, 5120, 17408), (40, 10240, 5120),
                                   (300, 512, 5120), (512, 10240, 5120)])
def test_split_k_with_and_without_acc(m, n, k):
    """Tiles that fill the GPU unevenly: K ranges split in slices whose exact
    int32 partial sums a second kernel adds; y is the same with or without
    acc.  Above 128 tokens the tiles are CTA pairs' 256 weight rows x 256
    tokens: with fewer tiles than pairs every tile is split (300 tokens), with
    more the whole waves stay whole and only the last wave's tiles are split
    (512 x 10240: 76 tiles whole, 4 in slices)."""
    assert B.tern_kernel_launches(B.TERN_OP_GEMM_PACKED, m, n, k) == 2
    codes = I.make_codes(31, n, k)
    scales = I.make_scales(31, n, k)
    bits, x = I.make_activations(31, m, k, 0.001, 50.0)
    lay = _layer(codes, scales)
    acc, y = _run(lay, bits, m)
    y2 = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
    ws = B.Workspace()
    ws.scratch(B.tern_workspace_bytes(B.TERN_OP_GEMM_PACKED, m, n, k)).fill_(0x5A)   # any contents
    B.prefill(lay, to_dev_bf16(bits), y=y2, from_packed=True, ws=ws)
    B.tern_check()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    rows = np.sort(np.random.default_rng(5).choice(n, 128, replace=False))
    r = O.linear_int8(x, codes[rows], scales[rows])
    rt = torch.from_numpy(rows).cuda()
    assert np.array_equal(acc[:, rt].cpu().numpy().astype(np.int64), r["acc"])
    assert np.array_equal(bf16_to_f32(y[:, rt]).view(np.uint32), r["y"].view(np.uint32))


def test_workspace_required():
    m, n, k = 64, 512, 5120
    lay = _layer(np.zeros((n, k), np.int8), np.zeros((n, k // 128), np.float16))
    need = B.tern_workspace_bytes(B.TERN_OP_GEMM_PACKED, m, n, k)
    assert need > 0 and need % (m * n * 4) == 0   # one int32 plane per K slice
    xq = to_dev(np.ones((m, k), np.float16))
    ts = to_dev(np.ones(m, np.float32))
    y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    acc = torch.empty((m, n), dtype=torch.int32, device="cuda")
    for a in (None, acc.data_ptr()):
        st = B.lib().tern_gemm_prefill_packed(xq.data_ptr(), ts.data_ptr(),
                                              lay.packed.data_ptr(), lay.q.data_ptr(),
                                              lay.rscale.data_ptr(), m, n, k, y.data_ptr(), a,
                                              None, 0, None)
        assert st == 6   # TERN_ERR_WORKSPACE


def test_zero_and_empty():
    m, n, k = 40, 256, 1024
    lay = _layer(np.zeros((n, k), np.int8), np.zeros((n, k // 128), np.float16))
    y = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
    acc = poison(torch.empty((m, n), dtype=torch.int32, device="cuda"))
    xq = to_dev(np.ones((m, k), np.float16))
    B.tern_gemm_prefill_packed(xq, to_dev(np.ones(m, np.float32)), lay.packed, lay.q, lay.rscale,
                               m, n, k, y, acc, *_ws(m, n, k))
    B.tern_check()
    assert not acc.cpu().numpy().any() and not bf16_to_f32(y).any()
    # M = 0 and N = 0 are no-ops
    B.tern_gemm_prefill_packed(xq, to_dev(np.ones(m, np.float32)), lay.packed, lay.q, lay.rscale,
                               0, n, k, y, acc)
    B.tern_gemm_prefill_packed(xq, to_dev(np.ones(m, np.float32)), lay.packed, lay.q, lay.rscale,
                               m, 0, k, y, acc)


@pytest.mark.parametrize("m", [4, 16, 17, 128, 129, 256, 257, 300])
def test_forward_picks_the_path(m):
    """binding.forward: the decode GEMV up to 16 tokens, the packed GEMM up to
    256, the expanded GEMM above -- each call equal to its path's own call."""
    n, k = 512, 2048
    codes = I.make_codes(33, n, k)
    scales = I.make_scales(33, n, k)
    bits, x = I.make_activations(33, m, k, 0.001, 50.0)
    lay = _layer(codes, scales, expand=True)
    xd = to_dev_bf16(bits)
    ws = B.Workspace()
    got = B.forward(lay, xd, ws=ws)
    if m <= 16:
        want = B.decode(lay, xd, ws)
    else:
        want = B.prefill(lay, xd, from_packed=m <= 256, ws=ws)
    B.tern_check()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    tol = 4e-3 if m <= 16 else 2e-2
    assert O.rel_frobenius(bf16_to_f32(got), O.linear_f64(x, codes, scales)) <= tol
