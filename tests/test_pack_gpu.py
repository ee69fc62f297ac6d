"""GPU parity of tern_pack against the oracle (bitwise)."""

import numpy as np
import pytest
import torch

from oracle import tern_oracle as O
from ternary_weight_linear_block_gb300 import binding as B
from ternary_weight_linear_block_gb300 import inputs as I
from tests.gpu_helpers import ensure_lib, f16_bits, poison, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _pack(codes, scales):
    n, k = codes.shape
    cd, sd = to_dev(codes), to_dev(scales)
    packed = poison(torch.empty(B.tern_packed_bytes(n, k), dtype=torch.uint8, device="cuda"))
    q = poison(torch.empty((n, k // 128), dtype=torch.int8, device="cuda"))
    rs = poison(torch.empty(n, dtype=torch.float32, device="cuda"))
    w8 = poison(torch.empty((n, k), dtype=torch.int8, device="cuda"))
    B.tern_pack(cd, sd, n, k, packed, q, rs, w8)
    torch.cuda.synchronize()
    return packed, q, rs, w8


@pytest.mark.parametrize("n,k", [(256, 1024), (100, 2048), (16, 1024), (300, 3072), (5120, 17408), (10240, 5120)])
def test_pack_bitwise(n, k):
    codes = I.make_codes(5, n, k)
    scales = I.make_scales(5, n, k)
    scales[3 % n] = 0                          # a zero row
    if n > 10:
        scales[7, ::2] = -scales[7, ::2]       # negative scales
    packed, q, rs, w8 = _pack(codes, scales)
    assert np.array_equal(packed.cpu().numpy(), O.pack_weights(codes, scales))
    qo, ro, _ = O.decompose_scales(scales)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(rs.cpu().numpy().view(np.uint32), ro.view(np.uint32))
    w = O.w_int8(codes, qo)
    assert np.array_equal(w8.cpu().numpy(), w.astype(np.int8))
    assert np.abs(w).max() <= 127


def test_pack_full_gate_up_shape():
    layer = I.GATE_UP
    codes = I.make_codes(0, layer.n, layer.k)
    scales = I.make_scales(0, layer.n, layer.k)
    packed, q, rs, w8 = _pack(codes, scales)
    assert np.array_equal(packed.cpu().numpy(), O.pack_weights(codes, scales))
    qo, ro, _ = O.decompose_scales(scales)
    assert np.array_equal(q.cpu().numpy(), qo)
    rows = np.random.default_rng(0).choice(layer.n, 256, replace=False)
    w = O.w_int8(codes[rows], qo[rows])
    assert np.array_equal(w8[torch.from_numpy(rows).cuda()].cpu().numpy(), w.astype(np.int8))


@pytest.mark.parametrize("rows,cols", [(1, 16), (3, 48), (256, 1024), (5120, 17408)])
def test_widen_int8_exact(rows, cols):
    """tern_widen_int8 holds every int8 value, -128..127, exactly in fp16."""
    rng = np.random.default_rng(rows + cols)
    src = rng.integers(-128, 128, (rows, cols)).astype(np.int8)
    flat = src.reshape(-1)
    every = np.arange(-128, 128).astype(np.int8)
    flat[-min(256, flat.size):] = every[-min(256, flat.size):]
    dst = poison(torch.empty((rows, cols), dtype=torch.float16, device="cuda"))
    B.tern_widen_int8(to_dev(src), rows, cols, dst)
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().float().numpy(), src.astype(np.float32))


def test_pack_layer_keeps_both_weight_forms():
    n, k = 272, 2048
    codes = I.make_codes(9, n, k)
    scales = I.make_scales(9, n, k)
    lay = B.pack_layer(to_dev(codes), to_dev(scales), decode=False, prefill=True, int8=True)
    qo, _, _ = O.decompose_scales(scales)
    w = O.w_int8(codes, qo)
    assert np.array_equal(lay.w_int8.cpu().numpy(), w.astype(np.int8))
    assert np.array_equal(lay.w_q.cpu().float().numpy(), w.astype(np.float32))
