"""The allocation-free decode GEMV entry point (tern_gemv_decode_noalloc).

It exists for callers that cannot allocate device memory: an application
that owns all device memory through its own pool and hands the layer only its
inputs and outputs, or a decode loop that must not stall on cudaMalloc.  It
runs the same GEMV with its scratch in a fixed array inside the library.
Its output must match tern_gemv_decode (caller workspace) on two calls in a
row (the second call sees the array exactly as the first one left it).
Collected last so a failure here leaves every other test already run.
"""

import numpy as np
import pytest
import torch

from oracle import tern_oracle as O
from ternary_weight_linear_block_gb300 import binding as B
from ternary_weight_linear_block_gb300 import inputs as I
from tests.gpu_helpers import bf16_to_f32, ensure_lib, poison, to_dev, to_dev_bf16

TOL = 4e-3   # the decode tolerance used by the GEMV parity tests


def _compare(codes, scales, x_bits, m, n, k):
    """Two allocation-free calls in a row against the workspace call; returns
    the workspace call's output."""
    lay = B.pack_layer(to_dev(codes), to_dev(scales), decode=True, prefill=False)
    xh, xs = B.fwht(to_dev_bf16(x_bits), B.TERN_FWHT_DECODE)
    y_ref = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
    ws = B.Workspace()
    buf = ws.get(B.tern_workspace_bytes(B.TERN_OP_GEMV, m, n, k))
    B.tern_gemv_decode(lay.packed, xh, xs, m, n, k, y_ref, buf, buf.numel())
    torch.cuda.synchronize()
    ref = bf16_to_f32(y_ref)
    for _ in range(2):
        y = poison(torch.empty((m, n), dtype=torch.bfloat16, device="cuda"))
        B.tern_gemv_decode_noalloc(lay.packed, xh, xs, m, n, k, y)
        B.tern_check()
        got = bf16_to_f32(y)
        assert np.isfinite(got).all()
        assert O.rel_frobenius(got, ref) <= TOL
        assert np.array_equal(got, ref)          # same kernel and split: identical
    return ref


@pytest.mark.gpu
@pytest.mark.parametrize("layer,m", [(I.QKV, 4), (I.DOWN, 16), (I.TINY, 1), (I.GATE_UP, 16)])
def test_noalloc_matches_workspace_entry_point(layer, m):
    ensure_lib()
    n, k = layer.n, layer.k
    assert B.tern_workspace_bytes(B.TERN_OP_GEMV, m, n, k) <= B.TERN_NOALLOC_SCRATCH_BYTES
    d = I.make_layer(layer, m, seed=5)
    ref = _compare(d.codes, d.scales, d.x_bits, m, n, k)
    rows = np.random.default_rng(0).choice(n, 128, replace=False)
    exact = O.linear_f64(d.x, d.codes[rows], d.scales[rows])
    assert O.rel_frobenius(ref[:, rows], exact) <= TOL


@pytest.mark.gpu
def test_noalloc_limit_boundary():
    """Growing the row count in steps of 512 (K = 5120, M = 16): the last
    count whose scratch fits the array before the first one that does not
    runs and matches the workspace call; that next one is rejected with
    TERN_ERR_WORKSPACE before anything is launched."""
    ensure_lib()
    k, m = 5120, 16
    n = 512
    while B.tern_workspace_bytes(B.TERN_OP_GEMV, m, n + 512, k) <= B.TERN_NOALLOC_SCRATCH_BYTES:
        n += 512
    assert B.tern_workspace_bytes(B.TERN_OP_GEMV, m, n, k) <= B.TERN_NOALLOC_SCRATCH_BYTES
    assert n >= I.GATE_UP.n
    codes = I.make_codes(6, n, k)
    scales = I.make_scales(6, n, k)
    bits, _ = I.make_activations(6, m, k, 0.001, 50.0)
    _compare(codes, scales, bits, m, n, k)
    over = n + 512
    assert B.tern_workspace_bytes(B.TERN_OP_GEMV, m, over, k) > B.TERN_NOALLOC_SCRATCH_BYTES
    fake = 1 << 20                                  # aligned, never dereferenced
    st = B.lib().tern_gemv_decode_noalloc(fake, fake, fake, m, over, k, fake, None)
    assert st == B.TERN_ERR_WORKSPACE
