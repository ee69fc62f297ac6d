"""Column-parallel (N-split) layers on one GPU, the ranks' local phases run in
turn: each rank's rows through the library's own calls.  Prefill (int8) is
bit-identical to the whole layer (exact integer accumulators, per-row and
per-token rescale); decode is within the decode tolerance of the oracle (the
GEMV's summation grouping depends on N)."""

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


def _ranks(codes, scales, world, expand=True):
    n = codes.shape[0]
    lins = []
    for r in range(world):
        plan = TP.nsplit_plan(n, world, r)
        lins.append(TP.NSplitLinear(plan, to_dev(codes[plan.n0:plan.n1]),
                                    to_dev(scales[plan.n0:plan.n1]), expand=expand))
    return lins


@pytest.mark.parametrize("world,n,m,expand", [(3, 1040, 200, True), (2, 5120, 300, True),
                                              (2, 5120, 100, False)])
def test_prefill_rows_equal_the_whole_layer(world, n, m, expand):
    k = 5120
    codes, scales = I.make_codes(71, n, k), I.make_scales(71, n, k)
    bits, x = I.make_activations(71, m, k, 0.001, 50.0)
    xd = to_dev_bf16(bits)
    whole = B.pack_layer(to_dev(codes), to_dev(scales), decode=True, prefill=True, expand=expand)
    want = B.forward(whole, xd)
    got = torch.cat([TP.nsplit_local(lin, xd) for lin in _ranks(codes, scales, world, expand)],
                    dim=1)
    B.tern_check()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    rows = np.sort(np.random.default_rng(3).choice(n, 128, replace=False))
    r = O.linear_int8(x, codes[rows], scales[rows])
    assert np.array_equal(bf16_to_f32(got[:, torch.from_numpy(rows).cuda()]).view(np.uint32),
                          r["y"].view(np.uint32))


@pytest.mark.parametrize("world,n,m", [(2, 34816, 4), (3, 1040, 1), (4, 5120, 16)])
def test_decode_rows_within_tolerance(world, n, m):
    k = 5120
    codes, scales = I.make_codes(72, n, k), I.make_scales(72, n, k)
    bits, x = I.make_activations(72, m, k, 0.001, 50.0)
    xd = to_dev_bf16(bits)
    lins = _ranks(codes, scales, world)
    parts = [TP.nsplit_local(lin, xd) for lin in lins]
    B.tern_check()
    for lin, y in zip(lins, parts):
        p = lin.plan
        if p.nr:
            ref = O.linear_f64(x, codes[p.n0:p.n1], scales[p.n0:p.n1])
            assert O.rel_frobenius(bf16_to_f32(y), ref) <= 4e-3
    y = bf16_to_f32(torch.cat(parts, dim=1))
    rows = np.sort(np.random.default_rng(4).choice(n, 256, replace=False))
    assert O.rel_frobenius(y[:, rows], O.linear_f64(x, codes[rows], scales[rows])) <= 4e-3
