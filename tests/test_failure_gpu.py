"""The failure path of the bounded device-side waits, exercised without a GPU
fault: tern_selftest_wait runs one warp that waits, with the kernels' own
wait helper, on a barrier nothing completes.  The wait gives up after its
poll limit, the next tern_check reports TERN_ERR_TIMEOUT once, and the
context stays usable for the layer's own calls."""

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


def _timed_selftest(polls: int) -> float:
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    B.tern_selftest_wait(polls)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


@pytest.mark.parametrize("polls", [1, 64, 4096])
def test_wait_gives_up_and_is_reported_once(polls):
    B.tern_check()                          # nothing pending
    t = _timed_selftest(polls)
    assert t < 10.0                         # the wait is bounded
    with pytest.raises(B.TernError) as ei:
        B.tern_check()
    assert ei.value.status == B.TERN_ERR_TIMEOUT
    B.tern_check()                          # read and cleared: OK again


def test_context_usable_after_a_timeout():
    """After a wait gave up, decode and prefill calls still run and match
    the oracle, and tern_check is clean."""
    B.tern_selftest_wait(64)
    with pytest.raises(B.TernError):
        B.tern_check()
    d = I.make_layer(I.TINY, 8, seed=0)
    layer = B.pack_layer(to_dev(d.codes), to_dev(d.scales), decode=True, prefill=True)
    x = to_dev_bf16(d.x_bits)
    y = poison(torch.empty((8, layer.n), dtype=torch.bfloat16, device="cuda"))
    B.decode(layer, x, B.Workspace(), y=y)
    acc = poison(torch.empty((8, layer.n), dtype=torch.int32, device="cuda"))
    yp = poison(torch.empty((8, layer.n), dtype=torch.bfloat16, device="cuda"))
    B.prefill(layer, x, y=yp, acc=acc)
    B.tern_check()
    ref = O.linear_f64(d.x, d.codes, d.scales)
    assert O.rel_frobenius(bf16_to_f32(y), ref) <= 4e-3
    r = O.linear_int8(d.x, d.codes, d.scales)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), r["acc"])
