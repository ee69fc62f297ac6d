"""Column-parallel (N-split) tensor parallelism on CPU ranks.

The product's host orchestration (ternary_weight_linear_block_gb300.tp: the
row plan, the padded all-gather in rank order) runs on gloo ranks, with each
rank's compute replaced by the oracle (test code).  The gathered output
equals the whole layer's: bit for bit on the int8 path, whose integer
accumulators do not depend on how the rows are grouped.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import tern_oracle as O
from ternary_weight_linear_block_gb300 import inputs as I
from ternary_weight_linear_block_gb300 import tp as TP


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _layer(n, k, m):
    return I.make_codes(70, n, k), I.make_scales(70, n, k), I.make_activations(70, m, k, 0.001, 50.0)[1]


def _oracle_local(lin, x, sign=None, ws=None):
    """The int8 path of the rank's rows, by the oracle."""
    if lin.plan.nr == 0:
        return torch.empty((x.shape[0], 0), dtype=torch.float32)
    return torch.from_numpy(O.linear_int8(x.numpy(), lin.codes.numpy(), lin.scales.numpy())["y"])


def _worker(rank, world, port, n, k, m, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        codes, scales, x = _layer(n, k, m)
        plan = TP.nsplit_plan(n, world, rank)
        lin = TP.NSplitLinear(plan, torch.from_numpy(codes[plan.n0:plan.n1].copy()),
                              torch.from_numpy(scales[plan.n0:plan.n1].copy()), pack=False)
        xt = torch.from_numpy(x)
        y_all = TP.nsplit_forward(lin, xt, local=_oracle_local).numpy()
        y_own = TP.nsplit_forward(lin, xt, gather=False, local=_oracle_local).numpy()
        q.put((rank, y_all, y_own, (plan.n0, plan.n1)))
    except Exception:                      # report at once instead of timing out
        import traceback
        q.put((rank, traceback.format_exc(), None, None))
        raise
    finally:
        dist.destroy_process_group()


def _run(world, n, k, m):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n, k, m, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = []
    for _ in procs:
        r = q.get(timeout=300)
        assert not isinstance(r[1], str), r[1]
        res.append(r)
    res.sort(key=lambda t: t[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return res


def test_plan():
    assert [(p.n0, p.n1) for p in (TP.nsplit_plan(1040, 3, r) for r in range(3))] == \
        [(0, 352), (352, 704), (704, 1040)]
    assert [(p.n0, p.n1) for p in (TP.nsplit_plan(16, 3, r) for r in range(3))] == \
        [(0, 16), (16, 16), (16, 16)]
    for n, w in ((34816, 2), (5120, 4), (10240, 8), (1040, 3)):
        plans = [TP.nsplit_plan(n, w, r) for r in range(w)]
        assert plans[0].n0 == 0 and plans[-1].n1 == n
        assert all(a.n1 == b.n0 for a, b in zip(plans, plans[1:]))
        assert all(p.n0 % 16 == 0 for p in plans)
    with pytest.raises(ValueError):
        TP.nsplit_plan(1000, 2, 0)
    with pytest.raises(ValueError):
        TP.nsplit_plan(1024, 2, 2)


@pytest.mark.parametrize("world,n", [(2, 1024), (3, 1040), (3, 16)])
def test_gathered_rows_equal_the_whole_layer(world, n):
    k, m = 2048, 5
    codes, scales, x = _layer(n, k, m)
    want = O.linear_int8(x, codes, scales)["y"]
    res = _run(world, n, k, m)
    for rank, y_all, y_own, (n0, n1) in res:
        assert np.array_equal(y_all.view(np.uint32), want.view(np.uint32))
        assert np.array_equal(y_own.view(np.uint32), want[:, n0:n1].view(np.uint32))
