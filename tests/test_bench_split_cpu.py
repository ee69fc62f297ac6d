"""The split-layer bench path (bench.py --split n|k) on CPU ranks.

bench.split_shard / split_forward are the host side of the tensor-parallel
decode measurement: each rank builds its shard of the same layer and runs the
column-parallel (one all-gather) or row-parallel (half-block all-gather +
all-reduce) forward through torch.distributed.  Here they run on gloo ranks
(world sizes 2 and 3) with the library's kernels replaced by the oracle (test
code), and every rank's result must equal the whole layer: exactly for the
row split (each output row is computed whole on one rank), within the decode
tolerance for the K split (partial sums over column shards).
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


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _oracle_rows(lin, x, sign=None, ws=None):
    """The decode of the rank's rows, by the oracle (fp64)."""
    if lin.plan.nr == 0:
        return torch.empty((x.shape[0], 0), dtype=torch.float64)
    return torch.from_numpy(O.linear_f64(x.numpy(), lin.codes.numpy(), lin.scales.numpy()))


def _worker(rank, world, port, split, n, k, m, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from tests.test_ksplit_cpu import OracleOps
        codes = torch.from_numpy(I.make_codes(90, n, k))
        scales = torch.from_numpy(I.make_scales(90, n, k))
        _, x = I.make_activations(90, m, k, 0.001, 50.0)
        layer = I.Layer("test", k, n, 0.001, 50.0)
        lin = bench.split_shard(split, layer, world, rank, codes, scales, pack=False)
        y = bench.split_forward(split, lin, torch.from_numpy(x), world, ops=OracleOps(),
                                local=_oracle_rows)
        q.put((rank, y.double().numpy(), None))
    except Exception:                      # report at once instead of timing out
        import traceback
        q.put((rank, None, traceback.format_exc()))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("split,world", [("n", 2), ("n", 3), ("k", 2), ("k", 3)])
def test_split_bench_path_matches_whole_layer(split, world):
    n, k, m = 1040, 3072, 4                # k: 1.5 blocks per rank at world 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, split, n, k, m, q))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=120)
    for _, _, err in res:
        assert err is None, err
    for p in procs:
        assert p.exitcode == 0
    codes = I.make_codes(90, n, k)
    scales = I.make_scales(90, n, k)
    _, x = I.make_activations(90, m, k, 0.001, 50.0)
    exact = O.linear_f64(x, codes, scales)
    for _, y, _ in res:
        assert y.shape == (m, n)
        if split == "n":
            assert np.array_equal(y, exact)
        else:
            assert O.rel_frobenius(y, exact) <= 4e-3
    for _, y, _ in res[1:]:
        assert np.array_equal(y, res[0][1])     # every rank holds the same result


def test_split_value_is_strong_scaling():
    import bench
    # whole-layer bytes per step over the slowest rank's time, whatever the rank count
    assert bench.split_value(2_000_000_000, 10, 2.0) == pytest.approx(10.0)
