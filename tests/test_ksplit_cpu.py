"""K-split tensor parallelism (the page's section 1) on CPU ranks.

The product's host orchestration (ternary_weight_linear_block_gb300.tp: the
plan, the padded weight layout, which rank combines which halves with which
sign, the all-gather and the all-reduce) runs on two gloo ranks, with the
library's kernels replaced by the oracle's steps (OracleOps below, test code).
Checks: each rank's rotated columns equal the whole-width rotation bit for
bit; the all-reduced output matches the whole-width layer within the decode
and int8 tolerances; swapping the ranks' sum and difference is caught.
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


class OracleOps:
    """The kernels' steps, computed by the oracle on CPU tensors."""

    def __init__(self, swap=False):
        self.swap = swap

    def shard_rotate(self, plan, x, sign=None):
        xf = x.float().numpy()
        if sign is not None:
            xf = xf * sign.float().numpy()[None, :]
        m = xf.shape[0]
        xr = np.zeros((m, plan.kp), np.float32)
        h = np.zeros((2, m, 512), np.float32)
        if plan.lead:
            h[0] = O.fwht_half_f32(xf[:, :512])
        if plan.whole:
            a = 512 * plan.lead
            xr[:, 1024 * plan.lead:1024 * (plan.lead + plan.whole)] = O.fwht_f32(
                xf[:, a:a + 1024 * plan.whole])
        if plan.trail:
            h[1] = O.fwht_half_f32(xf[:, plan.kr - 512:])
        return torch.from_numpy(xr), torch.from_numpy(h)

    def combine(self, h_first, h_second, part, xr, blk):
        part = 1 - part if self.swap else part
        v = O.ksplit_combine(h_first.numpy(), h_second.numpy(), part)
        xr[:, 1024 * blk:1024 * blk + 512] = torch.from_numpy(v)
        xr[:, 1024 * blk + 512:1024 * (blk + 1)] = 0

    def decode(self, lin, xr, ws):
        xh, inv = O.f16_operand(xr.numpy())
        kp = xr.shape[1]
        x_eff = (xh.astype(np.float64).reshape(-1, kp // 1024, 1024) *
                 inv.astype(np.float64)[:, :, None]).reshape(-1, kp)
        w = O.dequant_f64(lin.codes_padded.numpy(), lin.scales_padded.numpy())
        return torch.from_numpy((x_eff @ w.T).astype(np.float32))

    def prefill(self, lin, xr, ws):
        xq, ts = O.quant_tokens(xr.numpy())
        q, rs, _ = O.decompose_scales(lin.scales_padded.numpy())
        acc = O.acc_int8(xq, O.w_int8(lin.codes_padded.numpy(), q))
        return torch.from_numpy(O.y_int8(acc, ts, rs))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _layer(k, n, m):
    codes = I.make_codes(50, n, k)
    scales = I.make_scales(50, n, k)
    bits, x = I.make_activations(50, m, k, 0.001, 50.0)
    return codes, scales, bits, x


def _worker(rank, world, port, k, n, m, swap, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        _body(rank, world, k, n, m, swap, q)
    except Exception:                      # report at once instead of timing out
        import traceback
        q.put((rank, traceback.format_exc(), None, None))
        raise
    finally:
        dist.destroy_process_group()


def _body(rank, world, k, n, m, swap, q):
    codes, scales, bits, x = _layer(k, n, m)
    plan = TP.ksplit_plan(k, world, rank)
    cr = torch.from_numpy(codes[:, plan.k0:plan.k1].copy())
    sr = torch.from_numpy(scales[:, plan.k0 // 128:plan.k1 // 128].copy())
    lin = TP.KSplitLinear(plan, cr, sr, pack=False)
    xb = torch.from_numpy(np.ascontiguousarray(bits[:, plan.k0:plan.k1]).view(np.int16)
                          ).view(torch.bfloat16)
    ops = OracleOps(swap)
    # rotated columns (exchange included), back in the shard's own order
    xr, h = TP.local_phase(lin, xb, ops=ops)
    h_all = [torch.empty_like(h) for _ in range(world)]
    dist.all_gather(h_all, h)
    TP.finish_phase(lin, xr, h_all, "decode", ops)   # fills the half blocks of xr
    cols = np.concatenate([xr.numpy()[:, p:p + ln] for p, s, ln in plan.padded_columns()],
                          axis=1)
    y_dec = TP.forward(lin, xb, mode="decode", ops=ops).numpy()
    y_pre = TP.forward(lin, xb, mode="prefill", ops=ops).numpy()
    q.put((rank, cols, y_dec, y_pre))


def _run(world, k, n, m, swap=False):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, k, n, m, swap, q))
             for r in range(world)]
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


def test_plan_and_padded_layout():
    p0 = TP.ksplit_plan(17408, 2, 0)
    p1 = TP.ksplit_plan(17408, 2, 1)
    assert (p0.k0, p0.k1, p0.lead, p0.trail, p0.whole, p0.kp) == (0, 8704, False, True, 8, 9216)
    assert (p1.k0, p1.k1, p1.lead, p1.trail, p1.whole, p1.kp) == (8704, 17408, True, False, 8, 9216)
    assert p0.padded_columns() == [(0, 0, 8192), (8192, 8192, 512)]
    assert p1.padded_columns() == [(0, 0, 512), (1024, 512, 8192)]
    mid = TP.ksplit_plan(4608 * 2, 3, 1)            # 3072 columns: lead + 2 whole + trail? no:
    assert (mid.k0 % 1024, mid.k1 % 1024) == (0, 0) and not mid.exchange
    p = TP.ksplit_plan(6144, 4, 1)                  # 1536: starts mid-block, ends on a boundary
    assert (p.lead, p.trail, p.whole, p.kp) == (True, False, 1, 2048)
    p = TP.ksplit_plan(6144, 4, 2)                  # [3072, 4608): whole block + trail half
    assert (p.lead, p.trail, p.whole, p.kp) == (False, True, 1, 2048)
    for bad in ((17408, 4, 0), (5120, 3, 0), (1000, 1, 0)):
        with pytest.raises(ValueError):
            TP.ksplit_plan(*bad)
    # padding: the shard's columns land in their runs, zeros elsewhere
    codes = torch.arange(1, 8705, dtype=torch.int32).remainder(3).sub(1).to(torch.int8)
    codes = codes[None, :].repeat(2, 1)
    scales = torch.arange(68, dtype=torch.float16)[None, :].repeat(2, 1) + 1
    cp, sp = TP.pad_shard(p1, codes, scales)
    assert torch.equal(cp[:, :512], codes[:, :512]) and not cp[:, 512:1024].any()
    assert torch.equal(cp[:, 1024:], codes[:, 512:])
    assert torch.equal(sp[:, :4], scales[:, :4]) and not sp[:, 4:8].any()
    assert torch.equal(sp[:, 8:], scales[:, 4:])


@pytest.mark.parametrize("world,k", [(2, 17408), (2, 3072), (4, 6144)])
def test_two_and_four_ranks_match_whole_width(world, k):
    n, m = 64, 3
    res = _run(world, k, n, m)
    codes, scales, bits, x = _layer(k, n, m)
    cols = np.concatenate([r[1] for r in res], axis=1)
    assert np.array_equal(cols.view(np.uint32), O.fwht_f32(x).view(np.uint32))
    exact = O.linear_f64(x, codes, scales)
    for _, _, y_dec, y_pre in res:                   # every rank holds the reduced output
        assert O.rel_frobenius(y_dec, exact) <= 4e-3
        assert O.rel_frobenius(y_pre, exact) <= 2e-2


def test_swapped_sum_and_difference_is_caught():
    n, m, k = 64, 3, 17408
    res = _run(2, k, n, m, swap=True)
    codes, scales, bits, x = _layer(k, n, m)
    exact = O.linear_f64(x, codes, scales)
    err = O.rel_frobenius(res[0][2], exact)
    assert err > 0.05
