"""Tensor parallelism of the ternary linear layer: K split (row-parallel,
below) and N split (column-parallel, at the end of the file).

Page "RTX 5070 x2 ... Ternary-Bonsai-2-27B on vLLM TP=2", section 1
("TP=2 への移植: アダマールブロックの真ん中で割れる"): a row-parallel layer's input
columns are split over the ranks, and the split can cut a 1024-wide Hadamard
block in the middle (down 17408 over two ranks: 8704 = 8.5 blocks).  With the
Sylvester structure H1024 [a; b] = [H512 a + H512 b ; H512 a - H512 b], each
rank transforms its own half with H512, the ranks exchange those halves with
one all-gather, and the rank holding the first half takes the sum while the
one holding the second half takes the difference.  The rotated activations
are then exactly those of the whole-width rotation (the stride-512 butterfly
is the last stage), and each rank multiplies its columns by its weight
columns; an all-reduce adds the ranks' partial outputs.

Host orchestration only: every step on the data runs in the library's
kernels (tern_fwht_shard, tern_fwht_combine, tern_quant_rotated, then the
GEMV or a GEMM); the exchange and the reduction are collectives of the
caller's process group.  A rank's padded layout is [lead block] [whole
blocks] [trail block]: a half block is padded with 512 zero columns (zero
weights), so the GEMV and the GEMMs run unchanged.

The forward is split into a rank-local phase and a finishing phase around the
exchange, so the same code runs under torch.distributed (one process per
rank) and, for a test on one device, with the ranks' phases called in turn.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as B

HBLOCK = 1024
HALF = 512
GROUP = 128


@dataclass(frozen=True)
class KSplitPlan:
    """Rank `rank` of `world` holds input columns [k0, k1) of a K-wide layer."""

    K: int
    world: int
    rank: int
    k0: int
    k1: int
    lead: bool     # the shard starts in the middle of a block (second half)
    trail: bool    # the shard ends in the middle of a block (first half)

    @property
    def kr(self) -> int:
        return self.k1 - self.k0

    @property
    def whole(self) -> int:
        """Number of whole 1024-blocks inside the shard."""
        return (self.kr - HALF * (self.lead + self.trail)) // HBLOCK

    @property
    def kp(self) -> int:
        """Width of the padded local layout."""
        return HBLOCK * (self.whole + self.lead + self.trail)

    @property
    def exchange(self) -> bool:
        """Whether any shard boundary of the layer cuts a block (all ranks
        then take part in the exchange)."""
        return (self.K // self.world) % HBLOCK != 0

    def padded_columns(self) -> list[tuple[int, int, int]]:
        """(padded start, shard start, length) of the shard's column runs in
        the padded layout; every other padded column is zero."""
        runs = []
        p = 0
        s = 0
        if self.lead:
            runs.append((0, 0, HALF))
            p, s = HBLOCK, HALF
        if self.whole:
            runs.append((p, s, HBLOCK * self.whole))
            p += HBLOCK * self.whole
            s += HBLOCK * self.whole
        if self.trail:
            runs.append((p, s, HALF))
        return runs


def ksplit_plan(K: int, world: int, rank: int) -> KSplitPlan:
    """Equal contiguous shards; each must be a whole number of half blocks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world size or rank")
    if K % HBLOCK or K % world or (K // world) % HALF:
        raise ValueError(f"K={K} does not split over {world} ranks at half-block boundaries")
    kr = K // world
    k0, k1 = rank * kr, (rank + 1) * kr
    return KSplitPlan(K, world, rank, k0, k1, k0 % HBLOCK != 0, k1 % HBLOCK != 0)


def pad_shard(plan: KSplitPlan, codes: torch.Tensor, scales: torch.Tensor):
    """The rank's weight columns (codes int8 [N, kr], fp16 scales [N, kr/128])
    in its padded layout: zero codes and zero scales in the padding."""
    n = codes.shape[0]
    if codes.shape[1] != plan.kr or scales.shape[1] != plan.kr // GROUP:
        raise ValueError("shard columns do not match the plan")
    cp = torch.zeros((n, plan.kp), dtype=codes.dtype, device=codes.device)
    sp = torch.zeros((n, plan.kp // GROUP), dtype=scales.dtype, device=scales.device)
    for p, s, ln in plan.padded_columns():
        cp[:, p:p + ln] = codes[:, s:s + ln]
        sp[:, p // GROUP:(p + ln) // GROUP] = scales[:, s // GROUP:(s + ln) // GROUP]
    return cp.contiguous(), sp.contiguous()


class KSplitLinear:
    """One rank's part of a K-split ternary linear layer, packed for decode
    and/or prefill (see binding.pack_layer) in the padded layout.  With
    pack=False the padded codes and scales are kept unpacked instead (for a
    reference implementation of the ops)."""

    def __init__(self, plan: KSplitPlan, codes: torch.Tensor, scales: torch.Tensor,
                 decode: bool = True, prefill: bool = True, expand: bool = True,
                 pack: bool = True):
        self.plan = plan
        self.n = codes.shape[0]
        cp, sp = pad_shard(plan, codes, scales)
        self.layer = None
        self.codes_padded = self.scales_padded = None
        if pack:
            self.layer = B.pack_layer(cp, sp, decode=decode, prefill=prefill, expand=expand)
        else:
            self.codes_padded, self.scales_padded = cp, sp


class GpuOps:
    """The library calls of the K-split forward (CUDA tensors)."""

    def shard_rotate(self, plan: KSplitPlan, x: torch.Tensor, sign=None):
        m = x.shape[0]
        xr = torch.empty((m, plan.kp), dtype=torch.float32, device=x.device)
        h = torch.zeros((2, m, HALF), dtype=torch.float32, device=x.device)
        B.tern_fwht_shard(x, m, plan.kr, plan.lead, plan.trail, sign, xr,
                          h[0] if plan.lead else None, h[1] if plan.trail else None)
        return xr, h

    def combine(self, h_first, h_second, part: int, xr: torch.Tensor, blk: int):
        B.tern_fwht_combine(h_first.contiguous(), h_second.contiguous(), xr.shape[0], part, xr,
                            xr.shape[1], blk)

    def decode(self, lin: KSplitLinear, xr: torch.Tensor, ws: B.Workspace) -> torch.Tensor:
        m, kp = xr.shape
        xh = torch.empty((m, kp), dtype=torch.float16, device=xr.device)
        xs = B.decode_aux(kp, xr.device)
        B.tern_quant_rotated(xr, m, kp, B.TERN_FWHT_DECODE, xh, xs)
        y = torch.empty((m, lin.n), dtype=torch.bfloat16, device=xr.device)
        nb = B.tern_workspace_bytes(B.TERN_OP_GEMV, m, lin.n, kp)
        buf = ws.get(nb)
        B.tern_gemv_decode(lin.layer.packed, xh, xs, m, lin.n, kp, y, buf, buf.numel())
        return y

    def prefill(self, lin: KSplitLinear, xr: torch.Tensor, ws: B.Workspace) -> torch.Tensor:
        m, kp = xr.shape
        xq = torch.empty((m, kp), dtype=torch.float16, device=xr.device)
        ts = torch.empty(m, dtype=torch.float32, device=xr.device)
        B.tern_quant_rotated(xr, m, kp, B.TERN_FWHT_I8H, xq, ts)
        y = torch.empty((m, lin.n), dtype=torch.bfloat16, device=xr.device)
        lay = lin.layer
        if lay.w_q is not None:
            nb = B.tern_workspace_bytes(B.TERN_OP_GEMM, m, lin.n, kp)
            buf = ws.scratch(nb) if nb else None
            B.tern_gemm_prefill_int8h(xq, ts, lay.w_q, lay.rscale, m, lin.n, kp, y, None, buf, nb)
        else:
            nb = B.tern_workspace_bytes(B.TERN_OP_GEMM_PACKED, m, lin.n, kp)
            buf = ws.scratch(nb) if nb else None
            B.tern_gemm_prefill_packed(xq, ts, lay.packed, lay.q, lay.rscale, m, lin.n, kp, y,
                                       None, buf, nb)
        return y


def local_phase(lin: KSplitLinear, x: torch.Tensor, sign=None, ops=None):
    """Rank-local step: rotate the whole blocks and transform the half
    blocks.  Returns (xr in the padded layout, h [2, M, 512]: the leading
    and trailing halves' H512, zero where absent) -- h is what the ranks
    exchange."""
    ops = ops or GpuOps()
    return ops.shard_rotate(lin.plan, x, sign)


def finish_phase(lin: KSplitLinear, xr, h_all, mode: str = "decode", ops=None, ws=None):
    """After the exchange (h_all[r] = rank r's h): combine this rank's half
    blocks -- the first-half rank takes the sum, the second-half rank the
    difference -- then quantise and multiply.  Returns this rank's partial
    output [M, N]."""
    ops = ops or GpuOps()
    plan = lin.plan
    r = plan.rank
    if plan.lead:   # second half of the block shared with rank r - 1
        ops.combine(h_all[r - 1][1], h_all[r][0], 1, xr, 0)
    if plan.trail:  # first half of the block shared with rank r + 1
        ops.combine(h_all[r][1], h_all[r + 1][0], 0, xr, plan.kp // HBLOCK - 1)
    ws = ws or B.Workspace(xr.device)
    if mode == "decode":
        return ops.decode(lin, xr, ws)
    if mode == "prefill":
        return ops.prefill(lin, xr, ws)
    raise ValueError(mode)


def forward(lin: KSplitLinear, x: torch.Tensor, group=None, mode: str = "decode", sign=None,
            ops=None, ws=None) -> torch.Tensor:
    """The K-split forward on one rank of a torch.distributed process group:
    local phase, all-gather of the half-block transforms (only when some
    shard boundary cuts a block), finishing phase, all-reduce (sum) of the
    partial outputs.  x: this rank's input columns [M, kr] (bf16)."""
    import torch.distributed as dist
    xr, h = local_phase(lin, x, sign, ops)
    world = lin.plan.world
    if lin.plan.exchange:
        h_all = [torch.empty_like(h) for _ in range(world)]
        dist.all_gather(h_all, h.contiguous(), group=group)
    else:
        h_all = [h] * world
    y = finish_phase(lin, xr, h_all, mode, ops, ws)
    dist.all_reduce(y, group=group)
    return y


# ---------------------------------------------------------------------------
# Column-parallel (N-split): each rank holds a contiguous block of output
# rows.  Every rank rotates the whole input and computes its own rows with
# the layer's usual calls, so the data path has no collective; one optional
# all-gather joins the rows.

@dataclass(frozen=True)
class NSplitPlan:
    """Rank `rank` of `world` holds output rows [n0, n1) of an N-row layer;
    every rank's block starts at a multiple of `per` rows."""

    N: int
    world: int
    rank: int
    per: int
    n0: int
    n1: int

    @property
    def nr(self) -> int:
        return self.n1 - self.n0


def nsplit_plan(N: int, world: int, rank: int, align: int = 16) -> NSplitPlan:
    """Blocks of ceil(N / world) rows rounded up to `align` (the GEMMs take
    N % 16 == 0); the last ranks take what is left, possibly nothing."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world size or rank")
    if N % align:
        raise ValueError(f"N={N} is not a multiple of {align}")
    per = -(-N // world)
    per = -(-per // align) * align
    n0 = min(rank * per, N)
    return NSplitPlan(N, world, rank, per, n0, min(n0 + per, N))


class NSplitLinear:
    """One rank's rows of a column-parallel ternary linear layer: codes int8
    [nr, K] and scales fp16 [nr, K/128] of rows [n0, n1), packed like any
    layer (binding.pack_layer); with pack=False they are kept as given (for
    a reference implementation of the compute)."""

    def __init__(self, plan: NSplitPlan, codes: torch.Tensor, scales: torch.Tensor,
                 decode: bool = True, prefill: bool = True, expand: bool = True,
                 pack: bool = True):
        if codes.shape[0] != plan.nr or scales.shape[0] != plan.nr:
            raise ValueError("shard rows do not match the plan")
        self.plan = plan
        self.layer = None
        self.codes = self.scales = None
        if pack and plan.nr:
            self.layer = B.pack_layer(codes.contiguous(), scales.contiguous(), decode=decode,
                                      prefill=prefill, expand=expand)
        elif not pack:
            self.codes, self.scales = codes, scales


def nsplit_local(lin: NSplitLinear, x: torch.Tensor, sign=None, ws=None) -> torch.Tensor:
    """This rank's columns of y, [M, nr]: the layer's own forward (rotation of
    the whole input included) on the rank's rows."""
    if lin.plan.nr == 0:
        return torch.empty((x.shape[0], 0), dtype=torch.bfloat16, device=x.device)
    return B.forward(lin.layer, x, ws=ws, sign=sign)


def nsplit_forward(lin: NSplitLinear, x: torch.Tensor, group=None, gather: bool = True,
                   sign=None, ws=None, local=None) -> torch.Tensor:
    """The column-parallel forward on one rank of a torch.distributed process
    group: the rank's columns of y, and with `gather` all of y [M, N] in rank
    order (one all-gather of the blocks, padded to `per` columns so that
    every rank sends the same size).  `local` replaces nsplit_local (for a
    reference implementation of the compute)."""
    import torch.distributed as dist
    y = (local or nsplit_local)(lin, x, sign=sign, ws=ws)
    if not gather:
        return y
    plan = lin.plan
    ypad = torch.zeros((x.shape[0], plan.per), dtype=y.dtype, device=y.device)
    ypad[:, :plan.nr] = y
    parts = [torch.empty_like(ypad) for _ in range(plan.world)]
    dist.all_gather(parts, ypad, group=group)
    return torch.cat(parts, dim=1)[:, :plan.N]
