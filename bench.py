"""Benchmark of the ternary-weight linear layer on GB300.

Workload (default): decode through the fused gate/up projection,
K = 5120 -> N = 34816, one batch of M = 1 and one of M = 4 tokens per step.
A step is one pass of the decode hot path for each batch: the block-Hadamard
rotation into the fp16 decode operand, then the 2-bit GEMV.  Weights rotate
through independent synthetic copies totalling more than 4x L2 (129 MB), so
every step streams its weights from HBM.  Metric: decode weight GB/s =
(2-bit code bytes + fp16 scale bytes) per step / step time.

The JSON line also carries the prefill int8 path (M = 2048 through the same
layer) as its own object, the roofline of the dominant kernel, the end-to-end
number through the public API with host buffers, clocks sampled during the
timed region, and the CPU oracle timed on a bounded sample.

Multi-GPU (torchrun): every rank runs the same per-GPU workload on its own
weights (independent layers, no collective in the data path; weak scaling);
value = bytes processed by all ranks / max time over ranks.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from ternary_weight_linear_block_gb300 import binding as B  # noqa: E402
from ternary_weight_linear_block_gb300 import inputs as I  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
METRIC = "ternary linear: decode weight GB/s (% HBM peak); prefill int8 TOPS (% peak)"
DECODE_MS = (1, 4)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------- distributed

def _dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, ws, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v: float, ws: int) -> float:
    """The slowest rank's time (every rank gets it)."""
    if ws <= 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank: int) -> int:
    """Each rank streams its own weights (independent layers): weak scaling."""
    return 1000 * rank


def aggregate_value(bytes_per_step: int, steps: int, ws: int, t_max: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
    return bytes_per_step * steps * ws / t_max / 1e9


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        # "under load": samples within 80% of the highest seen
        hi = max(sm)
        loaded = [v for v in sm if v >= 0.8 * hi] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workload

def _make_layers(layer: I.Layer, copies: int, seed: int, prefill: bool):
    """Synthetic weights drawn on the device (seeded), packed by tern_pack."""
    g = torch.Generator(device="cuda")
    out = []
    for c in range(copies):
        g.manual_seed(seed * 1000 + c)
        codes = (torch.randint(0, 3, (layer.n, layer.k), dtype=torch.int8, device="cuda",
                               generator=g) - 1).to(torch.int8)
        scales = (0.02 * torch.randn((layer.n, layer.k // 128), device="cuda", generator=g).abs()
                  + 1e-3).to(torch.float16)
        out.append(B.pack_layer(codes, scales, decode=True, prefill=prefill))
        del codes, scales
    torch.cuda.synchronize()
    return out


def _activations(layer: I.Layer, m: int, seed: int) -> torch.Tensor:
    bits, _ = I.make_activations(seed, m, layer.k, layer.outlier_frac, layer.outlier_mult)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


class DecodeRunner:
    """Preallocated buffers for the decode step over a rotation of layers."""

    def __init__(self, layers, xs_host, stream):
        self.layers = layers
        self.stream = stream
        self.n, self.k = layers[0].n, layers[0].k
        self.ms = [x.shape[0] for x in xs_host]
        self.x = [x.cuda() for x in xs_host]
        self.xh = [torch.empty((m, self.k), dtype=torch.float16, device="cuda") for m in self.ms]
        self.xs = [B.decode_aux(self.k) for m in self.ms]
        self.y = [torch.empty((m, self.n), dtype=torch.bfloat16, device="cuda") for m in self.ms]
        self.ws = []
        for m in self.ms:
            nb = max(B.tern_workspace_bytes(B.TERN_OP_GEMV, m, self.n, self.k), 256)
            w = torch.empty(nb, dtype=torch.uint8, device="cuda")
            B.tern_workspace_init(w, nb, stream)
            self.ws.append(w)
        self.i = 0

    def step(self):
        """One decode pass per batch; each batch streams the next weight copy.
        The batches are independent, so their rotations are issued first and
        overlap each other; then the GEMVs run back to back."""
        st = self.stream.cuda_stream
        for b, m in enumerate(self.ms):
            B.tern_fwht_quant(self.x[b], m, self.k, None, B.TERN_FWHT_DECODE, self.xh[b],
                              self.xs[b], st)
        for b, m in enumerate(self.ms):
            layer = self.layers[self.i % len(self.layers)]
            self.i += 1
            B.tern_gemv_decode(layer.packed, self.xh[b], self.xs[b], m, self.n, self.k, self.y[b],
                               self.ws[b], self.ws[b].numel(), st)

    def step_fused(self):
        """The same decode pass with the rotation folded into the GEMV
        (tern_linear_decode, one launch per batch)."""
        st = self.stream.cuda_stream
        for b, m in enumerate(self.ms):
            layer = self.layers[self.i % len(self.layers)]
            self.i += 1
            B.tern_linear_decode(self.x[b], None, layer.packed, m, self.n, self.k, self.y[b],
                                 self.ws[b], self.ws[b].numel(), st)

    def gemv_only(self, b):
        st = self.stream.cuda_stream
        m = self.ms[b]
        layer = self.layers[self.i % len(self.layers)]
        self.i += 1
        B.tern_gemv_decode(layer.packed, self.xh[b], self.xs[b], m, self.n, self.k, self.y[b],
                           self.ws[b], self.ws[b].numel(), st)

    def launches_per_step(self):
        # per batch: the rotation kernel, then the GEMV (and its fixup kernel
        # at shapes where a row block is shared by many CTAs)
        return sum(1 + B.tern_kernel_launches(B.TERN_OP_GEMV, m, self.n, self.k)
                   for m in self.ms)

    def bytes_per_step(self):
        return sum(self.layers[0].weight_bytes for _ in self.ms)


def _time_region(fn, steps, stream, ws, lead_cycles=2_000_000):
    """Device time of `steps` calls of fn on `stream` (CUDA events on that
    stream, a barrier and a synchronisation on both sides).  A short device
    spin (about 1 ms) is queued before the first event, so the host has
    enqueued the first launches when the timed region starts: the region
    measures the GPU, not the host's launch rate (the end-to-end figure
    covers the host)."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    _barrier(ws)
    torch.cuda.synchronize()
    if lead_cycles:
        with torch.cuda.stream(stream):
            torch.cuda._sleep(lead_cycles)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    _barrier(ws)
    return e0.elapsed_time(e1) / 1e3   # seconds


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the timed kernels at the bench's shapes, from one ncu capture on GB300 of
# the current kernels; they change only when a kernel changes.
TRAFFIC_GEMV_GATEUP_M4 = 47_464_192 + 2_048           # gemv_kernel<1>, 5120 -> 34816, M = 4
TRAFFIC_GEMM_I8_GATEUP_M2048 = 402_740_992 + 130_555_392   # gemm_i8_kernel (CTA pairs, last wave split), M = 2048


def _gemv_algorithmic_bytes(m, n, k):
    """Bytes one GEMV launch must move: codes + scales + the fp16 activation
    operand + its 192-byte group records + bf16 output."""
    return n * k // 4 + n * (k // 128) * 2 + 2 * m * k + (k // 128) * 192 + m * n * 2


def run_decode(args, rank, ws, local):
    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    layer = I.GATE_UP
    per_copy = B.tern_packed_bytes(layer.n, layer.k)
    copies = max(4, int(np.ceil(4 * L2_BYTES / per_copy)) + 1)
    hbm_peak, tc_peak, peak_kind = _peaks()
    with torch.cuda.stream(stream):
        layers = _make_layers(layer, copies, seed=rank_seed(rank), prefill=False)
        xs_host = [_activations(layer, m, seed=rank * 10 + m) for m in DECODE_MS]
        run = DecodeRunner(layers, xs_host, stream)
        for _ in range(args.warmup):
            run.step()
        torch.cuda.synchronize()

        with ClockSampler(local) as clk:
            t = _time_region(run.step, args.steps, stream, ws)
        clocks = clk.summary()
        t = _max_over_ranks(t, ws)

        # dominant kernel alone (same launch configuration), M = 4 batch
        kb = DECODE_MS.index(4) if 4 in DECODE_MS else 0
        kernel_launches = max(200, args.steps)
        tk = _time_region(lambda: run.gemv_only(kb), kernel_launches, stream, 1)
        gemv_us = tk / kernel_launches * 1e6
        # the fused path (rotation inside the GEMV), same steps
        for _ in range(args.warmup):
            run.step_fused()
        fused_steps = max(200, args.steps)
        tf = _time_region(run.step_fused, fused_steps, stream, 1)

        # end to end through the public API (B.DecodeStepGraph): every step
        # copies the batches' pinned host activations in, rotates, multiplies
        # and copies y back to pinned host memory (one graph per step), then
        # waits
        plans = [B.DecodeStepGraph([(lay, m) for m in DECODE_MS]) for lay in layers]
        for pl in plans:
            for b in range(len(DECODE_MS)):
                pl.x_host[b].copy_(xs_host[b])
        e2e_i = [0]

        def e2e_step():
            plans[e2e_i[0] % len(layers)].launch()
            e2e_i[0] += 1
            stream.synchronize()

        for _ in range(args.warmup):
            e2e_step()
        e2e_steps = max(50, args.steps // 20)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        te2e = time.perf_counter() - t0
        te2e = _max_over_ranks(te2e, ws)

    bytes_step = run.bytes_per_step()
    value = aggregate_value(bytes_step, args.steps, ws, t)
    m = DECODE_MS[kb]
    alg = _gemv_algorithmic_bytes(m, layer.n, layer.k)
    achieved = alg / (gemv_us * 1e-6) / 1e9
    h2d = sum(m * layer.k * 2 for m in DECODE_MS)
    d2h = sum(m * layer.n * 2 for m in DECODE_MS)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 products (2*code x fp16 activations), f32 accumulate",
        "data": "synthetic (seeded uniform ternary codes, |N(0,1)|-based fp16 g128 scales, "
                "bf16 N(0,1) activations with 0.1% outlier channels x50)",
        "config": {"workload": "decode gate/up 5120->34816", "K": layer.k, "N": layer.n,
                   "M": list(DECODE_MS), "weight_copies": copies,
                   "weight_bytes_per_copy": layers[0].weight_bytes,
                   "l2": "inputs larger than L2: weights rotate over "
                         f"{copies} copies ({copies * layers[0].weight_bytes / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{ws} (independent layers per GPU)"},
        "pct_hbm_peak": round(100 * value / ws / hbm_peak, 1),
        "roofline": {"bound": "hbm", "kernel": "tern_gemv_decode (M=%d)" % m,
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4),
                     "traffic": TRAFFIC_GEMV_GATEUP_M4 if m == 4 else None,
                     "algorithmic_bytes": alg, "avg_launch_us": round(gemv_us, 3),
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)"},
        "e2e": {"value": round(bytes_step * e2e_steps * ws / te2e / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(te2e / e2e_steps * 1e3, 4),
                "transfer": ("kernels read x from and write y to pinned host memory in place"
                             if plans[0].zero_copy else "memcpy nodes in the step's graph")},
        "fused_step": {"what": "rotation folded into the GEMV (tern_linear_decode), one launch "
                                "per batch, the same weights and batches",
                       "value": round(bytes_step * fused_steps / tf / 1e9, 1), "unit": "GB/s",
                       "ms_per_step": round(tf / fused_steps * 1e3, 5)},
        "gpu_launches": run.launches_per_step() * args.steps,
        "clocks": clocks,
    }
    return out, layers


# ---------------------------------------------------------------- split layer (--split)

SPLIT_LAYERS = (I.GATE_UP, I.DOWN)


def split_shard(split, layer, world, rank, codes, scales, pack=True):
    """This rank's part of one layer: its output rows (split "n", column
    parallel) or its input columns (split "k", row parallel with the page's
    half-block exchange), packed for decode (pack=False keeps the codes and
    scales for a reference compute)."""
    from ternary_weight_linear_block_gb300 import tp as TP
    if split == "n":
        plan = TP.nsplit_plan(layer.n, world, rank)
        return TP.NSplitLinear(plan, codes[plan.n0:plan.n1].contiguous(),
                               scales[plan.n0:plan.n1].contiguous(), decode=True, prefill=False,
                               pack=pack)
    plan = TP.ksplit_plan(layer.k, world, rank)
    return TP.KSplitLinear(plan, codes[:, plan.k0:plan.k1].contiguous(),
                           scales[:, plan.k0 // 128:plan.k1 // 128].contiguous(), decode=True,
                           prefill=False, expand=False, pack=pack)


def split_forward(split, lin, x, world, group=None, ops=None, local=None):
    """One decode forward of a split layer on this rank: x is the whole input
    [M, K]; returns the whole output (split "n": the all-gathered rows; split
    "k": the all-reduced sum of the ranks' partials).  With one rank there is
    no collective."""
    from ternary_weight_linear_block_gb300 import tp as TP
    if split == "n":
        if world == 1:
            return (local or TP.nsplit_local)(lin, x)
        return TP.nsplit_forward(lin, x, group=group, local=local)
    xs = x[:, lin.plan.k0:lin.plan.k1].contiguous()
    if world == 1:
        xr, h = TP.local_phase(lin, xs, ops=ops)
        return TP.finish_phase(lin, xr, [h], "decode", ops)
    return TP.forward(lin, xs, group=group, mode="decode", ops=ops)


def split_value(whole_bytes_per_step, steps, t_max):
    """Strong scaling: the whole layers' weight bytes per step (each step
    processes every layer once, however it is split) over the slowest rank's
    time."""
    return whole_bytes_per_step * steps / t_max / 1e9


def run_split(args, rank, ws, local):
    """Decode of gate/up and down split over the ranks (tensor parallel), both
    batches (M = 1 and 4) per step; weights rotate over shard copies larger
    than L2 on every rank; NCCL collectives in the data path."""
    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    split = args.split
    with torch.cuda.stream(stream):
        g = torch.Generator(device="cuda")
        shards = {}
        copies = {}
        for layer in SPLIT_LAYERS:
            shard_bytes = B.tern_packed_bytes(layer.n, layer.k) // ws
            copies[layer.name] = max(2, int(np.ceil(2 * L2_BYTES / max(shard_bytes, 1))) + 1)
            shards[layer.name] = []
            for c in range(copies[layer.name]):
                g.manual_seed(4242 + c)            # the same layer on every rank
                codes = (torch.randint(0, 3, (layer.n, layer.k), dtype=torch.int8, device="cuda",
                                       generator=g) - 1).to(torch.int8)
                scales = (0.02 * torch.randn((layer.n, layer.k // 128), device="cuda",
                                             generator=g).abs() + 1e-3).to(torch.float16)
                shards[layer.name].append(split_shard(split, layer, ws, rank, codes, scales))
                del codes, scales
        xs = {(layer.name, m): _activations(layer, m, seed=500 + m).cuda()
              for layer in SPLIT_LAYERS for m in DECODE_MS}
        it = [0]

        def step():
            for layer in SPLIT_LAYERS:
                lin = shards[layer.name][it[0] % copies[layer.name]]
                for m in DECODE_MS:
                    split_forward(split, lin, xs[(layer.name, m)], ws)
            it[0] += 1

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        t = _time_region(step, args.steps, stream, ws, lead_cycles=0)
        t = _max_over_ranks(t, ws)
        B.tern_check(stream)
    whole = sum(B.tern_packed_bytes(l.n, l.k) for l in SPLIT_LAYERS) * len(DECODE_MS)
    how = ("column-parallel N split: each rank its output rows, one all-gather"
           if split == "n" else
           "row-parallel K split: each rank its input columns, half-block all-gather "
           "+ all-reduce of the partial outputs")
    return {
        "metric": METRIC, "value": round(split_value(whole, args.steps, t), 1), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 5), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None,
        "dtype": "f16 products (code x fp16 activations), f32 accumulate",
        "data": "synthetic (seeded uniform ternary codes, |N(0,1)|-based fp16 g128 scales, "
                "bf16 N(0,1) activations with 0.1% outlier channels x50)",
        "config": {"workload": "decode gate/up 5120->34816 and down 17408->5120, split over "
                               "the GPUs", "M": list(DECODE_MS),
                   "parallelism": f"tp{ws} {how}",
                   "l2": "inputs larger than L2: each rank's shards rotate over copies"},
        "gpu_launches": None}


def run_prefill(args, local, m=2048):
    """Prefill int8 path through gate/up 5120->34816 at M tokens: the rotation
    with per-token int8 quantisation, then the exact int8 GEMM (int8 values,
    fp16 tensor pipe) with its per-row / per-token rescale to bf16."""
    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    layer = I.GATE_UP
    _, tc_peak, peak_kind = _peaks()
    with torch.cuda.stream(stream):
        g = torch.Generator(device="cuda")
        g.manual_seed(7000)
        codes = (torch.randint(0, 3, (layer.n, layer.k), dtype=torch.int8, device="cuda",
                               generator=g) - 1).to(torch.int8)
        scales = (0.02 * torch.randn((layer.n, layer.k // 128), device="cuda", generator=g).abs()
                  + 1e-3).to(torch.float16)
        lay = B.pack_layer(codes, scales, decode=True, prefill=True, int8=True)
        w_h = B.expand_fp16(codes, scales)
        del codes, scales
        x = _activations(layer, m, seed=77).cuda()
        xq = torch.empty((m, layer.k), dtype=torch.float16, device="cuda")
        ts = torch.empty(m, dtype=torch.float32, device="cuda")
        y = torch.empty((m, layer.n), dtype=torch.bfloat16, device="cuda")
        st = stream.cuda_stream

        nbd = B.tern_workspace_bytes(B.TERN_OP_GEMM, m, layer.n, layer.k)
        wsd = B.Workspace().scratch(nbd) if nbd else None

        def step():
            B.tern_fwht_quant(x, m, layer.k, None, B.TERN_FWHT_I8H, xq, ts, st)
            B.tern_gemm_prefill_int8h(xq, ts, lay.w_q, lay.rscale, m, layer.n, layer.k, y, None,
                                     wsd, nbd, stream=st)

        def gemm_only():
            B.tern_gemm_prefill_int8h(xq, ts, lay.w_q, lay.rscale, m, layer.n, layer.k, y, None,
                                     wsd, nbd, stream=st)

        nbp = B.tern_workspace_bytes(B.TERN_OP_GEMM_PACKED, m, layer.n, layer.k)
        wsp = B.Workspace().scratch(nbp) if nbp else None

        def packed_only():
            B.tern_gemm_prefill_packed(xq, ts, lay.packed, lay.q, lay.rscale, m, layer.n,
                                       layer.k, y, None, wsp, nbp, stream=st)

        # the int8-typed boundary: int8 xq and W_int8, widened in the workspace per call
        xq8 = torch.empty((m, layer.k), dtype=torch.int8, device="cuda")
        nb8 = B.tern_workspace_bytes(B.TERN_OP_GEMM_INT8, m, layer.n, layer.k)
        ws8 = B.Workspace().scratch(nb8)

        def int8_step():
            B.tern_fwht_quant(x, m, layer.k, None, B.TERN_FWHT_I8, xq8, ts, st)
            B.tern_gemm_prefill_int8(xq8, ts, lay.w_int8, lay.rscale, m, layer.n, layer.k, y,
                                     None, ws8, nb8, stream=st)

        def int8_only():
            B.tern_gemm_prefill_int8(xq8, ts, lay.w_int8, lay.rscale, m, layer.n, layer.k, y,
                                     None, ws8, nb8, stream=st)

        xh = torch.empty((m, layer.k), dtype=torch.float16, device="cuda")
        xs = torch.empty((m, layer.k // 1024), dtype=torch.float32, device="cuda")
        B.tern_fwht_quant(x, m, layer.k, None, B.TERN_FWHT_F16, xh, xs, st)

        def fp16_only():
            B.tern_gemm_prefill_fp16(xh, xs, w_h, m, layer.n, layer.k, y, wsd, nbd, st)

        for _ in range(max(3, args.warmup // 4)):
            step()
            packed_only()
            fp16_only()
            int8_step()
        torch.cuda.synchronize()
        n = 20
        t = _time_region(step, n, stream, 1)
        tg = _time_region(gemm_only, n, stream, 1)
        tp = _time_region(packed_only, n, stream, 1)
        th = _time_region(fp16_only, n, stream, 1)
        t8 = _time_region(int8_step, n, stream, 1)
        tg8 = _time_region(int8_only, n, stream, 1)
        B.tern_check(stream)
    ops = 2.0 * m * layer.n * layer.k
    del lay, w_h, ws8
    torch.cuda.empty_cache()
    return {"metric": "prefill int8 TOPS (2*M*N*K / step time)", "value": round(ops * n / t / 1e12, 1),
            "unit": "TOPS", "workload": f"prefill gate/up 5120->34816, M={m}",
            "ms_per_step": round(t / n * 1e3, 4),
            "roofline": {"bound": "tensor",
                         "kernel": "tern_gemm_prefill_int8h (W_int8 held in fp16)",
                         "achieved": round(ops * n / tg / 1e12, 1), "peak": tc_peak,
                         "unit": "TFLOP/s", "frac": round(ops * n / tg / 1e12 / tc_peak, 4),
                         "avg_launch_us": round(tg / n * 1e6, 2),
                         "traffic": TRAFFIC_GEMM_I8_GATEUP_M2048 if m == 2048 else None,
                         "algorithmic_bytes": layer.n * layer.k * 2 + m * layer.k * 2
                                              + m * layer.n * 2 + 4 * (m + layer.n),
                         "peak_source": f"{peak_kind} bf16_tflops (MEASURED_PEAKS.json): the "
                                        "int8 values run on the fp16/bf16 tensor pipe; "
                                        "sm_103a has no tcgen05 int8 kind"},
            "packed": {"kernel": "tern_gemm_prefill_packed (no expanded weight in memory)",
                       "achieved": round(ops * n / tp / 1e12, 1), "unit": "TFLOP/s",
                       "frac": round(ops * n / tp / 1e12 / tc_peak, 4),
                       "avg_launch_us": round(tp / n * 1e6, 2),
                       "weight_bytes": layer.n * layer.k // 4 + layer.n * (layer.k // 128) * 3,
                       "expanded_weight_bytes": layer.n * layer.k * 2},
            "int8_typed": {"kernel": "tern_gemm_prefill_int8 (int8 xq and W_int8; both "
                                     "widened to fp16 in the workspace on every call)",
                           "achieved": round(ops * n / tg8 / 1e12, 1), "unit": "TFLOP/s",
                           "frac": round(ops * n / tg8 / 1e12 / tc_peak, 4),
                           "avg_call_us": round(tg8 / n * 1e6, 2),
                           "ms_per_step": round(t8 / n * 1e3, 4),
                           "vs_fp16_held": round(tg / tg8, 4)},
            "fp16_variant": {"kernel": "tern_gemm_prefill_fp16 (decode operand x fp16 code*s, "
                                       "no int8 quantisation)",
                             "achieved": round(ops * n / th / 1e12, 1), "unit": "TFLOP/s",
                             "frac": round(ops * n / th / 1e12 / tc_peak, 4),
                             "avg_launch_us": round(th / n * 1e6, 2)}}


def run_mid_m(args, local, ms=(32, 64, 128, 256, 512)):
    """Mid-size M (17..512 tokens) through each linear shape: the packed GEMM
    (2-bit weights; 128-token tiles up to M = 128, weight rows on the MMA's M
    side with 256-token tiles above; split along K when its tiles do not fill
    the GPU) against the GEMM on the expanded weight; GEMM alone, weights
    rotating over copies larger than L2, bit-identical outputs."""
    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    out = []
    with torch.cuda.stream(stream):
        st = stream.cuda_stream
        for shp in I.STACK_LAYERS:
            # both weight forms rotate over more than twice the L2
            copies = max(2, int(np.ceil(2 * L2_BYTES / B.tern_packed_bytes(shp.n, shp.k))))
            lays = _make_layers(shp, copies, seed=11, prefill=True)
            for m in ms:
                xq = torch.randint(-127, 128, (m, shp.k), device="cuda").half()
                ts = torch.full((m,), 1e-3, device="cuda")
                y = torch.empty((m, shp.n), dtype=torch.bfloat16, device="cuda")
                nb = B.tern_workspace_bytes(B.TERN_OP_GEMM_PACKED, m, shp.n, shp.k)
                wsb = B.Workspace().scratch(nb) if nb else None
                nbe = B.tern_workspace_bytes(B.TERN_OP_GEMM, m, shp.n, shp.k)
                wse = B.Workspace().scratch(nbe) if nbe else None
                i = [0]

                def packed():
                    l = lays[i[0] % copies]
                    i[0] += 1
                    B.tern_gemm_prefill_packed(xq, ts, l.packed, l.q, l.rscale, m, shp.n, shp.k,
                                               y, None, wsb, nb, stream=st)

                def expanded():
                    l = lays[i[0] % copies]
                    i[0] += 1
                    B.tern_gemm_prefill_int8h(xq, ts, l.w_q, l.rscale, m, shp.n, shp.k, y, None,
                                             wse, nbe, stream=st)

                for f in (packed, expanded):
                    for _ in range(3):
                        f()
                reps = 30
                tp = _time_region(packed, reps, stream, 1) / reps
                te = _time_region(expanded, reps, stream, 1) / reps
                out.append({"linear": shp.name, "M": m, "packed_us": round(tp * 1e6, 2),
                            "expanded_us": round(te * 1e6, 2),
                            "packed_launches": B.tern_kernel_launches(B.TERN_OP_GEMM_PACKED, m,
                                                                      shp.n, shp.k)})
            del lays
            torch.cuda.empty_cache()
        B.tern_check(stream)
    return out


def run_prefill_configs(args, local, configs=((I.GATE_UP, 512), (I.DOWN, 512), (I.DOWN, 2048))):
    """The other prefill configurations (gate/up and down at M = 512 and
    2048): rotation + int8 quantisation + the int8 GEMM on the expanded
    weight (with its K-split workspace), and the GEMM alone, expanded and
    packed."""
    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    _, tc_peak, _ = _peaks()
    out = []
    with torch.cuda.stream(stream):
        st = stream.cuda_stream
        for layer, m in configs:
            lay = _make_layers(layer, 1, seed=8, prefill=True)[0]
            x = _activations(layer, m, seed=88).cuda()
            xq = torch.empty((m, layer.k), dtype=torch.float16, device="cuda")
            ts = torch.empty(m, dtype=torch.float32, device="cuda")
            y = torch.empty((m, layer.n), dtype=torch.bfloat16, device="cuda")
            nbd = B.tern_workspace_bytes(B.TERN_OP_GEMM, m, layer.n, layer.k)
            wsd = B.Workspace().scratch(nbd) if nbd else None
            nbp = B.tern_workspace_bytes(B.TERN_OP_GEMM_PACKED, m, layer.n, layer.k)
            wsp = B.Workspace().scratch(nbp) if nbp else None

            def gemm():
                B.tern_gemm_prefill_int8h(xq, ts, lay.w_q, lay.rscale, m, layer.n, layer.k, y,
                                         None, wsd, nbd, stream=st)

            def step():
                B.tern_fwht_quant(x, m, layer.k, None, B.TERN_FWHT_I8H, xq, ts, st)
                gemm()

            def packed():
                B.tern_gemm_prefill_packed(xq, ts, lay.packed, lay.q, lay.rscale, m, layer.n,
                                           layer.k, y, None, wsp, nbp, stream=st)

            for f in (step, packed):
                for _ in range(3):
                    f()
            torch.cuda.synchronize()
            n = 20
            t = _time_region(step, n, stream, 1)
            tg = _time_region(gemm, n, stream, 1)
            tp = _time_region(packed, n, stream, 1)
            B.tern_check(stream)
            ops = 2.0 * m * layer.n * layer.k
            out.append({"workload": f"prefill {layer.name}, M={m}",
                        "TOPS": round(ops * n / t / 1e12, 1),
                        "ms_per_step": round(t / n * 1e3, 4),
                        "gemm_us": round(tg / n * 1e6, 2),
                        "gemm_frac_of_bf16_peak": round(ops * n / tg / 1e12 / tc_peak, 4),
                        "gemm_launches": B.tern_kernel_launches(B.TERN_OP_GEMM, m, layer.n,
                                                                layer.k),
                        "packed_gemm_us": round(tp / n * 1e6, 2)})
            del lay
            torch.cuda.empty_cache()
    return out


def run_decode_configs(args, local, shapes=(I.DOWN, I.QKV, I.O_PROJ), ms=(1, 4, 8, 16)):
    """The decode configurations of down 17408->5120, qkv 5120->10240 and o
    5120->5120 at M = 1, 4, 8 and 16: a step of rotation + GEMV (+ fixup), and the GEMV
    alone, each call streaming the next of several weight copies that
    together exceed L2 by more than 3x."""
    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    hbm_peak, _, _ = _peaks()
    out = []
    with torch.cuda.stream(stream):
        st = stream.cuda_stream
        for shp in shapes:
            copies = max(3, int(np.ceil(3 * L2_BYTES / B.tern_packed_bytes(shp.n, shp.k))))
            lays = _make_layers(shp, copies, seed=12, prefill=False)
            wbytes = lays[0].weight_bytes
            for m in ms:
                x = _activations(shp, m, seed=120 + m).cuda()
                xh = torch.empty((m, shp.k), dtype=torch.float16, device="cuda")
                xs = B.decode_aux(shp.k)
                y = torch.empty((m, shp.n), dtype=torch.bfloat16, device="cuda")
                nb = B.tern_workspace_bytes(B.TERN_OP_GEMV, m, shp.n, shp.k)
                ws = B.Workspace().get(nb)
                i = [0]

                def gemv():
                    lay = lays[i[0] % copies]
                    i[0] += 1
                    B.tern_gemv_decode(lay.packed, xh, xs, m, shp.n, shp.k, y, ws, ws.numel(), st)

                def step():
                    B.tern_fwht_quant(x, m, shp.k, None, B.TERN_FWHT_DECODE, xh, xs, st)
                    gemv()

                for _ in range(5):
                    step()
                torch.cuda.synchronize()
                reps = 200
                ts = _time_region(step, reps, stream, 1) / reps
                tg = _time_region(gemv, reps, stream, 1) / reps
                B.tern_check(stream)
                out.append({"workload": f"decode {shp.name}, M={m}", "shape": shp.name, "M": m,
                            "weight_GBps": round(wbytes / ts / 1e9, 1),
                            "pct_hbm_peak": round(100 * wbytes / ts / 1e9 / hbm_peak, 1),
                            "step_us": round(ts * 1e6, 2), "gemv_us": round(tg * 1e6, 2),
                            "launches_per_step": 1 + B.tern_kernel_launches(B.TERN_OP_GEMV, m,
                                                                            shp.n, shp.k)})
            del lays
            torch.cuda.empty_cache()
    return out


def run_stack(args, local, n_layers=64, decode_ms=(1, 4, 8, 16), prefill_ms=(128, 512, 2048)):
    """The 64-layer linear stack of a 27B hybrid model: per layer qkv
    5120->10240, o 5120->5120, gate/up 5120->34816, down 17408->5120, each with
    its own seeded weights (seed = 4 * layer + linear).  The linears are not
    chained (there is no model): each shape has its own synthetic input.  A
    decode step runs rotation + GEMV through all 256 linears (captured as one
    CUDA graph, replayed); a prefill step runs rotation + int8 quantisation +
    the int8 GEMM through all 256."""
    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    shapes = I.STACK_LAYERS
    hbm_peak, tc_peak, _ = _peaks()
    with torch.cuda.stream(stream):
        g = torch.Generator(device="cuda")
        layers = []
        for li in range(n_layers):
            row = []
            for si, shp in enumerate(shapes):
                g.manual_seed(4 * li + si)
                codes = (torch.randint(0, 3, (shp.n, shp.k), dtype=torch.int8, device="cuda",
                                       generator=g) - 1).to(torch.int8)
                scales = (0.02 * torch.randn((shp.n, shp.k // 128), device="cuda", generator=g)
                          .abs() + 1e-3).to(torch.float16)
                row.append(B.pack_layer(codes, scales, decode=True, prefill=True))
                del codes, scales
            layers.append(row)
        torch.cuda.synchronize()
        packed_bytes = sum(l.weight_bytes for row in layers for l in row)
        wq_bytes = sum(l.w_q.numel() * 2 for row in layers for l in row)
        st = stream.cuda_stream
        out = {"layers": n_layers, "linears": [s.name for s in shapes],
               "packed_bytes": packed_bytes, "w_int8_held_as_fp16_bytes": wq_bytes,
               "inputs": "each linear shape has its own seeded synthetic input (not chained)",
               "decode": [], "prefill": []}
        for m in decode_ms:
            xs_in = [_activations(shp, m, seed=900 + si).cuda() for si, shp in enumerate(shapes)]
            xh = [torch.empty((m, shp.k), dtype=torch.float16, device="cuda") for shp in shapes]
            sc = [B.decode_aux(shp.k) for shp in shapes]
            ys = [torch.empty((m, shp.n), dtype=torch.bfloat16, device="cuda") for shp in shapes]
            wss = [B.Workspace().get(B.tern_workspace_bytes(B.TERN_OP_GEMV, m, shp.n, shp.k))
                   for shp in shapes]

            def decode_step(st_handle):
                for row in layers:
                    for si, (shp, lay) in enumerate(zip(shapes, row)):
                        B.tern_fwht_quant(xs_in[si], m, shp.k, None, B.TERN_FWHT_DECODE, xh[si],
                                          sc[si], st_handle)
                        B.tern_gemv_decode(lay.packed, xh[si], sc[si], m, shp.n, shp.k, ys[si],
                                           wss[si], wss[si].numel(), st_handle)

            decode_step(st)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                decode_step(torch.cuda.current_stream().cuda_stream)
            for _ in range(3):
                graph.replay()
            torch.cuda.synchronize()
            reps = 10
            t = _time_region(graph.replay, reps, stream, 1)
            B.tern_check(stream)
            gbps = packed_bytes * reps / t / 1e9
            out["decode"].append({"M": m, "ms_per_step": round(t / reps * 1e3, 4),
                                  "weight_GBps": round(gbps, 1),
                                  "pct_hbm_peak": round(100 * gbps / hbm_peak, 1),
                                  "launches_per_step": n_layers * sum(
                                      1 + B.tern_kernel_launches(B.TERN_OP_GEMV, m, shp.n, shp.k)
                                      for shp in shapes)})
            del graph
        ops_step = sum(2.0 * shp.n * shp.k for shp in shapes) * n_layers
        for m in prefill_ms:
            xs_in = [_activations(shp, m, seed=950 + si).cuda() for si, shp in enumerate(shapes)]
            xq = [torch.empty((m, shp.k), dtype=torch.float16, device="cuda") for shp in shapes]
            ts = [torch.empty(m, dtype=torch.float32, device="cuda") for shp in shapes]
            ys = [torch.empty((m, shp.n), dtype=torch.bfloat16, device="cuda") for shp in shapes]

            nbs = [B.tern_workspace_bytes(B.TERN_OP_GEMM_PACKED, m, shp.n, shp.k)
                   for shp in shapes]
            wsp = B.Workspace().scratch(max(nbs)) if max(nbs) else None
            nbe = [B.tern_workspace_bytes(B.TERN_OP_GEMM, m, shp.n, shp.k) for shp in shapes]
            wse = B.Workspace().scratch(max(nbe)) if max(nbe) else None

            def prefill_step(packed=False):
                for row in layers:
                    for si, (shp, lay) in enumerate(zip(shapes, row)):
                        B.tern_fwht_quant(xs_in[si], m, shp.k, None, B.TERN_FWHT_I8H, xq[si],
                                          ts[si], st)
                        if packed:
                            B.tern_gemm_prefill_packed(xq[si], ts[si], lay.packed, lay.q,
                                                       lay.rscale, m, shp.n, shp.k, ys[si], None,
                                                       wsp, nbs[si], stream=st)
                        else:
                            B.tern_gemm_prefill_int8h(xq[si], ts[si], lay.w_q, lay.rscale, m,
                                                     shp.n, shp.k, ys[si], None, wse, nbe[si],
                                                     stream=st)

            prefill_step()
            prefill_step(packed=True)
            torch.cuda.synchronize()
            reps = 3
            t = _time_region(prefill_step, reps, stream, 1)
            tp = _time_region(lambda: prefill_step(packed=True), reps, stream, 1)
            B.tern_check(stream)
            tops = ops_step * m * reps / t / 1e12
            out["prefill"].append({"M": m, "ms_per_step": round(t / reps * 1e3, 3),
                                   "TOPS": round(tops, 1),
                                   "frac_of_bf16_peak": round(tops / tc_peak, 4),
                                   "packed_ms_per_step": round(tp / reps * 1e3, 3),
                                   "packed_TOPS": round(ops_step * m * reps / tp / 1e12, 1)})
            del xq, ys
    del layers
    torch.cuda.empty_cache()
    return out


def _oracle_rate(budget_s):
    """The oracle (fp64 dense reference) timed on a bounded sample of the
    decode workload: weight bytes per second, repetitions, seconds."""
    from oracle import tern_oracle as O
    layer = I.GATE_UP
    rows = 2048
    d = I.make_layer(layer, 4, seed=0, n=rows)
    xs = {m: d.x[:m] for m in DECODE_MS}
    O.linear_f64(xs[1], d.codes[:16], d.scales[:16])     # warm the H matrix cache
    done_bytes = 0
    t0 = time.perf_counter()
    reps = 0
    while True:
        for m in DECODE_MS:
            O.linear_f64(xs[m], d.codes, d.scales)
            done_bytes += rows * layer.k // 4 + rows * (layer.k // 128) * 2
        reps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return done_bytes / dt, reps, dt, rows, layer


def _oracle_rate_one_core(budget_s):
    """The same on one core: a child process whose BLAS libraries start with
    one thread (their thread count is fixed when numpy loads)."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                "BLIS_NUM_THREADS"):
        env[var] = "1"
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "r = bench._oracle_rate(%r); print(json.dumps([r[0], r[1], r[2]]))" % (ROOT, budget_s))
    try:
        p = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=budget_s + 120)
        rate, reps, dt = json.loads(p.stdout.strip().splitlines()[-1])
        return rate, reps, dt
    except (subprocess.SubprocessError, ValueError, IndexError):
        return None


_SHAPES = {l.name: l for l in (I.TINY, I.GATE_UP, I.DOWN, I.QKV, I.O_PROJ)}


def _oracle_config_rate(kind, shape_name, m, rows, budget_s):
    """The oracle on a seeded row sample of one configuration, repeated for
    about budget_s seconds.  kind "decode": O1 (fp64 dense reference), rate in
    weight bytes per second of the sampled rows; kind "prefill": O2 (the
    int8 path), rate in int8 ops (2 M rows K) per second."""
    from oracle import tern_oracle as O
    layer = _SHAPES[shape_name]
    d = I.make_layer(layer, m, seed=5, n=rows)
    work = (rows * layer.k // 4 + rows * (layer.k // 128) * 2) if kind == "decode" \
        else 2.0 * m * rows * layer.k
    fn = (lambda: O.linear_f64(d.x, d.codes, d.scales)) if kind == "decode" \
        else (lambda: O.linear_int8(d.x, d.codes, d.scales))
    fn()                                   # warm (the dense H cache, allocator)
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return work * reps / dt, reps, dt


def _one_core(fn_name, fn_args, budget_s):
    """bench.<fn_name>(*fn_args) in a child process whose BLAS libraries start
    with one thread (their thread count is fixed when numpy loads)."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                "BLIS_NUM_THREADS"):
        env[var] = "1"
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "r = bench.%s(*%r); print(json.dumps([r[0], r[1], r[2]]))" % (ROOT, fn_name, fn_args))
    try:
        p = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=budget_s + 120)
        return tuple(json.loads(p.stdout.strip().splitlines()[-1]))
    except (subprocess.SubprocessError, ValueError, IndexError):
        return None


def _host_cores():
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        blas = max((i.get("num_threads", 1) for i in threadpool_info()), default=cores)
        cores = min(cores, blas)
    except ImportError:
        pass
    return cores


def config_cpu_baseline(kind, layer, m, rows, budget_s=1.5, one_core_s=1.0):
    """The oracle beside one GPU configuration, on the host's cores and on one."""
    rate, reps, dt = _oracle_config_rate(kind, layer.name, m, rows, budget_s)
    unit, scale = ("GB/s", 1e9) if kind == "decode" else ("TOPS", 1e12)
    out = {"value": round(rate / scale, 6), "unit": unit, "cores": _host_cores(), "kind": "oracle",
           "sample": f"{'fp64 dense oracle (O1)' if kind == 'decode' else 'int8-path oracle (O2)'} "
                     f"on {rows} of {layer.n} rows of {layer.name}, M={m}, "
                     f"{reps} repetitions in {dt:.1f} s"}
    if one_core_s > 0:
        r1 = _one_core("_oracle_config_rate", [kind, layer.name, m, rows, one_core_s], one_core_s)
        if r1 is not None:
            out["one_core"] = {"value": round(r1[0] / scale, 6), "unit": unit, "cores": 1,
                               "sample": f"the same sample, {r1[1]} repetitions in {r1[2]:.1f} s"}
    return out


def run_cpu_baseline(args, budget_s=15.0, one_core_s=5.0):
    """The oracle (fp64 dense reference) timed on a bounded sample of the
    workload, on the host's cores, and (one_core_s > 0) on one core."""
    rate, reps, dt, rows, layer = _oracle_rate(budget_s)
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        blas = max((i.get("num_threads", 1) for i in threadpool_info()), default=cores)
        cores = min(cores, blas)
    except ImportError:
        pass
    out = {"value": round(rate / 1e9, 4), "unit": "GB/s", "cores": cores,
           "kind": "oracle",
           "sample": f"fp64 dense oracle on {rows} of {layer.n} rows of gate/up 5120->34816, "
                     f"M=1 and M=4, {reps} repetitions in {dt:.1f} s"}
    if one_core_s > 0:
        r1 = _oracle_rate_one_core(one_core_s)
        if r1 is not None:
            out["one_core"] = {"value": round(r1[0] / 1e9, 4), "unit": "GB/s", "cores": 1,
                               "sample": f"the same sample, {r1[1]} repetitions in {r1[2]:.1f} s"}
    return out


def _oracle_step(rows, layer, d_x):
    """One reference step: the fp64 oracle on `rows` seeded rows of gate/up for
    each decode batch; returns the weight bytes it covered."""
    from oracle import tern_oracle as O
    done = 0
    for m in DECODE_MS:
        O.linear_f64(d_x[:m], rows[0], rows[1])
        done += rows[0].shape[0] * layer.k // 4 + rows[0].shape[0] * (layer.k // 128) * 2
    return done


def run_reference(args, rank, ws):
    """The reference arm: the oracle (fp64 dense reference) timed on the host
    cores, exactly --steps steps after --warmup untimed ones, each step a
    seeded row sample of the decode workload (both batches) sized so the run
    stays within about two minutes."""
    if rank != 0:
        return None
    layer = I.GATE_UP
    d = I.make_layer(layer, 4, seed=0, n=2048)
    per_step = min(1.0, 120.0 / max(1, args.steps + args.warmup))
    # calibrate: time one step on 64 rows, then size the sample to per_step
    t0 = time.perf_counter()
    _oracle_step((d.codes[:64], d.scales[:64]), layer, d.x)
    t64 = time.perf_counter() - t0
    rows = int(max(1, min(2048, 64 * per_step / max(t64, 1e-6))))
    sample = (d.codes[:rows], d.scales[:rows])
    for _ in range(args.warmup):
        _oracle_step(sample, layer, d.x)
    done = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        done += _oracle_step(sample, layer, d.x)
    dt = time.perf_counter() - t0
    v = round(done / dt / 1e9, 5)
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count()
    base = {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 dense oracle on {rows} of {layer.n} rows of gate/up 5120->34816 "
                      f"per step, M=1 and M=4, {args.steps} steps in {dt:.1f} s"}
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / max(1, args.steps) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode gate/up 5120->34816", "K": 5120, "N": 34816,
                       "M": list(DECODE_MS)},
            "cpu_baseline": base,
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-stack", action="store_true")
    ap.add_argument("--split", choices=["n", "k"], default=None,
                    help="split gate/up and down over the GPUs (tensor parallel) instead of "
                         "running independent replicas")
    ap.add_argument("--no-decode-configs", action="store_true",
                    help="skip the down / qkv decode configurations (for profiling)")
    ap.add_argument("--stack-layers", type=int, default=64,
                    help="layers of the linear stack section (64 = the 27B model's stack)")
    ap.add_argument("--stack-only", action="store_true",
                    help="run only the stack section (for profiling); prints its JSON object")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank, ws, local = _dist_init()
    if args.impl == "reference":
        line = run_reference(args, rank, ws)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    from ternary_weight_linear_block_gb300 import build as BUILD
    if BUILD.is_stale():          # missing, or older than a source file
        if rank == 0:
            BUILD.build()
        _barrier(ws)
    if args.split:
        line = run_split(args, rank, ws, local)
        if rank == 0:
            print(json.dumps(line), flush=True)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    if args.stack_only:
        if rank == 0:
            print(json.dumps({"stack": run_stack(args, local, n_layers=args.stack_layers)}),
                  flush=True)
        return
    line, layers = run_decode(args, rank, ws, local)
    del layers
    torch.cuda.empty_cache()
    cpu = not args.no_cpu_baseline and ws == 1 and rank == 0
    if rank == 0 and not args.no_decode_configs:
        line["decode_configs"] = run_decode_configs(args, local)
        if cpu:
            for e in line["decode_configs"]:
                e["cpu_baseline"] = config_cpu_baseline(
                    "decode", _SHAPES[e["shape"]], e["M"], rows=256, budget_s=1.0,
                    one_core_s=1.0 if e["M"] == 4 else 0)
    if not args.no_prefill:
        line["prefill"] = run_prefill(args, local)
        if cpu:
            line["prefill"]["cpu_baseline"] = config_cpu_baseline(
                "prefill", I.GATE_UP, 512, rows=64, budget_s=2.0, one_core_s=1.5)
        if rank == 0:
            line["prefill"]["other_configs"] = run_prefill_configs(args, local)
    if not args.no_prefill and rank == 0:
        line["mid_m"] = run_mid_m(args, local)
    if not args.no_stack and rank == 0:
        line["stack"] = run_stack(args, local, n_layers=args.stack_layers)
        if cpu:
            # each distinct shape's oracle rate at M = 1, times the layers
            secs = 0.0
            for shp in I.STACK_LAYERS:
                r = config_cpu_baseline("decode", shp, 1, rows=256, budget_s=1.0, one_core_s=0)
                secs += B.tern_packed_bytes(shp.n, shp.k) / (r["value"] * 1e9)
            secs *= args.stack_layers
            line["stack"]["cpu_baseline"] = {
                "value": round(line["stack"]["packed_bytes"] / secs / 1e9, 6), "unit": "GB/s",
                "ms_per_step": round(secs * 1e3, 1), "cores": _host_cores(), "kind": "oracle",
                "sample": "fp64 dense oracle (O1) at M=1 on 256 rows of each of the four linear "
                          "shapes, its per-byte rate applied to each shape's weights, times "
                          f"{args.stack_layers} layers"}
    if rank == 0:
        if not args.no_cpu_baseline and ws == 1:
            line["cpu_baseline"] = run_cpu_baseline(args)
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
