"""Thin ctypes binding over libtern.so (include/tern.h).

The functions named ``tern_*`` mirror the C entry points one to one and only
marshal arguments: torch tensors supply device memory (their data pointers)
and the current CUDA stream supplies ``stream``.  Every step of the layer runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback, and a
missing library raises.

``pack_layer`` / ``decode`` / ``prefill`` are conveniences that allocate the
outputs with torch and call the entry points in order.
"""

from __future__ import annotations

import ctypes
import os
import re
import weakref
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtern.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "tern.h")

TERN_OK = 0
TERN_ERR_INVALID_ARG = 1
TERN_ERR_UNSUPPORTED = 4
TERN_ERR_WORKSPACE = 6
TERN_ERR_TIMEOUT = 7
TERN_NOALLOC_SCRATCH_BYTES = 24 << 20     # include/tern.h, tern_gemv_decode_noalloc
TERN_FWHT_F32 = 0
TERN_FWHT_DECODE = 1
TERN_FWHT_I8 = 2
TERN_FWHT_F16 = 3
TERN_FWHT_I8H = 4
TERN_OP_GEMV = 1
TERN_OP_GEMM = 2
TERN_OP_GEMM_PACKED = 3
TERN_OP_GEMV_F32 = 4
TERN_OP_GEMM_INT8 = 5
STATUS_NAMES = {0: "TERN_OK", 1: "TERN_ERR_INVALID_ARG", 2: "TERN_ERR_SHAPE", 3: "TERN_ERR_ALIGN",
                4: "TERN_ERR_UNSUPPORTED", 5: "TERN_ERR_CUDA", 6: "TERN_ERR_WORKSPACE",
                7: "TERN_ERR_TIMEOUT"}

_i64 = ctypes.c_int64
_p = ctypes.c_void_p
_sz = ctypes.c_size_t
_SIGS = {
    "tern_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "tern_version": (ctypes.c_int, []),
    "tern_packed_bytes": (_sz, [_i64, _i64]),
    "tern_workspace_bytes": (_sz, [ctypes.c_int, _i64, _i64, _i64]),
    "tern_kernel_launches": (ctypes.c_int, [ctypes.c_int, _i64, _i64, _i64]),
    "tern_host_accessible": (ctypes.c_int, [_p]),
    "tern_workspace_init": (ctypes.c_int, [_p, _sz, _p]),
    "tern_pack": (ctypes.c_int, [_p, _p, _i64, _i64, _p, _p, _p, _p, _p]),
    "tern_fwht_quant": (ctypes.c_int, [_p, _i64, _i64, _p, ctypes.c_int, _p, _p, _p]),
    "tern_gemv_decode": (ctypes.c_int, [_p, _p, _p, _i64, _i64, _i64, _p, _p, _sz, _p]),
    "tern_expand_fp16": (ctypes.c_int, [_p, _p, _i64, _i64, _p, _p]),
    "tern_gemm_prefill_fp16": (ctypes.c_int, [_p, _p, _p, _i64, _i64, _i64, _p, _p, _sz, _p]),
    "tern_fwht_shard": (ctypes.c_int, [_p, _i64, _i64, ctypes.c_int, ctypes.c_int, _p, _p, _p, _p,
                                       _p]),
    "tern_fwht_combine": (ctypes.c_int, [_p, _p, _i64, ctypes.c_int, _p, _i64, _i64, _p]),
    "tern_quant_rotated": (ctypes.c_int, [_p, _i64, _i64, ctypes.c_int, _p, _p, _p]),
    "tern_widen_int8": (ctypes.c_int, [_p, _i64, _i64, _p, _p]),
    "tern_gemm_prefill_int8": (ctypes.c_int, [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _p, _sz,
                                              _p]),
    "tern_gemm_prefill_int8h": (ctypes.c_int, [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _p, _sz,
                                               _p]),
    "tern_gemm_prefill_packed": (ctypes.c_int, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _p,
                                                _p, _sz, _p]),
    "tern_check": (ctypes.c_int, [_p]),
    "tern_selftest_wait": (ctypes.c_int, [ctypes.c_uint32, _p]),
    "tern_gemv_decode_noalloc": (ctypes.c_int, [_p, _p, _p, _i64, _i64, _i64, _p, _p]),
    "tern_linear_decode": (ctypes.c_int, [_p, _p, _p, _i64, _i64, _i64, _p, _p, _sz, _p]),
    "tern_gemv_decode_f32": (ctypes.c_int, [_p, _p, _i64, _i64, _i64, _p, _p, _sz, _p]),
}

_lib = None


class TernError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libtern.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libtern.so not built ({LIB_PATH}); run "
                               "ternary_weight_linear_block_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def header_functions() -> list[str]:
    """Names of the functions declared in include/tern.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(tern_\w+)\s*\(", text, re.M)))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return stream


def _call(name, *args):
    st = getattr(lib(), name)(*args)
    if st != TERN_OK:
        raise TernError(name, st)
    return st


# ---------------------------------------------------------------- C mirrors

def tern_status_str(status: int) -> str:
    return lib().tern_status_str(status).decode()


def tern_version() -> int:
    return lib().tern_version()


def tern_packed_bytes(n: int, k: int) -> int:
    return lib().tern_packed_bytes(n, k)


def tern_workspace_bytes(op: int, m: int, n: int, k: int) -> int:
    return lib().tern_workspace_bytes(op, m, n, k)


def tern_kernel_launches(op: int, m: int, n: int, k: int) -> int:
    return lib().tern_kernel_launches(op, m, n, k)


def tern_host_accessible(t) -> bool:
    """Whether the GPU can read and write this host buffer in place."""
    return bool(lib().tern_host_accessible(_ptr(t)))


def tern_workspace_init(ws, nbytes: int | None = None, stream=None):
    nb = ws.numel() * ws.element_size() if nbytes is None else nbytes
    return _call("tern_workspace_init", _ptr(ws), nb, _stream(stream))


def tern_pack(codes, scales, n, k, packed, q, rscale, w_int8, stream=None):
    return _call("tern_pack", _ptr(codes), _ptr(scales), n, k, _ptr(packed), _ptr(q),
                 _ptr(rscale), _ptr(w_int8), _stream(stream))


def tern_widen_int8(src, rows, cols, dst, stream=None):
    return _call("tern_widen_int8", _ptr(src), rows, cols, _ptr(dst), _stream(stream))


def tern_fwht_quant(x, m, k, sign, mode, out, out_scale, stream=None):
    return _call("tern_fwht_quant", _ptr(x), m, k, _ptr(sign), mode, _ptr(out), _ptr(out_scale),
                 _stream(stream))


def tern_gemv_decode(packed, xh, xs, m, n, k, y, ws, ws_bytes, stream=None):
    return _call("tern_gemv_decode", _ptr(packed), _ptr(xh), _ptr(xs), m, n, k, _ptr(y), _ptr(ws),
                 ws_bytes, _stream(stream))


def tern_gemm_prefill_int8(xq, tscale, w_int8, rscale, m, n, k, y, acc=None, ws=None,
                           ws_bytes=0, stream=None):
    return _call("tern_gemm_prefill_int8", _ptr(xq), _ptr(tscale), _ptr(w_int8), _ptr(rscale), m,
                 n, k, _ptr(y), _ptr(acc), _ptr(ws), ws_bytes, _stream(stream))


def tern_gemm_prefill_int8h(xq, tscale, w_q, rscale, m, n, k, y, acc=None, ws=None, ws_bytes=0,
                            stream=None):
    return _call("tern_gemm_prefill_int8h", _ptr(xq), _ptr(tscale), _ptr(w_q), _ptr(rscale), m,
                 n, k, _ptr(y), _ptr(acc), _ptr(ws), ws_bytes, _stream(stream))


def tern_gemm_prefill_packed(xq, tscale, packed, q, rscale, m, n, k, y, acc=None, ws=None,
                             ws_bytes=0, stream=None):
    return _call("tern_gemm_prefill_packed", _ptr(xq), _ptr(tscale), _ptr(packed), _ptr(q),
                 _ptr(rscale), m, n, k, _ptr(y), _ptr(acc), _ptr(ws), ws_bytes, _stream(stream))


def tern_expand_fp16(codes, scales, n, k, w_h, stream=None):
    return _call("tern_expand_fp16", _ptr(codes), _ptr(scales), n, k, _ptr(w_h), _stream(stream))


def tern_gemm_prefill_fp16(xh, xs, w_h, m, n, k, y, ws=None, ws_bytes=0, stream=None):
    return _call("tern_gemm_prefill_fp16", _ptr(xh), _ptr(xs), _ptr(w_h), m, n, k, _ptr(y),
                 _ptr(ws), ws_bytes, _stream(stream))


def tern_fwht_shard(x, m, kr, lead, trail, sign, xr, h_lead, h_trail, stream=None):
    return _call("tern_fwht_shard", _ptr(x), m, kr, int(lead), int(trail), _ptr(sign), _ptr(xr),
                 _ptr(h_lead), _ptr(h_trail), _stream(stream))


def tern_fwht_combine(h_first, h_second, m, part, xr, kp, blk, stream=None):
    return _call("tern_fwht_combine", _ptr(h_first), _ptr(h_second), m, part, _ptr(xr), kp, blk,
                 _stream(stream))


def tern_quant_rotated(xr, m, k, mode, out, out_scale, stream=None):
    return _call("tern_quant_rotated", _ptr(xr), m, k, mode, _ptr(out), _ptr(out_scale),
                 _stream(stream))


def tern_check(stream=None):
    """Synchronise and report bounded-wait timeouts.  After a timeout the
    decode GEMV may have left published partial sums (nonzero words) in its
    workspace, so every live ``Workspace`` is marked dirty (its next ``get``
    zero-fills it again)."""
    st = lib().tern_check(_stream(stream))
    if st == TERN_ERR_TIMEOUT:
        for w in list(_WORKSPACES):
            w.clean = 0
    if st != TERN_OK:
        raise TernError("tern_check", st)
    return st


def tern_selftest_wait(polls: int, stream=None):
    """Launch the bounded-wait self-test (a wait that gives up after ``polls``
    polls); the next tern_check raises TERN_ERR_TIMEOUT."""
    return _call("tern_selftest_wait", polls, _stream(stream))


def tern_gemv_decode_f32(packed, xr, m, n, k, y, ws, ws_bytes, stream=None):
    return _call("tern_gemv_decode_f32", _ptr(packed), _ptr(xr), m, n, k, _ptr(y), _ptr(ws),
                 ws_bytes, _stream(stream))


def tern_linear_decode(x, sign, packed, m, n, k, y, ws, ws_bytes, stream=None):
    return _call("tern_linear_decode", _ptr(x), _ptr(sign), _ptr(packed), m, n, k, _ptr(y),
                 _ptr(ws), ws_bytes, _stream(stream))


def tern_gemv_decode_noalloc(packed, xh, xs, m, n, k, y, stream=None):
    """Decode GEMV with the library's fixed scratch array (no workspace, no
    allocation), for callers that cannot allocate device memory."""
    return _call("tern_gemv_decode_noalloc", _ptr(packed), _ptr(xh), _ptr(xs), m, n, k, _ptr(y),
                 _stream(stream))


# ---------------------------------------------------------------- conveniences

def _need(t, dtype, name):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name}: expected a contiguous CUDA tensor of {dtype}")


@dataclass
class PackedLayer:
    n: int
    k: int
    packed: torch.Tensor | None         # uint8, codes + scales in 17408-byte units
    q: torch.Tensor | None              # int8 [N, G]
    rscale: torch.Tensor | None         # float32 [N]
    w_q: torch.Tensor | None            # float16 [N, K] holding W_int8 (exact)
    w_int8: torch.Tensor | None = None  # int8 [N, K]

    @property
    def weight_bytes(self) -> int:
        """Algorithmic bytes of the decode weights: 2-bit codes + fp16 scales."""
        return self.n * self.k // 4 + self.n * (self.k // 128) * 2


def pack_layer(codes: torch.Tensor, scales: torch.Tensor, decode: bool = True,
               prefill: bool = True, expand: bool = True, int8: bool = False,
               stream=None) -> PackedLayer:
    """Run tern_pack on device codes (int8 [N,K]) and scales (fp16 [N,G]).
    ``decode`` keeps the packed 2-bit units, ``prefill`` the scale split
    (q, rscale); with ``expand`` the layer also keeps W_int8 held in fp16
    (w_q, tern_widen_int8 of tern_pack's int8 weight), the operand of
    tern_gemm_prefill_int8h, and with ``int8`` the int8 weight itself
    (w_int8, for tern_gemm_prefill_int8).  Without either, prefill reads
    the packed units (tern_gemm_prefill_packed)."""
    _need(codes, torch.int8, "codes")
    _need(scales, torch.float16, "scales")
    n, k = codes.shape
    dev = codes.device
    packed = q = rs = wq = w8 = None
    if decode:
        packed = torch.empty(tern_packed_bytes(n, k), dtype=torch.uint8, device=dev)
    if prefill:
        q = torch.empty((n, k // 128), dtype=torch.int8, device=dev)
        rs = torch.empty(n, dtype=torch.float32, device=dev)
        if expand or int8:
            w8 = torch.empty((n, k), dtype=torch.int8, device=dev)
    tern_pack(codes, scales, n, k, packed, q, rs, w8, stream)
    if expand and w8 is not None:
        wq = torch.empty((n, k), dtype=torch.float16, device=dev)
        tern_widen_int8(w8, n, k, wq, stream)
    return PackedLayer(n, k, packed, q, rs, wq, w8 if int8 else None)


def decode_aux(k: int, device="cuda") -> torch.Tensor:
    """The float [K/128][48] group records of the decode operand
    (TERN_FWHT_DECODE's out_scale)."""
    return torch.empty((k // 128, 48), dtype=torch.float32, device=device)


def fwht(x: torch.Tensor, mode: int, sign: torch.Tensor | None = None, stream=None):
    """Rotation (+ quantisation) of bf16 activations [M,K]; returns (out, out_scale)."""
    _need(x, torch.bfloat16, "x")
    m, k = x.shape
    dev = x.device
    if mode == TERN_FWHT_F32:
        out, sc = torch.empty((m, k), dtype=torch.float32, device=dev), None
    elif mode == TERN_FWHT_DECODE:
        out = torch.empty((m, k), dtype=torch.float16, device=dev)
        sc = decode_aux(k, dev)
    elif mode == TERN_FWHT_F16:
        out = torch.empty((m, k), dtype=torch.float16, device=dev)
        sc = torch.empty((m, k // 1024), dtype=torch.float32, device=dev)
    else:
        dt = torch.int8 if mode == TERN_FWHT_I8 else torch.float16
        out = torch.empty((m, k), dtype=dt, device=dev)
        sc = torch.empty(m, dtype=torch.float32, device=dev)
    tern_fwht_quant(x, m, k, sign, mode, out, sc, stream)
    return out, sc


# Every live Workspace, so that a timeout reported by tern_check marks them
# all dirty.
_WORKSPACES: "weakref.WeakSet[Workspace]" = weakref.WeakSet()


class Workspace:
    """A device workspace for the library's calls, grown on demand; use it
    from one stream.  The decode GEMV needs the bytes it uses zero-filled and
    leaves them so, while the split GEMMs leave partial sums behind: ``get``
    returns the buffer ready for the GEMV (zero-filling it on the stream
    first if a GEMM used it since), ``scratch`` returns it for a GEMM."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = None
        self.clean = 0        # leading bytes known to be zero
        _WORKSPACES.add(self)

    def _ensure(self, nbytes: int) -> int:
        nbytes = max(int(nbytes), 256)
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            self.clean = 0
        return nbytes

    def get(self, nbytes: int, stream=None) -> torch.Tensor:
        """The buffer with at least ``nbytes`` zero bytes, for tern_gemv_decode
        or tern_linear_decode."""
        nbytes = self._ensure(nbytes)
        if self.clean < nbytes:
            tern_workspace_init(self.buf, self.buf.numel(), stream)
            self.clean = self.buf.numel()
        return self.buf

    def scratch(self, nbytes: int, stream=None) -> torch.Tensor:
        """The buffer of at least ``nbytes`` bytes, any contents, for a GEMM
        (which leaves partial sums in it)."""
        self._ensure(nbytes)
        self.clean = 0
        return self.buf


def decode(layer: PackedLayer, x: torch.Tensor, ws: Workspace, y: torch.Tensor | None = None,
           sign=None, stream=None, fused: bool = False) -> torch.Tensor:
    """Decode forward for M <= 16 bf16 tokens: rotation, then the GEMV (the
    two calls, or one launch of tern_linear_decode with ``fused=True``; the
    results agree bit for bit)."""
    m = x.shape[0]
    _need(x, torch.bfloat16, "x")
    if y is None:
        y = torch.empty((m, layer.n), dtype=torch.bfloat16, device=x.device)
    nb = tern_workspace_bytes(TERN_OP_GEMV, m, layer.n, layer.k)
    buf = ws.get(nb, stream)
    if fused:
        tern_linear_decode(x, sign, layer.packed, m, layer.n, layer.k, y, buf, buf.numel(), stream)
        return y
    xh, xs = fwht(x, TERN_FWHT_DECODE, sign, stream)
    tern_gemv_decode(layer.packed, xh, xs, m, layer.n, layer.k, y, buf, buf.numel(), stream)
    return y


class _DecodeCall:
    """Device and pinned host buffers of one decode forward (layer, M).  With
    zero_copy the kernels read x from, and write y to, the pinned host
    buffers in place; otherwise the graph copies them (memcpy nodes)."""

    def __init__(self, layer: PackedLayer, m: int, sign, fused: bool, device, zero_copy):
        self.layer, self.m, self.sign, self.fused = layer, m, sign, fused
        self.x_host = torch.zeros((m, layer.k), dtype=torch.bfloat16).pin_memory()
        self.y_host = torch.empty((m, layer.n), dtype=torch.bfloat16).pin_memory()
        if zero_copy is None:
            zero_copy = tern_host_accessible(self.x_host) and tern_host_accessible(self.y_host)
        self.zero_copy = bool(zero_copy)
        if self.zero_copy:
            self.x, self.y = self.x_host, self.y_host
        else:
            self.x = torch.empty((m, layer.k), dtype=torch.bfloat16, device=device)
            self.y = torch.empty((m, layer.n), dtype=torch.bfloat16, device=device)
        self.xh = torch.empty((m, layer.k), dtype=torch.float16, device=device)
        self.xs = decode_aux(layer.k, device)
        nb = tern_workspace_bytes(TERN_OP_GEMV, m, layer.n, layer.k)
        self.ws = Workspace(device).get(nb)

    def first(self):
        """The input's copy (if any) and the rotation (the fused call: all of it)."""
        lay, m = self.layer, self.m
        st = torch.cuda.current_stream().cuda_stream
        if not self.zero_copy:
            self.x.copy_(self.x_host, non_blocking=True)
        x, y = self.x.data_ptr(), self.y.data_ptr()
        if self.fused:
            tern_linear_decode(x, self.sign, lay.packed, m, lay.n, lay.k, y, self.ws,
                               self.ws.numel(), st)
        else:
            tern_fwht_quant(x, m, lay.k, self.sign, TERN_FWHT_DECODE, self.xh, self.xs, st)

    def second(self):
        """The GEMV (two-call form) and the output's copy (if any)."""
        lay, m = self.layer, self.m
        st = torch.cuda.current_stream().cuda_stream
        if not self.fused:
            tern_gemv_decode(lay.packed, self.xh, self.xs, m, lay.n, lay.k, self.y.data_ptr(),
                             self.ws, self.ws.numel(), st)
        if not self.zero_copy:
            self.y_host.copy_(self.y, non_blocking=True)


class DecodeStepGraph:
    """Several decode forwards -- (layer, M) pairs, e.g. the batches or the
    layers of one decode step -- captured once as a single CUDA graph with
    their host transfers: each call copies its pinned host input
    ``x_host[i]`` to the device, rotates, multiplies (tern_fwht_quant +
    tern_gemv_decode, or tern_linear_decode with ``fused=True``) and copies
    its bf16 result back to the pinned ``y_host[i]``.  ``run()`` replays the
    graph on the current stream and waits for it, so the whole step pays one
    graph launch and one wait.  The buffers belong to the graph: write the
    inputs into ``x_host`` and read ``y_host`` after ``run`` returns.

    Where the GPU can address the pinned buffers directly
    (tern_host_accessible, e.g. over NVLink-C2C on Grace-Blackwell) the
    rotation reads x from host memory and the GEMV writes y into it, with no
    copy (``zero_copy=None`` chooses; True forces it, False uses copies).

    Every call reads its own host input, so the calls are independent: the
    graph issues all the rotations first (they overlap one another) and then
    the GEMVs back to back."""

    def __init__(self, entries, sign: torch.Tensor | None = None, fused: bool = False,
                 device="cuda", zero_copy: bool | None = None):
        self.calls = [_DecodeCall(layer, m, sign, fused, device, zero_copy)
                      for layer, m in entries]
        self.zero_copy = all(c.zero_copy for c in self.calls)
        self.x_host = [c.x_host for c in self.calls]
        self.y_host = [c.y_host for c in self.calls]
        self._body()                      # first launch outside capture (sets kernel attributes)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._body()

    def _body(self):
        for c in self.calls:
            c.first()
        for c in self.calls:
            c.second()

    def launch(self):
        """Replay on the current stream without waiting."""
        self.graph.replay()

    def run(self):
        """Replay and wait; returns the pinned host outputs."""
        self.launch()
        torch.cuda.current_stream().synchronize()
        return self.y_host


class DecodeGraph(DecodeStepGraph):
    """One layer's decode forward for a fixed M (a DecodeStepGraph of one
    call), with ``x_host`` / ``y_host`` the call's pinned buffers."""

    def __init__(self, layer: PackedLayer, m: int, sign: torch.Tensor | None = None,
                 fused: bool = False, device="cuda", zero_copy: bool | None = None):
        super().__init__([(layer, m)], sign, fused, device, zero_copy)
        self.layer, self.m, self.sign, self.fused = layer, m, sign, fused
        self.x_host = self.calls[0].x_host
        self.y_host = self.calls[0].y_host

    def launch(self, x: torch.Tensor | None = None):
        """Replay on the current stream without waiting."""
        if x is not None:
            self.x_host.copy_(x)
        self.graph.replay()

    def run(self, x: torch.Tensor | None = None) -> torch.Tensor:
        """Replay and wait; returns the pinned host output."""
        self.launch(x)
        torch.cuda.current_stream().synchronize()
        return self.y_host


def expand_fp16(codes: torch.Tensor, scales: torch.Tensor, stream=None) -> torch.Tensor:
    """The fp16 weight code * s [N, K] of the fp16 prefill variant."""
    _need(codes, torch.int8, "codes")
    _need(scales, torch.float16, "scales")
    n, k = codes.shape
    w_h = torch.empty((n, k), dtype=torch.float16, device=codes.device)
    tern_expand_fp16(codes, scales, n, k, w_h, stream)
    return w_h


def prefill_fp16(w_h: torch.Tensor, x: torch.Tensor, y: torch.Tensor | None = None, sign=None,
                 stream=None, ws: Workspace | None = None) -> torch.Tensor:
    """fp16 prefill variant: rotation to the fp16 operand (fp16 + per-block
    factors), then one tensor-core GEMM against w_h with the factors applied
    per 1024-block in the epilogue."""
    m = x.shape[0]
    n, k = w_h.shape
    xh, xs = fwht(x, TERN_FWHT_F16, sign, stream)
    if y is None:
        y = torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    nb = tern_workspace_bytes(TERN_OP_GEMM, m, n, k)
    buf = (ws or Workspace(x.device)).scratch(nb, stream) if nb > 0 else None
    tern_gemm_prefill_fp16(xh, xs, w_h, m, n, k, y, buf, nb, stream)
    return y


def prefill(layer: PackedLayer, x: torch.Tensor, y: torch.Tensor | None = None,
            acc: torch.Tensor | None = None, sign=None, stream=None,
            from_packed: bool | None = None, ws: Workspace | None = None) -> torch.Tensor:
    """Prefill forward: rotation + per-token int8 quantisation, then the int8
    GEMM -- straight from the packed units (``from_packed``; the default when
    the layer holds no expanded weight), on the fp16-held weight w_q, or on
    the int8 weight w_int8 (int8-typed operands, tern_gemm_prefill_int8).
    All three give bit-identical results."""
    m = x.shape[0]
    if from_packed is None:
        from_packed = layer.w_q is None and layer.w_int8 is None
    ws = ws or Workspace(x.device)
    if y is None:
        y = torch.empty((m, layer.n), dtype=torch.bfloat16, device=x.device)
    if from_packed or layer.w_q is not None:
        xq, ts = fwht(x, TERN_FWHT_I8H, sign, stream)
        op = TERN_OP_GEMM_PACKED if from_packed else TERN_OP_GEMM
        nb = tern_workspace_bytes(op, m, layer.n, layer.k)
        buf = ws.scratch(nb, stream) if nb > 0 else None
        nb = 0 if buf is None else buf.numel()
        if from_packed:
            tern_gemm_prefill_packed(xq, ts, layer.packed, layer.q, layer.rscale, m, layer.n,
                                     layer.k, y, acc, buf, nb, stream=stream)
        else:
            tern_gemm_prefill_int8h(xq, ts, layer.w_q, layer.rscale, m, layer.n, layer.k, y, acc,
                                    buf, nb, stream=stream)
        return y
    if layer.w_int8 is None:
        raise ValueError("prefill needs packed units, w_q or w_int8")
    xq, ts = fwht(x, TERN_FWHT_I8, sign, stream)
    nb = tern_workspace_bytes(TERN_OP_GEMM_INT8, m, layer.n, layer.k)
    buf = ws.scratch(nb, stream)
    tern_gemm_prefill_int8(xq, ts, layer.w_int8, layer.rscale, m, layer.n, layer.k, y, acc, buf,
                           buf.numel(), stream=stream)
    return y


def forward(layer: PackedLayer, x: torch.Tensor, y: torch.Tensor | None = None,
            ws: Workspace | None = None, sign=None, stream=None) -> torch.Tensor:
    """The layer for any number of tokens, on the path measured fastest on
    GB300 for that M: the decode GEMV for M <= 16; the int8 GEMM straight from
    the packed weights for 16 < M <= 256 (or whenever the layer holds no
    expanded weight); the int8 GEMM on the expanded weight w_q above that.
    The decode path keeps fp16 activations; the int8 paths quantise them per
    token (the page's section 4), so results differ by the int8 tolerance
    across the M = 16 boundary."""
    m = x.shape[0]
    ws = ws or Workspace(x.device)
    if m <= 16 and layer.packed is not None:
        return decode(layer, x, ws, y=y, sign=sign, stream=stream)
    if layer.q is None:
        raise ValueError("prefill needs the layer packed with prefill=True (q, rscale)")
    from_packed = layer.packed is not None and (
        (layer.w_q is None and layer.w_int8 is None) or m <= 256)
    return prefill(layer, x, y=y, sign=sign, stream=stream, from_packed=from_packed, ws=ws)

