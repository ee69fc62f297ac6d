"""Host-side checks of the C-ABI library (no GPU needed).

The library must load, export every function that include/tern.h declares,
and reject bad arguments on the host before any CUDA call.
"""

import ctypes
import os

import pytest
import torch

from ternary_weight_linear_block_gb300 import binding as B
from ternary_weight_linear_block_gb300 import build as BUILD


@pytest.fixture(scope="session")
def lib():
    BUILD.ensure_built()          # missing, or older than a source file
    return B.lib()


def test_every_header_function_is_exported(lib):
    names = B.header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(B._SIGS), "binding and header disagree"


def test_status_strings_and_version(lib):
    assert B.tern_version() == 100
    for code, name in B.STATUS_NAMES.items():
        assert B.tern_status_str(code) == name
    assert B.tern_status_str(99) == "TERN_ERR_UNKNOWN"


def test_sizes(lib):
    # codes (2 bits) + fp16 scales per 128 elements, rows padded to 512
    assert B.tern_packed_bytes(34816, 5120) == 34816 * 5120 // 4 + 34816 * 40 * 2
    assert B.tern_packed_bytes(100, 1024) == 512 * 1024 // 4 + 512 * 8 * 2
    assert B.tern_packed_bytes(-1, 1024) == 0
    assert B.tern_workspace_bytes(B.TERN_OP_GEMV, 0, 10, 1024) == 0
    assert B.tern_workspace_bytes(B.TERN_OP_GEMV, 4, 34816, 5120) > 0


def test_kernel_launch_counts(lib):
    # 152 SMs (the host default with no device, and GB300's count)
    G = B.TERN_OP_GEMV
    assert B.tern_kernel_launches(G, 0, 34816, 5120) == 0
    assert B.tern_kernel_launches(99, 4, 34816, 5120) == 0
    # 1088 gate/up pair tiles on 76 pairs: the last wave's tiles split along K,
    # finished by a second kernel
    assert B.tern_kernel_launches(B.TERN_OP_GEMM, 2048, 34816, 5120) == 2
    # gate/up: 68 blocks x 40 groups over 152 CTAs (17.9 units each): a block
    # has at most 4 owners, summed in place at M <= 8; any sharing at M > 8
    assert B.tern_kernel_launches(G, 1, 34816, 5120) == 1
    assert B.tern_kernel_launches(G, 8, 34816, 5120) == 1
    assert B.tern_kernel_launches(G, 9, 34816, 5120) == 2
    # down: 10 blocks x 136 groups -> about 16 owners per block
    assert B.tern_kernel_launches(G, 1, 5120, 17408) == 2
    # 152 blocks of 8 groups: one block per CTA, nothing shared
    assert B.tern_kernel_launches(G, 16, 152 * 512, 1024) == 1
    # one block of 8 groups split over 8 CTAs
    assert B.tern_kernel_launches(G, 16, 512, 1024) == 2
    # the packed GEMM: 8 x 136 pair tiles on 76 pairs, the last wave's 24
    # tiles split in 3 K slices (a second kernel adds the [256][256] int32
    # pieces); down at 128 tokens has 20 CTA tiles, all split along K
    P = B.TERN_OP_GEMM_PACKED
    assert B.tern_kernel_launches(P, 2048, 34816, 5120) == 2
    assert B.tern_workspace_bytes(P, 2048, 34816, 5120) == 24 * 3 * 256 * 256 * 4
    # gate/up at 512 tokens: 272 tiles, kept whole
    assert B.tern_kernel_launches(P, 512, 34816, 5120) == 1
    assert B.tern_workspace_bytes(P, 512, 34816, 5120) == 0
    assert B.tern_kernel_launches(P, 128, 5120, 17408) == 2
    # 20 tiles -> 7 slices of whole 128-groups (140 units), one int32 plane each
    assert B.tern_workspace_bytes(P, 128, 5120, 17408) == 7 * 128 * 5120 * 4


FAKE = 1 << 20          # an aligned, never dereferenced address


def _st(fn, *args):
    return getattr(B.lib(), fn)(*args)


def test_pack_argument_errors(lib):
    assert _st("tern_pack", FAKE, FAKE, 16, 1000, FAKE, None, None, None, None) == 2
    assert _st("tern_pack", FAKE, FAKE, -1, 1024, FAKE, None, None, None, None) == 1
    assert _st("tern_pack", FAKE, FAKE, 16, 1024, FAKE, FAKE, None, None, None) == 1
    assert _st("tern_pack", FAKE, FAKE, 16, 1024, None, None, None, FAKE, None) == 1
    assert _st("tern_pack", None, FAKE, 16, 1024, FAKE, None, None, None, None) == 1
    assert _st("tern_pack", FAKE + 4, FAKE, 16, 1024, FAKE, None, None, None, None) == 3
    assert _st("tern_pack", FAKE, FAKE, 0, 1024, FAKE, None, None, None, None) == 0
    assert _st("tern_pack", FAKE, FAKE, 16, 1024 * 65, FAKE, None, None, None, None) == 2


def test_fwht_argument_errors(lib):
    assert _st("tern_fwht_quant", FAKE, 4, 1000, None, 0, FAKE, None, None) == 2
    assert _st("tern_fwht_quant", FAKE, 4, 1024, None, 7, FAKE, None, None) == 1
    assert _st("tern_fwht_quant", FAKE, 4, 1024, None, 1, FAKE, None, None) == 1   # no scale out
    assert _st("tern_fwht_quant", FAKE, 4, 1024 * 33, None, 2, FAKE, FAKE, None) == 2
    assert _st("tern_fwht_quant", FAKE + 2, 4, 1024, None, 0, FAKE, None, None) == 3
    assert _st("tern_fwht_quant", None, 4, 1024, None, 0, FAKE, None, None) == 1
    assert _st("tern_fwht_quant", FAKE, 0, 1024, None, 0, FAKE, None, None) == 0
    assert _st("tern_fwht_quant", FAKE, -3, 1024, None, 0, FAKE, None, None) == 1
    assert _st("tern_fwht_quant", FAKE, 17, 1024, None, 1, FAKE, FAKE, None) == 2  # decode: M <= 16
    assert _st("tern_fwht_quant", FAKE, 4, 1024, None, 3, FAKE, None, None) == 1   # fp16: no scale out
    assert _st("tern_quant_rotated", FAKE, 17, 1024, 1, FAKE, FAKE, None) == 2
    assert _st("tern_quant_rotated", FAKE, 4, 1024, 0, FAKE, FAKE, None) == 1      # no f32 mode


def test_gemv_argument_errors(lib):
    ws = B.tern_workspace_bytes(B.TERN_OP_GEMV, 4, 256, 1024)
    args = lambda m=4, n=256, k=1024, ws_ptr=FAKE, ws_b=ws, y=FAKE: (
        FAKE, FAKE, FAKE, m, n, k, y, ws_ptr, ws_b, None)
    assert _st("tern_gemv_decode", *args(m=17)) == 2
    assert _st("tern_gemv_decode", *args(k=1536)) == 2
    assert _st("tern_gemv_decode", *args(y=None)) == 1
    assert _st("tern_gemv_decode", *args(y=FAKE + 8)) == 3
    assert _st("tern_gemv_decode", *args(ws_b=ws - 1)) == 6
    assert _st("tern_gemv_decode", *args(ws_ptr=None)) == 6
    assert _st("tern_gemv_decode", *args(m=0)) == 0
    # the fp32-input sibling: a larger workspace (GEMV part, then the operand)
    wf = B.tern_workspace_bytes(B.TERN_OP_GEMV_F32, 4, 256, 1024)
    assert wf >= ws + 4 * 1024 * 2 + 8 * 192
    assert B.tern_workspace_bytes(B.TERN_OP_GEMV_F32, 17, 256, 1024) == 0
    f32 = lambda m=4, k=1024, xr=FAKE, ws_b=wf, y=FAKE: (FAKE, xr, m, 256, k, y, FAKE, ws_b, None)
    assert _st("tern_gemv_decode_f32", *f32(m=17)) == 2
    assert _st("tern_gemv_decode_f32", *f32(k=1536)) == 2
    assert _st("tern_gemv_decode_f32", *f32(xr=None)) == 1
    assert _st("tern_gemv_decode_f32", *f32(xr=FAKE + 4)) == 3
    assert _st("tern_gemv_decode_f32", *f32(ws_b=ws)) == 6
    assert _st("tern_gemv_decode_f32", *f32(m=0)) == 0
    assert _st("tern_gemv_decode_f32", *f32()) == 4            # valid, but no GPU here


def test_gemm_argument_errors(lib):
    a = lambda m=64, n=256, k=1024, y=FAKE, ws=None, nb=0: (FAKE, FAKE, FAKE, FAKE, m, n, k, y,
                                                            None, ws, nb, None)
    for fn in ("tern_gemm_prefill_int8h", "tern_gemm_prefill_int8"):
        assert _st(fn, *a(n=250)) == 2
        assert _st(fn, *a(k=100)) == 2
        assert _st(fn, *a(y=None)) == 1
        assert _st(fn, *a(y=FAKE + 2)) == 3
        assert _st(fn, *a(m=0)) == 0
    # the int8-typed call needs its workspace: both operands widened, then the split pieces
    nb = B.tern_workspace_bytes(B.TERN_OP_GEMM_INT8, 64, 256, 1024)
    assert nb >= (64 + 256) * 1024 * 2
    assert B.tern_workspace_bytes(B.TERN_OP_GEMM_INT8, 2048, 34816, 5120) >= (
        (2048 + 34816) * 5120 * 2 + B.tern_workspace_bytes(B.TERN_OP_GEMM, 2048, 34816, 5120))
    assert _st("tern_gemm_prefill_int8", *a()) == B.TERN_ERR_WORKSPACE
    assert _st("tern_gemm_prefill_int8", *a(ws=FAKE, nb=nb - 1)) == B.TERN_ERR_WORKSPACE
    assert _st("tern_gemm_prefill_int8", *a(ws=FAKE + 8, nb=nb)) == 3
    assert B.tern_kernel_launches(B.TERN_OP_GEMM_INT8, 64, 256, 1024) in (3, 4)
    assert B.tern_kernel_launches(B.TERN_OP_GEMM_INT8, 0, 256, 1024) == 0


def test_widen_argument_errors(lib):
    w = lambda rows=4, cols=32, src=FAKE, dst=FAKE: (src, rows, cols, dst, None)
    assert _st("tern_widen_int8", *w(rows=-1)) == 1
    assert _st("tern_widen_int8", *w(cols=24)) == 2
    assert _st("tern_widen_int8", *w(rows=0, src=None)) == 0
    assert _st("tern_widen_int8", *w(src=None)) == 1
    assert _st("tern_widen_int8", *w(dst=FAKE + 2)) == 3


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_is_unsupported(lib):
    assert _st("tern_fwht_quant", FAKE, 4, 1024, None, 0, FAKE, None, None) == 4
    assert _st("tern_selftest_wait", 64, None) == B.TERN_ERR_UNSUPPORTED


def test_selftest_wait_argument_errors(lib):
    """The poll count is checked before anything else (no GPU needed)."""
    assert _st("tern_selftest_wait", 0, None) == B.TERN_ERR_INVALID_ARG
    assert _st("tern_selftest_wait", (1 << 20) + 1, None) == B.TERN_ERR_INVALID_ARG


def test_binding_raises_named_error(lib):
    with pytest.raises(B.TernError) as ei:
        B.tern_fwht_quant(FAKE, 4, 1000, None, 0, FAKE, None, stream=0)
    assert ei.value.status == 2 and "TERN_ERR_SHAPE" in str(ei.value)


def test_gemm_packed_argument_errors(lib):
    need = B.tern_workspace_bytes(B.TERN_OP_GEMM_PACKED, 64, 256, 5120)
    a = lambda m=64, n=256, k=5120, y=FAKE, ws=FAKE, wsb=need: (
        FAKE, FAKE, FAKE, FAKE, FAKE, m, n, k, y, None, ws, wsb, None)
    assert need > 0                                            # 1 x 1 tile: split along K
    assert _st("tern_gemm_prefill_packed", *a(n=250)) == 2       # N % 16
    assert _st("tern_gemm_prefill_packed", *a(k=1536)) == 2
    assert _st("tern_gemm_prefill_packed", *a(m=-1)) == 1
    assert _st("tern_gemm_prefill_packed", *a(y=None)) == 1
    assert _st("tern_gemm_prefill_packed", *a(y=FAKE + 2)) == 3
    assert _st("tern_gemm_prefill_packed", *a(wsb=need - 1)) == 6
    assert _st("tern_gemm_prefill_packed", *a(ws=None)) == 6
    assert _st("tern_gemm_prefill_packed", *a(ws=FAKE + 8)) == 3
    assert _st("tern_gemm_prefill_packed", *a(m=0)) == 0
    assert _st("tern_gemm_prefill_packed", *a(n=0)) == 0


def test_ksplit_argument_errors(lib):
    sh = lambda m=2, kr=8704, lead=0, trail=1, x=FAKE, xr=FAKE, hl=None, ht=FAKE: (
        x, m, kr, lead, trail, None, xr, hl, ht, None)
    assert _st("tern_fwht_shard", *sh(trail=0)) == 2                 # 8.5 blocks, no half marked
    assert _st("tern_fwht_shard", *sh(lead=2)) == 1
    assert _st("tern_fwht_shard", *sh(ht=None)) == 1                 # trailing half, no output
    assert _st("tern_fwht_shard", *sh(lead=1, trail=1, kr=9216, hl=None)) == 1
    assert _st("tern_fwht_shard", *sh(x=None)) == 1
    assert _st("tern_fwht_shard", *sh(x=FAKE + 2)) == 3
    assert _st("tern_fwht_shard", *sh(kr=512 + 65536)) == 2          # padded width > 65536
    assert _st("tern_fwht_shard", *sh(m=0)) == 0
    cb = lambda m=2, part=0, kp=9216, blk=8, hf=FAKE: (hf, FAKE, m, part, FAKE, kp, blk, None)
    assert _st("tern_fwht_combine", *cb(part=2)) == 1
    assert _st("tern_fwht_combine", *cb(blk=9)) == 2
    assert _st("tern_fwht_combine", *cb(kp=9000)) == 2
    assert _st("tern_fwht_combine", *cb(hf=None)) == 1
    assert _st("tern_fwht_combine", *cb(hf=FAKE + 4)) == 3
    assert _st("tern_fwht_combine", *cb(m=0)) == 0
    qr = lambda m=2, k=9216, mode=1, sc=FAKE: (FAKE, m, k, mode, FAKE, sc, None)
    assert _st("tern_quant_rotated", *qr(mode=0)) == 1               # only DECODE and I8
    assert _st("tern_quant_rotated", *qr(k=8704)) == 2
    assert _st("tern_quant_rotated", *qr(sc=None)) == 1
    assert _st("tern_quant_rotated", *qr(m=0)) == 0


def test_fp16_variant_argument_errors(lib):
    assert _st("tern_expand_fp16", FAKE, FAKE, 16, 1000, FAKE, None) == 2
    assert _st("tern_expand_fp16", FAKE, FAKE, -1, 1024, FAKE, None) == 1
    assert _st("tern_expand_fp16", FAKE, FAKE, 16, 1024, None, None) == 1
    assert _st("tern_expand_fp16", FAKE + 1, FAKE, 16, 1024, FAKE, None) == 3
    assert _st("tern_expand_fp16", FAKE, FAKE, 0, 1024, FAKE, None) == 0
    g = lambda m=64, n=256, k=1024, y=FAKE, ws=None: (FAKE, FAKE, FAKE, m, n, k, y, ws, 0, None)
    assert _st("tern_gemm_prefill_fp16", *g(n=250)) == 2
    assert _st("tern_gemm_prefill_fp16", *g(k=1536)) == 2
    assert _st("tern_gemm_prefill_fp16", *g(y=None)) == 1
    assert _st("tern_gemm_prefill_fp16", *g(y=FAKE + 2)) == 3
    assert _st("tern_gemm_prefill_fp16", *g(ws=FAKE + 4)) == 3
    assert _st("tern_gemm_prefill_fp16", *g(m=0)) == 0
    # the expanded GEMMs' optional split: 20 tiles of down at 128 tokens
    assert B.tern_workspace_bytes(B.TERN_OP_GEMM, 128, 5120, 17408) > 0
    assert B.tern_kernel_launches(B.TERN_OP_GEMM, 128, 5120, 17408) == 2
    # ... and the last wave of gate/up at 2048 tokens (24 of 76 pairs busy)
    assert B.tern_workspace_bytes(B.TERN_OP_GEMM, 2048, 34816, 5120) > 0
    assert B.tern_kernel_launches(B.TERN_OP_GEMM, 2048, 34816, 5120) == 2
    # o at 512 tokens: 40 pair tiles, one wave, kept whole
    assert B.tern_workspace_bytes(B.TERN_OP_GEMM, 512, 5120, 5120) == 0
    assert B.tern_kernel_launches(B.TERN_OP_GEMM, 512, 5120, 5120) == 1


def test_host_accessible_query(lib):
    assert B.lib().tern_host_accessible(None) == 0
    if not torch.cuda.is_available():
        assert B.lib().tern_host_accessible(FAKE) == 0        # no device: never


def test_workspace_zero_fills_for_the_gemv_after_a_gemm(monkeypatch):
    """Workspace bookkeeping (host logic; the zero-fill call is faked on a
    CPU tensor): ``get`` zero-fills a new or GEMM-used buffer once, and not
    again while only GEMV calls use it."""
    fills = []

    def fake_init(ws, nbytes=None, stream=None):
        ws[:nbytes].zero_()
        fills.append(nbytes)
        return B.TERN_OK

    monkeypatch.setattr(B, "tern_workspace_init", fake_init)
    ws = B.Workspace(device="cpu")
    a = ws.get(1000)
    assert a.numel() == 1000 and not a.any() and fills == [1000]
    ws.get(600)
    assert fills == [1000]                      # still clean
    s = ws.scratch(800)
    assert s.data_ptr() == a.data_ptr()
    s.fill_(0x5A)                               # what a split GEMM may leave
    b = ws.get(600)
    assert not b.any() and fills == [1000, 1000]
    ws.scratch(4000).fill_(7)                   # grows: a new buffer, contents undefined
    c = ws.get(100)
    assert c.numel() == 4000 and not c.any() and fills[-1] == 4000


def test_a_timeout_marks_every_workspace_dirty(monkeypatch):
    """After tern_check reports a bounded wait that gave up, the GEMV may have
    left published partial sums in its workspace: every live Workspace's next ``get``
    zero-fills again (host logic; tern_check and the fill are faked)."""
    fills = []

    def fake_init(ws, nbytes=None, stream=None):
        ws[:nbytes].zero_()
        fills.append(nbytes)
        return B.TERN_OK

    class FakeLib:
        status = B.TERN_OK

        def tern_check(self, stream):
            return self.status

    fake = FakeLib()
    monkeypatch.setattr(B, "tern_workspace_init", fake_init)
    monkeypatch.setattr(B, "lib", lambda: fake)
    a, b = B.Workspace(device="cpu"), B.Workspace(device="cpu")
    a.get(512)
    b.get(256)
    assert fills == [512, 256]
    B.tern_check(stream=0)                      # OK: nothing changes
    a.get(512)
    b.get(256)
    assert fills == [512, 256]
    fake.status = B.TERN_ERR_TIMEOUT
    with pytest.raises(B.TernError) as ei:
        B.tern_check(stream=0)
    assert ei.value.status == B.TERN_ERR_TIMEOUT
    a.get(512)
    b.get(256)
    assert fills == [512, 256, 512, 256]


def test_binding_constants_match_the_header():
    import re
    with open(B.HEADER) as f:
        text = f.read()
    m = re.search(r"#define TERN_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == B.TERN_NOALLOC_SCRATCH_BYTES
    for name in ("TERN_ERR_WORKSPACE", "TERN_ERR_TIMEOUT", "TERN_ERR_INVALID_ARG",
                 "TERN_ERR_UNSUPPORTED"):
        m = re.search(r"\b%s = (\d+)" % name, text)
        assert m and int(m.group(1)) == getattr(B, name), name
    for name in ("TERN_OP_GEMV", "TERN_OP_GEMM", "TERN_OP_GEMM_PACKED", "TERN_OP_GEMV_F32",
                 "TERN_OP_GEMM_INT8", "TERN_FWHT_F32", "TERN_FWHT_DECODE", "TERN_FWHT_I8",
                 "TERN_FWHT_F16", "TERN_FWHT_I8H"):
        m = re.search(r"#define %s (\d+)" % name, text)
        assert m and int(m.group(1)) == getattr(B, name), name
