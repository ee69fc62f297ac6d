"""GPU parity of tern_fwht_quant against the oracle (bitwise)."""

import numpy as np
import pytest
import torch

from oracle import tern_oracle as O
from ternary_weight_linear_block_gb300 import binding as B
from ternary_weight_linear_block_gb300 import inputs as I
from tests.gpu_helpers import bf16_to_f32, ensure_lib, f16_bits, poison, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

CASES = [  # (M, K, outlier fraction, factor): the workloads' activation mixes
    (1, 1024, 0.01, 20.0), (8, 1024, 0.01, 20.0), (1, 5120, 0.001, 50.0), (4, 5120, 0.001, 50.0),
    (3, 17408, 0.001, 50.0), (16, 17408, 0.001, 50.0), (13, 2048, 0.01, 20.0),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _run(xd, m, k, mode, sign=None):
    dev = "cuda"
    if mode == B.TERN_FWHT_F32:
        out, sc = poison(torch.empty((m, k), dtype=torch.float32, device=dev)), None
    elif mode == B.TERN_FWHT_DECODE:
        out = poison(torch.empty((m, k), dtype=torch.float16, device=dev))
        sc = poison(B.decode_aux(k, dev))
    elif mode == B.TERN_FWHT_F16:
        out = poison(torch.empty((m, k), dtype=torch.float16, device=dev))
        sc = poison(torch.empty((m, k // 1024), dtype=torch.float32, device=dev))
    else:
        dt = torch.int8 if mode == B.TERN_FWHT_I8 else torch.float16
        out = poison(torch.empty((m, k), dtype=dt, device=dev))
        sc = poison(torch.empty(m, dtype=torch.float32, device=dev))
    B.tern_fwht_quant(xd, m, k, sign, mode, out, sc)
    torch.cuda.synchronize()
    return out, sc


@pytest.mark.parametrize("m,k,frac,mult", CASES)
def test_fwht_f32_bitwise(m, k, frac, mult):
    bits, x = I.make_activations(1, m, k, frac, mult)
    out, _ = _run(to_dev_bf16(bits), m, k, B.TERN_FWHT_F32)
    ref = O.fwht_f32(x)
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("m,k,frac,mult", CASES)
def test_fwht_decode_operand_bitwise(m, k, frac, mult):
    """The decode operand (per-step scaled fp16) and its group records
    (offsets, fold factors, zeros for tokens M..15) bit for bit, written over
    a poisoned buffer."""
    bits, x = I.make_activations(2, m, k, frac, mult)
    out, sc = _run(to_dev_bf16(bits), m, k, B.TERN_FWHT_DECODE)
    vals, aux = O.decode_operand(O.fwht_f32(x))
    assert np.array_equal(f16_bits(out), vals.view(np.uint16))
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), aux.view(np.uint32))


@pytest.mark.parametrize("m,k,frac,mult", CASES + [(40, 5120, 0.001, 50.0)])
def test_fwht_f16_operand_bitwise(m, k, frac, mult):
    bits, x = I.make_activations(2, m, k, frac, mult)
    out, sc = _run(to_dev_bf16(bits), m, k, B.TERN_FWHT_F16)
    vals, inv = O.f16_operand(O.fwht_f32(x))
    assert np.array_equal(f16_bits(out), vals.view(np.uint16))
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), inv.view(np.uint32))


def test_decode_mode_rejects_more_than_16_tokens():
    x = torch.zeros((17, 1024), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((17, 1024), dtype=torch.float16, device="cuda")
    st = B.lib().tern_fwht_quant(x.data_ptr(), 17, 1024, None, B.TERN_FWHT_DECODE,
                                 out.data_ptr(), B.decode_aux(1024).data_ptr(), None)
    assert st == 2                                  # TERN_ERR_SHAPE


@pytest.mark.parametrize("m,k,frac,mult", CASES + [(64, 17408, 0.001, 50.0), (37, 5120, 0.001, 50.0),
                                           (5, 19456, 0.001, 50.0), (3, 32768, 0.001, 50.0)])
def test_fwht_i8_bitwise(m, k, frac, mult):
    """One CTA per token, one warp per block: up to 18 blocks two CTAs per
    SM, up to the mode's limit of 32 blocks one; both give the oracle's xq
    and tscale."""
    bits, x = I.make_activations(3, m, k, frac, mult)
    xd = to_dev_bf16(bits)
    out, sc = _run(xd, m, k, B.TERN_FWHT_I8)
    xq, ts = O.quant_tokens(O.fwht_f32(x))
    assert out.dtype == torch.int8
    assert np.array_equal(out.cpu().numpy(), xq.astype(np.int8))
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), ts.view(np.uint32))
    # the same integers held in fp16, the tensor cores' operand
    out_h, sc_h = _run(xd, m, k, B.TERN_FWHT_I8H)
    assert np.array_equal(out_h.cpu().float().numpy(), xq.astype(np.float32))
    assert torch.equal(sc, sc_h)


def test_sign_vector_all_modes():
    m, k = 5, 3072
    bits, x = I.make_activations(4, m, k, 0.01, 20.0)
    rng = np.random.default_rng(44)
    sign = rng.choice(np.array([-1, 1], np.int8), k)
    sd = to_dev(sign)
    xd = to_dev_bf16(bits)
    out, _ = _run(xd, m, k, B.TERN_FWHT_F32, sd)
    ref = O.fwht_f32(x, sign.astype(np.float32))
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    out, sc = _run(xd, m, k, B.TERN_FWHT_I8, sd)
    xq, ts = O.quant_tokens(ref)
    assert np.array_equal(out.cpu().float().numpy(), xq.astype(np.float32))
    out, sc = _run(xd, m, k, B.TERN_FWHT_DECODE, sd)
    vals, aux = O.decode_operand(ref)
    assert np.array_equal(f16_bits(out), vals.view(np.uint16))
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), aux.view(np.uint32))
    # unaligned sign pointer (the header allows it)
    buf = torch.zeros(k + 1, dtype=torch.int8, device="cuda")
    buf[1:] = sd
    out2, _ = _run(xd, m, k, B.TERN_FWHT_F32, buf[1:])
    assert np.array_equal(out2.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_degenerate_inputs():
    k = 2048
    x = np.zeros((6, k), np.float32)
    x[1] = 3.0e30                      # huge, same sign everywhere
    x[2, 7] = -1.0e-30                 # one tiny value
    x[3, ::2] = 1.0
    x[3, 1::2] = -1.0
    x[4, 3] = 1.0e-37                  # rotated values +-3e-39: a subnormal tscale
    x[5, 0], x[5, 1] = 3.0, 1.0        # rotated 4/32 and 2/32: v / tscale next to 63.5
    from ternary_weight_linear_block_gb300.inputs import to_bf16_bits, bf16_bits_to_f32
    bits = to_bf16_bits(x)
    xf = bf16_bits_to_f32(bits)
    xd = to_dev_bf16(bits)
    out, _ = _run(xd, 6, k, B.TERN_FWHT_F32)
    ref = O.fwht_f32(xf)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    out, sc = _run(xd, 6, k, B.TERN_FWHT_DECODE)
    vals, aux = O.decode_operand(ref)
    assert np.array_equal(f16_bits(out), vals.view(np.uint16))
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), aux.view(np.uint32))
    out, sc = _run(xd, 6, k, B.TERN_FWHT_F16)
    vals, inv = O.f16_operand(ref)
    assert np.array_equal(f16_bits(out), vals.view(np.uint16))
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), inv.view(np.uint32))
    out, sc = _run(xd, 6, k, B.TERN_FWHT_I8)
    xq, ts = O.quant_tokens(ref)
    assert np.array_equal(out.cpu().float().numpy(), xq.astype(np.float32))
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), ts.view(np.uint32))
    assert ts[0] == 0 and not xq[0].any()
    assert 0 < ts[4] < np.finfo(np.float32).tiny      # the subnormal case is exercised
    assert set(np.unique(np.abs(xq[5]))) <= {0, 63, 64, 127}


def test_m_zero_is_a_noop():
    out = poison(torch.empty(16, dtype=torch.float32, device="cuda"))
    B.tern_fwht_quant(out, 0, 1024, None, B.TERN_FWHT_F32, out, None)
    torch.cuda.synchronize()
    assert (out.view(torch.int32) == -1).all()
