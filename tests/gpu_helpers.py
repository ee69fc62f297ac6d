"""Shared helpers for the GPU parity tests (marshalling only)."""

import numpy as np
import torch

from ternary_weight_linear_block_gb300 import binding as B
from ternary_weight_linear_block_gb300 import build as BUILD


def ensure_lib():
    BUILD.ensure_built()          # missing, or older than a source file
    return B.lib()


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def poison(t: torch.Tensor) -> torch.Tensor:
    """Fill a tensor with a NaN-like byte pattern so untouched outputs show."""
    t.view(torch.uint8).fill_(0xFF)
    return t


def f16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy()
