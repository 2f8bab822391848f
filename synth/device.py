"""Moving the seeded bf16 bit patterns to and from torch tensors (no arithmetic)."""
from __future__ import annotations

import numpy as np
import torch

from . import bf16_bits_to_f64


def bf16_to_torch(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t


def torch_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def torch_bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return bf16_bits_to_f64(torch_to_bits(t))
