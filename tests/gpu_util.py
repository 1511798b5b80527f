"""Helpers shared by the GPU tests (no arithmetic of the method here)."""
import numpy as np
import pytest
import torch


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_verification_gb300 import build
    build.build()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bfloat16 tensor (any device)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def np_(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def rand_codes(shape, seed, lo=-127, hi=127):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int8)


def rand_scales(n, seed, lo=1e-4, hi=1e-2):
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(n, generator=g, dtype=torch.float64) * (hi - lo) + lo).to(torch.float32)
