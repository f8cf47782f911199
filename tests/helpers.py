"""Small conversions shared by the tests (no arithmetic of the method)."""
import numpy as np
import torch


def bits(t: torch.Tensor) -> np.ndarray:
    """A bfloat16 tensor's bit patterns as a uint16 numpy array (CPU copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """uint16 bit patterns -> bfloat16 CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def f32(t) -> np.ndarray:
    return t.detach().cpu().float().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float32)
