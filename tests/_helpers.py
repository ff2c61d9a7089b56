"""Small conversions shared by the tests (no method arithmetic)."""
import numpy as np
import torch


def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> its uint16 bit patterns as a numpy array."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_from_float(x) -> np.ndarray:
    """Round float values to bf16 (torch's RNE cast) and return the bit patterns."""
    return bits16(torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def bf16_value(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)
