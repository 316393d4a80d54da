"""bf16 rounding on NumPy float32 arrays (test infrastructure only).

bf16 keeps the top 16 bits of an IEEE binary32 value; rounding to nearest,
ties to even, is the rounding a bf16 decoder applies when it stores a tensor.
"""
import numpy as np


def round_bf16(x) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even); returns
    float32 holding bf16-representable values.  Finite inputs only."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    b = x.view(np.uint32).astype(np.uint64)
    bias = ((b >> 16) & 1) + 0x7FFF
    r = ((b + bias) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).reshape(x.shape)


def bits_bf16(x) -> np.ndarray:
    """uint16 bit patterns of bf16-representable float32 values."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def from_bits(u16) -> np.ndarray:
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


def mm(a, w) -> np.ndarray:
    """a @ w.T accumulated in float64, rounded once to float32."""
    return (np.asarray(a, np.float64) @ np.asarray(w, np.float64).T).astype(np.float32)
