"""Comparison helpers for the parity tests (no step arithmetic)."""
import numpy as np


def ordered16(bits: np.ndarray) -> np.ndarray:
    """Map 16-bit sign-magnitude float patterns to integers ordered like the values."""
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_diff16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(ordered16(a) - ordered16(b))


def rel_err(got: np.ndarray, ref: np.ndarray, tiny: float = 1e-30) -> np.ndarray:
    """|got - ref| / |ref|, or the absolute difference where |ref| < tiny."""
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    d = np.abs(got - ref)
    return np.where(np.abs(ref) < tiny, d, d / np.maximum(np.abs(ref), tiny))


def scaled_err(got: np.ndarray, ref: np.ndarray, prev: np.ndarray, tiny: float = 1e-30) -> np.ndarray:
    """|got - ref| / max(|ref|, |prev|): the error relative to the larger of the
    result and the value it was computed from (the operands' scale)."""
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    scale = np.maximum(np.maximum(np.abs(ref), np.abs(prev.astype(np.float64))), tiny)
    d = np.abs(got - ref)
    return np.where(scale <= tiny, d, d / scale)
