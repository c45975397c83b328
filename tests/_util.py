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


def ulp16_at(bits: np.ndarray, dtype_is_bf16: bool) -> np.ndarray:
    """Spacing of the 16-bit format at each value's magnitude (subnormal floor)."""
    b = bits.astype(np.int64) & 0x7FFF
    if dtype_is_bf16:
        e = b >> 7
        return np.ldexp(1.0, np.maximum(e, 1) - 127 - 7)
    e = b >> 10
    return np.ldexp(1.0, np.maximum(e, 1) - 15 - 10)


def params_close(got_bits, ref_bits, ref_vals, got_vals, master_err_bound, dtype_is_bf16):
    """Cast-out params agree within 1 ulp, or -- where the master itself sits
    at a cancellation -- within 1 ulp plus the master's allowed error."""
    ulp = ulp16_at(ref_bits, dtype_is_bf16)
    diff = np.abs(got_vals.astype(np.float64) - ref_vals.astype(np.float64))
    return (ulp_diff16(got_bits, ref_bits) <= 1) | (diff <= ulp + master_err_bound)
