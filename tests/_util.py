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


# ---------------------------------------------------------------------------
# How often the relaxed checks are needed
# ---------------------------------------------------------------------------
# The fp32-state check scales the error by the largest magnitude an element
# has held, and the parameter check allows the master's error on top of
# 1 ulp. Both relaxations are meant for the few elements an update cancels
# towards zero. Every check records how many elements needed them, and
# asserts a cap, so that an error spread over many elements cannot pass as
# "cancellation".
TOL_STATS = []
# Per tensor: at most this fraction of the checked elements (or FLOOR
# elements, for small tensors) may fail the plain element-wise bar (1e-5
# relative for master/m/v, 1 ulp for the parameters). Measured on GB300 over
# the whole GPU suite, the worst check had 0.19 % of masters, 0.73 % of m
# (the 300-step mixed run: m = 0.9 m + 0.1 g cancels often), no v and 2 of
# 620K parameters; the caps are about 2.5 times those. v has no cancellation
# (every term is non-negative), so it must pass the plain bar everywhere.
PLAIN_FAIL_CAP = {"master": (5e-3, 32), "m": (2e-2, 32), "v": (0.0, 0), "params": (1e-5, 4)}


def record_plain(where: str, name: str, n_checked: int, plain_fail: int, max_plain: float) -> dict:
    import os
    rec = {"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], "where": where,
           "tensor": name, "n": int(n_checked), "plain_fail": int(plain_fail),
           "max_plain": float(max_plain)}
    TOL_STATS.append(rec)
    frac, floor = PLAIN_FAIL_CAP[name]
    cap = max(floor, frac * n_checked)
    if os.environ.get("ZERO_TOL_CAP", "on") != "off":  # "off": record the counts only
        assert plain_fail <= cap, (f"{name}: {plain_fail} of {n_checked} elements fail the plain "
                                   f"element-wise bar (cap {cap:.0f})")
    return rec


def plain_state_stats(where, name, got, ref, rtol):
    """Elements of an fp32 state tensor beyond rtol in plain relative error."""
    plain = rel_err(got, ref)
    bad = plain > rtol
    return record_plain(where, name, got.size, int(bad.sum()),
                        float(plain[bad].max()) if bad.any() else 0.0)


def plain_param_stats(where, got_bits, ref_bits, mask=None):
    """Cast-out params more than 1 ulp from the oracle's (plain check)."""
    d = ulp_diff16(got_bits, ref_bits)
    if mask is not None:
        d = d[mask]
    bad = d > 1
    return record_plain(where, "params", d.size, int(bad.sum()), float(d.max()) if d.size else 0.0)
