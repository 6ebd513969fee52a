"""bfloat16 rounding for the oracle's BF16-operand mode (test infrastructure).

bfloat16 keeps the upper 16 bits of an IEEE float32.  Rounding a float32 to
the nearest bfloat16, ties to even, is integer arithmetic on the bit pattern:
add 0x7FFF plus the lowest kept bit, then drop the low 16 bits.  A carry out
of the mantissa correctly bumps the exponent (and turns the largest finite
values into infinity).  NaNs are kept quiet.  Written from the IEEE 754
definition of round-to-nearest-even; pinned against torch's own conversion.
"""
import numpy as np


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest bfloat16 (ties to even), returned as float32."""
    x = np.asarray(x)
    if x.dtype != np.float32:
        raise TypeError("round_bf16 takes float32 input; round wider values to "
                        "float32 first so the rounding sequence is explicit")
    u = x.view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)) & np.uint64(0xFFFF)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x0040)) & np.uint64(0xFFFF)
    return (r.astype(np.uint32) << np.uint32(16)).view(np.float32).reshape(x.shape)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bfloat16 bit patterns -> float32 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)
