"""Storage-format rounding used by the oracle (test infrastructure only).

The bf16 configuration stores every weight as bfloat16.  The oracle widens
those stored values back to float and computes in fp64, so the only bf16
effect it models is the rounding of the weights themselves.
"""
import numpy as np


def round_to_bf16(x) -> np.ndarray:
    """Round fp32 values to the nearest bfloat16 (ties to even), returned as fp32.

    bfloat16 keeps the top 16 bits of an IEEE binary32 value.  Rounding to
    nearest-even adds 0x7FFF plus the lowest kept bit to the bit pattern
    before truncation.  Inputs are finite (no NaN handling is needed for
    weights drawn from a normal distribution).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    # finite inputs have u <= 0xFF7FFFFF, so adding at most 0x8000 cannot wrap
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32).reshape(x.shape)
