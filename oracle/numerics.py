"""Scalar numerics for the oracle (test infrastructure only; see ``oracle/__init__``).

All functions take and return float64 numpy arrays.
"""

import numpy as np


def f64(a):
    """Exact upcast of whatever the kernels consume (bf16 / fp32 / int) to float64."""
    return np.asarray(a, dtype=np.float64)


def round_f32(x):
    """Round float64 values to the nearest float32 (IEEE round-to-nearest-even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_bf16(x):
    """Round to bfloat16 the way a kernel that computes in fp32 and stores bf16 does.

    bfloat16 is the upper half of an IEEE-754 binary32 word (1 sign, 8 exponent,
    7 fraction bits).  The value is first rounded to float32, then the low 16
    bits of the float32 pattern are rounded away to nearest, ties to even.
    Finite inputs only (the path never produces NaN).
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    keep_lsb = (bits >> np.uint64(16)) & np.uint64(1)
    bits = (bits + np.uint64(0x7FFF) + keep_lsb) & np.uint64(0xFFFF0000)
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def sigmoid(z):
    """Logistic function 1 / (1 + e^-z)."""
    z = f64(z)
    return 1.0 / (1.0 + np.exp(-z))


def softplus(z):
    """softplus(z) = log(1 + e^z), evaluated without overflow."""
    return np.logaddexp(0.0, f64(z))


def silu(z):
    """SiLU (swish): z * sigmoid(z)."""
    z = f64(z)
    return z * sigmoid(z)
