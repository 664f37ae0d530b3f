"""Test-side MXFP4 packing, written independently of the oracle's decoder.

A dense float64 matrix whose entries are exactly E2M1 values times a per-32-block power
of two is turned into packed bytes (low nibble = even K index) and E8M0 scale bytes by
table inversion; the tests then compare oracle results on the packed form with dense
float64 matmuls on the matrix itself.
"""

import numpy as np

E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
_POS = {v: c for c, v in enumerate(E2M1_TABLE[:8])}


def random_mx_matrix(rng, rows, cols, exp_lo=-8, exp_hi=-4):
    """(dense float64 [rows, cols], codes [rows, cols] 0..15, exps [rows, cols/32])."""
    codes = rng.integers(0, 16, size=(rows, cols))
    exps = rng.integers(exp_lo, exp_hi + 1, size=(rows, cols // 32))
    vals = np.array(E2M1_TABLE)[codes] * np.repeat(2.0 ** exps, 32, axis=1)
    return vals, codes, exps


def pack(codes, exps):
    """Pack codes [R, K] (0..15) and block exponents [R, K/32] into (q uint8, s uint8)."""
    codes = np.asarray(codes, dtype=np.uint8)
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    s = (np.asarray(exps) + 127).astype(np.uint8)
    return q, s


def encode_dense(w, exps):
    """Inverse of the dense construction: codes from values given the block exponents."""
    scaled = w / np.repeat(2.0 ** np.asarray(exps), 32, axis=1)
    codes = np.zeros(w.shape, dtype=np.uint8)
    for v, c in _POS.items():
        codes[np.abs(scaled) == v] = c
    codes |= np.where(np.signbit(scaled), 8, 0).astype(np.uint8)
    return pack(codes, exps)
