"""Number formats of the W4A8 MXFP4 experts and the FP8 LM head, from their bit fields.

Test infrastructure (see ``oracle/__init__.py``): only tests, smoke() and the bench's
CPU-baseline legs use this module.

The pages name the formats only ("Humming MXFP4 kernels compile at run time for the
model's real shapes": the official W4A8 recipe with MXFP4 MoE kernels; "Online FP8
quantization halves the LM head weight reads": FP8 head; runbyai.xyz/posts/593 para. 3:
the head is stored in BF16). The bit layouts written out below are the published OCP
definitions of those names:

* E2M1 (MXFP4 element): 1 sign bit (bit 3), 2 exponent bits (bits 2-1, bias 1),
  1 mantissa bit (bit 0). Exponent 0 is subnormal: value = mantissa * 0.5.
  Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* E8M0 (MX block scale): 8 exponent bits, bias 127, no sign, no mantissa;
  value 2**(e - 127); 255 is NaN.
* E4M3 "fn" (FP8): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; no infinities;
  S.1111.111 is NaN; largest finite 448; exponent 0 is subnormal with value m/8 * 2**-6.
* BF16: the upper 16 bits of an IEEE binary32.

Quantisers (activations, the SwiGLU output and the LM head) are defined as IEEE binary32
operations followed by a round-to-nearest-even, saturating conversion to E4M3; they are
emulated here in numpy float32 so the codes are exact, not approximations.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0

# ----------------------------------------------------------------------------- decode


def e2m1_to_float(codes) -> np.ndarray:
    """Decode 4-bit E2M1 codes (low 4 bits of each integer) to float64."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    normal = np.ldexp(1.0 + 0.5 * m, (e - 1).astype(np.int64))  # 2^(e-1) * (1 + m/2)
    sub = 0.5 * m                                               # 2^(1-1) * (m/2)
    return sign * np.where(e == 0, sub, normal)


def e8m0_to_float(bytes_) -> np.ndarray:
    """Decode E8M0 scale bytes to float64 (255 -> NaN)."""
    b = np.asarray(bytes_).astype(np.int64) & 0xFF
    v = np.ldexp(1.0, b - 127)
    return np.where(b == 255, np.nan, v)


def e4m3_to_float(bytes_) -> np.ndarray:
    """Decode E4M3 (fn variant) bytes to float64 (S.1111.111 -> NaN)."""
    b = np.asarray(bytes_).astype(np.int64) & 0xFF
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, e - 7)
    sub = np.ldexp(m / 8.0, -6)
    v = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((b & 7) == 7), np.nan, v)


# Lookup tables built from the decoders above (a convenience for speed on large arrays;
# each entry is the decoder's own output).
E2M1_LUT = e2m1_to_float(np.arange(16))
E4M3_LUT = e4m3_to_float(np.arange(256))

# ----------------------------------------------------------------------------- encode


def float_to_e4m3_rne_sat(v) -> np.ndarray:
    """Round float32 values to E4M3 codes: round to nearest, ties to even, saturating.

    Saturation ("satfinite"): a magnitude above 448 becomes 448, never NaN. The sign of a
    zero result follows the sign bit of the input (IEEE conversions keep it).
    The quotient a/q below is exact (q is a power of two) and ``np.rint`` rounds half to
    even, so the result is the correctly rounded E4M3 value.
    """
    v32 = np.asarray(v, dtype=np.float32)
    a = np.abs(v32.astype(np.float64))
    neg = np.signbit(v32)
    _, ex = np.frexp(a)                           # a = f * 2^ex, f in [0.5, 1)
    # quantum: 2^(floor(log2 a) - 3) in the normal range (a >= 2^-6), 2^-9 below it
    q = np.where(a >= 2.0 ** -6, np.ldexp(1.0, ex - 1 - 3), 2.0 ** -9)
    r = np.rint(a / q) * q
    r = np.minimum(r, E4M3_MAX)
    # encode the (now representable) magnitude r
    _, ex2 = np.frexp(np.where(r > 0, r, 1.0))
    p = ex2 - 1                                   # floor(log2 r)
    is_sub = r < 2.0 ** -6
    e_field = np.where(is_sub, 0, p + 7)
    m_field = np.where(is_sub, r / 2.0 ** -9, (np.ldexp(r, -p) - 1.0) * 8.0)
    code = (e_field.astype(np.int64) << 3) | np.rint(m_field).astype(np.int64)
    code = np.where(r == 0, 0, code)
    code = code | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)


def f32_to_bf16_bits(v) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns the 16-bit patterns."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def bf16_bits_to_float(b) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_f64_to_bf16(v) -> np.ndarray:
    """Round float64 values directly to the nearest bf16 (ties to even); returns float32.

    bf16 keeps 8 significant bits; rounding the float64 significand once avoids the
    double rounding of a float64 -> float32 -> bf16 chain. Values stay in the normal
    range for every use here (hidden states of order 1..1e4).
    """
    v = np.asarray(v, dtype=np.float64)
    f, e = np.frexp(v)                  # v = f * 2^e, |f| in [0.5, 1)
    r = np.ldexp(np.rint(np.ldexp(f, 8)), e - 8)
    return r.astype(np.float32)


# ----------------------------------------------------------------------------- quantiser


def quantize_fp8_lastdim(v):
    """Per-vector dynamic FP8 quantisation along the last axis, in emulated float32.

    For each vector: amax = max |v| (exact); scale = float32(amax) / float32(448),
    correctly rounded; t = float32(v) / scale, correctly rounded; code = E4M3(t) with
    round-to-nearest-even and saturation. An all-zero vector gets scale 1 and all-zero
    codes. Returns (codes uint8 [..., K], scale float32 [...]).

    This is the "dynamic FP8 quantization" of the LM head ("Online FP8 quantization
    halves the LM head weight reads", one scale per vocabulary row) and the per-token
    activation quantisation of the W4A8 recipe ("Humming MXFP4 kernels ...": the A8 half).
    """
    v32 = np.asarray(v, dtype=np.float32)
    amax = np.max(np.abs(v32), axis=-1)
    scale = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32),
                     np.float32(1.0)).astype(np.float32)
    t = (v32 / scale[..., None]).astype(np.float32)
    return float_to_e4m3_rne_sat(t), scale
