"""FP8 E4M3 codec written from the OCP 8-bit floating point format definition (oracle).

The pages fix only that an FP8 KV cache is a byte container viewed as the
platform FP8 type, with a per-layer k_scale / v_scale that the write side and
the read side must interpret the same way ("vLLM 源码完全拆解（六）：Attention
Backend", section «KV Cache 视图必须匹配 Kernel ABI»; "SGLang 源码完全拆解(八)：
Attention Backend", section «层与后端的边界»: set_kv_buffer(..., k, v,
*kv_write_scales)).  The reading taken here:

* real value = decode(code) * scale;
* code = encode(float32(x) * inv_scale), with inv_scale = float32(1) / float32(scale)
  and the product rounded once to float32;
* encode rounds to nearest, ties to even, and saturates finite overflow to
  +-448 (there is no infinity in E4M3); NaN encodes to 0x7F.

E4M3 layout: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.
Exponent field 0 is subnormal (m * 2^-9); S.1111.111 is NaN; the largest
finite magnitude is 1.75 * 2^8 = 448; the smallest normal is 2^-6.
"""

from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0
MIN_NORMAL = 2.0 ** -6
SUBNORMAL_QUANTUM = 2.0 ** -9
NAN_CODE = 0x7F


def decode(codes) -> np.ndarray:
    """Exact float64 value of each E4M3 code (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * SUBNORMAL_QUANTUM, (8 + m) * np.exp2(e.astype(np.float64) - 10.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def decode_table() -> np.ndarray:
    """All 256 codes decoded, indexed by code."""
    return decode(np.arange(256))


def encode(x) -> np.ndarray:
    """Round float values to E4M3 codes: nearest-even, saturate to +-448, NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    # exponent of the binade holding a: a = f * 2^E, f in [0.5, 1) -> a in [2^(E-1), 2^E)
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    e = E.astype(np.int64) - 1
    normal = a >= MIN_NORMAL
    quantum = np.where(normal, np.exp2(np.clip(e, -6, 8).astype(np.float64) - 3.0), SUBNORMAL_QUANTUM)
    q = np.rint(a / quantum) * quantum  # np.rint rounds halves to even
    q = np.minimum(q, MAX_FINITE)
    q = np.where(a > MAX_FINITE, MAX_FINITE, q)
    # bits of the rounded magnitude
    _, Eq = np.frexp(np.where(q > 0, q, 1.0))
    eq = Eq.astype(np.int64) - 1
    is_sub = q < MIN_NORMAL
    sub_bits = np.rint(q / SUBNORMAL_QUANTUM).astype(np.int64)
    man = np.rint(q / np.exp2(eq.astype(np.float64) - 3.0)).astype(np.int64) - 8
    norm_bits = ((eq + 7) << 3) | man
    bits = np.where(is_sub, sub_bits, norm_bits)
    bits = np.where(neg, bits | 0x80, bits)
    bits = np.where(nan, NAN_CODE, bits)
    return bits.astype(np.uint8)


def quantize(x_fp32, scale: float) -> np.ndarray:
    """Store side: code = encode(float32(x) * float32(1 / scale)), product rounded to float32."""
    inv = np.float32(1.0) / np.float32(scale)
    prod = (np.asarray(x_fp32, dtype=np.float32) * inv).astype(np.float32)
    return encode(prod.astype(np.float64))


def dequantize(codes, scale: float) -> np.ndarray:
    """Read side: real = decode(code) * scale, in float64."""
    return decode(codes) * np.float64(np.float32(scale))
