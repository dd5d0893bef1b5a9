"""FP8 E4M3 codec and per-(token, KV head) quantisation of K/V (NumPy). Test infrastructure only.

Reading of the pages: quantising the KV cache is one of the cache strategies and changes how it is
stored ("¿Cuánta memoria reservar para la caché KV?", "Adaptar el presupuesto a la estrategia de
caché"); changing the K/V precision can change the numerics, so it gets its own contract ("Servicio
de modelos de lenguaje con un presupuesto de memoria" §4 and §6).

Format (OCP FP8 E4M3, the "fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no
infinities; S.1111.111 is NaN; largest finite 448; subnormals m * 2^-9.

Quantisation (the library's reading, per stored row of D values of one token and one KV head):
    amax  = max |x|                         (float32, exact)
    scale = amax / 448 in float32 (IEEE round to nearest), 1 when amax == 0
    code  = e4m3(x / scale), x / scale in float32 (IEEE), rounded to nearest even, saturated to ±448
and the dequantised value is decode(code) * scale.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

MAX_FINITE = 448.0


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """uint8 codes -> float64 values, from the bit layout."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.power(2.0, e - 7))
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return sign * val


_POS_CODES = np.arange(0x7F, dtype=np.uint8)          # 0x00 .. 0x7E: all non-negative finite codes
_POS_VALUES = decode_e4m3(_POS_CODES)                  # strictly increasing


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """float values -> uint8 codes: round to nearest, ties to the even code, saturate to ±448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), MAX_FINITE)
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, len(_POS_VALUES) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALUES) - 1)
    d_hi = _POS_VALUES[hi] - a
    d_lo = a - _POS_VALUES[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & ((_POS_CODES[lo] & 1) == 0))
    code = np.where(pick_lo, _POS_CODES[lo], _POS_CODES[hi]).astype(np.uint8)
    code = np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def quantize_rows(x: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """x float32 [..., D] -> (codes uint8 [..., D], scale float32 [...]) with the rules above."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(MAX_FINITE), np.float32(1.0)).astype(np.float32)
    y = (x / scale[..., None]).astype(np.float32)
    return encode_e4m3(y), scale


def dequantize(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """decode(codes) * scale in float64 (exact: a 4-bit significand times a float32)."""
    return decode_e4m3(codes) * np.asarray(scale, dtype=np.float64)[..., None]


# Byte position, within a 16-token group of a dim-major V page, of token j (a layout convention of
# the library's fp8 pools): the group is stored in the token order 0,1,8,9,2,3,10,11,4,5,12,13,6,7,14,15.
V_GROUP_ORDER = [0, 1, 8, 9, 2, 3, 10, 11, 4, 5, 12, 13, 6, 7, 14, 15]
V_POSITION = [V_GROUP_ORDER.index(j) for j in range(16)]


def v_byte_offset(off: int) -> int:
    """Byte position of in-block token offset ``off`` in a dim-major V page row."""
    return (off - off % 16) + V_POSITION[off % 16]


def reshape_and_cache_fp8(k8: np.ndarray, ks: np.ndarray, v8t: np.ndarray, vs: np.ndarray, k: np.ndarray,
                          v: np.ndarray, slots) -> None:
    """Quantise new K/V rows and scatter them into an fp8 pool, in place.

    Layout (the library's): k8 [NB][Hkv][B][D] codes, v8t [NB][Hkv][D][B] codes (V stored dim-major
    within a page, 16-token groups in the order V_GROUP_ORDER), ks / vs [NB][Hkv][B] float32 scales.
    k, v: [n_tokens][Hkv][D] float32 values (decoded bf16 inputs). A negative slot skips its token.
    """
    B = k8.shape[2]
    kc, ksc = quantize_rows(k)
    vc, vsc = quantize_rows(v)
    for i, s in enumerate(slots):
        s = int(s)
        if s < 0:
            continue
        blk, off = s // B, s % B
        k8[blk, :, off, :] = kc[i]
        ks[blk, :, off] = ksc[i]
        v8t[blk, :, :, v_byte_offset(off)] = vc[i]
        vs[blk, :, off] = vsc[i]


def dequantize_pool(k8: np.ndarray, ks: np.ndarray, v8t: np.ndarray, vs: np.ndarray):
    """float64 K and V caches in the standard [NB][Hkv][B][D] layout from an fp8 pool."""
    K = decode_e4m3(k8) * ks.astype(np.float64)[..., None]
    B = v8t.shape[3]
    tok_order = np.array([v_byte_offset(off) for off in range(B)])
    V = decode_e4m3(np.swapaxes(v8t[..., tok_order], 2, 3)) * vs.astype(np.float64)[..., None]
    return K, V
