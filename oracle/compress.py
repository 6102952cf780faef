"""Compressed shared pool: int8 keys, 3-bit rotated values (test oracle).

Follows the PolyKV summary, section 2B ("Asymmetrisch Compressieschema"):

* keys: int8 with one linear scale per tensor (item 1);
* values: rotate with a fast Walsh-Hadamard transform so the coordinates are
  close to a unit normal, map each coordinate to the nearest of the 8
  Lloyd-Max levels for N(0,1), and decode by looking the levels up and
  applying the inverse transform (item 2);
* the code-bit ratio against bf16 is ``16 / ((8 + 3) / 2)`` (same section,
  "Compressieverhouding").

Readings where the page is silent:

* "per tensor" = one scale for all keys (every token and kv head) of one
  layer: ``scale = max|K| / 127`` stored as fp32 (1.0 when all keys are 0);
  codes ``clamp(round_half_even(K / scale), -127, 127)``; -128 unused.
* The rotation is the unnormalised Sylvester Hadamard ``H`` (entries +-1,
  ``H H = d I``), no random sign flips.  A vector ``v`` keeps its norm
  ``n = |v|`` (fp32) and is coded as ``z = H v / n`` whose coordinates have
  unit RMS; decoding is ``v_hat = n * H z_hat / d``.  ``n = 0`` decodes to 0.
* Levels are the classical 8-level Lloyd-Max quantiser of a unit normal
  (J. Max, "Quantizing for minimum distortion", 1960); the decision
  boundaries are the midpoints between levels and a value exactly on a
  boundary takes the upper level.
* Bit packing: three bit planes of ``d/8`` bytes; plane ``b`` holds bit ``b``
  of every code, code ``i`` at bit ``i % 8`` of byte ``i // 8``.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

LLOYD_MAX_N01_8 = np.array([-2.1520, -1.3439, -0.7560, -0.2451,
                            0.2451, 0.7560, 1.3439, 2.1520], dtype=np.float64)
LLOYD_MAX_BOUNDARIES = 0.5 * (LLOYD_MAX_N01_8[1:] + LLOYD_MAX_N01_8[:-1])


def compression_ratio(base_bits: int = 16, k_bits: int = 8,
                      v_bits: int = 3) -> float:
    """Code-bit ratio of the asymmetric scheme against a ``base_bits`` cache."""
    return base_bits / ((k_bits + v_bits) / 2.0)


def fwht(x: np.ndarray) -> np.ndarray:
    """Unnormalised fast Walsh-Hadamard transform along the last axis.

    Butterfly in natural (Sylvester) order: equals ``x @ H`` with
    ``H[i, j] = (-1)^popcount(i & j)``.
    """
    y = np.array(x, dtype=np.float64, copy=True)
    n = y.shape[-1]
    if n & (n - 1):
        raise ValueError("FWHT length must be a power of two")
    h = 1
    while h < n:
        y = y.reshape(y.shape[:-1] + (n // (2 * h), 2, h))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(y.shape[:-3] + (n,))
        h *= 2
    return y


def k_int8_scale(k: np.ndarray) -> np.float32:
    """Per-tensor key scale ``max|K| / 127`` as fp32 (1.0 for an all-zero K)."""
    m = float(np.max(np.abs(np.asarray(k, dtype=np.float64)))) if np.size(k) else 0.0
    if m == 0.0:
        return np.float32(1.0)
    return np.float32(m / 127.0)


def k_int8_encode(k: np.ndarray, scale) -> np.ndarray:
    """``clamp(round_half_even(K / scale), -127, 127)`` as int8."""
    qk = np.rint(np.asarray(k, dtype=np.float64) / float(np.float32(scale)))
    return np.clip(qk, -127, 127).astype(np.int8)


def k_int8_decode(qk: np.ndarray, scale) -> np.ndarray:
    return np.asarray(qk, dtype=np.float64) * float(np.float32(scale))


def v3_encode(v: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Codes ``[..., d]`` (uint8, 0..7) and fp32 norms ``[...]`` of ``v``."""
    v = np.asarray(v, dtype=np.float64)
    n = np.sqrt(np.sum(v * v, axis=-1))
    hv = fwht(v)
    safe = np.where(n > 0, n, 1.0)
    z = np.where(n[..., None] > 0, hv / safe[..., None], 0.0)
    idx = np.searchsorted(LLOYD_MAX_BOUNDARIES, z, side="right")
    return idx.astype(np.uint8), n.astype(np.float32)


def v3_decode(codes: np.ndarray, norms: np.ndarray) -> np.ndarray:
    """``v_hat = n * H z_hat / d`` with ``z_hat`` the looked-up levels."""
    zh = LLOYD_MAX_N01_8[np.asarray(codes, dtype=np.int64)]
    d = zh.shape[-1]
    return np.asarray(norms, dtype=np.float64)[..., None] * fwht(zh) / d


def pack_planes(codes: np.ndarray) -> np.ndarray:
    """``[..., d]`` 3-bit codes -> ``[..., 3*d/8]`` uint8 bit planes."""
    c = np.asarray(codes, dtype=np.uint8)
    d = c.shape[-1]
    planes = []
    for b in range(3):
        bits = (c >> b) & 1                                   # [..., d]
        bits = bits.reshape(c.shape[:-1] + (d // 8, 8))
        weights = (1 << np.arange(8)).astype(np.uint16)
        planes.append((bits.astype(np.uint16) * weights).sum(-1).astype(np.uint8))
    return np.concatenate(planes, axis=-1)


def unpack_planes(packed: np.ndarray, d: int) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    nb = d // 8
    codes = np.zeros(p.shape[:-1] + (d,), dtype=np.uint8)
    for b in range(3):
        plane = p[..., b * nb:(b + 1) * nb]
        bits = (plane[..., :, None] >> np.arange(8, dtype=np.uint8)) & 1
        codes |= (bits.reshape(p.shape[:-1] + (d,)) << b).astype(np.uint8)
    return codes


def encode_pages(pages_k, pages_v, slot_fill: np.ndarray):
    """Encode a layer's page store ``[n, P, H_kv, d]``.

    The key scale is taken over the filled rows of every page (the layer's
    whole key tensor).  Returns ``(kq int8 [n,P,H,d], k_scale fp32,
    vcodes uint8 [n,P,H,d], vnorm fp32 [n,P,H])``; unfilled rows are coded
    as zeros.
    """
    from .residual_attention import _f64
    pk, pv = _f64(pages_k), _f64(pages_v)
    n, P = pk.shape[:2]
    live = (np.arange(P)[None, :] < np.asarray(slot_fill)[:, None])  # [n, P]
    k_live = pk[live]
    scale = k_int8_scale(k_live)
    kq = np.where(live[..., None, None], k_int8_encode(pk, scale), 0).astype(np.int8)
    codes, norms = v3_encode(pv)
    codes = np.where(live[..., None, None], codes, 0).astype(np.uint8)
    norms = np.where(live[..., None], norms, 0).astype(np.float32)
    return kq, scale, codes, norms


def decode_pages(kq, k_scale, vcodes, vnorm):
    """Dequantised ``(K_hat, V_hat)`` page stores (float64)."""
    return k_int8_decode(kq, k_scale), v3_decode(vcodes, vnorm)
