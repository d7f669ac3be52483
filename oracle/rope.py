"""Oracle: rotary embedding at absolute positions and the paged K/V append.

Sources: "Chunked Prefill 的 Token 预算" (zwjcode.cn), section 07 -- a chunk's
position ids start at its absolute offset c and are never reset to 0, or the
rotary phase repeats and chunked prefill stops matching full prefill;
section 06 -- each new token's K/V goes to the physical slot named by
``slot_mapping``; "Chunked Prefill: Ending the Great Stall", section 05 -- the
paged blocks are filled token by token whatever chunk writes them.

Readings where the pages are silent (the plainest common form):

* rotate-half pairing (element i with element i + D/2), base 10000;
* the cos/sin table is computed in double precision with the C library
  (``math.cos``/``math.sin``/``**``) and rounded to fp32;
* each rotated element is three IEEE fp32 round-to-nearest operations
  (two products, then one sum or difference), never fused, then rounded to
  bf16 with round-to-nearest-even;
* the cache holds the rotated K and the unrotated V.

bf16 values are carried as uint16 bit patterns (numpy has no bf16 type).
"""
from __future__ import annotations

import math

import numpy as np


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exactly equal fp32 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_to_f32(bits).astype(np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest, ties to even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def rope_tables(positions, D: int, base: float = 10000.0):
    """cos and sin of p * base**(-2i/D) for the given positions, i < D/2, as fp32 [len, D/2]."""
    pos = [int(p) for p in np.asarray(positions).reshape(-1)]
    half = D // 2
    inv_freq = [base ** (-(2 * i) / D) for i in range(half)]
    cos = np.empty((len(pos), half), dtype=np.float32)
    sin = np.empty((len(pos), half), dtype=np.float32)
    for r, p in enumerate(pos):
        for i in range(half):
            ang = p * inv_freq[i]
            cos[r, i] = math.cos(ang)
            sin[r, i] = math.sin(ang)
    return cos, sin


def rope_rotate(x_bits: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate bf16 rows x [n, H, D] by per-row cos/sin [n, D/2]; returns bf16 bits.

    y[i]       = x[i] * cos_i - x[i + D/2] * sin_i
    y[i + D/2] = x[i + D/2] * cos_i + x[i] * sin_i
    """
    x = bf16_to_f32(x_bits)
    D = x.shape[-1]
    half = D // 2
    c = cos[:, None, :].astype(np.float32)
    s = sin[:, None, :].astype(np.float32)
    x1 = x[..., :half]
    x2 = x[..., half:]
    # numpy evaluates each float32 product and sum separately, rounding each
    y1 = np.subtract(np.multiply(x1, c), np.multiply(x2, s))
    y2 = np.add(np.multiply(x2, c), np.multiply(x1, s))
    y = np.concatenate([y1, y2], axis=-1).astype(np.float32)
    return f32_to_bf16_bits(y)


def kv_append(q_bits, k_bits, v_bits, positions, slot_mapping, k_pool_bits, v_pool_bits,
              page_size: int = 16, base: float = 10000.0):
    """Rotate q and k at their absolute positions and write k, v into the pools.

    q [T, H_q, D], k and v [T, H_kv, D] and the pools [P, H_kv, page, D] are
    bf16 bit arrays.  Slot -1 means "do not write".  Returns q_rot and the
    updated pools (copies).
    """
    D = q_bits.shape[-1]
    cos, sin = rope_tables(positions, D, base)
    q_rot = rope_rotate(q_bits, cos, sin)
    k_rot = rope_rotate(k_bits, cos, sin)
    kp = np.array(k_pool_bits, copy=True)
    vp = np.array(v_pool_bits, copy=True)
    for t, slot in enumerate(np.asarray(slot_mapping).reshape(-1)):
        slot = int(slot)
        if slot < 0:
            continue
        page, off = divmod(slot, page_size)
        kp[page, :, off, :] = k_rot[t]
        vp[page, :, off, :] = v_bits[t]
    return q_rot, kp, vp
