"""Oracle number formats — TEST INFRASTRUCTURE (see the package docstring).

The pages name the formats (a four-bit "tiled" matrix with per-32-column
groups, int8 activations, an eight-bit head) but never spell out their
encodings; these are the readings this oracle fixes:

* 4-bit weights, group 32 along K: per output row n and group g,
  ``s = f16(max|w| / 7)`` (the division in f32, then round-to-nearest-even to
  f16), ``q = clamp(rint(w / f32(s)), -8, 7)``; a group whose f16 scale is 0
  has ``q = 0``.
* int8 rows (activations feeding a matmul, and the head's rows):
  ``s = max|x| / 127`` in f32, ``q = clamp(rint(x / s), -127, 127)``, a zero
  row has ``s = 0, q = 0``.
* the quantised matvec (the int32 group sums are exact integers):
  ``acc[t,n,g] = sum_{k in g} qx[t,k] * qw[n,k]``,
  ``y[t,n] = sx[t] * sum_g f32(s[n,g]) * acc[t,n,g]``;
  the head: ``y[t,n] = sx[t] * sw[n] * sum_k qx[t,k] * qw[n,k]``.

Every decision that turns a float into an integer (the codes) is taken in
float32 with IEEE division and round-half-to-even, as a kernel takes it.
"""
from __future__ import annotations

import numpy as np

GROUP = 32


def quantize_rows_i8(x):
    """Symmetric int8 per row: returns (q int8 [..., K], s float32 [...])."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    s = (amax / np.float32(127)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1))
    q = np.rint(x32 / safe[..., None])
    q = np.where(s[..., None] > 0, q, 0)
    q = np.clip(q, -127, 127).astype(np.int8)
    return q, s


def quantize_q4g32(w):
    """4-bit weights, groups of 32 along the last axis.

    Returns (q int8 [N, K] with values in [-8, 7], s float16 [N, K // 32]).
    """
    w32 = np.asarray(w, dtype=np.float32)
    n, k = w32.shape
    if k % GROUP:
        raise ValueError(f"K = {k} is not a multiple of {GROUP}")
    wg = w32.reshape(n, k // GROUP, GROUP)
    amax = np.max(np.abs(wg), axis=-1)
    s16 = (amax / np.float32(7)).astype(np.float16)
    sf = s16.astype(np.float32)
    safe = np.where(sf > 0, sf, np.float32(1))
    q = np.rint(wg / safe[..., None])
    q = np.where(sf[..., None] > 0, q, 0)
    q = np.clip(q, -8, 7).astype(np.int8).reshape(n, k)
    return q, s16


def dequant_q4g32(q, s16, dtype=np.float32):
    """The real values a 4-bit matrix stands for: s * q (exact in f32)."""
    n, k = q.shape
    sf = np.asarray(s16, dtype=np.float32).astype(dtype)
    return (q.reshape(n, k // GROUP, GROUP).astype(dtype) * sf[..., None]).reshape(n, k)


def q4_group_sums(qx, qw):
    """The int32 group sums of the quantised matvec, by plain integer
    arithmetic: acc[t, n, g] = sum over the 32 columns k of group g of
    qx[t, k] * qw[n, k].  Returns int64 [T, N, K // 32]."""
    qx = np.asarray(qx, dtype=np.int64)
    qw = np.asarray(qw, dtype=np.int64)
    t, k = qx.shape
    n = qw.shape[0]
    g = k // GROUP
    xg = qx.reshape(t, g, GROUP)
    wg = qw.reshape(n, g, GROUP)
    out = np.zeros((t, n, g), dtype=np.int64)
    for gi in range(g):
        out[:, :, gi] = xg[:, gi, :] @ wg[:, gi, :].T
    return out


def q4_matvec_by_definition(qx, sx, qw, s16):
    """y[t, n] = sx[t] * sum_g s[n, g] * acc[t, n, g], summed in float64 in
    group order from the exact integer group sums."""
    acc = q4_group_sums(qx, qw).astype(np.float64)
    sf = np.asarray(s16, dtype=np.float32).astype(np.float64)
    y = np.einsum("tng,ng->tn", acc, sf)
    return y * np.asarray(sx, dtype=np.float32).astype(np.float64)[:, None]


def i8_matvec_by_definition(qx, sx, qw, sw):
    """The head: y[t, n] = sx[t] * sw[n] * sum_k qx[t, k] * qw[n, k] (exact
    integer sum, scales applied in float64)."""
    acc = np.asarray(qx, dtype=np.int64) @ np.asarray(qw, dtype=np.int64).T
    return (acc.astype(np.float64) * np.asarray(sx, dtype=np.float32).astype(np.float64)[:, None]
            * np.asarray(sw, dtype=np.float32).astype(np.float64)[None, :])
