"""Oracle: the q/k prologue -- per-head RMSNorm with gain, then the 3D (t,h,w)
rotary embedding on the first 96 of 128 head dims ("rot96").

Follows
* [SPARK] "What this config does": the Q path is RMSNorm, then rot96 RoPE
  (the norm comes first, the rotation second);
* [PR26] encoder text-tower commit: per-head q/k RMSNorm (each head's
  128-vector is normalised on its own);
* [PR26] "The device-resident forward (W2b)": the rotary is plain NeoX
  rotate_half, only the angles are unusual -- three axes read off the fp64
  position grid through a per-row cos/sin cache;
* [PR26] device-encoder commit (M-RoPE note): the cache is cat(freqs, freqs),
  so cos/sin repeat across the two halves of the rotated dims;
* [PR26] video-VAE ViT3D commit: the per-axis frequency blocks are
  concatenated before being tiled twice over the rotated dims.

Readings where the pages are silent (each listed in the design notes):
* the 96 rotated dims are one NeoX block: dim j pairs with j + 48, and the 48
  angles are [t: 16 | h: 16 | w: 16];
* per-axis frequencies omega_k = base ** (-2k / 32), k = 0..15, base 10000;
* eps sits inside the square root: r = 1 / sqrt(mean(x^2) + eps);
* the gain is one fp32 [128] vector per tensor, shared across heads, or a
  [H, 128] array when given per head.

Everything is fp64 from the bf16 input values; no intermediate rounding.
Parity: pinned (rotation preserves the norm, relative-position property,
closed forms for unit inputs, the plain-RMSNorm special case).
"""
from __future__ import annotations

import numpy as np

N_AXES = 3


def axis_inv_freq(base: float, rope_dims: int) -> np.ndarray:
    """omega_k = base ** (-2k / d_axis) for k = 0 .. d_axis/2 - 1, d_axis = rope_dims / 3."""
    d_axis = rope_dims // N_AXES
    k = np.arange(d_axis // 2, dtype=np.float64)
    return np.float64(base) ** (-(2.0 * k) / d_axis)


def rope_angles(pos: np.ndarray, base: float = 10000.0, rope_dims: int = 96) -> np.ndarray:
    """fp64 [S, rope_dims/2]: theta = p_axis * omega_k, blocks ordered t, h, w."""
    w = axis_inv_freq(base, rope_dims)
    return np.concatenate([pos[:, a:a + 1] * w[None, :] for a in range(N_AXES)], axis=1)


def rms_norm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """y = x * gain / sqrt(mean_j x_j^2 + eps) over the last axis (one head).

    x: [S, H, D]; gain: [D] (shared by all heads) or [H, D]."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(ms + eps)
    g = gain[None, None, :] if gain.ndim == 1 else gain[None, :, :]
    return x * r * g


def apply_rope(y: np.ndarray, theta: np.ndarray, rope_dims: int = 96) -> np.ndarray:
    """NeoX rotate-half on dims [0, rope_dims): y*cos + rotate_half(y)*sin,
    rotate_half(a, b) = (-b, a), cos/sin = cat(cos theta, cos theta).
    Dims >= rope_dims are returned unchanged.  theta: [S, rope_dims/2]."""
    half = rope_dims // 2
    c = np.cos(theta)[:, None, :]
    s = np.sin(theta)[:, None, :]
    a = y[..., :half]
    b = y[..., half:rope_dims]
    out = y.copy()
    out[..., :half] = a * c - b * s
    out[..., half:rope_dims] = b * c + a * s
    return out


def qk_prologue(x: np.ndarray, gain: np.ndarray, pos: np.ndarray, eps: float = 1e-6,
                base: float = 10000.0, rope_dims: int = 96) -> np.ndarray:
    """RMSNorm (with gain) then rot96 rotary, fp64.  x: [S, H, 128]."""
    return apply_rope(rms_norm(x, gain, eps), rope_angles(pos, base, rope_dims), rope_dims)
