"""KV compressor, RMSNorm and rotary position embedding, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows "DeepSeek V4 in vLLM: Efficient Long-context Attention":
* Background, "compressing the KV cache across tokens": a c4a entry is a
  weighted sum of 8 uncompressed tokens at stride 4, a c128a entry a weighted
  sum of 128 tokens at stride 128.
* Method details, kernel fusion (1): after compression the compressed K goes
  through RMSNorm, then RoPE, then into the cache (main or indexer).
* Appendix, "why inverse RoPE": R_m is an orthogonal rotation with
  R_m^T R_m = I and R_m R_n = R_{m+n}; the attention output is rotated back by
  R_m^{-1}.

Readings taken where the page is silent:
* Window weights: w = softmax_j(g[p_j] + b_j) over the window's positions
  p_j >= 0, with one scalar gate logit g per token and one bias b_j per
  window offset j.  Positions < 0 ("negative indices count as 0") contribute
  nothing and take no softmax weight (logit -inf).
* RMSNorm: c / sqrt(mean(c^2) + eps) * gamma, eps = 1e-6.
* RoPE acts on the last ``rope_dims`` dimensions in interleaved pairs
  (D-R+2j, D-R+2j+1), j = 0..R/2-1, with angle pos * theta^(-2j/R):
  [a, b] -> [a cos - b sin, a sin + b cos].  The inverse uses -angle.
"""
from __future__ import annotations

import numpy as np

RMS_EPS = 1e-6


def window_weights(gates: np.ndarray, bias: np.ndarray, valid: np.ndarray) -> np.ndarray:
    """Softmax over the valid window offsets of gate + per-offset bias."""
    logit = np.where(valid, gates + bias, -np.inf)
    mx = np.max(logit[valid])
    e = np.where(valid, np.exp(logit - mx), 0.0)
    return e / e.sum()


def compress_window(xs: np.ndarray, gates: np.ndarray, bias: np.ndarray,
                    valid: np.ndarray) -> np.ndarray:
    """Weighted sum of the window's token vectors xs[j] (rows)."""
    w = window_weights(gates, bias, valid)
    xs = np.where(valid[:, None], xs, 0.0)
    return w @ xs


def rms_norm(c: np.ndarray, gamma: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    return c / np.sqrt(np.mean(c * c) + eps) * gamma


def rope_angles(pos: float, rope_dims: int, theta: float) -> np.ndarray:
    j = np.arange(rope_dims // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * j / rope_dims)
    return float(pos) * inv_freq


def rope(v: np.ndarray, pos: float, rope_dims: int, theta: float,
         inverse: bool = False) -> np.ndarray:
    """Rotate the last ``rope_dims`` dims of v (last axis) by R_pos (or R_pos^-1)."""
    v = np.array(v, dtype=np.float64, copy=True)
    d = v.shape[-1]
    ang = rope_angles(pos, rope_dims, theta)
    if inverse:
        ang = -ang
    c, s = np.cos(ang), np.sin(ang)
    a = v[..., d - rope_dims + 0::2].copy()
    b = v[..., d - rope_dims + 1::2].copy()
    v[..., d - rope_dims + 0::2] = a * c - b * s
    v[..., d - rope_dims + 1::2] = a * s + b * c
    return v


def compressed_entry(x_of, g_of, i: int, ratio: int, bias: np.ndarray,
                     gamma: np.ndarray, rope_dims: int, theta: float,
                     eps: float = RMS_EPS) -> np.ndarray:
    """Entry i of one sequence before encoding.

    ``x_of(p)`` / ``g_of(p)`` return the compressor input vector / gate logit
    of native position p >= 0.
    """
    from .geometry import window_positions, anchor
    pos = window_positions(i, ratio)
    valid = np.array([p >= 0 for p in pos])
    xs = np.stack([x_of(p) if p >= 0 else np.zeros_like(gamma) for p in pos])
    gs = np.array([g_of(p) if p >= 0 else 0.0 for p in pos], dtype=np.float64)
    c = compress_window(xs, gs, np.asarray(bias, np.float64), valid)
    n = rms_norm(c, gamma, eps)
    return rope(n, anchor(i, ratio), rope_dims, theta)
