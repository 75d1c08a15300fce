"""Shared-K=V sparse attention and the inverse-RoPE output stage, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows "DeepSeek V4 in vLLM: Efficient Long-context Attention":
* Background: keys and values share one vector per cached entry; the
  attention output is rotated back by inverse RoPE (appendix "why inverse
  RoPE": with v_n = k_n = R_n k the output carries absolute position, and
  R_m^{-1} o_m = sum softmax(q_m^T k_n) R_{n-m} k restores relative position).
* Background: the query attends to the top-k compressed entries plus the
  uncompressed tokens of a 128-token sliding window [m-127, m].
* Method details, fusion (2): the attention output goes through inverse RoPE
  and then fp8 quantisation.

Readings taken where the page is silent:
* One softmax over the union of the selected compressed entries and the
  window tokens (a compressed entry and the raw tokens it summarises are
  different keys and both count).  Scale tau = 1/sqrt(D) (the appendix omits
  the scale "for brevity").
* fp8 output: one fp32 scale per token over all heads and dims, amax/448.
"""
from __future__ import annotations

import numpy as np

from .compressor import rope
from .formats import fp8_token_encode


def shared_kv_attention(q: np.ndarray, keys: np.ndarray, tau: float):
    """q [H][D], keys [N][D] (also the values) -> (o [H][D], lse [H])."""
    z = tau * (q @ keys.T)                          # [H][N]
    mx = np.max(z, axis=1, keepdims=True)
    e = np.exp(z - mx)
    s = e.sum(axis=1, keepdims=True)
    o = (e / s) @ keys
    lse = (mx + np.log(s))[:, 0]
    return o, lse


def inverse_rope(o: np.ndarray, m: int, rope_dims: int, theta: float) -> np.ndarray:
    """R_m^{-1} applied to every head of o [H][D]."""
    return rope(o, m, rope_dims, theta, inverse=True)


def quant_fp8_per_token(o: np.ndarray):
    """o [H][D] -> (codes [H][D], scale) with one scale for the whole token."""
    codes, s = fp8_token_encode(o.reshape(-1))
    return codes.reshape(o.shape), s
