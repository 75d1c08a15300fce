"""Pins of the compressor, RMSNorm and RoPE: closed forms, group identities
and chunk == sequence of steps."""
import math

import numpy as np
import pytest

from oracle import compressor as C
from oracle import formats as F
from oracle import geometry as G
from oracle import layer as L


def test_equal_logits_give_the_mean_and_dominant_logit_copies():
    rng = np.random.default_rng(0)
    xs = rng.standard_normal((8, 16))
    valid = np.ones(8, bool)
    mean = C.compress_window(xs, np.full(8, 0.3), np.zeros(8), valid)
    assert np.allclose(mean, xs.mean(axis=0), rtol=0, atol=1e-14)
    g = np.zeros(8)
    g[5] = 800.0
    assert np.allclose(C.compress_window(xs, g, np.zeros(8), valid), xs[5], atol=1e-14)
    # bias and gate add: moving the logit from the gate to the bias changes nothing
    b = rng.standard_normal(8)
    g2 = rng.standard_normal(8)
    assert np.allclose(C.compress_window(xs, g2 + b, np.zeros(8), valid),
                       C.compress_window(xs, g2, b, valid), atol=1e-14)


def test_first_c4a_entry_uses_only_positions_0_to_3():
    rng = np.random.default_rng(1)
    xs = rng.standard_normal((8, 4))
    valid = np.array([False] * 4 + [True] * 4)
    w = C.window_weights(rng.standard_normal(8), rng.standard_normal(8), valid)
    assert np.all(w[:4] == 0) and math.isclose(w.sum(), 1.0)
    ref = C.compress_window(xs[4:], np.zeros(4), np.zeros(4), np.ones(4, bool))
    got = C.compress_window(xs, np.zeros(8), np.zeros(8), valid)
    assert np.allclose(got, ref, atol=1e-15)


def test_rms_norm_unit_rms():
    rng = np.random.default_rng(2)
    c = rng.standard_normal(512) * 7
    n = C.rms_norm(c, np.ones(512), eps=0.0)
    assert math.isclose(np.sqrt(np.mean(n * n)), 1.0, rel_tol=1e-14)
    g = rng.standard_normal(512)
    assert np.allclose(C.rms_norm(c, g, 0.0), n * g)


def test_rope_hand_values_and_group_identities():
    D, R, th = 128, 64, 10000.0
    e = np.zeros(D)
    e[D - R] = 1.0                       # first rotated pair, first component
    r = C.rope(e, 1, R, th)
    assert math.isclose(r[D - R], math.cos(1.0)) and math.isclose(r[D - R + 1], math.sin(1.0))
    e2 = np.zeros(D)
    e2[D - R + 3] = 1.0                  # pair j=1, second component
    r2 = C.rope(e2, 5, R, th)
    ang = 5 * th ** (-2.0 / R)
    assert math.isclose(r2[D - R + 2], -math.sin(ang)) and math.isclose(r2[D - R + 3], math.cos(ang))
    rng = np.random.default_rng(3)
    v = rng.standard_normal(D)
    assert np.array_equal(C.rope(v, 7, R, th)[:D - R], v[:D - R])     # nope dims untouched
    for m, n in ((3, 11), (1000, 777777), (1048575, 1)):
        a = C.rope(v, m, R, th)
        assert math.isclose(np.linalg.norm(a), np.linalg.norm(v), rel_tol=1e-13)   # R^T R = I
        assert np.allclose(C.rope(a, n, R, th), C.rope(v, m + n, R, th), atol=1e-9)  # R_m R_n
        assert np.allclose(C.rope(a, m, R, th, inverse=True), v, atol=1e-12)         # R_-m R_m
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    d1 = C.rope(q, 100, R, th) @ C.rope(k, 40, R, th)
    d2 = C.rope(q, 5100, R, th) @ C.rope(k, 5040, R, th)
    assert math.isclose(d1, d2, rel_tol=1e-10)                          # relative position only


def _comp(ratio, dim, B, cap, rng):
    return L.Compressor(ratio=ratio, dim=dim, rope_dims=dim // 2 if dim < 128 else 64,
                        theta=10000.0, bias=rng.standard_normal(G.window_len(ratio)) * 0.5,
                        gamma=1 + 0.1 * rng.standard_normal(dim),
                        ring_x=F.bf16_encode(rng.standard_normal((B, cap, dim))),
                        ring_gate=rng.standard_normal((B, cap)))


@pytest.mark.parametrize("ratio,start,C_new", [(4, 13, 19), (4, 0, 9), (128, 250, 140)])
def test_chunk_equals_sequence_of_single_token_calls(ratio, start, C_new):
    rng = np.random.default_rng(4)
    dim = 32
    W = G.window_len(ratio)
    cap = W - 1 + C_new
    comp = _comp(ratio, dim, 1, cap, rng)
    x = F.bf16_encode(rng.standard_normal((C_new, dim)))
    g = rng.standard_normal(C_new)
    pos = np.arange(start, start + C_new)
    chunk = L.compress(np.zeros(C_new, int), pos, x, g, comp)
    # replay one token at a time, writing each token into the ring afterwards
    ring_x, ring_g = comp.ring_x.copy(), comp.ring_gate.copy()
    step = {}
    for t in range(C_new):
        c1 = L.Compressor(**{**comp.__dict__, "ring_x": ring_x.copy(), "ring_gate": ring_g.copy()})
        step.update(L.compress(np.zeros(1, int), pos[t:t + 1], x[t:t + 1], g[t:t + 1], c1))
        ring_x[0, pos[t] % cap] = x[t]
        ring_g[0, pos[t] % cap] = g[t]
    assert chunk.keys() == step.keys()
    assert len(chunk) == sum(1 for p in pos if (p + 1) % ratio == 0)
    for key in chunk:
        assert np.array_equal(chunk[key], step[key])


def test_compressed_entry_matches_hand_composition():
    rng = np.random.default_rng(5)
    dim = 16
    xs = {p: rng.standard_normal(dim) for p in range(0, 40)}
    gs = {p: rng.standard_normal() for p in range(0, 40)}
    bias = rng.standard_normal(8)
    gamma = rng.standard_normal(dim)
    i = 5
    pos = list(range(16, 24))
    logits = np.array([gs[p] + bias[j] for j, p in enumerate(pos)])
    w = np.exp(logits - logits.max())
    w /= w.sum()
    c = sum(w[j] * xs[p] for j, p in enumerate(pos))
    n = c / math.sqrt(np.mean(c * c) + 1e-6) * gamma
    ang = (4 * i + 3) * 10000.0 ** (-2.0 * np.arange(4) / 8)
    out = n.copy()
    a, b = n[8::2].copy(), n[9::2].copy()
    out[8::2] = a * np.cos(ang) - b * np.sin(ang)
    out[9::2] = a * np.sin(ang) + b * np.cos(ang)
    got = C.compressed_entry(lambda p: xs[p], lambda p: gs[p], i, 4, bias, gamma, 8, 10000.0)
    assert np.allclose(got, out, atol=1e-13)
