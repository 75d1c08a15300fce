"""Pins of indexer top-k and shared-K=V attention: brute force on tiny
inputs, the tie rule, the dense special case against torch fp64, window
coverage and translation invariance after inverse RoPE."""
import itertools
import math

import numpy as np
import torch

from oracle import attention as A
from oracle import compressor as C
from oracle import indexer as I


def test_scores_brute_force_loops():
    rng = np.random.default_rng(0)
    q, w, keys = rng.standard_normal((4, 8)), rng.uniform(0, 1, 4), rng.standard_normal((30, 8))
    s = I.index_scores(q, w, keys)
    for i in range(30):
        ref = sum(w[h] * max(0.0, sum(q[h, d] * keys[i, d] for d in range(8))) for h in range(4))
        assert math.isclose(s[i], ref, rel_tol=1e-12, abs_tol=1e-14)


def test_topk_brute_force_sort():
    rng = np.random.default_rng(1)
    for n, k in ((10, 3), (40, 40), (7, 12), (100, 33)):
        s = np.round(rng.standard_normal(n), 1)          # plenty of exact ties
        got = I.topk_set(s, k)
        order = sorted(range(n), key=lambda i: (-s[i], i))[:min(n, k)]
        assert got[:min(n, k)].tolist() == sorted(order)
        assert np.all(got[min(n, k):] == -1)


def test_all_ties_take_lowest_indices():
    keys = np.random.default_rng(2).standard_normal((50, 8))
    s = I.index_scores(np.ones((4, 8)), np.zeros(4), keys)       # w = 0: every score 0
    assert np.all(s == 0)
    assert I.topk_set(s, 16).tolist() == list(range(16))


def test_sparse_equals_dense_when_k_covers_everything():
    rng = np.random.default_rng(3)
    H, D, n = 4, 32, 20
    q, keys = rng.standard_normal((H, D)), rng.standard_normal((n, D))
    tau = 1 / math.sqrt(D)
    sel = I.topk_set(rng.standard_normal(n), 64)        # k > n: all entries
    o, lse = A.shared_kv_attention(q, keys[sel[sel >= 0]], tau)
    qt, kt = torch.from_numpy(q), torch.from_numpy(keys)
    p = torch.softmax(tau * qt @ kt.T, dim=-1)
    ref = (p @ kt).numpy()
    assert np.allclose(o, ref, atol=1e-13)
    assert np.allclose(lse, torch.logsumexp(tau * qt @ kt.T, dim=-1).numpy(), atol=1e-12)


def test_translation_invariance_after_inverse_rope():
    rng = np.random.default_rng(4)
    H, D, R, th = 3, 64, 32, 10000.0
    q0 = rng.standard_normal((H, D))
    k0 = rng.standard_normal((9, D))
    key_pos = np.array([3, 7, 11, 15, 90, 91, 92, 93, 94])
    m = 94
    tau = 1 / math.sqrt(D)

    def run(delta, inverse):
        q = C.rope(q0, m + delta, R, th)
        keys = np.stack([C.rope(k0[j], key_pos[j] + delta, R, th) for j in range(9)])
        o, _ = A.shared_kv_attention(q, keys, tau)
        return A.inverse_rope(o, m + delta, R, th) if inverse else o

    base = run(0, True)
    for delta in (1, 1000, 123457):
        assert np.allclose(run(delta, True), base, atol=1e-9)
    # negative control: without the inverse rotation the output moves with position
    assert not np.allclose(run(1000, False), run(0, False), atol=1e-3)


def test_fp8_output_quant_one_scale_per_token():
    rng = np.random.default_rng(5)
    o = rng.standard_normal((4, 16))
    codes, s = A.quant_fp8_per_token(o)
    assert codes.shape == (4, 16)
    assert math.isclose(s, np.max(np.abs(o)) / 448, rel_tol=1e-7)


def test_attention_softmax_is_a_distribution_over_union():
    # duplicates count as separate keys: attending to [k, k] equals attending to k
    rng = np.random.default_rng(6)
    q, k = rng.standard_normal((2, 8)), rng.standard_normal((1, 8))
    o1, _ = A.shared_kv_attention(q, k, 0.5)
    o2, lse2 = A.shared_kv_attention(q, np.concatenate([k, k]), 0.5)
    assert np.allclose(o1, o2) and np.allclose(o1, np.repeat(k, 2, axis=0))
    assert np.allclose(lse2, 0.5 * (q @ k.T)[:, 0] + math.log(2))
    for perm in itertools.permutations(range(3)):
        ks = rng.standard_normal((3, 8)) if perm == (0, 1, 2) else ks
        a, _ = A.shared_kv_attention(q, ks, 0.3)
        b, _ = A.shared_kv_attention(q, ks[list(perm)], 0.3)
        assert np.allclose(a, b, atol=1e-14)


# ---- hand-worked examples (values computed by hand, not by the oracle) -------

def test_index_score_hand_example():
    """Two heads: q_1.k = 3, q_2.k = -2 (ReLU drops it), w = (0.5, 2):
    score = 0.5 * 3 + 2 * 0 = 1.5.  A second key with q_1.k = -1, q_2.k = 4
    scores 2 * 4 = 8 and ranks first."""
    q = np.array([[1.0, 1.0, 0.0], [0.0, -1.0, 1.0]])
    w = np.array([0.5, 2.0])
    keys = np.array([[1.0, 2.0, 0.0],      # q1.k = 3, q2.k = -2
                     [0.0, -1.0, 3.0]])    # q1.k = -1, q2.k = 4
    s = I.index_scores(q, w, keys)
    assert s.tolist() == [1.5, 8.0]
    assert I.topk_set(s, 1).tolist() == [1]


def test_attention_two_keys_hand_example():
    """tau = ln(3)/2, q = (1, 0), k1 = (2, 0), k2 = (0, 5): logits ln 3 and 0,
    weights 3/4 and 1/4, output 3/4 k1 + 1/4 k2 = (1.5, 1.25), lse = ln 4."""
    tau = math.log(3.0) / 2.0
    q = np.array([[1.0, 0.0]])
    keys = np.array([[2.0, 0.0], [0.0, 5.0]])
    o, lse = A.shared_kv_attention(q, keys, tau)
    assert np.allclose(o, [[1.5, 1.25]], rtol=0, atol=1e-15)
    assert math.isclose(lse[0], math.log(4.0), rel_tol=1e-15)


def test_attention_three_keys_two_heads_hand_example():
    """tau = ln 2.  Head 1 (q = (2, 0)): logits 2 ln 2, ln 2, 0 -> weights
    4/7, 2/7, 1/7; head 2 (q = (0, 1)): keys' second coordinates 0, 0, 1 ->
    logits 0, 0, ln 2 -> weights 1/4, 1/4, 1/2.  Keys are the values."""
    tau = math.log(2.0)
    q = np.array([[2.0, 0.0], [0.0, 1.0]])
    keys = np.array([[1.0, 0.0], [0.5, 0.0], [0.0, 1.0]])
    o, lse = A.shared_kv_attention(q, keys, tau)
    exp1 = (4 * keys[0] + 2 * keys[1] + 1 * keys[2]) / 7     # (5/7, 1/7)
    exp2 = (1 * keys[0] + 1 * keys[1] + 2 * keys[2]) / 4     # (3/8, 1/2)
    assert np.allclose(o[0], [5 / 7, 1 / 7], atol=1e-15) and np.allclose(o[0], exp1, atol=1e-15)
    assert np.allclose(o[1], [3 / 8, 1 / 2], atol=1e-15) and np.allclose(o[1], exp2, atol=1e-15)
    assert np.allclose(lse, [math.log(7.0), math.log(4.0)], atol=1e-15)


def test_inverse_rope_of_a_hand_output():
    """Rope dims 2 (one pair), theta irrelevant for pair 0 (frequency 1): at
    position m = 1 the angle is 1 rad, so R_1^{-1} (cos 1, sin 1) = (1, 0) and
    the non-rope dims are untouched."""
    o = np.array([[7.0, math.cos(1.0), math.sin(1.0)]])
    r = A.inverse_rope(o, 1, 2, 10000.0)
    assert np.allclose(r, [[7.0, 1.0, 0.0]], atol=1e-15)
