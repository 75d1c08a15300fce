"""Pins of counts, windows, causality and slot mapping against the page's
closed forms and brute-force enumeration."""
import json
import os

import numpy as np

from oracle import geometry as G

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


def test_entries_per_block_from_page():
    assert G.BLOCK_POSITIONS == GOLD["block_positions"]["value"]
    assert G.entries_per_block(4) == GOLD["entries_per_block"]["c4a"]
    assert G.entries_per_block(128) == GOLD["entries_per_block"]["c128a"]


def test_windows_match_page_ranges():
    for ratio, key in ((4, "c4a_window"), (128, "c128a_window")):
        g = GOLD[key]
        for i in (0, 1, 7, 1000):
            pos = G.window_positions(i, ratio)
            assert pos[0] == g["stride"] * i + g["first"]
            assert pos[-1] == g["stride"] * i + g["last"]
            assert G.anchor(i, ratio) == g["stride"] * i + g["anchor"] == pos[-1]
    assert G.window_len(4) == GOLD["compressor_state_window"]["c4a"] == 8
    assert G.window_len(128) == GOLD["compressor_state_window"]["c128a"] == 128


def test_c4a_windows_overlap_by_four_and_c128a_tile():
    for i in range(1, 50):
        a, b = set(G.window_positions(i - 1, 4)), set(G.window_positions(i, 4))
        assert len(a & b) == 4
        assert len(set(G.window_positions(i - 1, 128)) & set(G.window_positions(i, 128))) == 0
    cover = sorted(p for i in range(6) for p in G.window_positions(i, 128))
    assert cover == list(range(6 * 128))
    assert [p for p in G.window_positions(0, 4) if p >= 0] == [0, 1, 2, 3]


def test_visible_counts_brute_force():
    for ratio in (4, 128):
        for m in range(0, 3000, 7):
            brute = sum(1 for i in range(m + 2) if G.anchor(i, ratio) <= m)
            assert G.n_visible(m, ratio) == brute
            e = G.emits_at(m, ratio)
            if e is not None:
                assert G.anchor(e, ratio) == m
            else:
                assert all(G.anchor(i, ratio) != m for i in range(m + 2))


def test_counts_at_one_million():
    m = (1 << 20) - 1
    assert G.n_visible(m, 4) == 262144
    assert abs(G.n_visible(m, 4) - GOLD["c4a_entries_at_1m_approx"]["value"]) / 250000 < 0.05
    assert G.n_visible(m, 128) == 8192
    assert G.n_visible(m, 128) <= GOLD["k_default"]["c128a"]     # c128a k=8192 is "all"
    # entry 262,143 completes at m = 4*262143+3 = 1,048,575
    assert G.emits_at(m, 4) == 262143


def test_c128a_query_before_first_anchor_sees_no_entry_but_window():
    for m in range(0, 127):
        assert G.n_visible(m, 128) == 0
        assert G.swa_positions(m) == list(range(0, m + 1))
    assert G.n_visible(127, 128) == 1
    assert G.swa_positions(1000) == list(range(873, 1001))
    assert len(G.swa_positions(1000)) == GOLD["swa_window"]["value"]


def test_slot_mapping_has_no_collisions():
    rng = np.random.default_rng(0)
    for ratio in (4, 128):
        B, maxblk = 5, 9
        table = rng.permutation(B * maxblk).reshape(B, maxblk)
        seen = {}
        e = G.entries_per_block(ratio)
        for b in range(B):
            for i in range(maxblk * e):
                blk, slot = G.slot_of(table[b], i, ratio)
                assert 0 <= slot < e
                assert (blk, slot) not in seen
                seen[(blk, slot)] = (b, i)
                # the logical block holds the 256 native positions of entry i's anchor
                assert G.anchor(i, ratio) // 256 == i // e
        assert len(seen) == B * maxblk * e
