"""Positions, windows, causality and slot mapping.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows "DeepSeek V4 in vLLM: Efficient Long-context Attention":
* Appendix, "exact position ranges and causality": c4a entry i (0-based) is
  a weighted sum of the native tokens at positions [4i-4, 4i+3], negative
  positions counting as absent; c128a entry i covers [128i, 128i+127].  RoPE
  is applied once, at the entry's anchor = its last native position (4i+3 or
  128i+127).  A query at position m may use entry i only if anchor(i) <= m.
* Method details, "A single logical block size": every compressed layer's
  logical block is 256 native positions, i.e. 256/ratio entries per physical
  block (64 for c4a, 2 for c128a); slot mapping needs no branch on the ratio.
* Background, "short sliding window": the window holds the uncompressed
  tokens [m-127, m]; appendix "why the short window" (a c128a query with
  m < 127 sees no compressed entry).
"""
from __future__ import annotations

BLOCK_POSITIONS = 256
SWA_WINDOW = 128


def entries_per_block(ratio: int) -> int:
    return BLOCK_POSITIONS // ratio


def window_positions(i: int, ratio: int) -> list[int]:
    """Native positions summed into compressed entry ``i`` (may be < 0)."""
    if ratio == 4:
        return list(range(4 * i - 4, 4 * i + 4))
    if ratio == 128:
        return list(range(128 * i, 128 * i + 128))
    raise ValueError(ratio)


def window_len(ratio: int) -> int:
    return 8 if ratio == 4 else 128


def anchor(i: int, ratio: int) -> int:
    """Position at which entry i is rotated: its last native token."""
    return ratio * i + ratio - 1


def emits_at(t: int, ratio: int) -> int | None:
    """Entry index completed by native token t, or None."""
    if (t + 1) % ratio == 0:
        return (t + 1) // ratio - 1
    return None


def n_visible(m: int, ratio: int) -> int:
    """Number of entries a query at position m may use: #{i : anchor(i) <= m}."""
    return (m + 1) // ratio


def swa_positions(m: int, window: int = SWA_WINDOW) -> list[int]:
    return list(range(max(0, m - window + 1), m + 1))


def slot_of(block_table_row, i: int, ratio: int) -> tuple[int, int]:
    """(physical block, slot within block) of logical entry i."""
    e = entries_per_block(ratio)
    return int(block_table_row[i // e]), i % e
