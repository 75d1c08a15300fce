"""Comparison helpers for the GPU parity tests (GPU output vs fp64 oracle)."""
from __future__ import annotations

import json
import os

import numpy as np

from oracle import formats as F
from oracle import geometry as G

BF16_TOL = (2e-2, 2e-3)     # attention output, bf16 caches: max-abs, mean-abs
FP8_TOL = (6e-2, 6e-3)      # attention output, fp8 / fp4 caches
TOPK_REL = 1e-5             # near-tie band around the k-th score

# With V4A_PARITY_RECORD set to a file path, every comparison below appends
# what it observed (errors, swap counts) as one JSON line there; the committed
# parity record under profiles/ is a summary of such a file from a GPU run.
_RECORD = os.environ.get("V4A_PARITY_RECORD")


def record(kind: str, where: str, **stats):
    if not _RECORD:
        return
    with open(_RECORD, "a") as f:
        f.write(json.dumps({"kind": kind, "where": str(where), **stats}) + "\n")


def check_topk(gpu_idx: np.ndarray, ref_idx: np.ndarray, scores: np.ndarray, k: int, where=""):
    """Sets equal except swaps among scores within TOPK_REL of the k-th score;
    the GPU row must be ascending, unique, -1 padded and inside the visible range."""
    n = scores.shape[0]
    g = gpu_idx.tolist()
    valid = [v for v in g if v >= 0]
    assert len(valid) == min(n, k), (where, len(valid), min(n, k))
    assert g[:len(valid)] == sorted(valid) and len(set(valid)) == len(valid), where
    assert all(v == -1 for v in g[len(valid):]), where
    assert all(0 <= v < n for v in valid), where
    if n <= k:
        assert sorted(valid) == list(range(n)), where
        return 0
    kth = np.sort(scores)[::-1][k - 1]
    diff = set(valid) ^ set(int(v) for v in ref_idx if v >= 0)
    worst = 0.0
    for e in diff:
        rel = abs(scores[e] - kth) / max(abs(kth), 1e-30)
        worst = max(worst, rel)
        assert rel <= TOPK_REL, (where, e, scores[e], kth)
    record("topk", where, swaps=len(diff) // 2, worst_swap_rel_to_kth=worst, k=k, entries=n)
    return len(diff)


def check_close(gpu: np.ndarray, ref: np.ndarray, tol, where=""):
    err = np.abs(np.asarray(gpu, np.float64) - ref)
    mx, mean = float(err.max()), float(err.mean())
    record("close", where, max_abs=mx, mean_abs=mean, tol_max=tol[0], tol_mean=tol[1])
    assert mx <= tol[0] and mean <= tol[1], (where, mx, mean)
    return mx, mean


# The kernels compute in fp32: a sum of up to 128 weighted terms, or a
# rotation, leaves an absolute error of a few fp32 ulps of the row's largest
# element.  An element that cancels to near zero cannot be within one bf16
# ulp of its own tiny value, so each element may also differ by this floor
# (2^-18 of the row's max, about 1e-3 of a bf16 ulp at that magnitude).
FP32_FLOOR = 2.0 ** -18


def check_bf16_row(gpu_bits: np.ndarray, ref: np.ndarray, where=""):
    """Stored bf16 within 1 ulp of the fp64 value (plus the fp32 floor)."""
    got = F.bf16_decode(gpu_bits)
    ulp = F.bf16_ulp(ref)
    floor = FP32_FLOOR * float(np.max(np.abs(ref)))
    bad = np.abs(got - ref) > ulp * 1.0000001 + floor + 1e-30
    assert not bad.any(), (where, np.nonzero(bad)[0][:5], got[bad][:5], ref[bad][:5])


def check_fp8_row(codes: np.ndarray, scale: float, ref: np.ndarray, where=""):
    """Per-row fp8: scale = amax/448 (relative 1e-6), values within 1 e4m3 ulp * scale."""
    amax = np.max(np.abs(ref))
    assert abs(scale - amax / 448) <= 1e-6 * amax / 448 + 1e-30, (where, scale, amax / 448)
    got = F.e4m3_decode(codes) * scale
    ulp = F.e4m3_ulp(ref / scale) * scale
    bad = np.abs(got - ref) > ulp * 1.0000001 + 1e-30
    assert not bad.any(), (where, np.nonzero(bad)[0][:5])


def check_fp8_blocks(codes, scales, ref, block, where=""):
    for b in range(ref.shape[0] // block):
        check_fp8_row(codes[b * block:(b + 1) * block], float(scales[b]), ref[b * block:(b + 1) * block],
                      f"{where}/blk{b}")


def check_fp4_blocks(packed, scales, ref, where=""):
    nib = F.unpack_nibbles(packed)
    for b in range(ref.shape[0] // 32):
        seg = ref[32 * b:32 * b + 32]
        amax = np.max(np.abs(seg))
        s = float(scales[b])
        assert abs(s - amax / 6) <= 1e-6 * amax / 6 + 1e-30, (where, b, s, amax / 6)
        got = F.e2m1_decode(nib[32 * b:32 * b + 32]) * s
        ulp = F.e2m1_ulp(seg / s) * s
        bad = np.abs(got - seg) > ulp * 1.0000001 + 1e-30
        assert not bad.any(), (where, b, np.nonzero(bad)[0][:5])


def check_fp4_mx_blocks(packed, scales, ref, where=""):
    """MX fp4: every scale a power of two equal to the oracle's shared scale
    (or the neighbouring one when the fp32 amax rounds across a power of two),
    codes within 1 e2m1 ulp, values above 6 * scale clipped to 6 * scale."""
    nib = F.unpack_nibbles(packed)
    for b in range(ref.shape[0] // 32):
        seg = ref[32 * b:32 * b + 32]
        s = float(scales[b])
        m, _ = np.frexp(s)
        assert m == 0.5, (where, b, s)
        want = F.mx_shared_scale(seg)
        amax = float(np.max(np.abs(seg)))
        near_pow2 = abs(np.frexp(amax)[0] - 0.5) < 1e-6 or abs(np.frexp(amax)[0] - 1.0) < 1e-6
        assert s == want or (near_pow2 and s in (want / 2, want * 2)), (where, b, s, want)
        got = F.e2m1_decode(nib[32 * b:32 * b + 32]) * s
        clipped = np.clip(seg, -6 * s, 6 * s)
        ulp = F.e2m1_ulp(clipped / s) * s
        bad = np.abs(got - clipped) > ulp * 1.0000001 + 1e-30
        assert not bad.any(), (where, b, np.nonzero(bad)[0][:5])


def check_dsv4_row(row: np.ndarray, ref: np.ndarray, where=""):
    """DeepSeek-V4 584-byte row: every nope block's scale byte equal to the
    oracle's rule on the fp64 values (or a neighbour when the block's amax
    lies within fp32 rounding of a scale boundary), codes within 1 e4m3 ulp of
    value / scale, rope elements within 1 bf16 ulp, pad byte 0."""
    assert row.shape == (F.DSV4_ROW,) and row[-1] == 0, where
    for j in range(F.DSV4_NOPE // F.DSV4_QBLOCK):
        seg = ref[64 * j:64 * (j + 1)]
        b = int(row[F.DSV4_NOPE + 2 * F.DSV4_ROPE + j])
        want = F.ue8m0_e4m3_scale_byte(seg)
        amax = float(np.max(np.abs(seg)))
        edge = amax > 0 and any(abs(amax / (448.0 * 2.0 ** (w - 127)) - 1.0) < 1e-6 for w in (want, want - 1))
        assert b == want or (edge and abs(b - want) == 1), (where, j, b, want)
        s = 2.0 ** (b - 127)
        got = F.e4m3_decode(row[64 * j:64 * (j + 1)]) * s
        ulp = F.e4m3_ulp(np.clip(seg / s, -448, 448)) * s
        bad = np.abs(got - np.clip(seg, -448 * s, 448 * s)) > ulp * 1.0000001 + 1e-30
        assert not bad.any(), (where, j, np.nonzero(bad)[0][:5])
    check_bf16_row(row[F.DSV4_NOPE:F.DSV4_NOPE + 2 * F.DSV4_ROPE].copy().view(np.uint16), ref[F.DSV4_NOPE:],
                   f"{where}/rope")


def kv_slot_bytes(pool: np.ndarray, spec, blk: int, slot: int):
    """(row bytes, scale or None) of one shared-KV entry."""
    E, D = spec.entries_per_block, spec.dim
    base = blk * spec.kv_block_bytes
    if spec.kv_fmt == F.KV_BF16:
        return pool[base + slot * 2 * D: base + (slot + 1) * 2 * D].copy().view(np.uint16), None
    if spec.kv_fmt == F.KV_FP8_DSV4:
        return pool[base + slot * F.DSV4_ROW: base + (slot + 1) * F.DSV4_ROW].copy(), None
    row = pool[base + slot * D: base + (slot + 1) * D].copy()
    sc = pool[base + E * D + 4 * slot: base + E * D + 4 * slot + 4].copy().view(np.float32)[0]
    return row, float(sc)


def ix_slot_bytes(pool: np.ndarray, spec, blk: int, slot: int):
    d, fmt = spec.ix_dim, spec.ix_fmt
    base = blk * spec.ix_block_bytes
    if fmt == F.IX_BF16:
        return pool[base + slot * 2 * d: base + (slot + 1) * 2 * d].copy().view(np.uint16), None
    rb = d if fmt == F.IX_FP8_B128 else d // 2
    ns = d // 128 if fmt == F.IX_FP8_B128 else d // 32
    row = pool[base + slot * rb: base + (slot + 1) * rb].copy()
    off = base + 64 * rb + 4 * ns * slot
    sc = pool[off: off + 4 * ns].copy().view(np.float32).astype(np.float64)
    return row, sc


def entry_slots(spec, block_table: np.ndarray, entries: dict, ratio: int):
    return {(b, i): G.slot_of(block_table[b], i, ratio) for (b, i) in entries}
