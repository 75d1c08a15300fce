"""Pins of the oracle's number formats against library casts and the OCP tables."""
import math

import numpy as np
import pytest
import torch

from oracle import formats as F


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = F.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def _e4m3_probe_values():
    pos = F.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[1:] + pos[:-1]) / 2
    rng = np.random.default_rng(0)
    rand = rng.standard_normal(20000) * rng.choice([1e-3, 0.1, 1, 30, 200], 20000)
    v = np.concatenate([pos, mids, mids * (1 + 1e-9), mids * (1 - 1e-9), rand])
    v = v[np.abs(v) <= 448]
    return np.concatenate([v, -v])


def test_e4m3_encode_matches_torch_cast():
    v = _e4m3_probe_values().astype(np.float32).astype(np.float64)  # torch casts from fp32
    ours = F.e4m3_decode(F.e4m3_encode(v))
    ref = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates_and_roundtrips():
    assert F.e4m3_decode(F.e4m3_encode(np.array([1e6, -500.0, 470.0])).tolist()).tolist() == [448.0, -448.0, 448.0]
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    back = F.e4m3_encode(F.e4m3_decode(codes))
    # +0 and -0 both decode to 0; everything else round-trips exactly
    assert np.array_equal(F.e4m3_decode(back), F.e4m3_decode(codes))
    assert np.array_equal(back[codes != 0x80], codes[codes != 0x80])


OCP_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_is_ocp_table():
    vals = F.e2m1_decode(np.arange(16))
    assert vals[:8].tolist() == OCP_E2M1
    assert (-vals[8:]).tolist() == OCP_E2M1


def test_e2m1_encode_nearest_even_brute_force():
    table = np.array(OCP_E2M1)
    rng = np.random.default_rng(1)
    mids = (table[1:] + table[:-1]) / 2
    v = np.concatenate([table, mids, rng.uniform(-7, 7, 5000), [6.5, 100.0]])
    for x in v:
        mag = min(abs(x), 6.0)
        d = np.abs(table - mag)
        best = np.nonzero(d == d.min())[0]
        code = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]
        got = int(F.e2m1_encode(np.array([x]))[0])
        assert got & 7 == code, (x, got, code)
        assert (got >> 3) == (1 if np.signbit(x) else 0)
    # ties printed explicitly: 0.25->0, 0.75->1, 1.25->1, 2.5->2, 5->4
    assert F.e2m1_decode(F.e2m1_encode(np.array([0.25, 0.75, 1.25, 2.5, 5.0]))).tolist() == [0, 1, 1, 2, 4]


def test_bf16_encode_matches_torch_on_fp32_and_brute_force_on_fp64():
    rng = np.random.default_rng(2)
    v32 = np.concatenate([rng.standard_normal(20000) * 10 ** rng.uniform(-30, 30, 20000),
                          [0.0, -0.0, 1.0, 3.0e38, 1e-40]]).astype(np.float32)
    ours = F.bf16_encode(v32.astype(np.float64))
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    v64 = rng.standard_normal(2000) * 10 ** rng.uniform(-5, 5, 2000)
    for x in v64:
        b = int(F.bf16_encode(np.array([x]))[0])
        lo = F.bf16_decode(np.array([b - 1], np.uint16))[0]
        hi = F.bf16_decode(np.array([b + 1], np.uint16))[0]
        mid = F.bf16_decode(np.array([b], np.uint16))[0]
        assert abs(mid - x) <= abs(lo - x) and abs(mid - x) <= abs(hi - x)


def test_fp8_token_quant_scale_rule_and_error():
    rng = np.random.default_rng(3)
    v = rng.standard_normal(512)
    codes, s = F.fp8_token_encode(v)
    assert s == pytest.approx(np.max(np.abs(v)) / 448, rel=1e-7)
    dq = F.e4m3_decode(codes) * s
    assert np.all(np.abs(dq - v) <= 0.5 * F.e4m3_ulp(v / s) * s * (1 + 1e-6) + 1e-12)
    assert np.max(np.abs(F.e4m3_decode(codes))) == 448.0
    z, s0 = F.fp8_token_encode(np.zeros(8))
    assert s0 == 1.0 and np.all(z == 0)


def test_fp4_blocks_quant_and_nibble_order():
    rng = np.random.default_rng(4)
    v = rng.standard_normal(128)
    packed, sc = F.fp4_blocks_encode(v, 32)
    assert packed.shape == (64,) and sc.shape == (4,)
    for b in range(4):
        assert sc[b] == pytest.approx(np.max(np.abs(v[32 * b:32 * b + 32])) / 6, rel=1e-7)
    nib = F.unpack_nibbles(packed)
    assert np.array_equal(nib[0::2], packed & 0xF)   # element 2j in the low nibble
    assert np.array_equal(F.pack_nibbles(nib), packed)
    dq = F.e2m1_decode(nib) * np.repeat(sc, 32)
    assert np.all(np.abs(dq - v) <= 0.5 * F.e2m1_ulp(v / np.repeat(sc, 32)) * np.repeat(sc, 32) + 1e-12)


def test_block_layout_bytes_and_decode():
    assert F.ix_block_bytes(F.IX_FP8_B128, 128) == 64 * 132          # 132 B per entry
    assert F.ix_block_bytes(F.IX_FP4_B32, 128) == 64 * 80            # 64 B + 4 scales
    assert F.kv_block_bytes(F.KV_FP8_TOKEN, 64, 512) == 64 * 516
    assert F.kv_block_bytes(F.KV_BF16, 2, 512) == 2048
    rng = np.random.default_rng(5)
    rows = rng.standard_normal((64, 128))
    raw = np.zeros(F.ix_block_bytes(F.IX_FP8_B128, 128), np.uint8)
    expect = np.zeros((64, 128))
    for e in range(64):
        c, s = F.fp8_blocks_encode(rows[e], 128)
        raw[e * 128:(e + 1) * 128] = c
        raw[64 * 128 + 4 * e: 64 * 128 + 4 * e + 4] = np.array(s, np.float32).view(np.uint8)
        expect[e] = F.e4m3_decode(c) * s[0]
    assert np.array_equal(F.ix_block_decode(raw, F.IX_FP8_B128, 128), expect)


def test_nibble_order_hand_bytes():
    # byte 0x21 holds element 0 = code 1 (0.5) and element 1 = code 2 (1.0);
    # byte 0xF8 holds element 2 = code 8 (-0) and element 3 = code 15 (-6)
    nib = F.unpack_nibbles(np.array([0x21, 0xF8], np.uint8))
    assert nib.tolist() == [1, 2, 8, 15]
    assert F.e2m1_decode(nib).tolist() == [0.5, 1.0, -0.0, -6.0]


def test_kv_fp8_and_ix_fp4_block_decode_apply_scales():
    E, D = 64, 512
    raw = np.zeros(F.kv_block_bytes(F.KV_FP8_TOKEN, E, D), np.uint8)
    raw[0] = 0x38                      # e4m3 1.0 at entry 0, dim 0
    raw[D * 5 + 7] = 0xC0              # e4m3 -2.0 at entry 5, dim 7
    sc = np.ones(E, np.float32)
    sc[0], sc[5] = 0.25, 3.0
    raw[E * D:] = sc.view(np.uint8)
    dec = F.kv_block_decode(raw, F.KV_FP8_TOKEN, E, D)
    assert dec[0, 0] == 0.25 and dec[5, 7] == -6.0 and dec.sum() == 0.25 - 6.0
    dI = 128
    raw = np.zeros(F.ix_block_bytes(F.IX_FP4_B32, dI), np.uint8)
    raw[3 * 64 + 20] = 0x70            # entry 3: element 40 = 0 (low), element 41 = code 7 (6.0)
    s4 = np.ones((64, 4), np.float32)
    s4[3, 1] = 0.5                     # elements 32..63 of entry 3
    raw[64 * 64:] = s4.reshape(-1).view(np.uint8)
    dec = F.ix_block_decode(raw, F.IX_FP4_B32, dI)
    assert dec[3, 41] == 3.0 and np.count_nonzero(dec) == 1


def test_mx_shared_scale_rule_hand_worked():
    # OCP MX rule: X = 2^(floor(log2 amax) - 2) for e2m1 (emax_elem = 2)
    assert F.mx_shared_scale(np.array([5.0, -0.7, 0.3])) == 1.0          # floor(log2 5) = 2
    assert F.mx_shared_scale(np.array([-4.0, 1.0])) == 1.0              # exact power of two: 2 - 2 = 0
    assert F.mx_shared_scale(np.array([3.99, 0.0])) == 0.5              # floor(log2 3.99) = 1
    assert F.mx_shared_scale(np.array([0.2, -0.1])) == 2.0 ** -5        # floor(log2 0.2) = -3
    assert F.mx_shared_scale(np.array([1000.0])) == 2.0 ** 7            # floor(log2 1000) = 9
    assert F.mx_shared_scale(np.zeros(32)) == 1.0
    assert F.mx_shared_scale(np.array([1e-45])) == 2.0 ** -126          # clamped to a normal fp32 word


def test_fp4_mx_block_hand_worked_codes():
    v = np.zeros(32)
    v[:6] = [5.0, -0.7, 0.3, 7.5, 6.0, -2.6]
    packed, sc = F.fp4_mx_blocks_encode(v)
    assert sc.tolist() == [1.0]                                            # amax 7.5 -> floor(log2) = 2
    nib = F.unpack_nibbles(packed)
    # 5.0 is the midpoint of 4 and 6 -> even code (4); -0.7 -> -0.5; 0.3 -> 0.5;
    # 7.5 saturates to 6; 6 stays; -2.6 -> -3 (nearest)
    assert F.e2m1_decode(nib[:6]).tolist() == [4.0, -0.5, 0.5, 6.0, 6.0, -3.0]
    assert nib[:6].tolist() == [0x6, 0x9, 0x1, 0x7, 0x7, 0xD]
    assert not np.any(nib[6:])


def test_fp4_mx_scales_are_powers_of_two_and_error_bounded():
    rng = np.random.default_rng(11)
    for _ in range(300):
        v = rng.standard_normal(128) * 10.0 ** rng.uniform(-4, 4)
        packed, sc = F.fp4_mx_blocks_encode(v)
        m, e = np.frexp(sc)
        assert np.all(m == 0.5), "every MX scale is an exact power of two"
        dec = F.e2m1_decode(F.unpack_nibbles(packed)) * np.repeat(sc, 32)
        for b in range(4):
            seg, d = v[32 * b:32 * b + 32], dec[32 * b:32 * b + 32]
            amax = np.abs(seg).max()
            assert 4.0 <= amax / sc[b] < 8.0
            # inside the e2m1 range the error is at most half a step of the grid
            # at that magnitude; above 6 * X the value clips to 6 * X
            inside = np.abs(seg) <= 6.0 * sc[b]
            assert np.all(np.abs(seg - d)[inside] <= F.e2m1_ulp(seg[inside] / sc[b]) * sc[b] / 2 + 1e-300)
            assert np.all(np.abs(d[~inside]) == 6.0 * sc[b])


def test_fp4_mx_layout_equals_fp4_layout():
    assert F.ix_block_bytes(F.IX_FP4_MX32, 128) == F.ix_block_bytes(F.IX_FP4_B32, 128) == 64 * 80
    rng = np.random.default_rng(2)
    raw = rng.integers(0, 256, F.ix_block_bytes(F.IX_FP4_B32, 128), dtype=np.uint8)
    raw[64 * 64:] = np.ldexp(1.0, rng.integers(-5, 5, 64 * 4)).astype(np.float32).view(np.uint8)
    assert np.array_equal(F.ix_block_decode(raw, F.IX_FP4_MX32, 128), F.ix_block_decode(raw, F.IX_FP4_B32, 128))


# ---- DeepSeek-V4 fp8 row (SGLang KV-pool article, section "DeepSeek-V4") ----

def test_dsv4_row_and_page_arithmetic_from_the_pages():
    # the article's per-token byte list: 448 fp8 + 64 x bf16 + 448 / 64 scales + 1 pad
    assert 448 + 64 * 2 + 448 // 64 + 1 == 584 == F.DSV4_ROW
    # pages padded to 576-byte units: ceil(page_size * 584 / 576) * 576
    assert F.kv_block_bytes(F.KV_FP8_DSV4, 64, 512) == math.ceil(64 * 584 / 576) * 576 == 37440
    assert F.kv_block_bytes(F.KV_FP8_DSV4, 2, 512) == 1728


def test_dsv4_scale_byte_hand_values_and_brute_force():
    # hand-worked: 448 = 0.875 * 2^9 fits scale 1; 449 needs 2; 1.0 fits 2^-8 (1 / 2^-8 = 256 <= 448 < 512)
    assert F.ue8m0_e4m3_scale_byte(np.array([448.0])) == 127
    assert F.ue8m0_e4m3_scale_byte(np.array([-449.0, 3.0])) == 128
    assert F.ue8m0_e4m3_scale_byte(np.array([1.0, -0.25])) == 119
    assert F.ue8m0_e4m3_scale_byte(np.array([896.5])) == 129
    assert F.ue8m0_e4m3_scale_byte(np.zeros(64)) == 127
    rng = np.random.default_rng(5)
    for amax in np.exp(rng.uniform(-20, 20, 300)):
        k = -140
        while amax / 2.0 ** k > 448.0:      # smallest power of two that keeps amax within e4m3
            k += 1
        assert F.ue8m0_e4m3_scale_byte(np.array([amax])) == k + 127


def test_dsv4_row_bytes_match_library_casts():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(6)
    v = rng.normal(0, 1, 512) * np.exp(rng.uniform(-3, 3, 512))
    row = F.dsv4_row_encode(v)
    assert row.shape == (584,) and row[583] == 0
    for j in range(7):
        seg = v[64 * j:64 * (j + 1)]
        b = int(row[576 + j])
        want = torch.from_numpy(np.ldexp(seg, 127 - b)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(row[64 * j:64 * (j + 1)], want)
        assert np.max(np.abs(seg)) <= 448.0 * 2.0 ** (b - 127) < 2 * np.max(np.abs(seg))
    rope = torch.from_numpy(v[448:]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint8)
    assert np.array_equal(row[448:576], rope)
    # decode: codes times their block's power of two; rope as stored
    dec = F.dsv4_row_decode(row)
    codes = torch.from_numpy(row[:448].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(dec[:448], codes * np.repeat(2.0 ** (row[576:583].astype(np.int64) - 127), 64))
    assert np.array_equal(dec[448:], torch.from_numpy(v[448:]).to(torch.bfloat16).to(torch.float64).numpy())
