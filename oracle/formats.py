"""Number formats and paged-cache byte layouts, written from their definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources and readings
--------------------
* bf16 cache ("DeepSeek V4 in vLLM", section "Method details": prefill keeps a
  bfloat16 KV cache).  bf16 = 1 sign, 8 exponent, 7 stored mantissa bits.
* fp8 per-token cache (same section: decode partly uses a token-wise fp8
  cache; deployment flags use ``--kv-cache-dtype fp8``).  The page names no
  variant; reading taken: OCP e4m3fn (bias 7, max 448, no infinities, one NaN
  pattern per sign), round-to-nearest-even, saturating to +-448.  One fp32
  scale per token: scale = amax/448, or 1 when amax == 0; value = code*scale.
* fp8 indexer cache with one fp32 scale per 128 elements: the SGLang KV-pool
  article, section "DSA", gives 128 fp8 bytes + 4 scale bytes = 132 B per
  token for index_head_dim 128 and quant_block_size 128.
* fp4 indexer cache (vLLM page, "Background": fp4 indexer cache; SGLang
  article, section "FP4": two 4-bit values per byte).  Reading taken: OCP
  e2m1 (values 0, .5, 1, 1.5, 2, 3, 4, 6), round-to-nearest-even, saturating to
  +-6, one fp32 scale per 32 elements = amax/6 (1 when amax == 0); element 2j
  in the low nibble and 2j+1 in the high nibble of byte j.
* fp4 indexer cache with power-of-two block scales (the same bytes; reading
  of the summary article's remark that the indexer "computes in true FP4": a
  native fp4 tensor-core product scales each 32-element block by a power of
  two, the OCP Microscaling (MX) v1.0 convention for e2m1 with an E8M0 shared
  scale).  The scale is chosen by the MX conversion rule,
  X = 2^(floor(log2 amax) - 2), written into the fp32 scale word; codes are
  e2m1 of v / X (nearest-even, saturating to +-6).
* DeepSeek-V4 fp8 row of the SGLang KV-pool article (section "DeepSeek-V4",
  the per-token byte list): 448 fp8 "nope" elements, then the 64 rope
  elements in bf16 (128 B), then one scale byte per 64 nope elements (7 B),
  then 1 pad byte: 584 B per token; a page of P tokens is padded to
  ceil(P * 584 / 576) * 576 bytes.  Readings taken: the nope part is the
  first D - 64 elements of a D = 512 row and the rope part its last 64 (the
  rotary dims of every other layout here); a scale byte is an unsigned
  power-of-two exponent (UE8M0, value 2^(byte - 127)), chosen as the smallest
  power of two s with amax / s <= 448 (so no code saturates; 1 for amax = 0);
  codes are e4m3 of v / s (nearest-even); the pad byte is 0; the page's
  rows are consecutive from its first byte.
* Block layout (vLLM page, "A single logical block size": every compressed
  layer's logical block is 256 native positions, so a c4a block holds 64
  entries and a c128a block 2).  Reading taken for the bytes inside one
  physical block: all entries' data rows first ([entries][row]), then all
  scale words ([entries][scales per row] fp32).
"""
from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# bf16
# --------------------------------------------------------------------------

def bf16_decode(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _round_to_grid(mag: np.ndarray, mant_bits: int, min_exp_ulp: int) -> np.ndarray:
    """Round non-negative finite ``mag`` to the nearest value with
    ``mant_bits`` stored mantissa bits, ties to even; ``min_exp_ulp`` is
    log2 of the subnormal spacing.  Works because scaling by a power of two
    is exact in float64 and np.rint rounds half to even."""
    mag = np.asarray(mag, dtype=np.float64)
    _, e = np.frexp(mag)                      # mag = f * 2**e, f in [0.5, 1)
    ulp_exp = np.maximum(e - 1 - mant_bits, min_exp_ulp)
    ulp = np.ldexp(1.0, ulp_exp)
    return np.rint(mag / ulp) * ulp


def bf16_encode(x) -> np.ndarray:
    """float64 -> bf16 bit patterns, round-to-nearest-even, overflow -> inf."""
    x = np.asarray(x, dtype=np.float64)
    mag = _round_to_grid(np.abs(x), 7, -133)
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    mag = np.where(mag > bf16_max, np.inf, mag)
    val = np.where(np.signbit(x), -mag, mag)
    val = np.where(np.isnan(x), np.nan, val)
    bits = val.astype(np.float32).view(np.uint32) >> np.uint32(16)
    return bits.astype(np.uint16)


def bf16_round(x) -> np.ndarray:
    """float64 -> nearest bf16 value (as float64)."""
    return bf16_decode(bf16_encode(x))


def bf16_ulp(x) -> np.ndarray:
    """Spacing of bf16 values at |x| (the ulp of the bf16 binade of x)."""
    mag = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(mag == 0, 1e-300, mag))
    return np.ldexp(1.0, np.maximum(e - 8, -133))

# --------------------------------------------------------------------------
# fp8 e4m3fn
# --------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """uint8 e4m3fn codes -> float64; code 0x7f / 0xff decode to NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    sub = np.ldexp(man / 8.0, -6)
    nrm = np.ldexp(1.0 + man / 8.0, exp - 7)
    mag = np.where(exp == 0, sub, nrm)
    mag = np.where((exp == 15) & (man == 7), np.nan, mag)
    return sign * mag


_E4M3_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))   # codes 0..0x7e


def e4m3_encode(x) -> np.ndarray:
    """float64 -> e4m3fn codes, round-to-nearest-even, saturate to +-448."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.minimum(_round_to_grid(np.abs(x), 3, -9), E4M3_MAX)
    mag = np.where(np.isnan(x), 0.0, mag)
    code = np.searchsorted(_E4M3_POS, mag).astype(np.uint8)
    assert np.all(_E4M3_POS[code] == mag), "e4m3 grid rounding left the table"
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def e4m3_ulp(x) -> np.ndarray:
    """Spacing of e4m3 values at |x|."""
    mag = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(mag == 0, 1e-300, mag))
    return np.ldexp(1.0, np.maximum(e - 4, -9))

# --------------------------------------------------------------------------
# fp4 e2m1
# --------------------------------------------------------------------------

E2M1_MAX = 6.0
# OCP MX e2m1 magnitudes for codes 0..7 (sign in bit 3).
E2M1_TABLE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_decode(codes) -> np.ndarray:
    """4-bit e2m1 codes (0..15) -> float64, computed from the bit fields."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 0x8, -1.0, 1.0)
    exp = (c >> 1) & 0x3
    man = c & 0x1
    mag = np.where(exp == 0, 0.5 * man, np.ldexp(1.0 + man / 2.0, exp - 1))
    return sign * mag


def e2m1_encode(x) -> np.ndarray:
    """float64 -> e2m1 codes (uint8 0..15), nearest-even, saturate to +-6."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.minimum(_round_to_grid(np.abs(x), 1, -1), E2M1_MAX)
    code = np.searchsorted(E2M1_TABLE, mag).astype(np.uint8)
    assert np.all(E2M1_TABLE[code] == mag), "e2m1 grid rounding left the table"
    return np.where(np.signbit(x), code | 0x8, code).astype(np.uint8)


def e2m1_ulp(x) -> np.ndarray:
    mag = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(mag == 0, 1e-300, mag))
    return np.ldexp(1.0, np.maximum(e - 2, -1))

# --------------------------------------------------------------------------
# Scaled quantisers (conventions stated in the module docstring)
# --------------------------------------------------------------------------

def quant_scale(block: np.ndarray, qmax: float) -> float:
    amax = float(np.max(np.abs(block))) if block.size else 0.0
    return amax / qmax if amax > 0 else 1.0


def fp8_token_encode(v: np.ndarray):
    """One vector -> (e4m3 codes, fp32-representable scale as float64)."""
    s = float(np.float32(quant_scale(v, E4M3_MAX)))
    return e4m3_encode(v / s), s


def fp8_blocks_encode(v: np.ndarray, block: int):
    """Per-``block``-element fp8 quantisation of one vector."""
    n = v.shape[-1] // block
    codes = np.empty(v.shape[-1], np.uint8)
    scales = np.empty(n, np.float64)
    for b in range(n):
        seg = v[b * block:(b + 1) * block]
        s = float(np.float32(quant_scale(seg, E4M3_MAX)))
        codes[b * block:(b + 1) * block] = e4m3_encode(seg / s)
        scales[b] = s
    return codes, scales


def fp4_blocks_encode(v: np.ndarray, block: int = 32):
    """Per-32-element fp4 quantisation of one vector -> (packed bytes, scales)."""
    n = v.shape[-1] // block
    nib = np.empty(v.shape[-1], np.uint8)
    scales = np.empty(n, np.float64)
    for b in range(n):
        seg = v[b * block:(b + 1) * block]
        s = float(np.float32(quant_scale(seg, E2M1_MAX)))
        nib[b * block:(b + 1) * block] = e2m1_encode(seg / s)
        scales[b] = s
    return pack_nibbles(nib), scales


def mx_shared_scale(block: np.ndarray, emax_elem: int = 2) -> float:
    """Shared power-of-two scale of one block under the OCP Microscaling (MX)
    rule: X = 2^(floor(log2(amax)) - emax_elem), emax_elem = 2 for e2m1 (its
    largest power of two is 4).  amax = 0 gives 1 (the convention of the other
    scaled formats here).  The exponent is clamped to the normal fp32 range
    [-126, 127] because the scale is stored as an fp32 word."""
    amax = float(np.max(np.abs(block))) if block.size else 0.0
    if amax == 0.0:
        return 1.0
    _, e = np.frexp(amax)            # amax = f * 2^e, f in [0.5, 1)  ->  floor(log2 amax) = e - 1
    x = int(e) - 1 - emax_elem
    return float(np.ldexp(1.0, min(max(x, -126), 127)))


def fp4_mx_blocks_encode(v: np.ndarray, block: int = 32):
    """Per-32-element fp4 quantisation with OCP MX shared scales -> (packed
    bytes, scales).  v / X lies in [4, 8) for the block's largest element, so
    e2m1's saturation to +-6 clips what lies above 6 (as the MX conversion
    prescribes); every scale is an exact power of two."""
    n = v.shape[-1] // block
    nib = np.empty(v.shape[-1], np.uint8)
    scales = np.empty(n, np.float64)
    for b in range(n):
        seg = v[b * block:(b + 1) * block]
        s = mx_shared_scale(seg)
        nib[b * block:(b + 1) * block] = e2m1_encode(seg / s)
        scales[b] = s
    return pack_nibbles(nib), scales


def pack_nibbles(nib: np.ndarray) -> np.ndarray:
    nib = np.asarray(nib, np.uint8)
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, np.uint8)
    out = np.zeros(p.shape[:-1] + (p.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out

# --------------------------------------------------------------------------
# Paged-block byte layouts
# --------------------------------------------------------------------------

KV_BF16, KV_FP8_TOKEN, KV_FP8_DSV4 = 0, 1, 2
DSV4_NOPE, DSV4_ROPE, DSV4_QBLOCK, DSV4_ROW, DSV4_PAGE_UNIT = 448, 64, 64, 584, 576
# IX_FP4_MX32: the IX_FP4_B32 byte layout with every scale a power of two
# chosen by the OCP MX rule (mx_shared_scale).
IX_BF16, IX_FP8_B128, IX_FP4_B32, IX_FP4_MX32 = 0, 1, 2, 3
FP4_FORMATS = (IX_FP4_B32, IX_FP4_MX32)


def kv_block_bytes(fmt: int, entries: int, dim: int) -> int:
    """Bytes of one physical block of the shared-K=V compressed cache."""
    if fmt == KV_BF16:
        return entries * dim * 2
    if fmt == KV_FP8_TOKEN:
        return entries * dim + entries * 4
    if fmt == KV_FP8_DSV4:
        assert dim == DSV4_NOPE + DSV4_ROPE
        return -(-entries * DSV4_ROW // DSV4_PAGE_UNIT) * DSV4_PAGE_UNIT
    raise ValueError(fmt)


def ue8m0_e4m3_scale_byte(block: np.ndarray) -> int:
    """Scale byte b of one nope block: s = 2^(b - 127) is the smallest power
    of two with amax / s <= 448.  With amax = f * 2^e (f in [0.5, 1)) and
    448 = 0.875 * 2^9: amax / 2^k <= 448 iff f * 2^(e - 9 - k) <= 0.875, so
    k = e - 9, plus 1 when f > 0.875."""
    amax = float(np.max(np.abs(block))) if block.size else 0.0
    if amax == 0.0:
        return 127
    f, e = np.frexp(amax)
    k = int(e) - 9 + (1 if f > 0.875 else 0)
    return min(max(k + 127, 1), 254)


def dsv4_row_encode(v: np.ndarray) -> np.ndarray:
    """One D = 512 row -> its 584 bytes."""
    v = np.asarray(v, np.float64)
    out = np.zeros(DSV4_ROW, np.uint8)
    for j in range(DSV4_NOPE // DSV4_QBLOCK):
        seg = v[j * DSV4_QBLOCK:(j + 1) * DSV4_QBLOCK]
        b = ue8m0_e4m3_scale_byte(seg)
        out[j * DSV4_QBLOCK:(j + 1) * DSV4_QBLOCK] = e4m3_encode(np.ldexp(seg, 127 - b))
        out[DSV4_NOPE + 2 * DSV4_ROPE + j] = b
    out[DSV4_NOPE:DSV4_NOPE + 2 * DSV4_ROPE] = bf16_encode(v[DSV4_NOPE:]).view(np.uint8)
    return out


def dsv4_row_decode(raw: np.ndarray) -> np.ndarray:
    """584 bytes [..., 584] -> float64 [..., 512]."""
    raw = np.ascontiguousarray(raw, np.uint8)
    lead = raw.shape[:-1]
    codes = raw[..., :DSV4_NOPE].reshape(lead + (DSV4_NOPE // DSV4_QBLOCK, DSV4_QBLOCK))
    b = raw[..., DSV4_NOPE + 2 * DSV4_ROPE:DSV4_NOPE + 2 * DSV4_ROPE + DSV4_NOPE // DSV4_QBLOCK]
    nope = np.ldexp(e4m3_decode(codes), b.astype(np.int64)[..., None] - 127).reshape(lead + (DSV4_NOPE,))
    rope = bf16_decode(raw[..., DSV4_NOPE:DSV4_NOPE + 2 * DSV4_ROPE].copy().view(np.uint16))
    return np.concatenate([nope, rope], axis=-1)


def ix_block_bytes(fmt: int, dim: int, entries: int = 64) -> int:
    """Bytes of one physical block of the indexer-key cache."""
    if fmt == IX_BF16:
        return entries * dim * 2
    if fmt == IX_FP8_B128:
        return entries * dim + entries * (dim // 128) * 4
    if fmt in FP4_FORMATS:
        return entries * dim // 2 + entries * (dim // 32) * 4
    raise ValueError(fmt)


def kv_block_decode(raw: np.ndarray, fmt: int, entries: int, dim: int) -> np.ndarray:
    """Bytes of blocks [..., block_bytes] -> float64 [..., entries, dim]."""
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    lead = raw.shape[:-1]
    if fmt == KV_BF16:
        bits = raw[..., :entries * dim * 2].copy().view(np.uint16)
        return bf16_decode(bits).reshape(lead + (entries, dim))
    if fmt == KV_FP8_TOKEN:
        codes = raw[..., :entries * dim].reshape(lead + (entries, dim))
        scales = raw[..., entries * dim:entries * dim + 4 * entries].copy().view(np.float32)
        return e4m3_decode(codes) * scales.astype(np.float64)[..., None]
    if fmt == KV_FP8_DSV4:
        rows = raw[..., :entries * DSV4_ROW].reshape(lead + (entries, DSV4_ROW))
        return dsv4_row_decode(rows)
    raise ValueError(fmt)


def ix_block_decode(raw: np.ndarray, fmt: int, dim: int, entries: int = 64) -> np.ndarray:
    """Bytes of indexer blocks [..., block_bytes] -> float64 [..., entries, dim]."""
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    lead = raw.shape[:-1]
    if fmt == IX_BF16:
        bits = raw[..., :entries * dim * 2].copy().view(np.uint16)
        return bf16_decode(bits).reshape(lead + (entries, dim))
    if fmt == IX_FP8_B128:
        nb = dim // 128
        codes = raw[..., :entries * dim].reshape(lead + (entries, dim))
        sc = raw[..., entries * dim:entries * dim + 4 * entries * nb].copy().view(np.float32)
        sc = sc.astype(np.float64).reshape(lead + (entries, nb))
        return e4m3_decode(codes) * np.repeat(sc, 128, axis=-1)
    if fmt in FP4_FORMATS:
        nb = dim // 32
        packed = raw[..., :entries * dim // 2].reshape(lead + (entries, dim // 2))
        sc = raw[..., entries * dim // 2:entries * dim // 2 + 4 * entries * nb].copy().view(np.float32)
        sc = sc.astype(np.float64).reshape(lead + (entries, nb))
        return e2m1_decode(unpack_nibbles(packed)) * np.repeat(sc, 32, axis=-1)
    raise ValueError(fmt)
