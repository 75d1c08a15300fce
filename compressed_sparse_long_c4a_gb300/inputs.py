"""Seeded synthetic workloads for the compressed sparse attention layer.

This module only draws random numbers and lays them out in the library's
buffer formats.  It holds none of the method's arithmetic (no compression,
normalisation, rotation, quantisation rule, scoring or attention), so both the
CUDA path and the fp64 oracle can take their inputs from it.

Each workload is one layer step over a ragged batch: every sequence has
``cached`` native tokens already processed (caches, rings and the sliding
window filled "as if by earlier steps" with random contents) and ``new``
tokens arriving at positions cached .. cached+new-1.  The new tokens are also
the queries.  Distributions follow the five workloads of the layer:

* compressor inputs x ~ N(0,1) (bf16), gate logits ~ N(0,1), per-offset bias
  ~ N(0, 0.5^2), RMSNorm gamma ~ 1 + N(0, 0.1^2);
* queries, window keys and bf16 cache entries ~ N(0,1) (bf16);
* indexer head weights ~ U(0,1);
* fp8 codes are the e4m3 cast (a library cast) of N(0,1)*100, clamped to
  +-448, with fp32 scales ~ U(0.5,1.5)/100, so decoded values are ~N(0,1);
* DeepSeek-V4 584-byte rows: e4m3 codes as above, scale bytes uniform on
  {119, 120, 121} (2^-8 .. 2^-6), rope values ~ N(0,1) in bf16;
* fp4 codes are drawn from a fixed categorical law over the 8 e2m1
  magnitudes (small codes most likely) with a random sign, with fp32 scales
  ~ U(0.5,1.5)/2, or, for the power-of-two (MX) scale format, scales 2^e with
  e uniform on {-3, -2, -1};
* block tables are a seeded random permutation of the physical pool.

Sub-seeds: every tensor gets its own generator seeded with (seed, tensor id).
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import torch

BLOCK_POSITIONS = 256
KV_BF16, KV_FP8_TOKEN, KV_FP8_DSV4 = 0, 1, 2
IX_BF16, IX_FP8_B128, IX_FP4_B32, IX_FP4_MX32 = 0, 1, 2, 3
Q_BF16, Q_FP8_HEAD = 0, 1
OUT_BF16, OUT_FP8_TOKEN = 0, 1


@dataclass(frozen=True)
class LayerSpec:
    """One layer step: geometry, formats and the ragged batch shape."""
    name: str
    ratio: int                 # 4 (c4a) or 128 (c128a)
    batch: int                 # sequences
    heads: int                 # query heads H
    dim: int                   # shared K=V dim D
    cached: tuple              # per-sequence cached native tokens (before the step)
    new: int = 1               # new tokens (queries) per sequence
    rope_dims: int = 64
    theta: float = 10000.0
    kv_fmt: int = KV_BF16
    swa_fmt: int = KV_BF16
    ix_heads: int = 0          # 0: no indexer (c128a attends to every entry)
    ix_dim: int = 0
    ix_fmt: int = IX_BF16
    ix_q_fmt: int = Q_BF16
    topk: int = 0              # 0: all visible entries
    swa: int = 128
    out_fmt: int = OUT_BF16
    spare_blocks: int = 3      # unused physical blocks in the pool
    window_only: bool = False  # pure sliding-window layer: attention over the window alone
    q_prep: bool = False       # the step normalises and rotates the raw queries (fusion (3))
    ix_q_prep: bool = False    # the step rotates + encodes the raw indexer query (fp8 query only)

    @property
    def entries_per_block(self) -> int:
        return BLOCK_POSITIONS // self.ratio

    @property
    def ix_rope_dims(self) -> int:
        return self.ix_dim // 2

    @property
    def ix_w_mult(self) -> float:
        """Constant of the indexer weights' multiplication: 1/sqrt(H_I * d_I)."""
        return float((self.ix_heads * self.ix_dim) ** -0.5) if self.ix_heads else 1.0

    @property
    def window(self) -> int:
        return 8 if self.ratio == 4 else 128

    @property
    def tokens(self) -> int:
        return self.batch * self.new

    @property
    def max_pos(self) -> int:
        return max(self.cached) + self.new - 1

    @property
    def max_blocks(self) -> int:
        return (self.max_pos + BLOCK_POSITIONS) // BLOCK_POSITIONS

    @property
    def num_blocks(self) -> int:
        return self.batch * self.max_blocks + self.spare_blocks

    @property
    def kv_block_bytes(self) -> int:
        e = self.entries_per_block
        if self.kv_fmt == KV_FP8_DSV4:      # 584-byte rows, pages padded to 576-byte units
            return -(-e * 584 // 576) * 576
        return e * self.dim * 2 if self.kv_fmt == KV_BF16 else e * self.dim + 4 * e

    @property
    def ix_block_bytes(self) -> int:
        d = self.ix_dim
        if self.ix_fmt == IX_BF16:
            return 64 * d * 2
        if self.ix_fmt == IX_FP8_B128:
            return 64 * d + 64 * (d // 128) * 4
        return 64 * d // 2 + 64 * (d // 32) * 4

    @property
    def ring_cap(self) -> int:
        """Compressor ring capacity: window - 1 + new tokens per call."""
        return self.window - 1 + self.new

    @property
    def ix_ring_cap(self) -> int:
        return 8 - 1 + self.new

    @property
    def swa_cap(self) -> int:
        return self.swa - 1 + self.new


def _gen(seed: int, tid: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed((seed * 1_000_003 + tid * 7919) & 0x7FFF_FFFF_FFFF)
    return g


def _randn(shape, seed, tid, std=1.0, mean=0.0):
    return torch.randn(shape, generator=_gen(seed, tid), dtype=torch.float32) * std + mean


def _rand(shape, seed, tid, lo=0.0, hi=1.0):
    return torch.rand(shape, generator=_gen(seed, tid), dtype=torch.float32) * (hi - lo) + lo


def _bf16(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.bfloat16)


def _fp8_codes(shape, seed, tid) -> torch.Tensor:
    v = (_randn(shape, seed, tid) * 100.0).clamp(-448.0, 448.0)
    return v.to(torch.float8_e4m3fn).view(torch.uint8)


_FP4_MAG_LAW = torch.tensor([0.14, 0.20, 0.20, 0.15, 0.12, 0.10, 0.06, 0.03])


def _fp4_bytes(nbytes_shape, seed, tid) -> torch.Tensor:
    g = _gen(seed, tid)
    n = int(math.prod(nbytes_shape)) * 2
    mag = torch.multinomial(_FP4_MAG_LAW, n, replacement=True, generator=g).to(torch.uint8)
    sign = (torch.rand(n, generator=g) < 0.5).to(torch.uint8) << 3
    nib = (mag | sign).view(-1, 2)
    return (nib[:, 0] | (nib[:, 1] << 4)).view(nbytes_shape)


def _scales(n, seed, tid, base) -> torch.Tensor:
    return _rand((n,), seed, tid, 0.5, 1.5) / base


def _pow2_scales(n, seed, tid) -> torch.Tensor:
    e = torch.randint(-3, 0, (n,), generator=_gen(seed, tid))
    return torch.pow(2.0, e.to(torch.float32))


@dataclass
class Case:
    """All tensors of one layer step (CPU), in the library's layouts."""
    spec: LayerSpec
    seed: int
    seq_ids: torch.Tensor          # [T] int32
    positions: torch.Tensor        # [T] int32
    block_table: torch.Tensor      # [B][max_blocks] int32 (-1 = unallocated)
    kv_pool: torch.Tensor          # [NB * kv_block_bytes] uint8
    x: torch.Tensor                # [T][D] bf16 main compressor input
    gate: torch.Tensor             # [T] fp32
    bias: torch.Tensor             # [window] fp32
    gamma: torch.Tensor            # [D] fp32
    ring_x: torch.Tensor           # [B][Rc][D] bf16
    ring_gate: torch.Tensor        # [B][Rc] fp32
    k_swa: torch.Tensor            # [T][D] bf16 (pre-RoPE window key)
    swa_ring: torch.Tensor         # [B][Rs][D] bf16 or uint8
    swa_scale: torch.Tensor        # [B][Rs] fp32 (fp8 window only; else empty)
    q: torch.Tensor                # [T][H][D] bf16 (already rotated; the step's output when q_prep)
    ix_pool: torch.Tensor | None = None
    x_i: torch.Tensor | None = None
    gate_i: torch.Tensor | None = None
    bias_i: torch.Tensor | None = None
    gamma_i: torch.Tensor | None = None
    ring_x_i: torch.Tensor | None = None
    ring_gate_i: torch.Tensor | None = None
    q_i: torch.Tensor | None = None        # [T][HI][dI] bf16 or uint8 codes
    q_i_scale: torch.Tensor | None = None  # [T][HI] fp32 (fp8 query)
    w_i: torch.Tensor | None = None        # [T][HI] fp32
    o_in: torch.Tensor | None = None       # [T][H][D] bf16 (input of the output stage)
    q_raw: torch.Tensor | None = None      # [T][H][D] bf16 query before norm + RoPE (q_prep)
    gamma_q: torch.Tensor | None = None    # [D] fp32 query RMSNorm weight (q_prep)
    q_i_raw: torch.Tensor | None = None    # [T][HI][dI] bf16 indexer query before RoPE + fp8 (ix_q_prep)
    w_i_raw: torch.Tensor | None = None    # [T][HI] fp32 head weights before the multiplication (ix_q_prep)


def make_case(spec: LayerSpec, seed: int = 0) -> Case:
    s = spec
    B, T, D, C = s.batch, s.tokens, s.dim, s.new
    seq_ids = torch.arange(B, dtype=torch.int32).repeat_interleave(C)
    positions = torch.cat([torch.arange(c, c + C, dtype=torch.int32) for c in s.cached])

    perm = torch.randperm(s.num_blocks, generator=_gen(seed, 1)).to(torch.int32)
    bt = torch.full((B, s.max_blocks), -1, dtype=torch.int32)
    for b in range(B):
        need = (s.cached[b] + C - 1) // BLOCK_POSITIONS + 1
        bt[b, :need] = perm[b * s.max_blocks: b * s.max_blocks + need]

    nb = s.num_blocks
    e = s.entries_per_block
    if s.kv_fmt == KV_BF16:
        kv = _bf16(_randn((nb, e * D), seed, 2)).view(torch.uint8).reshape(nb, -1)
    elif s.kv_fmt == KV_FP8_DSV4:
        # 584-byte rows: 448 e4m3 codes, 64 bf16 rope values, 7 scale bytes
        # (2^-8 .. 2^-6: with the codes' ~N(0,1)*100 the decoded values are
        # ~N(0,1) within a factor of two), 1 zero pad byte; zero page padding
        codes = _fp8_codes((nb, e, 448), seed, 2)
        rope = _bf16(_randn((nb, e, 64), seed, 3)).view(torch.uint8).reshape(nb, e, 128)
        sb = torch.randint(119, 122, (nb, e, 7), generator=_gen(seed, 15), dtype=torch.int64).to(torch.uint8)
        rows = torch.cat([codes, rope, sb, torch.zeros((nb, e, 1), dtype=torch.uint8)], dim=2).reshape(nb, -1)
        kv = torch.cat([rows, torch.zeros((nb, s.kv_block_bytes - e * 584), dtype=torch.uint8)], dim=1)
    else:
        codes = _fp8_codes((nb, e * D), seed, 2)
        sc = _scales(nb * e, seed, 3, 100.0).view(torch.uint8).reshape(nb, -1)
        kv = torch.cat([codes, sc], dim=1)
    kv_pool = kv.reshape(-1).contiguous()

    W = s.window
    case = Case(
        spec=s, seed=seed, seq_ids=seq_ids, positions=positions, block_table=bt,
        kv_pool=kv_pool,
        x=_bf16(_randn((T, D), seed, 4)),
        gate=_randn((T,), seed, 5),
        bias=_randn((W,), seed, 6, std=0.5),
        gamma=_randn((D,), seed, 7, std=0.1, mean=1.0),
        ring_x=_bf16(_randn((B, s.ring_cap, D), seed, 8)),
        ring_gate=_randn((B, s.ring_cap), seed, 9),
        k_swa=_bf16(_randn((T, D), seed, 10)),
        swa_ring=(_bf16(_randn((B, s.swa_cap, D), seed, 11)) if s.swa_fmt == KV_BF16
                  else _fp8_codes((B, s.swa_cap, D), seed, 11)),
        swa_scale=(torch.empty(0) if s.swa_fmt == KV_BF16
                   else _scales(B * s.swa_cap, seed, 12, 100.0).view(B, s.swa_cap)),
        q=_bf16(_randn((T, s.heads, D), seed, 13)),
        o_in=_bf16(_randn((T, s.heads, D), seed, 14, std=0.3)),
    )
    if s.ix_heads:
        HI, dI = s.ix_heads, s.ix_dim
        if s.ix_fmt == IX_BF16:
            ix = _bf16(_randn((nb, 64 * dI), seed, 20)).view(torch.uint8).reshape(nb, -1)
        elif s.ix_fmt == IX_FP8_B128:
            codes = _fp8_codes((nb, 64 * dI), seed, 20)
            sc = _scales(nb * 64 * (dI // 128), seed, 21, 100.0).view(torch.uint8).reshape(nb, -1)
            ix = torch.cat([codes, sc], dim=1)
        else:
            packed = _fp4_bytes((nb, 64 * dI // 2), seed, 20)
            if s.ix_fmt == IX_FP4_MX32:
                sc = _pow2_scales(nb * 64 * (dI // 32), seed, 21)
            else:
                sc = _scales(nb * 64 * (dI // 32), seed, 21, 2.0)
            ix = torch.cat([packed, sc.view(torch.uint8).reshape(nb, -1)], dim=1)
        case.ix_pool = ix.reshape(-1).contiguous()
        case.x_i = _bf16(_randn((T, dI), seed, 22))
        case.gate_i = _randn((T,), seed, 23)
        case.bias_i = _randn((8,), seed, 24, std=0.5)
        case.gamma_i = _randn((dI,), seed, 25, std=0.1, mean=1.0)
        case.ring_x_i = _bf16(_randn((B, s.ix_ring_cap, dI), seed, 26))
        case.ring_gate_i = _randn((B, s.ix_ring_cap), seed, 27)
        if s.ix_q_fmt == Q_BF16:
            case.q_i = _bf16(_randn((T, HI, dI), seed, 28))
            case.q_i_scale = torch.ones((T, HI), dtype=torch.float32)
        else:
            case.q_i = _fp8_codes((T, HI, dI), seed, 28)
            case.q_i_scale = _scales(T * HI, seed, 29, 100.0).view(T, HI)
        case.w_i = _rand((T, HI), seed, 30)
    if s.q_prep:
        case.q_raw = _bf16(_randn((T, s.heads, D), seed, 31, std=2.0))
        case.gamma_q = _randn((D,), seed, 32, std=0.1, mean=1.0)
    if s.ix_q_prep:
        assert s.ix_heads and s.ix_q_fmt == Q_FP8_HEAD
        case.q_i_raw = _bf16(_randn((T, s.ix_heads, s.ix_dim), seed, 33))
        case.w_i_raw = _rand((T, s.ix_heads), seed, 34)
    return case


def uniform_lengths(batch: int, lo: int, hi: int, seed: int, tid: int) -> list[int]:
    g = _gen(seed, tid)
    return [int(v) for v in torch.randint(lo, hi + 1, (batch,), generator=g)]


# --------------------------------------------------------------------------
# The five workloads of the layer (seed 0)
# --------------------------------------------------------------------------

def c4a_decode_1k() -> LayerSpec:
    """c4a decode, 1 sequence, 1024 cached tokens + 1 query (m = 1024)."""
    return LayerSpec(name="c4a_decode_b1_1k", ratio=4, batch=1, heads=16, dim=128,
                     cached=(1024,), ix_heads=4, ix_dim=64, ix_fmt=IX_BF16,
                     ix_q_fmt=Q_BF16, topk=32)


def c4a_decode_b32_32k_64k(seed: int = 0) -> LayerSpec:
    """c4a decode, batch 32, contexts ~U[32k, 64k]; four sequences pinned to
    compression and block boundaries (emit, first-slot emit, last-slot emit,
    block start)."""
    L = uniform_lengths(32, 32768, 65536, seed, 100)
    L[0] = 4 * 9000 + 3              # m = 4i+3: emits entry i
    L[1] = 256 * 200 + 3             # emits into the first slot of a block
    L[2] = 256 * 201 + 255           # emits into the last slot of a block
    L[3] = 256 * 202                 # first position of a fresh block
    return LayerSpec(name="c4a_decode_b32_32k_64k", ratio=4, batch=32, heads=64, dim=512,
                     cached=tuple(L), ix_heads=64, ix_dim=128, ix_fmt=IX_FP8_B128,
                     ix_q_fmt=Q_FP8_HEAD, topk=512)


def c128a_decode_b64_64k_128k(seed: int = 0) -> LayerSpec:
    """c128a decode, batch 64, contexts ~U[64k, 128k], all entries + window."""
    L = uniform_lengths(64, 65536, 131072, seed, 101)
    L[0] = 128 * 700 + 127           # emits a c128a entry (second slot of a block)
    L[1] = 128 * 702 + 127           # emits into the first slot of a block
    return LayerSpec(name="c128a_decode_b64_64k_128k", ratio=128, batch=64, heads=64,
                     dim=512, cached=tuple(L), topk=0)


def c4a_prefill_4x4k() -> LayerSpec:
    """c4a chunked prefill: 4 sequences x (32768 cached + 4096 new)."""
    return LayerSpec(name="c4a_prefill_4x32k_plus_4k", ratio=4, batch=4, heads=64, dim=512,
                     cached=(32768,) * 4, new=4096, ix_heads=64, ix_dim=128,
                     ix_fmt=IX_FP8_B128, ix_q_fmt=Q_FP8_HEAD, topk=512)


def c4a_decode_1m() -> LayerSpec:
    """c4a decode at 1M context, batch 4, fp8 attention cache, fp4 indexer,
    fp8 output (the queries arrive normalised and rotated).  m = 1,048,575
    emits entry 262,143 (the last slot of a block), so each query sees
    262,144 entries."""
    return LayerSpec(name="c4a_decode_b4_1m", ratio=4, batch=4, heads=128, dim=512,
                     cached=(1_048_575,) * 4, kv_fmt=KV_FP8_TOKEN, swa_fmt=KV_FP8_TOKEN,
                     ix_heads=64, ix_dim=128, ix_fmt=IX_FP4_B32, ix_q_fmt=Q_FP8_HEAD,
                     topk=2048, out_fmt=OUT_FP8_TOKEN, spare_blocks=1)


def c4a_decode_1m_dsv4() -> LayerSpec:
    """c4a_decode_b4_1m with the attention cache in the DeepSeek-V4 584-byte
    fp8 layout of the SGLang KV-pool article (448 fp8 nope with a scale byte
    per 64, 64 bf16 rope, pages padded to 576-byte units)."""
    return dataclasses.replace(c4a_decode_1m(), name="c4a_decode_b4_1m_dsv4", kv_fmt=KV_FP8_DSV4)


def c4a_decode_1m_mx() -> LayerSpec:
    """c4a_decode_b4_1m with the fp4 indexer's per-32 fp32 scales restricted to
    powers of two (the OCP MX rule; same bytes per entry), which the tensor
    cores apply inside a block-scaled MMA."""
    return dataclasses.replace(c4a_decode_1m(), name="c4a_decode_b4_1m_mx", ix_fmt=IX_FP4_MX32)


def c4a_decode_1m_qprep() -> LayerSpec:
    """c4a_decode_b4_1m with the queries' RMSNorm + RoPE inside the step
    (the query side of the horizontal fusion with the window-key insert)."""
    return dataclasses.replace(c4a_decode_1m(), name="c4a_decode_b4_1m_qprep", q_prep=True)


def c4a_decode_1m_ixprep() -> LayerSpec:
    """c4a_decode_b4_1m with the indexer query's RoPE + per-head fp8 + weight
    multiplication inside the step."""
    return dataclasses.replace(c4a_decode_1m(), name="c4a_decode_b4_1m_ixprep", ix_q_prep=True)


def c4a_decode_128k() -> LayerSpec:
    """c4a_decode_b4_1m at 128k context: m = 131,071 emits entry 32,767 (the
    last slot of a block), so each query sees 32,768 entries (the low end of
    the 128k-1M range the decode target names)."""
    return dataclasses.replace(c4a_decode_1m(), name="c4a_decode_b4_128k", cached=(131_071,) * 4)


def swa_decode_1m() -> LayerSpec:
    """A pure sliding-window layer of the same model at 1M context, batch 4:
    attention over the last 128 tokens only (no compressed entries), fp8
    window, fp8 output.  The compressed-cache geometry is c128a's (its cache
    is allocated but never read)."""
    return LayerSpec(name="swa_decode_b4_1m", ratio=128, batch=4, heads=128, dim=512,
                     cached=(1_048_575,) * 4, kv_fmt=KV_FP8_TOKEN, swa_fmt=KV_FP8_TOKEN,
                     out_fmt=OUT_FP8_TOKEN, spare_blocks=1, window_only=True)


def c128a_decode_1m() -> LayerSpec:
    """A c128a layer of the same model at 1M context, batch 4: attention over
    all 8,192 compressed entries plus the window, fp8 caches and output."""
    return LayerSpec(name="c128a_decode_b4_1m", ratio=128, batch=4, heads=128, dim=512,
                     cached=(1_048_575,) * 4, kv_fmt=KV_FP8_TOKEN, swa_fmt=KV_FP8_TOKEN,
                     out_fmt=OUT_FP8_TOKEN, spare_blocks=1)


WORKLOADS = {
    "c4a_decode_b1_1k": c4a_decode_1k,
    "c4a_decode_b32_32k_64k": c4a_decode_b32_32k_64k,
    "c128a_decode_b64_64k_128k": c128a_decode_b64_64k_128k,
    "c4a_prefill_4x32k_plus_4k": c4a_prefill_4x4k,
    "c4a_decode_b4_1m": c4a_decode_1m,
    "c4a_decode_b4_1m_mx": c4a_decode_1m_mx,
    "c4a_decode_b4_128k": c4a_decode_128k,
    "c128a_decode_b4_1m": c128a_decode_1m,
    "c4a_decode_b4_1m_dsv4": c4a_decode_1m_dsv4,
    "c4a_decode_b4_1m_qprep": c4a_decode_1m_qprep,
}


def shrink(spec: LayerSpec, **kw) -> LayerSpec:
    """A smaller variant of a workload (same formats), for fast tests."""
    return dataclasses.replace(spec, **kw)
