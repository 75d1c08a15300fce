"""The page allocator (v4a_pages.h) on the host: the DeepSeek-V4 cache stack
folds into the three page-size buckets of "DeepSeek V4 in vLLM: Efficient
Long-context Attention" (Method details, "keeping the KV cache memory
packed"), a logical block is 256 native positions in every layer, and the
free lists never hand out a page twice."""
import os
import random

import numpy as np
import pytest

from compressed_sparse_long_c4a_gb300 import inputs as I
from compressed_sparse_long_c4a_gb300 import pages as P
from compressed_sparse_long_c4a_gb300 import v4a


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(v4a.LIB_PATH):
        from compressed_sparse_long_c4a_gb300 import build
        build.build()


def _v4_kinds(kv_fmt=I.KV_FP8_TOKEN, n_c4a=30, n_c128a=31, n_swa=0):
    """The five cache kinds of the model's layers (c4a KV, c4a indexer KV,
    c128a KV; SWA KV and the three compressor states as rings), with the 1M
    decode workloads' formats."""
    import dataclasses
    c4 = dataclasses.replace(I.c4a_decode_1m(), kv_fmt=kv_fmt)
    c128 = dataclasses.replace(I.c128a_decode_1m(), kv_fmt=kv_fmt)
    swa_slot = c4.dim + 4                               # fp8 window row + its scale
    kinds = [P.block_kind(c4.kv_block_bytes, n_c4a),                       # 0 c4a KV
             P.block_kind(c4.ix_block_bytes, n_c4a),                       # 1 indexer KV
             P.block_kind(c128.kv_block_bytes, n_c128a),                   # 2 c128a KV
             P.ring_kind(swa_slot, c4.swa_cap, 0, n_c4a + n_c128a + n_swa),  # 3 SWA KV
             P.ring_kind(2 * c4.dim + 4, c4.ring_cap, 0, n_c4a),           # 4 c4a state
             P.ring_kind(2 * c128.dim + 4, c128.ring_cap, 0, n_c128a),     # 5 c128a state
             P.ring_kind(2 * c4.ix_dim + 4, c4.ix_ring_cap, 1, n_c4a)]     # 6 indexer state
    return kinds, c4, c128


@pytest.mark.parametrize("kv_fmt", [I.KV_FP8_TOKEN, I.KV_FP8_DSV4])
def test_deepseek_v4_stack_folds_into_three_buckets(kv_fmt):
    kinds, c4, c128 = _v4_kinds(kv_fmt)
    a = P.PageAllocator(kinds, max_seqs=4, max_blocks=64, budget_bytes=1 << 34)
    assert a.num_buckets == 3
    pb = [b.page_bytes for b in a.buckets()]
    assert pb == sorted(pb, reverse=True)
    # largest: c4a KV, SWA KV, both compressor states; middle: the indexer KV
    # and the indexer's state; smallest: c128a KV
    want = {0: 0, 1: 1, 2: 2, 3: 0, 4: 0, 5: 0, 6: 1}
    assert {k: a.info(k).bucket for k in range(len(kinds))} == want
    # one logical block = 256 native positions: 64 c4a entries, 2 c128a entries
    if kv_fmt == I.KV_FP8_TOKEN:
        assert pb == [64 * (512 + 4), 64 * (128 // 2 + 4 * 128 // 32), 2 * (512 + 4)]
    else:   # 584-byte rows, pages padded to 576-byte units
        assert pb[0] == -(-64 * 584 // 576) * 576 == 65 * 576
        assert pb[2] == -(-2 * 584 // 576) * 576 == 3 * 576
        assert pb[1] == 64 * (64 + 16)


def test_ring_geometry():
    kinds, c4, c128 = _v4_kinds()
    a = P.PageAllocator(kinds, max_seqs=2, max_blocks=8, budget_bytes=1 << 32)
    for k in range(3, 7):
        i, kd = a.info(k), kinds[k]
        page = a.bucket(i.bucket).page_bytes
        assert i.slots == page // kd.slot_bytes >= 1
        assert i.ring_pages == -(-kd.ring_slots // i.slots)
        assert i.ring_cap == i.slots * i.ring_pages >= kd.ring_slots
        assert i.table_cols == i.ring_pages
        assert page % 16 == 0 and i.slots * kd.slot_bytes <= page
    # SWA: 64 fp8 rows of 516 B fill a c4a page exactly; 128 slots = 2 pages
    swa = a.info(3)
    assert (swa.slots, swa.ring_pages, swa.ring_cap) == (64, 2, 128)
    # the c128a state (window 128) takes 4 pages of 32 slots; c4a's (window 8) one
    assert (a.info(5).ring_pages, a.info(5).ring_cap) == (4, 128)
    assert (a.info(4).ring_pages, a.info(4).ring_cap) == (1, 32)


def test_pool_sizing_from_budget():
    kinds, _, _ = _v4_kinds(n_c4a=2, n_c128a=3)
    S, MB = 3, 40
    probe = P.PageAllocator(kinds, S, MB, budget_bytes=1 << 40)   # capped by S * MB blocks
    bk = probe.buckets()
    ring = [0, 0, 0]
    blk = [0, 0, 0]
    for k, kd in enumerate(kinds):
        i = probe.info(k)
        if kd.kind == P.RING:
            ring[i.bucket] += kd.layers * i.ring_pages
        else:
            blk[i.bucket] += kd.layers
    assert [b.num_pages for b in bk] == [S * r + S * MB * c for r, c in zip(ring, blk)]
    ring_bytes = sum(S * r * b.page_bytes for r, b in zip(ring, bk))
    per_block = sum(c * b.page_bytes for c, b in zip(blk, bk))
    budget = ring_bytes + 17 * per_block + per_block // 2
    a = P.PageAllocator(kinds, S, MB, budget_bytes=budget)
    assert [b.num_pages for b in a.buckets()] == [S * r + 17 * c for r, c in zip(ring, blk)]
    assert sum(b.num_pages * b.page_bytes for b in a.buckets()) <= budget
    assert all(b.free_pages == b.num_pages for b in a.buckets())
    with pytest.raises(v4a.V4AError) as e:
        P.PageAllocator(kinds, S, MB, budget_bytes=ring_bytes + per_block - 1)
    assert e.value.code == P.ERR_OUT_OF_PAGES


def _check_invariants(a: P.PageAllocator, kinds, model_blocks: dict):
    """Every table entry of an open sequence is a distinct page of its
    bucket; closed sequences and blocks beyond a sequence's count hold -1;
    free + used = pool size."""
    used = {b: [] for b in range(a.num_buckets)}
    for k, kd in enumerate(kinds):
        i = a.info(k)
        for layer in range(kd.layers):
            t = a.table(k, layer)
            for s in range(a.max_seqs):
                row = t[s]
                if s not in model_blocks:
                    assert (row == -1).all()
                elif kd.kind == P.RING:
                    assert (row >= 0).all()
                    used[i.bucket] += row.tolist()
                else:
                    n = model_blocks[s]
                    assert (row[:n] >= 0).all() and (row[n:] == -1).all()
                    used[i.bucket] += row[:n].tolist()
    for b in range(a.num_buckets):
        bk = a.bucket(b)
        assert len(set(used[b])) == len(used[b])                 # no page handed out twice
        assert all(0 <= p < bk.num_pages for p in used[b])
        assert bk.free_pages + len(used[b]) == bk.num_pages
    for s in range(a.max_seqs):
        assert a.blocks(s) == model_blocks.get(s, -1)


def test_random_open_reserve_close_keeps_the_books():
    kinds, _, _ = _v4_kinds(n_c4a=2, n_c128a=2, n_swa=1)
    S, MB = 5, 24
    probe = P.PageAllocator(kinds, S, MB, budget_bytes=1 << 40)
    ring_b = sum(S * kd.layers * probe.info(k).ring_pages * probe.bucket(probe.info(k).bucket).page_bytes
                 for k, kd in enumerate(kinds) if kd.kind == P.RING)
    per_block = sum(kd.layers * kd.page_bytes for kd in kinds if kd.kind == P.BLOCK)
    a = P.PageAllocator(kinds, S, MB, budget_bytes=ring_b + 40 * per_block)   # 40 of 120 blocks
    rng = random.Random(7)
    model = {}
    n_out = 0
    for _ in range(400):
        s = rng.randrange(S)
        op = rng.random()
        before = a.tables().copy()
        if s not in model:
            if op < 0.2:
                with pytest.raises(v4a.V4AError):
                    a.reserve(s, 10)                    # not open
                continue
            a.open(s)
            model[s] = 0
        elif op < 0.2:
            a.close(s)
            del model[s]
        else:
            pos = rng.randrange(0, MB * 256 + 1)
            need = -(-pos // 256)
            grow = max(0, need - model[s])
            if grow > a.bucket(2).free_pages // 2:      # c128a KV: 2 layers per block
                with pytest.raises(v4a.V4AError) as e:
                    a.reserve(s, pos)
                assert e.value.code == P.ERR_OUT_OF_PAGES
                assert np.array_equal(a.tables(), before)   # a failed reserve changes nothing
                n_out += 1
            else:
                a.reserve(s, pos)
                model[s] = max(model[s], need)
        _check_invariants(a, kinds, model)
    assert n_out > 0


def test_block_reserves_256_positions_in_every_layer():
    kinds, _, _ = _v4_kinds(n_c4a=3, n_c128a=2)
    a = P.PageAllocator(kinds, 2, 16, budget_bytes=1 << 36)
    a.open(1)
    for pos, blocks in ((1, 1), (256, 1), (257, 2), (3 * 256, 3), (100, 3)):   # never shrinks
        a.reserve(1, pos)
        assert a.blocks(1) == blocks
        for k, kd in enumerate(kinds):
            if kd.kind == P.BLOCK:
                for layer in range(kd.layers):
                    row = a.table(k, layer)[1]
                    assert (row[:blocks] >= 0).all() and (row[blocks:] == -1).all()
    with pytest.raises(v4a.V4AError):
        a.reserve(1, 16 * 256 + 1)                      # beyond max_blocks


def test_freed_pages_serve_another_kind_of_the_bucket():
    """One pool per bucket: pages that held a sequence's c4a KV are handed to
    the rings (SWA KV, compressor states) of a later sequence."""
    kinds, _, _ = _v4_kinds(n_c4a=1, n_c128a=1)
    probe = P.PageAllocator(kinds, 2, 64, budget_bytes=1 << 36)
    ring_b = sum(2 * kd.layers * probe.info(k).ring_pages * probe.bucket(probe.info(k).bucket).page_bytes
                 for k, kd in enumerate(kinds) if kd.kind == P.RING)
    per_block = sum(kd.layers * kd.page_bytes for kd in kinds if kd.kind == P.BLOCK)
    a = P.PageAllocator(kinds, 2, 64, budget_bytes=ring_b + 64 * per_block)   # rings of 2 + 64 blocks
    a.open(0)
    a.reserve(0, 64 * 256)
    kv_pages = set(a.table(0, 0)[0].tolist())
    assert len(kv_pages) == 64
    a.close(0)
    a.open(1)
    a.open(0)                                           # the rest of the bucket: former KV pages
    ring_pages = set()
    for k in (3, 4, 5):                                 # SWA, c4a state, c128a state
        for layer in range(kinds[k].layers):
            ring_pages |= set(a.table(k, layer)[0].tolist())
    assert ring_pages and ring_pages <= kv_pages
    a.reserve(0, 64 * 256)                              # the bucket's last 64 pages
    assert a.bucket(0).free_pages == 0
    with pytest.raises(v4a.V4AError) as e:
        a.reserve(1, 1)
    assert e.value.code == P.ERR_OUT_OF_PAGES


def test_rejected_plans_and_calls():
    kinds, c4, c128 = _v4_kinds()
    E = v4a.V4AError
    with pytest.raises(E):      # a ring naming a bucket that does not exist
        P.PageAllocator(kinds + [P.ring_kind(100, 8, 3, 1)], 2, 8, 1 << 34)
    with pytest.raises(E):      # a slot larger than the bucket's page
        P.PageAllocator(kinds + [P.ring_kind(10 ** 6, 8, 0, 1)], 2, 8, 1 << 34)
    with pytest.raises(E):      # a ring in a bucket whose page is not a multiple of 16 (1032 B)
        P.PageAllocator(kinds + [P.ring_kind(100, 8, 2, 1)], 2, 8, 1 << 34)
    with pytest.raises(E):      # rings only: no page size
        P.PageAllocator([P.ring_kind(100, 8, 0, 1)], 2, 8, 1 << 34)
    with pytest.raises(E):
        P.PageAllocator(kinds, 0, 8, 1 << 34)
    a = P.PageAllocator(kinds, 2, 8, 1 << 34)
    a.open(0)
    with pytest.raises(E):
        a.open(0)               # already open
    with pytest.raises(E):
        a.close(1)              # not open
    with pytest.raises(E):
        a.open(2)               # out of range
    assert a.blocks(1) == -1 and a.blocks(0) == 0
