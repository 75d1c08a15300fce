"""Edge cases of the GPU path through the C ABI: empty batches, fewer visible
entries than k, all-tied scores (both top-k paths), the first c4a entry, an
unallocated block (device status bit, no fault), and a prefill chunk equal
byte for byte to the same tokens fed one at a time."""
from __future__ import annotations

import ctypes as C
import dataclasses

import numpy as np
import pytest
import torch

from compressed_sparse_long_c4a_gb300 import inputs as I
from oracle import formats as F
from oracle import geometry as G
from tests import gpu_util as U
from tests import oracle_bridge as OB

pytestmark = pytest.mark.gpu


def _v4a():
    from compressed_sparse_long_c4a_gb300 import v4a
    return v4a


def test_empty_batch_launches_nothing():
    v4a = _v4a()
    case = I.make_case(I.c4a_decode_1k(), seed=0)
    L = v4a.DeviceLayer.from_case(case)
    step = v4a.Step(L)
    a, keep = L.compress_args()
    a.batch.num_tokens = 0
    assert v4a.lib().v4a_compress_insert(C.byref(a), None) == 0
    ia = L.index_args(step.idx)
    ia.batch.num_tokens = 0
    assert v4a.lib().v4a_index_topk(C.byref(ia), None, 0, None) == 0
    aa = L.attn_args(step.idx, step.o, step.lse)
    aa.batch.num_tokens = 0
    assert v4a.lib().v4a_sparse_attn(C.byref(aa), None, 0, None) == 0
    torch.cuda.synchronize()


def test_fewer_entries_than_k_and_first_entry():
    """m = 3 emits entry 0 from positions 0..3 only; m = 41 sees 10 < k entries."""
    v4a = _v4a()
    spec = dataclasses.replace(I.c4a_decode_1k(), name="short", batch=2, cached=(3, 41))
    case = I.make_case(spec, seed=1)
    L = v4a.DeviceLayer.from_case(case)
    step = v4a.Step(L, fused_out=False)   # the bf16 attention output is checked
    step.run()
    torch.cuda.synchronize()
    assert int(L.status.item()) == 0
    main, ix, swa = OB.oracle_compress(case)
    assert (0, 0) in main and (0, 0) in ix
    kv, ixp, ring, rsc = OB.oracle_state_after_compress(case, main, ix, swa)
    blk, slot = G.slot_of(case.block_table.numpy()[0], 0, 4)
    row, _ = U.kv_slot_bytes(L.t["kv_pool"].cpu().numpy(), spec, blk, slot)
    U.check_bf16_row(row, main[(0, 0)], "entry 0")
    idx, scores = OB.oracle_index(case, ixp)
    gpu = step.idx.cpu().numpy()
    for t in range(2):
        U.check_topk(gpu[t], idx[t], scores[t], spec.topk, f"t={t}")
    assert list(gpu[0][:2]) == [0, -1] and list(gpu[1][:10]) == list(range(10)) and gpu[1][10] == -1
    att = OB.oracle_attention(case, kv, ring, rsc, idx)
    U.check_close(step.o.float().cpu().numpy(), np.stack([att[t][0] for t in range(2)]), U.BF16_TOL)


@pytest.mark.parametrize("fmt", [I.IX_FP4_B32, I.IX_FP4_MX32])
@pytest.mark.parametrize("cached", [(12000, 16000), (40003, 39000), (150003, 140000)])
def test_all_tied_scores_take_lowest_indices(cached, fmt):
    """w = 0 makes every score 0: the top-k must be the k lowest entry indices
    (single-CTA path while a block-table row spans <= 32K entries, multi-CTA
    path beyond: 150,003 positions give rows of 37,504 entries)."""
    v4a = _v4a()
    spec = dataclasses.replace(I.c4a_decode_1m(), name="ties", batch=2, cached=cached, ix_fmt=fmt)
    case = I.make_case(spec, seed=2)
    case.w_i = torch.zeros_like(case.w_i)
    L = v4a.DeviceLayer.from_case(case)
    step = v4a.Step(L)
    v4a.index_topk(L, step.idx, step.ws_index)
    torch.cuda.synchronize()
    assert int(L.status.item()) == 0
    gpu = step.idx.cpu().numpy()
    for t in range(2):
        assert gpu[t].tolist() == list(range(spec.topk))


def test_unallocated_block_sets_status_without_fault():
    v4a = _v4a()
    spec = dataclasses.replace(I.c4a_decode_b32_32k_64k(), name="holes", batch=2, cached=(5003, 9000))
    case = I.make_case(spec, seed=3)
    case.block_table[1, 3] = -1           # a block the indexer and attention both need
    L = v4a.DeviceLayer.from_case(case)
    step = v4a.Step(L, fused_out=False)
    step.run()
    torch.cuda.synchronize()
    st = int(L.status.item())
    assert st & v4a.DEV_BAD_BLOCK
    assert not st & 8                    # no timeout
    o = step.o.float().cpu().numpy()
    assert np.isfinite(o).all()
    # the fused attention + output call on the same holes: same status, finite output
    L2 = v4a.DeviceLayer.from_case(case)
    fused = v4a.Step(L2, fused_out=True)
    fused.run()
    torch.cuda.synchronize()
    st2 = int(L2.status.item())
    assert st2 & v4a.DEV_BAD_BLOCK and not st2 & 8
    assert torch.equal(fused.out.cpu(), step.out.cpu())


def _sub_batch(L, case, rows):
    """Batch struct + kept tensors for the tokens `rows` of `case`."""
    v4a = _v4a()
    idx = torch.tensor(rows, dtype=torch.long)
    keep = {}
    for f in ("seq_ids", "positions", "x", "gate", "x_i", "gate_i", "k_swa"):
        v = getattr(case, f)
        if v is not None:
            keep[f] = v[idx].contiguous().cuda()
    return keep


def test_chunk_equals_single_token_steps():
    v4a = _v4a()
    spec = dataclasses.replace(I.c4a_prefill_4x4k(), name="chunk", batch=2, cached=(1000, 1535), new=37,
                               topk=64)
    case = I.make_case(spec, seed=4)
    A = v4a.DeviceLayer.from_case(case)
    v4a.compress_insert(A)
    B = v4a.DeviceLayer.from_case(case)
    s = spec
    for j in range(s.new):
        rows = [b * s.new + j for b in range(s.batch)]
        k = _sub_batch(B, case, rows)
        saved = {f: B.t[f] for f in k}
        B.t.update(k)
        a, keep = B.compress_args()
        a.batch.num_tokens = len(rows)
        a.batch.max_new_per_seq = 1
        rc = v4a.lib().v4a_compress_insert(C.byref(a), C.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0
        torch.cuda.synchronize()
        B.t.update(saved)
    torch.cuda.synchronize()
    assert int(A.status.item()) == 0 and int(B.status.item()) == 0
    for f in ("kv_pool", "ix_pool", "swa_ring", "ring_x", "ring_gate", "ring_x_i", "ring_gate_i"):
        assert torch.equal(A.t[f], B.t[f]), f
