"""GPU parity of the paths that only some shapes reach, against the fp64
oracle, through the C ABI:

* the CUDA-core indexer scan (bf16 keys; fp8 / fp4 / MX fp4 keys with a head
  count the tensor-core scans do not take) on rows long enough for the
  multi-CTA top-k (histogram kernel, filter, final);
* the long-row top-k after each tensor-core scan (fp8, fp4, MX fp4 keys);
* the CUDA-core attention (head dim 64; 256 heads);
* the window ring read from pages of a pool, on both attention paths.

Scores must agree entry by entry within 1e-5 of the query's score scale; the
top-k sets may differ only by swaps within 1e-5 of the k-th score; attention
within the bf16 tolerances of the workload."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from compressed_sparse_long_c4a_gb300 import inputs as I
from tests import gpu_util as U
from tests import oracle_bridge as OB

pytestmark = pytest.mark.gpu


def _v4a():
    from compressed_sparse_long_c4a_gb300 import v4a
    return v4a


def _index_specs():
    one_k, b32, m1 = I.c4a_decode_1k(), I.c4a_decode_b32_32k_64k(), I.c4a_decode_1m()
    r = dataclasses.replace
    return {
        # CUDA-core scan: bf16 keys (4 heads x 64), rows of 37,504 entries (> 32,768: multi-CTA top-k)
        "simt_bf16_long": r(one_k, name="simt_bf16_long", batch=2, cached=(4 * 30000 + 3, 150001)),
        # CUDA-core scan: 32 heads (the tensor-core scans take 64)
        "simt_fp8_32h": r(b32, name="simt_fp8_32h", batch=2, cached=(4 * 30000 + 3, 140001), ix_heads=32),
        "simt_fp4_32h": r(m1, name="simt_fp4_32h", batch=2, cached=(150003, 140001), ix_heads=32),
        "simt_mx_32h": r(m1, name="simt_mx_32h", batch=2, cached=(150003, 140001), ix_heads=32,
                         ix_fmt=I.IX_FP4_MX32),
        # tensor-core scans on rows of ~100k entries
        "tc_fp8_long": r(b32, name="tc_fp8_long", batch=2, cached=(4 * 100000 + 3, 300001)),
        "tc_fp4_long": r(m1, name="tc_fp4_long", batch=3, cached=(4 * 100000 + 3, 300001, 256 * 700 + 255)),
        "tc_mx_long": r(m1, name="tc_mx_long", batch=3, cached=(4 * 100000 + 3, 300001, 256 * 700 + 255),
                        ix_fmt=I.IX_FP4_MX32),
    }


INDEX = _index_specs()


@pytest.mark.parametrize("name", list(INDEX))
def test_index_scores_and_topk(name):
    v4a = _v4a()
    spec = INDEX[name]
    case = I.make_case(spec, seed=7)
    L = v4a.DeviceLayer.from_case(case)
    step = v4a.Step(L)
    v4a.index_scores(L, step.idx, step.ws_index)
    torch.cuda.synchronize()
    assert int(L.status.item()) == 0
    sc = v4a.index_scores_view(L, step.ws_index).cpu().numpy()
    idx, scores = OB.oracle_index(case, OB.u8(case.ix_pool))
    for t, ref in scores.items():
        got = sc[t, :ref.shape[0]].astype(np.float64)
        err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
        assert err <= 1e-5, (name, t, err)
    v4a.index_topk(L, step.idx, step.ws_index)
    torch.cuda.synchronize()
    assert int(L.status.item()) == 0
    gpu = step.idx.cpu().numpy()
    for t in idx:
        U.check_topk(gpu[t], idx[t], scores[t], spec.topk, f"{name} t={t}")


def _attn_specs():
    one_k = I.c4a_decode_1k()
    r = dataclasses.replace
    return {
        "simt_attn_d64": r(one_k, name="simt_attn_d64", batch=3, dim=64, rope_dims=32,
                           cached=(1024, 3001, 700)),
        "simt_attn_h256": r(one_k, name="simt_attn_h256", batch=2, heads=256, cached=(1024, 2047)),
    }


ATTN = _attn_specs()


@pytest.mark.parametrize("name", list(ATTN))
def test_cuda_core_attention(name):
    """Attention on the oracle's own selection over the generator's caches."""
    v4a = _v4a()
    spec = ATTN[name]
    case = I.make_case(spec, seed=8)
    L = v4a.DeviceLayer.from_case(case)
    step = v4a.Step(L, fused_out=False)
    oidx, _ = OB.oracle_index(case, OB.u8(case.ix_pool))
    full = np.full((spec.tokens, spec.topk), -1, np.int64)
    for t, v in oidx.items():
        full[t] = v
    idx_t = torch.from_numpy(full.astype(np.int32)).cuda()
    v4a.sparse_attn(L, idx_t, step.o, step.lse, step.ws_attn)
    torch.cuda.synchronize()
    assert int(L.status.item()) == 0
    ring = OB.u16(case.swa_ring)
    ref = OB.oracle_attention(case, OB.u8(case.kv_pool), ring, None, {t: full[t] for t in range(spec.tokens)})
    o = step.o.float().cpu().numpy()
    U.check_close(o, np.stack([ref[t][0] for t in range(spec.tokens)]), U.BF16_TOL, name)
    assert np.allclose(step.lse.cpu().numpy(), np.stack([ref[t][1] for t in range(spec.tokens)]),
                       atol=1e-3, rtol=1e-4)


def _paged_window(case, spec, slots, seed):
    """The case's window ring as slots in pages of one pool under a shuffled
    page table (the v4a_ring_pages layout: [slots][row] then [slots] fp32)."""
    B, cap, D = spec.batch, spec.swa_cap, spec.dim
    fp8 = spec.swa_fmt == I.KV_FP8_TOKEN
    rb = D if fp8 else 2 * D
    pb = -(-slots * (rb + (4 if fp8 else 0)) // 16) * 16
    per = cap // slots
    assert per * slots == cap
    g = torch.Generator().manual_seed(seed)
    npages = B * per + 3
    table = torch.randperm(npages, generator=g)[:B * per].to(torch.int32).view(B, per)
    pool = torch.zeros(npages * pb, dtype=torch.uint8)
    rows = case.swa_ring.contiguous().view(torch.uint8).view(B, cap, rb)
    for b in range(B):
        for s in range(cap):
            base = int(table[b, s // slots]) * pb
            j = s % slots
            pool[base + j * rb: base + (j + 1) * rb] = rows[b, s]
            if fp8:
                pool[base + slots * rb + 4 * j: base + slots * rb + 4 * j + 4] = \
                    case.swa_scale[b, s].reshape(1).view(torch.uint8)
    return pool.cuda(), table.cuda(), npages, pb


PAGED_WINDOW = {
    "simt_attn_d64": (ATTN["simt_attn_d64"], 32),
    "simt_attn_h256": (ATTN["simt_attn_h256"], 64),
    "tc_fp8_window": (dataclasses.replace(I.c4a_decode_1m(), name="tc_fp8_window", batch=2,
                                          cached=(4 * 3000 + 3, 9001)), 16),
    "tc_bf16_window": (dataclasses.replace(I.c4a_decode_1k(), name="tc_bf16_window", batch=3,
                                           cached=(1024, 3001, 700)), 128),
}


@pytest.mark.parametrize("name", list(PAGED_WINDOW))
def test_paged_window_equals_dense_window(name):
    """Attention over every visible entry with the window read from pages of
    a pool (shuffled page table) writes the same output and lse bytes as
    with the per-sequence ring: CUDA-core path (head dim 64, 256 heads) and
    tensor-core path (fp8 and bf16 windows)."""
    import ctypes as C
    v4a = _v4a()
    spec, slots = PAGED_WINDOW[name]
    case = I.make_case(spec, seed=5)
    L = v4a.DeviceLayer.from_case(case)
    T, H, D = spec.tokens, spec.heads, spec.dim
    ws = torch.empty(max(v4a.attn_workspace_bytes(L, False), 256), dtype=torch.uint8, device="cuda")
    o1 = torch.empty((T, H, D), dtype=torch.bfloat16, device="cuda")
    l1 = torch.empty((T, H), dtype=torch.float32, device="cuda")
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    v4a.sparse_attn(L, None, o1, l1, ws)
    pool, table, npages, pb = _paged_window(case, spec, slots, seed=11)
    rp = v4a.RingPages(pool.data_ptr(), npages, pb, table.data_ptr(), slots)
    a = L.attn_args(None, o2, l2)
    a.window, a.window_scale, a.window_pages = None, None, C.pointer(rp)
    rc = v4a.lib().v4a_sparse_attn(C.byref(a), ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(L.status.item()) == 0
    assert torch.equal(o1.cpu(), o2.cpu()) and torch.equal(l1.cpu(), l2.cpu())
