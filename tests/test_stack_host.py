"""Host side of the attention stack: the layer mix, and a pin of the oracle's
window-only attention against the textbook softmax attention computed here
from library casts."""
import math

import numpy as np
import torch

from compressed_sparse_long_c4a_gb300 import inputs as I
from compressed_sparse_long_c4a_gb300 import stack as S
from tests import oracle_bridge as OB


def test_deepseek_v4_mix_counts_and_order():
    kinds = S.deepseek_v4_mix()
    assert len(kinds) == 61 and kinds.count("c4a") == 30 and kinds.count("c128a") == 31
    assert kinds[:4] == ["c128a", "c4a", "c128a", "c4a"] and kinds[-1] == "c128a"
    assert S.deepseek_v4_mix(2, 1, 3) == ["c128a", "c4a", "c4a", "swa", "swa", "swa"]


def test_oracle_window_only_attention_is_softmax_over_the_window():
    import dataclasses
    spec = dataclasses.replace(I.swa_decode_1m(), name="swa_tiny", batch=2, heads=4, dim=128,
                               rope_dims=64, cached=(300, 40))
    case = I.make_case(spec, 3)
    att = OB.oracle_attention(case, OB.u8(case.kv_pool), OB.u8(case.swa_ring), case.swa_scale.double().numpy(),
                              {t: np.zeros(0, np.int64) for t in range(spec.tokens)})
    tau = 1.0 / math.sqrt(spec.dim)
    for t in range(spec.tokens):
        b, m = int(case.seq_ids[t]), int(case.positions[t])
        lo = max(0, m - spec.swa + 1)
        slots = [p % spec.swa_cap for p in range(lo, m + 1)]
        codes = case.swa_ring[b, slots]                                    # e4m3 codes
        keys = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy() * \
            case.swa_scale[b, slots].double().numpy()[:, None]
        q = case.q[t].to(torch.float64).numpy()
        z = tau * q @ keys.T
        p = np.exp(z - z.max(axis=1, keepdims=True))
        o = (p / p.sum(axis=1, keepdims=True)) @ keys
        lse = np.log(p.sum(axis=1)) + z.max(axis=1)
        assert np.allclose(att[t][0], o, rtol=1e-12, atol=1e-12)
        assert np.allclose(att[t][1], lse, rtol=1e-12, atol=1e-12)


def test_paged_stack_places_every_slot_the_kernels_read():
    """The paged stack built on the CPU (no kernel runs): every cache block
    of the synthetic cases is in the page its table names, and every ring
    position a step reads (the compressor windows and the attention window)
    is at page table[b][s // slots], index s % slots, s = p % ring_cap, with
    its fp32 after the page's rows (the v4a_ring_pages layout)."""
    cases = S.shared_context_cases()
    kinds = ["c4a", "c128a", "swa", "c4a"]
    st = S.AttentionStack(kinds, cases, device="cpu", paged=True)
    assert len(st.pools) == 3
    seen = {}
    for k, L in zip(kinds, st.layers):
        li = seen.get(k, 0)
        seen[k] = li + 1
        case = cases[k]
        s = case.spec
        bt = case.block_table.numpy()
        caches = [] if k == "swa" else [(f"{k}.kv", case.kv_pool)] + ([("c4a.ix", case.ix_pool)] if k == "c4a" else [])
        for name, dense in caches:
            dev, host, info = st._table(name, li)
            pb = st.alloc.bucket(info.bucket).page_bytes
            pages = st.pools[info.bucket].view(-1, pb)
            for b in range(s.batch):
                for lb in np.nonzero(bt[b] >= 0)[0]:
                    assert torch.equal(pages[host[b, lb]], dense.view(-1, pb)[bt[b, lb]]), (name, b, lb)
            assert torch.equal(dev, torch.from_numpy(host))
        rings = [(f"{k}.swa", case.swa_ring, case.swa_scale if case.swa_scale.numel() else None, s.swa - 1)]
        if k != "swa":
            rings.append((f"{k}.state", case.ring_x, case.ring_gate, s.window - 1))
        if k == "c4a":
            rings.append(("c4a.ix_state", case.ring_x_i, case.ring_gate_i, 7))
        for name, rows, side, back in rings:
            dev, host, info = st._table(name, li)
            pb = st.alloc.bucket(info.bucket).page_bytes
            pool = st.pools[info.bucket]
            cap = rows.shape[1]
            rb = rows[0, 0].numel() * rows.element_size()
            rows8 = rows.contiguous().view(torch.uint8).view(s.batch, cap, rb)
            for b in range(s.batch):
                for p in range(max(0, s.cached[b] - back), s.cached[b]):
                    sp = p % info.ring_cap
                    page, j = int(host[b, sp // info.slots]), sp % info.slots
                    base = page * pb
                    assert torch.equal(pool[base + j * rb: base + (j + 1) * rb], rows8[b, p % cap]), (name, b, p)
                    if side is not None:
                        got = pool[base + info.slots * rb + 4 * j: base + info.slots * rb + 4 * j + 4]
                        assert torch.equal(got, side[b, p % cap].reshape(1).view(torch.uint8)), (name, b, p)


def test_paged_stack_rejects_what_the_allocator_cannot_plan():
    """One context per sequence in every layer (a logical block reserves the
    same 256 positions everywhere), and at least one compressed cache to
    size the pages; a c128a-only stack's one bucket (1,032-byte pages) cannot
    hold rings, whose pages need 16-byte strides."""
    import pytest
    cases = S.shared_context_cases()
    mixed = dict(cases, c128a=S.shrink_cases()["c128a"])          # another context
    with pytest.raises(ValueError):
        S.AttentionStack(["c4a", "c128a"], mixed, device="cpu", paged=True)
    with pytest.raises(ValueError):
        S.AttentionStack(["swa"], cases, device="cpu", paged=True)
    from compressed_sparse_long_c4a_gb300 import v4a
    with pytest.raises(v4a.V4AError):
        S.AttentionStack(["c128a"], cases, device="cpu", paged=True)
