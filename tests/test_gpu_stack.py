"""Pure sliding-window layers (attention over the window alone) and the
attention stack replayed from one CUDA graph."""
import numpy as np
import pytest
import torch

from compressed_sparse_long_c4a_gb300 import stack as S
from oracle import formats as F
from tests import gpu_util as U
from tests import oracle_bridge as OB

pytestmark = pytest.mark.gpu


def test_window_only_attention_matches_oracle():
    from compressed_sparse_long_c4a_gb300 import v4a
    case = S.shrink_cases()["swa"]
    s = case.spec
    L = v4a.DeviceLayer.from_case(case)
    step = v4a.Step(L, fused_out=False)
    step.run()
    torch.cuda.synchronize()
    assert int(L.status.item()) == 0
    # the oracle's chain on its own window insert, attention over no compressed entry
    main, ix, swa = OB.oracle_compress(case)
    kv, ixp, ring, rsc = OB.oracle_state_after_compress(case, main, ix, swa)
    att = OB.oracle_attention(case, kv, ring, rsc, {t: np.zeros(0, np.int64) for t in range(s.tokens)},
                              q_bits=OB.step_q_bits(case))
    U.check_close(step.o.float().cpu().numpy(), np.stack([att[t][0] for t in range(s.tokens)]), U.FP8_TOL,
                  "window only")
    lse_ref = np.stack([att[t][1] for t in range(s.tokens)])
    assert np.allclose(step.lse.cpu().numpy(), lse_ref, atol=1e-3, rtol=1e-4)
    # the fused call takes the same shapes and writes the same bytes
    Lf = v4a.DeviceLayer.from_case(case)
    fused = v4a.Step(Lf)
    fused.run()
    torch.cuda.synchronize()
    assert fused.fused_out and torch.equal(fused.out.cpu(), step.out.cpu())


def test_stack_graph_replay_equals_layer_by_layer():
    """A graph of the mixed stack, replayed once, leaves every layer's output
    and caches as running its layers one after another does."""
    cases = S.shrink_cases()
    kinds = ["c128a", "c4a", "swa", "c4a", "c128a"]
    a, b = S.AttentionStack(kinds, cases), S.AttentionStack(kinds, cases)
    a.run()
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = b.capture(stream)
    g.replay()
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    for la, lb, sa, sb in zip(a.layers, b.layers, a.steps, b.steps):
        assert torch.equal(sa.out.cpu(), sb.out.cpu())
        for k in ("kv_pool", "swa_ring", "ix_pool"):
            if k in la.t:
                assert torch.equal(la.t[k].cpu(), lb.t[k].cpu()), k
    assert a.launches_per_step() > len(kinds)


def test_c128a_fp8_layer_matches_oracle():
    """A c128a layer with fp8 caches (2 x 516-byte entries per block: rows on
    8 bytes, so the CUDA-core attention takes it) against the oracle."""
    from compressed_sparse_long_c4a_gb300 import v4a
    case = S.shrink_cases()["c128a"]
    s = case.spec
    L = v4a.DeviceLayer.from_case(case)
    step = v4a.Step(L, fused_out=False)
    step.run()
    torch.cuda.synchronize()
    assert int(L.status.item()) == 0
    main, ix, swa = OB.oracle_compress(case)
    kv, ixp, ring, rsc = OB.oracle_state_after_compress(case, main, ix, swa)
    att = OB.oracle_attention(case, kv, ring, rsc, None, q_bits=OB.step_q_bits(case))
    U.check_close(step.o.float().cpu().numpy(), np.stack([att[t][0] for t in range(s.tokens)]), U.FP8_TOL,
                  "c128a fp8")
    assert np.allclose(step.lse.cpu().numpy(), np.stack([att[t][1] for t in range(s.tokens)]), atol=1e-3,
                       rtol=1e-4)


def _pages_of(stack, name, li):
    dev, host, info = stack._table(name, li)
    bk = stack.alloc.bucket(info.bucket)
    return stack.pools[info.bucket].view(-1, bk.page_bytes), host


def test_paged_stack_equals_dense_stack():
    """Caches and rings of every layer as pages of the allocator's three
    bucket pools, replayed from one CUDA graph: the same output bytes and
    selections as the stack with per-layer buffers, and every cache block
    (the step's new entries included) holds the same bytes in its page."""
    cases = S.shared_context_cases()
    kinds = ["c128a", "c4a", "swa", "c4a", "c128a"]
    dense = S.AttentionStack(kinds, cases)
    paged = S.AttentionStack(kinds, cases, paged=True)
    assert len(paged.pools) == 3
    assert [paged.alloc.info(paged.slot[n]).bucket for n in ("c4a.kv", "c4a.swa", "c4a.state", "c128a.state",
                                                             "c128a.swa", "swa.swa")] == [0] * 6
    assert [paged.alloc.info(paged.slot[n]).bucket for n in ("c4a.ix", "c4a.ix_state", "c128a.kv")] == [1, 1, 2]
    dense.run()
    stream = torch.cuda.Stream()
    g = paged.capture(stream)
    g.replay()
    torch.cuda.synchronize()
    assert dense.status() == 0 and paged.status() == 0
    seen = {}
    for k, ld, lp, sd, sp in zip(kinds, dense.layers, paged.layers, dense.steps, paged.steps):
        li = seen.get(k, 0)
        seen[k] = li + 1
        assert torch.equal(sd.out.cpu(), sp.out.cpu()), k
        if sd.out_scale is not None:
            assert torch.equal(sd.out_scale.cpu(), sp.out_scale.cpu()), k
        if sd.idx is not None:
            assert torch.equal(sd.idx.cpu(), sp.idx.cpu()), k
        if k == "swa":
            continue
        bt = cases[k].block_table.numpy()
        mask = bt >= 0
        for pool_key, name in (("kv_pool", f"{k}.kv"), ("ix_pool", f"{k}.ix")):
            if pool_key not in ld.t:
                continue
            pages, host = _pages_of(paged, name, li)
            dpool = ld.t[pool_key].view(-1, pages.shape[1])
            src = torch.from_numpy(bt[mask].astype(np.int64)).cuda()
            dst = torch.from_numpy(host[mask].astype(np.int64)).cuda()
            assert torch.equal(dpool[src].cpu(), pages[dst].cpu()), name


def test_paged_layers_match_oracle():
    """A c128a layer and a window-only layer read their caches and windows
    from pages (compress, then attention with per-call outputs) and agree
    with the oracle's chain on the same case."""
    from compressed_sparse_long_c4a_gb300 import v4a
    cases = S.shared_context_cases()
    st = S.AttentionStack(["c4a", "c128a", "swa"], cases, paged=True)
    for li, kind in ((1, "c128a"), (2, "swa")):
        case = cases[kind]
        s = case.spec
        L = st.layers[li]
        step = v4a.Step(L, fused_out=False)
        step.run()
        torch.cuda.synchronize()
        assert int(L.status.item()) == 0, kind
        main, ix, swa = OB.oracle_compress(case)
        kv, ixp, ring, rsc = OB.oracle_state_after_compress(case, main, ix, swa)
        sel = {t: np.zeros(0, np.int64) for t in range(s.tokens)} if kind == "swa" else None
        att = OB.oracle_attention(case, kv, ring, rsc, sel, q_bits=OB.step_q_bits(case))
        U.check_close(step.o.float().cpu().numpy(), np.stack([att[t][0] for t in range(s.tokens)]), U.FP8_TOL,
                      f"paged {kind}")
        assert np.allclose(step.lse.cpu().numpy(), np.stack([att[t][1] for t in range(s.tokens)]), atol=1e-3,
                           rtol=1e-4)
