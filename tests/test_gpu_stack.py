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
    att = OB.oracle_attention(case, kv, ring, rsc, {t: np.zeros(0, np.int64) for t in range(s.tokens)})
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
    att = OB.oracle_attention(case, kv, ring, rsc, None)
    U.check_close(step.o.float().cpu().numpy(), np.stack([att[t][0] for t in range(s.tokens)]), U.FP8_TOL,
                  "c128a fp8")
    assert np.allclose(step.lse.cpu().numpy(), np.stack([att[t][1] for t in range(s.tokens)]), atol=1e-3,
                       rtol=1e-4)
