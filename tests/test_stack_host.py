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
