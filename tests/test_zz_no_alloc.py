"""v4a_index_topk_static: the indexer top-k with the library's fixed device
scratch instead of a caller workspace.  It must select exactly what
v4a_index_topk selects, call after call (the shared scratch carries the
previous call's leftovers), and refuse, launching nothing, arguments that need
more scratch than the fixed array holds.

This file is collected last so the GPU tests also run after every other test
in the same process; it passes on its own as well."""
from __future__ import annotations

import ctypes as C
import dataclasses
import os

import pytest
import torch

from compressed_sparse_long_c4a_gb300 import inputs as I
from compressed_sparse_long_c4a_gb300 import v4a

V4A_ERR_WORKSPACE = 4


def _lib():
    if not os.path.exists(v4a.LIB_PATH):
        from compressed_sparse_long_c4a_gb300 import build
        build.build()
    return v4a.lib()


def _shape_only_args(spec) -> v4a.IndexArgs:
    """Index arguments with every pointer NULL: enough to size the scratch."""
    s = spec
    batch = v4a.Batch(s.tokens, None, None, s.batch, s.new)
    keys = v4a.Cache(4, s.ix_dim, s.ix_rope_dims, s.theta, s.ix_fmt, None, s.num_blocks, None, s.max_blocks)
    return v4a.IndexArgs(batch, keys, s.ix_heads, s.ix_q_fmt, None, None, None, s.topk, None, None)


def _oversize_spec():
    # 90 prefill queries over ~50K entries: ~20 MB of scratch (> 16 MiB)
    return dataclasses.replace(I.c4a_decode_1m(), name="static_oversize", batch=1, cached=(200001,), new=90)


def test_oversize_rejected_on_host():
    """The size check comes before any CUDA call, so it runs without a GPU."""
    lib = _lib()
    a = _shape_only_args(_oversize_spec())
    assert lib.v4a_index_workspace_size(C.byref(a)) > v4a.INDEX_STATIC_SCRATCH_BYTES
    assert lib.v4a_index_topk_static(C.byref(a), None) == V4A_ERR_WORKSPACE


def _cases():
    return [
        I.c4a_decode_1k(),                                           # one-CTA top-k path
        dataclasses.replace(I.c4a_decode_1m(), name="static_multi", batch=2,
                            cached=(150003, 200001)),                # multi-CTA path (rows > 32K)
    ]


@pytest.mark.gpu
def test_static_scratch_matches_workspace_call_twice_in_a_row():
    _lib()
    layers = []
    for n, spec in enumerate(_cases()):
        case = I.make_case(spec, seed=40 + n)
        L = v4a.DeviceLayer.from_case(case)
        v4a.compress_insert(L)
        ws = torch.empty(max(v4a.index_workspace_bytes(L), 256), dtype=torch.uint8, device="cuda")
        assert ws.numel() <= v4a.INDEX_STATIC_SCRATCH_BYTES
        ref = torch.full((spec.tokens, spec.topk), -7, dtype=torch.int32, device="cuda")
        v4a.index_topk(L, ref, ws)
        layers.append((spec, L, ref))
    torch.cuda.synchronize()
    # each case twice in a row, then the cases again in the other order: every
    # call starts from the previous call's leftovers in the shared scratch
    order = [0, 0, 1, 1, 0, 1]
    for i in order:
        spec, L, ref = layers[i]
        got = torch.full_like(ref, -9)
        v4a.index_topk_static(L, got)
        torch.cuda.synchronize()
        assert int(L.status.item()) == 0, spec.name
        assert torch.equal(got, ref), spec.name     # integer indices: exact


@pytest.mark.gpu
def test_static_scratch_refuses_oversize_and_launches_nothing():
    _lib()
    spec = _oversize_spec()
    case = I.make_case(spec, seed=43)
    L = v4a.DeviceLayer.from_case(case)
    assert v4a.index_workspace_bytes(L) > v4a.INDEX_STATIC_SCRATCH_BYTES
    out = torch.full((spec.tokens, spec.topk), -5, dtype=torch.int32, device="cuda")
    with pytest.raises(v4a.V4AError) as e:
        v4a.index_topk_static(L, out)
    assert e.value.code == V4A_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == -5).all())
    assert int(L.status.item()) == 0
