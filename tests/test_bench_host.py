"""Host logic of bench.py that needs no GPU: the timed-window statistics and
the --gpus launcher contract (N ranks started through torch.distributed.run
when no launcher did it; a mismatched world size is an error)."""
import sys
import types

import pytest

import bench


def test_window_stats_median_and_spread():
    st = bench.window_stats([1.0, 1.2, 0.9, 1.1, 1.05])
    assert st["count"] == 5
    assert st["median"] == pytest.approx(1.05)
    assert st["min"] == 0.9 and st["max"] == 1.2
    assert st["spread_pct"] == pytest.approx((1.2 - 0.9) / 1.05 * 100.0)
    assert st["ms_per_step"] == [1.0, 1.2, 0.9, 1.1, 1.05]   # in window order


def test_gpus_n_without_launcher_starts_n_ranks(monkeypatch):
    calls = []
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: calls.append(cmd) or 0)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "4", "--steps", "5"])
    with pytest.raises(SystemExit) as e:
        bench._relaunch_if_needed(types.SimpleNamespace(gpus=4))
    assert e.value.code == 0
    (cmd,) = calls
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"]
    assert "--nproc-per-node=4" in cmd and "127.0.0.1" in cmd
    assert cmd[-4:] == ["--gpus", "4", "--steps", "5"]


def test_gpus_n_launch_failure_is_nonzero(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: 3)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "2"])
    with pytest.raises(SystemExit) as e:
        bench._relaunch_if_needed(types.SimpleNamespace(gpus=2))
    assert e.value.code == 3


def test_world_size_mismatch_exits_nonzero(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit) as e:
        bench._relaunch_if_needed(types.SimpleNamespace(gpus=4))
    assert e.value.code not in (0, None)


def test_single_gpu_and_matching_launcher_run_in_process(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench._relaunch_if_needed(types.SimpleNamespace(gpus=1))
    monkeypatch.setenv("WORLD_SIZE", "4")
    bench._relaunch_if_needed(types.SimpleNamespace(gpus=4))
