"""The timeout path of the bounded waits, exercised without a fault: a
test-only kernel (tests/cuda/wait_timeout_probe.cu, compiled here, never part
of libv4a) waits on an mbarrier that nothing completes.  The library's wait
must give up after its limit, set V4A_DEV_TIMEOUT in the status word and
return; a kernel launched afterwards must still run (the context is usable)."""
import ctypes
import os
import shutil
import subprocess
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "compressed_sparse_long_c4a_gb300", "csrc")
SRC = os.path.join(ROOT, "tests", "cuda", "wait_timeout_probe.cu")
V4A_DEV_TIMEOUT = 8


def _build(tmp_path) -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    so = str(tmp_path / "libwait_probe.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"), "-I", CSRC, SRC, "-o", so],
                   check=True, capture_output=True)
    return so


def test_probe_source_compiles_for_sm103a(tmp_path):
    """Host-only: the probe builds (nvcc cross-compiles without a GPU)."""
    if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        pytest.skip("no nvcc")
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
def test_bounded_wait_reports_timeout_and_context_survives(tmp_path):
    import torch
    lib = ctypes.CDLL(_build(tmp_path))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gave_up = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    rc = lib.v4a_probe_wait_timeout(ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(gave_up.data_ptr()))
    waited = time.time() - t0
    assert rc == 0, f"the probe kernel failed (cuda error {rc})"
    assert int(gave_up.item()) == 1
    assert int(status.item()) & V4A_DEV_TIMEOUT
    assert waited < 30.0
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.v4a_probe_after(ctypes.c_void_p(out.data_ptr()), 1234) == 0
    assert int(out.item()) == 1234
    # and the library itself still runs a call on the same device
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == pytest.approx(1023 * 1024 / 2)
