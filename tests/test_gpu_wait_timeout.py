"""Failure detection on the GPU without a fault: the kernels' bounded mbarrier
wait, run against a barrier nothing arrives at, gives up after its limit, sets
DCP_ERR_TIMEOUT in the status word, and leaves the context usable."""

from __future__ import annotations

import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "context_decode_attention_paged_gb300", "csrc")
DCP_ERR_TIMEOUT = 4


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    out = tmp_path_factory.mktemp("wait") / "libwait_timeout.so"
    from context_decode_attention_paged_gb300.build import ARCH, nvcc
    cmd = [nvcc(), *ARCH, "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-I", CSRC,
           "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "cuda", "wait_timeout.cu"),
           "-o", str(out)]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(str(out))
    lib.wait_timeout_probe.restype = ctypes.c_int
    lib.wait_timeout_probe.argtypes = [ctypes.c_ulonglong, ctypes.c_int] + [ctypes.c_void_p] * 4
    return lib


@pytest.mark.parametrize("limit_ms", [5, 50])
def test_bounded_wait_gives_up_and_reports(probe, limit_ms):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    gave_up = torch.zeros(1, dtype=torch.int32, device="cuda")
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    threads = 64
    rc = probe.wait_timeout_probe(limit_ms * 1_000_000, threads, status.data_ptr(), elapsed.data_ptr(),
                                  gave_up.data_ptr(), counter.data_ptr())
    assert rc == 0, rc
    assert int(status.item()) == DCP_ERR_TIMEOUT
    assert int(gave_up.item()) == threads          # every waiting thread gave up
    ms = int(elapsed.item()) / 1e6
    assert limit_ms <= ms < limit_ms + 1000, ms    # no earlier than the limit, and bounded
    assert int(counter.item()) == 128              # the context still runs kernels
    # and the library's own calls still work on the same context
    x = torch.ones(4, device="cuda")
    assert float(x.sum().item()) == 4.0
