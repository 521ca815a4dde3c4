"""tcgen05 operand forms (A in TMEM, K-major 128B/64B-swizzled B, MN-major B)
checked on one CTA against torch matmuls."""

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


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    out = tmp_path_factory.mktemp("umma") / "libumma_selftest.so"
    from context_decode_attention_paged_gb300.build import ARCH, nvcc
    cmd = [nvcc(), *ARCH, "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-I", CSRC,
           "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "cuda", "umma_selftest.cu"),
           "-o", str(out)]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(str(out))
    lib.umma_probe.restype = ctypes.c_int
    lib.umma_probe.argtypes = [ctypes.c_void_p] * 6
    return lib


def test_umma_operand_forms(probe):
    g = torch.Generator(device="cuda").manual_seed(7)
    A = torch.randn((128, 288), generator=g, device="cuda").to(torch.bfloat16)
    B = torch.randn((64, 576), generator=g, device="cuda").to(torch.bfloat16)
    P = torch.rand((128, 64), generator=g, device="cuda").to(torch.bfloat16)
    D1 = torch.full((128, 64), float("nan"), device="cuda")
    D2 = torch.full((128, 256), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.umma_probe(A.data_ptr(), B.data_ptr(), P.data_ptr(), D1.data_ptr(), D2.data_ptr(),
                          status.data_ptr())
    assert rc == 0, rc
    assert int(status.item()) == 0
    dims = list(range(256)) + list(range(512, 544))
    ref1 = A.double() @ B[:, dims].double().T
    ref2 = P.double() @ B[:, :256].double()
    assert torch.isfinite(D1).all() and torch.isfinite(D2).all()
    assert (D1.double() - ref1).abs().max().item() < 1e-3 * ref1.abs().max().item()
    assert (D2.double() - ref2).abs().max().item() < 1e-3 * ref2.abs().max().item()
