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


@pytest.fixture(scope="module")
def probe_t(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    out = tmp_path_factory.mktemp("umma_t") / "libumma_selftest_t.so"
    from context_decode_attention_paged_gb300.build import ARCH, nvcc
    cmd = [nvcc(), *ARCH, "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-I", CSRC,
           "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "cuda", "umma_selftest_t.cu"),
           "-o", str(out), "-lcuda"]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(str(out))
    lib.umma_probe_t.restype = ctypes.c_int
    lib.umma_probe_t.argtypes = [ctypes.c_int] + [ctypes.c_void_p] * 10
    return lib


@pytest.mark.parametrize("ncol", [16, 32, 64])
def test_umma_transposed_forms(probe_t, ncol):
    """Keys-as-M forms: S^T = K Q^T (A = K tile, B = Q rows under the 128-byte
    swizzle) and O^T = V^T P^T (A = V tile read MN-major, B = P rows under the
    ncol-wide swizzle, stored by threads and, separately, by TMA); and S^T again
    with descriptors built once and advanced per K-step by adding the offset to
    the start-address field (as a 64-bit add and on the low word only)."""
    g = torch.Generator(device="cuda").manual_seed(11 + ncol)
    K = torch.randn((128, 128), generator=g, device="cuda").to(torch.bfloat16)
    V = torch.randn((128, 128), generator=g, device="cuda").to(torch.bfloat16)
    Q = torch.randn((ncol, 128), generator=g, device="cuda").to(torch.bfloat16)
    P = torch.rand((128, ncol), generator=g, device="cuda").to(torch.bfloat16)
    D = [torch.full((128, ncol), float("nan"), device="cuda") for _ in range(5)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe_t.umma_probe_t(ncol, K.data_ptr(), V.data_ptr(), Q.data_ptr(), P.data_ptr(),
                              D[0].data_ptr(), D[1].data_ptr(), D[2].data_ptr(), D[3].data_ptr(),
                              D[4].data_ptr(), status.data_ptr())
    assert rc == 0, rc
    assert int(status.item()) == 0
    ref_s = K.double() @ Q.double().T
    ref_o = V.double().T @ P.double()
    for got, ref, what in ((D[0], ref_s, "S^T"), (D[1], ref_o, "O^T (P by threads)"),
                           (D[2], ref_o, "O^T (P by TMA)"), (D[3], ref_s, "S^T (64-bit descriptor advance)"),
                           (D[4], ref_s, "S^T (low-word descriptor advance)")):
        assert torch.isfinite(got).all(), what
        err = (got.double() - ref).abs().max().item()
        assert err < 1e-3 * ref.abs().max().item(), (what, err)
