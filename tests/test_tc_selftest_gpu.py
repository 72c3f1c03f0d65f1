"""tcgen05 building blocks on the device: a single-CTA GEMM through the same
descriptors, instruction descriptor, TMEM loads/stores and MMA forms the
tensor-core kernels use, compared with a host matmul."""
import ctypes

import pytest
import torch

from tests.native import build as nbuild

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    lib = ctypes.CDLL(nbuild.build())
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.kata_tc_selftest.argtypes = [P, P, P, I, I, I, P, P]
    lib.kata_tc_selftest.restype = I
    return lib


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("K", [16, 32, 64, 128])
@pytest.mark.parametrize("N", [16, 64, 80, 128])
def test_gemm_probe(lib, mode, K, N):
    g = torch.Generator().manual_seed(K * 1000 + N * 10 + mode)
    A = torch.randn(128, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = A.double() @ B.double().T
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.kata_tc_selftest(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), K, N, mode,
                              status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(status.item()) == 0
    err = (D.double().cpu() - ref).abs().max().item()
    assert err <= 1e-3 * max(1.0, ref.abs().max().item()), err


def test_bounded_wait_gives_up_and_context_stays_usable(lib):
    # an mbarrier nothing arrives on: the library's bounded wait returns after
    # its budget, the kernel reports it, and the next kernel still runs
    P = ctypes.c_void_p
    lib.kata_wait_selftest.argtypes = [P, P, ctypes.c_ulonglong, P]
    lib.kata_wait_selftest.restype = ctypes.c_int
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    budget = 5_000_000  # 5 ms
    rc = lib.kata_wait_selftest(status.data_ptr(), elapsed.data_ptr(), budget,
                                torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert int(status[0].item()) == 1, "the wait did not give up"
    assert budget <= int(elapsed.item()) < 1_000_000_000
    assert int(status[1].item()) == 42, "the context did not survive the timeout"
