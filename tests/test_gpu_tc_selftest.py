"""Tensor-core building blocks of the prefill kernels, checked against a plain fp32 matmul:
operand layouts (K-major / MN-major, 128-byte swizzle), descriptors, negate-A,
accumulation, TMEM readback and a TMA-loaded operand.  Products of bf16 values are exact
in fp32, so the only difference is the fp32 summation order.  The self-test kernel lives in
the test-only library libkda_selftest.so, built beside libkda.so."""
import ctypes
import functools

import pytest
import torch

from kda_state_chunked_gb300 import build as kda_build

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=1)
def _selftest_lib():
    kda_build.build()
    return ctypes.CDLL(kda_build.SELFTEST_SO)


def _run(K, N, a_mn, b_mn, neg, use_tma, seed=0):
    L = _selftest_lib()
    f = L.kda_internal_mma_selftest
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 6 + [ctypes.c_void_p, ctypes.c_void_p]
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = torch.randn(128, K, generator=g, device="cuda").to(torch.bfloat16)
    B = torch.randn(K, N, generator=g, device="cuda").to(torch.bfloat16)
    D = torch.full((128, N), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = f(A.data_ptr(), B.data_ptr(), D.data_ptr(), K, N, a_mn, b_mn, neg, use_tma, err.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = (A.float() @ B.float()) * (-2.0 if neg else 2.0)
    return (D - ref).abs().max().item() / ref.abs().max().item()


@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_mma_layouts(K, N, a_mn, b_mn):
    assert _run(K, N, a_mn, b_mn, 0, 0) < 1e-5


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 1)])
def test_mma_negate_a(a_mn, b_mn):
    assert _run(128, 64, a_mn, b_mn, 1, 0) < 1e-5


@pytest.mark.parametrize("K,N", [(64, 64), (128, 128)])
def test_mma_tma_loaded_operand(K, N):
    assert _run(K, N, 0, 0, 0, 1) < 1e-5


@pytest.mark.parametrize("K,N,b_mn,neg", [(64, 64, 0, 0), (128, 64, 1, 1), (128, 128, 0, 0), (64, 128, 1, 0)])
def test_mma_a_operand_from_tmem(K, N, b_mn, neg):
    """A read from tensor memory (bf16 pairs packed along K per 32-bit column)."""
    assert _run(K, N, 0, b_mn, neg, 2) < 1e-5
