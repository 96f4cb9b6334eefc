"""gemm_scale_relu_noalloc: the entry point for callers that cannot let the library
allocate device memory (a runtime with a fixed memory plan, or a latency-critical loop
that cannot take a first-time cudaMalloc's synchronisation).  It runs the small-M kernel
with its scratch in a fixed array inside the library; its results must match the
ordinary entry point's, call after call, although every call reuses the same array.

This file is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

import tensor_core_gemm_multistage_gb300 as gsr
from tensor_core_gemm_multistage_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

ATOL = 1e-2   # the tolerance of the parity tests (the tutorial's assert_close)
RTOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    gsr.build()
    yield


def _noalloc(dA, dB, dC, alpha, stream):
    M, K = dA.shape
    N = dB.shape[1]
    return gsr.lib().gemm_scale_relu_noalloc(
        ctypes.c_void_p(dA.data_ptr()), ctypes.c_void_p(dB.data_ptr()),
        ctypes.c_void_p(dC.data_ptr()), M, N, K, ctypes.c_float(alpha),
        ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("M,N,K,alpha", [(16, 4096, 8192, 0.5), (48, 1000, 2048, 1.0),
                                         (1, 8, 100000 - 100000 % 8, 0.75)])
def test_noalloc_matches_the_allocating_entry_point(M, N, K, alpha):
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    A, B = make_inputs(M, N, K, seed=M + N, b_std_inv_sqrt_k=True)
    dA, dB = A.to(dev), B.to(dev)
    ref = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    gsr.gemm_scale_relu(dA, dB, ref, alpha, stream=stream)
    torch.cuda.synchronize()
    want = ref.float().cpu().numpy()
    assert not np.isnan(want).any()
    for call in range(2):          # two calls in a row share the same scratch array
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        assert _noalloc(dA, dB, out, alpha, stream) == gsr.Status.OK
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert not np.isnan(got).any(), "call %d left outputs unwritten" % call
        assert np.all(np.abs(got - want) <= ATOL + RTOL * np.abs(want)), "call %d" % call


def test_noalloc_rejects_what_it_cannot_hold():
    stream = torch.cuda.current_stream(torch.device("cuda", 0))
    L = gsr.lib()
    vp = ctypes.c_void_p
    A, B, C = vp(0x10000), vp(1 << 36), vp(1 << 40)   # never touched: rejected first
    s = L.gemm_scale_relu_noalloc(A, B, C, 64, 1 << 29, 8, ctypes.c_float(1.0),
                                  vp(stream.cuda_stream))
    assert s == gsr.Status.ERR_SCRATCH_LIMIT
    s = L.gemm_scale_relu_noalloc(A, B, C, 65, 64, 8, ctypes.c_float(1.0), vp(stream.cuda_stream))
    assert s == gsr.Status.ERR_INVALID_ARG
