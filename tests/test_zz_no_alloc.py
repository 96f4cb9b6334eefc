"""gemm_scale_relu_noalloc: the entry point for callers that cannot let the library allocate
device memory (a runtime with a fixed memory plan, or a latency-critical loop that cannot take
a first-time cudaMalloc's synchronisation).  It runs the small-M kernel with its scratch in a
fixed array inside the library, so every call reuses the same array.

Checked here, through the C ABI:
  * its output against the fp64 oracle with the parity tests' acceptance (per element
    |gpu - oracle| <= 1e-2 + 1e-2 |oracle|, relative Frobenius <= 1e-3, exact zeros where
    alpha * sum < -1e-2), on two calls in a row;
  * bit-equality with the allocating entry point: both run the same kernel with the same
    K split and sum the partial tiles in the same order, so a stale or missing partial in
    the shared array would show;
  * a call with a deep K split followed by one with a shallow split (stale partials lie in
    the array where the second call's slots are);
  * that calls after the first one change neither the device's free memory nor PyTorch's
    reserved pool;
  * that a timeout inside it is reported by gsr_device_status and the next call is correct.

This file is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import tensor_core_gemm_multistage_gb300 as gsr
from tensor_core_gemm_multistage_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

ATOL = 1e-2        # per element, as in the parity tests (the tutorial's assert_close)
RTOL = 1e-2
FROB = 1e-3        # relative Frobenius error
ZERO_BELOW = -1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    gsr.build()
    oracle.build()
    yield
    gsr.set_test_flags(0)
    gsr.set_wait_timeout_ns(1_000_000_000)


def _noalloc(dA, dB, dC, alpha, stream):
    M, K = dA.shape
    N = dB.shape[1]
    return gsr.lib().gemm_scale_relu_noalloc(
        ctypes.c_void_p(dA.data_ptr()), ctypes.c_void_p(dB.data_ptr()),
        ctypes.c_void_p(dC.data_ptr()), M, N, K, ctypes.c_float(alpha),
        ctypes.c_void_p(stream.cuda_stream))


def _check_oracle(got, A, B, alpha, label):
    ref, z = oracle.gemm_scale_relu(A, B, alpha, return_pre=True)
    x = got.astype(np.float64)
    y = ref.astype(np.float64)
    assert not np.isnan(x).any(), "%s: outputs left unwritten" % label
    assert np.all(np.abs(x - y) <= ATOL + RTOL * np.abs(y)), "%s: outside tolerance" % label
    ny = np.linalg.norm(y)
    if ny > 0:
        assert np.linalg.norm(x - y) / ny <= FROB, "%s: Frobenius" % label
    assert np.all(x[z < ZERO_BELOW] == 0), "%s: ReLU zeros" % label


def _allocating(dA, dB, alpha, stream):
    # the allocating entry point on the same kernel (small B alone would take one-CTA tiles)
    M, N = dA.shape[0], dB.shape[1]
    ref = torch.full((M, N), float("nan"), dtype=torch.float16, device=dA.device)
    gsr.set_path_override(gsr.PATH_SKINNY)
    try:
        gsr.gemm_scale_relu(dA, dB, ref, alpha, stream=stream)
    finally:
        gsr.set_path_override(gsr.PATH_AUTO)
    torch.cuda.synchronize()
    return ref


@pytest.mark.parametrize("M,N,K,alpha", [(16, 4096, 8192, 0.5),       # 32 tiles x 4 K slabs
                                         (48, 1000, 2048, 1.0),       # 8 tiles x 19 slabs, ragged N
                                         (1, 8, 100000 - 100000 % 8, 0.75)])   # 1 tile x 152 slabs
def test_noalloc_matches_the_oracle_and_the_allocating_entry_point(M, N, K, alpha):
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    A, B = make_inputs(M, N, K, seed=M + N, b_std_inv_sqrt_k=True)
    dA, dB = A.to(dev), B.to(dev)
    ref = _allocating(dA, dB, alpha, stream)
    for call in range(2):          # two calls in a row share the same scratch array
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        assert _noalloc(dA, dB, out, alpha, stream) == gsr.Status.OK
        torch.cuda.synchronize()
        _check_oracle(out.cpu().numpy(), A, B, alpha, "call %d" % call)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), "call %d" % call


def test_stale_partials_from_a_deeper_split_are_never_read():
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    # 4 tiles x 38 slabs first (partial slots 0..151 written), then 32 tiles x 4 slabs, whose
    # slots (tile * 4 + slab) all hold the first call's partials when it starts
    for M, N, K, seed in ((64, 512, 16384, 1), (64, 4096, 2048, 2), (40, 1024, 4096, 3)):
        A, B = make_inputs(M, N, K, seed=seed, b_std_inv_sqrt_k=True)
        dA, dB = A.to(dev), B.to(dev)
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        assert _noalloc(dA, dB, out, 0.5, stream) == gsr.Status.OK
        torch.cuda.synchronize()
        ref = _allocating(dA, dB, 0.5, stream)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), (M, N, K)
        _check_oracle(out.cpu().numpy(), A, B, 0.5, "%dx%dx%d" % (M, N, K))


def test_calls_after_the_first_allocate_nothing():
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    cases = [(16, 4096, 8192), (32, 2048, 4096), (64, 1024, 2048), (5, 16384, 1024), (1, 8, 64)]
    bufs = []
    for M, N, K in cases:
        A, B = make_inputs(M, N, K, seed=M * 7 + N)
        bufs.append((A.to(dev), B.to(dev),
                     torch.empty(M, N, dtype=torch.float16, device=dev)))
    # one call does the set-up on this device (it may load the library's module)
    assert _noalloc(*bufs[0], 0.5, stream) == gsr.Status.OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    reserved0 = torch.cuda.memory_reserved(dev)
    for _ in range(2):
        for b in bufs:
            assert _noalloc(*b, 0.5, stream) == gsr.Status.OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0, "device free memory moved by %d bytes" % (free0 - free1)
    assert torch.cuda.memory_reserved(dev) == reserved0


def test_a_timeout_is_reported_and_the_next_call_is_correct():
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    M, N, K = 16, 4096, 8192
    A, B = make_inputs(M, N, K, seed=31, b_std_inv_sqrt_k=True)
    dA, dB = A.to(dev), B.to(dev)
    out = torch.zeros(M, N, dtype=torch.float16, device=dev)
    assert gsr.device_status(stream) == (gsr.Status.OK, 0)
    gsr.set_wait_timeout_ns(50_000_000)       # 50 ms
    gsr.set_test_flags(1)                     # the first CTA's first fill is skipped
    try:
        assert _noalloc(dA, dB, out, 0.5, stream) == gsr.Status.OK
        status, code = gsr.device_status(stream)
    finally:
        gsr.set_test_flags(0)
        gsr.set_wait_timeout_ns(1_000_000_000)
    assert status == gsr.Status.ERR_DEVICE_TIMEOUT
    assert code & 0xF00 == 0x200 and (code & 0xFF) in (1, 2, 3, 4, 5)
    assert gsr.device_status(stream) == (gsr.Status.OK, 0)      # read once, then cleared
    out.fill_(float("nan"))
    assert _noalloc(dA, dB, out, 0.5, stream) == gsr.Status.OK
    assert gsr.device_status(stream) == (gsr.Status.OK, 0)
    _check_oracle(out.cpu().numpy(), A, B, 0.5, "after the timeout")


def test_noalloc_argument_checks():
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    # M above the small-M kernel's 64 rows: refused before any work (real buffers, so a
    # regression that let it through could only compute, never touch foreign memory)
    dA = torch.zeros(65, 64, dtype=torch.float16, device=dev)
    dB = torch.zeros(64, 64, dtype=torch.float16, device=dev)
    dC = torch.zeros(65, 64, dtype=torch.float16, device=dev)
    assert _noalloc(dA, dB, dC, 1.0, stream) == gsr.Status.ERR_INVALID_ARG
    # K == 0 clears C
    dA0 = torch.empty(8, 0, dtype=torch.float16, device=dev)
    dB0 = torch.empty(0, 64, dtype=torch.float16, device=dev)
    dC0 = torch.full((8, 64), float("nan"), dtype=torch.float16, device=dev)
    assert _noalloc(dA0, dB0, dC0, 1.0, stream) == gsr.Status.OK
    torch.cuda.synchronize()
    assert torch.all(dC0 == 0)
