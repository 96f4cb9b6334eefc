"""Failure detection without a GPU fault.

Every wait inside the kernels is bounded.  A test-only flag makes the first CTA's TMA
producer (bit 0), or on the CTA-pair kernel the first pair's second CTA (bit 4), skip its
first shared-memory fill, so the MMA issuer waits for data that never comes.  With a short limit the wait runs out, the kernel records a code in the
stream's error word, drains what it started, frees its tensor memory and exits; the host
reads GSR_ERR_DEVICE_TIMEOUT from gsr_device_status.  Nothing traps, and a normal call
right after must still be correct (same context, small-M tickets reset).
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_core_gemm_multistage_gb300 as gsr
from tensor_core_gemm_multistage_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    gsr.build()
    oracle.build()
    yield
    gsr.set_test_flags(0)
    gsr.set_wait_timeout_ns(1_000_000_000)
    gsr.set_path_override(gsr.PATH_AUTO)


# The skipped fill turns into a timeout once the producer has to wait for the stage it never
# filled, so each CTA's work must run past its ring of stages (on CTA pairs K = 4096: 32 stages
# per tile against a ring of 3 or 4).
@pytest.mark.parametrize("M,N,K,path,kernel,flags", [(512, 1024, 1024, gsr.PATH_TILED, 0x100, 1),
                                                     (1024, 2048, 4096, gsr.PATH_PAIR, 0x100, 1),
                                                     (1024, 2048, 4096, gsr.PATH_PAIR_128, 0x100, 1),
                                                     # the first pair's second CTA skips its fill
                                                     (1024, 2048, 4096, gsr.PATH_PAIR, 0x100, 16),
                                                     (1024, 2048, 4096, gsr.PATH_PAIR_128, 0x100, 16),
                                                     (2000, 3000, 1000, gsr.PATH_PAIR, 0x100, 16),
                                                     (300, 512, 1024, gsr.PATH_TILED_64, 0x100, 1),
                                                     (16, 4096, 8192, gsr.PATH_SKINNY, 0x200, 1),
                                                     (200, 4096, 8192, gsr.PATH_SKINNY, 0x200, 1)])
def test_timeout_is_reported_and_the_gpu_stays_usable(M, N, K, path, kernel, flags):
    dev = torch.device("cuda", 0)
    A, B = make_inputs(M, N, K, seed=21)
    dA, dB = A.to(dev), B.to(dev)
    dC = torch.zeros(M, N, dtype=torch.float16, device=dev)
    gsr.set_path_override(path)
    gsr.set_wait_timeout_ns(50_000_000)        # 50 ms
    gsr.set_test_flags(flags)
    try:
        gsr.gemm_scale_relu(dA, dB, dC, 0.5)
        status, code = gsr.device_status()
    finally:
        gsr.set_test_flags(0)
        gsr.set_wait_timeout_ns(1_000_000_000)
    assert status == gsr.Status.ERR_DEVICE_TIMEOUT
    assert code & 0xF00 == kernel and (code & 0xFF) in (1, 2, 3, 4, 5)
    # the error word was cleared by the read
    assert gsr.device_status() == (gsr.Status.OK, 0)

    # same process, same context: a normal call is correct again
    dC.fill_(float("nan"))
    try:
        gsr.gemm_scale_relu(dA, dB, dC, 0.5)
        status, code = gsr.device_status()
    finally:
        gsr.set_path_override(gsr.PATH_AUTO)
    assert status == gsr.Status.OK, hex(code)
    ref = oracle.gemm_scale_relu(A, B, 0.5).astype(np.float64)
    got = dC.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))


def test_small_m_timeout_needs_no_status_call_to_recover():
    # A small-M launch that gives up leaves its tile tickets at zero by itself: a caller that
    # never reads gsr_device_status still gets correct results from the next call.
    dev = torch.device("cuda", 0)
    M, N, K = 16, 4096, 8192            # 32 tiles x 4 K slabs: every tile takes 4 tickets
    A, B = make_inputs(M, N, K, seed=23, b_std_inv_sqrt_k=True)
    dA, dB = A.to(dev), B.to(dev)
    dC = torch.zeros(M, N, dtype=torch.float16, device=dev)
    gsr.set_wait_timeout_ns(50_000_000)
    gsr.set_test_flags(1)
    try:
        gsr.gemm_scale_relu(dA, dB, dC, 0.5)
        torch.cuda.synchronize()
    finally:
        gsr.set_test_flags(0)
        gsr.set_wait_timeout_ns(1_000_000_000)
    ref, z = oracle.gemm_scale_relu(A, B, 0.5, return_pre=True)
    ref = ref.astype(np.float64)
    for _ in range(2):
        dC.fill_(float("nan"))
        gsr.gemm_scale_relu(dA, dB, dC, 0.5)
        torch.cuda.synchronize()
        got = dC.cpu().numpy().astype(np.float64)
        assert not np.isnan(got).any()
        assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))
        assert np.all(got[z < -1e-2] == 0)
    # the timeout is still on record for whoever asks
    status, code = gsr.device_status()
    assert status == gsr.Status.ERR_DEVICE_TIMEOUT and code & 0xF00 == 0x200
    assert gsr.device_status() == (gsr.Status.OK, 0)


def test_host_entry_point_blocks_time_out_and_recover():
    # The pipelined host path with B and C in column blocks (3 blocks x 8 row chunks, 24 pair
    # launches): every launch loses its first copy and gives up.  The call still completes (the
    # copy streams are joined back to the caller's stream), the timeout is reported on that
    # stream, and the next call on the same buffers is correct everywhere.
    M, N, K = 8192, 16384, 512
    A, B = make_inputs(M, N, K, seed=25)
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = torch.full((M, N), float("nan"), dtype=torch.float16).pin_memory()
    dev = torch.device("cuda", 0)
    dA = torch.empty(M, K, dtype=torch.float16, device=dev)
    dB = torch.empty(K, N, dtype=torch.float16, device=dev)
    dC = torch.empty(M, N, dtype=torch.float16, device=dev)
    stream = torch.cuda.Stream()
    gsr.set_wait_timeout_ns(20_000_000)        # 20 ms
    gsr.set_test_flags(1)
    try:
        gsr.gemm_scale_relu_host(hA, hB, hC, dA, dB, dC, 0.5, stream=stream)
        stream.synchronize()
        status, code = gsr.device_status(stream)
    finally:
        gsr.set_test_flags(0)
        gsr.set_wait_timeout_ns(1_000_000_000)
    assert status == gsr.Status.ERR_DEVICE_TIMEOUT and code & 0xF00 == 0x100, hex(code)
    hC.fill_(float("nan"))
    gsr.gemm_scale_relu_host(hA, hB, hC, dA, dB, dC, 0.5, stream=stream)
    stream.synchronize()
    assert gsr.device_status(stream) == (gsr.Status.OK, 0)
    C = hC.clone()
    assert not torch.isnan(C).any()
    rows = np.unique(np.concatenate([np.arange(0, M, 1024), np.arange(1023, M, 1024),
                                     np.random.default_rng(5).integers(0, M, 64)]))
    ref = oracle.gemm_scale_relu(A, B, 0.5, rows=rows).astype(np.float64)
    got = C[rows].numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))


def test_release_stream_frees_and_the_stream_stays_usable():
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream(dev)
    M, N, K = 16, 2048, 4096
    A, B = make_inputs(M, N, K, seed=29)
    dA, dB = A.to(dev), B.to(dev)
    ref, z = oracle.gemm_scale_relu(A, B, 0.5, return_pre=True)
    for _ in range(2):                  # state allocated, released, allocated again
        dC = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        with torch.cuda.stream(s):
            gsr.gemm_scale_relu(dA, dB, dC, 0.5, stream=s)
        assert gsr.device_status(s) == (gsr.Status.OK, 0)
        got = dC.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref.astype(np.float64)))
        gsr.release_stream(s)
        gsr.release_stream(s)           # nothing left: a no-op
    assert gsr.device_status(s) == (gsr.Status.OK, 0)
