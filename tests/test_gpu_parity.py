"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Acceptance, per element of C:   |gpu - oracle| <= 1e-2 + 1e-2 * |oracle|
(the tutorial's own check, torch.testing.assert_close(rtol=1e-2, atol=1e-2), in
"Tutorial14: 使用TileLang语言编写attention算子", section 2), plus
    relative Frobenius error ||gpu - oracle||_F / ||oracle||_F <= 1e-3
(the relative-Frobenius `check` the aikraft.ru TileLang tutorial survey recommends for
fp16), plus exact zeros wherever the oracle's pre-ReLU value alpha * sum is below -1e-2.
Every output buffer is pre-filled with NaN so an element the kernel never writes fails.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_core_gemm_multistage_gb300 as gsr
from tensor_core_gemm_multistage_gb300.workloads import WORKLOADS, make_inputs, sample_rows, workload_inputs

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2
FROB = 1e-3
ZERO_BELOW = -1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    gsr.build()
    oracle.build()
    yield
    gsr.set_path_override(gsr.PATH_AUTO)


def run_gpu(A, B, alpha, path=gsr.PATH_AUTO, stream=None):
    """A, B: CPU fp16 tensors. Returns C as a CPU fp16 tensor."""
    dev = torch.device("cuda", 0)
    dA = A.to(dev)
    dB = B.to(dev)
    dC = torch.full((A.shape[0], B.shape[1]), float("nan"), dtype=torch.float16, device=dev)
    gsr.set_path_override(path)
    try:
        gsr.gemm_scale_relu(dA, dB, dC, alpha, stream=stream)
        status, code = gsr.device_status(stream)
    finally:
        gsr.set_path_override(gsr.PATH_AUTO)
    assert status == gsr.Status.OK, (status, hex(code))
    return dC.cpu()


def check(C_gpu, C_ref, Z_ref, label=""):
    x = C_gpu.numpy().astype(np.float64) if hasattr(C_gpu, "numpy") else C_gpu.astype(np.float64)
    y = C_ref.astype(np.float64)
    assert x.shape == y.shape
    assert not np.isnan(x).any(), "%s: %d elements never written" % (label, int(np.isnan(x).sum()))
    err = np.abs(x - y)
    bound = ATOL + RTOL * np.abs(y)
    bad = err > bound
    assert not bad.any(), "%s: %d elements out of tolerance, worst %g at %s" % (
        label, int(bad.sum()), float(err.max()), np.unravel_index(np.argmax(err - bound), err.shape))
    ny = np.linalg.norm(y)
    if ny > 0:
        rel = np.linalg.norm(x - y) / ny
        assert rel <= FROB, "%s: relative Frobenius error %g" % (label, rel)
    neg = Z_ref < ZERO_BELOW
    assert np.all(x[neg] == 0), "%s: non-zero output where alpha*sum < -1e-2" % label


def parity(M, N, K, alpha, path=gsr.PATH_AUTO, seed=0, b_scaled=False, rows=None):
    A, B = make_inputs(M, N, K, seed=seed, b_std_inv_sqrt_k=b_scaled)
    C = run_gpu(A, B, alpha, path)
    if rows is None:
        ref, z = oracle.gemm_scale_relu(A, B, alpha, return_pre=True)
        check(C, ref, z, "%dx%dx%d" % (M, N, K))
    else:
        ref, z = oracle.gemm_scale_relu(A, B, alpha, rows=rows, return_pre=True)
        check(C[rows], ref, z, "%dx%dx%d rows" % (M, N, K))


# ---------------------------------------------------------------------------- the five workloads

@pytest.mark.parametrize("name", ["square1024", "ragged2000x3000x1000", "skinny_decode"])
def test_workload_full(name):
    w = WORKLOADS[name]
    parity(w.M, w.N, w.K, w.alpha, b_scaled=w.b_std_inv_sqrt_k)


@pytest.mark.parametrize("name", ["square8192", "llm_mlp_up"])
def test_workload_sampled_rows(name):
    # Too big for the oracle in full: a seeded sample of 128 whole rows plus the tile edges.
    w = WORKLOADS[name]
    parity(w.M, w.N, w.K, w.alpha, b_scaled=w.b_std_inv_sqrt_k, rows=sample_rows(w.M))


def test_page_instance_against_torch_reference():
    # The tutorial's own check: seed 0, 1024^3, scale 0.5, against relu((a @ b) * scale)
    # with rtol = atol = 1e-2.  A test-only cross-check; the oracle is the authority.
    A, B = make_inputs(1024, 1024, 1024, seed=0)
    C = run_gpu(A, B, 0.5)
    ref = torch.relu((A.cuda() @ B.cuda()) * 0.5).cpu()
    torch.testing.assert_close(C, ref, rtol=1e-2, atol=1e-2)


# ---------------------------------------------------------------------------- tile edges

EDGE_SHAPES = [
    (1, 8, 8), (1, 64, 64), (7, 136, 72), (16, 128, 64), (17, 264, 1000), (33, 8, 16),
    (64, 512, 56), (65, 256, 64), (127, 128, 64), (128, 256, 64), (129, 264, 72),
    (255, 120, 200), (256, 256, 128), (257, 392, 136), (300, 8, 8), (1000, 1000, 8),
    (130, 6144, 64), (384, 512, 1024),
]


@pytest.mark.parametrize("M,N,K", EDGE_SHAPES)
def test_edges_auto(M, N, K):
    parity(M, N, K, 0.5, seed=M + N + K)


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (129, 264, 72), (255, 120, 200), (257, 392, 136),
                                   (16, 16384, 1024), (640, 768, 4096)])
@pytest.mark.parametrize("path", [gsr.PATH_TILED_256, gsr.PATH_TILED_128, gsr.PATH_TILED_64, gsr.PATH_PAIR,
                                  gsr.PATH_PAIR_128])
def test_edges_every_tiled_kernel(M, N, K, path):
    parity(M, N, K, 1.0, path=path, seed=7 * M + N + K)


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (5, 40, 8), (16, 128, 64), (16, 136, 72),
                                   (17, 1000, 1000), (32, 4096, 4096), (33, 264, 1024),
                                   (48, 2048, 8192), (64, 640, 64), (64, 16384, 2048),
                                   (3, 8, 100000 - 100000 % 8)])
def test_small_m_path(M, N, K):
    # forced (the automatic choice takes the small-M kernel only from 16 MiB of B on)
    parity(M, N, K, 0.75, path=gsr.PATH_SKINNY, seed=M * N + K, b_scaled=True)


@pytest.mark.parametrize("M,N,K,slabs", [(16, 1024, 2048, 1),     # no split: one item per tile
                                          (16, 1024, 2048, 3),     # 32 k-blocks in slabs of 10/11/11
                                          (40, 1000, 1000, 16),    # 16 k-blocks, one per slab
                                          (40, 1000, 1000, 99),    # asked for more: clamped to 16
                                          (64, 4096, 8192, 64)])   # more slabs than the default 4
def test_small_m_split_override(M, N, K, slabs):
    # gsr_set_split_k: any slab count sums every k-block once (slab order is fixed, so a second
    # call gives the same bytes); the per-stream workspace grows for more slabs than the default
    A, B = make_inputs(M, N, K, seed=M + slabs, b_std_inv_sqrt_k=True)
    gsr.set_split_k(slabs)
    try:
        C = run_gpu(A, B, 0.5, gsr.PATH_SKINNY)
        C2 = run_gpu(A, B, 0.5, gsr.PATH_SKINNY)
    finally:
        gsr.set_split_k(0)
    ref, z = oracle.gemm_scale_relu(A, B, 0.5, return_pre=True)
    check(C, ref, z, "split %d" % slabs)
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))


@pytest.mark.parametrize("M,N,K,rows", [(65, 264, 136, None), (100, 1000, 1000, None), (128, 520, 2048, None),
                                         (129, 8, 8, None), (200, 4096, 512, None), (256, 640, 64, None),
                                         (192, 16384, 1024, [0, 1, 63, 64, 127, 128, 190, 191]),
                                         (256, 16384, 2048, [0, 1, 127, 128, 129, 200, 254, 255])])
def test_small_m_path_forced_up_to_256_rows(M, N, K, rows):
    # 65 to 256 rows on the small-M kernel (forced): an MMA N of 128 or 256 and the epilogue
    # walking the accumulator in 32-column chunks, with K split into slabs (every shape but the
    # two with N = 16384, whose 128 tiles fill the SMs alone); the split runs twice, for the
    # same bytes (the slab order is fixed)
    A, B = make_inputs(M, N, K, seed=M * 7 + N + K, b_std_inv_sqrt_k=True)
    gsr.set_path_override(gsr.PATH_SKINNY)
    try:
        assert gsr.select_path(M, N, K) == gsr.KERNEL_SKINNY
    finally:
        gsr.set_path_override(gsr.PATH_AUTO)
    C = run_gpu(A, B, 0.75, gsr.PATH_SKINNY)
    if rows is None:
        ref, z = oracle.gemm_scale_relu(A, B, 0.75, return_pre=True)
        check(C, ref, z, "%dx%dx%d forced small-M" % (M, N, K))
        C2 = run_gpu(A, B, 0.75, gsr.PATH_SKINNY)
        assert torch.equal(C.view(torch.int16), C2.view(torch.int16))
    else:
        ref, z = oracle.gemm_scale_relu(A, B, 0.75, rows=rows, return_pre=True)
        check(C[rows], ref, z, "%dx%dx%d forced small-M rows" % (M, N, K))


@pytest.mark.parametrize("M,N,K", [(100, 4096, 14336), (128, 4096, 16384), (65, 3072, 20480)])
def test_small_m_chosen_for_up_to_128_rows(M, N, K):
    # the automatic choice of the small-M kernel for 65-128 rows (B streamed from HBM, few
    # one-CTA tiles)
    assert gsr.select_path(M, N, K) == gsr.KERNEL_SKINNY
    parity(M, N, K, 0.5, seed=M + N + K, b_scaled=True, rows=[0, 1, 31, 32, 63, 64, M - 2, M - 1])


@pytest.mark.parametrize("name", ["square1024", "ragged2000x3000x1000"])
@pytest.mark.parametrize("path", [gsr.PATH_TILED_128, gsr.PATH_TILED_64, gsr.PATH_PAIR, gsr.PATH_PAIR_128])
def test_small_workloads_on_each_tiled_kernel(name, path):
    w = WORKLOADS[name]
    parity(w.M, w.N, w.K, w.alpha, path=path)


@pytest.mark.parametrize("path", [gsr.PATH_PAIR, gsr.PATH_PAIR_128])
@pytest.mark.parametrize("M,N,K", [(512, 1024, 1024), (300, 768, 200), (520, 192, 136)])
def test_pair_kernel_with_and_without_3d_b_copies(M, N, K, path):
    # N % 64 == 0: B normally arrives as one 3-D copy per stage; test flag bit 1 forces the
    # two-box 2-D copies.  Both must match the oracle.
    A, B = make_inputs(M, N, K, seed=M + N + K)
    ref, z = oracle.gemm_scale_relu(A, B, 0.5, return_pre=True)
    for flags in (0, 2):
        gsr.set_test_flags(flags)
        try:
            C = run_gpu(A, B, 0.5, path)
        finally:
            gsr.set_test_flags(0)
        check(C, ref, z, "pair path=%d flags=%d" % (path, flags))


def test_big_workloads_use_the_pair_kernel():
    for name in ("square8192", "llm_mlp_up"):
        w = WORKLOADS[name]
        assert gsr.select_path(w.M, w.N, w.K) == gsr.KERNEL_PAIR
    w = WORKLOADS["ragged2000x3000x1000"]
    assert gsr.select_path(w.M, w.N, w.K) == gsr.KERNEL_PAIR


@pytest.mark.parametrize("M,N,K", [(7600, 576, 264),     # 90 tiles: 76 whole, 14 split; second halves past N
                                   (4096, 4096, 1024),   # 256 tiles: 228 whole, 28 split
                                   (512, 1024, 1024)])   # 8 tiles, all split into 16 halves
@pytest.mark.parametrize("flags", [0, 2])               # 3-D boxes of one chunk / 2-D boxes for B
def test_pair_kernel_half_width_tail(M, N, K, flags):
    # The 256 x 256 pair kernel runs a last wave that would keep at most half the pairs busy
    # as 256 x 128 half units; a half unit past N writes nothing.
    A, B = make_inputs(M, N, K, seed=M + 3 * N + K)
    rows = None if M * N * K <= 2 ** 31 else sample_rows(M)
    ref, z = oracle.gemm_scale_relu(A, B, 0.5, rows=rows, return_pre=True)
    gsr.set_test_flags(flags)
    try:
        C = run_gpu(A, B, 0.5, gsr.PATH_PAIR)
    finally:
        gsr.set_test_flags(0)
    check(C if rows is None else C[rows], ref, z, "half tail %dx%dx%d flags=%d" % (M, N, K, flags))


_RASTER_REF = {}


def _raster_reference(M, N, K):
    if (M, N, K) not in _RASTER_REF:
        A, B = make_inputs(M, N, K, seed=M + N + K + 1)
        rows = None if M * N * K <= 2 ** 33 else sample_rows(M)
        _RASTER_REF[(M, N, K)] = (A, B, rows) + oracle.gemm_scale_relu(A, B, 0.5, rows=rows,
                                                                       return_pre=True)
    return _RASTER_REF[(M, N, K)]


@pytest.mark.parametrize("M,N,K", [(2000, 3000, 1000),   # pair: 96 tiles, the last 20 split; partial groups
                                   (7600, 576, 264)])    # 30 row blocks of 256, 60 of 128: ragged groups
@pytest.mark.parametrize("path", [gsr.PATH_TILED_256, gsr.PATH_TILED_128, gsr.PATH_PAIR, gsr.PATH_PAIR_128])
@pytest.mark.parametrize("group", [1, 3, 4, 16, 64])
def test_raster_groups(M, N, K, path, group):
    # gsr_set_raster_group changes which CTA computes which tile (the "L2 swizzle" knob); every
    # grouping, including ones that leave the last group partial, must give the same result.
    A, B, rows, ref, z = _raster_reference(M, N, K)
    gsr.set_raster_group(group)
    try:
        C = run_gpu(A, B, 0.5, path)
    finally:
        gsr.set_raster_group(0)
    check(C if rows is None else C[rows], ref, z, "raster %d path %d %dx%dx%d" % (group, path, M, N, K))


def test_skinny_workload_through_tiled_path():
    w = WORKLOADS["skinny_decode"]
    parity(w.M, w.N, w.K, w.alpha, path=gsr.PATH_TILED, b_scaled=True)


# ---------------------------------------------------------------------------- structure

@pytest.mark.parametrize("M,K,path", [(64, 64, gsr.PATH_AUTO), (130, 72, gsr.PATH_AUTO),
                                      (300, 256, gsr.PATH_TILED_128), (40, 136, gsr.PATH_SKINNY),
                                      (200, 200, gsr.PATH_TILED_64),
                                      (520, 264, gsr.PATH_PAIR)])
def test_identity_b_is_exact(M, K, path):
    # the sum has one non-zero term, so fp32 accumulation is exact and C must equal the
    # oracle bit for bit
    A, _ = make_inputs(M, 8, K, seed=3)
    B = torch.eye(K, dtype=torch.float16)
    C = run_gpu(A, B, 0.5, path)
    ref = oracle.gemm_scale_relu(A, B, 0.5)
    assert np.array_equal(C.numpy().view(np.uint16), ref.view(np.uint16))


@pytest.mark.parametrize("M,N,K,alpha,path", [(200, 264, 1000, 0.5, gsr.PATH_AUTO),
                                              (8, 64, 3000, 1.0, gsr.PATH_SKINNY),
                                              (130, 128, 2048, 1.0, gsr.PATH_TILED_256),
                                              (260, 200, 4096, 0.5, gsr.PATH_TILED_64),
                                              (300, 520, 1000, 0.5, gsr.PATH_PAIR)])
def test_all_ones_is_exact(M, N, K, alpha, path):
    A = torch.ones(M, K, dtype=torch.float16)
    B = torch.ones(K, N, dtype=torch.float16)
    C = run_gpu(A, B, alpha, path)
    assert torch.all(C == float(np.float16(alpha * K)))


@pytest.mark.parametrize("path", [gsr.PATH_TILED, gsr.PATH_SKINNY, gsr.PATH_PAIR, gsr.PATH_PAIR_128])
def test_one_hot_rows(path):
    M, N, K = 48, 392, 320
    rng = np.random.default_rng(4)
    ks = rng.integers(0, K, M)
    A = torch.zeros(M, K, dtype=torch.float16)
    A[torch.arange(M), torch.from_numpy(ks)] = 1
    _, B = make_inputs(8, N, K, seed=5)
    C = run_gpu(A, B, 1.0, path)
    ref = oracle.gemm_scale_relu(A, B, 1.0)
    assert np.array_equal(C.numpy().view(np.uint16), ref.view(np.uint16))


@pytest.mark.parametrize("M", [16, 300])
def test_negative_alpha_nonnegative_inputs(M):
    A, B = make_inputs(M, 520, 264, seed=6)
    C = run_gpu(A.abs(), B.abs(), -0.5)
    assert torch.all(C == 0)


def test_k_zero_writes_zeros():
    dC = torch.full((33, 64), float("nan"), dtype=torch.float16, device="cuda")
    dA = torch.empty(33, 0, dtype=torch.float16, device="cuda")
    dB = torch.empty(0, 64, dtype=torch.float16, device="cuda")
    gsr.gemm_scale_relu(dA, dB, dC, 0.5)
    torch.cuda.synchronize()
    assert torch.all(dC == 0)


def test_empty_output_leaves_buffers_alone():
    dA = torch.ones(0, 64, dtype=torch.float16, device="cuda")
    dB = torch.ones(64, 8, dtype=torch.float16, device="cuda")
    dC = torch.empty(0, 8, dtype=torch.float16, device="cuda")
    gsr.gemm_scale_relu(dA, dB, dC, 0.5)
    torch.cuda.synchronize()


def test_repeated_calls_are_deterministic():
    for M in (16, 512):
        A, B = make_inputs(M, 2048, 4096, seed=9)
        c1 = run_gpu(A, B, 0.5)
        c2 = run_gpu(A, B, 0.5)
        assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


def test_streams_do_not_share_workspace():
    # two small-M launches in flight on two streams at once; each must be correct
    dev = torch.device("cuda", 0)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    A1, B1 = make_inputs(16, 4096, 8192, seed=11)
    A2, B2 = make_inputs(24, 4096, 8192, seed=12)
    d = [(A1.to(dev), B1.to(dev)), (A2.to(dev), B2.to(dev))]
    outs = [torch.full((16, 4096), float("nan"), dtype=torch.float16, device=dev),
            torch.full((24, 4096), float("nan"), dtype=torch.float16, device=dev)]
    torch.cuda.synchronize()
    for _ in range(3):
        for (a, b), c, s in zip(d, outs, (s1, s2)):
            with torch.cuda.stream(s):
                gsr.gemm_scale_relu(a, b, c, 0.5, stream=s)
    for s in (s1, s2):
        assert gsr.device_status(s)[0] == gsr.Status.OK
    for (A, B), c in zip(((A1, B1), (A2, B2)), outs):
        ref, z = oracle.gemm_scale_relu(A, B, 0.5, return_pre=True)
        check(c.cpu(), ref, z, "stream")


def test_every_gemm_kernel_on_two_streams_at_once():
    # CTA-pair, one-CTA and small-M launches queued alternately on two streams, three rounds:
    # whatever overlaps on the GPU, each result must match the oracle
    dev = torch.device("cuda", 0)
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    shapes = [(2048, 4096, 512), (1000, 1024, 512), (16, 4096, 2048), (2304, 2560, 520)]
    cases = []
    for i, (M, N, K) in enumerate(shapes):
        A, B = make_inputs(M, N, K, seed=40 + i)
        cases.append((A, B, A.to(dev), B.to(dev),
                      torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)))
    assert [gsr.select_path(M, N, K) for M, N, K in shapes] == [gsr.KERNEL_PAIR, gsr.KERNEL_TILED,
                                                               gsr.KERNEL_SKINNY, gsr.KERNEL_PAIR]
    torch.cuda.synchronize()
    for _ in range(3):
        for i, (_, _, dA, dB, dC) in enumerate(cases):
            s = streams[i % 2]
            with torch.cuda.stream(s):
                gsr.gemm_scale_relu(dA, dB, dC, 0.5, stream=s)
    for s in streams:
        assert gsr.device_status(s)[0] == gsr.Status.OK
    for A, B, _, _, dC in cases:
        rows = sample_rows(A.shape[0])
        ref, z = oracle.gemm_scale_relu(A, B, 0.5, rows=rows, return_pre=True)
        check(dC.cpu()[rows], ref, z, "two streams %dx%dx%d" % (A.shape[0], B.shape[1], A.shape[1]))


def test_host_entry_point_round_trip():
    M, N, K = 256, 384, 512
    A, B = make_inputs(M, N, K, seed=13)
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = torch.empty(M, N, dtype=torch.float16).pin_memory()
    dA = torch.empty(M, K, dtype=torch.float16, device="cuda")
    dB = torch.empty(K, N, dtype=torch.float16, device="cuda")
    dC = torch.empty(M, N, dtype=torch.float16, device="cuda")
    gsr.gemm_scale_relu_host(hA, hB, hC, dA, dB, dC, 0.5)
    torch.cuda.synchronize()
    ref, z = oracle.gemm_scale_relu(A, B, 0.5, return_pre=True)
    check(hC.clone(), ref, z, "host")


@pytest.mark.parametrize("M,N,K,chunk", [(1200, 1000, 1024, 0),         # below the threshold: one piece
                                          (2000, 3000, 1000, 1024),      # 1024 rows + 976
                                          (2500, 4096, 4096, 512),       # 4 x 512 rows + 452
                                          (4096, 4096, 4096, 512),       # 8 x 512 rows
                                          # C larger than A and B: B and C in 3 column blocks of
                                          # 5632, 5632 and 5120 columns, strided copies both ways
                                          (8192, 16384, 512, 1024),
                                          # the same with 7 x 1024 rows + 32 (joined to the 7th)
                                          # and a last block of 5112 columns (not a multiple of 64)
                                          (7200, 16376, 512, 1024)])
def test_host_entry_point_in_chunks(M, N, K, chunk):
    # Large enough for the pipelined host path: A's rows in chunks (and B and C in column
    # blocks where C is the larger transfer), each block's product and copy back overlapping
    # the copies in of later ones.  Every element must arrive.
    A, B = make_inputs(M, N, K, seed=M + K)
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = torch.full((M, N), float("nan"), dtype=torch.float16).pin_memory()
    dA = torch.empty(M, K, dtype=torch.float16, device="cuda")
    dB = torch.empty(K, N, dtype=torch.float16, device="cuda")
    dC = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    stream = torch.cuda.Stream()
    gsr.gemm_scale_relu_host(hA, hB, hC, dA, dB, dC, 0.5, stream=stream)
    stream.synchronize()
    assert gsr.device_status(stream)[0] == gsr.Status.OK
    C = hC.clone()
    assert not torch.isnan(C).any()
    if chunk == 0:
        ref, z = oracle.gemm_scale_relu(A, B, 0.5, return_pre=True)
        check(C, ref, z, "host")
    else:
        # the seeded row sample plus the first and last row of every chunk
        edges = [e for c0 in range(0, M, chunk) for e in (c0, min(c0 + chunk, M) - 1)]
        r = np.unique(np.concatenate([np.asarray(sample_rows(M)), np.asarray(edges)]))
        ref, z = oracle.gemm_scale_relu(A, B, 0.5, rows=r, return_pre=True)
        check(C[r], ref, z, "host chunks rows")
    # a second call on the same buffers (events and copy streams reused) gives the same bytes
    hC2 = torch.zeros_like(hC).pin_memory()
    gsr.gemm_scale_relu_host(hA, hB, hC2, dA, dB, dC, 0.5, stream=stream)
    stream.synchronize()
    assert torch.equal(hC2.view(torch.int16), C.view(torch.int16))


def test_gpu_validation_codes():
    dA = torch.empty(64, 64, dtype=torch.float16, device="cuda")
    dB = torch.empty(64, 64, dtype=torch.float16, device="cuda")
    assert gsr.gemm_scale_relu_ptr(dA.data_ptr(), dB.data_ptr(), dA.data_ptr(), 64, 64, 64, 1.0) \
        == gsr.Status.ERR_ALIAS
    assert gsr.gemm_scale_relu_ptr(dA.data_ptr() + 2, dB.data_ptr(), dB.data_ptr(), 8, 8, 8, 1.0) \
        == gsr.Status.ERR_ALIGNMENT


@pytest.mark.parametrize("flags", [4, 8, 32, 64, 4 | 32])
def test_pair_kernel_l2_switches(flags):
    # The pair kernel walks K backwards in every other wave of tiles by default; bit 2 walks
    # it forward everywhere, bit 3 drops the evict-first hint of the C stores, bits 5/6 change
    # the L2 hint of the B copies.  4096 x 4096 x 1024 has three and a half waves of tiles.
    A, B, rows, ref, z = _raster_reference(4096, 4096, 1024)
    gsr.set_test_flags(flags)
    try:
        C = run_gpu(A, B, 0.5, gsr.PATH_PAIR)
    finally:
        gsr.set_test_flags(0)
    check(C if rows is None else C[rows], ref, z, "pair flags %d" % flags)


# ---------------------------------------------------------------------------- partial last waves

@pytest.mark.parametrize("M,N,K,path,full", [
    (2000, 3000, 1000, gsr.PATH_AUTO, True),    # 96 tiles: 76 whole, then 20 as 40 half-width units
    (3000, 2600, 200, gsr.PATH_AUTO, True),     # 132 tiles: a last wave of 56 whole tiles, two stages each
    (2560, 2560, 64, gsr.PATH_AUTO, True),      # 100 tiles, one stage each: 24 tiles as 48 halves
    (1024, 2048, 1024, gsr.PATH_PAIR, True),    # 32 tiles, no full wave
    (4096, 4096, 1024, gsr.PATH_AUTO, False),   # 256 tiles: 3 waves, then 28 tiles as 56 halves
    (6144, 3072, 2048, gsr.PATH_AUTO, False)])  # 288 tiles: 3 waves, then 60 whole tiles
def test_pair_partial_last_wave(M, N, K, path, full):
    # Pair launches whose last wave is partial, with 1 to 16 stages per tile; a second call on
    # the same inputs gives the same bytes (every output element is summed in one fixed order).
    A, B = make_inputs(M, N, K, seed=M + N + K, b_std_inv_sqrt_k=True)
    rows = None if full else sample_rows(M)
    ref, z = oracle.gemm_scale_relu(A, B, 0.5, rows=rows, return_pre=True)
    C = run_gpu(A, B, 0.5, path)
    check(C if full else C[rows], ref, z, "last wave %dx%dx%d" % (M, N, K))
    C2 = run_gpu(A, B, 0.5, path)
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))


# ---------------------------------------------------------------------------- random shapes

def _random_shapes(n, seed):
    # seeded shapes for the automatic path: every kernel and tile width the host can choose,
    # ragged in M, N and K (N, K multiples of 8 as the boundary requires)
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M = int(rng.choice([rng.integers(1, 65), rng.integers(65, 1600)]))
        N = int(rng.integers(1, 190)) * 8
        K = int(rng.integers(1, 129)) * 8
        out.append((M, N, K, float(rng.choice([0.5, 1.0, -0.75, 1.25]))))
    return out


@pytest.mark.parametrize("M,N,K,alpha", _random_shapes(24, 2026))
def test_random_shapes_auto(M, N, K, alpha):
    parity(M, N, K, alpha, seed=M + 3 * N + 7 * K, b_scaled=True)


def _random_large_shapes(n, seed):
    # at least a wave of 256 x 256 pair tiles: the CTA-pair kernels (whole tiles, half-width
    # last waves, 256- or 128-wide tiles), checked on sampled rows
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(2300, 6001)), int(rng.integers(16, 751)) * 8, int(rng.integers(8, 129)) * 8,
             float(rng.choice([0.5, 1.0, -0.75]))) for _ in range(n)]


@pytest.mark.parametrize("M,N,K,alpha", _random_large_shapes(8, 2027))
def test_random_large_shapes_auto(M, N, K, alpha):
    parity(M, N, K, alpha, seed=M + N + K, b_scaled=True, rows=sample_rows(M))


# ---------------------------------------------------------------------------- large sizes

def test_a_million_rows():
    # M = 10^6 (not a multiple of 256): 3907 pair tiles over 76 pairs, tile and raster
    # arithmetic far from the small cases; checked on a row sample that includes the last rows
    M, N, K = 1_000_000, 136, 72
    A, B = make_inputs(M, N, K, seed=77)
    rows = sorted(set(sample_rows(M)) | {M - 2, M - 129, M - 256, 999_935})
    C = run_gpu(A, B, 0.5)
    ref, z = oracle.gemm_scale_relu(A, B, 0.5, rows=rows, return_pre=True)
    check(C[rows], ref, z, "M=10^6")


@pytest.mark.parametrize("path", [gsr.PATH_AUTO, gsr.PATH_PAIR, gsr.PATH_TILED_128])
def test_a_long_k(path):
    # K = 2^17 - 8: 2048 k-blocks, so every ring slot's phase bit wraps hundreds of times within
    # one tile, and the last k-block is ragged
    M, N, K = 200, 256, (1 << 17) - 8
    A, B = make_inputs(M, N, K, seed=78, b_std_inv_sqrt_k=True)
    C = run_gpu(A, B, 1.0, path)
    ref, z = oracle.gemm_scale_relu(A, B, 1.0, return_pre=True)
    check(C, ref, z, "K=2^17-8 path %d" % path)


@pytest.mark.parametrize("K", [6136, 6144])
def test_pairs_below_a_wave_from_a_long_k(K):
    # 256 x 16384: 64 pair tiles, fewer than the 76 pairs of a wave.  Up to K = 6143 the library
    # takes 128 x 256 one-CTA tiles, from 6144 on CTA pairs (their faster K loop repays their
    # cost per launch); both sides of that boundary, checked on rows of both 128-row halves of
    # the pair tile and the last row
    M, N = 256, 16384
    assert gsr.select_path(M, N, K) == (gsr.KERNEL_TILED if K < 6144 else gsr.KERNEL_PAIR)
    parity(M, N, K, 1.0, seed=K, b_scaled=True, rows=[0, 1, 63, 127, 128, 129, 200, 255])
