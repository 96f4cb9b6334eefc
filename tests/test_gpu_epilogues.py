"""GPU parity of the further epilogues against the fp64 oracle (next rows of the build):

  gemm_scale:      C = alpha * A @ B   (alpha = 1: the plain tiled GEMM, make_matmul section
                                        of the aikraft.ru TileLang tutorial survey)
  gemm_bias_gelu:  C = GELU(A @ B + bias), tanh form (its make_matmul_bias_gelu section)

Same acceptance as the fused operator: per element |gpu - oracle| <= 1e-2 + 1e-2 |oracle| and
relative Frobenius error <= 1e-3; outputs pre-filled with NaN so unwritten elements fail.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_core_gemm_multistage_gb300 as gsr
from tensor_core_gemm_multistage_gb300.workloads import WORKLOADS, make_inputs, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    gsr.build()
    oracle.build()
    yield
    gsr.set_path_override(gsr.PATH_AUTO)


def make_bias(N, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(N, generator=g) * 2).half()


def run(kind, A, B, alpha=1.0, bias=None, path=gsr.PATH_AUTO):
    dev = torch.device("cuda", 0)
    dA, dB = A.to(dev), B.to(dev)
    dC = torch.full((A.shape[0], B.shape[1]), float("nan"), dtype=torch.float16, device=dev)
    gsr.set_path_override(path)
    try:
        if kind == oracle.EPI_SCALE:
            gsr.gemm_scale(dA, dB, dC, alpha)
        else:
            gsr.gemm_bias_gelu(dA, dB, bias.to(dev), dC)
        status, code = gsr.device_status()
    finally:
        gsr.set_path_override(gsr.PATH_AUTO)
    assert status == gsr.Status.OK, hex(code)
    return dC.cpu().numpy()


def check(C, ref, label):
    x = C.astype(np.float64)
    y = ref.astype(np.float64)
    assert not np.isnan(x).any(), "%s: unwritten outputs" % label
    err = np.abs(x - y)
    assert np.all(err <= 1e-2 + 1e-2 * np.abs(y)), "%s: worst %g" % (label, err.max())
    ny = np.linalg.norm(y)
    if ny > 0:
        assert np.linalg.norm(x - y) / ny <= 1e-3, label


PATHS = [gsr.PATH_TILED_256, gsr.PATH_TILED_128, gsr.PATH_TILED_64, gsr.PATH_PAIR, gsr.PATH_PAIR_128,
         gsr.PATH_SKINNY]
SHAPES = [(16, 264, 1000), (40, 128, 72), (129, 264, 72), (300, 776, 520), (1000, 1000, 8)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("path", PATHS)
def test_scale(M, N, K, path):
    if path == gsr.PATH_SKINNY and M > 256:
        pytest.skip("the small-M kernel serves at most 256 rows (65 to 256 only when forced)")
    A, B = make_inputs(M, N, K, seed=M + 2 * N + K)
    for alpha in (1.0, -0.75):
        C = run(oracle.EPI_SCALE, A, B, alpha, path=path)
        ref = oracle.gemm_epilogue(A, B, alpha, oracle.EPI_SCALE)
        check(C, ref, "scale %s alpha=%g path=%d" % ((M, N, K), alpha, path))


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("path", PATHS)
def test_bias_gelu(M, N, K, path):
    if path == gsr.PATH_SKINNY and M > 256:
        pytest.skip("the small-M kernel serves at most 256 rows (65 to 256 only when forced)")
    A, B = make_inputs(M, N, K, seed=M + 3 * N + K, b_std_inv_sqrt_k=True)
    bias = make_bias(N, seed=N)
    C = run(oracle.EPI_BIAS_GELU, A, B, bias=bias, path=path)
    ref = oracle.gemm_epilogue(A, B, kind=oracle.EPI_BIAS_GELU, bias=bias)
    check(C, ref, "bias_gelu %s path=%d" % ((M, N, K), path))


def test_plain_gemm_on_the_pages_instance():
    w = WORKLOADS["square1024"]
    A, B = make_inputs(w.M, w.N, w.K, seed=0)
    C = run(oracle.EPI_SCALE, A, B, 1.0)
    check(C, oracle.gemm_epilogue(A, B, 1.0, oracle.EPI_SCALE), "plain 1024")


def test_bias_gelu_llm_mlp_up_sampled_rows():
    # the MLP up-projection followed by its activation, at full size, on sampled rows
    w = WORKLOADS["llm_mlp_up"]
    A, B = make_inputs(w.M, w.N, w.K, seed=0, b_std_inv_sqrt_k=True)
    bias = make_bias(w.N, seed=5)
    C = run(oracle.EPI_BIAS_GELU, A, B, bias=bias)
    rows = sample_rows(w.M, count=32)
    ref = oracle.gemm_epilogue(A, B, kind=oracle.EPI_BIAS_GELU, bias=bias, rows=rows)
    check(C[rows], ref, "llm bias_gelu rows")


def test_bias_gelu_k_zero():
    bias = make_bias(72, seed=9)
    A = torch.zeros(5, 0, dtype=torch.float16)
    B = torch.zeros(0, 72, dtype=torch.float16)
    C = run(oracle.EPI_BIAS_GELU, A, B, bias=bias)
    ref = oracle.gemm_epilogue(A.numpy(), B.numpy(), kind=oracle.EPI_BIAS_GELU, bias=bias)
    check(C, ref, "K=0")


def test_bias_gelu_validation_on_device():
    dA = torch.empty(64, 64, dtype=torch.float16, device="cuda")
    dB = torch.empty(64, 64, dtype=torch.float16, device="cuda")
    dC = torch.empty(64, 64, dtype=torch.float16, device="cuda")
    bias = torch.empty(72, dtype=torch.float16, device="cuda")
    p = gsr.gemm_bias_gelu_ptr
    assert p(dA.data_ptr(), dB.data_ptr(), 0, dC.data_ptr(), 64, 64, 64) == gsr.Status.ERR_INVALID_ARG
    assert p(dA.data_ptr(), dB.data_ptr(), bias.data_ptr() + 2, dC.data_ptr(), 64, 64, 64) \
        == gsr.Status.ERR_ALIGNMENT
    assert p(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), dC.data_ptr(), 64, 64, 64) \
        == gsr.Status.ERR_ALIAS


@pytest.mark.parametrize("path", [gsr.PATH_PAIR, gsr.PATH_PAIR_128])
def test_pair_epilogues_beyond_two_waves(path):
    # The pair kernel has two copies: launches of at most two waves of work units (every shape
    # above) run the one whose epilogue loop is compiled per kind, longer launches the one that
    # reads the kind at run time.  This shape gives 190 units of 256 x 256 (171 tiles, the last
    # wave in halves) or 342 of 256 x 128 on 76 pairs: the second copy, every kind, checked whole.
    M, N, K = 2304, 4864, 136
    A, B = make_inputs(M, N, K, seed=11, b_std_inv_sqrt_k=True)
    C = run(oracle.EPI_SCALE, A, B, -0.75, path=path)
    check(C, oracle.gemm_epilogue(A, B, -0.75, oracle.EPI_SCALE), "scale path=%d" % path)
    bias = make_bias(N, seed=12)
    C = run(oracle.EPI_BIAS_GELU, A, B, bias=bias, path=path)
    check(C, oracle.gemm_epilogue(A, B, kind=oracle.EPI_BIAS_GELU, bias=bias), "bias_gelu path=%d" % path)
    dev = torch.device("cuda", 0)
    dA, dB = A.to(dev), B.to(dev)
    dC = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    gsr.set_path_override(path)
    try:
        gsr.gemm_scale_relu(dA, dB, dC, 0.5)
        status, code = gsr.device_status()
    finally:
        gsr.set_path_override(gsr.PATH_AUTO)
    assert status == gsr.Status.OK, hex(code)
    check(dC.cpu().numpy(), oracle.gemm_scale_relu(A, B, 0.5), "scale_relu path=%d" % path)
