"""The C ABI without a GPU: the library builds and loads, exports every function that
include/gsr.h declares, and rejects bad arguments before touching CUDA.  The device addresses
below are fake: every call here must be rejected before a launch (or run only where no GPU is
present), since a launch on them would fault a real GPU."""
import ctypes
import os
import re

import pytest

import tensor_core_gemm_multistage_gb300 as gsr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gsr.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    gsr.build()
    yield


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)      # drop comments
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for must in ("gemm_scale_relu", "gemm_scale_relu_host", "gsr_device_status", "gsr_version"):
        assert must in names


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(gsr.library_path())
    missing = [n for n in _declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_status_enum_matches_header():
    text = open(HEADER).read()
    for name, value in re.findall(r"GSR_(OK|ERR_\w+)\s*=\s*(\d+)", text):
        assert gsr.Status[name] == int(value)
        assert gsr.status_string(int(value)) == "GSR_" + name


def test_version():
    assert gsr.version().startswith("gsr ") and "sm_103a" in gsr.version()


# Fake, never-dereferenced device addresses: validation must answer before any CUDA call.
A, B, C = 0x10000, 0x200000, 0x4000000


@pytest.mark.parametrize("M,N,K", [(-1, 8, 8), (8, -8, 8), (8, 8, -8), (2 ** 31, 8, 8),
                                   (8, 2 ** 31, 8), (8, 8, 2 ** 31)])
def test_bad_sizes(M, N, K):
    assert gsr.gemm_scale_relu_ptr(A, B, C, M, N, K, 1.0) == gsr.Status.ERR_INVALID_ARG


@pytest.mark.parametrize("M,N", [(0, 8), (8, 0), (0, 0)])
def test_empty_output_is_a_no_op(M, N):
    assert gsr.gemm_scale_relu_ptr(0, 0, 0, M, N, 8, 1.0) == gsr.Status.OK


def test_null_pointers():
    assert gsr.gemm_scale_relu_ptr(A, B, 0, 4, 8, 8, 1.0) == gsr.Status.ERR_INVALID_ARG
    assert gsr.gemm_scale_relu_ptr(0, B, C, 4, 8, 8, 1.0) == gsr.Status.ERR_INVALID_ARG
    assert gsr.gemm_scale_relu_ptr(A, 0, C, 4, 8, 8, 1.0) == gsr.Status.ERR_INVALID_ARG


@pytest.mark.parametrize("a,b,c,N,K", [
    (A + 8, B, C, 8, 8), (A, B + 2, C, 8, 8), (A, B, C + 4, 8, 8),   # pointers not 16-byte aligned
    (A, B, C, 12, 8), (A, B, C, 8, 12), (A, B, C, 1, 8), (A, B, C, 8, 1)])   # pitches not 16 bytes
def test_alignment(a, b, c, N, K):
    assert gsr.gemm_scale_relu_ptr(a, b, c, 4, N, K, 1.0) == gsr.Status.ERR_ALIGNMENT


def test_alias():
    M, N, K = 64, 64, 64
    assert gsr.gemm_scale_relu_ptr(A, B, A, M, N, K, 1.0) == gsr.Status.ERR_ALIAS
    assert gsr.gemm_scale_relu_ptr(A, B, B + 16 * 64, M, N, K, 1.0) == gsr.Status.ERR_ALIAS
    # C ending exactly where A begins does not overlap.  That call passes every check and
    # would launch a kernel on these fake addresses, so it runs only where there is no GPU.
    import torch
    if not torch.cuda.is_available():
        assert gsr.gemm_scale_relu_ptr(A, B, A - M * N * 2, M, N, K, 1.0) != gsr.Status.ERR_ALIAS


def test_host_entry_validates_the_same_way():
    assert gsr.gemm_scale_relu_host_ptr(1, 1, 1, A, B, C, -1, 8, 8, 1.0) == gsr.Status.ERR_INVALID_ARG
    assert gsr.gemm_scale_relu_host_ptr(0, 1, 1, A, B, C, 4, 8, 8, 1.0) == gsr.Status.ERR_INVALID_ARG
    assert gsr.gemm_scale_relu_host_ptr(1, 1, 1, A, B, A, 4, 8, 8, 1.0) == gsr.Status.ERR_ALIAS


def test_path_selection_and_override():
    try:
        assert gsr.select_path(16, 16384, 16384) == 1
        assert gsr.select_path(64, 8192, 8192) == 1
        assert gsr.select_path(16, 4096, 2048) == 1          # B of exactly 16 MiB
        # up to 64 rows with a small B the launch is latency-bound: one-CTA tiles
        assert gsr.select_path(64, 8, 8) == gsr.KERNEL_TILED
        assert gsr.select_path(64, 1024, 2048) == gsr.KERNEL_TILED
        assert gsr.select_path(16, 4096, 2040) == gsr.KERNEL_TILED
        assert gsr.select_path(65, 8, 8) == gsr.KERNEL_TILED
        assert gsr.select_path(8192, 8192, 8192) == gsr.KERNEL_PAIR
        assert gsr.select_path(16384, 14336, 4096) == gsr.KERNEL_PAIR
        assert gsr.select_path(1024, 1024, 1024) == gsr.KERNEL_TILED
        # 96 256x256 pair tiles on 76 pairs: one full wave, then the other 20 tiles as 40
        # half-width units (~1.56 tile times); 192 tiles of 256x128 need three waves (~1.68)
        assert gsr.select_path(2000, 3000, 1000) == gsr.KERNEL_PAIR
        # 256 tiles of 16384 x 1024 leave 28 for a last wave of halves (~3.56 tile times)
        assert gsr.select_path(16384, 1024, 1024) == gsr.KERNEL_PAIR
        # N = 128: a 256 x 256 tile is half empty, 256 x 128 tiles do the same work in ~0.68
        assert gsr.select_path(20000, 128, 512) == gsr.KERNEL_PAIR_128
        # N = 384 and 640 at K = 4096: 256 x 256 tiles measured 4.7 % and 17 % faster than
        # 256 x 128 ones (2 against 3 waves, 3 against 5)
        assert gsr.select_path(16384, 384, 4096) == gsr.KERNEL_PAIR
        assert gsr.select_path(16384, 640, 4096) == gsr.KERNEL_PAIR
        assert gsr.select_path(4096, 4096, 4096) == gsr.KERNEL_PAIR
        # below a full wave of pair tiles: 128 x 256 single tiles up to K ~ 6000, pairs beyond
        # (their faster K loop repays their larger cost per launch); 128 x 128 single tiles,
        # which use twice the SMs, stay at any K
        assert gsr.select_path(256, 16384, 4096) == gsr.KERNEL_TILED
        assert gsr.select_path(256, 16384, 8192) == gsr.KERNEL_PAIR
        assert gsr.select_path(256, 16384, 6136) == gsr.KERNEL_TILED
        assert gsr.select_path(256, 16384, 6144) == gsr.KERNEL_PAIR
        assert gsr.select_path(2048, 2048, 2048) == gsr.KERNEL_TILED
        assert gsr.select_path(2048, 2048, 16384) == gsr.KERNEL_PAIR
        assert gsr.select_path(1024, 2048, 16384) == gsr.KERNEL_TILED
        # 65 to 128 rows: the small-M kernel (MMA N 128) where B is streamed from HBM (64 MiB
        # or more) and one-CTA tiles would keep under two thirds of the SMs busy
        assert gsr.select_path(100, 4096, 14336) == gsr.KERNEL_SKINNY    # 64 tiles, B 117 MB
        assert gsr.select_path(128, 4096, 16384) == gsr.KERNEL_SKINNY
        assert gsr.select_path(96, 6144, 9216) == gsr.KERNEL_SKINNY      # 96 tiles
        assert gsr.select_path(128, 2048, 4096) == gsr.KERNEL_TILED      # B 17 MB
        assert gsr.select_path(128, 4096, 8192) == gsr.KERNEL_SKINNY     # B 64 MiB
        assert gsr.select_path(128, 4096, 6144) == gsr.KERNEL_TILED      # B 48 MiB
        assert gsr.select_path(100, 8192, 8192) == gsr.KERNEL_TILED      # 128 tiles
        assert gsr.select_path(128, 16384, 16384) == gsr.KERNEL_TILED
        assert gsr.select_path(129, 4096, 14336) == gsr.KERNEL_TILED
        # at 128 rows or fewer a 256-row pair tile is at least half empty: one-CTA tiles
        assert gsr.select_path(100, 28672, 8192) == gsr.KERNEL_TILED
        assert gsr.select_path(128, 65536, 4096) == gsr.KERNEL_TILED
        assert gsr.select_path(129, 65536, 4096) == gsr.KERNEL_PAIR
        # up to K = 384 a tile is mostly its epilogue: one-CTA tiles, not pairs
        assert gsr.select_path(4096, 16384, 384) == gsr.KERNEL_TILED
        assert gsr.select_path(4096, 16384, 392) == gsr.KERNEL_PAIR
        gsr.set_path_override(gsr.PATH_TILED)
        assert gsr.select_path(16, 16384, 16384) == 0
        assert gsr.select_path(8192, 8192, 8192) == 0
        gsr.set_path_override(gsr.PATH_PAIR)
        assert gsr.select_path(1024, 1024, 1024) == gsr.KERNEL_PAIR
        assert gsr.select_path(2000, 3000, 1000) == gsr.KERNEL_PAIR
        gsr.set_path_override(gsr.PATH_PAIR_128)
        assert gsr.select_path(8192, 8192, 8192) == gsr.KERNEL_PAIR_128
        gsr.set_path_override(gsr.PATH_TILED_64)
        assert gsr.select_path(8192, 8192, 8192) == gsr.KERNEL_TILED
        assert gsr.select_path(16, 8, 8) == gsr.KERNEL_TILED
        gsr.set_path_override(gsr.PATH_SKINNY)
        assert gsr.select_path(16, 8, 8) == 1
        assert gsr.select_path(100, 8, 8) == 1      # forced, it also takes 65 to 256 rows
        assert gsr.select_path(256, 8, 8) == 1
        assert gsr.select_path(257, 8, 8) == 0
    finally:
        gsr.set_path_override(gsr.PATH_AUTO)


def test_without_a_gpu_a_valid_call_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    s = gsr.gemm_scale_relu_ptr(A, B, C, 4, 8, 8, 1.0)
    assert s == gsr.Status.ERR_CUDA
    assert gsr.last_cuda_error() != 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from tensor_core_gemm_multistage_gb300 import _build, binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "libgsr.so"))
    with pytest.raises(ImportError):
        binding.lib()


def test_bias_gelu_argument_checks_need_no_gpu():
    p = gsr.gemm_bias_gelu_ptr
    assert p(A, B, 0, C, 4, 8, 8) == gsr.Status.ERR_INVALID_ARG             # no bias
    assert p(A, B, 0x300008, C, 4, 8, 8) == gsr.Status.ERR_ALIGNMENT         # bias not 16-byte aligned
    assert p(A, B, C + 16, C, 4, 8, 8) == gsr.Status.ERR_ALIAS               # bias inside C
    assert p(A, B, 0, C, 0, 8, 8) == gsr.Status.OK                           # empty output


def test_scale_entry_validates_like_the_fused_one():
    L = gsr.lib()
    assert L.gemm_scale(A, B, C, -1, 8, 8, ctypes.c_float(1.0), None) == gsr.Status.ERR_INVALID_ARG
    assert L.gemm_scale(A, B, A, 64, 64, 64, ctypes.c_float(1.0), None) == gsr.Status.ERR_ALIAS


def test_noalloc_limits_are_checked_before_any_cuda_call():
    # gemm_scale_relu_noalloc refuses M > 64 and sizes whose per-tile tickets alone exceed its
    # fixed scratch array before it touches CUDA, so without a GPU these answer with the
    # specific codes rather than GSR_ERR_CUDA.  The addresses are fake (A small, B 8 GiB at
    # 64 GiB, C 64 GiB at 1 TiB: no overlaps), so this runs only where no GPU is present.
    import torch
    if torch.cuda.is_available():
        pytest.skip("fake device addresses: runs only where no GPU is present")
    L = gsr.lib()
    vp = ctypes.c_void_p
    a, b, c = vp(0x10000), vp(1 << 36), vp(1 << 40)
    one = ctypes.c_float(1.0)
    assert L.gemm_scale_relu_noalloc(a, b, c, 64, 1 << 29, 8, one, None) == gsr.Status.ERR_SCRATCH_LIMIT
    assert L.gemm_scale_relu_noalloc(a, b, c, 65, 64, 8, one, None) == gsr.Status.ERR_INVALID_ARG
    # below the device-independent limit the call goes on to query the (absent) device
    assert L.gemm_scale_relu_noalloc(a, b, c, 64, 1 << 20, 8, one, None) == gsr.Status.ERR_CUDA


def test_release_stream_without_a_gpu_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert gsr.lib().gsr_release_stream(None) == gsr.Status.ERR_CUDA
