"""GB300-native fused GEMM + scale + ReLU: C = ReLU(alpha * A @ B), fp16 in/out, fp32 sum.

The product is the C-ABI library ``libgsr.so`` (include/gsr.h) built from the CUDA
sources in ``csrc/`` for sm_103a; this package holds its ctypes binding and the seeded
input generators.  Operator: "Tutorial14: 使用TileLang语言编写attention算子", sections 2
and 3.
"""
from .binding import (KERNEL_PAIR, KERNEL_PAIR_128, KERNEL_SKINNY, KERNEL_TILED, PATH_AUTO, PATH_PAIR, PATH_PAIR_128,
                      PATH_SKINNY, PATH_TILED, PATH_TILED_64, PATH_TILED_128, PATH_TILED_256,
                      GsrError, Status, device_status, flash_attention_fwd, gemm_bias_gelu, release_stream,
                      gemm_bias_gelu_ptr,
                      gemm_scale, gemm_scale_relu, gemm_scale_relu_host,
                      gemm_scale_relu_host_ptr, gemm_scale_relu_ptr, last_cuda_error, lib,
                      library_path, select_path, set_path_override, set_raster_group, set_split_k, set_test_flags,
                      set_wait_timeout_ns, shutdown, status_string, version)
from ._build import build

__all__ = [
    "KERNEL_PAIR", "KERNEL_PAIR_128", "KERNEL_SKINNY", "KERNEL_TILED", "PATH_AUTO", "PATH_PAIR", "PATH_PAIR_128", "PATH_SKINNY", "PATH_TILED", "PATH_TILED_64", "PATH_TILED_128", "PATH_TILED_256", "GsrError",
    "Status", "build", "device_status", "flash_attention_fwd", "gemm_bias_gelu", "gemm_bias_gelu_ptr", "gemm_scale",
    "gemm_scale_relu", "gemm_scale_relu_host",
    "gemm_scale_relu_host_ptr", "gemm_scale_relu_ptr", "last_cuda_error", "lib", "library_path",
    "release_stream", "select_path", "set_path_override", "set_raster_group", "set_split_k", "set_test_flags", "set_wait_timeout_ns", "shutdown",
    "status_string", "version",
]
