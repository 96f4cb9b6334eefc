"""ctypes binding of libgsr: the same entry points as include/gsr.h, with argument
marshalling only.  Every step of C = ReLU(alpha * A @ B) runs in the library's CUDA
kernels; there is no Python or CPU fallback.  If libgsr.so is missing, the first call
raises instead of computing anything.

PyTorch is used only to hand over device memory and streams: tensors are passed as
raw pointers plus sizes, streams as their CUDA handles.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading

from . import _build


class Status(enum.IntEnum):
    OK = 0
    ERR_INVALID_ARG = 1
    ERR_ALIGNMENT = 2
    ERR_ALIAS = 3
    ERR_CUDA = 4
    ERR_DEVICE_TIMEOUT = 5
    ERR_UNSUPPORTED_DEVICE = 6
    ERR_SCRATCH_LIMIT = 7


class GsrError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = Status(status) if status in Status._value2member_map_ else status
        msg = "%s failed: %s" % (what, status_string(status))
        if status == Status.ERR_CUDA:
            msg += " (CUDA error %d)" % last_cuda_error()
        super().__init__(msg)


PATH_AUTO, PATH_TILED, PATH_SKINNY, PATH_TILED_256, PATH_TILED_128, PATH_PAIR, PATH_PAIR_128 = 0, 1, 2, 3, 4, 5, 6
PATH_TILED_64 = 7
KERNEL_TILED, KERNEL_SKINNY, KERNEL_PAIR, KERNEL_PAIR_128 = 0, 1, 2, 3

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded libgsr.so; raises ImportError when it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise ImportError(
                "libgsr.so not found at %s; build it first with "
                "`python -m tensor_core_gemm_multistage_gb300._build`" % path)
        L = ctypes.CDLL(path)
        vp, i64, f32, u32, u64, i32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_float,
                                       ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int)
        L.gemm_scale_relu.restype = i32
        L.gemm_scale_relu.argtypes = [vp, vp, vp, i64, i64, i64, f32, vp]
        L.gemm_scale.restype = i32
        L.gemm_scale.argtypes = [vp, vp, vp, i64, i64, i64, f32, vp]
        L.gemm_bias_gelu.restype = i32
        L.gemm_bias_gelu.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
        L.flash_attention_fwd.restype = i32
        L.flash_attention_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, f32, i32, vp]
        L.gemm_scale_relu_noalloc.restype = i32
        L.gemm_scale_relu_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, f32, vp]
        L.gemm_scale_relu_host.restype = i32
        L.gemm_scale_relu_host.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, f32, vp]
        L.gsr_device_status.restype = i32
        L.gsr_device_status.argtypes = [vp, ctypes.POINTER(i32)]
        L.gsr_release_stream.restype = i32
        L.gsr_release_stream.argtypes = [vp]
        L.gsr_select_path.restype = i32
        L.gsr_select_path.argtypes = [i64, i64, i64]
        L.gsr_set_path_override.restype = None
        L.gsr_set_path_override.argtypes = [i32]
        L.gsr_set_wait_timeout_ns.restype = None
        L.gsr_set_wait_timeout_ns.argtypes = [u64]
        L.gsr_set_raster_group.restype = None
        L.gsr_set_raster_group.argtypes = [i32]
        L.gsr_set_split_k.restype = None
        L.gsr_set_split_k.argtypes = [i32]
        L.gsr_set_test_flags.restype = None
        L.gsr_set_test_flags.argtypes = [u32]
        L.gsr_last_cuda_error.restype = i32
        L.gsr_last_cuda_error.argtypes = []
        L.gsr_status_string.restype = ctypes.c_char_p
        L.gsr_status_string.argtypes = [i32]
        L.gsr_version.restype = ctypes.c_char_p
        L.gsr_version.argtypes = []
        L.gsr_shutdown.restype = i32
        L.gsr_shutdown.argtypes = []
        _lib = L
        return L


# ---------------------------------------------------------------------------- raw C ABI

def gemm_scale_relu_ptr(A: int, B: int, C: int, M: int, N: int, K: int, alpha: float,
                        stream: int = 0) -> int:
    """The C entry point with raw integer pointers; returns the gsr_status code."""
    return lib().gemm_scale_relu(A or None, B or None, C or None, M, N, K, ctypes.c_float(alpha),
                                 stream or None)


def gemm_scale_relu_host_ptr(hA: int, hB: int, hC: int, dA: int, dB: int, dC: int, M: int, N: int,
                             K: int, alpha: float, stream: int = 0) -> int:
    return lib().gemm_scale_relu_host(hA or None, hB or None, hC or None, dA or None, dB or None,
                                      dC or None, M, N, K, ctypes.c_float(alpha), stream or None)


def select_path(M: int, N: int, K: int) -> int:
    return int(lib().gsr_select_path(M, N, K))


def set_path_override(path: int) -> None:
    lib().gsr_set_path_override(int(path))


def set_wait_timeout_ns(ns: int) -> None:
    lib().gsr_set_wait_timeout_ns(int(ns))


def set_raster_group(group: int) -> None:
    lib().gsr_set_raster_group(int(group))


def set_split_k(slabs: int) -> None:
    lib().gsr_set_split_k(int(slabs))


def set_test_flags(flags: int) -> None:
    lib().gsr_set_test_flags(int(flags))


def last_cuda_error() -> int:
    return int(lib().gsr_last_cuda_error())


def status_string(status: int) -> str:
    return lib().gsr_status_string(int(status)).decode()


def version() -> str:
    return lib().gsr_version().decode()


def shutdown() -> None:
    s = lib().gsr_shutdown()
    if s != Status.OK:
        raise GsrError(s, "gsr_shutdown")


# ---------------------------------------------------------------------------- torch tensors

def _stream_handle(stream, device) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check_matrix(t, name, shape=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != torch.float16:
        raise TypeError("%s must be float16, got %s" % (name, t.dtype))
    if t.dim() != 2:
        raise ValueError("%s must be 2-D, got shape %s" % (name, tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous (row-major)" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def gemm_scale_relu(A, B, C, alpha: float, stream=None):
    """C = ReLU(alpha * A @ B) into the preallocated fp16 tensor C (returned).

    A (M, K), B (K, N), C (M, N): contiguous float16 CUDA tensors on one device.
    Queued on ``stream`` (default: the current torch stream of that device).
    """
    import torch
    _check_matrix(A, "A")
    M, K = A.shape
    _check_matrix(B, "B")
    if B.shape[0] != K:
        raise ValueError("inner sizes differ: A %s, B %s" % (tuple(A.shape), tuple(B.shape)))
    N = B.shape[1]
    _check_matrix(C, "C", (M, N))
    dev = C.device
    if dev.type != "cuda" or A.device != dev or B.device != dev:
        raise ValueError("A, B and C must be CUDA tensors on one device")
    with torch.cuda.device(dev):
        s = lib().gemm_scale_relu(A.data_ptr() or None, B.data_ptr() or None, C.data_ptr() or None,
                                  M, N, K, ctypes.c_float(alpha), _stream_handle(stream, dev) or None)
    if s != Status.OK:
        raise GsrError(s, "gemm_scale_relu")
    return C


def _operands(A, B, C):
    _check_matrix(A, "A")
    M, K = A.shape
    _check_matrix(B, "B")
    if B.shape[0] != K:
        raise ValueError("inner sizes differ: A %s, B %s" % (tuple(A.shape), tuple(B.shape)))
    N = B.shape[1]
    _check_matrix(C, "C", (M, N))
    dev = C.device
    if dev.type != "cuda" or A.device != dev or B.device != dev:
        raise ValueError("A, B and C must be CUDA tensors on one device")
    return M, N, K, dev


def gemm_scale(A, B, C, alpha: float = 1.0, stream=None):
    """C = alpha * A @ B into the preallocated fp16 tensor C (alpha = 1: plain GEMM)."""
    import torch
    M, N, K, dev = _operands(A, B, C)
    with torch.cuda.device(dev):
        s = lib().gemm_scale(A.data_ptr() or None, B.data_ptr() or None, C.data_ptr() or None,
                             M, N, K, ctypes.c_float(alpha), _stream_handle(stream, dev) or None)
    if s != Status.OK:
        raise GsrError(s, "gemm_scale")
    return C


def gemm_bias_gelu(A, B, bias, C, stream=None):
    """C = GELU(A @ B + bias) (tanh form), bias an fp16 CUDA vector of length N."""
    import torch
    M, N, K, dev = _operands(A, B, C)
    if not isinstance(bias, torch.Tensor) or bias.dtype != torch.float16 or bias.dim() != 1 \
            or bias.shape[0] != N or not bias.is_contiguous() or bias.device != dev:
        raise ValueError("bias must be a contiguous float16 CUDA vector of length N on C's device")
    with torch.cuda.device(dev):
        s = lib().gemm_bias_gelu(A.data_ptr() or None, B.data_ptr() or None,
                                 bias.data_ptr() or None, C.data_ptr() or None, M, N, K,
                                 _stream_handle(stream, dev) or None)
    if s != Status.OK:
        raise GsrError(s, "gemm_bias_gelu")
    return C


def gemm_bias_gelu_ptr(A: int, B: int, bias: int, C: int, M: int, N: int, K: int,
                       stream: int = 0) -> int:
    return lib().gemm_bias_gelu(A or None, B or None, bias or None, C or None, M, N, K,
                                stream or None)


def flash_attention_fwd(Q, K, V, O, lse=None, softmax_scale: float = 0.0, causal: bool = False,
                        stream=None):
    """O = softmax(scale * Q K^T [causal]) V for fp16 CUDA tensors Q (B,H,Sq,D), K and V
    (B,H,Skv,D), O (B,H,Sq,D); D in {64, 128}; scale 0 means 1/sqrt(D).  ``lse``: optional
    float32 (B,H,Sq) receiving the log-sum-exp of the scaled scores."""
    import torch
    for name, t in (("Q", Q), ("K", K), ("V", V), ("O", O)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float16 or t.dim() != 4 \
                or not t.is_contiguous() or t.device.type != "cuda":
            raise ValueError("%s must be a contiguous 4-D float16 CUDA tensor" % name)
    B, H, Sq, D = Q.shape
    Skv = K.shape[2]
    if tuple(K.shape) != (B, H, Skv, D) or tuple(V.shape) != (B, H, Skv, D) \
            or tuple(O.shape) != (B, H, Sq, D):
        raise ValueError("shapes: Q %s K %s V %s O %s" % (tuple(Q.shape), tuple(K.shape),
                                                            tuple(V.shape), tuple(O.shape)))
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Sq)
                            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 (B, H, Sq) tensor")
    dev = O.device
    with torch.cuda.device(dev):
        s = lib().flash_attention_fwd(Q.data_ptr() or None, K.data_ptr() or None,
                                      V.data_ptr() or None, O.data_ptr() or None,
                                      lse.data_ptr() if lse is not None else None,
                                      B, H, Sq, Skv, D, ctypes.c_float(softmax_scale),
                                      1 if causal else 0, _stream_handle(stream, dev) or None)
    if s != Status.OK:
        raise GsrError(s, "flash_attention_fwd")
    return O


def gemm_scale_relu_host(hA, hB, hC, dA, dB, dC, alpha: float, stream=None):
    """Host-memory variant: hA, hB (pinned CPU fp16) are copied into dA, dB, the product
    is computed into dC and copied back into hC (pinned CPU fp16), all on ``stream``."""
    import torch
    _check_matrix(hA, "hA")
    M, K = hA.shape
    _check_matrix(hB, "hB")
    N = hB.shape[1]
    _check_matrix(hC, "hC", (M, N))
    _check_matrix(dA, "dA", (M, K))
    _check_matrix(dB, "dB", (K, N))
    _check_matrix(dC, "dC", (M, N))
    dev = dC.device
    with torch.cuda.device(dev):
        s = lib().gemm_scale_relu_host(hA.data_ptr() or None, hB.data_ptr() or None,
                                       hC.data_ptr() or None, dA.data_ptr() or None,
                                       dB.data_ptr() or None, dC.data_ptr() or None, M, N, K,
                                       ctypes.c_float(alpha), _stream_handle(stream, dev) or None)
    if s != Status.OK:
        raise GsrError(s, "gemm_scale_relu_host")
    return hC


def release_stream(stream=None, device=None):
    """Frees the library's error word and small-M workspace of ``stream`` (after waiting
    for it); a later call on the stream allocates afresh."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        s = lib().gsr_release_stream(_stream_handle(stream, dev) or None)
    if s != Status.OK:
        raise GsrError(s, "gsr_release_stream")


def device_status(stream=None, device=None):
    """Waits for ``stream`` and returns (Status, raw device error code)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    code = ctypes.c_int(0)
    with torch.cuda.device(dev):
        s = lib().gsr_device_status(_stream_handle(stream, dev) or None, ctypes.byref(code))
    return Status(s), int(code.value)
