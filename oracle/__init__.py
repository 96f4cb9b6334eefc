"""CPU oracle for the fused operator C = ReLU(alpha * A @ B) (fp16 in, fp64 sum, fp16 out).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The GPU library
never calls it and shares no code with it; the library fails loudly when its
CUDA extension is missing instead of falling back here.

The arithmetic lives in ``gsr_oracle.c`` (plain C, built with gcc); this module
only builds that file and marshals numpy arrays through ctypes.

Sources (page title and section):
  * the aikraft.ru TileLang tutorial survey ("TileLang: создание высокопроизводительных
    GPU-ядер"), sections 2 (make_matmul, plain tiled GEMM) and 4 (make_matmul_bias_gelu) for
    the further epilogues of ``gemm_epilogue``;
  * "Tutorial14: 使用TileLang语言编写attention算子", section 3 (operator formula)
    and section 2 (the gemm_fused kernel: fp16 inputs, float accumulator,
    multiply by the float32 scale, then max with 0, fp16 output);
  * "TileKernels：面向大语言模型的高性能GPU算子库解析", section 五 (the plain
    triple-loop custom_matmul example).

Pins: ``tests/test_oracle.py`` checks this oracle against the binary16 format
definition, numpy's independent codec, closed forms (identity B, all-ones,
one-hot rows, negative alpha) and exact rational brute force on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gsr_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libgsr_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gsr_oracle.c`` into ``oracle/_build/libgsr_oracle.so`` with gcc."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_gemm_scale_relu.restype = ctypes.c_int
        lib.oracle_gemm_scale_relu.argtypes = [
            u16p, u16p, u16p, f64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_float, i64p, ctypes.c_int64]
        lib.oracle_gemm_epilogue.restype = ctypes.c_int
        lib.oracle_gemm_epilogue.argtypes = [
            u16p, u16p, u16p, u16p, f64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_float, ctypes.c_int, i64p, ctypes.c_int64]
        lib.oracle_f16_decode_array.restype = None
        lib.oracle_f16_decode_array.argtypes = [u16p, f64p, ctypes.c_int64]
        lib.oracle_f16_encode_array.restype = None
        lib.oracle_f16_encode_array.argtypes = [f64p, u16p, ctypes.c_int64]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_set_num_threads.restype = None
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _as_bits(x) -> np.ndarray:
    """Return a C-contiguous uint16 view of fp16 data (numpy or torch CPU tensor)."""
    if hasattr(x, "detach"):             # torch tensor: keep the exact fp16 bytes
        x = x.detach().cpu().contiguous().view(dtype=_torch_int16()).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16 or x.dtype == np.int16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs must be binary16 data, got %s" % x.dtype)
    return x


def _torch_int16():
    import torch
    return torch.int16


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def gemm_scale_relu(A, B, alpha: float, rows=None, return_pre: bool = False):
    """C = ReLU(alpha * A @ B) for fp16 A (M,K), B (K,N), summed in fp64.

    ``rows`` (optional) restricts the output to those rows of C, in the given
    order.  Returns C as a float16 array of shape (R, N); with ``return_pre``
    also returns Z = alpha * A @ B in fp64 (before the ReLU), same shape.
    """
    lib = _load()
    a = _as_bits(A)
    b = _as_bits(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
        raise ValueError("shape mismatch: A %s, B %s" % (a.shape, b.shape))
    M, K = a.shape
    N = b.shape[1]
    if rows is None:
        R = M
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        R = rows_arr.shape[0]
    c = np.zeros((R, N), dtype=np.uint16)
    z = np.zeros((R, N), dtype=np.float64) if return_pre else None
    # empty arrays still need a valid pointer for ctypes
    a_buf = a if a.size else np.zeros(1, np.uint16)
    b_buf = b if b.size else np.zeros(1, np.uint16)
    c_buf = c if c.size else np.zeros(1, np.uint16)
    rc = lib.oracle_gemm_scale_relu(
        _ptr(a_buf, ctypes.c_uint16), _ptr(b_buf, ctypes.c_uint16), _ptr(c_buf, ctypes.c_uint16),
        _ptr(z, ctypes.c_double) if (z is not None and z.size) else None,
        M, N, K, ctypes.c_float(alpha),
        _ptr(rows_arr, ctypes.c_int64) if rows_arr is not None and R else None,
        R)
    if rc == -1:
        raise ValueError("oracle rejected the arguments (row index out of range?)")
    if rc != 0:
        raise MemoryError("oracle ran out of memory")
    c16 = c.view(np.float16)
    return (c16, z) if return_pre else c16


EPI_SCALE_RELU, EPI_SCALE, EPI_BIAS_GELU = 0, 1, 2


def gemm_epilogue(A, B, alpha: float = 1.0, kind: int = EPI_SCALE_RELU, bias=None, rows=None,
                  return_pre: bool = False):
    """C = epilogue(A @ B) for fp16 A (M,K), B (K,N), summed in fp64.

    kind 0: ReLU(alpha * sum); 1: alpha * sum; 2: GELU(sum + bias) (tanh form written with
    the exponential as x / (1 + exp(-2u)); ``bias`` fp16 of length N).  With ``return_pre`` also returns Y, the fp64
    value before the final rounding to fp16.
    """
    lib = _load()
    a = _as_bits(A)
    b = _as_bits(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
        raise ValueError("shape mismatch: A %s, B %s" % (a.shape, b.shape))
    M, K = a.shape
    N = b.shape[1]
    if kind == EPI_BIAS_GELU:
        bb = _as_bits(bias).reshape(-1)
        if bb.shape[0] != N:
            raise ValueError("bias must have N = %d values" % N)
    else:
        bb = np.zeros(max(N, 1), np.uint16)
    if rows is None:
        R, rows_arr = M, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        R = rows_arr.shape[0]
    c = np.zeros((R, N), dtype=np.uint16)
    y = np.zeros((R, N), dtype=np.float64) if return_pre else None
    a_buf = a if a.size else np.zeros(1, np.uint16)
    b_buf = b if b.size else np.zeros(1, np.uint16)
    bb_buf = bb if bb.size else np.zeros(1, np.uint16)
    c_buf = c if c.size else np.zeros(1, np.uint16)
    rc = lib.oracle_gemm_epilogue(
        _ptr(a_buf, ctypes.c_uint16), _ptr(b_buf, ctypes.c_uint16), _ptr(bb_buf, ctypes.c_uint16),
        _ptr(c_buf, ctypes.c_uint16),
        _ptr(y, ctypes.c_double) if (y is not None and y.size) else None,
        M, N, K, ctypes.c_float(alpha), int(kind),
        _ptr(rows_arr, ctypes.c_int64) if rows_arr is not None and R else None, R)
    if rc == -1:
        raise ValueError("oracle rejected the arguments")
    if rc != 0:
        raise MemoryError("oracle ran out of memory")
    c16 = c.view(np.float16)
    return (c16, y) if return_pre else c16


def f16_decode(bits) -> np.ndarray:
    """binary16 bit patterns (uint16) -> exact float64 values."""
    lib = _load()
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    out = np.empty(b.shape, dtype=np.float64)
    if b.size:
        lib.oracle_f16_decode_array(_ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double), b.size)
    return out


def f16_encode(x) -> np.ndarray:
    """float64 values -> binary16 bit patterns (uint16), round to nearest even."""
    lib = _load()
    v = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(v.shape, dtype=np.uint16)
    if v.size:
        lib.oracle_f16_encode_array(_ptr(v, ctypes.c_double), _ptr(out, ctypes.c_uint16), v.size)
    return out


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))
