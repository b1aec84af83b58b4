"""CPU oracle for the pipelined GEMM library -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the C-ABI library and
its Python binding) never imports, links or calls it, and it shares no code
with them: inputs reach both sides from ``pipelined_warp_specialized_gb300.inputs``,
which holds only the seeded random-number recipe.

What it computes (the plain definitions the pipelined kernels reach exactly,
up to rounding order):

* ``gemm_s32_nn`` -- Croqtile tutorial ch.6, section "使用 swap 的双缓冲":
  ``out[m,n] = sum_k lhs[m,k] * rhs[k,n]`` over int32 inputs, summed exactly
  and wrapped to int32 (two's complement).
* ``gemm_f16_nt_f64`` -- Croqtile tutorial ch.6, section "带 event 的 1P1C 内核":
  ``ref[m,n] = sum_k lhs[m,k] * rhs[n,k]`` with ``rhs`` stored ``[N,K]``
  (C = A . B^T), f16 inputs decoded exactly and summed in binary64.
* ``f64_to_f16`` / ``f16_to_f64`` -- the IEEE 754 binary16 format, rounding
  to nearest, ties to even, directly from binary64.
* ``f16_tolerance`` / ``check_f16`` -- the acceptance rule for the f16 path:
  ``|gpu - ref| <= ulp16(ref) + 1e-3 * sqrt(K)``, where ``ulp16(x)`` is the
  binary16 spacing at ``|x|`` (``2^(max(floor(log2|x|), -14) - 10)``; ``2^-24``
  at zero and in the subnormal range).

The arithmetic lives in ``gemm_oracle.c`` (plain C, built with gcc by
``build()``); this module only marshals numpy arrays.  ``ring_model`` holds a
CPU model of the S-slot full/empty credit protocol.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gemm_oracle.c`` into ``oracle/_build/liboracle.so`` with gcc."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f64.restype = ctypes.c_double
    lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_f16.restype = ctypes.c_uint16
    lib.oracle_f16_to_f64_array.argtypes = [p, p, i64]
    lib.oracle_f64_to_f16_array.argtypes = [p, p, i64]
    lib.oracle_gemm_s32_nn.argtypes = [i64, i64, i64, p, p, p, i32]
    lib.oracle_gemm_f16_nt.argtypes = [i64, i64, i64, p, p, p, i32]
    lib.oracle_gemm_f16_nt.restype = ctypes.c_int
    lib.oracle_gemm_f16_nt_entries.argtypes = [i64, p, p, p, p, i64, p, i32]
    lib.oracle_gemm_s32_nn_entries.argtypes = [i64, i64, p, p, p, p, i64, p, i32]
    _lib = lib
    return lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _f16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    if x.dtype == np.uint16:
        return x
    raise TypeError(f"expected float16 or uint16 bit patterns, got {x.dtype}")


# --------------------------------------------------------------------------
# binary16 codec
# --------------------------------------------------------------------------

def f16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode binary16 values (float16 or uint16 bit patterns) to float64."""
    h = _f16_bits(np.asarray(bits))
    out = np.empty(h.shape, dtype=np.float64)
    _load().oracle_f16_to_f64_array(_ptr(h), _ptr(out), h.size)
    return out


def f64_to_f16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to binary16 (nearest, ties to even); uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f64_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


# --------------------------------------------------------------------------
# the two products
# --------------------------------------------------------------------------

def gemm_s32_nn(lhs: np.ndarray, rhs: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """out[M,N] = lhs[M,K] . rhs[K,N], exact sum wrapped to int32."""
    lhs = np.ascontiguousarray(lhs, dtype=np.int32)
    rhs = np.ascontiguousarray(rhs, dtype=np.int32)
    M, K = lhs.shape
    K2, N = rhs.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    out = np.zeros((M, N), dtype=np.int32)
    if M and N:
        _load().oracle_gemm_s32_nn(M, N, K, _ptr(lhs), _ptr(rhs), _ptr(out),
                                   nthreads or default_threads())
    return out


def gemm_f16_nt_f64(lhs: np.ndarray, rhs: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """ref[M,N] = lhs[M,K] . rhs[N,K]^T summed in float64 (f16 inputs)."""
    a = _f16_bits(lhs)
    b = _f16_bits(rhs)
    M, K = a.shape
    N, K2 = b.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    out = np.zeros((M, N), dtype=np.float64)
    if M and N:
        rc = _load().oracle_gemm_f16_nt(M, N, K, _ptr(a), _ptr(b), _ptr(out),
                                        nthreads or default_threads())
        if rc != 0:
            raise MemoryError("oracle could not allocate decoded operands")
    return out


def gemm_f16_nt_entries(lhs: np.ndarray, rhs: np.ndarray, rows: np.ndarray, cols: np.ndarray,
                        nthreads: int | None = None) -> np.ndarray:
    """ref[i] = sum_k lhs[rows[i],k] * rhs[cols[i],k] in float64."""
    a = _f16_bits(lhs)
    b = _f16_bits(rhs)
    K = a.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in shape")
    if rows.size and (rows.min() < 0 or rows.max() >= a.shape[0] or cols.min() < 0 or cols.max() >= b.shape[0]):
        raise IndexError("entry index out of range")
    out = np.zeros(rows.shape, dtype=np.float64)
    if rows.size:
        _load().oracle_gemm_f16_nt_entries(K, _ptr(a), _ptr(b), _ptr(rows), _ptr(cols), rows.size,
                                           _ptr(out), nthreads or default_threads())
    return out


def gemm_s32_nn_entries(lhs: np.ndarray, rhs: np.ndarray, rows: np.ndarray, cols: np.ndarray,
                        nthreads: int | None = None) -> np.ndarray:
    """out[i] = sum_k lhs[rows[i],k] * rhs[k,cols[i]], wrapped to int32."""
    lhs = np.ascontiguousarray(lhs, dtype=np.int32)
    rhs = np.ascontiguousarray(rhs, dtype=np.int32)
    K, N = rhs.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= lhs.shape[0] or cols.min() < 0 or cols.max() >= N):
        raise IndexError("entry index out of range")
    out = np.zeros(rows.shape, dtype=np.int32)
    if rows.size:
        _load().oracle_gemm_s32_nn_entries(N, K, _ptr(lhs), _ptr(rhs), _ptr(rows), _ptr(cols),
                                           rows.size, _ptr(out), nthreads or default_threads())
    return out


# --------------------------------------------------------------------------
# acceptance rule for the f16 path
# --------------------------------------------------------------------------

def f16_ulp(ref: np.ndarray) -> np.ndarray:
    """Binary16 spacing at |ref|: 2^(max(floor(log2|ref|), -14) - 10)."""
    ref = np.asarray(ref, dtype=np.float64)
    _, e = np.frexp(np.abs(ref))          # |ref| = m * 2^e, m in [0.5, 1)
    expo = np.maximum(e - 1, -14)         # floor(log2|ref|), clamped to the subnormal range
    ulp = np.ldexp(1.0, expo - 10)
    return np.where(ref == 0.0, 2.0 ** -24, ulp)


def f16_tolerance(ref: np.ndarray, K: int) -> np.ndarray:
    return f16_ulp(ref) + 1e-3 * np.sqrt(float(K))


def check_f16(gpu: np.ndarray, ref: np.ndarray, K: int) -> dict:
    """Compare GPU f16 results with the float64 oracle.

    Returns a summary; ``ok`` is True when every element satisfies
    ``|gpu - ref| <= ulp16(ref) + 1e-3 sqrt(K)``.  Where the oracle's value
    rounds to an infinity in binary16 the GPU must hold the same infinity.
    """
    g = f16_to_f64(gpu)
    ref = np.asarray(ref, dtype=np.float64)
    ref16 = f16_to_f64(f64_to_f16(ref))
    tol = f16_tolerance(ref, K)
    inf_ref = np.isinf(ref16)
    err = np.abs(g - ref)
    bad = np.where(inf_ref, g != ref16, ~(err <= tol))
    finite = ~inf_ref
    return {
        "ok": not bool(bad.any()),
        "n_bad": int(bad.sum()),
        "n": int(ref.size),
        "max_err": float(err[finite].max()) if finite.any() else 0.0,
        "max_err_over_tol": float((err[finite] / tol[finite]).max()) if finite.any() else 0.0,
        "first_bad": (np.argwhere(bad)[0].tolist() if bad.any() else None),
    }


__all__ = [
    "build", "default_threads", "f16_to_f64", "f64_to_f16",
    "gemm_s32_nn", "gemm_f16_nt_f64", "gemm_f16_nt_entries", "gemm_s32_nn_entries",
    "f16_ulp", "f16_tolerance", "check_f16",
]
