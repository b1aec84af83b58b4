"""Python binding of the pipelined, warp-specialized GEMM library (sm_103a).

Argument marshalling only: every function here forwards to the entry point of
the same name in the C ABI (``include/pwsgemm.h``), implemented by the CUDA
library ``_build/libpwsgemm.so``.  PyTorch supplies device memory and streams.
There is no fallback: if the library is missing or fails to load, every call
raises.

    import torch, pipelined_warp_specialized_gb300 as pws
    a = torch.randn(4096, 4096, device="cuda", dtype=torch.float16)   # lhs [M, K]
    b = torch.randn(4096, 4096, device="cuda", dtype=torch.float16)   # rhs [N, K]
    c = pws.gemm_f16_nt(a, b, stages=4)                               # a @ b.T, f16
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpwsgemm.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "pwsgemm.h")

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_ALIGNMENT = 2
GEMM_ERR_UNSUPPORTED_STAGES = 3
GEMM_ERR_UNSUPPORTED_ARCH = 4
GEMM_ERR_LAUNCH = 5
GEMM_ERR_TIMEOUT = 6

GEMM_DEBUG_SKIP_EMPTY_SEED = 1
GEMM_DEBUG_FORCE_COPY_PRODUCER = 2
GEMM_DEBUG_FORCE_DIRECT_STORE = 4
GEMM_DEBUG_FORCE_SOLO_TILE = 8
GEMM_DEBUG_FORCE_PAIR_TILE = 16
GEMM_DEBUG_NO_SPLIT = 32
GEMM_DEBUG_FORCE_NARROW_TILE = 64
GEMM_DEBUG_FORCE_WIDE_TILE = 128
GEMM_DEBUG_SKIP_ACC_SEED = 256
GEMM_DEBUG_NO_KSPLIT = 512
GEMM_DEBUG_FORCE_KSPLIT = 1024
GEMM_DEBUG_SKIP_KSPLIT_SEND = 2048
GEMM_DEBUG_FORCE_DOUBLE_SLOT = 4096
GEMM_DEBUG_NO_DOUBLE_SLOT = 8192
GEMM_DEBUG_IN_PLACE = 16384

_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Loads the CUDA library (building nothing); raises if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"the CUDA library {p} is not built; run "
                          "`python -m pipelined_warp_specialized_gb300.build`")
    lib = ctypes.CDLL(p)
    i64, i32, vp, u32, u64 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_uint, ctypes.c_uint64
    lib.gemm_s32_nn.argtypes = [i64, i64, i64, vp, vp, vp, vp]
    lib.gemm_s32_nn.restype = i32
    lib.gemm_s32_nn_ring.argtypes = [i64, i64, i64, vp, vp, vp, i32, vp]
    lib.gemm_s32_nn_ring.restype = i32
    lib.gemm_f16_nt.argtypes = [i64, i64, i64, vp, vp, vp, i32, vp]
    lib.gemm_f16_nt.restype = i32
    lib.gemm_f16_nt_noalloc.argtypes = [i64, i64, i64, vp, vp, vp, i32, vp]
    lib.gemm_f16_nt_noalloc.restype = i32
    lib.gemm_device_status.argtypes = [vp]
    lib.gemm_device_status.restype = i32
    lib.gemm_status_string.argtypes = [i32]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_set_wait_timeout_ns.argtypes = [u64]
    lib.gemm_set_wait_timeout_ns.restype = i32
    lib.gemm_set_debug_flags.argtypes = [u32]
    lib.gemm_set_debug_flags.restype = i32
    lib.gemm_set_scratch_pool.argtypes = [i32]
    lib.gemm_set_scratch_pool.restype = i32
    lib.gemm_f16_nt_plan.argtypes = [i64, i64, i64, vp, vp, vp, i32, ctypes.POINTER(i64)]
    lib.gemm_f16_nt_plan.restype = i32
    if path is None:
        _lib = lib
    return lib


def header_functions(header: str = HEADER) -> list:
    """Names of the functions ``include/pwsgemm.h`` declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:int|const char\s*\*)\s*(\w+)\s*\(", text, flags=re.M)


def status_string(status: int) -> str:
    try:
        return load_library().gemm_status_string(int(status)).decode()
    except ImportError:
        return f"status {status}"


def _stream_ptr(stream, device) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, what: str) -> None:
    if status != GEMM_OK:
        raise GemmError(status, what)


def _same_device(name, lhs, rhs, out):
    """Every operand must live on lhs's device: the call launches there, and a
    pointer into another GPU's memory is not valid on it."""
    devs = {t.device for t in (lhs, rhs, out) if t is not None}
    if len(devs) > 1:
        raise ValueError(f"{name}: lhs, rhs and out must be on one device, got {sorted(map(str, devs))}")


def gemm_s32_nn(lhs, rhs, out=None, stream=None):
    """out[M,N] = lhs[M,K] @ rhs[K,N] over int32 (wrapping), on lhs's device."""
    import torch
    if lhs.dtype != torch.int32 or rhs.dtype != torch.int32:
        raise TypeError("gemm_s32_nn takes int32 tensors")
    if lhs.dim() != 2 or rhs.dim() != 2 or lhs.shape[1] != rhs.shape[0]:
        raise ValueError(f"shapes {tuple(lhs.shape)} x {tuple(rhs.shape)} do not form [M,K] x [K,N]")
    if not (lhs.is_cuda and rhs.is_cuda) or not lhs.is_contiguous() or not rhs.is_contiguous():
        raise ValueError("gemm_s32_nn takes contiguous CUDA tensors")
    _same_device("gemm_s32_nn", lhs, rhs, out)
    M, K = lhs.shape
    N = rhs.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.int32, device=lhs.device)
    elif out.shape != (M, N) or out.dtype != torch.int32 or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous int32 CUDA tensor of shape [M, N]")
    with torch.cuda.device(lhs.device):
        _check(load_library().gemm_s32_nn(M, N, K, lhs.data_ptr(), rhs.data_ptr(), out.data_ptr(),
                                          _stream_ptr(stream, lhs.device)), "gemm_s32_nn")
    return out


def gemm_s32_nn_ring(lhs, rhs, out=None, stages: int = 4, stream=None):
    """gemm_s32_nn with an S-slot ring (S = `stages`, 2..6); bit-identical results."""
    import torch
    if lhs.dtype != torch.int32 or rhs.dtype != torch.int32:
        raise TypeError("gemm_s32_nn_ring takes int32 tensors")
    if lhs.dim() != 2 or rhs.dim() != 2 or lhs.shape[1] != rhs.shape[0]:
        raise ValueError(f"shapes {tuple(lhs.shape)} x {tuple(rhs.shape)} do not form [M,K] x [K,N]")
    if not (lhs.is_cuda and rhs.is_cuda) or not lhs.is_contiguous() or not rhs.is_contiguous():
        raise ValueError("gemm_s32_nn_ring takes contiguous CUDA tensors")
    _same_device("gemm_s32_nn_ring", lhs, rhs, out)
    M, K = lhs.shape
    N = rhs.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.int32, device=lhs.device)
    elif out.shape != (M, N) or out.dtype != torch.int32 or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous int32 CUDA tensor of shape [M, N]")
    with torch.cuda.device(lhs.device):
        _check(load_library().gemm_s32_nn_ring(M, N, K, lhs.data_ptr(), rhs.data_ptr(), out.data_ptr(), int(stages),
                                               _stream_ptr(stream, lhs.device)), "gemm_s32_nn_ring")
    return out


def gemm_f16_nt(lhs, rhs, out=None, stages: int = 4, stream=None):
    """out[M,N] = f16(lhs[M,K] @ rhs[N,K].T) with fp32 accumulation, S = `stages` ring slots."""
    import torch
    if lhs.dtype != torch.float16 or rhs.dtype != torch.float16:
        raise TypeError("gemm_f16_nt takes float16 tensors")
    if lhs.dim() != 2 or rhs.dim() != 2 or lhs.shape[1] != rhs.shape[1]:
        raise ValueError(f"shapes {tuple(lhs.shape)} x {tuple(rhs.shape)} do not form [M,K] x [N,K]")
    if not (lhs.is_cuda and rhs.is_cuda) or not lhs.is_contiguous() or not rhs.is_contiguous():
        raise ValueError("gemm_f16_nt takes contiguous CUDA tensors")
    _same_device("gemm_f16_nt", lhs, rhs, out)
    M, K = lhs.shape
    N = rhs.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=lhs.device)
    elif out.shape != (M, N) or out.dtype != torch.float16 or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous float16 CUDA tensor of shape [M, N]")
    with torch.cuda.device(lhs.device):
        _check(load_library().gemm_f16_nt(M, N, K, lhs.data_ptr(), rhs.data_ptr(), out.data_ptr(), int(stages),
                                          _stream_ptr(stream, lhs.device)), "gemm_f16_nt")
    return out


def gemm_f16_nt_noalloc(lhs, rhs, out=None, stages: int = 4, stream=None):
    """gemm_f16_nt for callers that cannot allocate device memory.

    Where gemm_f16_nt would take scratch from its pool, this uses a fixed
    32 MiB device array loaded with the library, so no allocator is entered
    (for code under a fixed memory budget or that must not allocate).  Calls
    share that array: calls that can overlap on the GPU must be ordered.
    Raises GemmError(GEMM_ERR_INVALID_ARG) when more scratch would be needed.
    ``out`` should be preallocated by such callers (None allocates it here).
    """
    import torch
    if lhs.dtype != torch.float16 or rhs.dtype != torch.float16:
        raise TypeError("gemm_f16_nt_noalloc takes float16 tensors")
    if lhs.dim() != 2 or rhs.dim() != 2 or lhs.shape[1] != rhs.shape[1]:
        raise ValueError(f"shapes {tuple(lhs.shape)} x {tuple(rhs.shape)} do not form [M,K] x [N,K]")
    if not (lhs.is_cuda and rhs.is_cuda) or not lhs.is_contiguous() or not rhs.is_contiguous():
        raise ValueError("gemm_f16_nt_noalloc takes contiguous CUDA tensors")
    _same_device("gemm_f16_nt_noalloc", lhs, rhs, out)
    M, K = lhs.shape
    N = rhs.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=lhs.device)
    elif out.shape != (M, N) or out.dtype != torch.float16 or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous float16 CUDA tensor of shape [M, N]")
    with torch.cuda.device(lhs.device):
        _check(load_library().gemm_f16_nt_noalloc(M, N, K, lhs.data_ptr(), rhs.data_ptr(), out.data_ptr(),
                                                  int(stages), _stream_ptr(stream, lhs.device)),
               "gemm_f16_nt_noalloc")
    return out


def gemm_device_status(stream=None) -> int:
    """Synchronizes the stream; returns and clears the device status word."""
    return load_library().gemm_device_status(_stream_ptr(stream, None))


def gemm_status_string(status: int) -> str:
    return status_string(status)


def gemm_set_wait_timeout_ns(ns: int) -> None:
    _check(load_library().gemm_set_wait_timeout_ns(int(ns)), "gemm_set_wait_timeout_ns")


def gemm_set_debug_flags(flags: int) -> None:
    _check(load_library().gemm_set_debug_flags(int(flags)), "gemm_set_debug_flags")


def gemm_set_scratch_pool(enable: bool) -> None:
    """Lets later gemm_f16_nt calls copy operands TMA cannot address to pooled
    scratch (faster for large ones; allocates stream-ordered).  Off by default."""
    _check(load_library().gemm_set_scratch_pool(int(bool(enable))), "gemm_set_scratch_pool")


def gemm_f16_nt_plan(M: int, N: int, K: int, lhs_ptr: int = 1 << 40, rhs_ptr: int = 2 << 40,
                     out_ptr: int = 3 << 40, stages: int = 4) -> dict:
    """The launch plan gemm_f16_nt would use (host logic only; the pointers are
    only inspected for alignment and overlap, never dereferenced)."""
    plan = (ctypes.c_int64 * 11)()
    _check(load_library().gemm_f16_nt_plan(M, N, K, lhs_ptr, rhs_ptr, out_ptr, stages, plan), "gemm_f16_nt_plan")
    keys = ["bm", "bn", "bk", "cta_group", "producer", "copy_bytes", "store", "smem_bytes", "tiles", "k_blocks",
            "k_split"]
    return dict(zip(keys, list(plan)))


__all__ = [
    "GemmError", "load_library", "header_functions", "gemm_s32_nn", "gemm_f16_nt", "gemm_device_status",
    "gemm_status_string", "gemm_set_wait_timeout_ns", "gemm_set_debug_flags", "gemm_set_scratch_pool",
    "gemm_f16_nt_plan", "gemm_f16_nt_noalloc", "gemm_s32_nn_ring",
]
