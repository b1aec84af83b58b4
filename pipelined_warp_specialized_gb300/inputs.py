"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle's callers.

This module holds only the random-number recipe; it performs none of the
GEMM's arithmetic and imports neither the CUDA library nor the oracle.

Generator: splitmix64 used as a counter-based generator.  For stream ``j`` of
seed ``s`` the key is ``mix(s ^ (j * 0xD1B54A32D192ED03))`` and draw ``i`` is
``mix(key + (i + 1) * 0x9E3779B97F4A7C15)`` (all arithmetic modulo 2^64), where
``mix`` is the splitmix64 finaliser (xor-shift 30, multiply 0xBF58476D1CE4E5B9,
xor-shift 27, multiply 0x94D049BB133111EB, xor-shift 31).  A unit uniform is
``(draw >> 11) * 2^-53`` in [0, 1).

Value recipes (the pages fix none of them; these are the readings used):

* ``ints(lo, hi)``: ``lo + floor(u * (hi - lo + 1))`` -- both ends inclusive
  (17 values for [-8, 8]).
* ``uniform_f16(lo, hi)``: ``lo + (hi - lo) * u`` in binary64, rounded to
  binary16 (nearest, ties to even) by numpy's float64 -> float16 cast.
* ``normal_f16``: Box-Muller in binary64 on draws ``(2i, 2i+1)``:
  ``sqrt(-2 ln(1 - u1)) * cos(2 pi u2)``, then rounded to binary16.

``lhs`` uses stream 0 and ``rhs`` stream 1 of a configuration's seed.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_STREAM = 0xD1B54A32D192ED03
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def splitmix64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Draws ``offset .. offset+n-1`` of stream ``stream`` of ``seed`` (uint64)."""
    key_in = (int(seed) ^ ((int(stream) * _STREAM) & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
    key = _mix(np.array([key_in], dtype=np.uint64))[0]
    out = np.empty(n, dtype=np.uint64)
    chunk = 1 << 24
    with np.errstate(over="ignore"):
        for start in range(0, n, chunk):
            stop = min(n, start + chunk)
            ctr = np.arange(offset + start + 1, offset + stop + 1, dtype=np.uint64)
            out[start:stop] = _mix(key + ctr * _GAMMA)
    return out


def unit_uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """Uniform float64 draws in [0, 1)."""
    return (splitmix64(seed, stream, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def ints(seed: int, stream: int, shape, lo: int = -8, hi: int = 8) -> np.ndarray:
    n = int(np.prod(shape))
    u = unit_uniform(seed, stream, n)
    v = lo + np.floor(u * (hi - lo + 1)).astype(np.int64)
    return v.astype(np.int32).reshape(shape)


def uniform_f16(seed: int, stream: int, shape, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float16)
    chunk = 1 << 24
    for start in range(0, n, chunk):
        stop = min(n, start + chunk)
        u = (splitmix64(seed, stream, stop - start, offset=start) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        out[start:stop] = (lo + (hi - lo) * u).astype(np.float16)
    return out.reshape(shape)


def normal_f16(seed: int, stream: int, shape) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float16)
    chunk = 1 << 23
    for start in range(0, n, chunk):
        stop = min(n, start + chunk)
        d = splitmix64(seed, stream, 2 * (stop - start), offset=2 * start)
        u = (d >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        u1, u2 = u[0::2], u[1::2]
        z = np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)
        out[start:stop] = z.astype(np.float16)
    return out.reshape(shape)


@dataclass(frozen=True)
class Workload:
    """One seeded synthetic workload of the library."""
    name: str
    kind: str            # "s32_nn" or "f16_nt"
    M: int
    N: int
    K: int
    seed: int
    dist: str            # "ints", "uniform", "normal"
    stages: tuple        # stage counts the workload is run with

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def lhs(self) -> np.ndarray:
        if self.kind == "s32_nn":
            return ints(self.seed, 0, (self.M, self.K))
        return _f16(self.dist, self.seed, 0, (self.M, self.K))

    def lhs_rows(self, rows: int) -> np.ndarray:
        """The first `rows` rows of lhs() (the generator is counter-based in
        row-major element order, so they need not generate the rest)."""
        if self.kind == "s32_nn":
            return ints(self.seed, 0, (rows, self.K))
        return _f16(self.dist, self.seed, 0, (rows, self.K))

    def rhs(self) -> np.ndarray:
        if self.kind == "s32_nn":
            return ints(self.seed, 1, (self.K, self.N))
        return _f16(self.dist, self.seed, 1, (self.N, self.K))


def _f16(dist: str, seed: int, stream: int, shape) -> np.ndarray:
    if dist == "uniform":
        return uniform_f16(seed, stream, shape)
    if dist == "normal":
        return normal_f16(seed, stream, shape)
    raise ValueError(dist)


# The five workloads: shapes, value distributions and stage counts as the
# library's specification names them; seeds 1..5 in order.
WORKLOADS = {
    "s32_nn_128x256x256": Workload("s32_nn_128x256x256", "s32_nn", 128, 256, 256, 1, "ints", (2,)),
    "f16_nt_1024": Workload("f16_nt_1024", "f16_nt", 1024, 1024, 1024, 2, "uniform", (2,)),
    "f16_nt_4096": Workload("f16_nt_4096", "f16_nt", 4096, 4096, 4096, 3, "uniform", (4,)),
    "f16_nt_ragged_4000x3000x2050": Workload("f16_nt_ragged_4000x3000x2050", "f16_nt", 4000, 3000, 2050, 4,
                                             "normal", (3,)),
    "f16_nt_8192": Workload("f16_nt_8192", "f16_nt", 8192, 8192, 8192, 5, "uniform", (1, 2, 3, 4, 5, 6)),
}
