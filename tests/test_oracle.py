"""Pins for the CPU oracle (no GPU): each checks the oracle against something
other than itself -- the IEEE 754 binary16 definition, numpy's binary16
conversion, exact rational or big-integer arithmetic, closed forms of special
inputs, and invariants of the product."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from pipelined_warp_specialized_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _safe_eval(expr: str) -> float:
    allowed = set("0123456789.+-*/() e")
    if not set(expr) <= allowed:
        raise ValueError(expr)
    return float(eval(expr, {"__builtins__": {}}, {}))  # noqa: S307 -- digits and operators only


# ---------------------------------------------------------------- binary16 codec

def test_f16_decode_all_patterns_match_numpy(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signs of zeros too
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_f16_encode_round_trips_every_finite_value(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(vals)
    back = oracle_mod.f64_to_f16(vals[finite])
    assert np.array_equal(back, bits[finite])


def test_f16_encode_golden_fixture(oracle_mod):
    rows = []
    with open(os.path.join(GOLDEN, "f16_rounding.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            expr, hexbits, _why = [p.strip() for p in line.split("|")]
            rows.append((_safe_eval(expr), int(hexbits, 16), expr))
    assert len(rows) >= 20
    x = np.array([r[0] for r in rows])
    got = oracle_mod.f64_to_f16(x)
    for (val, want, expr), g in zip(rows, got):
        assert int(g) == want, f"{expr}: got {int(g):04x}, want {want:04x}"


def test_f16_encode_ties_go_to_even(oracle_mod):
    # every midpoint between adjacent positive finite binary16 values
    bits = np.arange(0, 0x7BFF, dtype=np.uint16)
    lo = bits.view(np.float16).astype(np.float64)
    hi = (bits + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2.0                      # exact in binary64
    got = oracle_mod.f64_to_f16(mid)
    want = np.where(bits % 2 == 0, bits, bits + 1).astype(np.uint16)
    assert np.array_equal(got, want)
    assert np.array_equal(oracle_mod.f64_to_f16(-mid), want | np.uint16(0x8000))


def test_f16_encode_matches_numpy_on_random_doubles(oracle_mod):
    rng = np.random.default_rng(12345)
    mags = np.ldexp(rng.random(400_000) + 0.5, rng.integers(-30, 18, 400_000))
    x = mags * rng.choice([-1.0, 1.0], 400_000)
    ours = oracle_mod.f64_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------- s32 product

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 7, 3), (5, 1, 6), (3, 4, 5), (7, 7, 7), (2, 3, 0)])
def test_s32_brute_force_big_ints(oracle_mod, M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    A = rng.integers(-2**31, 2**31, (M, K), dtype=np.int64).astype(np.int32)
    B = rng.integers(-2**31, 2**31, (K, N), dtype=np.int64).astype(np.int32)
    got = oracle_mod.gemm_s32_nn(A, B)
    for m in range(M):
        for n in range(N):
            s = sum(int(A[m, k]) * int(B[k, n]) for k in range(K))
            w = ((s + 2**31) % 2**32) - 2**31          # two's complement wrap
            assert int(got[m, n]) == w


def test_s32_closed_forms(oracle_mod):
    M, N, K = 9, 11, 13
    ones_a = np.ones((M, K), np.int32)
    ones_b = np.ones((K, N), np.int32)
    assert np.all(oracle_mod.gemm_s32_nn(ones_a, ones_b) == K)
    B = inputs.ints(7, 1, (K, N))
    eye = np.eye(K, dtype=np.int32)
    assert np.array_equal(oracle_mod.gemm_s32_nn(eye, B), B)
    # rank one: lhs[m,k] = a_m, rhs[k,n] = b_n  ->  K * a_m * b_n
    a = np.arange(-4, 5, dtype=np.int32)
    b = np.arange(-5, 6, dtype=np.int32)
    lhs = np.repeat(a[:, None], K, axis=1)
    rhs = np.repeat(b[None, :], K, axis=0)
    assert np.array_equal(oracle_mod.gemm_s32_nn(lhs, rhs), K * np.outer(a, b))


def test_s32_forced_overflow_wraps(oracle_mod):
    K = 8
    lhs = np.full((2, K), 2**31 - 1, np.int32)
    rhs = np.full((K, 3), 2**31 - 1, np.int32)
    exact = K * (2**31 - 1) ** 2
    want = ((exact + 2**31) % 2**32) - 2**31
    assert np.all(oracle_mod.gemm_s32_nn(lhs, rhs) == want)
    lhs[1] = -2**31
    exact2 = K * (-2**31) * (2**31 - 1)
    want2 = ((exact2 + 2**31) % 2**32) - 2**31
    assert np.all(oracle_mod.gemm_s32_nn(lhs, rhs)[1] == want2)


def test_s32_entries_match_full(oracle_mod):
    A = inputs.ints(3, 0, (37, 29))
    B = inputs.ints(3, 1, (29, 41))
    full = oracle_mod.gemm_s32_nn(A, B)
    rows = np.array([0, 36, 5, 17, 36])
    cols = np.array([0, 40, 33, 2, 0])
    assert np.array_equal(oracle_mod.gemm_s32_nn_entries(A, B, rows, cols), full[rows, cols])


def test_s32_page_geometry(oracle_mod):
    # lhs [128,256] x rhs [256,256] -> out [128,256]; |sum| <= 256 * 8 * 8
    wl = inputs.WORKLOADS["s32_nn_128x256x256"]
    A, B = wl.lhs(), wl.rhs()
    assert A.shape == (128, 256) and B.shape == (256, 256)
    assert A.min() >= -8 and A.max() <= 8
    out = oracle_mod.gemm_s32_nn(A, B)
    assert out.shape == (128, 256)
    assert np.abs(out).max() <= 256 * 64
    ref = (A.astype(np.int64) @ B.astype(np.int64))       # no wrap possible at this size
    assert np.array_equal(out, ref.astype(np.int32))


# ---------------------------------------------------------------- f16 product

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 5), (4, 1, 9), (3, 3, 17), (5, 6, 0)])
def test_f16_nt_within_exact_rational_bound(oracle_mod, M, N, K):
    A = inputs.normal_f16(M * 7 + K, 0, (M, K))
    B = inputs.normal_f16(N * 11 + K, 1, (N, K))
    got = oracle_mod.gemm_f16_nt_f64(A, B)
    Af = [[Fraction(float(v)) for v in row] for row in A.astype(np.float64)]
    Bf = [[Fraction(float(v)) for v in row] for row in B.astype(np.float64)]
    for m in range(M):
        for n in range(N):
            exact = sum((Af[m][k] * Bf[n][k] for k in range(K)), Fraction(0))
            abs_sum = sum((abs(Af[m][k] * Bf[n][k]) for k in range(K)), Fraction(0))
            # a K-term binary64 sum of exact products errs by at most K * 2^-53 * sum|terms|
            bound = Fraction(K) * Fraction(1, 2**53) * abs_sum
            assert abs(Fraction(float(got[m, n])) - exact) <= bound


def test_f16_nt_permutation_is_exact(oracle_mod):
    # lhs a permutation matrix P (M x K):  (P . B^T)[m, n] = B[n, perm[m]]
    K = 19
    perm = np.array([3, 0, 18, 7, 7, 11])                    # rows may repeat
    P = np.zeros((len(perm), K), np.float16)
    P[np.arange(len(perm)), perm] = 1.0
    B = inputs.uniform_f16(9, 1, (13, K))
    got = oracle_mod.gemm_f16_nt_f64(P, B)
    assert np.array_equal(got, B[:, perm].T.astype(np.float64))


def test_f16_nt_rank_one_dyadic_closed_form(oracle_mod):
    K = 64
    a = np.array([1.0, -1.0, 0.5, -0.5], np.float16)
    b = np.array([0.5, 1.0, -1.0, -0.5, 1.0], np.float16)
    A = np.repeat(a[:, None], K, axis=1)
    B = np.repeat(b[:, None], K, axis=1)
    got = oracle_mod.gemm_f16_nt_f64(A, B)
    want = K * np.outer(a.astype(np.float64), b.astype(np.float64))
    assert np.array_equal(got, want)


def test_f16_nt_is_a_times_b_transposed(oracle_mod):
    # a distinct-value test that a transposed operand or swapped index would fail
    A = np.array([[1, 2, 3], [4, 5, 6]], np.float16)           # M=2, K=3
    B = np.array([[1, 0, 0], [0, 1, 0], [1, 1, 1], [2, 0, -1]], np.float16)  # N=4, K=3
    want = np.array([[1, 2, 6, -1], [4, 5, 15, 2]], np.float64)
    assert np.array_equal(oracle_mod.gemm_f16_nt_f64(A, B), want)


def test_f16_nt_zero_padding_of_k_is_invariant(oracle_mod):
    A = inputs.uniform_f16(21, 0, (6, 45))
    B = inputs.uniform_f16(21, 1, (5, 45))
    Ap = np.concatenate([A, np.zeros((6, 19), np.float16)], axis=1)
    Bp = np.concatenate([B, np.zeros((5, 19), np.float16)], axis=1)
    assert np.array_equal(oracle_mod.gemm_f16_nt_f64(A, B), oracle_mod.gemm_f16_nt_f64(Ap, Bp))


def test_f16_nt_entries_match_full(oracle_mod):
    A = inputs.normal_f16(5, 0, (33, 70))
    B = inputs.normal_f16(5, 1, (21, 70))
    full = oracle_mod.gemm_f16_nt_f64(A, B)
    rows = np.array([0, 32, 11, 5])
    cols = np.array([20, 0, 13, 5])
    assert np.array_equal(oracle_mod.gemm_f16_nt_entries(A, B, rows, cols), full[rows, cols])


def test_f16_nt_thread_count_does_not_change_results(oracle_mod):
    A = inputs.uniform_f16(8, 0, (50, 300))
    B = inputs.uniform_f16(8, 1, (40, 300))
    one = oracle_mod.gemm_f16_nt_f64(A, B, nthreads=1)
    many = oracle_mod.gemm_f16_nt_f64(A, B, nthreads=7)
    assert np.array_equal(one, many)


# ---------------------------------------------------------------- acceptance rule

def test_f16_ulp_is_the_binary16_spacing(oracle_mod):
    # ulp16(x) must equal the gap from |x|'s binary16 value to its successor,
    # read from numpy's binary16 arithmetic, for x inside each binade.
    pos = np.arange(1, 0x7BFF, 37, dtype=np.uint16).view(np.float16)
    nxt = np.nextafter(pos, np.float16(np.inf))
    gap = nxt.astype(np.float64) - pos.astype(np.float64)
    assert np.array_equal(oracle_mod.f16_ulp(pos.astype(np.float64)), gap)
    assert oracle_mod.f16_ulp(np.array([0.0]))[0] == 2.0 ** -24
    assert oracle_mod.f16_ulp(np.array([1.0]))[0] == 2.0 ** -10
    assert oracle_mod.f16_ulp(np.array([-0.75]))[0] == 2.0 ** -11
    assert oracle_mod.f16_ulp(np.array([65504.0]))[0] == 32.0


def test_check_f16_accepts_rounded_and_rejects_planted_error(oracle_mod):
    K = 256
    A = inputs.uniform_f16(4, 0, (16, K))
    B = inputs.uniform_f16(4, 1, (24, K))
    ref = oracle_mod.gemm_f16_nt_f64(A, B)
    gpu_like = oracle_mod.f64_to_f16(ref)
    assert oracle_mod.check_f16(gpu_like, ref, K)["ok"]
    bad = gpu_like.copy()
    tol = oracle_mod.f16_tolerance(ref[3, 5], K)
    bad[3, 5] = oracle_mod.f64_to_f16(np.array([ref[3, 5] + 3 * tol]))[0]
    res = oracle_mod.check_f16(bad, ref, K)
    assert not res["ok"] and res["n_bad"] == 1 and res["first_bad"] == [3, 5]


def test_k_tolerance_term(oracle_mod):
    t = oracle_mod.f16_tolerance(np.array([1.0]), 8192)[0]
    assert math.isclose(t, 2.0 ** -10 + 1e-3 * math.sqrt(8192))


# ---------------------------------------------------------------- generator recipe

def test_generator_reference_values():
    # splitmix64 finaliser applied to 0x9E3779B97F4A7C15 (seed 0 key, first draw of a
    # classic splitmix64 stream starting from 0) is 0xE220A8397B1DCDAF.
    from pipelined_warp_specialized_gb300.inputs import _mix
    z = _mix(np.array([0x9E3779B97F4A7C15], dtype=np.uint64))[0]
    assert int(z) == 0xE220A8397B1DCDAF
    x = inputs.ints(1, 0, (4096,))
    assert x.min() == -8 and x.max() == 8 and len(np.unique(x)) == 17
    u = inputs.uniform_f16(2, 0, (100000,)).astype(np.float64)
    assert -1.0 <= u.min() and u.max() <= 1.0 and abs(u.mean()) < 0.01
    z = inputs.normal_f16(4, 0, (200000,)).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    # determinism and stream independence
    assert np.array_equal(inputs.uniform_f16(3, 0, (1000,)), inputs.uniform_f16(3, 0, (1000,)))
    assert not np.array_equal(inputs.uniform_f16(3, 0, (1000,)), inputs.uniform_f16(3, 1, (1000,)))
