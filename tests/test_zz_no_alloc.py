"""gemm_f16_nt_noalloc, the entry point for callers that cannot allocate
device memory (a fixed memory budget, memory reserved up front, or code that
must not enter an allocator).  It runs the same GEMM as gemm_f16_nt and
repacks operands TMA cannot address into the library's fixed device array,
whatever the scratch-pool setting; operands that would need more than the
array holds are read in place.  Results are checked against the oracle and
must equal gemm_f16_nt's bit for bit.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process (the
fixture builds and loads what it needs).
"""
import numpy as np
import pytest

import oracle
import pipelined_warp_specialized_gb300 as pws
from pipelined_warp_specialized_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from pipelined_warp_specialized_gb300 import build as libbuild
    libbuild.build()
    oracle.build()
    pws.load_library()
    pws.gemm_set_debug_flags(0)


def _pair(seed, M, N, K):
    a = inputs.normal_f16(seed, 0, (M, K))
    b = inputs.normal_f16(seed, 1, (N, K))
    return a, b


def _bits(t):
    return t.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("M,N,K,S,want", [
    # K = 1030: rows of 2060 bytes, which no tensor map describes: this call
    # repacks them into the array (1700 rows x 1032 x 2 bytes, well under
    # its 32 MiB), as gemm_f16_nt does (in 128-byte rows)
    (1000, 700, 1030, 3, {}),
    # the ragged workload: 7000 rows of 2056 elements, 28.7 MB of the array
    (4000, 3000, 2050, 3, {}),
    # 9 single-CTA tiles of 33 K blocks: the K split on repacked operands
    (300, 260, 2050, 2, {"k_split": 2}),
], ids=["1000x700x1030", "ragged_4000x3000x2050", "k_split_300x260x2050"])
def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(M, N, K, S, want):
    plan = pws.gemm_f16_nt_plan(M, N, K, stages=S)
    assert plan["producer"] == 2 and {k: plan[k] for k in want} == want, plan
    for seed in (71, 72):                       # two calls in a row share the array
        a_np, b_np = _pair(seed, M, N, K)
        a, b = torch.from_numpy(a_np).cuda(), torch.from_numpy(b_np).cuda()
        got = pws.gemm_f16_nt_noalloc(a, b, stages=S)
        torch.cuda.synchronize()
        assert pws.gemm_device_status() == pws.GEMM_OK
        res = oracle.check_f16(got.cpu().numpy(), oracle.gemm_f16_nt_f64(a_np, b_np), K)
        assert res["ok"], res
        # both entry points run the same sums in the same order
        want_out = pws.gemm_f16_nt(a, b, stages=S)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(got), _bits(want_out))


def test_noalloc_without_scratch_and_over_the_limit():
    # operands the accelerator addresses directly need no scratch
    a_np, b_np = _pair(73, 300, 260, 256)
    a, b = torch.from_numpy(a_np).cuda(), torch.from_numpy(b_np).cuda()
    want = pws.gemm_f16_nt(a, b, stages=2)
    got = pws.gemm_f16_nt_noalloc(a, b, stages=2)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(got), _bits(want))
    # 512 rows of 65544 elements would need 64 MiB of scratch, more than the
    # array holds: the operands are read in place instead, with the same result
    M, N, K = 256, 256, 65538
    a_np, b_np = _pair(74, M, N, K)
    a, b = torch.from_numpy(a_np).cuda(), torch.from_numpy(b_np).cuda()
    out = torch.empty(M, N, dtype=torch.float16, device="cuda")
    for _ in range(2):
        out.fill_(0)
        pws.gemm_f16_nt_noalloc(a, b, out, stages=3)
        torch.cuda.synchronize()
        assert pws.gemm_device_status() == pws.GEMM_OK
        res = oracle.check_f16(out.cpu().numpy(), oracle.gemm_f16_nt_f64(a_np, b_np), K)
        assert res["ok"], res
