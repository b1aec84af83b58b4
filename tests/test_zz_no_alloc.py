"""gemm_f16_nt_noalloc, the entry point for callers that cannot allocate
device memory (a fixed memory budget, memory reserved up front, or code that
must not enter an allocator).  It runs the same GEMM as gemm_f16_nt but takes
the scratch of the repack step from a fixed device array loaded with the
library instead of a memory pool.

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
    a = torch.from_numpy(inputs.normal_f16(seed, 0, (M, K))).cuda()
    b = torch.from_numpy(inputs.normal_f16(seed, 1, (N, K))).cuda()
    return a, b


def test_noalloc_matches_gemm_f16_nt_on_two_calls_in_a_row():
    # K = 1030: rows of 2060 bytes, so the GEMM needs the repack scratch
    # (1700 rows x 1032 x 2 bytes, well under the 32 MiB array)
    M, N, K = 1000, 700, 1030
    assert pws.gemm_f16_nt_plan(M, N, K)["producer"] == 2
    for seed in (71, 72):                       # two calls in a row share the array
        a, b = _pair(seed, M, N, K)
        want = pws.gemm_f16_nt(a, b, stages=3)
        got = pws.gemm_f16_nt_noalloc(a, b, stages=3)
        torch.cuda.synchronize()
        assert pws.gemm_device_status() == pws.GEMM_OK
        want_np = want.cpu().numpy()
        res = oracle.check_f16(got.cpu().numpy(), oracle.f16_to_f64(want_np), K)
        assert res["ok"], res


def test_noalloc_without_scratch_and_over_the_limit():
    # operands the accelerator addresses directly need no scratch
    a, b = _pair(73, 300, 260, 256)
    want = pws.gemm_f16_nt(a, b, stages=2)
    got = pws.gemm_f16_nt_noalloc(a, b, stages=2)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().view(np.uint16), want.cpu().numpy().view(np.uint16))
    # 16384 rows of 2056 elements need 64 MiB of scratch: refused before any launch
    big_a = torch.empty(8192, 2050, dtype=torch.float16, device="cuda")
    big_b = torch.empty(8192, 2050, dtype=torch.float16, device="cuda")
    out = torch.empty(8192, 8192, dtype=torch.float16, device="cuda")
    with pytest.raises(pws.GemmError) as e:
        pws.gemm_f16_nt_noalloc(big_a, big_b, out, stages=3)
    assert e.value.status == pws.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert pws.gemm_device_status() == pws.GEMM_OK
