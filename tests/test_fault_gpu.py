"""The bounded device waits: skipping the empty-credit seed (the deadlock the
Croqtile tutorial ch.6 describes in "消费者路径") must end in GEMM_ERR_TIMEOUT
from the status word, with the kernel returning on its own and the context
still usable.  Nothing here faults, traps or hangs the GPU: every wait in the
kernels gives up after the limit set below, and the roles drain and return."""
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
    pws.load_library()
    yield
    pws.gemm_set_debug_flags(0)
    pws.gemm_set_wait_timeout_ns(0)


@pytest.mark.parametrize("seed_flag", [pws.GEMM_DEBUG_SKIP_EMPTY_SEED, pws.GEMM_DEBUG_SKIP_ACC_SEED],
                         ids=["no_empty_seed", "no_acc_seed"])
@pytest.mark.parametrize("extra,N", [
    (0, 256), (pws.GEMM_DEBUG_FORCE_PAIR_TILE, 256), (pws.GEMM_DEBUG_FORCE_COPY_PRODUCER, 256),
    (pws.GEMM_DEBUG_FORCE_PAIR_TILE | pws.GEMM_DEBUG_FORCE_WIDE_TILE, 512),   # split accumulator, 8 epilogue warps
    (pws.GEMM_DEBUG_FORCE_KSPLIT, 256),                 # two CTAs per tile, one K half each
    (pws.GEMM_DEBUG_FORCE_KSPLIT | pws.GEMM_DEBUG_FORCE_COPY_PRODUCER, 256),
], ids=["solo_tma", "pair_tma", "solo_copy", "wide_tma", "ksplit_tma", "ksplit_copy"])
def test_missing_seed_times_out_and_context_survives(seed_flag, extra, N):
    # Without the empty seed the producer's first wait never completes: no
    # copy is ever issued.  Without the accumulator seed the multiply role's
    # first wait never completes while the producer has filled both slots
    # (K = 256 is four K blocks, S = 2): the roles give up with copies
    # issued, and a pair's producers drain them before the CTAs exit.  With the
    # K split, the owner warps' wait for the peer's partial sums gives up too
    # (their own CTA's abort, or the time limit), and every CTA meets its peer
    # at the cluster barrier before exiting.
    M, K = 256, 256
    a_np = inputs.uniform_f16(2, 0, (M, K))
    b_np = inputs.uniform_f16(2, 1, (N, K))
    a = torch.from_numpy(a_np).cuda()
    b = torch.from_numpy(b_np).cuda()
    assert pws.gemm_device_status() == pws.GEMM_OK          # clear anything earlier
    pws.gemm_set_wait_timeout_ns(200_000_000)               # 0.2 s per wait
    pws.gemm_set_debug_flags(seed_flag | extra)
    try:
        pws.gemm_f16_nt(a, b, stages=2)
        torch.cuda.synchronize()                             # the kernel returns by itself
        assert pws.gemm_device_status() == pws.GEMM_ERR_TIMEOUT
        assert pws.gemm_device_status() == pws.GEMM_OK       # the word was cleared
    finally:
        pws.gemm_set_debug_flags(0)
        pws.gemm_set_wait_timeout_ns(0)
    # the context is intact: a normal call still gives the right answer
    out = pws.gemm_f16_nt(a, b, stages=2)
    torch.cuda.synchronize()
    assert pws.gemm_device_status() == pws.GEMM_OK
    res = oracle.check_f16(out.cpu().numpy(), oracle.gemm_f16_nt_f64(a_np, b_np), K)
    assert res["ok"], res
    assert np.isfinite(out.float().cpu().numpy()).all()


@pytest.mark.parametrize("extra", [0, pws.GEMM_DEBUG_FORCE_COPY_PRODUCER], ids=["tma", "copy"])
def test_k_split_missing_partial_sums_time_out(extra):
    # In the K split the owner of each lane quarter waits for its peer CTA's
    # partial sums.  With the senders silenced, that wait alone runs out (0.2
    # s): every other role of both CTAs completes normally, both CTAs meet at
    # the final cluster barrier, the call reports GEMM_ERR_TIMEOUT, and the
    # next call is correct.
    M, N, K = 256, 256, 256
    a_np = inputs.uniform_f16(3, 0, (M, K))
    b_np = inputs.uniform_f16(3, 1, (N, K))
    a = torch.from_numpy(a_np).cuda()
    b = torch.from_numpy(b_np).cuda()
    flags = pws.GEMM_DEBUG_FORCE_KSPLIT | extra
    pws.gemm_set_debug_flags(flags)
    try:
        assert pws.gemm_f16_nt_plan(M, N, K, stages=2)["k_split"] == 2
    finally:
        pws.gemm_set_debug_flags(0)
    assert pws.gemm_device_status() == pws.GEMM_OK
    pws.gemm_set_wait_timeout_ns(200_000_000)
    pws.gemm_set_debug_flags(flags | pws.GEMM_DEBUG_SKIP_KSPLIT_SEND)
    try:
        pws.gemm_f16_nt(a, b, stages=2)
        torch.cuda.synchronize()
        assert pws.gemm_device_status() == pws.GEMM_ERR_TIMEOUT
        assert pws.gemm_device_status() == pws.GEMM_OK
    finally:
        pws.gemm_set_debug_flags(0)
        pws.gemm_set_wait_timeout_ns(0)
    pws.gemm_set_debug_flags(flags)
    try:
        out = pws.gemm_f16_nt(a, b, stages=2)
        torch.cuda.synchronize()
    finally:
        pws.gemm_set_debug_flags(0)
    assert pws.gemm_device_status() == pws.GEMM_OK
    res = oracle.check_f16(out.cpu().numpy(), oracle.gemm_f16_nt_f64(a_np, b_np), K)
    assert res["ok"], res


def _tiled_ternary_f16(seed, stream, rows, K, period=8200):
    # Seeded values in {-1, 0, 1}, a block `period` columns wide repeated
    # along K and cut at K (cheap to generate at K = 2^20).  Every partial sum
    # is then an integer below 2^24, exact in fp32 whatever the summation
    # order, so the GPU result must equal the oracle's exact sum rounded to
    # f16 bit for bit.  period is not a multiple of the 64-column K block, so
    # a K block summed twice or skipped changes the result.
    base = inputs.ints(seed, stream, (rows, period), -1, 1).astype(np.float16)
    reps = -(-K // period)
    return np.ascontiguousarray(np.tile(base, (1, reps))[:, :K])


@pytest.mark.parametrize("M,N,K,flags,want", [
    # one 128 x 128 tile, 16384 K blocks: the K split gives each CTA of the
    # cluster 8192 blocks, and the owners wait for the peer's partial sums
    (128, 128, 1 << 20, 0, {"cta_group": 1, "k_split": 2}),
    # one 256 x 512 wide pair tile, 4096 K blocks: the epilogue's wait for
    # the first half of the accumulator lasts the whole K loop
    (256, 512, 1 << 18, pws.GEMM_DEBUG_FORCE_PAIR_TILE | pws.GEMM_DEBUG_FORCE_WIDE_TILE,
     {"cta_group": 2, "bn": 512}),
], ids=["k_split_owner", "wide_epilogue"])
def test_long_k_loops_outlast_a_short_wait_limit(M, N, K, flags, want):
    # The wait limit bounds stalls, not work.  With a 2 ms limit and one ring
    # slot (S = 1: every K block waits for its copy, then its multiply), these
    # calls' K loops run several times longer than the limit; every wait for
    # the loop's result restarts its clock whenever the producer issues a K
    # block, so the calls complete and match the oracle exactly.
    limit_ms = 2.0
    a_np = _tiled_ternary_f16(21, 0, M, K)
    b_np = _tiled_ternary_f16(21, 1, N, K)
    a = torch.from_numpy(a_np).cuda()
    b = torch.from_numpy(b_np).cuda()
    pws.gemm_set_debug_flags(flags)
    try:
        plan = pws.gemm_f16_nt_plan(M, N, K, stages=1)
        assert {k: plan[k] for k in want} == want, plan
        out = torch.empty(M, N, dtype=torch.float16, device="cuda")
        pws.gemm_f16_nt(a, b, out, stages=1)              # warm: first-call set-up
        torch.cuda.synchronize()
        assert pws.gemm_device_status() == pws.GEMM_OK
        pws.gemm_set_wait_timeout_ns(int(limit_ms * 1e6))
        out.fill_(0)
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        pws.gemm_f16_nt(a, b, out, stages=1)
        stop.record()
        torch.cuda.synchronize()
        elapsed_ms = start.elapsed_time(stop)
        status = pws.gemm_device_status()
    finally:
        pws.gemm_set_debug_flags(0)
        pws.gemm_set_wait_timeout_ns(0)
    assert status == pws.GEMM_OK, (pws.gemm_status_string(status), elapsed_ms)
    # the loop really did outlast the limit, so the test means something
    assert elapsed_ms > limit_ms, elapsed_ms
    ref = oracle.gemm_f16_nt_f64(a_np, b_np)
    got = out.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.f64_to_f16(ref)), int((got != oracle.f64_to_f16(ref)).sum())


def test_timeouts_are_reported_to_their_own_stream():
    # A call that deadlocks (no empty seed, 0.2 s limit) on one stream beside
    # a normal call on another: each stream's status word holds only its own
    # call's outcome, so the normal stream reads GEMM_OK -- even while the
    # other stream's kernel is still waiting out its limit -- and the
    # deadlocked one reads GEMM_ERR_TIMEOUT once, then GEMM_OK.
    M, N, K = 256, 256, 256
    a_np = inputs.uniform_f16(9, 0, (M, K))
    b_np = inputs.uniform_f16(9, 1, (N, K))
    a = torch.from_numpy(a_np).cuda()
    b = torch.from_numpy(b_np).cuda()
    s_bad, s_good = torch.cuda.Stream(), torch.cuda.Stream()
    out_bad = torch.empty(M, N, dtype=torch.float16, device="cuda")
    out_good = torch.empty(M, N, dtype=torch.float16, device="cuda")
    torch.cuda.synchronize()
    assert pws.gemm_device_status(s_bad) == pws.GEMM_OK and pws.gemm_device_status(s_good) == pws.GEMM_OK
    pws.gemm_set_wait_timeout_ns(200_000_000)
    try:
        pws.gemm_set_debug_flags(pws.GEMM_DEBUG_SKIP_EMPTY_SEED)
        try:
            pws.gemm_f16_nt(a, b, out_bad, stages=2, stream=s_bad)
        finally:
            pws.gemm_set_debug_flags(0)
        pws.gemm_f16_nt(a, b, out_good, stages=2, stream=s_good)
        assert pws.gemm_device_status(s_good) == pws.GEMM_OK        # synchronizes s_good only
        assert pws.gemm_device_status(s_bad) == pws.GEMM_ERR_TIMEOUT
        assert pws.gemm_device_status(s_bad) == pws.GEMM_OK         # cleared
        assert pws.gemm_device_status(s_good) == pws.GEMM_OK
        assert pws.gemm_device_status() == pws.GEMM_OK               # the current stream's own word
    finally:
        pws.gemm_set_debug_flags(0)
        pws.gemm_set_wait_timeout_ns(0)
    torch.cuda.synchronize()
    res = oracle.check_f16(out_good.cpu().numpy(), oracle.gemm_f16_nt_f64(a_np, b_np), K)
    assert res["ok"], res
