"""GPU parity: the CUDA kernels, called through the C ABI, against the CPU oracle
on the same seeded inputs.

s32 is bit-exact.  f16 satisfies |gpu - ref| <= ulp16(ref) + 1e-3 sqrt(K)
(ref = the float64 oracle), is bit-exact where the exact sum is a binary16
value (closed forms), and is bitwise identical across stage counts S = 1..6.
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
    yield torch.device("cuda:0")
    pws.gemm_set_debug_flags(0)


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


# `flags` value standing for gemm_set_scratch_pool(1) in the parametrized tests
POOL = 1 << 30


def run_f16(a, b, stages, flags=0):
    pws.gemm_set_debug_flags(flags & ~POOL)
    pws.gemm_set_scratch_pool(bool(flags & POOL))
    try:
        out = pws.gemm_f16_nt(_dev(a), _dev(b), stages=stages)
        torch.cuda.synchronize()
        assert pws.gemm_device_status() == pws.GEMM_OK
    finally:
        pws.gemm_set_debug_flags(0)
        pws.gemm_set_scratch_pool(False)
    return out.cpu().numpy()


def run_s32(a, b):
    out = pws.gemm_s32_nn(_dev(a), _dev(b))
    torch.cuda.synchronize()
    return out.cpu().numpy()


def assert_f16_ok(gpu, ref, K):
    res = oracle.check_f16(gpu, ref, K)
    assert res["ok"], res


# ------------------------------------------------------------------ s32 NN

def test_s32_page_config_bit_exact():
    wl = inputs.WORKLOADS["s32_nn_128x256x256"]
    a, b = wl.lhs(), wl.rhs()
    assert np.array_equal(run_s32(a, b), oracle.gemm_s32_nn(a, b))


@pytest.mark.parametrize("M,N,K", [
    (1, 1, 1), (1, 300, 1), (17, 33, 15), (129, 257, 17), (64, 64, 16), (300, 500, 77),
    (1000, 1000, 1000), (2048, 2048, 48), (5, 7, 3),
])
def test_s32_shapes_bit_exact(M, N, K):
    a = inputs.ints(M + 3, 0, (M, K), -1000, 1000)
    b = inputs.ints(N + 5, 1, (K, N), -1000, 1000)
    assert np.array_equal(run_s32(a, b), oracle.gemm_s32_nn(a, b))


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (1, 1, 1), (17, 33, 15), (300, 500, 77), (1000, 1000, 1000),
                                   (33, 18, 130), (1000, 700, 333)])
def test_s32_ring_every_stage_count_bit_exact(M, N, K):
    a = inputs.ints(M + 11, 0, (M, K), -1000, 1000)
    b = inputs.ints(N + 13, 1, (K, N), -1000, 1000)
    want = oracle.gemm_s32_nn(a, b)
    da, db = _dev(a), _dev(b)
    two = pws.gemm_s32_nn(da, db)
    for s in range(2, 7):
        got = pws.gemm_s32_nn_ring(da, db, stages=s)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), want), f"S={s}"
        assert torch.equal(got, two)


def test_two_copies_of_the_library_in_one_process(tmp_path):
    # Each copy of the library keeps its own per-kernel shared-memory
    # settings, so launches that need more than 48 KB of dynamic shared
    # memory (the 64 x 64 ring tile at S = 6, every f16 kernel) work from
    # both copies in turn.
    import shutil
    from pipelined_warp_specialized_gb300 import build as libbuild
    second = str(tmp_path / "libpwsgemm_copy.so")
    shutil.copy(libbuild.LIB_PATH, second)
    first = pws.load_library()
    other = pws.load_library(second)
    a = inputs.ints(7, 0, (1000, 333), -1000, 1000)
    b = inputs.ints(8, 1, (333, 700), -1000, 1000)
    want = oracle.gemm_s32_nn(a, b)
    da, db = _dev(a), _dev(b)
    a16 = _dev(inputs.uniform_f16(9, 0, (1024, 1024)))
    b16 = _dev(inputs.uniform_f16(9, 1, (1024, 1024)))
    outs = []
    try:
        for lib in (other, first, other):
            pws._lib = lib
            got = pws.gemm_s32_nn_ring(da, db, stages=6)
            outs.append(pws.gemm_f16_nt(a16, b16, stages=4))
            torch.cuda.synchronize()
            assert pws.gemm_device_status() == pws.GEMM_OK
            assert np.array_equal(got.cpu().numpy(), want)
    finally:
        pws._lib = first
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_graph_capture_replays_correctly():
    # the entry points only enqueue work on the given stream, so they can be
    # captured into a CUDA graph and replayed
    wl = inputs.WORKLOADS["s32_nn_128x256x256"]
    a32, b32 = wl.lhs(), wl.rhs()
    da32, db32 = _dev(a32), _dev(b32)
    o32 = torch.empty(wl.M, wl.N, dtype=torch.int32, device="cuda")
    M, N, K = 520, 384, 320
    a16 = inputs.uniform_f16(61, 0, (M, K))
    b16 = inputs.uniform_f16(61, 1, (N, K))
    da16, db16 = _dev(a16), _dev(b16)
    o16 = torch.empty(M, N, dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                       # first calls outside the capture
        pws.gemm_s32_nn(da32, db32, o32, stream=s)
        pws.gemm_f16_nt(da16, db16, o16, stages=3, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pws.gemm_s32_nn(da32, db32, o32, stream=s)
        pws.gemm_f16_nt(da16, db16, o16, stages=3, stream=s)
    o32.zero_()
    o16.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pws.gemm_device_status() == pws.GEMM_OK
    assert np.array_equal(o32.cpu().numpy(), oracle.gemm_s32_nn(a32, b32))
    assert_f16_ok(o16.cpu().numpy(), oracle.gemm_f16_nt_f64(a16, b16), K)


@pytest.mark.parametrize("ring_stages", [None, 3])
def test_s32_very_tall_output(ring_stages):
    # 65 537 row tiles of 128: more than a grid's y extent (65 535) holds, so
    # the tiles are numbered along a 1-D grid
    M, N, K = 65536 * 128 + 77, 5, 3
    a = inputs.ints(70, 0, (M, K))
    b = inputs.ints(70, 1, (K, N))
    if ring_stages is None:
        got = run_s32(a, b)
    else:
        out = pws.gemm_s32_nn_ring(_dev(a), _dev(b), stages=ring_stages)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
    assert np.array_equal(got, oracle.gemm_s32_nn(a, b))


def test_s32_wraps_on_overflow():
    M, N, K = 40, 24, 64
    a = inputs.ints(1, 0, (M, K), -2**31, 2**31 - 1)
    b = inputs.ints(1, 1, (K, N), -2**31, 2**31 - 1)
    assert np.array_equal(run_s32(a, b), oracle.gemm_s32_nn(a, b))


def test_s32_k_zero_and_unaligned_rows():
    a = np.zeros((5, 0), np.int32)
    b = np.zeros((0, 6), np.int32)
    assert np.array_equal(run_s32(a, b), np.zeros((5, 6), np.int32))
    # a row-major view starting one element in: 4-byte aligned only (element copies)
    big = _dev(inputs.ints(9, 0, (33 * 18 + 1,), -50, 50))
    a_t = big[1:].view(33, 18)
    b_np = inputs.ints(9, 1, (18, 21), -50, 50)
    out = pws.gemm_s32_nn(a_t, _dev(b_np))
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.gemm_s32_nn(a_t.cpu().numpy(), b_np))


# ------------------------------------------------------------------ f16 NT

def test_f16_1024_config_full():
    wl = inputs.WORKLOADS["f16_nt_1024"]
    a, b = wl.lhs(), wl.rhs()
    assert_f16_ok(run_f16(a, b, 2), oracle.gemm_f16_nt_f64(a, b), wl.K)


@pytest.mark.parametrize("flags", [0, pws.GEMM_DEBUG_FORCE_PAIR_TILE, pws.GEMM_DEBUG_FORCE_COPY_PRODUCER],
                         ids=["solo_tma", "pair_tma", "solo_copy"])
def test_f16_stage_counts_bitwise_identical(flags):
    M, N, K = 700, 650, 1000          # several tiles, ragged M and N, a K tail of 40
    a = inputs.uniform_f16(31, 0, (M, K))
    b = inputs.uniform_f16(31, 1, (N, K))
    outs = [run_f16(a, b, s, flags) for s in range(1, 7)]
    for s in range(1, 6):
        assert np.array_equal(outs[s].view(np.uint16), outs[0].view(np.uint16)), f"S={s + 1} differs from S=1"
    assert_f16_ok(outs[0], oracle.gemm_f16_nt_f64(a, b), K)


@pytest.mark.parametrize("M,N,K", [
    (2560, 2560, 256),      # wide tile for S <= 2, 256 x 256 for S >= 3: the same bits
    (2048, 2048, 512),      # the pair tile by wave count (64 pair tiles against 256 single)
    (1024, 1152, 2100),     # the K split, the operands read in place
    (1024, 1024, 1024),     # multi-box slots (256 / 128 K columns) for S <= 3, one box for S >= 4
    (700, 900, 1000),       # multi-box slots, the last slot's later boxes past K (K = 1000)
    (300, 260, 136),        # multi-box slots, the last slot's last box partly inside K
])
def test_f16_stage_counts_bitwise_identical_where_the_plan_changes(M, N, K):
    a = inputs.uniform_f16(M + K, 0, (M, K))
    b = inputs.uniform_f16(M + K, 1, (N, K))
    tiles = {(p["bm"], p["bn"], p["bk"], p["k_split"])
             for p in (pws.gemm_f16_nt_plan(M, N, K, stages=s) for s in range(1, 7))}
    outs = [run_f16(a, b, s) for s in range(1, 7)]
    for s in range(1, 6):
        assert np.array_equal(outs[s].view(np.uint16), outs[0].view(np.uint16)), f"S={s + 1} differs ({tiles})"
    assert_f16_ok(outs[0], oracle.gemm_f16_nt_f64(a, b), K)


@pytest.mark.parametrize("M,N,K,flags", [
    (1, 1, 1, 0), (1, 1, 8, 0), (5, 3, 64, 0), (128, 128, 64, 0), (129, 130, 72, 0),
    (260, 300, 136, pws.GEMM_DEBUG_FORCE_PAIR_TILE),      # second pair row: the peer CTA is all padding
    (513, 257, 200, pws.GEMM_DEBUG_FORCE_PAIR_TILE),
    (65, 70, 33, 0),                                     # odd K: repacked, then TMA
    (96, 80, 34, 0),
    (65, 70, 33, pws.GEMM_DEBUG_FORCE_COPY_PRODUCER),    # odd K: 2-byte element copies
    (96, 80, 34, pws.GEMM_DEBUG_FORCE_COPY_PRODUCER),    # K % 4 == 2: 4-byte copies
    (96, 80, 44, pws.GEMM_DEBUG_FORCE_COPY_PRODUCER),    # K % 8 == 4: 8-byte copies
    (700, 600, 2050, pws.GEMM_DEBUG_FORCE_PAIR_TILE),    # repacked into the pair tile
    (100, 77, 64, 0),                                    # odd N: guarded plain stores
    (200, 136, 128, pws.GEMM_DEBUG_FORCE_DIRECT_STORE),
    (300, 280, 512, pws.GEMM_DEBUG_FORCE_COPY_PRODUCER | pws.GEMM_DEBUG_FORCE_DIRECT_STORE),
])
def test_f16_edge_shapes(M, N, K, flags):
    a = inputs.normal_f16(M * 3 + K, 0, (M, K))
    b = inputs.normal_f16(N * 7 + K, 1, (N, K))
    for s in (1, 3):
        assert_f16_ok(run_f16(a, b, s, flags), oracle.gemm_f16_nt_f64(a, b), K)


@pytest.mark.parametrize("M,N,K,flags", [
    (1024, 1024, 1024, pws.GEMM_DEBUG_NO_KSPLIT),         # 64 single tiles < 152 SMs: every tile split in 2
    (700, 650, 1000, pws.GEMM_DEBUG_FORCE_PAIR_TILE),     # 9 pair tiles < 76 pairs: every tile split in 2
    (2300, 2100, 768, 0),                                 # 9 x 9 pair tiles = 81 > 76: a 5-tile tail split
])
def test_f16_tail_split_matches_unsplit(M, N, K, flags):
    a = inputs.uniform_f16(M + N, 0, (M, K))
    b = inputs.uniform_f16(M + N, 1, (N, K))
    ref = oracle.gemm_f16_nt_f64(a, b)
    split = run_f16(a, b, 3, flags)
    whole = run_f16(a, b, 3, flags | pws.GEMM_DEBUG_NO_SPLIT)
    assert_f16_ok(split, ref, K)
    # a half-width unit runs the whole K loop for its columns: same sums, same order
    assert np.array_equal(split.view(np.uint16), whole.view(np.uint16))


KS = pws.GEMM_DEBUG_FORCE_KSPLIT


@pytest.mark.parametrize("M,N,K,flags", [
    (1024, 1024, 2048, 0),                               # 64 tiles, 128 CTAs, 32 K blocks
    (700, 650, 4000, 0),                                 # ragged M and N, a K tail of 32
    (1024, 1152, 2100, 0),                               # 72 tiles, 144 CTAs
    (65, 70, 2051, 0),                                   # odd K: repacked, then TMA
    (100, 77, 2048, 0),                                  # odd N: guarded plain stores
    (129, 130, 257, KS),                                 # 5 K blocks: halves of 3 and 2, the last ragged
    (1, 1, 256, KS), (5, 3, 300, KS),                    # one tile, almost all padding
    (300, 280, 512, KS | pws.GEMM_DEBUG_FORCE_COPY_PRODUCER),
    (96, 80, 1002, KS | pws.GEMM_DEBUG_FORCE_COPY_PRODUCER | pws.GEMM_DEBUG_FORCE_DIRECT_STORE),
    (300, 300, 128, KS),                                 # 2 K blocks: one each
    (2048, 2048, 512, KS | pws.GEMM_DEBUG_FORCE_SOLO_TILE),   # 256 clusters: more than fit at once
])
def test_f16_k_split(M, N, K, flags):
    # A cluster of two CTAs per single-CTA tile, one K half each; the senders
    # of each lane quarter write their fp32 partial sums into the owner's
    # shared memory, where the owner adds them before rounding.  Checked
    # against the oracle for S = 1, 2 and 6 (the smallest ring, whose 32 KB
    # hold the owners' output staging exactly, and the paired-slot MMA loop),
    # bitwise equal across them.
    pws.gemm_set_debug_flags(flags)
    try:
        assert pws.gemm_f16_nt_plan(M, N, K, stages=2)["k_split"] == 2
    finally:
        pws.gemm_set_debug_flags(0)
    a = inputs.normal_f16(M + 3 * K, 0, (M, K))
    b = inputs.normal_f16(N + 5 * K, 1, (N, K))
    ref = oracle.gemm_f16_nt_f64(a, b)
    outs = [run_f16(a, b, s, flags) for s in (1, 2, 6)]
    assert_f16_ok(outs[0], ref, K)
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint16), outs[0].view(np.uint16))
    # the unsplit sum is a different rounding of the same values
    assert_f16_ok(run_f16(a, b, 2, flags | pws.GEMM_DEBUG_NO_KSPLIT), ref, K)


def test_f16_k_split_every_stage_count():
    # 1024 x 1024 x 4096 runs the K split for every S, with one result
    M, N, K = 1024, 1024, 4096
    a = inputs.uniform_f16(77, 0, (M, K))
    b = inputs.uniform_f16(77, 1, (N, K))
    assert {pws.gemm_f16_nt_plan(M, N, K, stages=s)["k_split"] for s in range(1, 7)} == {2}
    outs = [run_f16(a, b, s) for s in range(1, 7)]
    for s in range(1, 6):
        assert np.array_equal(outs[s].view(np.uint16), outs[0].view(np.uint16)), f"S={s + 1}"
    assert_f16_ok(outs[0], oracle.gemm_f16_nt_f64(a, b), K)


WIDE = pws.GEMM_DEBUG_FORCE_PAIR_TILE | pws.GEMM_DEBUG_FORCE_WIDE_TILE
NARROW = pws.GEMM_DEBUG_FORCE_PAIR_TILE | pws.GEMM_DEBUG_FORCE_NARROW_TILE


def test_f16_wide_tile_bitwise_equals_narrow_and_solo():
    # 3 x 3 wide tiles: ragged M (700 = 2 x 256 + 188), N = 1100 leaves a last
    # tile column of 76 (its second B box wholly past N), K has a tail of 40
    M, N, K = 700, 1100, 1000
    a = inputs.uniform_f16(41, 0, (M, K))
    b = inputs.uniform_f16(41, 1, (N, K))
    narrow = run_f16(a, b, 3, NARROW)
    # (54 single tiles would take the K split, which adds two partial sums)
    solo = run_f16(a, b, 3, pws.GEMM_DEBUG_FORCE_SOLO_TILE | pws.GEMM_DEBUG_NO_KSPLIT)
    assert_f16_ok(narrow, oracle.gemm_f16_nt_f64(a, b), K)
    # every tiling sums each element over K in the same order
    assert np.array_equal(solo.view(np.uint16), narrow.view(np.uint16))
    for s in range(1, 5):
        for extra in (0, pws.GEMM_DEBUG_NO_SPLIT):
            wide = run_f16(a, b, s, WIDE | extra)
            assert np.array_equal(wide.view(np.uint16), narrow.view(np.uint16)), f"wide S={s} flags={extra}"


@pytest.mark.parametrize("M,N,K", [
    (1, 1, 8), (5, 3, 64),                 # one tile, almost all padding
    (260, 300, 136),                       # the peer CTA's rows and the second B box past M and N
    (256, 512, 64), (257, 513, 72),        # exact tile, and one row / column over
    (513, 257, 200), (300, 1030, 72),
    (700, 1100, 2050),                     # repacked operands into the wide tile
])
def test_f16_wide_tile_edge_shapes(M, N, K):
    a = inputs.normal_f16(M * 5 + K, 0, (M, K))
    b = inputs.normal_f16(N * 11 + K, 1, (N, K))
    ref = oracle.gemm_f16_nt_f64(a, b)
    for s in (1, 2, 4):
        assert_f16_ok(run_f16(a, b, s, WIDE), ref, K)


@pytest.mark.parametrize("M,N,K", [
    (1024, 1024, 512),      # 4 x 2 wide tiles, fewer than the CTA pairs: all split into halves
    (2300, 4600, 256),      # 9 x 9 = 81 wide tiles: one full wave and a tail of 5 split into halves
])
def test_f16_wide_tile_tail_split(M, N, K):
    a = inputs.uniform_f16(M + N + 7, 0, (M, K))
    b = inputs.uniform_f16(M + N + 7, 1, (N, K))
    split = run_f16(a, b, 4, WIDE)
    whole = run_f16(a, b, 4, WIDE | pws.GEMM_DEBUG_NO_SPLIT)
    narrow = run_f16(a, b, 4, NARROW | pws.GEMM_DEBUG_NO_SPLIT)
    assert np.array_equal(split.view(np.uint16), whole.view(np.uint16))
    assert np.array_equal(split.view(np.uint16), narrow.view(np.uint16))
    assert_f16_ok(split, oracle.gemm_f16_nt_f64(a, b), K)


@pytest.mark.parametrize("stages,flags", [
    (4, pws.GEMM_DEBUG_FORCE_PAIR_TILE | pws.GEMM_DEBUG_FORCE_WIDE_TILE),
    (6, pws.GEMM_DEBUG_FORCE_PAIR_TILE),
    (2, pws.GEMM_DEBUG_FORCE_SOLO_TILE),
], ids=["wide", "pair", "solo"])
def test_f16_long_k(stages, flags):
    # 1025 K blocks, the last one ragged: the ring laps each slot hundreds of
    # times, so every event's phase flips hundreds of times within one unit
    M, N, K = 300, 520, 65536 + 40
    a = inputs.uniform_f16(95, 0, (M, K))
    b = inputs.uniform_f16(95, 1, (N, K))
    assert_f16_ok(run_f16(a, b, stages, flags), oracle.gemm_f16_nt_f64(a, b), K)


@pytest.mark.parametrize("M,N,K,stages", [
    (131072 + 77, 64, 64, 6),        # 513 pair tile rows: 65 raster groups of 8
    (131072 + 77, 512, 72, 4),       # the same with the wide tile
    (64, 131072 + 296, 64, 4),       # 257 wide tile columns (the last one ragged), walked both ways
])
def test_f16_very_tall_and_very_wide(M, N, K, stages):
    a = inputs.normal_f16(96, 0, (M, K))
    b = inputs.normal_f16(96, 1, (N, K))
    assert_f16_ok(run_f16(a, b, stages), oracle.gemm_f16_nt_f64(a, b), K)


def test_f16_k_zero_and_empty():
    a = np.zeros((7, 0), np.float16)
    b = np.zeros((5, 0), np.float16)
    assert np.array_equal(run_f16(a, b, 2).view(np.uint16), np.zeros((7, 5), np.uint16))
    out = pws.gemm_f16_nt(torch.zeros(0, 16, dtype=torch.float16, device="cuda"),
                          torch.zeros(4, 16, dtype=torch.float16, device="cuda"))
    assert out.shape == (0, 4)


@pytest.mark.parametrize("flags", [0, pws.GEMM_DEBUG_IN_PLACE, pws.GEMM_DEBUG_IN_PLACE | pws.GEMM_DEBUG_FORCE_PAIR_TILE,
                                   pws.GEMM_DEBUG_IN_PLACE | pws.GEMM_DEBUG_FORCE_PAIR_TILE | pws.GEMM_DEBUG_FORCE_WIDE_TILE,
                                   pws.GEMM_DEBUG_IN_PLACE | pws.GEMM_DEBUG_FORCE_KSPLIT, POOL,
                                   pws.GEMM_DEBUG_FORCE_COPY_PRODUCER],
                         ids=["fixed_array", "realign", "realign_pair", "realign_wide", "realign_ksplit", "pooled",
                              "copy"])
def test_f16_unaligned_operands(flags):
    M, N, K = 150, 90, 128
    big_a = _dev(inputs.uniform_f16(5, 0, (M * K + 1,)))
    a_t = big_a[1:].view(M, K)                           # 2-byte aligned only
    b = inputs.uniform_f16(5, 1, (N, K))
    pws.gemm_set_debug_flags(flags & ~POOL)
    pws.gemm_set_scratch_pool(bool(flags & POOL))
    try:
        out = pws.gemm_f16_nt(a_t, _dev(b), stages=2)
        torch.cuda.synchronize()
    finally:
        pws.gemm_set_debug_flags(0)
        pws.gemm_set_scratch_pool(False)
    assert pws.gemm_device_status() == pws.GEMM_OK
    assert_f16_ok(out.cpu().numpy(), oracle.gemm_f16_nt_f64(a_t.cpu().numpy(), b), K)


@pytest.mark.parametrize("offset", range(8))
def test_f16_unaligned_every_row_alignment(offset):
    # The realigning producer and the repack both read each row as the aligned
    # 16-byte blocks that hold it and shift them into place.  lhs starts
    # `offset` elements into a buffer and rhs 7 - offset; with K odd,
    # consecutive rows start 2 bytes further on, so every even byte offset
    # 0..14 occurs as a row start, for both operands, and the last rows end
    # near the buffers' ends.  In place on the single-CTA, pair and wide
    # tiles; repacked into the fixed array (gemm_f16_nt's default and the
    # no-alloc call) and into pooled scratch.
    M, N, K = 37, 45, 1027
    big_a = _dev(inputs.normal_f16(60 + offset, 0, (M * K + 8,)))
    big_b = _dev(inputs.normal_f16(60 + offset, 1, (N * K + 8,)))
    a_t = big_a[offset:offset + M * K].view(M, K)
    b_t = big_b[7 - offset:7 - offset + N * K].view(N, K)
    assert pws.gemm_f16_nt_plan(M, N, K, a_t.data_ptr(), b_t.data_ptr(), 3 << 40)["producer"] == 2
    ref = oracle.gemm_f16_nt_f64(a_t.cpu().numpy(), b_t.cpu().numpy())
    outs = []
    for fn, flags in ((pws.gemm_f16_nt, pws.GEMM_DEBUG_IN_PLACE),
                      (pws.gemm_f16_nt, pws.GEMM_DEBUG_IN_PLACE | pws.GEMM_DEBUG_FORCE_PAIR_TILE),
                      (pws.gemm_f16_nt, pws.GEMM_DEBUG_IN_PLACE | pws.GEMM_DEBUG_FORCE_PAIR_TILE |
                       pws.GEMM_DEBUG_FORCE_WIDE_TILE),
                      (pws.gemm_f16_nt, 0), (pws.gemm_f16_nt, POOL), (pws.gemm_f16_nt_noalloc, 0)):
        pws.gemm_set_debug_flags(flags & ~POOL)
        pws.gemm_set_scratch_pool(bool(flags & POOL))
        try:
            out = fn(a_t, b_t, stages=2)
            torch.cuda.synchronize()
        finally:
            pws.gemm_set_debug_flags(0)
            pws.gemm_set_scratch_pool(False)
        assert pws.gemm_device_status() == pws.GEMM_OK
        assert_f16_ok(out.cpu().numpy(), ref, K)
        outs.append(out.cpu().numpy().view(np.uint16))
    # every tile sums each element over K in the same order: the same bits
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


@pytest.mark.parametrize("M,N,K,S,extra", [
    (1024, 1024, 1024, 2, 0),   # the 1024^3 workload: 64 tiles as 128 half-width units (tail split)
    (1000, 1100, 1090, 3, POOL),    # TMA on the repacked copy; the last slot's second box 2 columns deep
    (2048, 2048, 200, 1, pws.GEMM_DEBUG_FORCE_SOLO_TILE),    # 256 tiles: more than one wave
    (129, 77, 64, 2, 0),        # a single K block: one box per slot either way
])
def test_f16_two_box_slots_bitwise_equal_one_box(M, N, K, S, extra):
    a = inputs.uniform_f16(90, 0, (M, K))
    b = inputs.uniform_f16(90, 1, (N, K))
    pws.gemm_set_debug_flags((pws.GEMM_DEBUG_FORCE_DOUBLE_SLOT | extra) & ~POOL)
    pws.gemm_set_scratch_pool(bool(extra & POOL))
    try:
        bk = pws.gemm_f16_nt_plan(M, N, K, stages=S)["bk"]
    finally:
        pws.gemm_set_debug_flags(0)
        pws.gemm_set_scratch_pool(False)
    assert bk == (64 if K <= 64 else (192 if S <= 2 else 128))
    outs = [run_f16(a, b, S, f | extra) for f in (pws.GEMM_DEBUG_FORCE_DOUBLE_SLOT, pws.GEMM_DEBUG_NO_DOUBLE_SLOT)]
    assert np.array_equal(outs[0].view(np.uint16), outs[1].view(np.uint16))
    assert_f16_ok(outs[0], oracle.gemm_f16_nt_f64(a, b), K)


@pytest.mark.parametrize("M,N,K,S,extra", [
    (1024, 1024, 1024, 2, 0),   # the 1024^3 workload: 128 half-width units, 4 slots of 4 boxes
    (1024, 1024, 1024, 1, 0),
    (700, 900, 1000, 2, 0),     # the last slot's last box partly inside K
    (300, 260, 136, 2, 0),      # one slot: three boxes inside K, the fourth past it
    (1000, 1100, 1090, 2, POOL),    # TMA on the repacked copy
])
def test_f16_four_box_slots_bitwise_equal_one_and_three_boxes(M, N, K, S, extra):
    # where every tile runs as two half-width units, their half-size B boxes
    # let a slot hold four boxes of each operand: the K order, and so the
    # bits, stay those of one and of three boxes per slot
    a = inputs.uniform_f16(91, 0, (M, K))
    b = inputs.uniform_f16(91, 1, (N, K))
    pws.gemm_set_scratch_pool(bool(extra & POOL))
    try:
        assert pws.gemm_f16_nt_plan(M, N, K, stages=S)["bk"] == 256
    finally:
        pws.gemm_set_scratch_pool(False)
    outs = [run_f16(a, b, S, f | extra)
            for f in (0, pws.GEMM_DEBUG_FORCE_DOUBLE_SLOT, pws.GEMM_DEBUG_NO_DOUBLE_SLOT)]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint16), outs[0].view(np.uint16))
    assert_f16_ok(outs[0], oracle.gemm_f16_nt_f64(a, b), K)


@pytest.mark.parametrize("M,N,K,S,flags,want", [
    (300, 260, 1024, 2, 0, {"cta_group": 1, "k_split": 1}),                       # 9 single-CTA tiles
    (300, 260, 4096, 2, 0, {"cta_group": 1, "k_split": 2}),                       # K split
    (1000, 1000, 512, 3, pws.GEMM_DEBUG_FORCE_SOLO_TILE, {"cta_group": 1}),       # tail split, half-width units
    (2048, 2048, 1024, 2, 0, {"cta_group": 2, "bn": 256}),                        # pair tile, one wave
    (2600, 2500, 640, 1, pws.GEMM_DEBUG_FORCE_NARROW_TILE, {"cta_group": 2, "bn": 256}),   # 110 tiles: tail split
    (4000, 3000, 512, 3, 0, {"cta_group": 2, "bn": 512}),                         # wide tile, tail split
    (4000, 3000, 512, 4, pws.GEMM_DEBUG_NO_SPLIT, {"cta_group": 2, "bn": 512}),
    (8192, 2048, 256, 6, 0, {"cta_group": 2, "bn": 256}),                         # six slots (paired MMA waits)
])
def test_f16_realign_equals_tma_bitwise(M, N, K, S, flags, want):
    # With K a multiple of 8, operands that start 2 bytes past a 16-byte
    # boundary are read by the realigning producer; an aligned copy is read
    # by TMA.  Same tile, same split, same summation order: the same bits.
    a_np = inputs.uniform_f16(80, 0, (M, K))
    b_np = inputs.uniform_f16(80, 1, (N, K))
    big_a = torch.empty(M * K + 8, dtype=torch.float16, device="cuda")
    big_b = torch.empty(N * K + 8, dtype=torch.float16, device="cuda")
    a_u = big_a[1:1 + M * K].view(M, K)
    b_u = big_b[3:3 + N * K].view(N, K)
    a_u.copy_(torch.from_numpy(a_np))
    b_u.copy_(torch.from_numpy(b_np))
    a_al, b_al = _dev(a_np), _dev(b_np)
    flags |= pws.GEMM_DEBUG_IN_PLACE           # the unaligned operands are read in place
    pws.gemm_set_debug_flags(flags)
    try:
        p_u = pws.gemm_f16_nt_plan(M, N, K, a_u.data_ptr(), b_u.data_ptr(), 3 << 40, S)
        p_al = pws.gemm_f16_nt_plan(M, N, K, a_al.data_ptr(), b_al.data_ptr(), 3 << 40, S)
        assert p_u["producer"] == 3 and p_al["producer"] == 0
        assert {k: p_u[k] for k in want} == want, p_u
        assert all(p_u[k] == p_al[k] for k in ("bm", "bn", "cta_group", "k_split", "tiles")), (p_u, p_al)
        got = pws.gemm_f16_nt(a_u, b_u, stages=S)
        want_out = pws.gemm_f16_nt(a_al, b_al, stages=S)
        torch.cuda.synchronize()
    finally:
        pws.gemm_set_debug_flags(0)
    assert pws.gemm_device_status() == pws.GEMM_OK
    assert np.array_equal(got.cpu().numpy().view(np.uint16), want_out.cpu().numpy().view(np.uint16))
    rows, cols = _sampled_entries(M, N, 81, 4000)
    ref = oracle.gemm_f16_nt_entries(a_np, b_np, rows, cols)
    res = oracle.check_f16(got.cpu().numpy()[rows, cols], ref, K)
    assert res["ok"], res


@pytest.mark.parametrize("flags", [0, pws.GEMM_DEBUG_FORCE_PAIR_TILE, pws.GEMM_DEBUG_FORCE_COPY_PRODUCER,
                                   pws.GEMM_DEBUG_FORCE_KSPLIT,
                                   pws.GEMM_DEBUG_FORCE_KSPLIT | pws.GEMM_DEBUG_FORCE_COPY_PRODUCER])
def test_f16_closed_forms_bit_exact(flags):
    # rank one with dyadic values: every sum is K * a_m * b_n, exact in fp32 and in f16
    # (with the K split each half's sum is exact too, so the added halves must be)
    K = 1024
    a = np.array([1.0, -1.0, 0.5, -0.5] * 75, np.float16)            # M = 300
    b = np.array([0.5, 1.0, -1.0, -0.5, 1.0] * 52, np.float16)       # N = 260
    A = np.repeat(a[:, None], K, axis=1)
    B = np.repeat(b[:, None], K, axis=1)
    got = run_f16(A, B, 3, flags)
    want = (K * np.outer(a.astype(np.float64), b.astype(np.float64))).astype(np.float16)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    # identity: out = B^T exactly
    Kp = 256
    eye = np.eye(Kp, dtype=np.float16)
    Bm = inputs.normal_f16(3, 1, (200, Kp))
    got = run_f16(eye, Bm, 2, flags)
    assert np.array_equal(got.view(np.uint16), np.ascontiguousarray(Bm.T).view(np.uint16))


def test_f16_overflow_gives_inf():
    A = np.full((130, 16), 256.0, np.float16)
    B = np.full((140, 16), 256.0, np.float16)
    B[1] = -256.0
    got = run_f16(A, B, 2).astype(np.float64)
    assert np.all(np.isposinf(got[:, 0])) and np.all(np.isneginf(got[:, 1]))


def _sampled_entries(M, N, seed, n_random, tile=128):
    rng = np.random.default_rng(seed)
    rows = sorted({0, M - 1, tile - 1, tile, 2 * tile - 1, 2 * tile, M // 2} & set(range(M)))
    cols = sorted({0, N - 1, tile - 1, tile, 2 * tile - 1, 2 * tile, N // 2} & set(range(N)))
    rr, cc = [], []
    for r in rows:                       # full rows crossing every column tile
        rr.append(np.full(N, r))
        cc.append(np.arange(N))
    for c in cols:                       # full columns crossing every row tile
        rr.append(np.arange(M))
        cc.append(np.full(M, c))
    rr.append(rng.integers(0, M, n_random))
    cc.append(rng.integers(0, N, n_random))
    return np.concatenate(rr), np.concatenate(cc)


@pytest.mark.parametrize("M,N,K,S", [
    (1, 8192, 4096, 4),       # one output row: a single-CTA tile row, the K split
    (8192, 1, 4096, 4),       # one output column
    (65536, 128, 256, 3),     # tall: 512 single tiles or 256 pair tiles, several waves
    (128, 65536, 256, 2),     # wide: the same, transposed
    (33, 40000, 72, 1),       # one slot, a ragged single K block past 64
    (40000, 33, 1000, 6),     # six slots on the pair tile with one ragged column tile
    (2, 3, 70000, 2),         # long K on one tile: the K split, 1094 K blocks
])
def test_f16_extreme_aspect_ratios(M, N, K, S):
    # shapes at the edges of the plan's rules, against the f64 oracle on
    # whole rows and columns crossing every tile plus random entries, and
    # bitwise equal at another ring depth
    a = inputs.uniform_f16(M % 997 + 3, 0, (M, K))
    b = inputs.uniform_f16(N % 991 + 5, 1, (N, K))
    got = run_f16(a, b, S)
    other = run_f16(a, b, 1 if S != 1 else 3)
    assert np.array_equal(got.view(np.uint16), other.view(np.uint16))
    rows, cols = _sampled_entries(M, N, 7, 3000)
    ref = oracle.gemm_f16_nt_entries(a, b, rows, cols)
    res = oracle.check_f16(got[rows, cols], ref, K)
    assert res["ok"], res


def test_f16_4096_config_full():
    # every one of the 16.8 M outputs against the f64 oracle (about 3 s on 16 host cores)
    wl = inputs.WORKLOADS["f16_nt_4096"]
    a, b = wl.lhs(), wl.rhs()
    got = run_f16(a, b, 4)
    assert_f16_ok(got, oracle.gemm_f16_nt_f64(a, b), wl.K)


def test_f16_ragged_config_full():
    # K = 2050: rows of 4100 bytes, which no tensor map describes.  The
    # default path repacks them into the library's fixed array and runs the
    # wide pair tile on the copy; also read in place by the realigning
    # producer on the wide, 256 x 256 pair and single-CTA tiles, the pooled
    # repack and the async-copy producer.  All against the oracle, and the
    # tiles bitwise equal to each other.
    wl = inputs.WORKLOADS["f16_nt_ragged_4000x3000x2050"]
    a, b = wl.lhs(), wl.rhs()
    p = pws.gemm_f16_nt_plan(wl.M, wl.N, wl.K, stages=3)
    assert (p["producer"], p["cta_group"], p["bn"]) == (2, 2, 512)
    ref = oracle.gemm_f16_nt_f64(a, b)
    outs = []
    for flags in (0, pws.GEMM_DEBUG_IN_PLACE, pws.GEMM_DEBUG_IN_PLACE | pws.GEMM_DEBUG_FORCE_NARROW_TILE,
                  pws.GEMM_DEBUG_IN_PLACE | pws.GEMM_DEBUG_FORCE_SOLO_TILE, POOL,
                  pws.GEMM_DEBUG_FORCE_COPY_PRODUCER):
        got = run_f16(a, b, 3, flags)
        assert_f16_ok(got, ref, wl.K)
        outs.append(got.view(np.uint16))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_f16_repack_scratch_is_stream_ordered():
    # two unaligned-K GEMMs in flight on two streams, each with its own pooled
    # scratch (gemm_set_scratch_pool), repeated so the pool hands blocks
    # back and out again
    M, N, K = 640, 520, 1030
    cases = []
    for seed in (41, 42):
        a = inputs.uniform_f16(seed, 0, (M, K))
        b = inputs.uniform_f16(seed, 1, (N, K))
        cases.append((a, b, _dev(a), _dev(b), oracle.gemm_f16_nt_f64(a, b)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty(M, N, dtype=torch.float16, device="cuda") for _ in range(2)]
    for _ in range(3):
        pws.gemm_set_scratch_pool(True)
        try:
            assert pws.gemm_f16_nt_plan(M, N, K)["producer"] == 2
            for (a, b, da, db, _), s, o in zip(cases, streams, outs):
                pws.gemm_f16_nt(da, db, o, stages=4, stream=s)
        finally:
            pws.gemm_set_scratch_pool(False)
        torch.cuda.synchronize()
        assert pws.gemm_device_status() == pws.GEMM_OK
        for (a, b, da, db, ref), o in zip(cases, outs):
            assert_f16_ok(o.cpu().numpy(), ref, K)


def test_f16_fixed_array_shared_by_calls_on_four_streams():
    # Unaligned-K GEMMs on four streams, each repacked into the library's one
    # fixed array: every use is ordered after the previous one by an event,
    # so no call reads another's copy.  Rounds with different inputs, each
    # output against the oracle; also through the no-alloc entry point.
    M, N, K = 520, 640, 1030
    cases = []
    for seed in range(43, 47):
        a = inputs.uniform_f16(seed, 0, (M, K))
        b = inputs.uniform_f16(seed, 1, (N, K))
        cases.append((_dev(a), _dev(b), oracle.gemm_f16_nt_f64(a, b)))
    assert pws.gemm_f16_nt_plan(M, N, K)["producer"] == 2
    streams = [torch.cuda.Stream() for _ in range(4)]
    outs = [torch.empty(M, N, dtype=torch.float16, device="cuda") for _ in range(4)]
    torch.cuda.synchronize()
    for fn in (pws.gemm_f16_nt, pws.gemm_f16_nt_noalloc, pws.gemm_f16_nt):
        for r in range(3):
            for i, (st, o) in enumerate(zip(streams, outs)):
                da, db, _ = cases[(i + r) % 4]
                fn(da, db, o, stages=3, stream=st)
            torch.cuda.synchronize()
            for s_ in streams:
                assert pws.gemm_device_status(s_) == pws.GEMM_OK
            for i, o in enumerate(outs):
                assert_f16_ok(o.cpu().numpy(), cases[(i + r) % 4][2], K)


def test_f16_unaligned_calls_inside_graph_capture():
    # A stream being captured cannot wait for the fixed array's event, so
    # gemm_f16_nt reads unaligned operands in place there (the no-alloc call
    # uses the array, unordered); the replayed graph gives the same bits as
    # the eager calls, which repack into the array.
    M, N, K = 300, 260, 1030
    a_np = inputs.normal_f16(48, 0, (M, K))
    b_np = inputs.normal_f16(48, 1, (N, K))
    a, b = _dev(a_np), _dev(b_np)
    ref = oracle.gemm_f16_nt_f64(a_np, b_np)
    eager = pws.gemm_f16_nt(a, b, stages=2)
    torch.cuda.synchronize()
    for fn in (pws.gemm_f16_nt, pws.gemm_f16_nt_noalloc):
        out = torch.empty(M, N, dtype=torch.float16, device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn(a, b, out, stages=2, stream=s)          # first call of the process on this path: set-up
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn(a, b, out, stages=2, stream=s)
        out.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert pws.gemm_device_status(s) == pws.GEMM_OK
        assert_f16_ok(out.cpu().numpy(), ref, K)
        assert np.array_equal(out.cpu().numpy().view(np.uint16), eager.cpu().numpy().view(np.uint16))


def test_concurrent_gemms_on_four_streams():
    # independent f16 GEMMs (single-CTA, 256x256 and wide pair tiles, S = 1..4,
    # and two K splits, whose clusters run side by side) and s32 GEMMs issued
    # round-robin on four streams forked from one, first eagerly, then
    # captured as one fork/join graph and replayed
    f16_cases = []
    for i, (M, N, K) in enumerate([(300, 260, 200), (1024, 1024, 256), (4096, 4096, 64), (2304, 4608, 128),
                                   (700, 1100, 320), (260, 300, 2048), (129, 520, 2500)]):
        a = inputs.uniform_f16(70 + i, 0, (M, K))
        b = inputs.uniform_f16(70 + i, 1, (N, K))
        f16_cases.append((_dev(a), _dev(b), oracle.gemm_f16_nt_f64(a, b), K,
                          torch.empty(M, N, dtype=torch.float16, device="cuda")))
    s32_cases = []
    for i, (M, N, K) in enumerate([(128, 256, 256), (17, 33, 15), (300, 500, 77)]):
        a = inputs.ints(80 + i, 0, (M, K), -1000, 1000)
        b = inputs.ints(80 + i, 1, (K, N), -1000, 1000)
        s32_cases.append((_dev(a), _dev(b), oracle.gemm_s32_nn(a, b), torch.empty(M, N, dtype=torch.int32, device="cuda")))
    streams = [torch.cuda.Stream() for _ in range(4)]

    def launch_all(s0):
        for st in streams:
            st.wait_stream(s0)
        j = 0
        for da, db, _, _, o in f16_cases:
            pws.gemm_f16_nt(da, db, o, stages=j % 4 + 1, stream=streams[j % 4])
            j += 1
        for da, db, _, o in s32_cases:
            pws.gemm_s32_nn(da, db, o, stream=streams[j % 4])
            j += 1
        for st in streams:
            s0.wait_stream(st)

    def check_and_clear():
        torch.cuda.synchronize()
        assert pws.gemm_device_status() == pws.GEMM_OK
        for _, _, ref, K, o in f16_cases:
            assert_f16_ok(o.cpu().numpy(), ref, K)
            o.zero_()
        for _, _, ref, o in s32_cases:
            assert np.array_equal(o.cpu().numpy(), ref)
            o.zero_()
        torch.cuda.synchronize()

    s0 = torch.cuda.Stream()
    s0.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s0):
        launch_all(s0)
    check_and_clear()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s0):
        launch_all(s0)
    for _ in range(2):
        g.replay()
        check_and_clear()


@pytest.mark.parametrize("M,stages", [(1024, 2), (4096, 4)], ids=["single_tile", "wide_tile"])
def test_dependent_f16_chain_reads_completed_outputs(M, stages):
    # x <- f16(x . W^T) six times on one stream: each GEMM reads the previous
    # one's output.  Every kernel lets the next grid be scheduled while it runs
    # (programmatic dependent launch); the next one must still read the
    # completed output.  Each step is checked against the oracle applied to the
    # previous step's GPU output.  W is scaled by 1/32 (exact in f16) so the
    # values neither overflow nor vanish over the chain.
    K = M
    w = (inputs.uniform_f16(90, 0, (K, K)).astype(np.float32) / 32).astype(np.float16)
    x = inputs.uniform_f16(91, 0, (M, K))
    dw = _dev(w)
    cur = _dev(x)
    outs = []
    for _ in range(6):
        cur = pws.gemm_f16_nt(cur, dw, stages=stages)
        outs.append(cur)
    torch.cuda.synchronize()
    assert pws.gemm_device_status() == pws.GEMM_OK
    prev = x
    for i, o in enumerate(outs):
        got = o.cpu().numpy()
        if M > 2048:     # the oracle on sampled entries at the large size
            rows, cols = _sampled_entries(M, M, 50 + i, 4000, tile=256)
            assert_f16_ok(got[rows, cols], oracle.gemm_f16_nt_entries(prev, w, rows, cols), K)
        else:
            assert_f16_ok(got, oracle.gemm_f16_nt_f64(prev, w), K)
        assert np.abs(got.astype(np.float32)).max() > 1e-3, f"step {i} vanished"
        prev = got


def test_dependent_s32_chain_reads_completed_outputs():
    # c <- c . B four times on one stream (wrapping int32), each step bit-exact
    # against the oracle applied to the previous step's GPU output
    n = 512
    b = inputs.ints(92, 1, (n, n), -3, 3)
    c = inputs.ints(92, 0, (n, n), -3, 3)
    db = _dev(b)
    cur = _dev(c)
    outs = []
    for _ in range(4):
        cur = pws.gemm_s32_nn(cur, db)
        outs.append(cur)
    torch.cuda.synchronize()
    prev = c
    for o in outs:
        got = o.cpu().numpy()
        assert np.array_equal(got, oracle.gemm_s32_nn(prev, b))
        prev = got


def test_calls_from_concurrent_host_threads():
    # four host threads call the library at the same time (ctypes releases the
    # GIL), each on its own stream with a different tile and S, five calls each
    import threading
    cases = []
    for i, (M, N, K, S) in enumerate([(700, 1100, 320, 4), (1024, 1024, 256, 2), (300, 260, 200, 6),
                                      (2304, 2560, 128, 3)]):
        a = inputs.uniform_f16(100 + i, 0, (M, K))
        b = inputs.uniform_f16(100 + i, 1, (N, K))
        cases.append((_dev(a), _dev(b), oracle.gemm_f16_nt_f64(a, b), K, S))
    results, errors = [None] * len(cases), []

    def worker(i):
        try:
            torch.cuda.set_device(0)
            da, db, _, _, S = cases[i]
            st = torch.cuda.Stream()
            st.wait_stream(torch.cuda.default_stream())
            outs = [pws.gemm_f16_nt(da, db, stages=S, stream=st) for _ in range(5)]
            st.synchronize()
            results[i] = outs
        except Exception as e:          # reported below, in the test's own thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert pws.gemm_device_status() == pws.GEMM_OK
    for (_, _, ref, K, _), outs in zip(cases, results):
        for o in outs:
            assert_f16_ok(o.cpu().numpy(), ref, K)


def test_f16_8192_sweep_identical_across_stages():
    wl = inputs.WORKLOADS["f16_nt_8192"]
    a, b = wl.lhs(), wl.rhs()
    da, db = _dev(a), _dev(b)
    first = None
    for s in wl.stages:
        out = pws.gemm_f16_nt(da, db, stages=s)
        torch.cuda.synchronize()
        assert pws.gemm_device_status() == pws.GEMM_OK
        if first is None:
            first = out
        else:
            assert torch.equal(out.view(torch.int16), first.view(torch.int16)), f"S={s} differs"
    # every one of the 67 M outputs against the f64 oracle: 1.1 TFLOP of f64
    # work, about half a minute on 16 host cores
    assert_f16_ok(first.cpu().numpy(), oracle.gemm_f16_nt_f64(a, b), wl.K)


def _random_cases(n, seed=2026):
    rng = np.random.default_rng(seed)
    flag_sets = [0, pws.GEMM_DEBUG_FORCE_PAIR_TILE, pws.GEMM_DEBUG_FORCE_PAIR_TILE | pws.GEMM_DEBUG_FORCE_WIDE_TILE,
                 pws.GEMM_DEBUG_FORCE_SOLO_TILE, pws.GEMM_DEBUG_FORCE_KSPLIT, pws.GEMM_DEBUG_NO_SPLIT,
                 pws.GEMM_DEBUG_FORCE_DOUBLE_SLOT, pws.GEMM_DEBUG_FORCE_DIRECT_STORE, POOL]
    cases = []
    for _ in range(n):
        M = int(rng.integers(1, 1300))
        N = int(rng.integers(1, 1300))
        K = int(rng.integers(1, 1400))
        S = int(rng.integers(1, 7))
        offs = (int(rng.integers(0, 8)), int(rng.integers(0, 8)))
        flags = flag_sets[int(rng.integers(0, len(flag_sets)))]
        cases.append((M, N, K, S, offs, flags))
    return cases


@pytest.mark.parametrize("M,N,K,S,offs,flags", _random_cases(40))
def test_f16_random_shapes_offsets_and_plans_against_the_oracle(M, N, K, S, offs, flags):
    # Seeded random shapes, element offsets of each operand from a 16-byte
    # boundary (0 with K % 8 == 0: TMA; otherwise the realigning producer or,
    # with the pool, the repack), ring depths and plan switches: every output
    # against the oracle, and the status word clean.
    a_np = inputs.normal_f16(M * 7 + K, 0, (M, K))
    b_np = inputs.normal_f16(N * 5 + K, 1, (N, K))
    big_a = torch.zeros(M * K + 8, dtype=torch.float16, device="cuda")
    big_b = torch.zeros(N * K + 8, dtype=torch.float16, device="cuda")
    a_t = big_a[offs[0]:offs[0] + M * K].view(M, K)
    b_t = big_b[offs[1]:offs[1] + N * K].view(N, K)
    a_t.copy_(torch.from_numpy(a_np))
    b_t.copy_(torch.from_numpy(b_np))
    pws.gemm_set_debug_flags(flags & ~POOL)
    pws.gemm_set_scratch_pool(bool(flags & POOL))
    try:
        out = pws.gemm_f16_nt(a_t, b_t, stages=S)
        torch.cuda.synchronize()
    finally:
        pws.gemm_set_debug_flags(0)
        pws.gemm_set_scratch_pool(False)
    assert pws.gemm_device_status() == pws.GEMM_OK
    assert_f16_ok(out.cpu().numpy(), oracle.gemm_f16_nt_f64(a_np, b_np), K)
