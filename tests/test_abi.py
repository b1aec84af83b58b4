"""The C-ABI library on the host (no GPU): it builds, loads, exports every
function its header declares, and its host logic (argument checks, launch
plan) behaves as the header states.  No call here launches a kernel."""
import ctypes

import pytest

import pipelined_warp_specialized_gb300 as pws
from pipelined_warp_specialized_gb300 import build as libbuild


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return pws.load_library()


def test_exports_every_declared_function(lib):
    names = pws.header_functions()
    assert set(names) >= {"gemm_s32_nn", "gemm_f16_nt", "gemm_device_status", "gemm_status_string",
                          "gemm_set_wait_timeout_ns", "gemm_set_debug_flags", "gemm_f16_nt_plan"}
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_exports_only_the_declared_functions(lib):
    # built with hidden visibility, the library's dynamic symbol table holds
    # exactly the header's functions: no internal function and no
    # function-local static that a second copy loaded into the same process
    # could bind to
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm is not installed")
    out = subprocess.run([nm, "-D", "--defined-only", libbuild.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    syms = {ln.split()[-1]: ln.split()[-2] for ln in out.splitlines() if ln.strip()}
    assert set(syms) == set(pws.header_functions()), sorted(set(syms) ^ set(pws.header_functions()))
    assert set(syms.values()) == {"T"}


def test_binding_constants_match_the_header():
    # every GEMM_* enumerator the header declares has the same value in the
    # binding, and the binding defines no GEMM_* constant the header lacks
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(pws.__file__), os.pardir, "include", "pwsgemm.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    declared = {m.group(1): int(m.group(2), 0) for m in re.finditer(r"\b(GEMM_[A-Z_]+)\s*=\s*(\d+)u?\b", hdr)}
    assert "GEMM_DEBUG_FORCE_KSPLIT" in declared and "GEMM_ERR_TIMEOUT" in declared
    bound = {k: v for k, v in vars(pws).items() if k.startswith("GEMM_") and isinstance(v, int)}
    assert bound == declared
    # the debug flags are distinct single bits
    flags = [v for k, v in declared.items() if k.startswith("GEMM_DEBUG_")]
    assert all(f and f & (f - 1) == 0 for f in flags) and len(set(flags)) == len(flags)


def test_binding_refuses_operands_on_different_devices():
    # stand-ins for CUDA tensors (no GPU here): the wrappers must refuse
    # before any launch when the operands sit on different devices
    torch = pytest.importorskip("torch")

    class Stub:
        def __init__(self, shape, dtype, device):
            self.shape, self.dtype, self.device, self.is_cuda = tuple(shape), dtype, torch.device(device), True

        def dim(self):
            return len(self.shape)

        def is_contiguous(self):
            return True

    f16, s32 = torch.float16, torch.int32
    cases = [
        (pws.gemm_f16_nt, Stub((4, 8), f16, "cuda:0"), Stub((5, 8), f16, "cuda:1"), None),
        (pws.gemm_f16_nt, Stub((4, 8), f16, "cuda:0"), Stub((5, 8), f16, "cuda:0"), Stub((4, 5), f16, "cuda:1")),
        (pws.gemm_f16_nt_noalloc, Stub((4, 8), f16, "cuda:1"), Stub((5, 8), f16, "cuda:0"), None),
        (pws.gemm_s32_nn, Stub((4, 8), s32, "cuda:0"), Stub((8, 5), s32, "cuda:1"), None),
        (pws.gemm_s32_nn_ring, Stub((4, 8), s32, "cuda:0"), Stub((8, 5), s32, "cuda:0"), Stub((4, 5), s32, "cuda:2")),
    ]
    for fn, a, b, out in cases:
        with pytest.raises(ValueError, match="one device"):
            fn(a, b, out=out)


def test_status_strings(lib):
    for code, name in [(0, "GEMM_OK"), (1, "GEMM_ERR_INVALID_ARG"), (2, "GEMM_ERR_ALIGNMENT"),
                       (3, "GEMM_ERR_UNSUPPORTED_STAGES"), (4, "GEMM_ERR_UNSUPPORTED_ARCH"),
                       (5, "GEMM_ERR_LAUNCH"), (6, "GEMM_ERR_TIMEOUT")]:
        assert pws.gemm_status_string(code) == name
    assert pws.gemm_status_string(99) == "GEMM_ERR_UNKNOWN"


A = 1 << 40            # fake, 16-byte aligned addresses: never dereferenced on these paths
B = 2 << 40
C = 3 << 40


@pytest.mark.parametrize("args,want", [
    ((-1, 4, 4, A, B, C, 2), pws.GEMM_ERR_INVALID_ARG),
    ((4, -1, 4, A, B, C, 2), pws.GEMM_ERR_INVALID_ARG),
    ((4, 4, -1, A, B, C, 2), pws.GEMM_ERR_INVALID_ARG),
    ((1 << 31, 4, 4, A, B, C, 2), pws.GEMM_ERR_INVALID_ARG),
    ((4, 4, 4, A, B, C, 0), pws.GEMM_ERR_UNSUPPORTED_STAGES),
    ((4, 4, 4, A, B, C, 7), pws.GEMM_ERR_UNSUPPORTED_STAGES),
    ((4, 4, 4, 0, B, C, 2), pws.GEMM_ERR_INVALID_ARG),
    ((4, 4, 4, A, B, 0, 2), pws.GEMM_ERR_INVALID_ARG),
    ((4, 4, 4, A + 1, B, C, 2), pws.GEMM_ERR_ALIGNMENT),
    ((4, 4, 4, A, B, A + 16, 2), pws.GEMM_ERR_INVALID_ARG),     # out overlaps lhs
    ((0, 4, 4, 0, 0, 0, 2), pws.GEMM_OK),                       # empty output: no-op
    ((4, 0, 4, 0, 0, 0, 6), pws.GEMM_OK),
])
def test_f16_argument_checks_return_before_launch(lib, args, want):
    M, N, K, a, b, c, s = args
    assert lib.gemm_f16_nt(M, N, K, a, b, c, s, None) == want


@pytest.mark.parametrize("args,want", [
    ((-1, 4, 4, A, B, C), pws.GEMM_ERR_INVALID_ARG),
    ((4, 4, 4, A, 0, C), pws.GEMM_ERR_INVALID_ARG),
    ((4, 4, 4, A + 2, B, C), pws.GEMM_ERR_ALIGNMENT),
    ((4, 4, 4, A, B, B + 4), pws.GEMM_ERR_INVALID_ARG),          # out overlaps rhs
    ((0, 4, 4, 0, 0, 0), pws.GEMM_OK),
])
def test_s32_argument_checks_return_before_launch(lib, args, want):
    assert lib.gemm_s32_nn(*args, None) == want


@pytest.mark.parametrize("args,want", [
    ((4, 4, 4, A, B, C, 1), pws.GEMM_ERR_UNSUPPORTED_STAGES),
    ((4, 4, 4, A, B, C, 7), pws.GEMM_ERR_UNSUPPORTED_STAGES),
    ((-1, 4, 4, A, B, C, 3), pws.GEMM_ERR_INVALID_ARG),
    ((4, 4, 4, A + 2, B, C, 3), pws.GEMM_ERR_ALIGNMENT),
    ((0, 4, 4, 0, 0, 0, 3), pws.GEMM_OK),
])
def test_s32_ring_argument_checks_return_before_launch(lib, args, want):
    assert lib.gemm_s32_nn_ring(*args, None) == want


def test_debug_flags_and_timeout_setters(lib):
    assert lib.gemm_set_debug_flags(1 << 15) == pws.GEMM_ERR_INVALID_ARG
    assert lib.gemm_set_debug_flags(0) == pws.GEMM_OK
    assert lib.gemm_set_wait_timeout_ns(0) == pws.GEMM_OK


def test_plan_headline_shapes(lib):
    pws.gemm_set_debug_flags(0)
    # five and six slots: the 256 x 256 pair tile, 32 KB slots
    p = pws.gemm_f16_nt_plan(8192, 8192, 8192, stages=6)
    assert (p["bm"], p["bn"], p["bk"], p["cta_group"]) == (256, 256, 64, 2)
    assert p["producer"] == 0 and p["store"] == 0
    assert p["tiles"] == 32 * 32 and p["k_blocks"] == 128
    assert {k: v for k, v in pws.gemm_f16_nt_plan(8192, 8192, 8192, stages=5).items() if k != "smem_bytes"} == \
        {k: v for k, v in p.items() if k != "smem_bytes"}
    # one to four slots: the wide 256 x 512 pair tile, 48 KB slots (A and two B boxes per CTA)
    for s in range(1, 7):
        q = pws.gemm_f16_nt_plan(8192, 8192, 8192, stages=s)
        slot = 49152 if s <= 4 else 32768
        assert q["bn"] == (512 if s <= 4 else 256)
        assert q["tiles"] == 32 * (16 if s <= 4 else 32)
        # ring slots plus 32 KB of epilogue staging fit the 227 KB limit for every S
        assert s * slot + 32768 <= q["smem_bytes"] <= 232448


def test_plan_wide_tile_rule(lib):
    # the wide tile is used where its 512-column tiles add no padded block of 256 columns
    for n, wide in ((8192, True), (3000, True), (512, True), (4608, True), (256, False), (768, False),
                    (1100, False), (257, True)):
        q = pws.gemm_f16_nt_plan(32768, n, 1024, stages=4)      # M large enough for the pair tile
        assert q["cta_group"] == 2 and (q["bn"] == 512) == wide, n
    # the debug flags override it either way; six slots never fit the wide tile
    try:
        pws.gemm_set_debug_flags(pws.GEMM_DEBUG_FORCE_NARROW_TILE)
        assert pws.gemm_f16_nt_plan(8192, 8192, 8192, stages=4)["bn"] == 256
        pws.gemm_set_debug_flags(pws.GEMM_DEBUG_FORCE_WIDE_TILE)
        assert pws.gemm_f16_nt_plan(32768, 256, 1024, stages=4)["bn"] == 512
        assert pws.gemm_f16_nt_plan(32768, 256, 1024, stages=6)["bn"] == 256
        # the single-CTA tile has no wide form
        pws.gemm_set_debug_flags(pws.GEMM_DEBUG_FORCE_WIDE_TILE | pws.GEMM_DEBUG_FORCE_SOLO_TILE)
        assert (pws.gemm_f16_nt_plan(4096, 4096, 1024, stages=4)["bn"], pws.gemm_f16_nt_plan(4096, 4096, 1024, stages=4)["cta_group"]) == (128, 1)
    finally:
        pws.gemm_set_debug_flags(0)


def test_plan_wave_count_rules(lib):
    # pair tiles where they need fewer waves of the grid than single tiles
    # (152 SMs: 76 pairs), whatever S; ties keep the old rule
    pws.gemm_set_debug_flags(0)
    def tile(M, N, K, s):
        p = pws.gemm_f16_nt_plan(M, N, K, stages=s)
        return p["bm"], p["bn"]
    for s in range(1, 7):
        assert tile(2048, 2048, 2048, s) == (256, 256)      # 64 pair tiles (1 wave) vs 256 single (2)
        assert tile(1024, 4096, 2048, s) == (256, 256)
        assert tile(1536, 1536, 1536, s) == (128, 128)      # 1 wave either way, 36 pair tiles
        assert tile(1024, 1024, 1024, s) == (128, 128)
    # the wide tile gives way to 256 x 256 where that fills the pairs better
    # (same bits either way, so S may decide)
    for s in range(1, 5):
        assert tile(2048, 2048, 4096, s) == (256, 256)      # 64 narrow tiles fit one wave
        assert tile(2560, 2560, 2560, s) == ((256, 512) if s <= 2 else (256, 256))
        assert tile(3072, 3072, 3072, s) == (256, 512)      # narrow tail of 68 does not half-split
        assert tile(4096, 4096, 4096, s) == (256, 512)
        assert tile(2048, 4096, 4096, s) == (256, 512)
        assert tile(8192, 8192, 8192, s) == (256, 512)


def test_plan_sum_order_never_depends_on_stages(lib):
    # Results are bitwise identical across S because the choices that change
    # the summation (the K split) or could (single CTA vs pair) read the shape
    # only.  Checked over a grid of shapes around every threshold of the
    # rules: tile-count edges, the 32-block K-split edge, ragged sizes.
    pws.gemm_set_debug_flags(0)
    dims = [1, 64, 129, 256, 300, 640, 1000, 1024, 1152, 1216, 1536, 2048, 2304, 2560, 3072, 4096, 9728, 20000]
    ks = [1, 64, 200, 1984, 1985, 2048, 4100, 8192]
    for M in dims:
        for N in dims:
            for K in ks:
                plans = [pws.gemm_f16_nt_plan(M, N, K, stages=s) for s in range(1, 7)]
                assert len({(p["cta_group"], p["k_split"]) for p in plans}) == 1, (M, N, K)
                for s, p in enumerate(plans, start=1):
                    assert p["bn"] != 512 or s <= 4, (M, N, K, s)            # the wide tile needs <= 4 slots
                    # multi-box slots (192 or 256 K columns per slot for at
                    # most 2 slots, 128 for 3, multiplied in the same K
                    # order) only on the single-CTA tile, without the K split;
                    # four boxes only where every tile runs as two half-width
                    # units (the tiles fill at most half the SMs)
                    assert p["bk"] == 64 or (p["bk"] in ((192, 256) if s <= 2 else (128,)) and s <= 3
                                             and p["cta_group"] == 1 and p["k_split"] == 1), (M, N, K, s)
                    assert p["bk"] != 256 or 2 * p["tiles"] <= 152, (M, N, K, s)
                    assert p["k_blocks"] == -(-K // p["bk"]), (M, N, K, s)
                    assert p["k_split"] == 1 or p["cta_group"] == 1, (M, N, K)
                    assert p["k_split"] == 1 or p["k_blocks"] >= 32, (M, N, K)


def test_smoke_cases_plan_the_paths_they_check(lib):
    # smoke() runs on the GPU only at round end; its plan expectations are
    # host logic and are checked here first
    import __graft_entry__
    pws.gemm_set_debug_flags(0)
    __graft_entry__.check_smoke_plans()


def test_plan_k_split_rule(lib):
    # single-CTA tiles that leave at least half of the 152 SMs idle, with at
    # least 32 K blocks: two CTAs (a cluster) per tile, one K half each.  The
    # rule reads the shape only, never S.
    pws.gemm_set_debug_flags(0)
    for s in range(1, 7):
        p = pws.gemm_f16_nt_plan(1024, 1024, 4096, stages=s)
        assert (p["cta_group"], p["tiles"], p["k_blocks"], p["k_split"]) == (1, 64, 64, 2), s
        assert pws.gemm_f16_nt_plan(1024, 1024, 1024, stages=s)["k_split"] == 1      # 16 K blocks
    assert pws.gemm_f16_nt_plan(1024, 1024, 1985)["k_split"] == 2        # 32 K blocks, the last ragged
    assert pws.gemm_f16_nt_plan(1024, 1024, 1984)["k_split"] == 1        # 31 K blocks
    assert pws.gemm_f16_nt_plan(700, 650, 4000)["k_split"] == 2          # 6 x 6 tiles
    assert pws.gemm_f16_nt_plan(1024, 1152, 2048)["k_split"] == 2        # 8 x 9 = 72 tiles: 144 CTAs
    assert pws.gemm_f16_nt_plan(1024, 1216, 2048)["k_split"] == 1        # 8 x 10 = 80 tiles: 160 CTAs > 152
    assert pws.gemm_f16_nt_plan(4096, 4096, 4096)["k_split"] == 1        # pair tiles
    assert pws.gemm_f16_nt_plan(4000, 3000, 2050, stages=3)["k_split"] == 1
    assert pws.gemm_f16_nt_plan(65, 70, 2051)["k_split"] == 2            # repacked operands
    try:
        pws.gemm_set_debug_flags(pws.GEMM_DEBUG_FORCE_COPY_PRODUCER)
        assert pws.gemm_f16_nt_plan(700, 650, 4000)["k_split"] == 2
        pws.gemm_set_debug_flags(pws.GEMM_DEBUG_NO_KSPLIT)
        assert pws.gemm_f16_nt_plan(1024, 1024, 4096)["k_split"] == 1
        pws.gemm_set_debug_flags(pws.GEMM_DEBUG_FORCE_PAIR_TILE)
        assert pws.gemm_f16_nt_plan(1024, 1024, 4096)["k_split"] == 1
        pws.gemm_set_debug_flags(pws.GEMM_DEBUG_FORCE_KSPLIT | pws.GEMM_DEBUG_FORCE_SOLO_TILE)
        assert pws.gemm_f16_nt_plan(4096, 4096, 1024)["k_split"] == 2        # 1024 tiles
        assert pws.gemm_f16_nt_plan(300, 300, 128)["k_split"] == 2           # 2 K blocks
        assert pws.gemm_f16_nt_plan(300, 300, 64)["k_split"] == 1            # 1 K block
    finally:
        pws.gemm_set_debug_flags(0)


def test_plan_ragged_shape(lib):
    # K = 2050: rows of 4100 bytes are not 16-byte aligned, so no TMA descriptor
    # exists for the operands as given.  They fit the library's fixed 32 MiB
    # array in 128-byte rows (7000 x 2112 x 2 bytes): repacked there, then fed
    # by TMA; nothing is allocated
    p = pws.gemm_f16_nt_plan(4000, 3000, 2050, stages=3)
    assert p["producer"] == 2 and p["copy_bytes"] == 16
    assert p["cta_group"] == 2 and p["bm"] == 256               # 16 x 12 pair tiles >= 152 / 2
    assert p["bn"] == 512                       # N = 3000: 6 wide tile columns pad no more than 12 narrow ones
    assert p["store"] == 0                      # 6000-byte output rows are 16-byte aligned
    assert p["tiles"] == 16 * 6 and p["k_blocks"] == 33
    # read in place by the realigning producer: the same tile
    pws.gemm_set_debug_flags(pws.GEMM_DEBUG_IN_PLACE)
    try:
        r = pws.gemm_f16_nt_plan(4000, 3000, 2050, stages=3)
    finally:
        pws.gemm_set_debug_flags(0)
    assert r["producer"] == 3 and {k: r[k] for k in ("bm", "bn", "tiles")} == {k: p[k] for k in ("bm", "bn", "tiles")}
    # too large for the array (16384 rows of 2112 elements): read in place,
    # unless the scratch pool is allowed
    assert pws.gemm_f16_nt_plan(8192, 8192, 2050, stages=3)["producer"] == 3
    pws.gemm_set_scratch_pool(True)
    try:
        assert pws.gemm_f16_nt_plan(8192, 8192, 2050, stages=3)["producer"] == 2
    finally:
        pws.gemm_set_scratch_pool(False)
    assert pws.gemm_f16_nt_plan(8192, 8192, 2050, stages=3)["producer"] == 3      # the setter is host state
    # the async-copy producer reads them in place (single-CTA tile, 4-byte copies)
    pws.gemm_set_debug_flags(pws.GEMM_DEBUG_FORCE_COPY_PRODUCER)
    try:
        q = pws.gemm_f16_nt_plan(4000, 3000, 2050, stages=3)
    finally:
        pws.gemm_set_debug_flags(0)
    assert q["producer"] == 1 and q["copy_bytes"] == 4
    assert q["cta_group"] == 1 and q["bm"] == 128
    assert q["tiles"] == 32 * 24 and q["k_blocks"] == 33


def test_plan_rejects_tile_counts_beyond_int(lib):
    # 2^16 x 2^16 tiles of 128 x 128: no such output fits in memory, and the
    # plan's tile count would overflow; refused before any launch
    with pytest.raises(pws.GemmError) as e:
        pws.gemm_f16_nt_plan(1 << 23, 1 << 23, 16)
    assert e.value.status == pws.GEMM_ERR_INVALID_ARG
    assert lib.gemm_f16_nt(1 << 23, 1 << 23, 16, 1 << 40, 2 << 40, 3 << 40, 4, None) == pws.GEMM_ERR_INVALID_ARG
    p = pws.gemm_f16_nt_plan(1 << 23, 1 << 15, 16)
    assert p["tiles"] == (1 << 15) * (1 << 6)
    # the s32 calls number their (at smallest 16 x 16) tiles in a 1-D grid
    assert lib.gemm_s32_nn(1 << 20, 1 << 20, 4, 1 << 40, 2 << 40, 3 << 40, None) == pws.GEMM_ERR_INVALID_ARG
    assert lib.gemm_s32_nn_ring(1 << 20, 1 << 20, 4, 1 << 40, 2 << 40, 3 << 40, 3, None) == pws.GEMM_ERR_INVALID_ARG


def test_plan_edge_cases(lib):
    assert pws.gemm_f16_nt_plan(7, 9, 3)["producer"] == 2            # odd K: repacked into the fixed array
    assert pws.gemm_f16_nt_plan(7, 9, 3)["store"] == 1               # odd N: plain stores
    assert pws.gemm_f16_nt_plan(64, 64, 16, lhs_ptr=A + 2)["producer"] == 2   # unaligned base
    pws.gemm_set_debug_flags(pws.GEMM_DEBUG_IN_PLACE)
    try:
        assert pws.gemm_f16_nt_plan(7, 9, 3)["producer"] == 3
        assert pws.gemm_f16_nt_plan(64, 64, 16, lhs_ptr=A + 2)["producer"] == 3
        assert pws.gemm_f16_nt_plan(64, 64, 16)["producer"] == 0      # aligned: TMA either way
    finally:
        pws.gemm_set_debug_flags(0)
    assert pws.gemm_f16_nt_plan(64, 64, 16)["producer"] == 0
    pws.gemm_set_debug_flags(pws.GEMM_DEBUG_FORCE_COPY_PRODUCER)
    try:
        assert pws.gemm_f16_nt_plan(7, 9, 3)["copy_bytes"] == 2      # odd K: 2-byte copies
        assert pws.gemm_f16_nt_plan(64, 64, 12)["copy_bytes"] == 8   # K % 4 == 0, not % 8
        assert pws.gemm_f16_nt_plan(64, 64, 16, lhs_ptr=A + 2)["copy_bytes"] == 2
        assert pws.gemm_f16_nt_plan(64, 64, 16, lhs_ptr=A + 8)["copy_bytes"] == 8
        assert pws.gemm_f16_nt_plan(64, 64, 16)["producer"] == 1     # forced even when aligned
    finally:
        pws.gemm_set_debug_flags(0)
    with pytest.raises(pws.GemmError):
        pws.gemm_f16_nt_plan(64, 64, 16, stages=9)
    pws.gemm_set_debug_flags(pws.GEMM_DEBUG_FORCE_PAIR_TILE)
    try:
        assert pws.gemm_f16_nt_plan(300, 300, 64)["cta_group"] == 2
        assert pws.gemm_f16_nt_plan(300, 300, 66)["cta_group"] == 2   # repacked, or read in place, on the pair tile
    finally:
        pws.gemm_set_debug_flags(0)
    pws.gemm_set_debug_flags(pws.GEMM_DEBUG_FORCE_PAIR_TILE | pws.GEMM_DEBUG_FORCE_COPY_PRODUCER)
    try:
        assert pws.gemm_f16_nt_plan(300, 300, 66)["cta_group"] == 1   # copy producer: single CTA
    finally:
        pws.gemm_set_debug_flags(0)


def test_binding_rejects_bad_tensors():
    torch = pytest.importorskip("torch")
    with pytest.raises(TypeError):
        pws.gemm_f16_nt(torch.zeros(2, 2, dtype=torch.float32), torch.zeros(2, 2, dtype=torch.float32))
    with pytest.raises(ValueError):
        pws.gemm_s32_nn(torch.zeros(2, 3, dtype=torch.int32), torch.zeros(2, 3, dtype=torch.int32))
    with pytest.raises(ValueError):   # CPU tensors are refused, never computed on the host
        pws.gemm_f16_nt(torch.zeros(2, 2, dtype=torch.float16), torch.zeros(2, 2, dtype=torch.float16))
