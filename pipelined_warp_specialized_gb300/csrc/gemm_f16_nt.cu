// gemm_f16_nt.cu -- out[M,N] = f16( lhs[M,K] . rhs[N,K]^T ) on the 5th-generation
// tensor cores of sm_103a.
//
// The pipeline is the 1P1C kernel of the Croqtile tutorial ch.6, section
// "带 event 的 1P1C 内核", re-built for tcgen05/TMEM/TMA:
//
//   * ring      -- S shared-memory slots, each holding one 64-wide K strip of
//                  the A tile and of the B tile, laid out in the 128-byte
//                  swizzle that both the TMA and the tensor-core descriptors
//                  use.  Slot for K block k is stage = k % S ("环形索引").
//   * events    -- full[s] / empty[s] mbarriers, one pair per slot.  full[s]
//                  counts the transaction bytes of the slot's copies
//                  (expect-tx), empty[s] is arrived by the tensor-core
//                  commit.  Lap l of a slot is waited with parity l mod 2
//                  (TileLang tutorial ch.22, section 3.2).
//   * producer  -- one warp (one elected thread) issues the TMA copies:
//                  wait empty[s], arm full[s] with the byte count, copy A and
//                  B strips into slot s.  Where TMA cannot address the
//                  operands (rows not 16-byte aligned), the host first
//                  copies them to aligned rows (the library's fixed array or
//                  pooled scratch); where that is not possible, eight warps
//                  fill the same swizzled layout themselves -- aligned
//                  16-byte loads shifted into place in registers -- and
//                  arrive on full[s] once their stores have been fenced to
//                  the async proxy (CUDA tutorial ch.4, section 4.8.1).
//   * consumer  -- one warp (one elected thread) seeds every empty[s] once
//                  before its loop ("foreach {s} in [MATMUL_STAGES] trigger
//                  empty[s]"), then per K block waits full[s], issues four
//                  tcgen05.mma (K = 16 each; eight for the wide tile) into an
//                  fp32 accumulator in tensor memory, and commits to
//                  empty[s] -- the commit is
//                  the "mma.commit" fence: the slot is released only once the
//                  multiplies reading it have completed.
//   * epilogue  -- four warps, one per 32-lane quarter of tensor memory
//                  (eight, two per quarter, for the wide tile), wait for the
//                  accumulator, read it with tcgen05.ld, round to f16
//                  (nearest even), stage 32 x 64 blocks in swizzled shared
//                  memory and store them with TMA (clipped at M and N), or
//                  with guarded plain stores where TMA cannot address `out`.
//
// The kernel is persistent (the Croqtile tutorial ch.5 "持久调度与 if 守卫"):
// a fixed grid strides over work units (output tiles, or half tiles in a
// partial last wave), and the accumulator is double buffered in tensor memory
// so the epilogue of unit i overlaps the main loop of unit i+1 (two more
// event pairs, tmem_full[2] / tmem_empty[2], seeded by the epilogue warps the
// same way).
//
// Three tile shapes share the code.  A CTA pair (cta_group::2) computes
// 256 x 256 (each CTA loading its own 128 rows of A and 128 rows of B -- no
// multicast), or, for rings of up to four slots, 256 x 512 with two B boxes
// per slot and one 512-column accumulator drained in two halves; a single CTA
// computes 128 x 128.  The tile is chosen from the shape and S alone, and
// every tile sums each output element over K in the same order.
//
// Small outputs with a long K split it instead: a cluster of two single CTAs
// per 128 x 128 tile, each summing one K half into its own accumulator; the
// two fp32 partial sums meet over distributed shared memory and are added
// once before the rounding.  That choice reads M, N and K only.
//
// Grids are launched as programmatic dependents: set-up (barriers, tensor
// memory, cluster) overlaps the previous grid on the stream, and global
// memory is touched only once that grid has completed.
//
// Every wait is bounded (wait_timeout_ns); a role that gives up records a
// timeout in the status word of the call's stream, raises a CTA-local abort flag that
// the other roles poll, and every role then runs the common exit path, so
// the kernel always returns.  Waits that last about one K block (the ring's)
// count the limit from their start; the waits that last a whole K loop (a
// finished accumulator, the K split's partial sums) count it from the last K
// block the producer issued, so they end on a stall, not on a long K.
#include <cstdint>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "pwsgemm.h"

namespace pws {
namespace f16nt {

constexpr int BK = 64;                 // K per ring slot: 64 f16 = one 128-byte swizzle row
constexpr int UMMA_K = 16;             // K per tcgen05.mma of kind::f16
constexpr int BM_CTA = 128;            // A rows per CTA (tensor-memory lanes)
constexpr int BN_CTA = 128;            // B rows per CTA
constexpr int A_SLOT = BM_CTA * BK * 2;
constexpr int B_SLOT = BN_CTA * BK * 2;
constexpr int EPI_WARPS = 4;           // epilogue warps: one per tensor-memory lane quarter, two staging buffers each
constexpr int EPI_WARPS_WIDE = 8;      // the wide tile's: two per lane quarter, one staging buffer each
constexpr int EPI_COLS = 64;           // output columns per epilogue chunk (128 bytes of f16)
constexpr int EPI_BUF = 32 * EPI_COLS * 2;     // 32 rows x 64 columns
constexpr int EPI_BYTES = EPI_WARPS * 2 * EPI_BUF;
static_assert(EPI_WARPS_WIDE * EPI_BUF == EPI_BYTES, "both epilogue forms use the same staging bytes");
// The wide tile fed by TMA drains with eight warps (two per lane quarter, a
// half of the chunks each); fed by the realigning producer it drains with
// four, leaving the registers of a 13-warp block to the producer's loads.
template <int NW, int PK>
constexpr int epi_warps() { return NW == 2 && PK == 0 ? EPI_WARPS_WIDE : EPI_WARPS; }
constexpr int MAX_STAGES = 6;
constexpr int COPY_WARPS = 8;          // producer warps of the realigning and cp.async producers
constexpr int COPY_THREADS = COPY_WARPS * 32;
#ifndef PWS_GROUP_M
#define PWS_GROUP_M 8
#endif
constexpr int GROUP_M = PWS_GROUP_M;   // tile-row group height of the raster order

// kProducerRealign: aligned 16-byte loads shifted into place, any tile (the
// plan query reports the repack path as 2)
enum { kProducerTma = 0, kProducerCopy = 1, kProducerRealign = 3 };
enum { kStoreTma = 0, kStoreDirect = 1 };

struct Params {
    int M, N, K;
    int num_kb;                 // K blocks: cdiv(K, BK)
    int tiles_m, tiles_n, num_tiles;
    int producer;               // kProducerTma / kProducerCopy / kProducerRealign
    int copy_bytes;             // cp.async granularity (8, 4) or 2 (plain loads)
    int store;                  // kStoreTma / kStoreDirect
    unsigned flags;             // GEMM_DEBUG_* bits
    unsigned long long timeout_ns;
    const __half* lhs;
    const __half* rhs;
    __half* out;
    unsigned* status;
    // Work units: units 0 .. full_units-1 are whole output tiles (unit = tile).
    // With split == 2, each remaining tile (those of the last, partial wave)
    // is cut into two units, its left and right halves of columns, which run
    // the full K loop (no partial sums to combine): with a half-width MMA, or
    // for the wide tile with one of its two MMAs.
    int full_units;
    int split;
    int total_units;
    // K split (single-CTA tile only): 2 = each tile is computed by a cluster
    // of two CTAs, rank r summing its K blocks [kb0(r), kb1(r)) -- the first
    // ceil(num_kb / 2) blocks, or the rest -- and the two fp32 partial tiles
    // are added once before rounding.  One tile per cluster, no persistence.
    int ksplit;
};

// NW = MMAs per K step, each UMMA_N columns wide.  NW = 1: the accumulator is
// double buffered.  NW = 2 (CTA pair only, "wide" 256 x 512 tile): one
// accumulator fills all 512 tensor-memory columns and each slot carries two B
// boxes, so every byte copied into shared memory feeds 4/3 as many flops.
template <int CG, int NW = 1>
struct Shape {
    static constexpr int UMMA_M = BM_CTA * CG;        // tile rows (per CTA group)
    static constexpr int UMMA_N = BN_CTA * CG;        // columns per MMA
    static constexpr int TILE_N = UMMA_N * NW;        // tile columns
    static constexpr int ACC_COLS = TILE_N;           // fp32 columns per accumulator
    static constexpr int NBUF = NW == 1 ? 2 : 1;      // accumulator buffers
    static constexpr int TMEM_COLS = NBUF * ACC_COLS;
    // a split (half-width) unit covers HALF_N columns of its tile
    static constexpr int HALF_N = NW == 1 ? UMMA_N / 2 : UMMA_N;
    static_assert(TMEM_COLS <= 512, "tensor memory holds 512 columns");
};

// Shared-memory carve-up (offsets from a 1024-byte aligned base).  A slot
// holds KB 64-wide K boxes of each operand: slot s holds A box j at
// A + s * A_STRIDE + j * A_SLOT and B box j at B + s * B_STRIDE + j * B_BOX,
// or, for the wide tile (KB = 1), its NW B boxes at B + s * B_STRIDE + h * B_SLOT.
// KB = 4 serves half-width units only (every unit of the launch is one):
// their B boxes are 64 rows, half a B_SLOT, so four boxes of each operand fit
// where three full ones would.
template <int S, int NW = 1, int KB = 1>
struct Layout {
    static constexpr int B_BOX = KB == 4 ? B_SLOT / 2 : B_SLOT;
    static constexpr int A_STRIDE = KB * A_SLOT;
    static constexpr int B_STRIDE = NW * KB * B_BOX;
    static constexpr int A = 0;
    static constexpr int B = S * A_STRIDE;
    static constexpr int EPI = S * (A_STRIDE + B_STRIDE);
    static constexpr int BAR = EPI + EPI_BYTES;
    static constexpr int FULL = BAR;
    static constexpr int EMPTY = FULL + 8 * S;
    static constexpr int TFULL = EMPTY + 8 * S;
    static constexpr int TEMPTY = TFULL + 16;
    static constexpr int DRAIN = TEMPTY + 16;
    static constexpr int RECV = DRAIN + 8;                   // K split: a peer warp's partial rows are staged (x2)
    static constexpr int TMEM_SLOT = RECV + 16;
    static constexpr int ABORT = TMEM_SLOT + 4;
    static constexpr int PROGRESS = ABORT + 4;               // K blocks this CTA's producer has issued
    static constexpr int END = PROGRESS + 4;
    static constexpr int BYTES = END + 1024;                // + alignment slack
    // at least ~half the SM's shared memory so only one CTA is resident per SM
    // (each CTA owns up to all 512 tensor-memory columns)
    static constexpr int DYN = BYTES > 120 * 1024 ? BYTES : 120 * 1024;
};

// Instruction descriptor of tcgen05.mma kind::f16: D fp32, A and B f16, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
template <int M_, int N_>
constexpr uint32_t make_idesc() {
    return (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) | (0u << 16) |
           (static_cast<uint32_t>(N_ >> 3) << 17) | (static_cast<uint32_t>(M_ >> 4) << 24);
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle: rows of 128 bytes, 8-row atoms of 1024 bytes (stride-dimension
// offset), start address >> 4 in bits 0..13, descriptor version 1 at bit 46,
// layout "128-byte swizzle" (2) at bit 61.  Advancing K by 16 elements moves
// the start address by 32 bytes inside the swizzle row.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(16u >> 4) << 16;     // leading-dimension offset (unused here)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;   // stride-dimension offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Output tile of persistent work item `t`: tile rows are grouped GROUP_M at a
// time so the CTAs working at the same moment share A and B strips in L2,
// and odd groups walk the tile columns right to left, so a group starts on
// the B columns the previous one used last (on GB300: 7.7 % fewer DRAM bytes
// at 8192^3 with the wide tile).
__device__ __forceinline__ void tile_coords(int t, const Params& p, int& tm, int& tn) {
    const int group = GROUP_M * p.tiles_n;
    const int g = t / group;
    const int first = g * GROUP_M;
    const int rows = min(p.tiles_m - first, GROUP_M);
    const int r = t - g * group;
    tm = first + r % rows;
    tn = r / rows;
    if (g & 1) tn = p.tiles_n - 1 - tn;
}

// One persistent work unit: an output tile, or (half = 0 or 1) the left or
// right half of its columns.
struct Unit {
    int tile, half;
};

__device__ __forceinline__ Unit unit_of(int u, const Params& p) {
    if (p.split < 2 || u < p.full_units) return Unit{u, -1};
    const int v = u - p.full_units;
    return Unit{p.full_units + v / 2, v % 2};
}

// Bounded mbarrier wait.  Returns false if the wait gave up (time limit or
// another role's abort); the first role to give up records the timeout.
struct Waiter {
    unsigned long long timeout_ns;
    volatile uint32_t* abort;
    unsigned* status;
    unsigned role;

    template <bool CLUSTER_SCOPE = false>
    __device__ __forceinline__ bool probe(uint32_t bar, uint32_t parity) const {
        return CLUSTER_SCOPE ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    }

    __device__ __forceinline__ bool give_up() const {
        *abort = 1u;
        atomicOr(status, kStatusTimeout | role);
        return false;
    }

    // A wait that lasts about one K block (the ring's, the accumulator
    // hand-over's): the limit counts from the start of the wait.
    template <bool CLUSTER_SCOPE = false>
    __device__ bool wait(uint32_t bar, uint32_t parity) const {
        return wait_inline<CLUSTER_SCOPE>(bar, parity);
    }

    // The same, inlined into the caller: for a caller holding many registers
    // across the wait (the realigning producer's loads in flight).
    template <bool CLUSTER_SCOPE = false>
    __device__ __forceinline__ bool wait_inline(uint32_t bar, uint32_t parity) const {
        if (probe<CLUSTER_SCOPE>(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            if (probe<CLUSTER_SCOPE>(bar, parity)) return true;
            if (*abort) return false;
            if (globaltimer_ns() - t0 > timeout_ns) return give_up();
        }
    }

    // A wait that legitimately lasts a whole K loop: the epilogue's wait for
    // a finished accumulator, and the K split's wait for the peer's partial
    // sums.  The limit counts from the last change of the progress counter
    // that the producer of the CTA being waited for bumps once per K block
    // (`remote`: the counter lives in the other CTA of the cluster), so such
    // a wait gives up on a stall -- no K block issued for the whole limit --
    // and never on a long but live loop.  After the producer's last block the
    // wait still has to cover at most S blocks of multiplies and a drain.
    template <bool CLUSTER_SCOPE = false>
    __device__ bool wait_progress(uint32_t bar, uint32_t parity, uint32_t progress, bool remote) const {
        if (probe<CLUSTER_SCOPE>(bar, parity)) return true;
        uint64_t t0 = globaltimer_ns();
        uint32_t seen = remote ? ld_relaxed_cluster_u32(progress) : ld_volatile_shared_u32(progress);
        for (;;) {
            if (probe<CLUSTER_SCOPE>(bar, parity)) return true;
            if (*abort) return false;
            const uint32_t now_seen = remote ? ld_relaxed_cluster_u32(progress) : ld_volatile_shared_u32(progress);
            const uint64_t now = globaltimer_ns();
            if (now_seen != seen) {
                seen = now_seen;
                t0 = now;
            } else if (now - t0 > timeout_ns) {
                return give_up();
            }
        }
    }
};

__device__ __forceinline__ uint32_t pack_half2(uint32_t lo_bits, uint32_t hi_bits) {
    const __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// ---------------------------------------------------------------- copy producer
//
// Fills ring slots with cp.async where no tensor map can describe the
// operands (rows not a multiple of 16 bytes, or an unaligned base).  The
// slot layout is exactly the one TMA writes: row r of the strip at r * 128
// bytes, 16-byte chunk c of the row at chunk (c ^ (r mod 8)).  Copies are G
// bytes (8 or 4 with cp.async and zero fill; 2 with plain loads and stores).
template <int G>
struct CopyShape {
    static constexpr int E = G / 2;                      // f16 per copy
    static constexpr int CPR = 128 / G;                  // copies per 128-byte row
    static constexpr int RPJ = COPY_THREADS / CPR;       // rows covered by one sweep of the threads
    static constexpr int J = BM_CTA / RPJ;               // sweeps per 128-row strip
    static_assert(COPY_THREADS % CPR == 0 && BM_CTA % RPJ == 0, "copy mapping");
};

// One 64-wide K strip of 128 rows of one operand into the slot at `slot`.
// Thread t copies column (t mod CPR) of rows t / CPR + j * RPJ.
template <int G>
__device__ __forceinline__ void copy_strip(uint32_t slot, const __half* base, int rows_total, int row0, int K,
                                           int k0, int t) {
    using C = CopyShape<G>;
    const int col = t % C::CPR;
    const int rr0 = t / C::CPR;
    const int k = k0 + col * C::E;
    const uint32_t in_row = static_cast<uint32_t>(col * G);
    const bool kval = k < K;
    const int64_t row_step = static_cast<int64_t>(C::RPJ) * K;
    const __half* src0 = base + static_cast<int64_t>(row0 + rr0) * K + k;
    if constexpr (G == 2) {
        unsigned short v[C::J];
#pragma unroll
        for (int j = 0; j < C::J; ++j) {
            const bool ok = kval && row0 + rr0 + j * C::RPJ < rows_total;
            v[j] = ok ? __ldg(reinterpret_cast<const unsigned short*>(src0 + j * row_step)) : (unsigned short)0;
        }
#pragma unroll
        for (int j = 0; j < C::J; ++j) {
            const int rr = rr0 + j * C::RPJ;
            const uint32_t dst = slot + rr * 128 + (((in_row >> 4) ^ static_cast<uint32_t>(rr & 7)) << 4) + (in_row & 15u);
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(dst), "h"(v[j]) : "memory");
        }
    } else {
#pragma unroll
        for (int j = 0; j < C::J; ++j) {
            const int rr = rr0 + j * C::RPJ;
            const bool ok = kval && row0 + rr < rows_total;
            const __half* src = ok ? src0 + j * row_step : base;
            const uint32_t dst = slot + rr * 128 + (((in_row >> 4) ^ static_cast<uint32_t>(rr & 7)) << 4) + (in_row & 15u);
            cp_async<G>(dst, src, ok ? static_cast<uint32_t>(G) : 0u);
        }
    }
}

// The producer loop of the copy path.  Each thread's copies of K block k form
// one cp.async group; the slot of block k is signalled LAG blocks later, once
// the thread's groups up to k have landed (cp.async.wait_group), after a proxy
// fence (the tensor core reads through the async proxy) and a warp barrier,
// by one arrive per warp.  The MMA thread takes GROUP slots at a time (2 when
// S = 6), so LAG = S - GROUP keeps the ring live: the wait on empty for block
// k needs block k - S consumed, which needs full signalled up to block
// k - S + GROUP - 1.
template <int G, int S>
__device__ void copy_producer(const Params& p, const Waiter& W, uint32_t sA, uint32_t sB, uint32_t bFULL,
                              uint32_t bEMPTY, uint32_t progress, int cluster_id, int num_clusters, int kb0, int kb1,
                              int lane) {
    constexpr int LAG = S - (S >= 6 ? 2 : 1);
    const int t = threadIdx.x;                   // 0 .. COPY_THREADS - 1
    uint32_t stage = 0, phase = 0, issued = 0, signalled = 0;
    bool ok = true;
    for (int u = cluster_id; ok && u < p.total_units; u += num_clusters) {
        const Unit un = unit_of(u, p);
        int tm, tn;
        tile_coords(un.tile, p, tm, tn);
        for (int kb = kb0; kb < kb1; ++kb) {
            bool got = true;
            if (lane == 0) got = W.wait(bEMPTY + 8 * stage, phase);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) { ok = false; break; }
            copy_strip<G>(sA + stage * A_SLOT, p.lhs, p.M, tm * BM_CTA, p.K, kb * BK, t);
            copy_strip<G>(sB + stage * B_SLOT, p.rhs, p.N, tn * BN_CTA, p.K, kb * BK, t);
            cp_async_commit();
            ++issued;
            if (t == 0) st_volatile_shared_u32(progress, issued);
            if (issued - signalled > static_cast<uint32_t>(LAG)) {
                cp_async_wait_group<LAG>();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bFULL + 8 * (signalled % S));
                ++signalled;
            }
            if (++stage == S) { stage = 0; phase ^= 1u; }
        }
    }
    cp_async_wait_group<0>();
    if (ok) {
        fence_proxy_async_smem();
        __syncwarp();
        for (; signalled < issued; ++signalled)
            if (lane == 0) mbar_arrive(bFULL + 8 * (signalled % S));
    }
}

// ---------------------------------------------------------------- realigning producer
//
// Reads the operands in place where no tensor map can describe them (rows
// not a multiple of 16 bytes apart, or a base not 16-byte aligned) and writes
// the slot layout TMA writes, so any tile can use it and nothing is copied
// to scratch memory.  Partial tiles follow the pages' cdiv and if guards
// (Croqtile tutorial ch.6 "带 event 的 1P1C 内核", ch.5 "以 if 实现谓词执行"):
// rows past M or N and columns past K are written as zeros.
//
// A warp operation covers 4 rows of a strip, 8 lanes per row, each lane one
// 16-byte chunk of the row's 64-element K strip.  Its 4 rows are 8 rows
// apart: strip row i = c + 8 j, with class c = i mod 8.  A strip starts at a
// multiple of 64 rows and 8 rows span 16 K bytes, so every row of class c
// starts (base + 2 c K) mod 16 bytes past a 16-byte boundary in every strip
// and K block.  The 4 rows of an operation therefore share one shift, taken
// by a warp-uniform switch, and the 128-byte swizzle of their chunks (chunk
// XOR row mod 8) is the chunk index XOR c.  Each lane loads the aligned
// 16-byte block holding the start of its chunk and, unless the shift is zero,
// the next one, and shifts the chunk into place; each block read holds a
// byte the chunk needs, so no load leaves the operand's pages.
//
// A warp issues the loads of a batch of its operations before it waits for
// the slot (registers, not shared memory, hold them), then writes them; the
// slot is signalled after a proxy fence (the tensor core reads through the
// async proxy) with one arrive per warp -- on the leader CTA's full[s], at
// cluster scope, for a CTA pair.

// Bytes SH .. SH+15 of the 32 bytes lo | hi (little-endian), SH even.
template <int SH>
__device__ __forceinline__ uint4 shift_chunk(const uint4& lo, const uint4& hi) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    constexpr int q = SH / 4, r = SH % 4;
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = r == 0 ? w[i + q] : __funnelshift_r(w[i + q], w[i + q + 1], 8 * r);
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint4 shift_chunk_any(const uint4& lo, const uint4& hi, int sh) {
    switch (sh) {
        case 0: return lo;
        case 2: return shift_chunk<2>(lo, hi);
        case 4: return shift_chunk<4>(lo, hi);
        case 6: return shift_chunk<6>(lo, hi);
        case 8: return shift_chunk<8>(lo, hi);
        case 10: return shift_chunk<10>(lo, hi);
        case 12: return shift_chunk<12>(lo, hi);
        default: return shift_chunk<14>(lo, hi);
    }
}

// One unit's K loop of the realigning producer.  NOPS operations per warp
// and K block: the 4 of A's strip (operations w, w + 8, w + 16, w + 24 of its
// 32), then those of the B boxes; SMALL: one 64-row B box (half-width unit of
// the 256 x 256 / 128 x 128 tiles, 16 operations, class (w >> 1) + 4 i), else
// 128-row boxes (class (w >> 2) + 2 i, box h = i / 4).  Every per-operation
// quantity is a compile-time multiple of a per-lane term.  Returns false if
// a wait gave up.
template <int CG, int NW, int S, int NOPS, bool SMALL>
__device__ __forceinline__ bool realign_unit(const Params& p, const Waiter& W, uint32_t sA, uint32_t sB,
                                             uint32_t full_addr, uint32_t bEMPTY, uint32_t progress, int kb0,
                                             int kb1, int m_cta, int n_cta, uint32_t shA, uint32_t shB, int warp,
                                             int lane, uint32_t& stage, uint32_t& phase, uint32_t& issued) {
    using SH = Shape<CG, NW>;
    using L = Layout<S, NW>;
    const int r4 = lane >> 3, cl = lane & 7;
    const uint64_t rb = 2ull * static_cast<uint32_t>(p.K);          // bytes between rows
    // A (and 128-row B boxes): class c0 + 2 i, rows 8 j + class
    const int jA = 4 * (warp & 3) + r4, c0A = warp >> 2;
    // a 64-row B box: class c0 + 4 i
    const int jB = SMALL ? 4 * (warp & 1) + r4 : jA, c0B = SMALL ? warp >> 1 : c0A;
    const int rowA = m_cta + c0A + 8 * jA, rowB = n_cta + c0B + 8 * jB;
    const uintptr_t pA = reinterpret_cast<uintptr_t>(p.lhs) + static_cast<uintptr_t>(static_cast<uint64_t>(rowA) * rb);
    const uintptr_t pB = reinterpret_cast<uintptr_t>(p.rhs) + static_cast<uintptr_t>(static_cast<uint64_t>(rowB) * rb);
    const uint32_t dA = static_cast<uint32_t>(c0A + 8 * jA) * 128u, dB = static_cast<uint32_t>(c0B + 8 * jB) * 128u;
    const uint32_t xA = static_cast<uint32_t>(cl ^ c0A) << 4, xB = static_cast<uint32_t>(cl ^ c0B) << 4;
    const uint32_t shA0 = shA >> (4 * c0A), shB0 = shB >> (4 * c0B);
    for (int kb = kb0; kb < kb1; ++kb) {
        const int vb = min(2 * (p.K - kb * BK), 2 * BK);             // bytes of each row in this K block
        const uintptr_t koff = static_cast<uintptr_t>(kb) * (2 * BK);
        const uint32_t slotA = sA + stage * A_SLOT, slotB = sB + stage * L::B_STRIDE;
        const bool lo_in = 16 * cl < vb;
        uint4 lo[NOPS], hi[NOPS];
        // the loads of the whole K block first: they touch no shared memory,
        // so they are in flight while the warp waits for the slot
#pragma unroll
        for (int i = 0; i < NOPS; ++i) {
            const bool is_a = i < 4;
            const int q = is_a ? i : (SMALL ? i - 4 : (i - 4) & 3);
            const int h = is_a || SMALL ? 0 : (i - 4) >> 2;
            const int cstep = !is_a && SMALL ? 4 : 2;
            const int roff = h * SH::UMMA_N + cstep * q;
            const int sh = static_cast<int>(((is_a ? shA0 : shB0) >> (4 * cstep * q)) & 15u);
            const bool row_ok = is_a ? rowA + roff < p.M : rowB + roff < p.N;
            const uintptr_t src = (is_a ? pA : pB) + static_cast<uintptr_t>(static_cast<uint64_t>(roff) * rb) + koff;
            const uint4* blk = reinterpret_cast<const uint4*>(src - static_cast<uintptr_t>(sh)) + cl;
            lo[i] = make_uint4(0u, 0u, 0u, 0u);
            hi[i] = make_uint4(0u, 0u, 0u, 0u);
            if (row_ok && lo_in) lo[i] = __ldg(blk);
            if (row_ok && sh != 0 && 16 * (cl + 1) < sh + vb) hi[i] = __ldg(blk + 1);
        }
        bool got = true;
        if (lane == 0) got = W.wait_inline(bEMPTY + 8 * stage, phase);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) return false;
        const int rem = vb - 16 * cl;                                 // bytes of the chunk inside K
#pragma unroll
        for (int i = 0; i < NOPS; ++i) {
            const bool is_a = i < 4;
            const int q = is_a ? i : (SMALL ? i - 4 : (i - 4) & 3);
            const int h = is_a || SMALL ? 0 : (i - 4) >> 2;
            const int cstep = !is_a && SMALL ? 4 : 2;
            const int sh = static_cast<int>(((is_a ? shA0 : shB0) >> (4 * cstep * q)) & 15u);
            // strip row c + 8 j at 128 (c + 8 j); chunk cl at (cl ^ c) -- with
            // c = c0 + cstep q, cl ^ c = (cl ^ c0) ^ (cstep q)
            const uint32_t dst = (is_a ? slotA + dA : slotB + h * B_SLOT + dB) + static_cast<uint32_t>(cstep * q) * 128u +
                                 ((is_a ? xA : xB) ^ (static_cast<uint32_t>(cstep * q) << 4));
            uint4 o = shift_chunk_any(lo[i], hi[i], sh);
            if (rem < 16) {
                // the K tail: elements past K are zero
                uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = 4 * e + 4 <= rem ? w[e] : (4 * e + 2 == rem ? (w[e] & 0xFFFFu) : 0u);
                o = make_uint4(w[0], w[1], w[2], w[3]);
            }
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(o.x), "r"(o.y), "r"(o.z),
                         "r"(o.w)
                         : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if constexpr (CG == 1) mbar_arrive(full_addr + 8 * stage);
            else mbar_arrive_cluster(full_addr + 8 * stage);
        }
        ++issued;
        if (warp == 0 && lane == 0) st_volatile_shared_u32(progress, issued);
        if (++stage == S) { stage = 0; phase ^= 1u; }
    }
    return true;
}

template <int CG, int NW, int S>
__device__ void realign_producer(const Params& p, const Waiter& W, uint32_t sA, uint32_t sB, uint32_t bFULL,
                                 uint32_t bEMPTY, uint32_t progress, int cluster_id, int num_clusters, int kb0,
                                 int kb1, uint32_t rank, int warp, int lane) {
    using SH = Shape<CG, NW>;
    static_assert(COPY_WARPS == 8, "operation mapping: warp w takes operations w, w + 8, ...");
    const uint32_t full_addr = (CG == 2) ? mapa_shared(bFULL, 0) : bFULL;
    const uintptr_t a_base = reinterpret_cast<uintptr_t>(p.lhs), b_base = reinterpret_cast<uintptr_t>(p.rhs);
    const uint64_t rb = 2ull * static_cast<uint32_t>(p.K);
    // shift of the rows of class c (row mod 8) past a 16-byte boundary, 4 bits per class
    uint32_t shA = 0u, shB = 0u;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        shA |= static_cast<uint32_t>((a_base + static_cast<uintptr_t>(c * rb)) & 15u) << (4 * c);
        shB |= static_cast<uint32_t>((b_base + static_cast<uintptr_t>(c * rb)) & 15u) << (4 * c);
    }
    uint32_t stage = 0, phase = 0, issued = 0;
    for (int u = cluster_id; u < p.total_units; u += num_clusters) {
        const Unit un = unit_of(u, p);
        int tm, tn;
        tile_coords(un.tile, p, tm, tn);
        const bool halfw = un.half >= 0;
        const int m_cta = tm * SH::UMMA_M + static_cast<int>(rank) * BM_CTA;
        const int n_unit = tn * SH::TILE_N + (halfw ? un.half * SH::HALF_N : 0);
        bool ok;
        if (NW == 1 && halfw) {
            const int n_cta = n_unit + static_cast<int>(rank) * (BN_CTA / 2);
            ok = realign_unit<CG, NW, S, 6, true>(p, W, sA, sB, full_addr, bEMPTY, progress, kb0, kb1, m_cta, n_cta,
                                                  shA, shB, warp, lane, stage, phase, issued);
        } else if (NW == 2 && !halfw) {
            const int n_cta = n_unit + static_cast<int>(rank) * BN_CTA;
            ok = realign_unit<CG, NW, S, 12, false>(p, W, sA, sB, full_addr, bEMPTY, progress, kb0, kb1, m_cta,
                                                    n_cta, shA, shB, warp, lane, stage, phase, issued);
        } else {
            const int n_cta = n_unit + static_cast<int>(rank) * BN_CTA;
            ok = realign_unit<CG, NW, S, 8, false>(p, W, sA, sB, full_addr, bEMPTY, progress, kb0, kb1, m_cta, n_cta,
                                                   shA, shB, warp, lane, stage, phase, issued);
        }
        if (!ok) return;
    }
}

// PK = 1: launched with COPY_WARPS producer warps (the cp.async or the
// realigning producer), PK = 0: with one (TMA).  Single-CTA kernels serve
// every producer with one bound; a CTA pair has a kernel per producer kind,
// so the TMA one keeps the registers eight producer warps would take.
//
// KB = 2, 3 or 4 (single-CTA tile, TMA): each slot holds KB 64-wide K boxes
// of each operand, so a latency-bound K loop runs 1/KB as many slot round
// trips; the multiplies keep their K order, so the result bits do not
// change.  KB = 4 is for launches whose units are all half-width (the B
// boxes are half size).
template <int CG, int S, int NW, int PK, int KB = 1>
__global__ void __launch_bounds__(((CG == 1 || PK == 1 ? COPY_WARPS : 1) + 1 + epi_warps<NW, PK>()) * 32, 1)
gemm_f16_nt_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ Params p) {
    static_assert(NW == 1 || CG == 2, "the wide tile is a CTA-pair tile");
    using SH = Shape<CG, NW>;
    using L = Layout<S, NW, KB>;
    static_assert(KB == 1 || (CG == 1 && NW == 1 && PK == 0), "multi-box slots: single-CTA TMA tile only");
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const gbase = smem_raw + (base - raw);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    constexpr int EW = epi_warps<NW, PK>();
    const int P = static_cast<int>(blockDim.x / 32) - 1 - EW;          // producer warps
    const int mma_warp = P;
    const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
    // K split: a cluster of two single CTAs per tile; krank picks the K half
    const bool kpair = CG == 1 && p.ksplit == 2;
    const uint32_t krank = kpair ? cluster_ctarank() : 0u;
    const int csize = (CG == 2 || kpair) ? 2 : 1;
    const int cluster_id = blockIdx.x / csize;
    const int num_clusters = gridDim.x / csize;
    const int kb_mid = (p.num_kb + 1) / 2;
    const int kb0 = kpair && krank != 0 ? kb_mid : 0;
    const int kb1 = kpair && krank == 0 ? kb_mid : p.num_kb;

    const uint32_t sA = base + L::A, sB = base + L::B, sEPI = base + L::EPI;
    const uint32_t bFULL = base + L::FULL, bEMPTY = base + L::EMPTY;
    const uint32_t bTFULL = base + L::TFULL, bTEMPTY = base + L::TEMPTY, bDRAIN = base + L::DRAIN;
    const uint32_t bRECV = base + L::RECV;
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + L::ABORT);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::TMEM_SLOT);
    const uint32_t sPROGRESS = base + L::PROGRESS;

    // ------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        // TMA: one arrive.expect_tx per phase; otherwise one arrive per
        // producer warp (of both CTAs of a pair)
        const uint32_t full_count = p.producer == kProducerTma ? 1u : static_cast<uint32_t>(P * CG);
        for (int s = 0; s < S; ++s) {
            mbar_init(bFULL + 8 * s, full_count);
            mbar_init(bEMPTY + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bTFULL + 8 * b, 1);
            mbar_init(bTEMPTY + 8 * b, EW * CG);
        }
        mbar_init(bDRAIN, 1);
        // K split: the 32 lanes of the peer's warp for lane quarter 2*krank + j
        for (int j = 0; j < 2; ++j) mbar_init(bRECV + 8 * j, 32);
        *abort_flag = 0u;
        *reinterpret_cast<volatile uint32_t*>(gbase + L::PROGRESS) = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0 && p.producer == kProducerTma) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (p.store == kStoreTma) tma_prefetch_desc(&tmC);
    }
    if (warp == mma_warp) {
        tmem_alloc<CG>(base + L::TMEM_SLOT, SH::TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    __syncthreads();
    // A pair's peer issues MMAs into this CTA's tensor memory and copies
    // against its barriers: it must see them set up.  The K split's first
    // cross-CTA access comes only after the main loop (the epilogue's), so
    // its threads arrive here and wait later (the epilogue warps before their
    // loop, the others at tear-down), out of the way of the first loads.
    if (CG == 2) cluster_sync();
    else if (kpair) cluster_arrive_release();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Launched as a programmatic dependent: everything above (barriers, tensor
    // memory, cluster) overlapped the previous grid's tail; global memory is
    // touched only after that grid's writes are visible.  The next grid may
    // start its own set-up as soon as SMs free up.
    grid_dependency_wait();
    allow_dependent_launch();

    const bool is_leader = (CG == 1) || rank == 0;

    if (warp < P) {
        // ======================================================== producer
        if (p.producer == kProducerTma) {
            if (lane == 0) {
                const Waiter W{p.timeout_ns, abort_flag, p.status, kStatusRoleProducer};
                // the slot's full barrier lives in the leader CTA of a pair
                const uint32_t full_leader = (CG == 2) ? mapa_shared(bFULL, 0) : bFULL;
                uint32_t stage = 0, phase = 0;
                uint32_t issued = 0;
                bool ok = true;
                for (int u = cluster_id; ok && u < p.total_units; u += num_clusters) {
                    const Unit un = unit_of(u, p);
                    int tm, tn;
                    tile_coords(un.tile, p, tm, tn);
                    const int m_cta = tm * SH::UMMA_M + static_cast<int>(rank) * BM_CTA;
                    const bool halfw = un.half >= 0;
                    // NW = 1: a half-width unit loads half of the CTA's B rows
                    // (tmBh: a 64-row box).  NW = 2: box h of the CTA's B rows
                    // starts at column h * UMMA_N of the unit; a half-width unit
                    // is one such box.
                    const int n_unit = tn * SH::TILE_N + (halfw ? un.half * SH::HALF_N : 0);
                    const int n_cta = n_unit + static_cast<int>(rank) * (NW == 1 && halfw ? BN_CTA / 2 : BN_CTA);
                    const CUtensorMap* tb = NW == 1 && halfw ? &tmBh : &tmB;
                    const int nbox = NW == 1 || halfw ? 1 : NW;
                    const uint32_t bytes = NW == 1 && halfw ? A_SLOT + B_SLOT / 2 : A_SLOT + nbox * B_SLOT;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!W.wait(bEMPTY + 8 * stage, phase)) { ok = false; break; }
                        const uint32_t a_dst = sA + stage * L::A_STRIDE, b_dst = sB + stage * L::B_STRIDE;
                        if constexpr (CG == 1 && KB > 1) {
                            // the slot's boxes inside K (a box wholly past K is neither
                            // loaded nor multiplied)
                            const int nk = min(KB, (p.K - kb * KB * BK + BK - 1) / BK);
                            mbar_arrive_expect_tx(bFULL + 8 * stage, static_cast<uint32_t>(nk) * bytes);
                            for (int j = 0; j < nk; ++j) {
                                tma_load_2d(a_dst + j * A_SLOT, &tmA, (kb * KB + j) * BK, m_cta, bFULL + 8 * stage);
                                tma_load_2d(b_dst + j * L::B_BOX, tb, (kb * KB + j) * BK, n_cta, bFULL + 8 * stage);
                            }
                        } else if constexpr (CG == 1) {
                            mbar_arrive_expect_tx(bFULL + 8 * stage, bytes);
                            tma_load_2d(a_dst, &tmA, kb * BK, m_cta, bFULL + 8 * stage);
                            tma_load_2d(b_dst, tb, kb * BK, n_cta, bFULL + 8 * stage);
                        } else {
                            // the leader arms its barrier for the bytes of both CTAs
                            if (rank == 0) mbar_arrive_expect_tx(bFULL + 8 * stage, 2 * bytes);
                            tma_load_2d_pair(a_dst, &tmA, kb * BK, m_cta, full_leader + 8 * stage);
                            for (int h = 0; h < nbox; ++h)
                                tma_load_2d_pair(b_dst + h * B_SLOT, tb, kb * BK, n_cta + h * SH::UMMA_N,
                                                 full_leader + 8 * stage);
                        }
                        ++issued;
                        st_volatile_shared_u32(sPROGRESS, issued);
                        if (++stage == S) { stage = 0; phase ^= 1u; }
                    }
                }
                if (!ok && is_leader) {
                    // drain: wait (bounded) for the copies still in flight into this CTA
                    const Waiter D{p.timeout_ns, abort_flag, p.status, kStatusRoleProducer};
                    volatile uint32_t no_abort = 0;
                    const Waiter Dn{D.timeout_ns, &no_abort, D.status, D.role};
                    const uint32_t first = issued > static_cast<uint32_t>(S) ? issued - S : 0u;
                    for (uint32_t it = first; it < issued; ++it)
                        if (!Dn.wait(bFULL + 8 * (it % S), (it / S) & 1u)) break;
                } else if (!ok && issued > 0) {
                    // A pair's peer: its copies signal the leader's barriers,
                    // which it cannot wait on, and the leader may have given
                    // up before arming them.  A copy lands within microseconds;
                    // waiting 1 ms (bounded) before the exit path keeps any
                    // still in flight from landing after the CTA is gone.
                    const uint64_t t0 = globaltimer_ns();
                    while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
                }
            }
        } else if (p.producer == kProducerRealign) {
            if constexpr ((CG == 1 || PK == 1) && KB == 1) {
                const Waiter W{p.timeout_ns, abort_flag, p.status, kStatusRoleProducer};
                realign_producer<CG, NW, S>(p, W, sA, sB, bFULL, bEMPTY, sPROGRESS, cluster_id, num_clusters, kb0,
                                            kb1, rank, warp, lane);
            }
        } else if constexpr (CG == 1 && KB == 1) {
            // cp.async producer (single CTA only): COPY_WARPS warps fill the swizzled slot
            const Waiter W{p.timeout_ns, abort_flag, p.status, kStatusRoleProducer};
            if (p.copy_bytes == 8)
                copy_producer<8, S>(p, W, sA, sB, bFULL, bEMPTY, sPROGRESS, cluster_id, num_clusters, kb0, kb1, lane);
            else if (p.copy_bytes == 4)
                copy_producer<4, S>(p, W, sA, sB, bFULL, bEMPTY, sPROGRESS, cluster_id, num_clusters, kb0, kb1, lane);
            else
                copy_producer<2, S>(p, W, sA, sB, bFULL, bEMPTY, sPROGRESS, cluster_id, num_clusters, kb0, kb1, lane);
        }
        __syncwarp();
    } else if (warp == mma_warp) {
        // ======================================================== MMA issuer
        if (lane == 0) {
            // seed: every slot starts with one empty credit
            if (!(p.flags & GEMM_DEBUG_SKIP_EMPTY_SEED))
                for (int s = 0; s < S; ++s) mbar_arrive(bEMPTY + 8 * s);
        }
        if (is_leader && lane == 0) {
            const Waiter W{p.timeout_ns, abort_flag, p.status, kStatusRoleMma};
            // a pair's realigning producer warps arrive on full[s] from both
            // CTAs with release at cluster scope: acquire at cluster scope
            constexpr bool kFullCluster = CG == 2 && PK == 1;
            uint32_t stage = 0, phase = 0;
            bool ok = true, issued_any = false;
            if constexpr (NW == 1) {
                constexpr uint32_t IDESC = make_idesc<SH::UMMA_M, SH::UMMA_N>();
                constexpr uint32_t IDESC_HALF = make_idesc<SH::UMMA_M, SH::UMMA_N / 2>();   // half-width units
                uint32_t tcount = 0;
                for (int u = cluster_id; ok && u < p.total_units; u += num_clusters, ++tcount) {
                    const Unit un = unit_of(u, p);
                    const uint32_t b = tcount % SH::NBUF, aph = (tcount / SH::NBUF) & 1u;
                    if (!W.template wait<CG == 2>(bTEMPTY + 8 * b, aph)) { ok = false; break; }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + b * SH::ACC_COLS;
                    // a half-width unit is one MMA of N = UMMA_N / 2
                    const uint32_t idesc = un.half >= 0 ? IDESC_HALF : IDESC;
                    // With S = 6 the MMA thread takes the ring's slots two at a time:
                    // it waits for both, issues their 8 MMAs back to back and then
                    // commits both.  A wait/commit boundary after every 4 MMAs
                    // measurably idles the tensor pipe (about 2 % sustained at
                    // 8192^3).  Holding two slots leaves the producer S - 2 to fill
                    // ahead, which only the 6-slot ring can afford: measured on
                    // GB300, pairing is 11 % slower at S = 4 and 2 % slower at S = 5.
                    constexpr int GROUP = S >= 6 ? 2 : 1;
                    for (int kb = kb0; kb < kb1; kb += GROUP) {
                        const int nb = kb1 - kb < GROUP ? kb1 - kb : GROUP;
                        uint32_t st[GROUP], ph[GROUP];
                        st[0] = stage;
                        ph[0] = phase;
                        if constexpr (GROUP == 2) {
                            st[1] = stage + 1 == S ? 0u : stage + 1;
                            ph[1] = stage + 1 == S ? phase ^ 1u : phase;
                        }
                        for (int j = 0; j < nb; ++j)
                            if (!W.template wait<kFullCluster>(bFULL + 8 * st[j], ph[j])) { ok = false; break; }
                        if (!ok) break;
                        tc_fence_after_sync();
                        if (p.producer == kProducerCopy) fence_proxy_async_smem();
                        for (int j = 0; j < nb; ++j) {
#pragma unroll
                            for (int bx = 0; bx < KB; ++bx) {
                                // a box wholly past K was not loaded (two-box slots)
                                if (KB > 1 && ((kb + j) * KB + bx) * BK >= p.K) break;
                                const uint64_t adesc = make_sdesc(sA + st[j] * L::A_STRIDE + bx * A_SLOT);
                                const uint64_t bdesc = make_sdesc(sB + st[j] * L::B_STRIDE + bx * L::B_BOX);
#pragma unroll
                                for (int k = 0; k < BK / UMMA_K; ++k) {
                                    // +32 bytes of K per step: +2 in the (address >> 4) field
                                    tc_mma_f16<CG>(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc,
                                                   (kb + j) != kb0 || bx != 0 || k != 0);
                                }
                            }
                        }
                        issued_any = true;
                        // release the slots once these multiplies have read them
                        for (int j = 0; j < nb; ++j) {
                            if constexpr (CG == 1) tc_commit_1(bEMPTY + 8 * st[j]);
                            else tc_commit_2_mc(bEMPTY + 8 * st[j], 0x3);
                            if (++stage == S) { stage = 0; phase ^= 1u; }
                        }
                    }
                    if (!ok) break;
                    // accumulator of this tile is complete
                    if constexpr (CG == 1) tc_commit_1(bTFULL + 8 * b);
                    else tc_commit_2_mc(bTFULL + 8 * b, 0x3);
                }
            } else {
                // The wide tile's accumulator is one buffer, drained in two
                // halves of UMMA_N columns with an event pair each (tmem_full[h]
                // / tmem_empty[h]).  At both ends of a unit the K blocks of a
                // group of J run half 0 and then half 1 on the same, still held,
                // slots: the epilogue drains half 0 of unit i while the tensor
                // pipe finishes half 1, and half 1 while half 0 of unit i+1
                // starts, so the pipe does not wait for the whole accumulator.
                // J = S - 1 leaves the producer one slot to fill while a group
                // is held.  A half-width unit uses half 0 only.
                //
                // The issuing thread's own instructions between MMAs idle the
                // tensor pipe (measured on GB300: the same MMAs issued from a
                // general loop over groups, halves and blocks ran 30-50 %
                // slower), so each part of a unit is straight-line code with
                // compile-time trip counts, and the descriptors of slot s are
                // the slot-0 descriptors plus s times the slot size: the start
                // address field (bits 0..13, address >> 4) cannot carry, as all
                // of shared memory lies below 256 KB.
                constexpr uint32_t IDESC = make_idesc<SH::UMMA_M, SH::UMMA_N>();
                constexpr int J = S > 1 ? S - 1 : 1;
                const uint64_t adesc0 = make_sdesc(sA), bdesc0 = make_sdesc(sB);
                uint32_t used0 = 0u, used1 = 0u;   // units that have used half 0 / half 1 so far
                const int nkb = p.num_kb;
                auto slot = [](uint32_t x) { return x < static_cast<uint32_t>(S) ? x : x - S; };
                // the 4 MMAs of the K block in slot s for half h (`first`: the unit's first K block)
                auto mma_block = [&](uint32_t s, int h, bool first) {
                    const uint64_t a = adesc0 + s * (A_SLOT >> 4);
                    const uint64_t b = bdesc0 + s * (L::B_STRIDE >> 4) + h * (B_SLOT >> 4);
                    const uint32_t d = tmem_base + h * SH::UMMA_N;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        tc_mma_f16<CG>(d, a + 2 * k, b + 2 * k, IDESC, !(first && k == 0));
                };
                auto wait_full = [&]() {
                    if (!W.template wait<kFullCluster>(bFULL + 8 * stage, phase)) return false;
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                    return true;
                };
                auto wait_acc = [&](int h) {
                    if (!W.template wait<true>(bTEMPTY + 8 * h, (h == 0 ? used0 : used1) & 1u)) return false;
                    tc_fence_after_sync();
                    return true;
                };
                for (int u = cluster_id; ok && u < p.total_units; u += num_clusters) {
                    const Unit un = unit_of(u, p);
                    if (un.half >= 0) {
                        // half-width unit: one box, half 0 of the accumulator
                        for (int kb = 0; kb < nkb; ++kb) {
                            const uint32_t s0 = stage;
                            if (!wait_full()) { ok = false; break; }
                            tc_fence_after_sync();
                            if (kb == 0 && !wait_acc(0)) { ok = false; break; }
                            mma_block(s0, 0, kb == 0);
                            issued_any = true;
                            tc_commit_2_mc(bEMPTY + 8 * s0, 0x3);
                        }
                        if (!ok) break;
                        tc_commit_2_mc(bTFULL, 0x3);
                        ++used0;
                    } else if (nkb > 2 * J) {
                        // head group: K blocks 0 .. J-1
                        const uint32_t h0 = stage;
#pragma unroll
                        for (int j = 0; j < J; ++j)
                            if (ok && !wait_full()) ok = false;
                        if (!ok) break;
                        tc_fence_after_sync();
                        if (!wait_acc(0)) { ok = false; break; }
#pragma unroll
                        for (int j = 0; j < J; ++j) mma_block(slot(h0 + j), 0, j == 0);
                        issued_any = true;
                        if (!wait_acc(1)) { ok = false; break; }
#pragma unroll
                        for (int j = 0; j < J; ++j) mma_block(slot(h0 + j), 1, j == 0);
#pragma unroll
                        for (int j = 0; j < J; ++j) tc_commit_2_mc(bEMPTY + 8 * slot(h0 + j), 0x3);
                        // the blocks in between: both halves back to back
                        for (int kb = J; kb < nkb - J; ++kb) {
                            const uint32_t s0 = stage;
                            if (!wait_full()) { ok = false; break; }
                            tc_fence_after_sync();
                            mma_block(s0, 0, false);
                            mma_block(s0, 1, false);
                            tc_commit_2_mc(bEMPTY + 8 * s0, 0x3);
                        }
                        if (!ok) break;
                        // tail group: K blocks nkb-J .. nkb-1
                        const uint32_t t0 = stage;
#pragma unroll
                        for (int j = 0; j < J; ++j)
                            if (ok && !wait_full()) ok = false;
                        if (!ok) break;
                        tc_fence_after_sync();
#pragma unroll
                        for (int j = 0; j < J; ++j) mma_block(slot(t0 + j), 0, false);
                        tc_commit_2_mc(bTFULL, 0x3);          // half 0 of the accumulator is complete
#pragma unroll
                        for (int j = 0; j < J; ++j) mma_block(slot(t0 + j), 1, false);
#pragma unroll
                        for (int j = 0; j < J; ++j) tc_commit_2_mc(bEMPTY + 8 * slot(t0 + j), 0x3);
                        tc_commit_2_mc(bTFULL + 8, 0x3);      // half 1 too
                        ++used0;
                        ++used1;
                    } else {
                        // few K blocks: every block holds both halves' MMAs; the
                        // accumulator is taken before the first and released after
                        // the last block
                        for (int kb = 0; kb < nkb; ++kb) {
                            const uint32_t s0 = stage;
                            if (!wait_full()) { ok = false; break; }
                            tc_fence_after_sync();
                            if (kb == 0 && (!wait_acc(0) || !wait_acc(1))) { ok = false; break; }
                            mma_block(s0, 0, kb == 0);
                            mma_block(s0, 1, kb == 0);
                            issued_any = true;
                            tc_commit_2_mc(bEMPTY + 8 * s0, 0x3);
                        }
                        if (!ok) break;
                        tc_commit_2_mc(bTFULL, 0x3);
                        tc_commit_2_mc(bTFULL + 8, 0x3);
                        ++used0;
                        ++used1;
                    }
                }
            }
            if (issued_any) {
                // all multiplies have finished before tensor memory is released
                if constexpr (CG == 1) tc_commit_1(bDRAIN);
                else tc_commit_2_mc(bDRAIN, 0x1);
                volatile uint32_t no_abort = 0;
                const Waiter D{p.timeout_ns, &no_abort, p.status, kStatusRoleMma};
                D.wait(bDRAIN, 0);
            }
        }
        __syncwarp();
    } else {
        // ======================================================== epilogue
        const int e = warp - P - 1;              // 0 .. EW-1
        const int q = warp & 3;                  // tensor-memory lane quarter of this warp
        if (kpair) cluster_wait_acquire();       // the peer's barriers are set up
        const Waiter W{p.timeout_ns, abort_flag, p.status, kStatusRoleEpilogue};
        const uint32_t tempty_leader = (CG == 2) ? mapa_shared(bTEMPTY, 0) : bTEMPTY;
        // seed: both accumulator event pairs start free (the two buffers of
        // the 256 x 256 and 128 x 128 tiles, the two halves of the wide one)
        if (lane == 0 && !(p.flags & GEMM_DEBUG_SKIP_ACC_SEED)) {
            for (int b = 0; b < 2; ++b) {
                if constexpr (CG == 1) mbar_arrive(bTEMPTY + 8 * b);
                else mbar_arrive_cluster(tempty_leader + 8 * b);
            }
        }
        // K split.  Lane quarters 2*krank and 2*krank+1 of the tile are this
        // CTA's to store.  The warps of the other two quarters are senders:
        // they write their fp32 partial sums from registers straight into the
        // peer's epilogue staging area and arrive on the peer's recv barrier
        // (each lane's release publishes its own stores); the owner warp then
        // adds them, read locally, to its own partial sums before rounding.
        // The staging area is free for this from the start: the K split's
        // owners stage their f16 output in their own ring instead (idle once
        // their accumulator is complete; one tile per CTA).  Layout, 16 KB per
        // quarter: 16-byte unit u (fp32 columns 4u..4u+3) of lane l's row at
        // u * 512 + l * 16, so one unit of all 32 rows is one contiguous
        // 512-byte block (conflict-free, one request per warp).  Measured on
        // GB300: the owner reading the sums from the peer's shared memory
        // instead cost 0.35-0.5 us more per tile (each remote round trip
        // exposed), and 2-4 us more with a 512-byte row per lane.
        const bool sender = kpair && static_cast<uint32_t>(q >> 1) != krank;
        const uint32_t recv_lane = sEPI + static_cast<uint32_t>(q & 1) * (32u * 512u) + static_cast<uint32_t>(lane) * 16u;
        const uint32_t push_lane = sender ? mapa_shared(recv_lane, krank ^ 1u) : 0u;
        const uint32_t peer_sums = kpair && !sender ? recv_lane : 0u;
        const uint32_t peer_progress = kpair ? mapa_shared(sPROGRESS, krank ^ 1u) : 0u;
        static_assert(SH::ACC_COLS / 4 * 512 <= 32 * 512 || CG == 2, "a received quarter holds the single tile's 128 fp32 columns");
        static_assert(2 * 32 * 512 == EPI_BYTES, "the staging area holds the two received quarters");
        static_assert(EPI_WARPS * 2 * EPI_BUF <= A_SLOT + B_SLOT, "the owners' output staging fits in the smallest ring");
        // Reads 64 accumulator columns (chunk c of the columns starting at
        // tensor-memory address tbase) of this lane's row, adds the peer's
        // partial sums of the same columns (K split), and rounds them to 32
        // packed f16 pairs.
        auto load_chunk = [&](uint32_t tbase, int c, uint32_t(&h)[32]) {
            const uint32_t taddr = tbase + static_cast<uint32_t>(c * EPI_COLS);
            if (peer_sums) {
                // 32 columns at a time: own partial sums from tensor memory and
                // the peer's (units 16c + 8 half ..+7) in flight together, then
                // own + peer, one fp32 add per element (commutative, so the
                // same bits whichever K half is this CTA's)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[32], w[32];
                    tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(half * 32), v);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t u = static_cast<uint32_t>(c * 16 + half * 8 + i);
                        ld_shared_v4(peer_sums + u * 512u, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        h[half * 16 + k] =
                            pack_half2(__float_as_uint(__uint_as_float(v[2 * k]) + __uint_as_float(w[2 * k])),
                                       __float_as_uint(__uint_as_float(v[2 * k + 1]) + __uint_as_float(w[2 * k + 1])));
                }
                return;
            }
            uint32_t v0[32], v1[32];
            tmem_ld_32x32b_x32(taddr, v0);
            tmem_ld_32x32b_x32(taddr + 32, v1);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 16; ++k) h[k] = pack_half2(v0[2 * k], v0[2 * k + 1]);
#pragma unroll
            for (int k = 0; k < 16; ++k) h[16 + k] = pack_half2(v1[2 * k], v1[2 * k + 1]);
        };
        // Writes a chunk (this lane's row of a 32 x 64 block) into staging
        // buffer `buf` in the 128-byte swizzle the output tensor map uses.
        auto stage_chunk = [&](uint32_t buf, const uint32_t(&h)[32]) {
            const uint32_t row_addr = buf + static_cast<uint32_t>(lane) * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t dst = row_addr + ((static_cast<uint32_t>(j) ^ static_cast<uint32_t>(lane & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(h[4 * j]), "r"(h[4 * j + 1]),
                             "r"(h[4 * j + 2]), "r"(h[4 * j + 3])
                             : "memory");
            }
        };
        // Guarded plain stores of a chunk (outputs TMA cannot address).
        auto store_direct = [&](const uint32_t(&h)[32], int row0, int col0) {
            const int row = row0 + lane;
            if (row < p.M) {
                unsigned short* dst = reinterpret_cast<unsigned short*>(p.out) + static_cast<int64_t>(row) * p.N;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int col = col0 + 2 * i;
                    if (col < p.N) dst[col] = static_cast<unsigned short>(h[i] & 0xFFFFu);
                    if (col + 1 < p.N) dst[col + 1] = static_cast<unsigned short>(h[i] >> 16);
                }
            }
        };
        // Waits for accumulator event pair i (parity `par`), writes its ncols
        // columns starting at tensor-memory column acc_col0 to output columns
        // col_base.. of rows row0..row0+31, and releases the columns.  False
        // if the wait gave up.  With TMA stores the chunks go two at a time
        // through the warp's two staging buffers: one wait for the buffers,
        // one proxy fence and one bulk group per pair (measured per chunk on
        // GB300: the fence and the store issue cost about as much as the
        // tensor-memory load and the rounding together).
        auto drain = [&](uint32_t i, uint32_t par, uint32_t acc_col0, int ncols, int row0, int col_base) {
            bool got = true;
            if (lane == 0) got = W.wait_progress(bTFULL + 8 * i, par, sPROGRESS, false);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) return false;
            tc_fence_after_sync();
            const int nch = ncols / EPI_COLS;
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc_col0;
            // the wide tile's two warps of a lane quarter take half of the chunks each
            constexpr bool kHalfChunks = EW == EPI_WARPS_WIDE;
            const int cb = kHalfChunks ? (e / 4) * (nch / 2) : 0;
            const int ce = kHalfChunks ? cb + nch / 2 : nch;
            if (kHalfChunks && p.store == kStoreTma) {
                // one staging buffer per warp
                const uint32_t buf = sEPI + static_cast<uint32_t>(e) * EPI_BUF;
                for (int c = cb; c < ce; ++c) {
                    // the store issued from the buffer has finished reading it
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
                    uint32_t h[32];
                    load_chunk(tbase, c, h);
                    stage_chunk(buf, h);
                    fence_proxy_async_smem();
                    __syncwarp();
                    const int col0 = col_base + c * EPI_COLS;
                    if (lane == 0 && row0 < p.M && col0 < p.N) {
                        tma_store_2d(&tmC, buf, col0, row0);
                        bulk_commit_group();
                    }
                }
            } else if (NW == 2 && p.store == kStoreTma) {
                // four warps: each drains all chunks of its lane quarter, one
                // at a time through its two staging buffers in turn (a bulk
                // group per chunk, possibly empty, so that "at most one group
                // still reading" means the buffer about to be written is free)
                const uint32_t bufs = sEPI + static_cast<uint32_t>(e) * 2 * EPI_BUF;
                for (int c = 0; c < nch; ++c) {
                    const uint32_t buf = bufs + static_cast<uint32_t>(c & 1) * EPI_BUF;
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
                    uint32_t h[32];
                    load_chunk(tbase, c, h);
                    stage_chunk(buf, h);
                    fence_proxy_async_smem();
                    __syncwarp();
                    const int col0 = col_base + c * EPI_COLS;
                    if (lane == 0) {
                        if (row0 < p.M && col0 < p.N) tma_store_2d(&tmC, buf, col0, row0);
                        bulk_commit_group();
                    }
                }
            } else if (p.store == kStoreTma) {
                // (the K split's owners stage in their ring: the staging area
                // holds the peer's partial sums)
                const uint32_t bufs = (kpair ? sA : sEPI) + static_cast<uint32_t>(e) * 2 * EPI_BUF;
                for (int c = 0; c < nch; c += 2) {
                    const int nb = nch - c < 2 ? nch - c : 2;
                    // the stores issued from both buffers have finished reading them
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (t < nb) {
                            uint32_t h[32];
                            load_chunk(tbase, c + t, h);
                            stage_chunk(bufs + t * EPI_BUF, h);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        bool any = false;
                        for (int t = 0; t < nb; ++t) {
                            const int col0 = col_base + (c + t) * EPI_COLS;
                            // a box wholly past M or N (padding rows of a pair tile) is not stored
                            if (row0 < p.M && col0 < p.N) {
                                tma_store_2d(&tmC, bufs + t * EPI_BUF, col0, row0);
                                any = true;
                            }
                        }
                        if (any) bulk_commit_group();
                    }
                }
            } else {
                for (int c = cb; c < ce; ++c) {
                    uint32_t h[32];
                    load_chunk(tbase, c, h);
                    store_direct(h, row0, col_base + c * EPI_COLS);
                }
            }
            // this warp's reads of these accumulator columns are complete
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 1) mbar_arrive(bTEMPTY + 8 * i);
                else mbar_arrive_cluster(tempty_leader + 8 * i);
            }
            return true;
        };
        // K split, sender warps: wait for accumulator buffer i, write this
        // lane's row of it (128 fp32 columns) into the peer's staging area,
        // arrive on the peer's recv barrier and release the columns.  False
        // if the wait gave up.
        auto send = [&](uint32_t i, uint32_t par) {
            bool got = true;
            if (lane == 0) got = W.wait_progress(bTFULL + 8 * i, par, sPROGRESS, false);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) return false;
            tc_fence_after_sync();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + i * SH::ACC_COLS;
#pragma unroll 1
            for (int c = 0; c < (p.flags & GEMM_DEBUG_SKIP_KSPLIT_SEND ? 0 : SH::ACC_COLS / 64); ++c) {
                uint32_t v0[32], v1[32];
                tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(c * 64), v0);
                tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(c * 64 + 32), v1);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_cluster_v4(push_lane + static_cast<uint32_t>(c * 16 + j) * 512u, v0[4 * j],
                                         v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_cluster_v4(push_lane + static_cast<uint32_t>(c * 16 + 8 + j) * 512u, v1[4 * j],
                                         v1[4 * j + 1], v1[4 * j + 2], v1[4 * j + 3]);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (!(p.flags & GEMM_DEBUG_SKIP_KSPLIT_SEND))
                mbar_arrive_cluster(mapa_shared(bRECV + 8 * static_cast<uint32_t>(q & 1), krank ^ 1u));
            if (lane == 0) mbar_arrive(bTEMPTY + 8 * i);
            return true;
        };
        uint32_t tcount = 0;
        uint32_t used0 = 0u, used1 = 0u;     // wide tile: units that have used half 0 / half 1
        for (int u = cluster_id; u < p.total_units; u += num_clusters, ++tcount) {
            const Unit un = unit_of(u, p);
            int tm, tn;
            tile_coords(un.tile, p, tm, tn);
            const int row0 = tm * SH::UMMA_M + static_cast<int>(rank) * BM_CTA + q * 32;
            // a half-width unit holds HALF_N accumulator columns, starting at
            // column half * HALF_N of its tile
            const int col_base = tn * SH::TILE_N + (un.half > 0 ? SH::HALF_N : 0);
            if constexpr (NW == 1) {
                const uint32_t b = tcount & 1u, aph = (tcount >> 1) & 1u;
                const int ncols = un.half >= 0 ? SH::HALF_N : SH::ACC_COLS;
                if (kpair) {
                    if (sender) {
                        if (!send(b, aph)) break;
                        continue;
                    }
                    // the owner: every lane waits (its own acquire orders its
                    // reads of the peer's rows), and the warp goes on only if
                    // all lanes' waits completed.  The peer's sums come after
                    // the peer's whole K loop: the limit counts from the last
                    // K block the peer's producer issued.
                    bool got = W.template wait_progress<true>(bRECV + 8 * static_cast<uint32_t>(q & 1), 0,
                                                              peer_progress, true);
                    if (!__all_sync(0xffffffffu, got)) break;
                }
                if (!drain(b, aph, b * SH::ACC_COLS, ncols, row0, col_base)) break;
            } else {
                if (!drain(0u, used0 & 1u, 0u, SH::UMMA_N, row0, col_base)) break;
                ++used0;
                if (un.half < 0) {
                    if (!drain(1u, used1 & 1u, SH::UMMA_N, SH::UMMA_N, row0, col_base + SH::UMMA_N)) break;
                    ++used1;
                }
            }
        }
        // the staging buffers must stay until the last stores have read them;
        // the global writes themselves complete before the grid does
        if (lane == 0 && p.store == kStoreTma) bulk_wait_group_read<0>();
        __syncwarp();
    }

    // ------------------------------------------------------------ tear-down
    // (K split: the cluster barrier also keeps this CTA's staged partial sums
    // in place until the peer has read them)
    tc_fence_before_sync();
    __syncthreads();
    if (kpair && warp <= mma_warp) cluster_wait_acquire();     // the set-up barrier's wait
    if (CG == 2 || kpair) cluster_sync();
    if (warp == mma_warp) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem_base, SH::TMEM_COLS);
    }
}

// Fills a f16 [M,N] output with zeros (K == 0: the empty sum).
__global__ void zero_fill_u16(unsigned short* out, int64_t n) {
    grid_dependency_wait();             // launched as a programmatic dependent
    allow_dependent_launch();
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        out[i] = 0;
}

// Bytes sh .. sh+15 (sh even) of the 32 bytes lo | hi, little-endian.
__device__ __forceinline__ uint4 bytes_at(const uint4& lo, const uint4& hi, unsigned sh) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const unsigned q = sh >> 2, bits = (sh & 3u) * 8u;
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t x = q == 0 ? w[i] : q == 1 ? w[i + 1] : q == 2 ? w[i + 2] : w[i + 3];
        const uint32_t y = q == 0 ? w[i + 1] : q == 1 ? w[i + 2] : q == 2 ? w[i + 3] : w[i + 4];
        o[i] = __funnelshift_r(x, y, bits);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Copies the rows of lhs [ma, K] and rhs [nb, K] into destination rows Kp
// elements apart: a layout the tensor memory accelerator can address when
// K * 2 bytes is not a multiple of 16 or a base is not 16-byte aligned.  The
// first Kw = ceil(K/8)*8 elements of each row are written (the ones past K
// zeroed); the rest of a row (Kp > Kw) is padding that keeps rows 128-byte
// aligned and is never written or read.
//
// A row is copied by 2^tpr_log2 threads (as many as it has 16-byte chunks,
// up to the 256 of a block; a block takes 256 >> tpr_log2 rows), thread t
// writing chunks t, t + 2^tpr_log2, ...  A chunk wholly inside the row is
// read as the aligned 16-byte blocks that hold it (one, or two when the row
// does not start on a 16-byte boundary) and shifted into place; every block
// read holds at least one byte of the row, so no load leaves the pages the
// operand occupies.  The ragged last chunk of a row is read element by
// element.  Measured on GB300 for the 4000 x 3000 x 2050 operands (28.7 MB
// read, 12 us alone and cold, DRAM about 30 % busy): a thread per chunk with
// 4-byte loads and a 64-bit division per chunk ran as fast, one warp per row
// (9 dependent rounds of loads) and four chunks per thread with their loads
// issued together both ran slower.
__global__ void __launch_bounds__(256)
repack_rows_kernel(const uint16_t* __restrict__ a, int64_t ma, const uint16_t* __restrict__ b, int64_t nb, int K,
                   int Kw, int Kp, uint16_t* __restrict__ dst_a, uint16_t* __restrict__ dst_b, int tpr_log2) {
    // launched as a programmatic dependent; the GEMM that follows may start
    // its set-up while the copy finishes
    grid_dependency_wait();
    allow_dependent_launch();
    const int tpr = 1 << tpr_log2;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> tpr_log2) + (threadIdx.x >> tpr_log2);
    if (r >= ma + nb) return;
    const int t = threadIdx.x & (tpr - 1);
    const int chunks = Kw / 8, full = K / 8;
    const uint16_t* src = r < ma ? a + r * K : b + (r - ma) * K;
    uint16_t* dst = r < ma ? dst_a + r * Kp : dst_b + (r - ma) * Kp;
    const uintptr_t sa = reinterpret_cast<uintptr_t>(src);
    const unsigned sh = static_cast<unsigned>(sa & 15u);      // even: the operands are 2-byte aligned
    const uint4* blk = reinterpret_cast<const uint4*>(sa - sh);
    for (int j = t; j < chunks; j += tpr) {
        uint4 o;
        if (j < full) {
            const uint4 lo = blk[j];
            o = sh == 0 ? lo : bytes_at(lo, blk[j + 1], sh);
        } else {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int k = 8 * j + 2 * e;
                const uint32_t lo16 = k < K ? src[k] : 0u;
                const uint32_t hi16 = k + 1 < K ? src[k + 1] : 0u;
                w[e] = lo16 | (hi16 << 16);
            }
            o = make_uint4(w[0], w[1], w[2], w[3]);
        }
        *reinterpret_cast<uint4*>(dst + 8 * static_cast<int64_t>(j)) = o;
    }
}

// Launches repack_rows_kernel over the M + N rows (Kw elements written per
// destination row, rows Kp elements apart).
cudaError_t launch_repack(const void* lhs, int64_t M, const void* rhs, int64_t N, int64_t K, int64_t Kw, int64_t Kp,
                          uint16_t* da, uint16_t* db, cudaStream_t stream) {
    int tpr_log2 = 0;
    while ((1 << tpr_log2) < Kw / 8 && tpr_log2 < 8) ++tpr_log2;
    const int64_t rows_per_block = 256 >> tpr_log2;
    const int64_t blocks = (M + N + rows_per_block - 1) / rows_per_block;
    if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
    return launch_pdl(repack_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                      static_cast<const uint16_t*>(lhs), M, static_cast<const uint16_t*>(rhs), N, static_cast<int>(K),
                      static_cast<int>(Kw), static_cast<int>(Kp), da, db, tpr_log2);
}

struct Plan {
    int cg = 1;
    int nw = 1;                 // MMAs per K step (2: the wide 256 x 512 pair tile)
    bool repack = false;        // operands copied to 16-byte aligned rows, then TMA
    int producer = kProducerTma;
    int copy_bytes = 16;
    int store = kStoreTma;
    int tiles_m = 0, tiles_n = 0, num_tiles = 0, num_kb = 0;
    int smem = 0;
    int ksplit = 1;             // 2: two CTAs (a cluster) per single-CTA tile, one K half each
    int kb = 1;                 // 64-wide K boxes per ring slot (2, 3 or 4: single-CTA TMA tile, S <= 3)
};

// Fewest K blocks for which small single-CTA GEMMs split K over two CTAs.
constexpr int kKSplitMinBlocks = 32;

// Row alignment (elements) of a repacked copy: 64 elements, 128-byte rows,
// which TMA reads fastest (the fixed array falls back to 8 when 64 does not fit).
constexpr int64_t kPooledRowAlign = 64;

// The wide tile's 48 KB slots fit the shared memory up to this many stages.
constexpr int WIDE_MAX_STAGES = 4;

int smem_for(int stages, int nw, int kb = 1) {
    if (kb == 4) return stages == 1 ? Layout<1, 1, 4>::DYN : Layout<2, 1, 4>::DYN;
    if (kb == 3) return stages == 1 ? Layout<1, 1, 3>::DYN : Layout<2, 1, 3>::DYN;
    if (kb == 2) return Layout<3, 1, 2>::DYN;
    if (nw == 2) {
        switch (stages) {
            case 1: return Layout<1, 2>::DYN;
            case 2: return Layout<2, 2>::DYN;
            case 3: return Layout<3, 2>::DYN;
            default: return Layout<4, 2>::DYN;
        }
    }
    switch (stages) {
        case 1: return Layout<1>::DYN;
        case 2: return Layout<2>::DYN;
        case 3: return Layout<3>::DYN;
        case 4: return Layout<4>::DYN;
        case 5: return Layout<5>::DYN;
        default: return Layout<6>::DYN;
    }
}

// Argument checks shared by the plan query and the launch.
int validate(int64_t M, int64_t N, int64_t K, const void* lhs, const void* rhs, const void* out, int stages) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31)) return GEMM_ERR_INVALID_ARG;
    if (stages < 1 || stages > MAX_STAGES) return GEMM_ERR_UNSUPPORTED_STAGES;
    if (M == 0 || N == 0) return GEMM_OK;
    // the plan counts 128 x 128 tiles in an int (no output that large fits in
    // any device's memory: it would hold 2^31 * 2^14 elements)
    if (((M + 127) / 128) * ((N + 127) / 128) >= (1ll << 31)) return GEMM_ERR_INVALID_ARG;
    if (!out || (K > 0 && (!lhs || !rhs))) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(lhs) | reinterpret_cast<uintptr_t>(rhs)) & 1u)
        return GEMM_ERR_ALIGNMENT;
    const uint64_t out_b = static_cast<uint64_t>(M) * N * 2;
    if (K > 0 && (ranges_overlap(out, out_b, lhs, static_cast<uint64_t>(M) * K * 2) ||
                  ranges_overlap(out, out_b, rhs, static_cast<uint64_t>(N) * K * 2)))
        return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

// Destination row length of the repack: K rounded up to `align` elements.
// The pooled path uses 64 (128-byte rows): on GB300 a ring-slot copy from
// rows at a 16-byte but not 128-byte multiple runs the whole GEMM ~12 %
// slower (4096 x 3072 x 2056: 43.6 us; with K = 2048 or 2112: 38.8 / 38.7 us).
inline int64_t repack_ld(int64_t K, int64_t align) { return (K + align - 1) / align * align; }

// Bytes of scratch the repack path needs: both operands with rows of
// repack_ld(K, align) elements.
inline size_t repack_bytes(int64_t M, int64_t N, int64_t K, size_t* b_offset, int64_t align) {
    const int64_t Kp = repack_ld(K, align);
    const size_t a_bytes = (static_cast<size_t>(M) * Kp * 2 + 255) / 256 * 256;
    if (b_offset) *b_offset = a_bytes;
    return a_bytes + (static_cast<size_t>(N) * Kp * 2 + 255) / 256 * 256;
}

// Whether the wide pair tile (256 x 512) should replace the 256 x 256 one.  It
// copies a quarter fewer operand bytes into shared memory per flop, which on
// GB300 lets the power-capped clock run higher (measured 3-6 % faster from
// 4096^3 up, and never slower).  It is not used where its 512-column tiles
// would add a block of padding columns the 256-column tiles do not have.
bool want_wide(int64_t N) { return (N + 511) / 512 * 2 == (N + 255) / 256; }

// Where the wide tile would leave CTA pairs idle that the 256 x 256 tile
// fills (both give the same bits, so S may decide): when the 256 x 256 tiles
// fit in one wave of pairs (the wide ones would need the half split to fill
// them), or, from three slots on, when the wide tiles are fewer than the
// pairs while the 256 x 256 tiles take one wave and a tail that the half
// split runs at once.  Measured on GB300: 2048^2 x 4096, S = 1..4: 256 x 256
// 2-8 % faster; 2560^3, S = 3 / 4: 27.6 / 25.7 us against 29.9 / 29.9 us
// (at S = 1, 2 the wide tile wins: 56.5 / 32.5 against 65.2 / 36.5 us).
// Elsewhere the wide tile was as fast or faster (3072^3 to 8192^3).
bool narrow_fills_better(int64_t M, int64_t N, int stages, int64_t pair_cap) {
    const int64_t narrow = ((M + 255) / 256) * ((N + 255) / 256);
    const int64_t wide = ((M + 255) / 256) * ((N + 511) / 512);
    if (narrow <= pair_cap) return true;
    return stages >= 3 && wide < pair_cap && 2 * (narrow - pair_cap) <= pair_cap;
}

// Operands that no tensor map can describe are read in place by the
// realigning producer, unless `repack` is set: then they are copied to
// aligned rows in scratch memory first and read by TMA.
Plan make_plan(int64_t M, int64_t N, int64_t K, const void* lhs, const void* rhs, const void* out, int stages,
               int num_sms, unsigned flags, bool repack = false) {
    Plan pl;
    const uintptr_t a = reinterpret_cast<uintptr_t>(lhs), b = reinterpret_cast<uintptr_t>(rhs);
    const uintptr_t o = reinterpret_cast<uintptr_t>(out);
    const bool force_copy = flags & GEMM_DEBUG_FORCE_COPY_PRODUCER;
    const bool native_tma = K % 8 == 0 && a % 16 == 0 && b % 16 == 0;
    if (!force_copy && native_tma) {
        pl.producer = kProducerTma;
        pl.copy_bytes = 16;
    } else if (!force_copy && repack) {
        pl.repack = true;
        pl.producer = kProducerTma;
        pl.copy_bytes = 16;
    } else if (!force_copy) {
        pl.producer = kProducerRealign;
        pl.copy_bytes = 16;
    } else {
        pl.producer = kProducerCopy;
        if (K % 4 == 0 && a % 8 == 0 && b % 8 == 0) pl.copy_bytes = 8;
        else if (K % 2 == 0 && a % 4 == 0 && b % 4 == 0) pl.copy_bytes = 4;
        else pl.copy_bytes = 2;
    }
    pl.store = (!(flags & GEMM_DEBUG_FORCE_DIRECT_STORE) && N % 8 == 0 && o % 16 == 0) ? kStoreTma : kStoreDirect;
    // The CTA-pair tile when TMA feeds it and it needs fewer waves of the
    // persistent grid than the single-CTA tile (or as many, with enough pair
    // tiles to occupy the GPU); otherwise the single-CTA tile.  Small and
    // mid-size GEMMs are bound by each CTA's chain of K blocks through the
    // ring more than by the multiplies, so the wave count decides: a pair
    // block does twice a single CTA's work in about 1.2x the time.  Measured
    // on GB300 (S = 2 / 4): 2048^3 on 64 pair tiles (one wave) 18.6 / 13.9
    // us, on 256 single tiles (two waves) 27.5 / 19.3 us.  Decided from the
    // shape alone; the single-CTA tile keeps every shape the K split uses.
    const int64_t solo_tiles = ((M + 127) / 128) * ((N + 127) / 128);
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
    const int64_t pair_cap = num_sms / 2;
    const int64_t solo_waves = (solo_tiles + num_sms - 1) / num_sms;
    const int64_t pair_waves = (pair_tiles + pair_cap - 1) / pair_cap;
    const bool want_pair = (flags & GEMM_DEBUG_FORCE_PAIR_TILE) || pair_waves < solo_waves ||
                           (pair_waves == solo_waves && 2 * pair_tiles >= num_sms);
    pl.cg = (pl.producer != kProducerCopy && !(flags & GEMM_DEBUG_FORCE_SOLO_TILE) && want_pair) ? 2 : 1;
    pl.nw = (pl.cg == 2 && stages <= WIDE_MAX_STAGES && !(flags & GEMM_DEBUG_FORCE_NARROW_TILE) &&
             ((flags & GEMM_DEBUG_FORCE_WIDE_TILE) ||
              (want_wide(N) && !narrow_fills_better(M, N, stages, pair_cap))))
                ? 2
                : 1;
    const int tile_m = 128 * pl.cg, tile_n = 128 * pl.cg * pl.nw;
    pl.tiles_m = static_cast<int>((M + tile_m - 1) / tile_m);
    pl.tiles_n = static_cast<int>((N + tile_n - 1) / tile_n);
    pl.num_tiles = pl.tiles_m * pl.tiles_n;
    pl.num_kb = static_cast<int>((K + BK - 1) / BK);
    // K split: where single-CTA tiles leave at least half of the SMs idle and
    // K is long, a cluster of two CTAs computes each tile, one K half each.
    // Small GEMMs are bound by the chain of K blocks through the ring (each
    // block waits for a slot's load-to-use latency); halving the chain per CTA
    // pays once it outweighs the cluster launch and the exchange of partial
    // sums (about 1.5 us).  Measured on GB300 (S = 2 / 4): 1024 x 1024 x 4096
    // 23.4 -> 17.0 / 18.1 -> 13.2 us, 512 x 512 x 8192 43.1 -> 26.5 / 32.6 ->
    // 19.7 us, 1024 x 1024 x 2048 13.2 -> 10.9 / 10.7 -> 9.3 us; at 16 K blocks
    // (1024^3) it is even or slower (8.0 -> 7.9 / 6.9 -> 7.3 us).  Decided
    // from the shape alone, never from S.
    if (pl.cg == 1 && !(flags & GEMM_DEBUG_NO_KSPLIT)) {
        const bool forced = flags & GEMM_DEBUG_FORCE_KSPLIT;
        if (pl.num_kb >= (forced ? 2 : kKSplitMinBlocks) && (forced || 2ll * pl.num_tiles <= num_sms)) pl.ksplit = 2;
    }
    // Multi-box slots: on the single-CTA TMA tile with up to three slots,
    // when the tiles fit in one wave, so that each CTA's chain of K blocks
    // through the ring is what bounds the call: three boxes per slot for one
    // or two slots, two for three (the most that fit in shared memory).  When
    // every tile runs as two half-width units (the tail split of a launch
    // whose tiles fill at most half the SMs: the rule of run_plan, whose
    // grid for this tile is one CTA per SM), their half-size B boxes let one
    // or two slots hold four boxes.  Measured on GB300 (graph replay),
    // 1024^3 at S = 2 / 1: 6.46 / 9.05 us with three boxes, 6.25 / 8.30 us
    // with four; 1024 x 1024 x 512 at S = 2 the same either way.  Each
    // element keeps its K order: the result is the same for every choice.
    if (pl.cg == 1 && pl.ksplit == 1 && pl.producer == kProducerTma && stages <= 3 && pl.num_kb >= 2 &&
        !(flags & GEMM_DEBUG_NO_DOUBLE_SLOT) &&
        ((flags & GEMM_DEBUG_FORCE_DOUBLE_SLOT) || pl.num_tiles <= num_sms)) {
        pl.kb = stages <= 2 ? 3 : 2;
        if (stages <= 2 && !(flags & (GEMM_DEBUG_NO_SPLIT | GEMM_DEBUG_FORCE_DOUBLE_SLOT)) &&
            2 * pl.num_tiles <= num_sms)
            pl.kb = 4;
    }
    pl.num_kb = static_cast<int>((K + BK * pl.kb - 1) / (BK * pl.kb));
    pl.smem = smem_for(stages, pl.nw, pl.kb);
    return pl;
}

inline int block_threads(const Plan& pl) {
    const bool tma = pl.producer == kProducerTma;
    return ((tma ? 1 : COPY_WARPS) + 1 + (pl.nw == 2 && tma ? EPI_WARPS_WIDE : EPI_WARPS)) * 32;
}

// Sets the kernel's shared-memory limit (once per device) and returns how
// many CTA groups (pairs or single CTAs) can be resident at once: the size of
// the persistent grid.  0 on failure.
template <int CG, int S, int NW, int PK, int KB = 1>
int capacity(const DeviceInfo& info, int threads) {
    auto kern = gemm_f16_nt_kernel<CG, S, NW, PK, KB>;
    constexpr int smem = Layout<S, NW, KB>::DYN;
    static_assert(Layout<S, NW, KB>::BYTES <= 232448, "ring + staging exceed the per-block shared memory");
    // per-device caches; concurrent first calls from several host threads
    // compute and store the same values
    static std::atomic<int> configured[64] = {};
    static std::atomic<int> max_clusters[64] = {};
    if (!configured[info.device].load(std::memory_order_relaxed)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
        configured[info.device].store(1, std::memory_order_relaxed);
    }
    if constexpr (CG == 1) {
        return info.num_sms;
    } else {
        if (!max_clusters[info.device].load(std::memory_order_relaxed)) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            cfg.blockDim = dim3(threads, 1, 1);
            cfg.dynamicSmemBytes = smem;
            cfg.gridDim = dim3(2 * info.num_sms, 1, 1);
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
                cudaGetLastError();
                n = info.num_sms / 2;
            }
            max_clusters[info.device].store(n, std::memory_order_relaxed);
        }
        return max_clusters[info.device].load(std::memory_order_relaxed);
    }
}

template <int CG, int NW, int PK>
int capacity_for(int stages, const DeviceInfo& info, int threads) {
    switch (stages) {
        case 1: return capacity<CG, 1, NW, PK>(info, threads);
        case 2: return capacity<CG, 2, NW, PK>(info, threads);
        case 3: return capacity<CG, 3, NW, PK>(info, threads);
        case 4: return capacity<CG, 4, NW, PK>(info, threads);
    }
    if constexpr (NW == 1)
        return stages == 5 ? capacity<CG, 5, 1, PK>(info, threads) : capacity<CG, 6, 1, PK>(info, threads);
    return 0;
}

// PK of a plan's kernel: single-CTA kernels serve every producer (PK = 0);
// a CTA pair fed by the realigning producer has its own (PK = 1).
inline int pk_of(const Plan& pl) { return pl.cg == 2 && pl.producer != kProducerTma ? 1 : 0; }

int capacity_of(const Plan& pl, int stages, const DeviceInfo& info) {
    const int threads = block_threads(pl);
    if (pl.kb == 4) return stages == 1 ? capacity<1, 1, 1, 0, 4>(info, threads) : capacity<1, 2, 1, 0, 4>(info, threads);
    if (pl.kb > 1) {
        switch (stages) {
            case 1: return capacity<1, 1, 1, 0, 3>(info, threads);
            case 2: return capacity<1, 2, 1, 0, 3>(info, threads);
            case 3: return capacity<1, 3, 1, 0, 2>(info, threads);
        }
        return 0;
    }
    if (pl.cg == 1) return capacity_for<1, 1, 0>(stages, info, threads);
    if (pk_of(pl))
        return pl.nw == 2 ? capacity_for<2, 2, 1>(stages, info, threads) : capacity_for<2, 1, 1>(stages, info, threads);
    return pl.nw == 2 ? capacity_for<2, 2, 0>(stages, info, threads) : capacity_for<2, 1, 0>(stages, info, threads);
}

// Launches the persistent grid: one CTA group per work unit, at most as many
// as can be resident.
template <int CG, int S, int NW, int PK, int KB = 1>
int launch(const Plan& pl, const DeviceInfo& info, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbh,
           const CUtensorMap& tc, const Params& p, cudaStream_t stream) {
    auto kern = gemm_f16_nt_kernel<CG, S, NW, PK, KB>;
    const int threads = block_threads(pl);
    const int cap = capacity<CG, S, NW, PK, KB>(info, threads);
    if (cap <= 0) return GEMM_ERR_LAUNCH;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2] = {pdl_attribute(), {}};
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = Layout<S, NW, KB>::DYN;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool kpair = CG == 1 && p.ksplit == 2;
    if (CG == 2 || kpair) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    // K split: one cluster per tile (the staged partial sums use the ring, so
    // a CTA never moves on to a second tile); clusters beyond what fits at
    // once wait for the hardware to schedule them
    const int groups = kpair ? p.total_units : (p.total_units < cap ? p.total_units : cap);
    cfg.gridDim = dim3((kpair ? 2 : CG) * groups, 1, 1);
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tbh, tc, p) != cudaSuccess) return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}

template <int CG, int NW, int PK>
int launch_stages(int stages, const Plan& pl, const DeviceInfo& info, const CUtensorMap& ta, const CUtensorMap& tb,
                  const CUtensorMap& tbh, const CUtensorMap& tc, const Params& p, cudaStream_t stream) {
    switch (stages) {
        case 1: return launch<CG, 1, NW, PK>(pl, info, ta, tb, tbh, tc, p, stream);
        case 2: return launch<CG, 2, NW, PK>(pl, info, ta, tb, tbh, tc, p, stream);
        case 3: return launch<CG, 3, NW, PK>(pl, info, ta, tb, tbh, tc, p, stream);
        case 4: return launch<CG, 4, NW, PK>(pl, info, ta, tb, tbh, tc, p, stream);
    }
    if constexpr (NW == 1) {
        if (stages == 5) return launch<CG, 5, 1, PK>(pl, info, ta, tb, tbh, tc, p, stream);
        if (stages == 6) return launch<CG, 6, 1, PK>(pl, info, ta, tb, tbh, tc, p, stream);
    }
    return GEMM_ERR_UNSUPPORTED_STAGES;
}

int launch_plan(int stages, const Plan& pl, const DeviceInfo& info, const CUtensorMap& ta, const CUtensorMap& tb,
                const CUtensorMap& tbh, const CUtensorMap& tc, const Params& p, cudaStream_t stream) {
    if (pl.kb == 4) {
        // half-size B boxes: only a launch of half-width units may use them
        if (p.split != 2 || p.full_units != 0) return GEMM_ERR_LAUNCH;
        if (stages == 1) return launch<1, 1, 1, 0, 4>(pl, info, ta, tb, tbh, tc, p, stream);
        if (stages == 2) return launch<1, 2, 1, 0, 4>(pl, info, ta, tb, tbh, tc, p, stream);
        return GEMM_ERR_UNSUPPORTED_STAGES;
    }
    if (pl.kb > 1) {
        switch (stages) {
            case 1: return launch<1, 1, 1, 0, 3>(pl, info, ta, tb, tbh, tc, p, stream);
            case 2: return launch<1, 2, 1, 0, 3>(pl, info, ta, tb, tbh, tc, p, stream);
            case 3: return launch<1, 3, 1, 0, 2>(pl, info, ta, tb, tbh, tc, p, stream);
        }
        return GEMM_ERR_UNSUPPORTED_STAGES;
    }
    if (pl.cg == 1) return launch_stages<1, 1, 0>(stages, pl, info, ta, tb, tbh, tc, p, stream);
    if (pk_of(pl))
        return pl.nw == 2 ? launch_stages<2, 2, 1>(stages, pl, info, ta, tb, tbh, tc, p, stream)
                          : launch_stages<2, 1, 1>(stages, pl, info, ta, tb, tbh, tc, p, stream);
    return pl.nw == 2 ? launch_stages<2, 2, 0>(stages, pl, info, ta, tb, tbh, tc, p, stream)
                      : launch_stages<2, 1, 0>(stages, pl, info, ta, tb, tbh, tc, p, stream);
}

// Whether gemm_f16_nt repacks operands TMA cannot address (defined with the
// fixed scratch array below).
bool wants_repack(int64_t M, int64_t N, int64_t K, unsigned flags);

}  // namespace f16nt
}  // namespace pws

extern "C" int gemm_f16_nt_plan(int64_t M, int64_t N, int64_t K, const gemm_f16_t* lhs, const gemm_f16_t* rhs,
                                const gemm_f16_t* out, int stages, int64_t* plan) {
    using namespace pws::f16nt;
    const int rc = validate(M, N, K, lhs, rhs, out, stages);
    if (rc != GEMM_OK) return rc;
    if (!plan) return GEMM_ERR_INVALID_ARG;
    const unsigned flags = pws::debug_flags();
    const Plan pl = make_plan(M, N, K, lhs, rhs, out, stages, pws::sm_count_or_default(), flags,
                              wants_repack(M, N, K, flags));
    plan[0] = 128 * pl.cg;
    plan[1] = 128 * pl.cg * pl.nw;
    plan[2] = BK * pl.kb;
    plan[3] = pl.cg;
    plan[4] = pl.repack ? 2 : pl.producer;       // 0 TMA, 1 cp.async, 2 repack + TMA, 3 realigning loads
    plan[5] = pl.copy_bytes;
    plan[6] = pl.store;
    plan[7] = pl.smem;
    plan[8] = pl.num_tiles;
    plan[9] = pl.num_kb;
    plan[10] = pl.ksplit;
    return GEMM_OK;
}

namespace pws {
namespace f16nt {

// K == 0: the empty sum, zeros.
int zero_output(gemm_f16_t* out, int64_t M, int64_t N, const DeviceInfo& info, cudaStream_t stream) {
    const int64_t n = M * N;
    int blocks = static_cast<int>((n + 255) / 256);
    if (blocks > 8 * info.num_sms) blocks = 8 * info.num_sms;
    return launch_pdl(zero_fill_u16, dim3(blocks), dim3(256), 0, stream, reinterpret_cast<unsigned short*>(out), n) ==
                   cudaSuccess
               ? GEMM_OK
               : GEMM_ERR_LAUNCH;
}

// Encodes the tensor maps, fills the kernel parameters and launches the GEMM
// of plan `pl`.  The TMA producer reads the operands at a_src / b_src with
// rows `ld` elements apart (the caller's own, or a repacked copy); the
// copy producer reads lhs / rhs in place.
int run_plan(const Plan& pl, const DeviceInfo& info, int64_t M, int64_t N, int64_t K, const void* lhs,
             const void* rhs, void* out, const void* a_src, const void* b_src, int64_t ld, int stages, unsigned flags,
             cudaStream_t stream) {
    CUtensorMap ta, tb, tbh, tc;
    memset(&ta, 0, sizeof(ta));
    memset(&tb, 0, sizeof(tb));
    memset(&tbh, 0, sizeof(tbh));
    memset(&tc, 0, sizeof(tc));
    if (pl.producer == kProducerTma) {
        if (!encode_tmap_f16_2d(&ta, a_src, K, M, ld * 2, BK, BM_CTA) ||
            !encode_tmap_f16_2d(&tb, b_src, K, N, ld * 2, BK, BN_CTA))
            return GEMM_ERR_LAUNCH;
    }
    if (pl.store == kStoreTma) {
        if (!encode_tmap_f16_2d(&tc, out, N, M, N * 2, EPI_COLS, 32)) return GEMM_ERR_LAUNCH;
    }
    Params p;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_kb = pl.num_kb;
    p.tiles_m = pl.tiles_m;
    p.tiles_n = pl.tiles_n;
    p.num_tiles = pl.num_tiles;
    p.producer = pl.producer;
    p.copy_bytes = pl.copy_bytes;
    p.store = pl.store;
    p.flags = flags;
    p.timeout_ns = wait_timeout_ns();
    p.lhs = static_cast<const __half*>(lhs);
    p.rhs = static_cast<const __half*>(rhs);
    p.out = static_cast<__half*>(out);
    p.status = status_word(info, stream);
    p.full_units = pl.num_tiles;
    p.split = 0;
    p.total_units = pl.num_tiles;
    p.ksplit = pl.ksplit;

    // Tail split: when the tiles leave a last, partial wave of the persistent
    // grid (or fewer tiles than the grid) and twice that many units still
    // fit in one wave, each of those tiles runs as two half-width units on the
    // wave's otherwise idle CTA groups.  The TMA and the realigning producers
    // support it (with TMA the 256 x 256 and 128 x 128 tiles need a 64-row B
    // box; a half of the wide tile is one ordinary box).  Each output element is still one
    // in-order K sum; the decision depends on the shape and the device, never
    // on S.
    const int cap = capacity_of(pl, stages, info);
    if (cap <= 0) return GEMM_ERR_LAUNCH;
    const int waves = pl.num_tiles / cap;
    const int tail = pl.num_tiles - waves * cap;
    if (pl.producer != kProducerCopy && pl.ksplit == 1 && tail > 0 && 2 * tail <= cap &&
        !(flags & GEMM_DEBUG_NO_SPLIT)) {
        if (pl.producer == kProducerTma && pl.nw == 1 &&
            !encode_tmap_f16_2d(&tbh, b_src, K, N, ld * 2, BK, BN_CTA / 2))
            return GEMM_ERR_LAUNCH;
        p.full_units = waves * cap;
        p.split = 2;
        p.total_units = waves * cap + 2 * tail;
    }
    return launch_plan(stages, pl, info, ta, tb, tbh, tc, p, stream);
}

}  // namespace f16nt
}  // namespace pws

// ---------------------------------------------------------------- the library's fixed scratch array
//
// Operands whose rows the tensor memory accelerator cannot address are
// fastest copied once into aligned rows and read by TMA (the in-place
// producer realigns every K block of every tile it reads).  The copy needs
// scratch memory, and no call may allocate: so it goes to a fixed array in
// device memory that exists from the moment the library is loaded.  Every
// GPU that loads the library holds it until the process exits.
//
// Every use of the array on a device is ordered after the previous one: the
// call's stream waits for an event recorded after the previous user's GEMM,
// on whatever stream that was, and records it again after its own.  Calls on
// different streams therefore serialise on the GPU where they share the
// array, without any host synchronisation.  A stream being captured into a
// CUDA graph cannot wait for an event recorded outside the capture, so
// gemm_f16_nt reads the operands in place there, and gemm_f16_nt_noalloc uses
// the array unordered (its caller orders such calls).
namespace pws {
namespace f16nt {

constexpr size_t kFixedScratchBytes = static_cast<size_t>(32) << 20;   // 32 MiB

// The scratch array.  In host code its name only stands in for the symbol:
// it is not a device address, and passing it to a kernel would fault (or,
// where the GPU can reach host memory, silently use the wrong memory).  The
// device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

struct FixedScratch {
    std::mutex mu;                  // per-device state, and "wait; launch; record" as one step
    void* addr[64] = {};
    cudaEvent_t done[64] = {};      // recorded after the last user's GEMM
    bool used[64] = {};
};
FixedScratch g_fixed;

bool stream_capturing(cudaStream_t stream) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &st) != cudaSuccess) {
        cudaGetLastError();
        return true;                // unknown: take the path that needs no ordering
    }
    return st != cudaStreamCaptureStatusNone;
}

// Runs body(array address) for a call on `stream`; with `ordered`, after the
// previous user of the array and before the next.  The first use on a device
// looks up the address and creates the event.
template <class F>
int with_fixed_scratch(int device, cudaStream_t stream, bool ordered, F&& body) {
    if (device < 0 || device >= 64) return GEMM_ERR_LAUNCH;
    std::lock_guard<std::mutex> lk(g_fixed.mu);
    if (!g_fixed.addr[device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fixed_scratch) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        g_fixed.addr[device] = p;
    }
    if (ordered) {
        if (!g_fixed.done[device] &&
            cudaEventCreateWithFlags(&g_fixed.done[device], cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            g_fixed.done[device] = nullptr;
            return GEMM_ERR_LAUNCH;
        }
        if (g_fixed.used[device] && cudaStreamWaitEvent(stream, g_fixed.done[device], 0) != cudaSuccess)
            return GEMM_ERR_LAUNCH;
    }
    const int rc = body(g_fixed.addr[device]);
    if (ordered) {
        // recorded even after a failed launch: the stream's earlier work
        // still orders the next user correctly
        if (cudaEventRecord(g_fixed.done[device], stream) != cudaSuccess) return GEMM_ERR_LAUNCH;
        g_fixed.used[device] = true;
    }
    return rc;
}

// Repacks both operands into the array (rows `row_align` elements apart) and
// runs the TMA plan on the copy.
int run_repacked_in_array(void* scratch, const DeviceInfo& info, int64_t M, int64_t N, int64_t K, const void* lhs,
                          const void* rhs, void* out, int stages, unsigned flags, int64_t row_align,
                          cudaStream_t stream) {
    size_t b_off = 0;
    repack_bytes(M, N, K, &b_off, row_align);
    const Plan pl = make_plan(M, N, K, lhs, rhs, out, stages, info.num_sms, flags, true);
    // The repack writes every scratch byte the GEMM then reads (rows up to
    // ceil(K/8)*8 elements, the rest of a longer row is never read), so
    // nothing left over from an earlier call is ever used.
    const int64_t Kw = repack_ld(K, 8), Kp = repack_ld(K, row_align);
    uint16_t* da = static_cast<uint16_t*>(scratch);
    uint16_t* db = reinterpret_cast<uint16_t*>(static_cast<char*>(scratch) + b_off);
    if (launch_repack(lhs, M, rhs, N, K, Kw, Kp, da, db, stream) != cudaSuccess) return GEMM_ERR_LAUNCH;
    return run_plan(pl, info, M, N, K, lhs, rhs, out, da, db, Kp, stages, flags, stream);
}

// Row alignment (elements) of a repack into the array: 64 (128-byte rows,
// which TMA reads fastest) when that fits, else 8, else 0 (does not fit).
int64_t fixed_row_align(int64_t M, int64_t N, int64_t K) {
    if (repack_bytes(M, N, K, nullptr, kPooledRowAlign) <= kFixedScratchBytes) return kPooledRowAlign;
    if (repack_bytes(M, N, K, nullptr, 8) <= kFixedScratchBytes) return 8;
    return 0;
}

// Whether gemm_f16_nt repacks operands TMA cannot address (pooled scratch,
// or the fixed array where they fit), rather than reading them in place.
bool wants_repack(int64_t M, int64_t N, int64_t K, unsigned flags) {
    if (flags & GEMM_DEBUG_IN_PLACE) return false;
    return scratch_pool_enabled() || fixed_row_align(M, N, K) > 0;
}

}  // namespace f16nt
}  // namespace pws

extern "C" int gemm_f16_nt(int64_t M, int64_t N, int64_t K, const gemm_f16_t* lhs, const gemm_f16_t* rhs,
                           gemm_f16_t* out, int stages, cudaStream_t stream) {
    using namespace pws;
    using namespace pws::f16nt;
    int rc = validate(M, N, K, lhs, rhs, out, stages);
    if (rc != GEMM_OK) return rc;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceInfo info;
    rc = current_device(&info);
    if (rc != GEMM_OK) return rc;
    if (K == 0) return zero_output(out, M, N, info, stream);
    const unsigned flags = debug_flags();
    Plan pl = make_plan(M, N, K, lhs, rhs, out, stages, info.num_sms, flags, wants_repack(M, N, K, flags));

    // Operands whose rows TMA cannot address are copied to aligned rows and
    // read by TMA: into pooled scratch with gemm_set_scratch_pool(1), else
    // into the library's fixed array where they fit (ordered after its
    // previous user).  Otherwise -- too large, a stream being captured, the
    // pool out of memory -- the realigning producer reads them in place.
    if (pl.repack && !scratch_pool_enabled()) {
        const int64_t align = fixed_row_align(M, N, K);
        if (align > 0 && !stream_capturing(stream))
            return with_fixed_scratch(info.device, stream, true, [&](void* scratch) {
                return run_repacked_in_array(scratch, info, M, N, K, lhs, rhs, out, stages, flags, align, stream);
            });
        pl = make_plan(M, N, K, lhs, rhs, out, stages, info.num_sms, flags);
    }
    const void* a_src = lhs;
    const void* b_src = rhs;
    int64_t ld = K;
    void* scratch = nullptr;
    if (pl.repack) {
        size_t b_off = 0;
        const size_t bytes = repack_bytes(M, N, K, &b_off, kPooledRowAlign);
        scratch = scratch_alloc(info, bytes, stream);
        if (scratch) {
            const int64_t Kw = repack_ld(K, 8), Kp = repack_ld(K, kPooledRowAlign);
            uint16_t* da = static_cast<uint16_t*>(scratch);
            uint16_t* db = reinterpret_cast<uint16_t*>(static_cast<char*>(scratch) + b_off);
            if (launch_repack(lhs, M, rhs, N, K, Kw, Kp, da, db, stream) != cudaSuccess) {
                scratch_free(scratch, stream);
                return GEMM_ERR_LAUNCH;
            }
            a_src = da;
            b_src = db;
            ld = Kp;
        } else {
            pl = make_plan(M, N, K, lhs, rhs, out, stages, info.num_sms, flags);
        }
    }
    rc = run_plan(pl, info, M, N, K, lhs, rhs, out, a_src, b_src, ld, stages, flags, stream);
    scratch_free(scratch, stream);       // stream-ordered: after the GEMM has read it
    return rc;
}

// ---------------------------------------------------------------- no-allocation variant
//
// gemm_f16_nt_noalloc is gemm_f16_nt for callers that cannot allocate device
// memory: code running under a fixed device-memory budget that must not
// grow, code that must not call into the allocator at all (it can
// synchronise or fail at a point the caller cannot handle), or code that has
// reserved all device memory up front.  It never takes pooled scratch,
// whatever gemm_set_scratch_pool says: operands TMA cannot address go to the
// fixed array (rows ceil(K/8)*8 elements apart, the documented limit) or,
// when they do not fit, are read in place.
extern "C" int gemm_f16_nt_noalloc(int64_t M, int64_t N, int64_t K, const gemm_f16_t* lhs, const gemm_f16_t* rhs,
                                   gemm_f16_t* out, int stages, cudaStream_t stream) {
    using namespace pws;
    using namespace pws::f16nt;
    int rc = validate(M, N, K, lhs, rhs, out, stages);
    if (rc != GEMM_OK) return rc;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceInfo info;
    rc = current_device(&info);
    if (rc != GEMM_OK) return rc;
    if (K == 0) return zero_output(out, M, N, info, stream);
    const unsigned flags = debug_flags();
    const bool fits = repack_bytes(M, N, K, nullptr, 8) <= kFixedScratchBytes;
    const Plan pl = make_plan(M, N, K, lhs, rhs, out, stages, info.num_sms, flags,
                              fits && !(flags & GEMM_DEBUG_IN_PLACE));
    if (!pl.repack) return run_plan(pl, info, M, N, K, lhs, rhs, out, lhs, rhs, K, stages, flags, stream);
    return with_fixed_scratch(info.device, stream, !stream_capturing(stream), [&](void* scratch) {
        return run_repacked_in_array(scratch, info, M, N, K, lhs, rhs, out, stages, flags, 8, stream);
    });
}
