// gemm_s32_nn.cu -- out[M,N] = lhs[M,K] . rhs[K,N] over int32 on the CUDA cores.
//
// The schedule is the two-buffer swap pipeline of the Croqtile tutorial
// ch.6, section "使用 swap 的双缓冲": K is cut into tiles of 16
// ("with tile_k in 16"); the prologue issues the asynchronous copy of tile 0
// into buffer 0; each steady iteration t = 1..T-1 ("foreach tile_k(1:)")
// issues tile t into the other buffer, multiplies the buffer holding tile
// t-1, and swaps the two buffer names (a register swap; no data moves --
// section "swap：交换的是名称，不是字节"); the epilogue multiplies the last
// tile.  The copies are cp.async; as the TileLang tutorial ch.22 section 4.3
// notes, __syncthreads does not wait for them, so every read of a buffer is
// preceded by cp.async.wait_group and then __syncthreads (read after write),
// and every refill by a __syncthreads after the last read (write after read).
//
// Each thread owns a TM x TN block of outputs held in registers and does
// TM*TN wrapping 32-bit multiply-adds per K step (IMAD).
#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "pwsgemm.h"

namespace pws {
namespace s32nn {

// Only the largest tile of each kernel is chosen for outputs that can have
// more row tiles than a grid's y extent (65535); smaller tiles are chosen only
// while a few hundred row tiles fill the GPU.
constexpr int kPlainLargestTile = 128;
constexpr int kRingLargestTile = 64;

// For a kernel that may be launched on more row tiles than a grid's y extent
// holds: the origin of this block's tile from a 1-D grid numbering the tiles
// row by row, or from the 2-D grid (column tiles x row tiles) where that
// holds them.  gridDim.x equals the column-tile count only on the 2-D grid
// (or with one row of tiles, where both readings agree).  Other kernels read
// the 2-D grid directly: on the page's 128 x 256 x 256 problem any other
// form of that reading measured 0.1-0.8 us slower (the compiler schedules
// these latency-bound kernels differently).
template <int BN>
__device__ __forceinline__ int tall_row_tile(int N) {
    const unsigned tiles_n = static_cast<unsigned>((N + BN - 1) / BN);
    return static_cast<int>(gridDim.x == tiles_n ? blockIdx.y : blockIdx.x / tiles_n);
}
template <int BN>
__device__ __forceinline__ int tall_col_tile(int N) {
    const unsigned tiles_n = static_cast<unsigned>((N + BN - 1) / BN);
    return static_cast<int>(gridDim.x == tiles_n ? blockIdx.x : blockIdx.x % tiles_n);
}

constexpr int BK = 16;          // K per tile (the page's 256 / #tile_k)
constexpr int THREADS = 256;
constexpr int APAD = 4;         // words of padding per A row in shared memory

template <int BM, int BN, int TM, int TN, int ABYTES, int BBYTES>
__global__ void __launch_bounds__(THREADS)
gemm_s32_nn_kernel(int M, int N, int K, const int32_t* __restrict__ lhs, const int32_t* __restrict__ rhs,
                   int32_t* __restrict__ out) {
    static_assert((BM / TM) * (BN / TN) == THREADS, "one thread per TM x TN block");
    // Two buffers per operand: A tiles [BM][BK] (k contiguous), B tiles [BK][BN].
    __shared__ __align__(16) int32_t As[2][BM][BK + APAD];
    __shared__ __align__(16) int32_t Bs[2][BK][BN];

    const int tid = threadIdx.x;
    const int tx = tid % (BN / TN);
    const int ty = tid / (BN / TN);
    const int m0 = BM == kPlainLargestTile ? tall_row_tile<BN>(N) * BM : blockIdx.y * BM;
    const int n0 = BM == kPlainLargestTile ? tall_col_tile<BN>(N) * BN : blockIdx.x * BN;
    const int T = (K + BK - 1) / BK;
    // launched as a programmatic dependent: the previous grid's writes first
    grid_dependency_wait();
    allow_dependent_launch();

    // Issue the copies of K tile `t` into buffer `buf` (zero-fill outside M, N, K).
    auto issue = [&](int t, int buf) {
        const int k0 = t * BK;
        constexpr int AE = ABYTES / 4;                 // int32 per A copy
        constexpr int A_COPIES = BM * (BK / AE);
        for (int i = tid; i < A_COPIES; i += THREADS) {
            const int r = i / (BK / AE), c = (i % (BK / AE)) * AE;
            const int gm = m0 + r, gk = k0 + c;
            const bool ok = gm < M && gk < K;
            const int32_t* src = ok ? lhs + (int64_t)gm * K + gk : lhs;
            cp_async<ABYTES>(smem_u32(&As[buf][r][c]), src, ok ? ABYTES : 0);
        }
        constexpr int BE = BBYTES / 4;
        constexpr int B_COPIES = BK * (BN / BE);
        for (int i = tid; i < B_COPIES; i += THREADS) {
            const int r = i / (BN / BE), c = (i % (BN / BE)) * BE;
            const int gk = k0 + r, gn = n0 + c;
            const bool ok = gk < K && gn < N;
            const int32_t* src = ok ? rhs + (int64_t)gk * N + gn : rhs;
            cp_async<BBYTES>(smem_u32(&Bs[buf][r][c]), src, ok ? BBYTES : 0);
        }
        cp_async_commit();
    };

    uint32_t acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0u;       // the zero start of "+="

    // Multiply-accumulate over the 16 K values of buffer `buf`.
    auto compute = [&](int buf) {
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            uint32_t a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = static_cast<uint32_t>(As[buf][ty * TM + i][k]);
#pragma unroll
            for (int j = 0; j < TN; ++j) b[j] = static_cast<uint32_t>(Bs[buf][k][tx * TN + j]);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] += a[i] * b[j];   // wraps mod 2^32
        }
    };

    if (T > 0) {
        // prologue: tile 0 into buffer 0
        int cur = 0, nxt = 1;
        issue(0, cur);
        // steady state: load tile t, compute tile t-1, swap
        for (int t = 1; t < T; ++t) {
            issue(t, nxt);
            cp_async_wait_group<1>();      // tile t-1 has landed ...
            __syncthreads();               // ... and is visible to every thread
            compute(cur);
            __syncthreads();               // everyone is done reading `cur` before it is refilled
            const int tmp = cur;           // swap the names, not the bytes
            cur = nxt;
            nxt = tmp;
        }
        // epilogue: compute the last tile
        cp_async_wait_group<0>();
        __syncthreads();
        compute(cur);
    }

#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int gm = m0 + ty * TM + i;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int gn = n0 + tx * TN + j;
            if (gn < N) out[(int64_t)gm * N + gn] = static_cast<int32_t>(acc[i][j]);
        }
    }
}

// The grid: 2-D (column tiles x row tiles) where the row tiles fit in a
// grid's y extent, which measured 0.1-0.3 us faster on the page's problem
// than numbering the tiles along one dimension; 1-D beyond, at most 2^31 - 1
// tiles.  With the smallest (16 x 16) tile that bounds the output below
// 2^39 elements, more than any device holds.
inline bool too_many_tiles(int64_t M, int64_t N) { return ((M + 15) / 16) * ((N + 15) / 16) >= (1ll << 31); }

// A grid of 0 blocks (a launch error) if a kernel that reads only the 2-D
// grid would need the 1-D one.
inline dim3 tile_grid(int M, int N, int BM, int BN, bool tall_ok) {
    const unsigned tiles_m = static_cast<unsigned>((M + BM - 1) / BM), tiles_n = static_cast<unsigned>((N + BN - 1) / BN);
    if (tiles_m <= 65535u) return dim3(tiles_n, tiles_m);
    if (!tall_ok) return dim3(0);
    return dim3(static_cast<unsigned>(static_cast<uint64_t>(tiles_m) * tiles_n));
}

template <int BM, int BN, int TM, int TN>
cudaError_t launch_tile(int M, int N, int K, const int32_t* lhs, const int32_t* rhs, int32_t* out,
                        bool a16, bool b16, cudaStream_t stream) {
    const dim3 grid = tile_grid(M, N, BM, BN, BM == kPlainLargestTile);
    // 16-byte copies need 16-byte aligned rows; otherwise one element per copy.
    const bool b_vec = b16 && BN % 4 == 0;
    if (a16 && b_vec)
        return launch_pdl(gemm_s32_nn_kernel<BM, BN, TM, TN, 16, 16>, grid, dim3(THREADS), 0, stream, M, N, K, lhs, rhs, out);
    else if (a16)
        return launch_pdl(gemm_s32_nn_kernel<BM, BN, TM, TN, 16, 4>, grid, dim3(THREADS), 0, stream, M, N, K, lhs, rhs, out);
    else if (b_vec)
        return launch_pdl(gemm_s32_nn_kernel<BM, BN, TM, TN, 4, 16>, grid, dim3(THREADS), 0, stream, M, N, K, lhs, rhs, out);
    else
        return launch_pdl(gemm_s32_nn_kernel<BM, BN, TM, TN, 4, 4>, grid, dim3(THREADS), 0, stream, M, N, K, lhs, rhs, out);
}

}  // namespace s32nn
}  // namespace pws

extern "C" int gemm_s32_nn(int64_t M, int64_t N, int64_t K, const int32_t* lhs, const int32_t* rhs,
                           int32_t* out, cudaStream_t stream) {
    using namespace pws;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31)) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (s32nn::too_many_tiles(M, N)) return GEMM_ERR_INVALID_ARG;
    if (!out || (K > 0 && (!lhs || !rhs))) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(lhs) |
         reinterpret_cast<uintptr_t>(rhs)) & 3u)
        return GEMM_ERR_ALIGNMENT;
    const uint64_t out_b = (uint64_t)M * N * 4;
    if (K > 0 && (ranges_overlap(out, out_b, lhs, (uint64_t)M * K * 4) ||
                  ranges_overlap(out, out_b, rhs, (uint64_t)K * N * 4)))
        return GEMM_ERR_INVALID_ARG;

    DeviceInfo info;
    const int rc = current_device(&info);
    if (rc != GEMM_OK) return rc;

    const bool a16 = (K % 4 == 0) && (reinterpret_cast<uintptr_t>(lhs) % 16 == 0);
    const bool b16 = (N % 4 == 0) && (reinterpret_cast<uintptr_t>(rhs) % 16 == 0);
    // Largest output tile that still gives at least one block per SM; the
    // smallest (16 x 16, one output per thread: the page's [16,16]-thread
    // blocks) when none does.
    auto blocks = [&](int bm, int bn) { return ((M + bm - 1) / bm) * ((N + bn - 1) / bn); };
    cudaError_t e;
    if (blocks(128, 128) >= info.num_sms)
        e = s32nn::launch_tile<128, 128, 8, 8>((int)M, (int)N, (int)K, lhs, rhs, out, a16, b16, stream);
    else if (blocks(64, 64) >= info.num_sms)
        e = s32nn::launch_tile<64, 64, 4, 4>((int)M, (int)N, (int)K, lhs, rhs, out, a16, b16, stream);
    else if (blocks(32, 32) >= info.num_sms)
        e = s32nn::launch_tile<32, 32, 2, 2>((int)M, (int)N, (int)K, lhs, rhs, out, a16, b16, stream);
    else
        e = s32nn::launch_tile<16, 16, 1, 1>((int)M, (int)N, (int)K, lhs, rhs, out, a16, b16, stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

// ---------------------------------------------------------------- S-slot ring
//
// The same product with S shared-memory slots instead of two: the Croqtile
// tutorial ch.6 generalises swap(f0, f1) to rotate(f0, f1, f2) for three
// buffers ("swap：交换的是名称，不是字节"), and the CUDA tutorial ch.4,
// section 4.8.3 fills S - 1 slots before its main loop.  Here the prologue
// issues tiles 0 .. S-2; iteration t waits until tile t has landed
// (cp.async.wait_group, then __syncthreads), issues tile t + S - 1 into the
// slot tile t - 1 vacated and multiplies slot t mod S.  With S >= 3 the
// refill follows the barrier that publishes tile t, which also orders it
// after every read of tile t - 1: one barrier per tile.  With S = 2 the
// refill is issued before the wait and a second barrier guards the slot.
// Rotating the slot index is rotate() over S handles.
// With S tiles in flight the load latency of the small page-size problem is
// paid about T / (S - 1) times instead of T times; results are bit-identical
// to the two-buffer kernel (same products, same order, exact arithmetic).
namespace pws {
namespace s32nn {

template <int BM, int BN, int TM, int TN, int CBYTES, int S>
__global__ void __launch_bounds__(THREADS)
gemm_s32_nn_ring_kernel(int M, int N, int K, const int32_t* __restrict__ lhs, const int32_t* __restrict__ rhs,
                        int32_t* __restrict__ out) {
    static_assert(S >= 2 && S <= 6, "ring slots");
    static_assert((BM / TM) * (BN / TN) == THREADS, "one thread per TM x TN block");
    constexpr int A_WORDS = BM * (BK + APAD);      // one slot of A: [BM][BK + APAD]
    constexpr int B_WORDS = BK * BN;               // one slot of B: [BK][BN]
    extern __shared__ __align__(16) int32_t ring[];
    int32_t* const As = ring;
    int32_t* const Bs = ring + S * A_WORDS;

    const int tid = threadIdx.x;
    const int tx = tid % (BN / TN);
    const int ty = tid / (BN / TN);
    const int m0 = BM == kRingLargestTile ? tall_row_tile<BN>(N) * BM : blockIdx.y * BM;
    const int n0 = BM == kRingLargestTile ? tall_col_tile<BN>(N) * BN : blockIdx.x * BN;
    const int T = (K + BK - 1) / BK;
    // launched as a programmatic dependent: the previous grid's writes first
    grid_dependency_wait();
    allow_dependent_launch();

    auto issue = [&](int t, int slot) {
        const int k0 = t * BK;
        constexpr int E = CBYTES / 4;
        int32_t* a = As + slot * A_WORDS;
        int32_t* b = Bs + slot * B_WORDS;
        for (int i = tid; i < BM * (BK / E); i += THREADS) {
            const int r = i / (BK / E), c = (i % (BK / E)) * E;
            const int gm = m0 + r, gk = k0 + c;
            const bool ok = gm < M && gk < K;
            cp_async<CBYTES>(smem_u32(a + r * (BK + APAD) + c), ok ? lhs + (int64_t)gm * K + gk : lhs, ok ? CBYTES : 0);
        }
        for (int i = tid; i < BK * (BN / E); i += THREADS) {
            const int r = i / (BN / E), c = (i % (BN / E)) * E;
            const int gk = k0 + r, gn = n0 + c;
            const bool ok = gk < K && gn < N;
            cp_async<CBYTES>(smem_u32(b + r * BN + c), ok ? rhs + (int64_t)gk * N + gn : rhs, ok ? CBYTES : 0);
        }
    };

    uint32_t acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0u;

    // prologue: S - 1 tiles in flight
    for (int t = 0; t < S - 1; ++t) {
        if (t < T) issue(t, t);
        cp_async_commit();
    }
    // The slot names rotate by one per iteration (the page's rotate): tile t
    // is read from slot `cur`, tile t + S - 1 is loaded into slot `nxt`, the
    // one tile t - 1 vacated.  With S a run-time value, computing t mod S
    // made the loop execute 60 % more instructions and take twice the cycles
    // on GB300; with S fixed at compile time and the names incremented, the
    // loop is the two-buffer kernel's plus the extra slots in flight.
    //
    // With S >= 3 slots the refill of tile t + S - 1 is issued after the
    // barrier that publishes tile t: that barrier also follows every
    // thread's reads of tile t - 1, whose slot the refill overwrites, so one
    // barrier per tile orders both hazards while S - 2 later tiles are still
    // in flight during the wait.  With two slots that order would leave no
    // tile in flight during the wait, so S = 2 issues first and
    // synchronises twice (on the page's 128 x 256 x 256 problem, one barrier
    // measured 4.2-4.3 us at S = 3..6 against 4.7-4.8 us with two; at S = 2,
    // 5.2 us against 4.5 us).
    constexpr bool kOneBarrier = S >= 3;
    int cur = 0, nxt = S - 1;
    for (int t = 0; t < T; ++t) {
        if constexpr (kOneBarrier) {
            cp_async_wait_group<S - 2>();    // tile t has landed ...
            __syncthreads();                 // ... is visible, and tile t - 1's slot is free
            if (t + S - 1 < T) issue(t + S - 1, nxt);
            cp_async_commit();
        } else {
            if (t + S - 1 < T) issue(t + S - 1, nxt);
            cp_async_commit();
            cp_async_wait_group<S - 1>();    // tile t has landed ...
            __syncthreads();                 // ... and is visible to all threads
        }
        const int32_t* a = As + cur * A_WORDS;
        const int32_t* b = Bs + cur * B_WORDS;
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            uint32_t av[TM], bv[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) av[i] = static_cast<uint32_t>(a[(ty * TM + i) * (BK + APAD) + k]);
#pragma unroll
            for (int j = 0; j < TN; ++j) bv[j] = static_cast<uint32_t>(b[k * BN + tx * TN + j]);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] += av[i] * bv[j];
        }
        if constexpr (!kOneBarrier) __syncthreads();   // slot `cur` is free for tile t + S
        cur = cur + 1 == S ? 0 : cur + 1;
        nxt = nxt + 1 == S ? 0 : nxt + 1;
    }
    cp_async_wait_group<0>();

#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int gm = m0 + ty * TM + i;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int gn = n0 + tx * TN + j;
            if (gn < N) out[(int64_t)gm * N + gn] = static_cast<int32_t>(acc[i][j]);
        }
    }
}

template <int BM, int BN, int TM, int TN, int CBYTES, int S>
cudaError_t launch_ring_s(int M, int N, int K, const int32_t* lhs, const int32_t* rhs, int32_t* out, int device,
                          cudaStream_t stream) {
    const dim3 grid = tile_grid(M, N, BM, BN, BM == kRingLargestTile);
    constexpr size_t smem = static_cast<size_t>(S) * (BM * (BK + APAD) + BK * BN) * sizeof(int32_t);
    auto k = gemm_s32_nn_ring_kernel<BM, BN, TM, TN, CBYTES, S>;
    static std::atomic<bool> configured[64] = {};       // concurrent first calls store the same value
    if (smem > 48 * 1024 && !configured[device].load(std::memory_order_relaxed)) {   // above the default limit: opt in once
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
            return cudaGetLastError();
        configured[device].store(true, std::memory_order_relaxed);
    }
    return launch_pdl(k, grid, dim3(THREADS), smem, stream, M, N, K, lhs, rhs, out);
}

template <int BM, int BN, int TM, int TN, int CBYTES>
cudaError_t launch_ring_c(int M, int N, int K, int S, const int32_t* lhs, const int32_t* rhs, int32_t* out, int device,
                          cudaStream_t stream) {
    switch (S) {
        case 2: return launch_ring_s<BM, BN, TM, TN, CBYTES, 2>(M, N, K, lhs, rhs, out, device, stream);
        case 3: return launch_ring_s<BM, BN, TM, TN, CBYTES, 3>(M, N, K, lhs, rhs, out, device, stream);
        case 4: return launch_ring_s<BM, BN, TM, TN, CBYTES, 4>(M, N, K, lhs, rhs, out, device, stream);
        case 5: return launch_ring_s<BM, BN, TM, TN, CBYTES, 5>(M, N, K, lhs, rhs, out, device, stream);
        case 6: return launch_ring_s<BM, BN, TM, TN, CBYTES, 6>(M, N, K, lhs, rhs, out, device, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int BM, int BN, int TM, int TN>
cudaError_t launch_ring(int M, int N, int K, int S, const int32_t* lhs, const int32_t* rhs, int32_t* out,
                        bool vec16, int device, cudaStream_t stream) {
    return vec16 ? launch_ring_c<BM, BN, TM, TN, 16>(M, N, K, S, lhs, rhs, out, device, stream)
                 : launch_ring_c<BM, BN, TM, TN, 4>(M, N, K, S, lhs, rhs, out, device, stream);
}

}  // namespace s32nn
}  // namespace pws

extern "C" int gemm_s32_nn_ring(int64_t M, int64_t N, int64_t K, const int32_t* lhs, const int32_t* rhs,
                                int32_t* out, int stages, cudaStream_t stream) {
    using namespace pws;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31)) return GEMM_ERR_INVALID_ARG;
    if (stages < 2 || stages > 6) return GEMM_ERR_UNSUPPORTED_STAGES;
    if (M == 0 || N == 0) return GEMM_OK;
    if (s32nn::too_many_tiles(M, N)) return GEMM_ERR_INVALID_ARG;
    if (!out || (K > 0 && (!lhs || !rhs))) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(lhs) |
         reinterpret_cast<uintptr_t>(rhs)) & 3u)
        return GEMM_ERR_ALIGNMENT;
    const uint64_t out_b = (uint64_t)M * N * 4;
    if (K > 0 && (ranges_overlap(out, out_b, lhs, (uint64_t)M * K * 4) ||
                  ranges_overlap(out, out_b, rhs, (uint64_t)K * N * 4)))
        return GEMM_ERR_INVALID_ARG;
    DeviceInfo info;
    const int rc = current_device(&info);
    if (rc != GEMM_OK) return rc;
    // 16-byte copies need 16-byte aligned rows on both sides, else one element per copy
    const bool vec16 = (K % 4 == 0) && (N % 4 == 0) && (reinterpret_cast<uintptr_t>(lhs) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(rhs) % 16 == 0);
    auto blocks = [&](int bm, int bn) { return ((M + bm - 1) / bm) * ((N + bn - 1) / bn); };
    cudaError_t e;
    if (blocks(64, 64) >= info.num_sms)
        e = s32nn::launch_ring<64, 64, 4, 4>((int)M, (int)N, (int)K, stages, lhs, rhs, out, vec16, info.device, stream);
    else if (blocks(32, 32) >= info.num_sms)
        e = s32nn::launch_ring<32, 32, 2, 2>((int)M, (int)N, (int)K, stages, lhs, rhs, out, vec16, info.device, stream);
    else
        e = s32nn::launch_ring<16, 16, 1, 1>((int)M, (int)N, (int)K, stages, lhs, rhs, out, vec16, info.device, stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}
