/*
 * pwsgemm.h -- C ABI of the pipelined, warp-specialized GEMM library for
 * NVIDIA GB300 (sm_103a).
 *
 * Two products, both "a tiled matrix multiply whose K loop is software
 * pipelined" as the Croqtile tutorial ch.6 ("同步：流水线、事件与双缓冲")
 * builds it:
 *
 *   gemm_s32_nn  -- the s32 kernel of section "使用 swap 的双缓冲": a
 *                   two-buffer ring filled by asynchronous copies, with a
 *                   prologue load, steady iterations (load tile t, compute
 *                   tile t-1, swap the buffer names) and an epilogue compute.
 *                   Runs on the CUDA cores (wrapping 32-bit multiply-add).
 *   gemm_f16_nt  -- the f16 kernel of section "带 event 的 1P1C 内核": a
 *                   producer role fills an S-slot shared-memory ring guarded
 *                   by full[s]/empty[s] events (stage = k % S, every empty
 *                   seeded before the loop); a consumer role multiplies on
 *                   the tensor cores and releases each slot once its
 *                   multiply has completed ("mma.commit"), then writes the
 *                   output tile.  Accumulates in fp32, stores f16.
 *
 * Conventions shared by every entry point:
 *   - Matrices are dense and row-major, in DEVICE memory of the current CUDA
 *     device, owned by the caller.  `out` must not overlap `lhs` or `rhs`.
 *   - Calls are asynchronous and stream-ordered on `stream` (0 = the legacy
 *     default stream).  They do not synchronize and do not allocate device
 *     memory per call.
 *   - Kernels are launched with programmatic stream serialization: a call's
 *     kernel may be scheduled while the previous kernel on the stream is
 *     still running, but it reads and writes global memory only after that
 *     kernel has completed, so stream order holds for every memory effect.
 *     It also lets the next kernel on the stream be scheduled early; a
 *     caller's own kernel launched with that attribute after a call must
 *     execute griddepcontrol.wait (cudaGridDependencySynchronize) before
 *     reading the call's output, as that attribute always requires.
 *   - Argument errors are reported by the return value BEFORE any launch;
 *     nothing is written in that case.
 *   - M == 0 or N == 0 is a successful no-op.  K == 0 writes zeros to `out`
 *     (the empty sum).
 *   - A wait inside a kernel that exceeds the wait limit (see
 *     gemm_set_wait_timeout_ns) records GEMM_ERR_TIMEOUT in the status word
 *     of the call's stream and the kernel returns; gemm_device_status(stream)
 *     reads and clears it.
 *   - Per-device state (the status words, the no-alloc array's address, the
 *     kernels' shared-memory settings) is set up on the first call on a
 *     device and kept for the life of the process: after cudaDeviceReset the
 *     library must not be called again in that process.
 */
#ifndef PWSGEMM_H_
#define PWSGEMM_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The library is built with hidden visibility: the functions declared here
 * are its only exported symbols.  Its per-process state (tensor-map caches,
 * per-kernel shared-memory settings) therefore stays private to one copy of
 * the library even when several copies are loaded into the same process. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

/* Status codes returned by every entry point. */
typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,        /* negative size, null pointer, overlap, size too large */
    GEMM_ERR_ALIGNMENT = 2,          /* pointer not aligned to its element size               */
    GEMM_ERR_UNSUPPORTED_STAGES = 3, /* stages outside 1..6                                   */
    GEMM_ERR_UNSUPPORTED_ARCH = 4,   /* current device is not compute capability 10.3        */
    GEMM_ERR_LAUNCH = 5,             /* CUDA runtime or driver call failed                    */
    GEMM_ERR_TIMEOUT = 6             /* a bounded device wait expired (see gemm_device_status)*/
} gemm_status;

/* Binary16 values are passed as their IEEE 754 bit patterns. */
typedef uint16_t gemm_f16_t;

/*
 * gemm_s32_nn -- out[M,N] = lhs[M,K] . rhs[K,N] over int32.
 *
 * Croqtile tutorial ch.6, section "使用 swap 的双缓冲" (the s32 matmul with
 * "with tile_k in 16", "foreach tile_k(1:)" and swap(lf0, lf1)).
 *
 *   lhs : int32 [M, K], row-major (row stride K elements), 4-byte aligned
 *   rhs : int32 [K, N], row-major (row stride N elements), 4-byte aligned
 *   out : int32 [M, N], row-major, written (not accumulated into)
 *
 * The sum of products is computed with wrapping 32-bit arithmetic (two's
 * complement, i.e. the exact sum modulo 2^32).  K is cut into tiles of 16;
 * a partial last tile and partial edge tiles are zero-filled.
 *
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG (M, N or K negative or not below
 * 2^31, ceil(M/16) * ceil(N/16) not below 2^31, a null pointer with
 * M*N > 0, or out overlapping an input), GEMM_ERR_ALIGNMENT (a pointer not
 * 4-byte aligned), GEMM_ERR_UNSUPPORTED_ARCH or GEMM_ERR_LAUNCH.
 */
int gemm_s32_nn(int64_t M, int64_t N, int64_t K, const int32_t* lhs, const int32_t* rhs,
                int32_t* out, cudaStream_t stream);

/*
 * gemm_s32_nn_ring -- gemm_s32_nn with an S-slot ring instead of two buffers.
 *
 * Croqtile tutorial ch.6, section "swap：交换的是名称，不是字节" (rotate(f0, f1,
 * f2) over three buffers, generalised to S) and the CUDA tutorial ch.4,
 * section 4.8.3 (a pipeline that fills S - 1 slots before its main loop).
 * The prologue issues K tiles 0..S-2; iteration t issues tile t+S-1 into the
 * slot tile t-1 vacated, waits for tile t, multiplies it.  S - 1 tiles are in
 * flight while one is multiplied.
 *
 *   Arguments, layouts and wrapping arithmetic as gemm_s32_nn; the result is
 *   bit-identical to it.  stages : S, 2..6 (2 is the double buffer).
 *
 * Returns the codes of gemm_s32_nn, or GEMM_ERR_UNSUPPORTED_STAGES for S
 * outside 2..6.
 */
int gemm_s32_nn_ring(int64_t M, int64_t N, int64_t K, const int32_t* lhs, const int32_t* rhs,
                     int32_t* out, int stages, cudaStream_t stream);

/*
 * gemm_f16_nt -- out[M,N] = f16( lhs[M,K] . rhs[N,K]^T ), fp32 accumulation.
 *
 * Croqtile tutorial ch.6, section "带 event 的 1P1C 内核" (lhs declared
 * [M, K], rhs declared [N, K], multiplied with mma.row.row: C = A . B^T),
 * with the ring index of section "环形索引" and the seeding of "消费者路径";
 * the phase bit of each reused event follows TileLang tutorial ch.22,
 * section 3.2 (parity = (k / S) mod 2).
 *
 *   lhs    : binary16 [M, K], row-major (row stride K elements), 2-byte aligned
 *   rhs    : binary16 [N, K], row-major (row stride K elements), 2-byte aligned
 *   out    : binary16 [M, N], row-major, written; each element is the fp32 sum
 *            rounded to nearest-even binary16 (overflow gives +-inf)
 *   stages : S, the number of shared-memory ring slots, 1..6.  S = 1 is the
 *            single-buffer case (load and multiply serialise).  The result is
 *            bitwise identical for every S.
 *
 * The producer uses the tensor memory accelerator (TMA) when both operands
 * start on 16-byte boundaries and K is a multiple of 8 (row stride a multiple
 * of 16 bytes).  Otherwise the call first copies both operands into aligned
 * rows (ceil(K/64)*64 elements apart where that fits, else ceil(K/8)*8) of a
 * fixed 32 MiB array in device memory that the library holds from load time,
 * and TMA reads the copy; nothing is allocated.  Every use of that array on a
 * device is ordered after the previous one with an event (the call's stream
 * waits, on the GPU, for the previous user's GEMM), so calls on different
 * streams never overlap on it; such calls serialise with each other.  When
 * the copy does not fit in the array, or `stream` is being captured into a
 * CUDA graph (which cannot wait for an event recorded outside it), eight
 * producer warps per CTA read the operands in place instead: each row's K
 * strip is loaded as the aligned 16-byte blocks that hold it, shifted into
 * place in registers and written into the same swizzled ring slot TMA would
 * fill, on any tile (slower for large operands).  gemm_set_scratch_pool
 * offers pooled scratch instead of the array.  Every path gives the same
 * result bits.  Partial tiles are zero-filled on load and clipped on store.
 *
 * Output tiles: 256 x 256 on a CTA pair (two SMs sharing one tcgen05 MMA),
 * or 128 x 128 on one CTA.  The pair tile is used when TMA feeds it and it
 * needs fewer waves of CTA groups than the single-CTA tile (or as many, with
 * at least as many pair tiles as half the SMs); the asynchronous-copy
 * producer (GEMM_DEBUG_FORCE_COPY_PRODUCER) always uses the single-CTA tile.  With stages <= 4 the pair uses
 * a 256 x 512 tile instead where that adds no padding columns: each ring
 * slot then carries two B boxes, so each operand byte copied into shared
 * memory feeds 4/3 as many flops (5 and 6 slots of that size do not fit in
 * shared memory).  The 256 x 256 tile is kept where the 256 x 512 one would
 * leave pairs idle that it fills: when its tiles fit in one wave of pairs,
 * or, with 3 or 4 slots, when the 256 x 512 tiles are fewer than the pairs
 * and the 256 x 256 ones take one wave and a tail of at most half of it.
 * Every tile sums each output element over K in the same order, so the tile
 * choice never changes the result.
 *
 * K split: when the 128 x 128 tile is used, the tiles fill at most half of
 * the SMs and K spans at least 32 blocks of 64 (K > 1984), each tile is
 * computed by a cluster of two CTAs.  One sums the first ceil(nkb/2) K
 * blocks, the other the rest (nkb = ceil(K/64)), each into its own fp32
 * accumulator.  The two partial sums are added (one fp32 addition) before
 * the rounding to f16.  Such an output is therefore
 * f16(sum over the first half + sum over the second half), a different
 * rounding of the same exact sum than the one-pass tiles give.  The choice
 * depends on M, N and K only, so the result is still the same for every S.
 *
 * The kernel is persistent (the K split aside, which runs one cluster per
 * tile): a grid of as many CTA groups as fit on the GPU strides over the
 * output tiles.  When the tile count leaves a last, partial
 * wave that fills at most half of the grid, each tile of that wave runs as
 * two units, its left and right halves of columns, on the wave's otherwise
 * idle CTA groups.  Each half runs the whole K loop, so no partial sums are
 * combined, no scratch is needed and every output element has the same
 * summation order whether or not its tile was split.
 *
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_ALIGNMENT (a pointer not
 * 2-byte aligned), GEMM_ERR_UNSUPPORTED_STAGES, GEMM_ERR_UNSUPPORTED_ARCH or
 * GEMM_ERR_LAUNCH.  M, N, K must each be below 2^31, and the output must
 * hold fewer than 2^31 tiles of 128 x 128 (ceil(M/128) * ceil(N/128)), else
 * GEMM_ERR_INVALID_ARG.
 */
int gemm_f16_nt(int64_t M, int64_t N, int64_t K, const gemm_f16_t* lhs, const gemm_f16_t* rhs,
                gemm_f16_t* out, int stages, cudaStream_t stream);

/*
 * gemm_f16_nt_noalloc -- gemm_f16_nt for callers that cannot allocate device
 * memory.  The pages have no counterpart to this entry point.
 *
 * Same arguments, layouts, results and return codes as gemm_f16_nt, and the
 * same fixed 32 MiB array for operands whose rows the tensor memory
 * accelerator cannot address, with the same event ordering between its users.
 * Unlike gemm_f16_nt it never takes pooled scratch, whatever
 * gemm_set_scratch_pool says, so it never asks the driver or any allocator
 * for memory: this suits code running under a fixed device-memory budget,
 * code that has reserved all device memory up front, and code that must not
 * enter an allocator (which may synchronize or fail at a point the caller
 * cannot handle).  The array exists from the moment the library is loaded
 * until the process exits, on every GPU that loads it.
 *   - Scratch needed: round256(M*Kp*2) + round256(N*Kp*2) bytes, Kp = K
 *     rounded up to a multiple of 8.  Operands that would need more than the
 *     32 MiB (33554432 bytes) are read in place by the realigning producer
 *     instead (slower for large operands, same result bits).
 *     Operands the accelerator can address directly need no scratch at all.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *     The address is kept for the life of the process: after a
 *     cudaDeviceReset (or any other replacement of the device's primary
 *     context) this entry point must not be called again in that process.
 *   - All calls share the one array (with gemm_f16_nt).  Outside stream
 *     capture each use is ordered after the previous one, on the GPU, by an
 *     event.  A call made while `stream` is being captured into a CUDA graph
 *     cannot be ordered that way and uses the array unordered: calls that can
 *     overlap on the GPU then race on it, and the caller must order them.
 *     The array keeps the last call's contents; each call overwrites every
 *     byte it reads, so nothing needs clearing.
 */
int gemm_f16_nt_noalloc(int64_t M, int64_t N, int64_t K, const gemm_f16_t* lhs, const gemm_f16_t* rhs,
                        gemm_f16_t* out, int stages, cudaStream_t stream);

/*
 * gemm_device_status -- synchronizes `stream`, then returns and clears the
 * status word of that stream on the current device: GEMM_OK, or
 * GEMM_ERR_TIMEOUT if a bounded wait inside a kernel of this library launched
 * on `stream` expired since the last call for it.  Returns GEMM_ERR_LAUNCH if
 * the synchronization itself failed.
 *
 * Every device-side wait of the pipelines (mbarrier phase waits) gives up
 * after the wait limit; the waiting role then records the timeout, drains
 * what it has in flight and the kernel returns, so the CUDA context stays
 * usable.  This is the device analogue of the deadlock the Croqtile tutorial
 * ch.6 describes for a missing empty seed ("消费者路径").
 *
 * Each stream has its own word: a timeout in a call on one stream is neither
 * seen nor cleared by gemm_device_status on another.  The library keeps words
 * for the first 63 streams it sees on each device (keyed by the stream
 * handle, for the life of the process); later streams share one more word.
 * A handle reused by a new stream inherits the old stream's word.
 */
int gemm_device_status(cudaStream_t stream);

/* gemm_status_string -- a static, human-readable name for a status code. */
const char* gemm_status_string(int status);

/*
 * gemm_set_wait_timeout_ns -- sets the limit of every bounded device wait
 * for later launches (default 2e9 ns = 2 s; 0 restores the default).  Host
 * state only; returns GEMM_OK.
 */
int gemm_set_wait_timeout_ns(uint64_t ns);

/*
 * Debug flags for later launches (host state only; 0 = normal operation).
 *   GEMM_DEBUG_SKIP_EMPTY_SEED     : the consumer does not seed the empty
 *       events (Croqtile ch.6, "消费者路径": the producer's first wait then
 *       never completes); used to test that the bounded waits turn this
 *       deadlock into GEMM_ERR_TIMEOUT.
 *   GEMM_DEBUG_FORCE_COPY_PRODUCER : use the asynchronous-copy producer even
 *       where the tensor memory accelerator could be used.
 *   GEMM_DEBUG_FORCE_DIRECT_STORE  : store the output with guarded plain
 *       stores instead of the tensor memory accelerator.
 *   GEMM_DEBUG_FORCE_SOLO_TILE     : use the one-CTA 128x128 tile even where
 *       the CTA-pair 256x256 tile would be chosen.
 *   GEMM_DEBUG_FORCE_PAIR_TILE     : use the CTA-pair 256x256 tile whenever the
 *       TMA producer is used, even for small outputs.
 *   GEMM_DEBUG_NO_SPLIT            : do not split the last wave's tiles into
 *       half-width units (gemm_f16_nt normally does, see above).
 *   GEMM_DEBUG_FORCE_NARROW_TILE   : where the CTA pair is used, always use
 *       its 256x256 tile, never the wide 256x512 one.
 *   GEMM_DEBUG_FORCE_WIDE_TILE     : where the CTA pair is used and stages is
 *       at most 4, always use the wide 256x512 tile.
 *   GEMM_DEBUG_SKIP_ACC_SEED       : the epilogue does not seed the
 *       accumulator's empty events, so the multiply role's first wait for
 *       the accumulator never completes while the producer has already
 *       filled the ring; used to test that this deadlock, with copies
 *       issued, also ends in GEMM_ERR_TIMEOUT and a clean exit.
 *   GEMM_DEBUG_NO_KSPLIT           : never split K over a cluster of two
 *       CTAs (gemm_f16_nt does for small outputs, see above); the result is
 *       then the one-pass sum every other tile gives.
 *   GEMM_DEBUG_FORCE_KSPLIT        : split K wherever the single-CTA tile is
 *       used and there are at least 2 K blocks, however many tiles there are
 *       (clusters beyond those that fit at once run as the GPU frees SMs).
 *   GEMM_DEBUG_SKIP_KSPLIT_SEND    : in the K split, the warps that send
 *       their partial sums to the peer CTA send nothing and never signal it;
 *       used to test that the owners' wait for them ends in GEMM_ERR_TIMEOUT
 *       while the rest of the cluster finishes normally.
 *   GEMM_DEBUG_FORCE_DOUBLE_SLOT   : where the single-CTA tile is fed by TMA
 *       without the K split and stages <= 3, use ring slots of several
 *       64-wide K boxes (three for stages <= 2, two for 3) even when the
 *       tiles exceed one wave.
 *   GEMM_DEBUG_NO_DOUBLE_SLOT      : never use multi-box slots.
 *   GEMM_DEBUG_IN_PLACE            : read operands that the tensor memory
 *       accelerator cannot address in place (the realigning producer)
 *       rather than repacking them.
 * Returns GEMM_OK, or GEMM_ERR_INVALID_ARG for unknown bits.
 */
enum {
    GEMM_DEBUG_SKIP_EMPTY_SEED = 1u,
    GEMM_DEBUG_FORCE_COPY_PRODUCER = 2u,
    GEMM_DEBUG_FORCE_DIRECT_STORE = 4u,
    GEMM_DEBUG_FORCE_SOLO_TILE = 8u,
    GEMM_DEBUG_FORCE_PAIR_TILE = 16u,
    GEMM_DEBUG_NO_SPLIT = 32u,
    GEMM_DEBUG_FORCE_NARROW_TILE = 64u,
    GEMM_DEBUG_FORCE_WIDE_TILE = 128u,
    GEMM_DEBUG_SKIP_ACC_SEED = 256u,
    GEMM_DEBUG_NO_KSPLIT = 512u,
    GEMM_DEBUG_FORCE_KSPLIT = 1024u,
    GEMM_DEBUG_SKIP_KSPLIT_SEND = 2048u,
    GEMM_DEBUG_FORCE_DOUBLE_SLOT = 4096u,
    GEMM_DEBUG_NO_DOUBLE_SLOT = 8192u,
    GEMM_DEBUG_IN_PLACE = 16384u
};
int gemm_set_debug_flags(unsigned flags);

/*
 * gemm_set_scratch_pool -- whether later gemm_f16_nt calls may allocate
 * scratch memory (host state only; default 0 = never).
 *
 * On, operands that the tensor memory accelerator cannot address are copied
 * into rows of ceil(K/64)*64 elements in scratch memory taken stream-ordered
 * from a memory pool the library owns on the current device (about
 * (M+N)*ceil(K/64)*128 bytes per call, returned to the pool on `stream` after
 * the GEMM; the pool keeps freed memory, so repeated calls of one size request
 * no new memory from the driver), instead of into the library's fixed array.
 * Each call then has its own copy, so such calls on different streams can
 * overlap, and operands too large for the array are repacked rather than read
 * in place.  If the pool cannot supply the scratch, the call reads the
 * operands in place.  Results are bitwise identical either way.
 * gemm_f16_nt_noalloc ignores this setting.  Returns GEMM_OK.
 */
int gemm_set_scratch_pool(int enable);

/*
 * gemm_f16_nt_plan -- the launch plan gemm_f16_nt would use for these
 * arguments, without touching a device (host logic only).  Validates the
 * arguments exactly as gemm_f16_nt does and returns the same status.
 *   plan[0] tile rows per CTA group (BM)      plan[1] tile columns (BN)
 *   plan[2] K per ring slot (64; 256, 192 or 128 for multi-box slots)
 *   plan[3] CTAs per tile (1 or 2)
 *   plan[4] producer: 0 = tensor memory accelerator, 1 = async copy,
 *           2 = tensor memory accelerator on an aligned copy (in the fixed
 *           array, or in pooled scratch with gemm_set_scratch_pool; a call on
 *           a stream being captured reads in place instead), 3 = realigning
 *           loads in place
 *   plan[5] copy granularity in bytes (16 for TMA, else 8, 4 or 2)
 *   plan[6] output store: 0 = tensor memory accelerator, 1 = plain stores
 *   plan[7] dynamic shared memory bytes per CTA
 *   plan[8] number of output tiles
 *   plan[9] number of K blocks (of plan[2] columns each)
 *   plan[10] CTAs summing parts of K per tile: 1, or 2 (the K split)
 * `plan` must hold 11 int64 values.
 */
int gemm_f16_nt_plan(int64_t M, int64_t N, int64_t K, const gemm_f16_t* lhs, const gemm_f16_t* rhs,
                     const gemm_f16_t* out, int stages, int64_t* plan);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* PWSGEMM_H_ */
