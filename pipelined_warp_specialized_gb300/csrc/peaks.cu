// peaks.cu -- measurement kernels used by bench.py, built into their own
// library (_build/libpwspeaks.so); not part of the GEMM's C ABI.
//
//   pws_peaks_imad   -- the CUDA-core rate of 32-bit integer multiply-adds,
//                       the instruction the s32 kernels' inner product runs
//                       (mad.lo.u32), for the s32 path's roofline.
//   pws_peaks_empty  -- an empty kernel launched the way the GEMM kernels
//                       are (programmatic dependent launch), so a CUDA-graph
//                       replay of it gives the launch floor a small GEMM
//                       cannot go below.
//   pws_peaks_mma    -- the dense f16 -> fp32 tensor rate per SM per clock:
//                       one CTA per SM issues tcgen05.mma back to back from
//                       one shared-memory tile pair, timed in SM cycles.
#include <cstdint>

#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace pws {
namespace peaks {

// CHAINS independent multiply-add chains per thread, interleaved, so that
// each warp scheduler always has an independent mad.lo.u32 to issue.  The
// volatile asm keeps the compiler from folding the recurrences.
template <int CHAINS>
__global__ void __launch_bounds__(256) imad_kernel(uint32_t* sink, int iters, uint32_t m) {
    uint32_t a[CHAINS];
#pragma unroll
    for (int c = 0; c < CHAINS; ++c) a[c] = threadIdx.x + 977u * c;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < CHAINS; ++c)
            asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(a[c]) : "r"(m), "r"(static_cast<uint32_t>(c)));
    }
    uint32_t x = 0;
#pragma unroll
    for (int c = 0; c < CHAINS; ++c) x ^= a[c];
    if (x == 0x9E3779B9u) sink[0] = x;      // keeps every chain's result live
}

__global__ void empty_kernel() {
    grid_dependency_wait();
    allow_dependent_launch();
}

// tcgen05.mma kind::f16, M = 128, N = 256, K = 16: the instruction
// descriptor (fp32 D, f16 A and B, both K-major; N >> 3 at bit 17, M >> 4 at
// bit 24) and the shared-memory descriptor of a K-major operand in the
// 128-byte swizzle (start >> 4, 1024-byte stride between 8-row atoms,
// descriptor version 1, swizzle mode 2) -- the hardware formats the GEMM
// kernel uses too.
constexpr int kMmaM = 128, kMmaN = 256, kMmaK = 16, kMmaPerStep = 4;
constexpr uint32_t kMmaIdesc = (1u << 4) | (static_cast<uint32_t>(kMmaN >> 3) << 17) |
                               (static_cast<uint32_t>(kMmaM >> 4) << 24);
constexpr int kMmaSmem = 120 * 1024;     // one CTA per SM

__device__ __forceinline__ uint64_t mma_sdesc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Each CTA fills a 128 x 64 A tile and a 256 x 64 B tile with f16 values of
// random sign and mantissa in [0.125, 0.5), then one thread issues `steps`
// K steps of four MMAs into a 256-column fp32 accumulator and waits for
// them (bounded: `timeout_ns`).  out[2 b] = SM cycles, out[2 b + 1] =
// nanoseconds from the first issue to the completion of the last MMA of
// CTA b; a wait that gave up sets bit 0 of *status.
__global__ void __launch_bounds__(128, 1)
mma_kernel(int steps, unsigned long long timeout_ns, unsigned long long* out, unsigned* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const g = smem_raw + (base - raw);
    const uint32_t sA = base, sB = base + kMmaM * 128, bar = sB + kMmaN * 128, slot = bar + 8;
    uint16_t* const tiles = reinterpret_cast<uint16_t*>(g);
    for (int i = threadIdx.x; i < (kMmaM + kMmaN) * 64; i += blockDim.x) {
        uint32_t h = static_cast<uint32_t>(i) * 0x9E3779B1u ^ (blockIdx.x * 0x85EBCA77u);
        h ^= h >> 15;
        h *= 0x2C1B3C6Du;
        h ^= h >> 12;
        tiles[i] = static_cast<uint16_t>(0x3000u | (h & 0x07FFu) | ((h >> 16) & 0x8000u));
    }
    fence_proxy_async_smem();           // the tensor core reads what the threads wrote
    if (threadIdx.x < 32) {
        tmem_alloc<1>(slot, kMmaN);
        tmem_relinquish<1>();
    }
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(g + (slot - base));
    if (threadIdx.x == 0) {
        const uint64_t adesc = mma_sdesc(sA), bdesc = mma_sdesc(sB);
        const uint64_t c0 = clock64(), t0 = globaltimer_ns();
        for (int s = 0; s < steps; ++s) {
#pragma unroll
            for (int k = 0; k < kMmaPerStep; ++k)
                tc_mma_f16<1>(tmem, adesc + 2 * k, bdesc + 2 * k, kMmaIdesc, (s | k) != 0);
        }
        tc_commit_1(bar);
        bool done = false;
        while (!done) {
            done = mbar_try_wait(bar, 0);
            if (!done && globaltimer_ns() - t0 > timeout_ns) {
                atomicOr(status, 1u);
                break;
            }
        }
        out[2 * blockIdx.x] = clock64() - c0;
        out[2 * blockIdx.x + 1] = globaltimer_ns() - t0;
        if (!done) {
            // the multiplies are still in flight: wait for them (bounded
            // again) before the accumulator is released
            const uint64_t t1 = globaltimer_ns();
            while (!mbar_try_wait(bar, 0) && globaltimer_ns() - t1 < timeout_ns) {
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (threadIdx.x < 32) tmem_dealloc<1>(tmem, kMmaN);
}

}  // namespace peaks
}  // namespace pws

// The library is built with hidden visibility; these are its exports.
#pragma GCC visibility push(default)
extern "C" {

// Multiply-adds per thread: iters * pws_peaks_imad_chains().
int pws_peaks_imad_chains() { return 16; }

int pws_peaks_imad(int blocks, int threads, int iters, uint32_t* sink, cudaStream_t stream) {
    if (blocks <= 0 || threads <= 0 || threads > 256 || iters <= 0 || !sink) return 1;
    pws::peaks::imad_kernel<16><<<blocks, threads, 0, stream>>>(sink, iters, 0x01000193u);
    return cudaGetLastError() == cudaSuccess ? 0 : 5;
}

int pws_peaks_empty(int blocks, int threads, cudaStream_t stream) {
    if (blocks <= 0 || threads <= 0 || threads > 1024) return 1;
    return pws::launch_pdl(pws::peaks::empty_kernel, dim3(blocks), dim3(threads), 0, stream) == cudaSuccess ? 0 : 5;
}

// Flops of one CTA's K step in pws_peaks_mma: 2 * M * N * K * 4.
long long pws_peaks_mma_step_flops() {
    return 2ll * pws::peaks::kMmaM * pws::peaks::kMmaN * pws::peaks::kMmaK * pws::peaks::kMmaPerStep;
}

// `blocks` CTAs (at most one per SM) of `steps` K steps each; out holds 2 *
// blocks values (device memory), status one word (device memory, bit 0 set
// if a wait gave up).  Needs a device of compute capability 10.x.
int pws_peaks_mma(int blocks, int steps, unsigned long long timeout_ns, unsigned long long* out, unsigned* status,
                  cudaStream_t stream) {
    if (blocks <= 0 || steps <= 0 || !out || !status) return 1;
    // the shared-memory limit is a per-device setting of the kernel
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= 64) return 5;
    static bool configured[64] = {};
    if (!configured[device]) {
        if (cudaFuncSetAttribute(pws::peaks::mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 pws::peaks::kMmaSmem) != cudaSuccess)
            return 5;
        configured[device] = true;
    }
    pws::peaks::mma_kernel<<<blocks, 128, pws::peaks::kMmaSmem, stream>>>(steps, timeout_ns, out, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 5;
}

}  // extern "C"
#pragma GCC visibility pop
