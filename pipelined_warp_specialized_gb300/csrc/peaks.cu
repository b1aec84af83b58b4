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

}  // namespace peaks
}  // namespace pws

// The library is built with hidden visibility; these three are its exports.
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

}  // extern "C"
#pragma GCC visibility pop
