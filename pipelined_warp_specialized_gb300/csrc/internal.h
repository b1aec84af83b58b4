// internal.h -- host-side helpers shared by the translation units of the
// library (not part of the C ABI).
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime_api.h>

namespace pws {

// Bits of the device status word.
enum : unsigned {
    kStatusTimeout = 1u,          // a bounded wait expired
    kStatusRoleProducer = 1u << 8,
    kStatusRoleMma = 1u << 9,
    kStatusRoleEpilogue = 1u << 10,
};

// Status words per device: slot 0 is shared by streams beyond the first
// kStatusSlots - 1 seen on the device.
constexpr int kStatusSlots = 64;

struct DeviceInfo {
    int device = -1;
    int cc_major = 0, cc_minor = 0;
    int num_sms = 0;
    int max_smem_optin = 0;
    unsigned* status = nullptr;   // device address of this device's kStatusSlots status words
};

// Fills `info` for the current device.  Returns GEMM_OK,
// GEMM_ERR_UNSUPPORTED_ARCH (not compute capability 10.3) or GEMM_ERR_LAUNCH.
int current_device(DeviceInfo* info);

// The status word a launch on `stream` records its timeouts in, and the one
// gemm_device_status(stream) reads and clears.
unsigned* status_word(const DeviceInfo& info, cudaStream_t stream);

uint64_t wait_timeout_ns();
unsigned debug_flags();
// gemm_set_scratch_pool: gemm_f16_nt may copy unaligned operands to pooled scratch
bool scratch_pool_enabled();

// SM count of the current device if one is present, else the GB300 count.
int sm_count_or_default();

// The launch attribute of programmatic dependent launch: the grid may be
// scheduled while the previous grid in the stream finishes (its kernel calls
// grid_dependency_wait() before any global memory access), so the launch
// latency and the set-up overlap the previous grid's tail.
inline cudaLaunchAttribute pdl_attribute() {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

#ifdef __CUDACC__
// Launches `kernel` with the programmatic-dependent-launch attribute.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}
#endif

// Encodes a 2-D tiled tensor map over a row-major matrix of 2-byte elements:
// `inner` elements per row, `outer` rows, `row_bytes` between rows; a box of
// box_inner x box_outer elements with the 128-byte swizzle; out-of-bounds
// elements load as zero.  Returns false if the driver rejects it.
bool encode_tmap_f16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);

// Stream-ordered scratch memory from a library-owned memory pool of the
// current device (kept across calls: its release threshold is unlimited, so
// after the first call of a given size no memory is requested from the
// driver).  Returns nullptr if the pool cannot provide `bytes`.
void* scratch_alloc(const DeviceInfo& info, size_t bytes, cudaStream_t stream);
void scratch_free(void* p, cudaStream_t stream);

// True if [a, a+an) and [b, b+bn) (bytes) intersect.
inline bool ranges_overlap(const void* a, uint64_t an, const void* b, uint64_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    if (an == 0 || bn == 0) return false;
    return a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace pws
