// runtime.cu -- host runtime of the library: the per-device status word,
// device checks, wait limit and debug flags, tensor-map encoding, and the
// status entry points of the C ABI.
#include <atomic>
#include <mutex>

#include "internal.h"
#include "pwsgemm.h"

namespace pws {

namespace {

// Status words: kStatusSlots per device (a __device__ variable exists once in
// every context that loads this module).  A launch gets the word of its
// stream's slot and its kernels OR status bits into it, so that a timeout is
// reported to, and cleared by, the stream whose call had it.
__device__ unsigned g_status_words[kStatusSlots];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
bool g_info_ready[kMaxDevices] = {};

std::atomic<uint64_t> g_timeout_ns{0};
std::atomic<unsigned> g_flags{0};
std::atomic<int> g_scratch_pool{0};
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
bool g_encode_tried = false;

EncodeTiledFn encode_fn() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode_tried) {
        g_encode_tried = true;
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

}  // namespace

int current_device(DeviceInfo* info) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_LAUNCH;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_info_ready[dev]) {
            *info = g_info[dev];
        } else {
            DeviceInfo d;
            d.device = dev;
            if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                    cudaSuccess)
                return GEMM_ERR_LAUNCH;
            if (d.cc_major == 10 && d.cc_minor == 3) {
                void* p = nullptr;
                if (cudaGetSymbolAddress(&p, g_status_words) != cudaSuccess) return GEMM_ERR_LAUNCH;
                d.status = static_cast<unsigned*>(p);
            }
            g_info[dev] = d;
            g_info_ready[dev] = true;
            *info = d;
        }
    }
    if (info->cc_major != 10 || info->cc_minor != 3) return GEMM_ERR_UNSUPPORTED_ARCH;
    return GEMM_OK;
}

namespace {
// Stream -> status slot, per device: open addressing over slots
// 1 .. kStatusSlots-1 keyed by the stream handle (stored + 1, so 0 marks a
// free entry).  Entries are never evicted; once every slot is taken, further
// streams share slot 0.  A handle reused by a later stream inherits its slot.
std::mutex g_slot_mu;
uintptr_t g_slot_key[kMaxDevices][kStatusSlots] = {};
}  // namespace

int status_slot(int device, cudaStream_t stream) {
    if (device < 0 || device >= kMaxDevices) return 0;
    const uintptr_t key = reinterpret_cast<uintptr_t>(stream) + 1u;
    const int n = kStatusSlots - 1;
    int h = static_cast<int>(((key >> 4) * 0x9E3779B97F4A7C15ull) >> 40) % n;
    std::lock_guard<std::mutex> lk(g_slot_mu);
    for (int i = 0; i < n; ++i, h = h + 1 == n ? 0 : h + 1) {
        uintptr_t& e = g_slot_key[device][1 + h];
        if (e == key) return 1 + h;
        if (e == 0) {
            e = key;
            return 1 + h;
        }
    }
    return 0;
}

unsigned* status_word(const DeviceInfo& info, cudaStream_t stream) {
    return info.status ? info.status + status_slot(info.device, stream) : nullptr;
}

uint64_t wait_timeout_ns() {
    const uint64_t t = g_timeout_ns.load(std::memory_order_relaxed);
    return t ? t : kDefaultTimeoutNs;
}

unsigned debug_flags() { return g_flags.load(std::memory_order_relaxed); }

bool scratch_pool_enabled() { return g_scratch_pool.load(std::memory_order_relaxed) != 0; }

int sm_count_or_default() {
    int dev = -1, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
        return n;
    cudaGetLastError();   // clear the "no device" error of a CPU-only host
    return 152;
}

namespace {
cudaMemPool_t g_pool[kMaxDevices] = {};
bool g_pool_tried[kMaxDevices] = {};
}  // namespace

void* scratch_alloc(const DeviceInfo& info, size_t bytes, cudaStream_t stream) {
    cudaMemPool_t pool = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_pool_tried[info.device]) {
            g_pool_tried[info.device] = true;
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = info.device;
            cudaMemPool_t p = nullptr;
            if (cudaMemPoolCreate(&p, &props) == cudaSuccess) {
                uint64_t keep = ~0ull;      // never hand freed blocks back to the driver
                cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
                g_pool[info.device] = p;
            } else {
                cudaGetLastError();
            }
        }
        pool = g_pool[info.device];
    }
    if (!pool) return nullptr;
    void* ptr = nullptr;
    if (cudaMallocFromPoolAsync(&ptr, bytes, pool, stream) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return ptr;
}

void scratch_free(void* p, cudaStream_t stream) {
    if (p) cudaFreeAsync(p, stream);
}

bool encode_tmap_f16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace pws

extern "C" {

int gemm_device_status(cudaStream_t stream) {
    pws::DeviceInfo info;
    const int rc = pws::current_device(&info);
    if (rc != GEMM_OK) return rc;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_LAUNCH;
    unsigned* w = pws::status_word(info, stream);
    unsigned word = 0;
    if (cudaMemcpy(&word, w, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_LAUNCH;
    if (word) {
        const unsigned zero = 0;
        if (cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return GEMM_ERR_LAUNCH;
    }
    return (word & pws::kStatusTimeout) ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

const char* gemm_status_string(int status) {
    switch (status) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
        case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT";
        case GEMM_ERR_UNSUPPORTED_STAGES: return "GEMM_ERR_UNSUPPORTED_STAGES";
        case GEMM_ERR_UNSUPPORTED_ARCH: return "GEMM_ERR_UNSUPPORTED_ARCH";
        case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
        default: return "GEMM_ERR_UNKNOWN";
    }
}

int gemm_set_wait_timeout_ns(uint64_t ns) {
    pws::g_timeout_ns.store(ns, std::memory_order_relaxed);
    return GEMM_OK;
}

int gemm_set_scratch_pool(int enable) {
    pws::g_scratch_pool.store(enable ? 1 : 0, std::memory_order_relaxed);
    return GEMM_OK;
}

int gemm_set_debug_flags(unsigned flags) {
    const unsigned known = GEMM_DEBUG_SKIP_EMPTY_SEED | GEMM_DEBUG_FORCE_COPY_PRODUCER |
                           GEMM_DEBUG_FORCE_DIRECT_STORE | GEMM_DEBUG_FORCE_SOLO_TILE |
                           GEMM_DEBUG_FORCE_PAIR_TILE | GEMM_DEBUG_NO_SPLIT |
                           GEMM_DEBUG_FORCE_NARROW_TILE | GEMM_DEBUG_FORCE_WIDE_TILE |
                           GEMM_DEBUG_SKIP_ACC_SEED | GEMM_DEBUG_NO_KSPLIT | GEMM_DEBUG_FORCE_KSPLIT |
                           GEMM_DEBUG_SKIP_KSPLIT_SEND | GEMM_DEBUG_FORCE_DOUBLE_SLOT |
                           GEMM_DEBUG_NO_DOUBLE_SLOT | GEMM_DEBUG_IN_PLACE;
    if (flags & ~known) return GEMM_ERR_INVALID_ARG;
    pws::g_flags.store(flags, std::memory_order_relaxed);
    return GEMM_OK;
}

}  // extern "C"
