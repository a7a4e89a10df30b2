// q1_q8_gemv_noalloc: the decode GEMV for callers that cannot allocate device memory.
//
// q1_q8_gemv needs a small workspace (the activation's per-32-value constants and a tile
// counter) that the caller allocates.  Some callers cannot: code running inside another
// allocator's arena, plugins that are handed raw pointers, or real-time paths where an
// allocation could block or fail at the wrong moment.  This entry point uses a fixed block of
// device memory that is part of the library image instead: every GPU that loads the library holds
// it until the process exits, and no call allocates or frees anything.
//
// Set-up: the first call on each device looks up that array's device address with
// cudaGetSymbolAddress (with the device current) and caches it; make that first call before any
// stream capture on the device.  All calls share the array, so calls whose work overlaps on the
// GPU (different streams, or different host threads) race and must not be issued that way.
#include <mutex>

#include "gq_internal.cuh"

namespace {

constexpr int kNoAllocMaxN = GQ_NOALLOC_MAX_N;
// the activation constants for n = kNoAllocMaxN (96 bytes per 32 values) and the 16-byte counter
constexpr size_t kScratchBytes = static_cast<size_t>(kNoAllocMaxN / 32) * 96 + 16;

static __device__ __align__(256) unsigned char g_gemv_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_gemv_scratch);
        if (e != cudaSuccess) return static_cast<int>(e);
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return 0;
}

}  // namespace

extern "C" int q1_q8_gemv_noalloc(const void* packed_w, const void* act, float* y, int rows, int n,
                                  gq_stream_t stream) {
    if (rows < 1 || n < 128 || n % 128 != 0 || n > kNoAllocMaxN) return GQ_EINVAL_SHAPE;
    if (!packed_w || !act || !y) return GQ_EINVAL_PTR;
    const uintptr_t pw = reinterpret_cast<uintptr_t>(packed_w), pa = reinterpret_cast<uintptr_t>(act),
                    py = reinterpret_cast<uintptr_t>(y);
    if ((pw & 15) || (pa & 1) || (py & 3)) return GQ_EINVAL_PTR;
    void* scratch = nullptr;
    const int se = scratch_for_current_device(&scratch);
    if (se != 0) {
        gq::record_cuda_error(se);
        return GQ_ECUDA;
    }
    // The launch writes the constants for this n and zeroes the counter before the GEMV reads them.
    const cudaError_t e = gq::launch_q1_gemv(packed_w, act, y, rows, n, scratch, GQ_ACT_Q8_0,
                                                 reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        gq::record_cuda_error(static_cast<int>(e));
        return GQ_ECUDA;
    }
    return GQ_OK;
}
