// ggq_gemv_noalloc: the GEMV for callers that may not allocate device memory.
//
// ggq_gemv finishes rows whose columns were split between warp groups through
// a small workspace that the library allocates (cudaMalloc) the first time it
// is used on a stream.  Some callers cannot allow that: a server that reserves
// all device memory for its own pool at start-up and treats any later
// allocation as an error, or a latency-critical loop in which cudaMalloc /
// cudaFree (which can synchronise the whole device) must never run.  This
// entry point gives them the same kernel with its scratch in one fixed array
// of device memory that is part of the library itself.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "ggq_internal.h"

namespace ggq {
namespace {

// Limits of the built-in scratch.
constexpr int kNoAllocMaxGroups = 2048;        // warp groups a launch may use
constexpr int kNoAllocMaxRowBlocks = 32768;    // 32- or 64-row blocks per matrix
constexpr size_t kNoAllocPartialFloats = (size_t)kNoAllocMaxGroups * 2 * 4 * 32;
constexpr size_t kNoAllocBytes = kNoAllocPartialFloats * sizeof(float) + (size_t)(kNoAllocMaxRowBlocks + 32) * sizeof(int);

// Partial sums of split row blocks, then a stage counter padded to 128 bytes
// and one counter per row block.  Every device that loads the library holds these ~2.2 MB until
// the process exits; all calls on a device share them.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch on the current device, looked up once per
// device (cudaGetSymbolAddress; it allocates nothing).
int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(GGQ_EINVAL, "device %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GGQ_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace ggq

using namespace ggq;

extern "C" int ggq_gemv_noalloc(int type, const void* W, int64_t rows, int64_t cols, const float* x, float* y,
                                int M, void* stream) {
    clear_error();
    if (type != GGQ_Q8_0 && type != GGQ_Q4_K) return fail(GGQ_ETYPE, "ggq_gemv_noalloc: type %d not supported", type);
    if (!W || !x || !y) return fail(GGQ_EINVAL, "ggq_gemv_noalloc: NULL pointer");
    if (rows < 1 || rows > 0x7fffffff) return fail(GGQ_EINVAL, "ggq_gemv_noalloc: rows %lld out of range", (long long)rows);
    if (cols < 256 || cols % 256)
        return fail(GGQ_EINVAL, "ggq_gemv_noalloc: cols %lld not a positive multiple of 256", (long long)cols);
    if (M < 1 || M > 4) return fail(GGQ_EINVAL, "ggq_gemv_noalloc: M %d outside 1..4", M);
    if (!aligned(W, 16)) return fail(GGQ_EINVAL, "ggq_gemv_noalloc: W not 16-byte aligned");
    if (!aligned(x, 16)) return fail(GGQ_EINVAL, "ggq_gemv_noalloc: x not 16-byte aligned");
    if (!aligned(y, 4)) return fail(GGQ_EINVAL, "ggq_gemv_noalloc: y not 4-byte aligned");
    if (!stream_gemv_supported(type, cols, M, 1, &rows))
        return fail(GGQ_EINVAL, "ggq_gemv_noalloc: shape outside the built-in kernel's limits");
    void* base = nullptr;
    int rc = scratch_address(&base);
    if (rc) return rc;
    float* partials = static_cast<float*>(base);
    int* counters = reinterpret_cast<int*>(static_cast<unsigned char*>(base) + kNoAllocPartialFloats * sizeof(float));
    return launch_gemv_stream_scratch(type, W, rows, cols, x, y, M, static_cast<cudaStream_t>(stream), partials,
                                      kNoAllocMaxGroups, counters, kNoAllocMaxRowBlocks);
}
