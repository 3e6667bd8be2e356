// ggq_gemv_noalloc: the GEMV for callers that may not allocate device memory.
//
// Some callers cannot allow any device allocation at call time: a server that
// reserves all device memory for its own pool at start-up and treats any later
// allocation as an error, or a latency-critical loop in which cudaMalloc /
// cudaFree (which can synchronise the whole device) must never run.  This
// entry point runs the row-partitioned kernel, which needs no scratch memory
// at all (no row is split between CTAs), and refuses every shape that would
// need another kernel instead of falling back to it.
#include <cstdint>

#include <cuda_runtime.h>

#include "ggq_internal.h"

namespace ggq {
namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace ggq

using namespace ggq;

extern "C" int ggq_gemv_noalloc(int type, const void* W, int64_t rows, int64_t cols, const float* x, float* y,
                                int M, void* stream) {
    clear_error();
    if (type != GGQ_Q8_0 && type != GGQ_Q4_K && type != GGQ_Q4_0 && type != GGQ_Q6_K)
        return fail(GGQ_ETYPE, "ggq_gemv_noalloc: type %d not supported", type);
    if (!W || !x || !y) return fail(GGQ_EINVAL, "ggq_gemv_noalloc: NULL pointer");
    if (rows < 1 || rows > 0x7fffffff) return fail(GGQ_EINVAL, "ggq_gemv_noalloc: rows %lld out of range", (long long)rows);
    if (cols < 256 || cols % 256)
        return fail(GGQ_EINVAL, "ggq_gemv_noalloc: cols %lld not a positive multiple of 256", (long long)cols);
    if (M < 1 || M > 4) return fail(GGQ_EINVAL, "ggq_gemv_noalloc: M %d outside 1..4", M);
    if (!aligned(W, 16)) return fail(GGQ_EINVAL, "ggq_gemv_noalloc: W not 16-byte aligned");
    if (!aligned(x, 16)) return fail(GGQ_EINVAL, "ggq_gemv_noalloc: x not 16-byte aligned");
    if (!aligned(y, 4)) return fail(GGQ_EINVAL, "ggq_gemv_noalloc: y not 4-byte aligned");
    if (!stream_gemv_supported(type, cols, M, 1, &rows))
        return fail(GGQ_EINVAL, "ggq_gemv_noalloc: shape outside the allocation-free kernel's limits "
                                "(x' of one activation row must fit in shared memory)");
    const void* Ws[1] = {W};
    float* ys[1] = {y};
    return launch_gemv_stream(type, 1, Ws, &rows, cols, x, ys, M, static_cast<cudaStream_t>(stream));
}
