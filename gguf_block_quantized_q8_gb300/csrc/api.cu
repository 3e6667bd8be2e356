// C-ABI entry points: argument validation, dispatch to the kernels, error strings,
// and the device status word that the kernels' bounded waits report into.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "ggq_internal.h"
#include "ptx.cuh"

namespace ggq {

namespace {
thread_local char g_msg[512] = "";

// One int per device that loads the library: bit kStatusTimeout is set by a
// kernel whose bounded wait ran out.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// weights per block of the types the GEMV, decode and row-gather calls take; 0: none
int64_t block_of(int type) {
    switch (type) {
    case GGQ_F32: return 1;
    case GGQ_Q4_0:
    case GGQ_Q8_0: return 32;
    case GGQ_Q4_K:
    case GGQ_Q6_K: return 256;
    default: return 0;
    }
}
}  // namespace

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(e == cudaErrorMemoryAllocation ? GGQ_ENOMEM : GGQ_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

void clear_error() { g_msg[0] = '\0'; }

int* device_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

int read_and_clear_status(int* status) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "read status word");
    if (v) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "clear status word");
    }
    *status = v;
    return GGQ_OK;
}

}  // namespace ggq

using namespace ggq;

extern "C" int ggq_gemv(int type, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int M,
                        void* stream) {
    clear_error();
    const int64_t blk = block_of(type);
    if (blk == 0) return fail(GGQ_ETYPE, "ggq_gemv: type %d not supported", type);
    if (!W || !x || !y) return fail(GGQ_EINVAL, "ggq_gemv: NULL pointer");
    if (rows < 1 || rows > 0x7fffffff) return fail(GGQ_EINVAL, "ggq_gemv: rows %lld out of range", (long long)rows);
    if (cols > (int64_t)1 << 40) return fail(GGQ_EINVAL, "ggq_gemv: cols %lld out of range", (long long)cols);
    if (cols < blk || cols % blk) return fail(GGQ_EINVAL, "ggq_gemv: cols %lld not a positive multiple of %lld",
                                              (long long)cols, (long long)blk);
    if (M < 1 || M > 16) return fail(GGQ_EINVAL, "ggq_gemv: M %d outside 1..16", M);
    if (!aligned(W, 16)) return fail(GGQ_EINVAL, "ggq_gemv: W not 16-byte aligned");
    if (!aligned(x, 16)) return fail(GGQ_EINVAL, "ggq_gemv: x not 16-byte aligned");
    if (!aligned(y, 4)) return fail(GGQ_EINVAL, "ggq_gemv: y not 4-byte aligned");
    return launch_gemv(type, W, rows, cols, x, y, M, static_cast<cudaStream_t>(stream));
}

extern "C" int ggq_gemv_multi(int type, int n, const void* const* W, const int64_t* rows, int64_t cols,
                              const float* x, float* const* y, int M, void* stream) {
    clear_error();
    const int64_t blk = block_of(type);
    if (blk == 0) return fail(GGQ_ETYPE, "ggq_gemv_multi: type %d not supported", type);
    if (n < 1 || n > 4) return fail(GGQ_EINVAL, "ggq_gemv_multi: n %d outside 1..4", n);
    if (!W || !rows || !y || !x) return fail(GGQ_EINVAL, "ggq_gemv_multi: NULL pointer");
    if (cols > (int64_t)1 << 40) return fail(GGQ_EINVAL, "ggq_gemv_multi: cols %lld out of range", (long long)cols);
    if (cols < blk || cols % blk) return fail(GGQ_EINVAL, "ggq_gemv_multi: cols %lld not a positive multiple of %lld",
                                              (long long)cols, (long long)blk);
    if (M < 1 || M > 16) return fail(GGQ_EINVAL, "ggq_gemv_multi: M %d outside 1..16", M);
    if (!aligned(x, 16)) return fail(GGQ_EINVAL, "ggq_gemv_multi: x not 16-byte aligned");
    for (int i = 0; i < n; ++i) {
        if (!W[i] || !y[i]) return fail(GGQ_EINVAL, "ggq_gemv_multi: NULL pointer");
        if (rows[i] < 1 || rows[i] > 0x7fffffff) return fail(GGQ_EINVAL, "ggq_gemv_multi: rows out of range");
        if (!aligned(W[i], 16)) return fail(GGQ_EINVAL, "ggq_gemv_multi: W not 16-byte aligned");
        if (!aligned(y[i], 4)) return fail(GGQ_EINVAL, "ggq_gemv_multi: y not 4-byte aligned");
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (stream_gemv_supported(type, cols, M, n, rows)) return launch_gemv_stream(type, n, W, rows, cols, x, y, M, s);
    for (int i = 0; i < n; ++i) {
        int rc = launch_gemv(type, W[i], rows[i], cols, x, y[i], M, s);
        if (rc) return rc;
    }
    return GGQ_OK;
}

extern "C" int ggq_gemm_prefill(int type, const void* W, int64_t rows, int64_t cols, const uint16_t* X, float* Y,
                                int M, void* stream) {
    clear_error();
    if (type != GGQ_Q4_K && type != GGQ_Q8_0)
        return fail(GGQ_ETYPE, "ggq_gemm_prefill: type %d not supported", type);
    if (!W || !X || !Y) return fail(GGQ_EINVAL, "ggq_gemm_prefill: NULL pointer");
    if (rows < 128 || rows % 128 || rows > 0x7fffffff)
        return fail(GGQ_EINVAL, "ggq_gemm_prefill: rows %lld not a positive multiple of 128", (long long)rows);
    if (cols < 256 || cols % 256 || cols > (1 << 24))
        return fail(GGQ_EINVAL, "ggq_gemm_prefill: cols %lld not a positive multiple of 256", (long long)cols);
    if (M < 128 || M % 128 || M > 65536)
        return fail(GGQ_EINVAL, "ggq_gemm_prefill: M %d not a multiple of 128 in 128..65536", M);
    if (!aligned(W, 16) || !aligned(X, 16) || !aligned(Y, 16))
        return fail(GGQ_EINVAL, "ggq_gemm_prefill: W, X and Y must be 16-byte aligned");
    return launch_prefill(type, W, rows, cols, X, Y, M, static_cast<cudaStream_t>(stream));
}

extern "C" int ggq_dequantize(int type, const void* W, int64_t rows, int64_t cols, float* out, void* stream) {
    clear_error();
    const int64_t blk = block_of(type);
    if (blk == 0) return fail(GGQ_ETYPE, "ggq_dequantize: type %d not supported", type);
    if (!W || !out) return fail(GGQ_EINVAL, "ggq_dequantize: NULL pointer");
    if (rows < 0 || cols < 0 || cols % blk) return fail(GGQ_EINVAL, "ggq_dequantize: bad shape");
    if (!aligned(W, 16) || !aligned(out, 4)) return fail(GGQ_EINVAL, "ggq_dequantize: misaligned pointer");
    return launch_dequantize(type, W, rows, cols, out, static_cast<cudaStream_t>(stream));
}

extern "C" int ggq_embed(int type, const void* table, int64_t rows, int64_t cols, const int32_t* ids, int n,
                         float* out, void* stream) {
    clear_error();
    const int64_t blk = block_of(type);
    if (blk == 0) return fail(GGQ_ETYPE, "ggq_embed: type %d not supported", type);
    if (!table || !ids || !out) return fail(GGQ_EINVAL, "ggq_embed: NULL pointer");
    if (rows < 1 || rows > 0x7fffffff || cols < 1 || cols % blk) return fail(GGQ_EINVAL, "ggq_embed: bad shape");
    if (n < 1 || n > 65535) return fail(GGQ_EINVAL, "ggq_embed: n %d outside 1..65535", n);
    if (!aligned(table, type == GGQ_F32 ? 4 : 2) || !aligned(ids, 4) || !aligned(out, 4))
        return fail(GGQ_EINVAL, "ggq_embed: misaligned pointer");
    return launch_embed(type, table, rows, cols, ids, n, out, static_cast<cudaStream_t>(stream));
}

extern "C" int ggq_device_status(void) {
    clear_error();
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    int v = 0;
    int rc = read_and_clear_status(&v);
    if (rc) return rc;
    if (v & kStatusTimeout) {
        reset_prefill_sync();   // nothing runs now: the next prefill starts from clean sync words
        return fail(GGQ_ETIMEOUT, "a kernel's bounded wait ran out");
    }
    if (v & kStatusBadIndex) return fail(GGQ_EINVAL, "an embedding row id was outside the table");
    return GGQ_OK;
}

extern "C" const char* ggq_strerror(int code) {
    switch (code) {
    case GGQ_OK: return "success";
    case GGQ_EINVAL: return "invalid argument";
    case GGQ_ETYPE: return "unsupported tensor type";
    case GGQ_EIO: return "I/O error";
    case GGQ_EFORMAT: return "malformed GGUF file";
    case GGQ_ENOMEM: return "out of memory";
    case GGQ_ECUDA: return "CUDA error";
    case GGQ_ETIMEOUT: return "bounded wait timed out";
    case GGQ_ENOTFOUND: return "not found";
    default: return "unknown error";
    }
}

extern "C" const char* ggq_last_error(void) { return g_msg; }

extern "C" int ggq_abi_version(void) { return 1; }
