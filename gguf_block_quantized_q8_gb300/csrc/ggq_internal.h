// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cstdarg>
#include <cstdint>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "ggq.h"

struct ggq_model {
    uint32_t version = 0;
    uint64_t data_start = 0;
    struct Tensor {
        std::string name;
        int32_t type = 0;
        int32_t n_dims = 0;
        int64_t ne[4] = {1, 1, 1, 1};
        uint64_t offset = 0;
        uint64_t nbytes = 0;
        uint64_t arena_off = 0;   // offset inside the device arena
    };
    struct KV {
        std::string key;
        int32_t vtype = 0;
        std::vector<uint8_t> value;  // raw little-endian encoding of the value
    };
    std::vector<Tensor> tensors;
    std::vector<KV> kvs;
    void* arena = nullptr;           // one cudaMalloc for all payloads
    uint64_t arena_bytes = 0;
    int device = -1;
};

namespace ggq {

// thread-local error message; returns `code` for convenient `return fail(...)`
int fail(int code, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);
void clear_error();

// payload bytes for `n` elements of `type` (0 and GGQ_ETYPE if unknown)
int payload_bytes(int32_t type, uint64_t ne0, uint64_t n, uint64_t* out);

// kernel entry points (launchers live next to their kernels)
int launch_gemv(int type, const void* W, int64_t rows, int64_t cols, const float* x,
                float* y, int M, cudaStream_t stream);
// persistent row-partitioned GEMV over one or more matrices sharing x (M <= 4);
// needs no workspace
bool stream_gemv_supported(int type, int64_t cols, int M, int nseg, const int64_t* rows);
int launch_gemv_stream(int type, int nseg, const void* const* W, const int64_t* rows, int64_t cols,
                       const float* x, float* const* y, int M, cudaStream_t stream);
// warp-per-row GEMV for F32 (any cols), Q4_0 (cols % 32 == 0) and Q6_K
// (cols % 256 == 0), M up to 16
int launch_gemv_rows(int type, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int M,
                     cudaStream_t stream);
// small-batch dequant-GEMM on the tensor cores (Q8_0, Q4_K, Q4_0; M up to 16,
// cols % 256 == 0); ggq_gemv uses it from kSmallMMin activation rows on.  When
// it splits tiles along K it zeroes y first (a memset on the stream).
constexpr int kSmallMMin = 5;
bool smallm_supported(int type, int64_t rows, int64_t cols, int M);
int launch_smallm(int type, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int M,
                  cudaStream_t stream);
int launch_dequantize(int type, const void* W, int64_t rows, int64_t cols, float* out,
                      cudaStream_t stream);
int launch_prefill(int type, const void* W, int64_t rows, int64_t cols, const uint16_t* X,
                   float* Y, int M, cudaStream_t stream);

// device-side status word (bounded-wait timeouts); see ggq_device_status
int* device_status_word();       // device pointer for the current device (lazily zeroed)
int read_and_clear_status(int* status);
int reset_prefill_sync();   // after a timeout: zero the prefill split-tile sync words
int launch_embed(int type, const void* W, int64_t rows, int64_t cols, const int32_t* ids, int n, float* out,
                 cudaStream_t stream);

}  // namespace ggq
