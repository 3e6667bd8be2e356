// Block decode to fp32 in global memory (inspection / bit-exactness checks; the
// GEMV path never writes decoded weights).
//
// Q8_0 ("GGUF: The File Format...", "How a Q8_0 block is stored"): w = d * q.
// Q4_K (same section, k-quant paragraph; byte layout fp16 d, fp16 dmin, 12 bytes of
// packed 6-bit scales and mins, 128 bytes of nibbles): w = d*sc_j*q - dmin*m_j.
// Q4_0 (same section: the Q8_0 layout with 4-bit integers; byte layout fp16 d,
// then byte l holding the codes of weights l (low nibble) and 16 + l (high)):
// w = d * (code - 8).  Q6_K (same section; layout of real files: ql[128] low
// 4 bits, qh[64] high 2 bits, 16 signed 8-bit sub-block scales, fp16 d):
// w = d * sc[k/16] * (u - 32).  F32 rows are copied as they are.
// All are exact in fp32 except the single rounding of the Q4_K subtraction.
#include <cuda_runtime.h>

#include "ggq_internal.h"
#include "ptx.cuh"

namespace ggq {

namespace {

// one thread per Q8_0 block
__global__ void dequant_q8_kernel(const uint8_t* __restrict__ W, int64_t nblocks, float* __restrict__ out) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const uint8_t* blk = W + 34 * b;
    const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
    float* o = out + 32 * b;
#pragma unroll 8
    for (int i = 0; i < 32; ++i) o[i] = d * (float)(int8_t)blk[2 + i];
}

// one thread per Q4_0 block; the 18-byte block starts on an even address
__global__ void dequant_q40_kernel(const uint8_t* __restrict__ W, int64_t nblocks, float* __restrict__ out) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const uint8_t* blk = W + 18 * b;
    const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
    float* o = out + 32 * b;
#pragma unroll 4
    for (int l = 0; l < 16; ++l) {
        const int q = blk[2 + l];
        o[l] = d * (float)((q & 15) - 8);
        o[16 + l] = d * (float)((q >> 4) - 8);
    }
}

// the 6-bit code of weight k of a Q6_K super-block
__device__ __forceinline__ int q6k_code(const uint8_t* blk, int k) {
    const int h = k >> 7, g = (k >> 5) & 3, l = k & 31;
    const int lo = (blk[64 * h + 32 * (g & 1) + l] >> (4 * (g >> 1))) & 15;
    const int hi = (blk[128 + 32 * h + l] >> (2 * g)) & 3;
    return lo | (hi << 4);
}

// one thread per Q6_K sub-block (16 weights sharing a scale)
__global__ void dequant_q6k_kernel(const uint8_t* __restrict__ W, int64_t nsub, float* __restrict__ out) {
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= nsub) return;
    const int64_t sb = g >> 4;
    const int j = (int)(g & 15);
    const uint8_t* blk = W + 210 * sb;
    const float d = half_bits_to_float((uint32_t)blk[208] | ((uint32_t)blk[209] << 8));
    const float a = d * (float)(int8_t)blk[192 + j];
    float* o = out + 256 * sb + 16 * j;
#pragma unroll 4
    for (int l = 0; l < 16; ++l) o[l] = a * (float)(q6k_code(blk, 16 * j + l) - 32);
}

// one thread per Q4_K sub-block (32 weights)
__global__ void dequant_q4k_kernel(const uint8_t* __restrict__ W, int64_t nsub, float* __restrict__ out) {
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= nsub) return;
    const int64_t sb = g >> 3;
    const int j = (int)(g & 7);
    const uint8_t* blk = W + 144 * sb;
    const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
    const float dmin = half_bits_to_float((uint32_t)blk[2] | ((uint32_t)blk[3] << 8));
    const uint8_t* sc = blk + 4;
    int s, m;
    if (j < 4) {
        s = sc[j] & 63;
        m = sc[j + 4] & 63;
    } else {
        s = (sc[j + 4] & 15) | ((sc[j - 4] >> 6) << 4);
        m = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4);
    }
    const float a = d * (float)s, bm = dmin * (float)m;
    // sub-block j covers nibbles of qs[32*(j/2) + l]: low for even j, high for odd
    const uint8_t* qs = blk + 16 + 32 * (j >> 1);
    const int shift = (j & 1) ? 4 : 0;
    float* o = out + 256 * sb + 32 * j;
#pragma unroll 8
    for (int l = 0; l < 32; ++l) o[l] = fmaf(a, (float)((qs[l] >> shift) & 15), -bm);
}

// Token embedding rows ("GGUF Inferencer in R" section 4, "Input Embedding":
// the token's row of the embedding table; the C++ engine post's embed(table,
// token)): out[i, k] = w[ids[i], k].  One thread per output weight: the q
// bytes and the writes are coalesced, the block's scale bytes come from cache.
// An id outside [0, rows) gives a row of zeros and sets kStatusBadIndex.
template <int TYPE>
__global__ void embed_kernel(const uint8_t* __restrict__ W, int64_t rows, int64_t cols,
                             const int32_t* __restrict__ ids, float* __restrict__ out, int* status) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int i = blockIdx.y;
    if (k >= cols) return;
    const int32_t id = ids[i];
    float* o = out + (int64_t)i * cols + k;
    if (id < 0 || id >= rows) {
        *o = 0.0f;
        if (k == 0) atomicOr(status, kStatusBadIndex);
        return;
    }
    if constexpr (TYPE == GGQ_F32) {
        *o = reinterpret_cast<const float*>(W)[(int64_t)id * cols + k];
    } else if constexpr (TYPE == GGQ_Q8_0) {
        const uint8_t* blk = W + ((int64_t)id * (cols / 32) + k / 32) * 34;
        const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
        *o = d * (float)(int8_t)blk[2 + (k & 31)];
    } else if constexpr (TYPE == GGQ_Q6_K) {
        const uint8_t* blk = W + ((int64_t)id * (cols / 256) + k / 256) * 210;
        const int kk = (int)(k & 255);
        const float d = half_bits_to_float((uint32_t)blk[208] | ((uint32_t)blk[209] << 8));
        *o = d * (float)(int8_t)blk[192 + kk / 16] * (float)(q6k_code(blk, kk) - 32);
    } else if constexpr (TYPE == GGQ_Q4_0) {
        const uint8_t* blk = W + ((int64_t)id * (cols / 32) + k / 32) * 18;
        const int l = (int)(k & 31);
        const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
        const int q = (blk[2 + (l & 15)] >> (l >= 16 ? 4 : 0)) & 15;
        *o = d * (float)(q - 8);
    } else {
        const uint8_t* blk = W + ((int64_t)id * (cols / 256) + k / 256) * 144;
        const int kk = (int)(k & 255), j = kk >> 5, l = kk & 31;
        const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
        const float dmin = half_bits_to_float((uint32_t)blk[2] | ((uint32_t)blk[3] << 8));
        const uint8_t* sc = blk + 4;
        int s, m;
        if (j < 4) {
            s = sc[j] & 63;
            m = sc[j + 4] & 63;
        } else {
            s = (sc[j + 4] & 15) | ((sc[j - 4] >> 6) << 4);
            m = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4);
        }
        const int q = (blk[16 + 32 * (j >> 1) + l] >> ((j & 1) ? 4 : 0)) & 15;
        *o = fmaf(d * (float)s, (float)q, -(dmin * (float)m));
    }
}

}  // namespace

int launch_embed(int type, const void* W, int64_t rows, int64_t cols, const int32_t* ids, int n, float* out,
                 cudaStream_t stream) {
    int* status = device_status_word();
    if (!status) return fail(GGQ_ECUDA, "device status word unavailable");
    const dim3 grid((unsigned)((cols + 255) / 256), (unsigned)n);
    const uint8_t* w = static_cast<const uint8_t*>(W);
    if (type == GGQ_Q8_0)
        embed_kernel<GGQ_Q8_0><<<grid, 256, 0, stream>>>(w, rows, cols, ids, out, status);
    else if (type == GGQ_Q4_0)
        embed_kernel<GGQ_Q4_0><<<grid, 256, 0, stream>>>(w, rows, cols, ids, out, status);
    else if (type == GGQ_Q6_K)
        embed_kernel<GGQ_Q6_K><<<grid, 256, 0, stream>>>(w, rows, cols, ids, out, status);
    else if (type == GGQ_F32)
        embed_kernel<GGQ_F32><<<grid, 256, 0, stream>>>(w, rows, cols, ids, out, status);
    else
        embed_kernel<GGQ_Q4_K><<<grid, 256, 0, stream>>>(w, rows, cols, ids, out, status);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GGQ_OK : cuda_fail(e, "embed launch");
}

int launch_dequantize(int type, const void* W, int64_t rows, int64_t cols, float* out, cudaStream_t stream) {
    const uint8_t* w = static_cast<const uint8_t*>(W);
    if (type == GGQ_F32) {
        if (rows * cols == 0) return GGQ_OK;
        cudaError_t e = cudaMemcpyAsync(out, W, (size_t)(rows * cols) * 4, cudaMemcpyDeviceToDevice, stream);
        return e == cudaSuccess ? GGQ_OK : cuda_fail(e, "dequantize copy");
    }
    if (type == GGQ_Q8_0 || type == GGQ_Q4_0) {
        const int64_t nb = rows * (cols / 32);
        if (nb == 0) return GGQ_OK;
        if (type == GGQ_Q8_0)
            dequant_q8_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, stream>>>(w, nb, out);
        else
            dequant_q40_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, stream>>>(w, nb, out);
    } else if (type == GGQ_Q6_K) {
        const int64_t ns = rows * (cols / 256) * 16;
        if (ns == 0) return GGQ_OK;
        dequant_q6k_kernel<<<(unsigned)((ns + 255) / 256), 256, 0, stream>>>(w, ns, out);
    } else {
        const int64_t ns = rows * (cols / 256) * 8;
        if (ns == 0) return GGQ_OK;
        dequant_q4k_kernel<<<(unsigned)((ns + 255) / 256), 256, 0, stream>>>(w, ns, out);
    }
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GGQ_OK : cuda_fail(e, "dequantize launch");
}

}  // namespace ggq
