// Block decode to fp32 in global memory (inspection / bit-exactness checks; the
// GEMV path never writes decoded weights).
//
// Q8_0 ("GGUF: The File Format...", "How a Q8_0 block is stored"): w = d * q.
// Q4_K (same section, k-quant paragraph; byte layout fp16 d, fp16 dmin, 12 bytes of
// packed 6-bit scales and mins, 128 bytes of nibbles): w = d*sc_j*q - dmin*m_j.
// Both are exact in fp32 except the single rounding of the Q4_K subtraction.
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

}  // namespace

int launch_dequantize(int type, const void* W, int64_t rows, int64_t cols, float* out, cudaStream_t stream) {
    const uint8_t* w = static_cast<const uint8_t*>(W);
    if (type == GGQ_Q8_0) {
        const int64_t nb = rows * (cols / 32);
        if (nb == 0) return GGQ_OK;
        dequant_q8_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, stream>>>(w, nb, out);
    } else {
        const int64_t ns = rows * (cols / 256) * 8;
        if (ns == 0) return GGQ_OK;
        dequant_q4k_kernel<<<(unsigned)((ns + 255) / 256), 256, 0, stream>>>(w, ns, out);
    }
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GGQ_OK : cuda_fail(e, "dequantize launch");
}

}  // namespace ggq
