// Warp-per-row GEMV for F32 and Q6_K weights and for the Q4_0 shapes the
// streaming kernel does not take (cols % 256 != 0, cols < 768, x' of an
// activation row too wide for its shared memory); M up to 16.
//
//   y[m][r] = sum_c w[r][c] * x[m][c]      (matvec of the culpeo.ws kernel list)
//
// F32 ("GGUF: The File Format...", the practice script's tensor payload):
// little-endian fp32 weights, row after row.
// Q4_0 (same page, "How a Q8_0 block is stored": the Q8_0 layout with 4-bit
// integers, 18 bytes per 32 weights): fp16 d, then 16 bytes of 4-bit codes;
// weight l (l < 16) is the low nibble of byte l, weight 16 + l its high
// nibble, and w = d * (code - 8) (the layout of real Q4_0 files).
// Q6_K (same page: the k-quant paragraph and the bits/weight loop, 210 bytes
// per 256 weights; "Understanding quantization names like Q4_K_M": Q4_K_M
// files hold some tensors as Q6_K): ql[128] low 4 bits, qh[64] high 2 bits,
// 16 signed 8-bit sub-block scales, fp16 d; weight k = 128h + 32g + l has the
// code u = ql[64h + 32(g%2) + l] >> 4(g/2) & 15 | (qh[32h + l] >> 2g & 3) << 4
// and w = d * sc[k/16] * (u - 32) (the layout of real Q6_K files).
//
// One warp owns a row at a time (grid-stride over rows), lanes split the row's
// columns, a shuffle tree adds the lanes: every output is written by exactly
// one lane and the sum order is fixed.  Weights are streamed with evict-first
// loads (each byte is used once); x is read through the read-only cache.
// The kernels are bound by HBM for F32 rows (four 16-byte loads in flight per
// lane); the Q4_0 kernel here is the correct-for-every-shape path, not the
// fast one (the streaming kernel is, wherever it applies).
#include <cuda_runtime.h>

#include <algorithm>

#include "ggq_internal.h"
#include "ptx.cuh"

namespace ggq {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int MMAX>
__device__ __forceinline__ void store_row(float (&acc)[MMAX], float* y, int64_t rows, int64_t row, int M, int lane) {
#pragma unroll
    for (int m = 0; m < MMAX; ++m) {
        if (m < M) {
            const float v = warp_sum(acc[m]);
            if (lane == 0) y[(int64_t)m * rows + row] = v;
        }
    }
}

// VEC: cols % 4 == 0, so every row and every activation row is 16-byte aligned
// (W and x are) and read as float4.
template <int MMAX, bool VEC>
__global__ void __launch_bounds__(kThreads) gemv_f32_kernel(const float* __restrict__ W, const float* __restrict__ x,
                                                            float* __restrict__ y, int64_t rows, int64_t cols, int M) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t)gridDim.x * kWarps;
    pdl_launch_dependents();
    pdl_wait();   // x may come from the previous kernel in the stream
    for (int64_t row = warp0; row < rows; row += nwarps) {
        float acc[MMAX];
#pragma unroll
        for (int m = 0; m < MMAX; ++m) acc[m] = 0.0f;
        if constexpr (VEC) {
            const int64_t n4 = cols / 4;
            const float4* wr = reinterpret_cast<const float4*>(W + row * cols);
            int64_t q = lane;
            for (; q + 96 < n4; q += 128) {   // four loads of the row in flight
                float4 w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) w[i] = __ldcs(wr + q + 32 * i);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int m = 0; m < MMAX; ++m)
                        if (m < M) {
                            const float4 xv = __ldg(reinterpret_cast<const float4*>(x + m * cols) + q + 32 * i);
                            acc[m] = fmaf(w[i].x, xv.x, fmaf(w[i].y, xv.y, fmaf(w[i].z, xv.z, fmaf(w[i].w, xv.w, acc[m]))));
                        }
            }
            for (; q < n4; q += 32) {
                const float4 w = __ldcs(wr + q);
#pragma unroll
                for (int m = 0; m < MMAX; ++m)
                    if (m < M) {
                        const float4 xv = __ldg(reinterpret_cast<const float4*>(x + m * cols) + q);
                        acc[m] = fmaf(w.x, xv.x, fmaf(w.y, xv.y, fmaf(w.z, xv.z, fmaf(w.w, xv.w, acc[m]))));
                    }
            }
        } else {
            const float* wr = W + row * cols;
            for (int64_t c = lane; c < cols; c += 32) {
                const float w = __ldcs(wr + c);
#pragma unroll
                for (int m = 0; m < MMAX; ++m)
                    if (m < M) acc[m] = fmaf(w, __ldg(x + m * cols + c), acc[m]);
            }
        }
        store_row<MMAX>(acc, y, rows, row, M, lane);
    }
}

// Q4_0: a warp step covers 4 consecutive blocks of the row; lane (s, t) =
// (lane / 8, lane % 8) takes code bytes 2t, 2t+1 of block s of the step, that is
// weights 2t, 2t+1 (low nibbles) and 16+2t, 17+2t (high nibbles).  The 8 lanes
// of a block read its x as contiguous pairs (64 bytes for the low and 64 for the
// high half), and a step's 72 weight bytes are contiguous.  A block starts on
// an even address (W is 16-byte aligned, 18 is even): d and a lane's two code
// bytes are 16-bit loads.  0x4B000000 | u is the float 2^23 + u, so u - 8 is
// formed exactly by one subtraction.
template <int MMAX>
__global__ void __launch_bounds__(kThreads) gemv_q40_rows_kernel(const uint8_t* __restrict__ W,
                                                                 const float* __restrict__ x, float* __restrict__ y,
                                                                 int64_t rows, int64_t cols, int M) {
    const int lane = threadIdx.x & 31, sub = lane >> 3, t = lane & 7;
    const int64_t warp0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t)gridDim.x * kWarps;
    const int64_t nb = cols / 32;
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t row = warp0; row < rows; row += nwarps) {
        float acc[MMAX];
#pragma unroll
        for (int m = 0; m < MMAX; ++m) acc[m] = 0.0f;
        const uint8_t* rp = W + row * nb * 18;
#pragma unroll 4
        for (int64_t b = sub; b < nb; b += 4) {
            const unsigned short* bp = reinterpret_cast<const unsigned short*>(rp + 18 * b);
            const float d = half_bits_to_float(__ldcs(bp));
            const uint32_t q = __ldcs(bp + 1 + t);   // code bytes 2t (bits 0-7) and 2t+1 (bits 8-15)
            const float w0 = __uint_as_float(0x4B000000u | (q & 15u)) - 8388616.0f;           // weight 2t
            const float w1 = __uint_as_float(0x4B000000u | ((q >> 8) & 15u)) - 8388616.0f;    // 2t + 1
            const float w16 = __uint_as_float(0x4B000000u | ((q >> 4) & 15u)) - 8388616.0f;   // 16 + 2t
            const float w17 = __uint_as_float(0x4B000000u | ((q >> 12) & 15u)) - 8388616.0f;  // 17 + 2t
#pragma unroll
            for (int m = 0; m < MMAX; ++m) {
                if (m >= M) continue;
                const float* xb = x + m * cols + 32 * b + 2 * t;
                const float2 xl = __ldg(reinterpret_cast<const float2*>(xb));
                const float2 xh = __ldg(reinterpret_cast<const float2*>(xb + 16));
                acc[m] = fmaf(d, fmaf(w0, xl.x, fmaf(w1, xl.y, fmaf(w16, xh.x, w17 * xh.y))), acc[m]);
            }
        }
        store_row<MMAX>(acc, y, rows, row, M, lane);
    }
}

// Q6_K: a warp step is one 256-weight super-block of the row.  Lane (h, i) =
// (lane / 16, lane % 16) takes columns l = 2i, 2i+1 of half h in all four
// quarters g (weights 128h + 32g + l): the ql bytes 64h + l (g = 0 low nibble,
// g = 2 high) and 64h + 32 + l (g = 1, 3), and the qh bytes 32h + l (2 bits per
// g).  Each of the three is one 16-bit load covering both columns, and the 16
// lanes of a half read 32 contiguous bytes of each.  The 6-bit codes of a
// quarter are assembled two at a time in one register; a byte permute puts a
// code under 0x4B0000 (the float 2^23 + u), so u - 32 is one packed
// subtraction.  Weight k uses sub-block scale k / 16 = 8h + 2g + i / 8: lane j
// converts scale j % 16 (d * sc, no int-to-float instruction) and the lanes
// that need it read it by shuffle.  The super-block starts on an even address
// (W is 16-byte aligned, 210 is even).
//
// Rows with few super-blocks in flight per SM (few rows) are shared: P = 1, 2,
// 4 or 8 warps of a CTA take one row, each a contiguous range of its
// super-blocks, and add their parts in shared memory in warp order.
//
// MINB: CTAs per SM the registers must allow.  With one warp per row (P = 1)
// and M = 1, 6 (48 warps per SM, 40 registers) measured faster; where rows are
// shared (P > 1), 4 (up to 64 registers) did (14336x4096: 27.6 vs 33.3 us; the
// 4096x14336 ffn_down shape, P = 2: 41.4 vs 37.3 us).
template <int MMAX, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) gemv_q6k_rows_kernel(const uint8_t* __restrict__ W,
                                                                 const float* __restrict__ x, float* __restrict__ y,
                                                                 int64_t rows, int64_t cols, int M, int P) {
    __shared__ float red[kWarps][MMAX];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, h = lane >> 4, i = lane & 15;
    const int rpc = kWarps / P, slot = warp / P, part = warp - slot * P;   // rows per CTA step
    const int64_t ns = cols / 256;
    const int64_t u0 = ns * part / P, u1 = ns * (part + 1) / P;
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t base = (int64_t)blockIdx.x * rpc; base < rows; base += (int64_t)gridDim.x * rpc) {
        const int64_t row = base + slot;
        float2 acc[MMAX];
#pragma unroll
        for (int m = 0; m < MMAX; ++m) acc[m] = make_float2(0.0f, 0.0f);
        if (row < rows) {
            const uint8_t* rp = W + row * ns * 210;
            // super-blocks in flight per warp: more where the registers allow
            constexpr int kUnroll = MMAX <= 4 ? 2 : 1;
#pragma unroll kUnroll
            for (int64_t u = u0; u < u1; ++u) {
                const uint8_t* sb = rp + 210 * u;
                const unsigned short* sb16 = reinterpret_cast<const unsigned short*>(sb);
                const uint32_t a = __ldcs(sb16 + 32 * h + i);         // ql 64h + 2i, +1
                const uint32_t b = __ldcs(sb16 + 32 * h + 16 + i);    // ql 64h + 32 + 2i, +1
                const uint32_t c = __ldcs(sb16 + 64 + 16 * h + i);    // qh 32h + 2i, +1
                const float d = half_bits_to_float(__ldcs(sb16 + 104));
                // scale (lane % 16) as a float: (sc + 128) under 0x4B0000, minus 2^23 + 128
                const uint32_t ub = __ldcs(sb + 192 + (lane & 15));
                const float dsl = d * (__uint_as_float(0x4B000000u | (ub ^ 0x80u)) - 8388736.0f);
                // codes of columns 2i (byte 0) and 2i + 1 (byte 1) in quarter g
                const uint32_t q[4] = {(a & 0x0F0Fu) | ((c << 4) & 0x3030u), (b & 0x0F0Fu) | ((c << 2) & 0x3030u),
                                       ((a >> 4) & 0x0F0Fu) | (c & 0x3030u), ((b >> 4) & 0x0F0Fu) | ((c >> 2) & 0x3030u)};
                float2 w[4];
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float ds = __shfl_sync(0xffffffffu, dsl, 8 * h + 2 * g + (i >> 3));
                    const float2 f = make_float2(__uint_as_float(__byte_perm(q[g], 0x4B000000u, 0x7440)),
                                                 __uint_as_float(__byte_perm(q[g], 0x4B000000u, 0x7441)));
                    w[g] = __fmul2_rn(__fadd2_rn(f, make_float2(-8388640.0f, -8388640.0f)), make_float2(ds, ds));
                }
#pragma unroll
                for (int m = 0; m < MMAX; ++m) {
                    if (m >= M) continue;
                    const float* xb = x + m * cols + 256 * u + 128 * h + 2 * i;
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        acc[m] = __ffma2_rn(w[g], __ldg(reinterpret_cast<const float2*>(xb + 32 * g)), acc[m]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MMAX; ++m) {
            if (m >= M) continue;
            const float v = warp_sum(acc[m].x + acc[m].y);
            if (P == 1) {
                if (lane == 0 && row < rows) y[(int64_t)m * rows + row] = v;
            } else if (lane == 0) {
                red[warp][m] = v;
            }
        }
        if (P > 1) {
            __syncthreads();
            if (part == 0 && lane < M && lane < MMAX && row < rows) {
                float v = 0.0f;
                for (int p2 = 0; p2 < P; ++p2) v += red[warp + p2][lane];
                y[(int64_t)lane * rows + row] = v;
            }
            __syncthreads();   // red is reused by the next step
        }
    }
}

int num_sms() {
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

template <typename Kernel, typename WT, typename... Extra>
int launch(Kernel kernel, const WT* W, int64_t rows, int64_t cols, const float* x, float* y, int M,
           cudaStream_t stream, int rows_per_cta = kWarps, Extra... extra) {
    const int sms = num_sms();
    const int64_t want = (rows + rows_per_cta - 1) / rows_per_cta;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)std::max(sms, 1) * 8));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, W, x, y, rows, cols, M, extra...);
    return e == cudaSuccess ? GGQ_OK : cuda_fail(e, "gemv launch");
}

template <int MMAX>
int launch_mmax(int type, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int M,
                cudaStream_t stream) {
    if (type == GGQ_F32) {
        const float* w = static_cast<const float*>(W);
        if (cols % 4 == 0) return launch(gemv_f32_kernel<MMAX, true>, w, rows, cols, x, y, M, stream);
        return launch(gemv_f32_kernel<MMAX, false>, w, rows, cols, x, y, M, stream);
    }
    if (type == GGQ_Q6_K) {
        // warps per row: enough rows in flight for about 48 warps per SM
        const int64_t target = (int64_t)num_sms() * 48;
        int P = 1;
        while (P < kWarps && rows * P < target && cols / 256 >= 2 * P) P *= 2;
        if constexpr (MMAX == 1) {
            if (P == 1)
                return launch(gemv_q6k_rows_kernel<1, 6>, static_cast<const uint8_t*>(W), rows, cols, x, y, M, stream,
                              kWarps, 1);
        }
        constexpr int kMinB = MMAX <= 2 ? 4 : MMAX == 8 ? 3 : 2;   // the registers the build needs, no spills
        return launch(gemv_q6k_rows_kernel<MMAX, kMinB>, static_cast<const uint8_t*>(W), rows, cols, x, y, M, stream,
                      kWarps / P, P);
    }
    return launch(gemv_q40_rows_kernel<MMAX>, static_cast<const uint8_t*>(W), rows, cols, x, y, M, stream);
}

}  // namespace

int launch_gemv_rows(int type, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int M,
                     cudaStream_t stream) {
    if (type != GGQ_F32 && type != GGQ_Q4_0 && type != GGQ_Q6_K)
        return fail(GGQ_ETYPE, "gemv: type %d has no warp-per-row kernel", type);
    if (M <= 1) return launch_mmax<1>(type, W, rows, cols, x, y, M, stream);
    if (M <= 2) return launch_mmax<2>(type, W, rows, cols, x, y, M, stream);
    if (M <= 4) return launch_mmax<4>(type, W, rows, cols, x, y, M, stream);
    if (M <= 8) return launch_mmax<8>(type, W, rows, cols, x, y, M, stream);
    return launch_mmax<16>(type, W, rows, cols, x, y, M, stream);
}

}  // namespace ggq
