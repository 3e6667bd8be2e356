// Fused dequantize + GEMV / small-batch GEMM for Q8_0 and Q4_K weights.
//
//   y[m][r] = sum_c w[r][c] * x[m][c]      (matvec of the culpeo.ws kernel list;
//                                           "GGUF Inferencer in R" 5.2: normalized input times transposed weight)
//
// Q8_0 ("GGUF: The File Format...", "How a Q8_0 block is stored"): 32 weights per
// 34-byte block, fp16 d then 32 signed bytes q, w = d*q.
// Q4_K (same section, k-quant paragraph): 256 weights per 144-byte super-block,
// fp16 d, fp16 dmin, 12 bytes of packed 6-bit sub-block scales/mins, 128 bytes of
// nibbles; w = d*sc_j*q - dmin*m_j.
//
// Design (one GB300, HBM-bound at M = 1):
//  * A CTA owns 32 consecutive rows -- one per lane -- and a slice of the columns.
//    The CTAs that share a row block form a thread-block cluster (up to 8 along K);
//    their partial sums meet in distributed shared memory, so no global scratch
//    and no atomics are needed and the result is deterministic.
//  * The weight tile [32 rows x one unit] (unit = one Q4_K super-block column,
//    144 B per row, or one 8-block Q8_0 period, 272 B per row) arrives by a 2-D
//    bulk tensor copy (TMA).  Row pitches of 144 / 272 bytes make the per-lane
//    16-byte shared-memory reads conflict-free.
//  * Decoding costs one AND per weight: a nibble (or an offset byte) masked in
//    place inside a 32-bit word is a float bit pattern q * 2^(p-149) -- a
//    subnormal, or the first normal binade, which continue it linearly.  The
//    activations are pre-scaled by the matching power of two (x' = x * 2^(53-p)),
//    so the FFMA of pattern and x' adds exactly q*x*2^-96 to a per-sub-block sum.
//    Scales are applied once per 32 weights.  Q8_0 bytes are offset by 128 (XOR
//    0x80) to make them non-negative; 128 * sum(x) over the block is subtracted.
//  * x' and the per-sub-block sums of x are built once per CTA in shared memory;
//    every lane reads them as broadcasts.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "gemv_tile.cuh"
#include "ggq_internal.h"
#include "ptx.cuh"

namespace ggq {

namespace {

constexpr int kRows = 32;    // rows per CTA (one per lane)
constexpr int kWarps = 4;    // warps per CTA
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxCluster = 8;

// Q4_K unit: one super-block column of 32 rows
constexpr int kQ4kRowBytes = 144;
constexpr int kQ4kTile = kRows * kQ4kRowBytes;   // 4608
constexpr int kQ4kXp = 256;                      // x' floats per unit
// Q8_0 unit: 8 blocks = 256 weights = 272 bytes per row
constexpr int kQ8RowBytes = 272;
constexpr int kQ8Tile = kRows * kQ8RowBytes;     // 8704
constexpr int kQ8Xp = 272;                       // x' floats per unit (indexed by byte)

struct GemvParams {
    const float* x;
    float* y;
    int rows;
    int64_t cols;
    int M;
    int units;      // units per row (super-blocks or 8-block periods)
    int ksplit;     // CTAs per cluster along the columns
    int rbuf;       // unit buffers per CTA (units processed per round)
    int* status;
};

struct Smem {
    uint8_t* tiles;
    float* xp;
    float* sums;
    float* red;
    uint64_t* bars;   // [rbuf] weight tiles, then one for the x slice
    uint64_t* xbar;
};

template <int MMAX>
__device__ __forceinline__ Smem carve(uint8_t* smem, int rbuf, int tile, int xpn) {
    Smem s;
    s.tiles = smem;
    s.xp = reinterpret_cast<float*>(smem + (size_t)rbuf * tile);
    s.sums = s.xp + (size_t)MMAX * rbuf * xpn;
    s.red = s.sums + (size_t)MMAX * rbuf * 8;
    s.bars = reinterpret_cast<uint64_t*>(s.red + kWarps * MMAX * 32);
    s.xbar = s.bars + rbuf;
    return s;
}

// Final reduction: warps -> CTA partial -> cluster (rank order) -> y.
template <int MMAX>
__device__ __forceinline__ void reduce_store(const GemvParams& p, const Smem& s, const float (&acc)[MMAX],
                                             int rb, int ks) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int m = 0; m < MMAX; ++m) s.red[(warp * MMAX + m) * 32 + lane] = acc[m];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int m = 0; m < MMAX; ++m) {
            float v = s.red[m * 32 + lane];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) v += s.red[(w * MMAX + m) * 32 + lane];
            s.red[m * 32 + lane] = v;
        }
    }
    const int row = rb * kRows + lane;
    if (p.ksplit == 1) {
        if (warp == 0 && row < p.rows) {
            for (int m = 0; m < p.M; ++m) p.y[(int64_t)m * p.rows + row] = s.red[m * 32 + lane];
        }
        return;
    }
    cluster_sync();
    if (ks == 0 && warp == 0 && row < p.rows) {
        for (int m = 0; m < p.M; ++m) {
            float v = 0.0f;
            for (int r = 0; r < p.ksplit; ++r) v += ld_cluster_f32(&s.red[m * 32 + lane], (uint32_t)r);
            p.y[(int64_t)m * p.rows + row] = v;
        }
    }
    cluster_sync();  // keep every CTA's shared memory alive until rank 0 has read it
}

// ------------------------------------------------------------------- Q4_K ----

template <int MMAX>
__global__ void __launch_bounds__(kThreads) gemv_q4k_kernel(const __grid_constant__ CUtensorMap wmap,
                                                            const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ks = blockIdx.x % p.ksplit;
    const int rb = blockIdx.x / p.ksplit;
    const int u0 = (int)((int64_t)ks * p.units / p.ksplit);
    const int u1 = (int)((int64_t)(ks + 1) * p.units / p.ksplit);
    const int S = u1 - u0;
    const Smem s = carve<MMAX>(smem, p.rbuf, kQ4kTile, kQ4kXp);

    if (tid == 0) {
        prefetch_tensormap(&wmap);
        for (int u = 0; u < p.rbuf; ++u) mbar_init(&s.bars[u], 1);
        mbar_init(s.xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    float acc[MMAX];
#pragma unroll
    for (int m = 0; m < MMAX; ++m) acc[m] = 0.0f;

    int round = 0;
    for (int r0 = 0; r0 < S; r0 += p.rbuf, ++round) {
        const int n = min(p.rbuf, S - r0);
        if (tid == 0) {
            if (round == 0) {
                // warm L2 only; every copy waits for the previous kernel in the
                // stream, which may still be writing x (or W)
                for (int u = 0; u < n; ++u) tma_prefetch_2d(&wmap, (u0 + r0 + u) * kQ4kRowBytes, rb * kRows);
                pdl_wait();
            }
            for (int u = 0; u < n; ++u) {
                mbar_arrive_expect_tx(&s.bars[u], kQ4kTile);
                tma_load_2d(s.tiles + (size_t)u * kQ4kTile, &wmap, &s.bars[u], (u0 + r0 + u) * kQ4kRowBytes,
                            rb * kRows);
            }
            mbar_arrive_expect_tx(s.xbar, (uint32_t)(p.M * n * 1024));
            for (int m = 0; m < p.M; ++m)
                for (int u = 0; u < n; ++u)
                    bulk_load(s.xp + (size_t)(m * p.rbuf + u) * kQ4kXp,
                              p.x + (int64_t)m * p.cols + (int64_t)(u0 + r0 + u) * 256, 1024, s.xbar);
        }
        mbar_wait(s.xbar, round & 1, p.status);

        // x' = x * 2^(53 - p) (p = bit position of the weight's nibble in its
        // 32-bit word, see gemv_tile.cuh) and the sums of x per 32-weight
        // sub-block for the min term; one warp per unit reads the 256 floats in
        // natural order and writes them back in q4k_xslot order
        for (int job = warp; job < p.M * n; job += kWarps) {
            const int m = job / n, u = job - m * n;
            float* blk = s.xp + (size_t)(m * p.rbuf + u) * kQ4kXp;
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = blk[32 * i + lane];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float sum = warp_sum(v[i]);
                if (lane == 0) s.sums[(m * p.rbuf + u) * 8 + i] = sum;
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = 32 * i + lane;
                blk[q4k_xslot(k)] = v[i] * q4k_xscale(k);
            }
        }
        __syncthreads();

        for (int u = warp; u < n; u += kWarps) {
            mbar_wait(&s.bars[u], round & 1, p.status);
            q4k_tile_row<MMAX>(s.tiles + (size_t)u * kQ4kTile + lane * kQ4kRowBytes, s.xp + (size_t)u * kQ4kXp,
                               p.rbuf * kQ4kXp, s.sums + u * 8, p.rbuf * 8, acc);
        }
        __syncthreads();  // buffers are reused by the next round
    }
    reduce_store<MMAX>(p, s, acc, rb, ks);
}

// ------------------------------------------------------------------- Q8_0 ----

template <int MMAX>
__global__ void __launch_bounds__(kThreads) gemv_q8_kernel(const __grid_constant__ CUtensorMap wmap,
                                                           const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ks = blockIdx.x % p.ksplit;
    const int rb = blockIdx.x / p.ksplit;
    const int u0 = (int)((int64_t)ks * p.units / p.ksplit);
    const int u1 = (int)((int64_t)(ks + 1) * p.units / p.ksplit);
    const int S = u1 - u0;
    const Smem s = carve<MMAX>(smem, p.rbuf, kQ8Tile, kQ8Xp);

    if (tid == 0) {
        prefetch_tensormap(&wmap);
        for (int u = 0; u < p.rbuf; ++u) mbar_init(&s.bars[u], 1);
        mbar_init(s.xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    float acc[MMAX];
#pragma unroll
    for (int m = 0; m < MMAX; ++m) acc[m] = 0.0f;

    int round = 0;
    for (int r0 = 0; r0 < S; r0 += p.rbuf, ++round) {
        const int n = min(p.rbuf, S - r0);
        if (tid == 0) {
            if (round == 0) {
                // warm L2 only; every copy waits for the previous kernel in the stream
                for (int u = 0; u < n; ++u) tma_prefetch_2d(&wmap, (u0 + r0 + u) * (kQ8RowBytes / 2), rb * kRows);
                pdl_wait();
            }
            for (int u = 0; u < n; ++u) {
                mbar_arrive_expect_tx(&s.bars[u], kQ8Tile);
                // the map's elements are 2 bytes: 136 per 272-byte period
                tma_load_2d(s.tiles + (size_t)u * kQ8Tile, &wmap, &s.bars[u], (u0 + r0 + u) * (kQ8RowBytes / 2),
                            rb * kRows);
            }
            // raw x of unit u lands at float 16 of its 272-float region
            mbar_arrive_expect_tx(s.xbar, (uint32_t)(p.M * n * 1024));
            for (int m = 0; m < p.M; ++m)
                for (int u = 0; u < n; ++u)
                    bulk_load(s.xp + (size_t)(m * p.rbuf + u) * kQ8Xp + 16,
                              p.x + (int64_t)m * p.cols + (int64_t)(u0 + r0 + u) * 256, 1024, s.xbar);
        }
        mbar_wait(s.xbar, round & 1, p.status);

        // Move each x to the byte position B = 34b + 2 + i of its weight in the
        // period and scale it by 2^(53 - 8*min(B mod 4, 2)); 128 * sum(x) per block.
        // One warp walks a unit's blocks in order: block b writes [34b+2, 34b+34),
        // which never reaches the raw floats of blocks > b (they start at 32b+48).
        for (int job = warp; job < p.M * n; job += kWarps) {
            const int m = job / n, u = job - m * n;
            float* reg = s.xp + (size_t)(m * p.rbuf + u) * kQ8Xp;
#pragma unroll 1
            for (int b = 0; b < 8; ++b) {
                const float v = reg[16 + 32 * b + lane];
                const float sum = warp_sum(v);   // also orders the reads before the writes
                const int B = 34 * b + 2 + lane;
                reg[B] = v * q8_xscale(B);
                if (lane == 0) s.sums[(m * p.rbuf + u) * 8 + b] = 128.0f * sum;
                __syncwarp();
            }
        }
        __syncthreads();

        for (int u = warp; u < n; u += kWarps) {
            mbar_wait(&s.bars[u], round & 1, p.status);
            q8_tile_row<MMAX>(s.tiles + (size_t)u * kQ8Tile + lane * kQ8RowBytes, s.xp + (size_t)u * kQ8Xp,
                              p.rbuf * kQ8Xp, s.sums + u * 8, p.rbuf * 8, acc);
        }
        __syncthreads();
    }
    reduce_store<MMAX>(p, s, acc, rb, ks);
}

// Q8_0 with cols not a multiple of 256 (rows not 16-byte aligned): one warp per
// row, plain loads.  Correct for every shape; not the fast path.
__global__ void __launch_bounds__(kThreads) gemv_q8_simple_kernel(const uint8_t* __restrict__ W,
                                                                  const GemvParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    pdl_launch_dependents();
    pdl_wait();
    if (row >= p.rows) return;
    const int64_t nb = p.cols / 32;
    const uint8_t* rp = W + row * nb * 34;
    float acc[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) acc[m] = 0.0f;
    for (int64_t b = lane; b < nb; b += 32) {
        const uint8_t* blk = rp + 34 * b;
        const float d = half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8));
        for (int i = 0; i < 32; ++i) {
            const float w = d * (float)(int8_t)blk[2 + i];
#pragma unroll
            for (int m = 0; m < 16; ++m)
                if (m < p.M) acc[m] = fmaf(w, p.x[(int64_t)m * p.cols + 32 * b + i], acc[m]);
        }
    }
    for (int m = 0; m < p.M; ++m) {
        const float v = warp_sum(acc[m]);
        if (lane == 0) p.y[(int64_t)m * p.rows + row] = v;
    }
}

// --------------------------------------------------------------- host side ----

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D map over W viewed as [rows][row_bytes / elem] elements of 1 or 2 bytes.
int encode_weight_map(CUtensorMap* map, const void* W, int64_t rows, int64_t row_bytes, int elem_bytes,
                      int box_inner) {
    auto enc = tensor_map_encoder();
    if (!enc) return fail(GGQ_ECUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / elem_bytes), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)kRows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                     const_cast<void*>(W), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GGQ_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return GGQ_OK;
}

size_t smem_bytes(int mmax, int rbuf, int tile, int xpn) {
    return (size_t)rbuf * tile + (size_t)mmax * rbuf * xpn * 4 + (size_t)mmax * rbuf * 8 * 4 +
           (size_t)kWarps * mmax * 32 * 4 + (size_t)(rbuf + 1) * 8;
}

constexpr size_t kSmemLimit = 227 * 1024;

template <typename Kernel>
int launch(Kernel kernel, const CUtensorMap& map, const GemvParams& p, int grid, size_t smem, int cluster,
           cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (cluster > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)cluster;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kernel, map, p);
    if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
    return GGQ_OK;
}

template <int MMAX>
int launch_tma_gemv(int type, const void* W, int64_t rows, int64_t cols, GemvParams p, cudaStream_t stream) {
    const bool q4k = type == GGQ_Q4_K;
    const int tile = q4k ? kQ4kTile : kQ8Tile;
    const int xpn = q4k ? kQ4kXp : kQ8Xp;
    const int64_t units = cols / 256;
    const int64_t row_bytes = q4k ? cols / 256 * 144 : cols / 32 * 34;
    if (units > (1 << 24)) return fail(GGQ_EINVAL, "cols too large");
    // CTAs along K: aim at ~4 units per CTA, at most 8 (one cluster)
    int ksplit = (int)std::min<int64_t>(kMaxCluster, std::max<int64_t>(1, (units + 3) / 4));
    const int per_cta = (int)((units + ksplit - 1) / ksplit);
    int rbuf = per_cta;
    while (rbuf > 1 && smem_bytes(MMAX, rbuf, tile, xpn) > kSmemLimit) --rbuf;
    const size_t smem = smem_bytes(MMAX, rbuf, tile, xpn);
    if (smem > kSmemLimit) return fail(GGQ_EINVAL, "shape needs too much shared memory");
    CUtensorMap map;
    int rc = encode_weight_map(&map, W, rows, row_bytes, q4k ? 1 : 2, q4k ? kQ4kRowBytes : kQ8RowBytes / 2);
    if (rc) return rc;
    p.units = (int)units;
    p.ksplit = ksplit;
    p.rbuf = rbuf;
    const int64_t rowblocks = (rows + kRows - 1) / kRows;
    if (rowblocks * ksplit > 0x7fffffff) return fail(GGQ_EINVAL, "rows too large");
    const int grid = (int)(rowblocks * ksplit);
    if (q4k) return launch(gemv_q4k_kernel<MMAX>, map, p, grid, smem, ksplit, stream);
    return launch(gemv_q8_kernel<MMAX>, map, p, grid, smem, ksplit, stream);
}

}  // namespace

int launch_gemv(int type, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int M,
                cudaStream_t stream) {
    GemvParams p = {};
    p.x = x;
    p.y = y;
    p.rows = (int)rows;
    p.cols = cols;
    p.M = M;
    p.status = device_status_word();
    if (!p.status) return fail(GGQ_ECUDA, "device status word unavailable");
    if ((type == GGQ_Q4_0 || type == GGQ_Q6_K) && M >= kSmallMMin && smallm_supported(type, rows, cols, M))
        return launch_smallm(type, W, rows, cols, x, y, M, stream);   // one pass over W for all M rows
    if (M <= 4 || type == GGQ_Q4_0 || type == GGQ_Q6_K) {
        // the streaming kernel holds x' for up to 4 activation rows in shared
        // memory; where all M rows do not fit (4 rows of 14336 columns) or M > 4
        // (Q6_K, or a Q4_0 shape the small-M kernel does not take), it runs once
        // per group of g rows, the most that fit (x and y rows are contiguous)
        int g = std::min(M, 4);
        while (g > 0 && !stream_gemv_supported(type, cols, g, 1, &rows)) --g;
        if (g > 0) {
            for (int m0 = 0; m0 < M; m0 += g) {
                const void* Ws[1] = {W};
                float* ys[1] = {y + (int64_t)m0 * rows};
                const int rc = launch_gemv_stream(type, 1, Ws, &rows, cols, x + (int64_t)m0 * cols, ys,
                                                  std::min(g, M - m0), stream);
                if (rc) return rc;
            }
            return GGQ_OK;
        }
    }
    if (type == GGQ_F32 || type == GGQ_Q4_0 || type == GGQ_Q6_K)
        return launch_gemv_rows(type, W, rows, cols, x, y, M, stream);
    if (type == GGQ_Q8_0 && cols % 256 != 0) {
        const int64_t grid = (rows + kWarps - 1) / kWarps;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kThreads);
        cfg.stream = stream;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_q8_simple_kernel, static_cast<const uint8_t*>(W), p);
        return e == cudaSuccess ? GGQ_OK : cuda_fail(e, "gemv launch");
    }
    if (M >= kSmallMMin && smallm_supported(type, rows, cols, M))
        return launch_smallm(type, W, rows, cols, x, y, M, stream);
    if (M <= 1) return launch_tma_gemv<1>(type, W, rows, cols, p, stream);
    if (M <= 2) return launch_tma_gemv<2>(type, W, rows, cols, p, stream);
    if (M <= 4) return launch_tma_gemv<4>(type, W, rows, cols, p, stream);
    if (M <= 8) return launch_tma_gemv<8>(type, W, rows, cols, p, stream);
    return launch_tma_gemv<16>(type, W, rows, cols, p, stream);
}

}  // namespace ggq
