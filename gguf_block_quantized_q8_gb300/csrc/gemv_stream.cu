// Persistent stream-K GEMV: y = W x for one or several weight matrices that
// share x (e.g. the q, k and v projections of a layer), M = 1..4.
//
// Work is a flat sequence of tiles t = (row block, unit): 32 rows (one per lane)
// by one unit of columns (a Q4_K super-block column of 144 B per row, or an
// 8-block Q8_0 period of 272 B per row).  The sequence is cut into equal
// contiguous runs, one per warp, so every SM streams the same number of bytes
// whatever the shapes.  Each warp keeps its own ring of tile buffers filled by
// 2-D bulk tensor copies that its lane 0 issues as buffers free up.  x' (the
// pre-scaled activations, see gemv_tile.cuh) for all columns is built once per
// CTA in shared memory.
//
// A lane's dot product over a row block that lies wholly inside its warp's run
// is stored directly.  Row blocks cut by a run boundary are finished by the last
// warp to reach them: contributors write their partial sums to a workspace, bump
// a per-row-block counter, and the warp that brings the counter to the number
// of contributors adds the partials in warp order (deterministic), stores y and
// resets the counter to zero for the next launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <utility>

#include "gemv_tile.cuh"
#include "ggq_internal.h"
#include "ptx.cuh"

namespace ggq {

namespace {

constexpr int kRows = 32;
constexpr int kMaxWarps = 16;
constexpr int kMaxSeg = 4;
constexpr int kMaxM = 4;
constexpr size_t kSmemLimit = 227 * 1024;

struct Segment {
    float* y;     // [M][rows]
    int rows;
    int rb0;      // first global row block of this segment
};

struct Maps {
    CUtensorMap m[kMaxSeg];
};

struct StreamParams {
    const float* x;
    int64_t cols;
    int M;
    int units;          // units per row
    int nseg;
    Segment seg[kMaxSeg];
    int rb_total;       // row blocks over all segments
    int64_t tiles;      // rb_total * units
    int ngroups;        // warp groups with work
    int ring;           // tile buffers per warp
    int warps;          // warps per CTA
    float* partials;    // [ngroups][2][kMaxM][32]: R * M <= kMaxM values per lane
    int* counters;      // [rb_total], zero between launches
    int* status;
};

// A tile is 32*R rows (lane l owns rows l, l+32, ...) by one unit of columns.
template <bool Q4K, int R>
struct Unit {
    static constexpr int kRowBytes = Q4K ? 144 : 272;
    static constexpr int kTileRows = kRows * R;
    static constexpr int kTile = kTileRows * kRowBytes;
    static constexpr int kXp = Q4K ? 256 : 272;     // x' floats per unit (per activation row)
    static constexpr int kMapX = Q4K ? 144 : 136;   // map elements per unit (1 or 2 bytes each)
};

__device__ __forceinline__ int64_t run_start(int64_t g, int64_t T, int64_t NW) { return g * T / NW; }
// the group whose run contains tile t
__device__ __forceinline__ int64_t warp_of(int64_t t, int64_t T, int64_t NW) { return ((t + 1) * NW - 1) / T; }

__device__ __forceinline__ int seg_of(const StreamParams& p, int gr) {
    int s = 0;
#pragma unroll
    for (int i = 1; i < kMaxSeg; ++i)
        if (i < p.nseg && gr >= p.seg[i].rb0) s = i;
    return s;
}

// Warps work in groups of G sharing one ring of tiles: with G = 4 (Q4_K) warp w
// of a group decodes chunk w (64 columns) of every tile, so a tile is done four
// times sooner; with G = 1 a warp takes whole tiles.  Groups are numbered across
// CTAs first (group index = group-in-CTA * gridDim.x + CTA) so the active ones
// spread over all SMs when there are few tiles.
template <bool Q4K, int MMAX, int R, int W, int G>
__global__ void __launch_bounds__(32 * W, 1) gemv_stream_kernel(const __grid_constant__ Maps maps,
                                                                 const StreamParams p) {
    static_assert(R * MMAX <= kMaxM, "partials slot too small");
    static_assert(Q4K || G == 1, "Q8_0 tiles are taken whole");
    constexpr int kThreads = 32 * W;
    constexpr int NG = W / G;
    using U = Unit<Q4K, R>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = warp / G, wig = warp % G;
    const int64_t gg = (int64_t)grp * gridDim.x + blockIdx.x;
    const bool active = gg < p.ngroups;
    const int64_t T = p.tiles, NW = p.ngroups;
    const int64_t t0 = active ? run_start(gg, T, NW) : 0, t1 = active ? run_start(gg + 1, T, NW) : 0;
    const int n = (int)(t1 - t0);

    // shared memory: [group rings][x'][sums][row-block partials][barriers]
    uint8_t* ring = smem + (size_t)grp * p.ring * U::kTile;
    float* xp = reinterpret_cast<float*>(smem + (size_t)NG * p.ring * U::kTile);
    const int xs = Q4K ? (int)p.cols : p.units * U::kXp;            // x' floats per activation row
    const int nsub = (int)(p.cols / 32);                              // sums per activation row
    float* sums = xp + (size_t)MMAX * xs;
    float* red = sums + (size_t)MMAX * nsub;                          // [NG][2][G][R*MMAX][32] when G > 1
    uint64_t* bars = reinterpret_cast<uint64_t*>(red + (G > 1 ? NG * 2 * G * R * MMAX * 32 : 0));
    uint64_t* full = bars + grp * p.ring;
    uint64_t* empty = bars + NG * p.ring + grp * p.ring;

    const bool producer = active && wig == 0 && lane == 0;
    // The producer walks its group's run with a (row block, unit) cursor; tile i
    // of the run goes to buffer i % ring.
    int pgr = 0, pu = 0, pslot = 0;   // producer cursor and next buffer
    if (producer) {
        pgr = (int)(t0 / p.units);
        pu = (int)(t0 - (int64_t)pgr * p.units);
    }
    auto issue = [&](int /*i*/) {   // issues tiles strictly in order
        const int s = seg_of(p, pgr);
        mbar_arrive_expect_tx(&full[pslot], U::kTile);
        tma_load_2d(ring + (size_t)pslot * U::kTile, &maps.m[s], &full[pslot], pu * U::kMapX,
                    (pgr - p.seg[s].rb0) * U::kTileRows);
        if (++pu == p.units) { pu = 0; ++pgr; }
        if (++pslot == p.ring) pslot = 0;
    };

    if (tid == 0) {
        for (int i = 0; i < NG * p.ring; ++i) {
            mbar_init(&bars[i], 1);
            mbar_init(&bars[NG * p.ring + i], G);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    // Each group's producer starts its first tiles (weights never depend on the
    // previous kernel).  A producer may stall here while the copy engine is
    // backed up behind HBM; the other warps go on building x'.
    if (producer) {
        for (int s = 0; s < p.nseg; ++s) prefetch_tensormap(&maps.m[s]);
        for (int i = 0; i < min(n, p.ring); ++i) issue(i);
    }

    // x' for every column, built once per CTA with ordinary loads (they do not
    // queue behind the tile copies)
    pdl_wait();   // x may come from the previous kernel in the stream
    if (Q4K) {
        // one warp per super-block: scale each x, sum each 32-weight sub-block,
        // store in q4k_xslot order
        const int nsb = (int)(p.cols / 256);
        for (int job = warp; job < p.M * nsb; job += W) {
            const int m = job / nsb, sb = job - m * nsb;
            const float* src = p.x + (int64_t)m * p.cols + (int64_t)sb * 256;
            float* blk = xp + (size_t)m * xs + (size_t)sb * 256;
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = src[32 * i + lane];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = 32 * i + lane;
                blk[q4k_xslot(k)] = v[i] * q4k_xscale(k);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float sum = warp_sum(v[i]);
                if (lane == 0) sums[m * nsub + sb * 8 + i] = sum;
            }
        }
    } else {
        // each x goes to the byte position B = 34b + 2 + i of its weight in the
        // 272-byte period; 128 * sum(x) per block
        for (int job = warp; job < p.M * p.units; job += W) {
            const int m = job / p.units, u = job - m * p.units;
            const float* src = p.x + (int64_t)m * p.cols + (int64_t)u * 256;
            float* reg = xp + (size_t)m * xs + (size_t)u * U::kXp;
            float v[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) v[b] = src[32 * b + lane];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int B = 34 * b + 2 + lane;
                reg[B] = v[b] * q8_xscale(B);
            }
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const float sum = warp_sum(v[b]);
                if (lane == 0) sums[m * nsub + u * 8 + b] = 128.0f * sum;
            }
        }
    }
    __syncthreads();
    if (!active) return;

    float acc[R][MMAX];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MMAX; ++m) acc[r][m] = 0.0f;
    const int gr_first = (int)(t0 / p.units);
    int gr = gr_first;
    int u = (int)(t0 - (int64_t)gr * p.units);   // consumer cursor: tile t0 + i is (gr, u)
    bool covered_from_start = u == 0;
    int nflush = 0;

    // finish row block `cur`: sum the group's warps, then store directly if this
    // group covered all of it, otherwise deposit the partial and let the last
    // contributor add them up
    auto flush = [&](int cur, bool whole) {
        if constexpr (G > 1) {
            float* mine = red + ((size_t)((grp * 2 + (nflush & 1)) * G + wig) * R * MMAX) * 32;
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < MMAX; ++m) mine[(r * MMAX + m) * 32 + lane] = acc[r][m];
            asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(32 * G) : "memory");
            const float* all = red + ((size_t)(grp * 2 + (nflush & 1)) * G * R * MMAX) * 32;
            ++nflush;
            if (wig != 0) return;
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < MMAX; ++m) {
                    float v = all[(r * MMAX + m) * 32 + lane];
#pragma unroll
                    for (int w = 1; w < G; ++w) v += all[((size_t)w * R * MMAX + r * MMAX + m) * 32 + lane];
                    acc[r][m] = v;
                }
        }
        const int s = seg_of(p, cur);
        const int row0 = (cur - p.seg[s].rb0) * U::kTileRows + lane;
        const int rows = p.seg[s].rows;
        float* ys = p.seg[s].y;
        if (whole) {
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (row0 + 32 * r < rows)
#pragma unroll
                    for (int m = 0; m < MMAX; ++m)
                        if (m < p.M) ys[(int64_t)m * rows + row0 + 32 * r] = acc[r][m];
            return;
        }
        const int slot = cur == gr_first ? 0 : 1;
        float* part = p.partials + ((gg * 2 + slot) * kMaxM) * 32;
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MMAX; ++m) part[(r * MMAX + m) * 32 + lane] = acc[r][m];
        __threadfence();
        __syncwarp();
        const int64_t lo = warp_of((int64_t)cur * p.units, T, NW);
        const int64_t hi = warp_of((int64_t)(cur + 1) * p.units - 1, T, NW);
        int prev = 0;
        if (lane == 0) prev = atomicAdd(&p.counters[cur], 1);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev != (int)(hi - lo)) return;
        __threadfence();
        // add the contributors' partials in group order, eight loads in flight
        float v[R][MMAX];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MMAX; ++m) v[r][m] = 0.0f;
        for (int64_t c0 = lo; c0 <= hi; c0 += 8) {
            float q[8][R * MMAX];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int64_t c = c0 + j;
                if (c <= hi) {
                    const int cslot = (int)(run_start(c, T, NW) / p.units) == cur ? 0 : 1;
                    const float* src = p.partials + ((c * 2 + cslot) * kMaxM) * 32 + lane;
#pragma unroll
                    for (int k = 0; k < R * MMAX; ++k) q[j][k] = __ldcg(src + k * 32);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (c0 + j <= hi)
#pragma unroll
                    for (int r = 0; r < R; ++r)
#pragma unroll
                        for (int m = 0; m < MMAX; ++m) v[r][m] += q[j][r * MMAX + m];
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (row0 + 32 * r < rows)
#pragma unroll
                for (int m = 0; m < MMAX; ++m)
                    if (m < p.M) ys[(int64_t)m * rows + row0 + 32 * r] = v[r][m];
        if (lane == 0) atomicExch(&p.counters[cur], 0);
    };

    int slot = 0;
    uint32_t parity = 0;   // phase of buffer `slot` for tile i: (i / ring) & 1
    for (int i = 0; i < n; ++i) {
        if (i > 0 && u == 0) {
            flush(gr - 1, covered_from_start);   // the run passed the previous row block's end
            covered_from_start = true;
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < MMAX; ++m) acc[r][m] = 0.0f;
        }
        mbar_wait(&full[slot], parity, p.status);
        const uint8_t* rp = ring + (size_t)slot * U::kTile + lane * U::kRowBytes;
        if constexpr (Q4K) {
            if constexpr (G == 4)
                q4k_chunk_rows<MMAX, R>(rp, 32 * U::kRowBytes, wig, xp + (size_t)u * 256, xs, sums + u * 8, nsub, acc);
            else
                q4k_tile_rows<MMAX, R>(rp, 32 * U::kRowBytes, xp + (size_t)u * 256, xs, sums + u * 8, nsub, acc);
        } else {
            q8_tile_row<MMAX>(rp, xp + (size_t)u * U::kXp, xs, sums + u * 8, nsub, acc[0]);
        }
        if (++u == p.units) { u = 0; ++gr; }
        __syncwarp();
        if constexpr (G == 1) {
            if (lane == 0 && i + p.ring < n) {
                fence_proxy_async_smem();   // our reads of this buffer before the copy that overwrites it
                issue(i + p.ring);
            }
        } else {
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (producer && i + p.ring < n) {
                mbar_wait(&empty[slot], parity, p.status);   // every warp of the group is done with it
                fence_proxy_async_smem();
                issue(i + p.ring);
            }
        }
        if (++slot == p.ring) { slot = 0; parity ^= 1u; }
    }
    // the row block holding the run's last tile
    if (u == 0) flush(gr - 1, covered_from_start);
    else flush(gr, false);
}

// ------------------------------------------------------------------ host ----

struct Workspace {
    float* partials = nullptr;
    int* counters = nullptr;
    int max_warps = 0;
    int max_rb = 0;
};

std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

int num_sms() {
    static int sms[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 1;
    if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    return sms[dev] > 0 ? sms[dev] : 1;
}

// Per (device, stream) workspace; allocated on the first call that needs it
// (and grown if a later call needs more row blocks).
int get_workspace(cudaStream_t stream, int warps, int rb, Workspace** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace& ws = g_ws[{dev, stream}];
    if (ws.max_warps < warps) {
        if (ws.partials) cudaFree(ws.partials);
        ws.partials = nullptr;
        const int want = std::max(warps, 152 * kMaxWarps);
        e = cudaMalloc(&ws.partials, (size_t)want * 2 * kMaxM * 32 * sizeof(float));
        if (e != cudaSuccess) { ws.max_warps = 0; return cuda_fail(e, "workspace allocation"); }
        ws.max_warps = want;
    }
    if (ws.max_rb < rb) {
        if (ws.counters) cudaFree(ws.counters);
        ws.counters = nullptr;
        const int want = std::max(rb, 1 << 17);
        e = cudaMalloc(&ws.counters, (size_t)want * sizeof(int));
        if (e != cudaSuccess) { ws.max_rb = 0; return cuda_fail(e, "workspace allocation"); }
        e = cudaMemsetAsync(ws.counters, 0, (size_t)want * sizeof(int), stream);
        if (e != cudaSuccess) return cuda_fail(e, "workspace clear");
        ws.max_rb = want;
    }
    *out = &ws;
    return GGQ_OK;
}

int encode_map(CUtensorMap* map, const void* W, int64_t rows, int64_t row_bytes, bool q4k, int box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    if (!fn) return fail(GGQ_ECUDA, "cuTensorMapEncodeTiled unavailable");
    const int elem = q4k ? 1 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / elem), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)(q4k ? 144 : 136), (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(map, q4k ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                    const_cast<void*>(W), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GGQ_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return GGQ_OK;
}

// Launch shape: warps per CTA, warps per tile group, rows per lane.
// GGQ_STREAM_SHAPE="warps,group,rows" overrides the default (a tuning aid).
struct Shape {
    int warps;
    int group;
    int rows;
};

Shape stream_shape(bool q4k, int mmax) {
    Shape sh = q4k ? (mmax == 1 ? Shape{16, 4, 2} : Shape{16, 4, 1}) : Shape{8, 1, 1};
    if (const char* e = getenv("GGQ_STREAM_SHAPE")) {
        int w = 0, g = 0, r = 0;
        if (sscanf(e, "%d,%d,%d", &w, &g, &r) == 3 && (w == 8 || w == 16) && (g == 1 || (g == 4 && q4k)) &&
            (r == 1 || (r == 2 && q4k && mmax == 1)))
            sh = {w, g, r};
    }
    return sh;
}

int rows_per_lane(bool q4k, int mmax) { return stream_shape(q4k, mmax).rows; }

size_t stream_smem(bool q4k, int mmax, int ring, int64_t cols) {
    const Shape sh = stream_shape(q4k, mmax);
    const int ng = sh.warps / sh.group;
    const int tile = kRows * sh.rows * (q4k ? 144 : 272);
    const int64_t xs = q4k ? cols : cols / 256 * 272;
    const size_t red = sh.group > 1 ? (size_t)ng * 2 * sh.group * sh.rows * mmax * 32 * 4 : 0;
    return (size_t)ng * ring * tile + (size_t)mmax * xs * 4 + (size_t)mmax * (cols / 32) * 4 + red +
           (size_t)(2 * ng * ring) * 8;
}

template <bool Q4K, int MMAX, int R, int W, int G>
int launch_stream_t(const Maps& maps, StreamParams& p, int grid, cudaStream_t stream) {
    const size_t smem = stream_smem(Q4K, MMAX, p.ring, p.cols);
    auto kernel = gemv_stream_kernel<Q4K, MMAX, R, W, G>;
    static int configured[64] = {};   // largest dynamic smem set so far, per device
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t e = cudaSuccess;
    if (dev < 0 || dev >= 64 || configured[dev] < (int)smem) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        if (dev >= 0 && dev < 64) configured[dev] = (int)smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(32 * W);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, maps, p);
    if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
    return GGQ_OK;
}

}  // namespace

bool stream_gemv_supported(int type, int64_t cols, int M, int nseg, const int64_t* rows) {
    if (M > kMaxM || nseg < 1 || nseg > kMaxSeg || cols % 256) return false;
    const bool q4k = type == GGQ_Q4_K;
    const int mmax = M <= 1 ? 1 : M <= 2 ? 2 : 4;
    const int trows = kRows * rows_per_lane(q4k, mmax);
    int64_t rb = 0;
    for (int s = 0; s < nseg; ++s) rb += (rows[s] + trows - 1) / trows;
    if (rb > (1 << 22)) return false;
    return stream_smem(q4k, mmax, 1, cols) <= kSmemLimit;
}

int launch_gemv_stream(int type, int nseg, const void* const* W, const int64_t* rows, int64_t cols, const float* x,
                       float* const* y, int M, cudaStream_t stream) {
    const bool q4k = type == GGQ_Q4_K;
    const int mmax = M <= 1 ? 1 : M <= 2 ? 2 : 4;
    const int64_t units = cols / 256;
    const int64_t row_bytes = q4k ? units * 144 : units * 272;
    Maps maps;
    StreamParams p = {};
    p.x = x;
    p.cols = cols;
    p.M = M;
    p.units = (int)units;
    p.nseg = nseg;
    const int trows = kRows * rows_per_lane(q4k, mmax);
    int rb = 0;
    for (int s = 0; s < nseg; ++s) {
        int rc = encode_map(&maps.m[s], W[s], rows[s], row_bytes, q4k, trows);
        if (rc) return rc;
        p.seg[s].y = y[s];
        p.seg[s].rows = (int)rows[s];
        p.seg[s].rb0 = rb;
        rb += (int)((rows[s] + trows - 1) / trows);
    }
    p.rb_total = rb;
    p.tiles = (int64_t)rb * units;
    // ring depth: as deep as shared memory allows (up to 8 tiles per group)
    const Shape sh = stream_shape(q4k, mmax);
    int ring = 8;
    while (ring > 1 && stream_smem(q4k, mmax, ring, cols) > kSmemLimit) --ring;
    if (stream_smem(q4k, mmax, ring, cols) > kSmemLimit) return fail(GGQ_EINVAL, "shape needs too much shared memory");
    p.ring = ring;
    // groups: one run of >= 1 tile each, at most (SMs x groups per CTA); one CTA
    // per SM
    const int ng = sh.warps / sh.group;
    const int64_t max_groups = (int64_t)num_sms() * ng;
    p.ngroups = (int)std::max<int64_t>(1, std::min<int64_t>(max_groups, p.tiles));
    const int grid = (int)std::min<int64_t>(num_sms(), p.ngroups);
    Workspace* ws = nullptr;
    int rc = get_workspace(stream, p.ngroups, rb, &ws);
    if (rc) return rc;
    p.partials = ws->partials;
    p.counters = ws->counters;
    p.status = device_status_word();
    if (!p.status) return fail(GGQ_ECUDA, "device status word unavailable");
    if (q4k) {
        if (mmax == 1) {
            if (sh.group == 4) {
                if (sh.rows == 2) return sh.warps == 16 ? launch_stream_t<true, 1, 2, 16, 4>(maps, p, grid, stream)
                                                        : launch_stream_t<true, 1, 2, 8, 4>(maps, p, grid, stream);
                return sh.warps == 16 ? launch_stream_t<true, 1, 1, 16, 4>(maps, p, grid, stream)
                                      : launch_stream_t<true, 1, 1, 8, 4>(maps, p, grid, stream);
            }
            if (sh.rows == 2) return launch_stream_t<true, 1, 2, 8, 1>(maps, p, grid, stream);
            return launch_stream_t<true, 1, 1, 8, 1>(maps, p, grid, stream);
        }
        if (mmax == 2) return launch_stream_t<true, 2, 1, 16, 4>(maps, p, grid, stream);
        return launch_stream_t<true, 4, 1, 16, 4>(maps, p, grid, stream);
    }
    if (mmax == 1) return sh.warps == 16 ? launch_stream_t<false, 1, 1, 16, 1>(maps, p, grid, stream)
                                         : launch_stream_t<false, 1, 1, 8, 1>(maps, p, grid, stream);
    if (mmax == 2) return launch_stream_t<false, 2, 1, 8, 1>(maps, p, grid, stream);
    return launch_stream_t<false, 4, 1, 8, 1>(maps, p, grid, stream);
}

// Same launch with caller-provided scratch instead of the per-stream workspace:
// `partials` holds max_groups * 2 * kMaxM * 32 floats and `counters`
// max_row_blocks ints.  The counters this call uses are cleared first
// (cudaMemsetAsync on `stream`); nothing is allocated.
int launch_gemv_stream_scratch(int type, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int M,
                               cudaStream_t stream, float* partials, int max_groups, int* counters,
                               int max_row_blocks) {
    const bool q4k = type == GGQ_Q4_K;
    const int mmax = M <= 1 ? 1 : M <= 2 ? 2 : 4;
    const int64_t units = cols / 256;
    const int64_t row_bytes = q4k ? units * 144 : units * 272;
    const int trows = kRows * rows_per_lane(q4k, mmax);
    const int64_t rb = (rows + trows - 1) / trows;
    if (rb > max_row_blocks)
        return fail(GGQ_EINVAL, "rows %lld exceed the %lld rows the built-in scratch can finish",
                    (long long)rows, (long long)max_row_blocks * trows);
    Maps maps;
    StreamParams p = {};
    p.x = x;
    p.cols = cols;
    p.M = M;
    p.units = (int)units;
    p.nseg = 1;
    int rc = encode_map(&maps.m[0], W, rows, row_bytes, q4k, trows);
    if (rc) return rc;
    p.seg[0].y = y;
    p.seg[0].rows = (int)rows;
    p.seg[0].rb0 = 0;
    p.rb_total = (int)rb;
    p.tiles = rb * units;
    const Shape sh = stream_shape(q4k, mmax);
    int ring = 8;
    while (ring > 1 && stream_smem(q4k, mmax, ring, cols) > kSmemLimit) --ring;
    if (stream_smem(q4k, mmax, ring, cols) > kSmemLimit) return fail(GGQ_EINVAL, "shape needs too much shared memory");
    p.ring = ring;
    const int ng = sh.warps / sh.group;
    const int64_t most = std::min<int64_t>((int64_t)num_sms() * ng, max_groups);
    p.ngroups = (int)std::max<int64_t>(1, std::min<int64_t>(most, p.tiles));
    const int grid = (int)std::min<int64_t>(num_sms(), p.ngroups);
    p.partials = partials;
    p.counters = counters;
    p.status = device_status_word();
    if (!p.status) return fail(GGQ_ECUDA, "device status word unavailable");
    cudaError_t e = cudaMemsetAsync(counters, 0, (size_t)rb * sizeof(int), stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the scratch counters");
    if (q4k) {
        if (mmax == 1) {
            if (sh.group == 4) {
                if (sh.rows == 2) return sh.warps == 16 ? launch_stream_t<true, 1, 2, 16, 4>(maps, p, grid, stream)
                                                        : launch_stream_t<true, 1, 2, 8, 4>(maps, p, grid, stream);
                return sh.warps == 16 ? launch_stream_t<true, 1, 1, 16, 4>(maps, p, grid, stream)
                                      : launch_stream_t<true, 1, 1, 8, 4>(maps, p, grid, stream);
            }
            if (sh.rows == 2) return launch_stream_t<true, 1, 2, 8, 1>(maps, p, grid, stream);
            return launch_stream_t<true, 1, 1, 8, 1>(maps, p, grid, stream);
        }
        if (mmax == 2) return launch_stream_t<true, 2, 1, 16, 4>(maps, p, grid, stream);
        return launch_stream_t<true, 4, 1, 16, 4>(maps, p, grid, stream);
    }
    if (mmax == 1) return sh.warps == 16 ? launch_stream_t<false, 1, 1, 16, 1>(maps, p, grid, stream)
                                         : launch_stream_t<false, 1, 1, 8, 1>(maps, p, grid, stream);
    if (mmax == 2) return launch_stream_t<false, 2, 1, 8, 1>(maps, p, grid, stream);
    return launch_stream_t<false, 4, 1, 8, 1>(maps, p, grid, stream);
}

}  // namespace ggq
