// Persistent row-partitioned GEMV over a chain of dependent stages.
//
// A stage is up to four weight matrices of one type and width that share their
// input x (e.g. the q, k and v projections of a layer): y_i = W_i x.  A chain is
// a list of stages run in order; stage s+1 reads its x only after every output
// of stage s is written, so the x of a later stage may be the y of an earlier
// one.  A single GEMV is a chain of one stage.
//
// Work unit: one 256-column block of one row (SB) -- a Q4_K super-block
// (144 B) or a Q8_0 period of 8 blocks (272 B).  The rows of a stage's
// matrices are numbered one after another; SB S = row * U + u (U = cols/256)
// sits right after SB S - 1 in memory inside one matrix.
//
//   * CTA b (one per SM) owns rows [R*b/G, R*(b+1)/G): whole rows, so no output
//     is ever split between CTAs and no cross-CTA reduction exists.
//   * Its SB range is cut into W equal contiguous pieces, one per warp.  A warp
//     streams its piece through its own ring of tiles of 32 SBs with 1-D bulk
//     copies (lane 0 issues them; weights do not depend on earlier stages, so
//     the ring runs ahead into the next stages while the chain waits at a stage
//     boundary).
//   * Lane l decodes SB l of a tile in registers against x', the pre-scaled
//     activations of its column block (interleaved across column blocks so
//     lanes reading different blocks hit different banks).  A segmented warp
//     sum adds the SBs of each row; a row that a warp sees from start to end is
//     stored directly, a row cut between warps is finished in shared memory by
//     the warp where it starts, adding the others' parts in warp order
//     (deterministic).
//   * Stage boundary: every CTA adds one to a device counter with release
//     semantics after its outputs are stored; CTAs wait (acquire, bounded) for
//     the count of all CTAs before reading the next stage's x.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "gemv_tile.cuh"
#include "ggq_internal.h"
#include "ptx.cuh"

namespace ggq {

namespace {

constexpr int kMaxSeg = 4;
constexpr int kMaxM = 4;
constexpr int kLanes = 32;
constexpr size_t kSmemLimit = 227 * 1024;

// One stage of a chain (device-visible: kernel parameter or global table).
struct StageDesc {
    const uint8_t* W[kMaxSeg];
    float* y[kMaxSeg];          // [M][rows]
    const float* x;             // [M][cols]
    int rows[kMaxSeg];
    int row0[kMaxSeg + 1];      // first row of each matrix in the stage's numbering; row0[nseg] = rows of the stage
    int nseg;
    int cols;
    int units;                  // U = cols / 256
};

struct ChainParams {
    const StageDesc* table;     // the stages in device memory, or null: the inline stage only
    int nstages;
    int M;
    int ring;                   // tiles per warp ring
    int xs;                     // x' floats per activation row (widest stage)
    int nsub;                   // x sums per activation row (widest stage)
    int* counter;               // stage counter (chains of > 1 stage); zero between launches
    int* status;
};

template <bool Q4K>
struct Blk {
    static constexpr int kBytes = Q4K ? 144 : 272;   // one SB
    static constexpr int kTile = kLanes * kBytes;
};

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int ld_relaxed(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int atom_acq_rel_add(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_relaxed(int* p, int v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits are bounded (kWaitLimitNs).  Once any wait of any CTA has run out (the
// status word is set) the others shorten theirs to kDrainNs: the kernel then
// only drains its own copies in flight and ends, instead of timing out once
// per remaining tile.
constexpr unsigned long long kDrainNs = 1000000ull;   // 1 ms

// Wait until *counter >= target (other CTAs finishing a stage).
__device__ __forceinline__ void wait_count(const int* counter, int target, int* status) {
    if (ld_acquire(counter) >= target) return;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ld_acquire(counter) >= target) return;   // each poll is an L2 round trip
        if ((it & 15u) == 0) {
            if (ld_relaxed(status) != 0) return;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                atomicOr(status, kStatusTimeout);
                return;
            }
        }
    }
}

// Wait for phase `parity` of a tile buffer's full barrier.
__device__ __forceinline__ void wait_full(uint64_t* bar, uint32_t parity, int* status) {
    if (mbar_try_wait(bar, parity)) return;
    const unsigned long long t0 = globaltimer_ns();
    unsigned long long limit = kWaitLimitNs;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return;
        if ((it & 255u) == 0) {
            const unsigned long long dt = globaltimer_ns() - t0;
            if (limit == kWaitLimitNs && ld_relaxed(status) != 0) limit = dt + kDrainNs;
            if (dt > limit) {
                atomicOr(status, kStatusTimeout);
                return;
            }
        }
    }
}

// The SB range [ws, we) of warp w (of nw) of CTA b (of nb) in a stage.
__device__ __forceinline__ void warp_range(const StageDesc* sd, int b, int nb, int w, int nw, int& ws, int& we) {
    const long long R = sd->row0[sd->nseg];
    const long long rlo = R * b / nb, rhi = R * (b + 1) / nb;
    const long long base = rlo * sd->units, n = (rhi - rlo) * sd->units;
    ws = (int)(base + n * w / nw);
    we = (int)(base + n * (w + 1) / nw);
}

__device__ __forceinline__ int seg_of_row(const StageDesc* sd, int g) {
    int s = 0;
#pragma unroll
    for (int i = 1; i < kMaxSeg; ++i)
        if (i < sd->nseg && g >= sd->row0[i]) s = i;
    return s;
}

// Issue the bulk copies of SBs [a, b) of a stage into `dst` (one thread).
template <bool Q4K>
__device__ __forceinline__ void issue_tile(const StageDesc* sd, int a, int b, uint8_t* dst, uint64_t* bar) {
    using B = Blk<Q4K>;
    fence_proxy_async_smem();   // this warp's reads of the buffer come before the copy's writes
    mbar_arrive_expect_tx(bar, (uint32_t)(b - a) * B::kBytes);
    const int U = sd->units;
    for (int s = 0; s < sd->nseg; ++s) {
        const int lo = max(a, sd->row0[s] * U), hi = min(b, sd->row0[s + 1] * U);
        if (lo < hi)
            bulk_load(dst + (size_t)(lo - a) * B::kBytes, sd->W[s] + (size_t)(lo - sd->row0[s] * U) * B::kBytes,
                      (uint32_t)(hi - lo) * B::kBytes, bar);
    }
}

template <bool Q4K, int MMAX, int W>
__global__ void __launch_bounds__(32 * W, 1) rows_kernel(const __grid_constant__ StageDesc inl, const ChainParams p) {
    using B = Blk<Q4K>;
    constexpr int kThreads = 32 * W;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int D = p.ring;

    // shared memory: [warp rings][x'][sums][cut-row parts][barriers]
    uint8_t* ring = smem + (size_t)warp * D * B::kTile;
    float* xp = reinterpret_cast<float*>(smem + (size_t)W * D * B::kTile);
    float* sums = xp + (size_t)MMAX * p.xs;
    float* cut_val = sums + (size_t)MMAX * p.nsub;                 // [2][W][MMAX]: row part before / after
    int* cut_row = reinterpret_cast<int*>(cut_val + 2 * W * MMAX);   // [2][W]
    uint64_t* full = reinterpret_cast<uint64_t*>(cut_row + 2 * W) + warp * D;   // 8-byte aligned: all sizes even

    if (lane == 0) {
        for (int i = 0; i < D; ++i) mbar_init(&full[i], 1);
        fence_mbar_init();
    }
    __syncwarp();
    pdl_launch_dependents();

    // ---- copy cursor of this warp: its tiles of every stage, in order
    int cs = -1, cj = 0, cn = 0, cws = 0, cwe = 0;   // stage, next tile, tiles in stage, range
    int issued = 0, consumed = 0;
    auto refill = [&]() {   // keep up to D tiles in flight or resident
        while (issued - consumed < D) {
            while (cj == cn && cs < p.nstages) {   // next stage in which this warp has tiles
                if (++cs == p.nstages) break;
                const StageDesc* sd = p.table ? p.table + cs : &inl;
                warp_range(sd, blockIdx.x, gridDim.x, warp, W, cws, cwe);
                cj = 0;
                cn = (cwe - cws + kLanes - 1) / kLanes;
            }
            if (cs >= p.nstages) break;
            const StageDesc* sd = p.table ? p.table + cs : &inl;
            const int a = cws + cj * kLanes, b = min(a + kLanes, cwe);
            const int slot = issued % D;
            if (lane == 0) issue_tile<Q4K>(sd, a, b, ring + (size_t)slot * B::kTile, &full[slot]);
            ++cj;
            ++issued;
        }
    };
    refill();

    for (int s = 0; s < p.nstages; ++s) {
        const StageDesc* sd = p.table ? p.table + s : &inl;
        if (s == 0) {
            pdl_wait();   // x may come from the previous kernel in the stream
        } else {
            // every CTA has finished stage s-1 (its outputs are visible)
            if (tid == 0) wait_count(p.counter, s * (int)gridDim.x, p.status);
            __syncthreads();
        }
        const int cols = sd->cols, U = sd->units;
        const int xs = p.xs, nsub = p.nsub;

        // ---- x' and the 32-column sums of this stage, interleaved over column
        // blocks: float4 group q of block u at index q*U + u.  x may have been
        // written by other CTAs: read it from L2.
        {
            const int nx = p.M * cols;
            for (int k0 = warp * 32; k0 < nx; k0 += kThreads * 4) {
                float v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int k = k0 + i * kThreads + lane;
                    v[i] = k < nx ? __ldcg(sd->x + k) : 0.0f;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int kb = k0 + i * kThreads;   // warp-uniform: one 32-column block of x
                    if (kb >= nx) break;
                    const int m = kb / cols, kc = kb - m * cols + lane;
                    const int u = kc >> 8, kk = kc & 255;
                    const float sum = warp_sum(v[i]);
                    float* xm = xp + (size_t)m * xs;
                    if (Q4K) {
                        const int slot = q4k_xslot(kk);
                        xm[((slot >> 2) * U + u) * 4 + (slot & 3)] = v[i] * q4k_xscale(kk);
                        if (lane == 0) sums[m * nsub + (kk >> 5) * U + u] = sum;
                    } else {
                        const int pos = 34 * (kk >> 5) + 2 + (kk & 31);   // byte position in the period
                        xm[((pos >> 2) * U + u) * 4 + (pos & 3)] = v[i] * q8_xscale(pos);
                        if (lane == 0) sums[m * nsub + (kk >> 5) * U + u] = 128.0f * sum;
                    }
                }
            }
        }
        if (tid < 2 * W) cut_row[tid] = -1;
        __syncthreads();

        // ---- this warp's SBs
        int ws, we;
        warp_range(sd, blockIdx.x, gridDim.x, warp, W, ws, we);
        int g_open = -1;          // row continued from the previous tile (warp-uniform)
        float acc_open[MMAX];
#pragma unroll
        for (int m = 0; m < MMAX; ++m) acc_open[m] = 0.0f;
        for (int a = ws; a < we; a += kLanes) {
            const int b = min(a + kLanes, we);
            const int slot = consumed % D;
            wait_full(&full[slot], (uint32_t)(consumed / D) & 1u, p.status);
            const int S = a + lane;
            const bool valid = S < b;
            const int g = valid ? S / U : -1;   // row in the stage's numbering
            const int u = valid ? S - g * U : 0;
            float v[MMAX];
#pragma unroll
            for (int m = 0; m < MMAX; ++m) v[m] = 0.0f;
            if (valid) {
                const uint8_t* blk = ring + (size_t)slot * B::kTile + lane * B::kBytes;
                if constexpr (Q4K) {
                    float r1[1][MMAX];
#pragma unroll
                    for (int m = 0; m < MMAX; ++m) r1[0][m] = 0.0f;
                    q4k_tile_rows<MMAX, 1>(blk, 0, xp + 4 * u, xs, sums + u, nsub, r1, 4 * U, U);
#pragma unroll
                    for (int m = 0; m < MMAX; ++m) v[m] = r1[0][m];
                } else {
                    q8_tile_row<MMAX>(blk, xp + 4 * u, xs, sums + u, nsub, v, 4 * U, U);
                }
            }
            __syncwarp();   // every lane is done with the buffer
            ++consumed;
            refill();

            // segmented sum over lanes of the same row: afterwards the first lane
            // of each row's run holds the run's total
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int go = __shfl_down_sync(0xffffffffu, g, off);
#pragma unroll
                for (int m = 0; m < MMAX; ++m) {
                    const float t = __shfl_down_sync(0xffffffffu, v[m], off);
                    if (lane + off < 32 && go == g) v[m] += t;
                }
            }
            const int gp = __shfl_up_sync(0xffffffffu, g, 1);
            const bool head = valid && (lane == 0 || gp != g);
            if (head && g == g_open) {
#pragma unroll
                for (int m = 0; m < MMAX; ++m) v[m] += acc_open[m];
            }
            const bool ends = (g + 1) * U <= b;   // the row's last SB is in this tile
            const bool started = g * U >= ws;      // the row's first SB is in this warp's range
            // the tile's last run may continue into the next tile of this warp
            const unsigned heads = __ballot_sync(0xffffffffu, head);
            const int last = 31 - __clz(heads);
            const bool cont = head && lane == last && !ends && b < we;
            if (head && !cont) {
                if (ends && started) {
                    const int sg = seg_of_row(sd, g);
                    const int r = g - sd->row0[sg], rows = sd->rows[sg];
                    float* ys = sd->y[sg];
#pragma unroll
                    for (int m = 0; m < MMAX; ++m)
                        if (m < p.M) ys[(int64_t)m * rows + r] = v[m];
                } else {
                    // cut by the warp range: part of a row that started before it
                    // (slot 0) or that goes on past it (slot 1)
                    const int k = started ? 1 : 0;
#pragma unroll
                    for (int m = 0; m < MMAX; ++m) cut_val[(k * W + warp) * MMAX + m] = v[m];
                    cut_row[k * W + warp] = g;
                }
            }
            const bool any_cont = __shfl_sync(0xffffffffu, cont, last);
            g_open = any_cont ? __shfl_sync(0xffffffffu, g, last) : -1;
#pragma unroll
            for (int m = 0; m < MMAX; ++m) acc_open[m] = __shfl_sync(0xffffffffu, v[m], last);
        }
        __syncthreads();

        // ---- rows cut between warps: the warp where the row starts adds the
        // later warps' parts in order and stores it
        if (lane == 0 && cut_row[W + warp] >= 0) {
            const int g = cut_row[W + warp];
            float t[MMAX];
#pragma unroll
            for (int m = 0; m < MMAX; ++m) t[m] = cut_val[(W + warp) * MMAX + m];
            // the row goes on in the next warps that have SBs (warps with an empty
            // range are skipped) while their part of a started row is this row
            for (int w2 = warp + 1; w2 < W; ++w2) {
                int ws2, we2;
                warp_range(sd, blockIdx.x, gridDim.x, w2, W, ws2, we2);
                if (ws2 == we2) continue;
                if (cut_row[w2] != g) break;
#pragma unroll
                for (int m = 0; m < MMAX; ++m) t[m] += cut_val[w2 * MMAX + m];
            }
            const int sg = seg_of_row(sd, g);
            const int r = g - sd->row0[sg], rows = sd->rows[sg];
            float* ys = sd->y[sg];
#pragma unroll
            for (int m = 0; m < MMAX; ++m)
                if (m < p.M) ys[(int64_t)m * rows + r] = t[m];
        }

        // ---- stage s done in this CTA: publish it (the CTA barrier orders every
        // warp's stores before thread 0's release); the last CTA of the chain
        // resets the counter for the next launch
        if (p.nstages > 1) {
            __syncthreads();
            if (tid == 0) {
                if (s + 1 < p.nstages) {
                    red_release_add(p.counter, 1);
                } else if (atom_acq_rel_add(p.counter, 1) == p.nstages * (int)gridDim.x - 1) {
                    st_relaxed(p.counter, 0);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ host ----

int num_sms() {
    static int sms[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 1;
    if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    return sms[dev] > 0 ? sms[dev] : 1;
}

int mmax_of(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : 4; }

// Warps per CTA.  GGQ_STREAM_WARPS=8|12|16 overrides the default for M = 1 (a
// tuning aid; read once, so a chain keeps the layout it was created with).
int warps_of(bool q4k, int mmax) {
    static const int env = [] {
        const char* v = getenv("GGQ_STREAM_WARPS");
        const int w = v ? atoi(v) : 0;
        return (w == 8 || w == 12 || w == 16) ? w : 0;
    }();
    if (env && mmax == 1) return env;
    if (!q4k) return 8;
    return mmax == 4 ? 8 : 16;
}

size_t rows_smem(bool q4k, int mmax, int ring, int64_t cols_max) {
    const int W = warps_of(q4k, mmax);
    const int64_t U = cols_max / 256;
    const size_t tile = (size_t)kLanes * (q4k ? 144 : 272);
    const size_t xs = (size_t)(q4k ? U * 256 : U * 272);
    const size_t cut = (size_t)2 * W * mmax * 4 + (size_t)2 * W * 4;
    return (size_t)W * ring * tile + (size_t)mmax * xs * 4 + (size_t)mmax * 8 * U * 4 + cut + (size_t)W * ring * 8;
}

int rows_ring(bool q4k, int mmax, int64_t cols_max) {
    int ring = 4;
    while (ring > 1 && rows_smem(q4k, mmax, ring, cols_max) > kSmemLimit) --ring;
    return rows_smem(q4k, mmax, ring, cols_max) <= kSmemLimit ? ring : 0;
}

void make_stage(int n, const void* const* W, const int64_t* rows, int64_t cols, const float* x, float* const* y,
                StageDesc* sd) {
    memset(sd, 0, sizeof(*sd));
    int r = 0;
    for (int s = 0; s < n; ++s) {
        sd->W[s] = static_cast<const uint8_t*>(W[s]);
        sd->y[s] = y[s];
        sd->rows[s] = (int)rows[s];
        sd->row0[s] = r;
        r += (int)rows[s];
    }
    sd->row0[n] = r;
    sd->nseg = n;
    sd->x = x;
    sd->cols = (int)cols;
    sd->units = (int)(cols / 256);
}

template <bool Q4K, int MMAX, int W>
int launch_t(const StageDesc& inl, const ChainParams& p, cudaStream_t stream, size_t smem, bool cooperative) {
    auto kernel = rows_kernel<Q4K, MMAX, W>;
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
    cfg.gridDim = dim3((unsigned)num_sms());
    cfg.blockDim = dim3(32 * W);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1].id = cudaLaunchAttributeCooperative;   // stage boundaries need every CTA resident
    attrs[1].val.cooperative = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = cooperative ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kernel, inl, p);
    if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
    return GGQ_OK;
}

// Launch the kernel: `table` (device) holds nstages stages, or is null and
// `inl` is the only stage.
int launch_rows(int type, int M, const StageDesc& inl, const StageDesc* table, int nstages, int64_t cols_max,
                int* counter, cudaStream_t stream) {
    const bool q4k = type == GGQ_Q4_K;
    const int mmax = mmax_of(M);
    const int W = warps_of(q4k, mmax);
    ChainParams p = {};
    p.table = table;
    p.nstages = nstages;
    p.M = M;
    p.ring = rows_ring(q4k, mmax, cols_max);
    if (p.ring == 0) return fail(GGQ_EINVAL, "shape needs too much shared memory");
    p.xs = (int)(q4k ? cols_max : cols_max / 256 * 272);
    p.nsub = (int)(cols_max / 32);
    p.counter = counter;
    p.status = device_status_word();
    if (!p.status) return fail(GGQ_ECUDA, "device status word unavailable");
    const size_t smem = rows_smem(q4k, mmax, p.ring, cols_max);
    const bool coop = nstages > 1;
    if (q4k) {
        if (mmax == 1) {
            if (W == 8) return launch_t<true, 1, 8>(inl, p, stream, smem, coop);
            if (W == 12) return launch_t<true, 1, 12>(inl, p, stream, smem, coop);
            return launch_t<true, 1, 16>(inl, p, stream, smem, coop);
        }
        if (mmax == 2) return launch_t<true, 2, 16>(inl, p, stream, smem, coop);
        return launch_t<true, 4, 8>(inl, p, stream, smem, coop);
    }
    if (mmax == 1) {
        if (W == 12) return launch_t<false, 1, 12>(inl, p, stream, smem, coop);
        if (W == 16) return launch_t<false, 1, 16>(inl, p, stream, smem, coop);
        return launch_t<false, 1, 8>(inl, p, stream, smem, coop);
    }
    if (mmax == 2) return launch_t<false, 2, 8>(inl, p, stream, smem, coop);
    return launch_t<false, 4, 8>(inl, p, stream, smem, coop);
}

}  // namespace

bool stream_gemv_supported(int type, int64_t cols, int M, int nseg, const int64_t* rows) {
    if (M > kMaxM || nseg < 1 || nseg > kMaxSeg || cols % 256 || cols > (1 << 20)) return false;
    int64_t r = 0;
    for (int s = 0; s < nseg; ++s) r += rows[s];
    if (r * (cols / 256) >= (1ll << 31)) return false;   // SB indices are 32-bit
    return rows_ring(type == GGQ_Q4_K, mmax_of(M), cols) > 0;
}

int launch_gemv_stream(int type, int nseg, const void* const* W, const int64_t* rows, int64_t cols, const float* x,
                       float* const* y, int M, cudaStream_t stream) {
    StageDesc sd;
    make_stage(nseg, W, rows, cols, x, y, &sd);
    return launch_rows(type, M, sd, nullptr, 1, cols, nullptr, stream);
}

}  // namespace ggq

// ------------------------------------------------------------ chain ABI ----

using namespace ggq;

struct ggq_chain {
    int type = 0;
    int M = 0;
    int nstages = 0;
    int64_t cols_max = 0;
    int device = -1;
    StageDesc* table = nullptr;   // device memory
    int* counter = nullptr;       // device memory, zero between runs
};

extern "C" int ggq_chain_create(int type, int M, int nstages, const ggq_chain_stage* stages, ggq_chain** out) {
    clear_error();
    if (!out) return fail(GGQ_EINVAL, "ggq_chain_create: out is NULL");
    *out = nullptr;
    if (type != GGQ_Q8_0 && type != GGQ_Q4_K) return fail(GGQ_ETYPE, "ggq_chain_create: type %d not supported", type);
    if (M < 1 || M > kMaxM) return fail(GGQ_EINVAL, "ggq_chain_create: M %d outside 1..%d", M, kMaxM);
    if (nstages < 1 || nstages > 65536 || !stages) return fail(GGQ_EINVAL, "ggq_chain_create: bad stage list");
    std::vector<StageDesc> host((size_t)nstages);
    int64_t cols_max = 0;
    for (int s = 0; s < nstages; ++s) {
        const ggq_chain_stage& st = stages[s];
        if (st.n < 1 || st.n > kMaxSeg || !st.x) return fail(GGQ_EINVAL, "ggq_chain_create: stage %d malformed", s);
        if ((reinterpret_cast<uintptr_t>(st.x) & 15) != 0)
            return fail(GGQ_EINVAL, "ggq_chain_create: stage %d x not 16-byte aligned", s);
        for (int i = 0; i < st.n; ++i) {
            if (!st.W[i] || !st.y[i] || st.rows[i] < 1 || st.rows[i] > 0x7fffffff)
                return fail(GGQ_EINVAL, "ggq_chain_create: stage %d matrix %d malformed", s, i);
            if ((reinterpret_cast<uintptr_t>(st.W[i]) & 15) != 0 || (reinterpret_cast<uintptr_t>(st.y[i]) & 3) != 0)
                return fail(GGQ_EINVAL, "ggq_chain_create: stage %d matrix %d misaligned", s, i);
        }
        if (!stream_gemv_supported(type, st.cols, M, st.n, st.rows))
            return fail(GGQ_EINVAL, "ggq_chain_create: stage %d shape unsupported (cols %% 256, size)", s);
        cols_max = std::max<int64_t>(cols_max, st.cols);
    }
    if (rows_ring(type == GGQ_Q4_K, mmax_of(M), cols_max) == 0)
        return fail(GGQ_EINVAL, "ggq_chain_create: widest stage needs too much shared memory");
    for (int s = 0; s < nstages; ++s) {   // all stages valid: encode them
        const ggq_chain_stage& st = stages[s];
        make_stage(st.n, st.W, st.rows, st.cols, st.x, st.y, &host[(size_t)s]);
    }
    ggq_chain* c = new (std::nothrow) ggq_chain();
    if (!c) return fail(GGQ_ENOMEM, "host allocation failed");
    cudaGetDevice(&c->device);
    cudaError_t e = cudaMalloc(&c->table, sizeof(StageDesc) * (size_t)nstages);
    if (e == cudaSuccess) e = cudaMalloc(&c->counter, sizeof(int));
    if (e == cudaSuccess)
        e = cudaMemcpy(c->table, host.data(), sizeof(StageDesc) * (size_t)nstages, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(c->counter, 0, sizeof(int));
    if (e != cudaSuccess) {
        if (c->table) cudaFree(c->table);
        if (c->counter) cudaFree(c->counter);
        delete c;
        return cuda_fail(e, "ggq_chain_create: device state");
    }
    c->type = type;
    c->M = M;
    c->nstages = nstages;
    c->cols_max = cols_max;
    *out = c;
    return GGQ_OK;
}

extern "C" int ggq_chain_run(const ggq_chain* c, void* stream) {
    clear_error();
    if (!c) return fail(GGQ_EINVAL, "ggq_chain_run: NULL chain");
    StageDesc none;
    memset(&none, 0, sizeof(none));
    return launch_rows(c->type, c->M, none, c->table, c->nstages, c->cols_max, c->counter,
                       static_cast<cudaStream_t>(stream));
}

extern "C" int ggq_chain_reset(ggq_chain* c) {
    clear_error();
    if (!c) return fail(GGQ_EINVAL, "ggq_chain_reset: NULL chain");
    cudaError_t e = cudaMemset(c->counter, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "ggq_chain_reset");
    return GGQ_OK;
}

extern "C" void ggq_chain_free(ggq_chain* c) {
    if (!c) return;
    if (c->table) cudaFree(c->table);
    if (c->counter) cudaFree(c->counter);
    delete c;
}
