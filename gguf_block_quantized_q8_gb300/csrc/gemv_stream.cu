// Persistent stream-K GEMV over a chain of dependent stages.
//
// A stage is up to four weight matrices of one type and width that share their
// input x (e.g. the q, k and v projections of a layer): y_i = W_i x.  A chain is
// a list of stages run in order; stage s+1 reads its x only after every output
// of stage s is written, so the x of a later stage may be the y of an earlier
// one.  A single GEMV is a chain of one stage.
//
// Work of a stage is a flat sequence of tiles t = (row block, unit): 32*R rows
// (lane l owns rows l, l+32, ...) by one unit of columns -- a Q4_K super-block
// column (144 B per row) or an 8-block Q8_0 period (272 B per row).  The
// sequence is cut into equal contiguous runs, one per warp group, so every SM
// streams the same number of bytes whatever the shapes.
//
// CTA layout (one CTA per SM, all CTAs resident: cooperative launch):
//   * W compute warps in groups of G.  With G = 4 (Q4_K) warp w of a group
//     decodes chunk w (64 columns) of every tile of its group's run; with G = 1
//     a warp takes whole tiles.
//   * one producer warp whose lane 0 keeps every group's ring of tile buffers
//     full with 2-D bulk tensor copies, stage after stage: weights never depend
//     on earlier stages, so the next stage's first tiles are already in shared
//     memory while the chain waits at a stage boundary.
//   * x' (the pre-scaled activations, see gemv_tile.cuh) for all columns of the
//     current stage, built once per CTA in shared memory.
//
// Row blocks cut by a run boundary are finished by the last group to reach
// them: contributors write partial sums to a workspace, bump a per-row-block
// counter, and the group that brings it to the number of contributors adds
// the partials in group order (deterministic), stores y and resets the counter.
// A stage is complete when every CTA has added one to the stage counter (with
// release semantics, after all its groups are done); CTAs wait for that count
// (acquire) before reading the next stage's x.  The last CTA of the chain
// resets the counter, so the workspace is back at zero for the next launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "gemv_tile.cuh"
#include "ggq_internal.h"
#include "ptx.cuh"

namespace ggq {

namespace {

constexpr int kRows = 32;
// counters[0] is the stage counter; the row-block counters start a 128-byte
// line later, so polling the stage counter does not slow the row-block atomics
constexpr int kRbCounter0 = 32;
constexpr int kMaxSeg = 4;
constexpr int kMaxM = 4;
constexpr size_t kSmemLimit = 227 * 1024;

// One stage of a chain (device-visible: kernel parameter or global table).
struct StageDesc {
    CUtensorMap maps[kMaxSeg];
    const float* x;            // [M][cols]
    float* y[kMaxSeg];         // [M][rows]
    int rows[kMaxSeg];
    int rb0[kMaxSeg + 1];      // first row block of each matrix; rb0[nseg] = row blocks of the stage
    int nseg;
    int cols;
    int units;                 // units per row
    int ngroups;               // groups with a run in this stage (<= groups of the grid)
    int rem;                   // tiles % ngroups: the first `rem` runs are one tile longer
    long long tiles;           // row blocks * units
    long long quot;            // tiles / ngroups
};

struct ChainParams {
    const StageDesc* table;    // the stages in device memory, or null: the inline stage only
    int nstages;
    int M;
    int ring;                  // tile buffers per group
    int xs;                    // x' floats per activation row (largest stage)
    int nsub;                  // x sums per activation row (largest stage)
    float* partials;           // [groups][2][kMaxM][32]
    int* counters;             // [0]: stage counter; [kRbCounter0 + rb]: row-block counters; zero between launches
    int* status;
};

template <bool Q4K, int R>
struct Unit {
    static constexpr int kRowBytes = Q4K ? 144 : 272;
    static constexpr int kTileRows = kRows * R;
    static constexpr int kTile = kTileRows * kRowBytes;
    static constexpr int kXp = Q4K ? 256 : 272;     // x' floats per unit (per activation row)
    static constexpr int kMapX = Q4K ? 144 : 136;   // map elements per unit (1 or 2 bytes each)
};

// Runs: group g of a stage takes tiles [run_start(g), run_start(g + 1)); the
// first `rem` groups take quot + 1 tiles, the others quot (quot >= 1).
__device__ __forceinline__ long long run_start(const StageDesc* sd, long long g) {
    return g * sd->quot + (g < sd->rem ? g : sd->rem);
}
// the group whose run contains tile t
__device__ __forceinline__ long long group_of(const StageDesc* sd, long long t) {
    const long long big = (long long)sd->rem * (sd->quot + 1);
    return t < big ? t / (sd->quot + 1) : sd->rem + (t - big) / sd->quot;
}

__device__ __forceinline__ int seg_of(const StageDesc* sd, int gr) {
    int s = 0;
#pragma unroll
    for (int i = 1; i < kMaxSeg; ++i)
        if (i < sd->nseg && gr >= sd->rb0[i]) s = i;
    return s;
}

__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

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

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Waits of the chain kernel are bounded (kWaitLimitNs), and once any wait of
// any CTA has run out (the status word is set) the others shorten theirs to
// kDrainNs: the kernel then only drains its own copies in flight and ends,
// instead of timing out once per remaining tile.
constexpr unsigned long long kDrainNs = 1000000ull;   // 1 ms

// Wait until *counter >= target (other CTAs' groups finishing a stage).
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

template <bool Q4K, int MMAX, int R, int W, int G>
__global__ void __launch_bounds__(32 * (W + 1), 1) chain_kernel(const __grid_constant__ StageDesc inl,
                                                                 const ChainParams p) {
    static_assert(R * MMAX <= kMaxM, "partials slot too small");
    static_assert(Q4K || G == 1, "Q8_0 tiles are taken whole");
    constexpr int NG = W / G;
    constexpr int kCompute = 32 * W;
    using U = Unit<Q4K, R>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // shared memory: [group rings][x'][sums][row-block partials][barriers]
    uint8_t* rings = smem;
    float* xp = reinterpret_cast<float*>(smem + (size_t)NG * p.ring * U::kTile);
    float* sums = xp + (size_t)MMAX * p.xs;
    float* red = sums + (size_t)MMAX * p.nsub;      // [NG][2][G][R*MMAX][32] when G > 1
    uint64_t* full = reinterpret_cast<uint64_t*>(red + (G > 1 ? NG * 2 * G * R * MMAX * 32 : 0));
    uint64_t* empty = full + NG * p.ring;

    if (tid == 0) {
        for (int i = 0; i < NG * p.ring; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], G);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    // ------------------------------------------------------------- producer
    if (warp == W) {
        if (lane != 0) return;
        struct Cursor {
            int s;            // stage
            long long t, end; // next tile of the run, run end
            int gr, u;        // (row block, unit) of tile t
            int slot, wraps;  // next buffer; times the ring has wrapped
            int issued;
        };
        Cursor c[NG];
        for (int gi = 0; gi < NG; ++gi) c[gi] = Cursor{-1, 0, 0, 0, 0, 0, 0, 0};
        if (!p.table)
            for (int s = 0; s < inl.nseg; ++s) prefetch_tensormap(&inl.maps[s]);
        int finished = 0;
        unsigned long long idle_since = 0;
        unsigned spins = 0;
        while (finished < NG) {
            bool progress = false;
            for (int gi = 0; gi < NG; ++gi) {
                Cursor& q = c[gi];
                if (q.s >= p.nstages) continue;
                while (q.t == q.end) {   // move on to the next stage in which this group has tiles
                    if (++q.s >= p.nstages) { ++finished; break; }
                    const StageDesc* sd = p.table ? p.table + q.s : &inl;
                    const long long gg = (long long)gi * gridDim.x + blockIdx.x;
                    if (gg < sd->ngroups) {
                        q.t = run_start(sd, gg);
                        q.end = run_start(sd, gg + 1);
                        q.gr = (int)(q.t / sd->units);
                        q.u = (int)(q.t - (long long)q.gr * sd->units);
                    } else {
                        q.t = q.end = 0;
                    }
                }
                if (q.s >= p.nstages) continue;
                const int b = gi * p.ring + q.slot;
                if (q.issued >= p.ring && !mbar_try_wait(&empty[b], (uint32_t)(q.wraps - 1) & 1u)) continue;
                const StageDesc* sd = p.table ? p.table + q.s : &inl;
                const int seg = seg_of(sd, q.gr);
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&full[b], U::kTile);
                tma_load_2d(rings + (size_t)b * U::kTile, &sd->maps[seg], &full[b], q.u * U::kMapX,
                            (q.gr - sd->rb0[seg]) * U::kTileRows);
                ++q.t;
                if (++q.u == sd->units) { q.u = 0; ++q.gr; }
                ++q.issued;
                if (++q.slot == p.ring) { q.slot = 0; ++q.wraps; }
                progress = true;
            }
            // idle: every ring full.  Consumers may sit at a stage boundary for up to
            // kWaitLimitNs, so give up only after twice that (or soon after another
            // wait has run out)
            if (progress) {
                idle_since = 0;
            } else if ((++spins & 255u) == 0) {
                const unsigned long long now = globaltimer_ns();
                if (idle_since == 0) {
                    idle_since = now;
                } else if (now - idle_since > 2 * kWaitLimitNs ||
                           (now - idle_since > kDrainNs && ld_relaxed(p.status) != 0)) {
                    atomicOr(p.status, kStatusTimeout);
                    return;
                }
            }
        }
        return;
    }

    // -------------------------------------------------------- compute warps
    const int grp = warp / G, wig = warp % G;
    const long long gg = (long long)grp * gridDim.x + blockIdx.x;
    int slot = 0;
    uint32_t parity = 0;   // phase of buffer `slot` for the group's next tile
    int nflush = 0;
    uint8_t* ring = rings + (size_t)grp * p.ring * U::kTile;

    for (int s = 0; s < p.nstages; ++s) {
        const StageDesc* sd = p.table ? p.table + s : &inl;
        if (s == 0) {
            pdl_wait();   // x may come from the previous kernel in the stream
        } else {
            // every CTA has finished stage s-1 (its outputs are visible)
            if (tid == 0) wait_count(p.counters, s * (int)gridDim.x, p.status);
            named_sync(1, kCompute);
        }
        const int cols = sd->cols, units = sd->units;
        const int xs = p.xs;

        // x' of this stage.  x may have been written by other CTAs: it is read
        // from L2 (cp.async.cg / ld.cg), after the stage barrier's acquire.
        if (Q4K) {
            // raw x into the x' area, then per 32-column sub-block: its sum, and
            // the values scaled and permuted in place (8 lanes a sub-block)
            const int c4 = cols / 4;
            for (int i = tid; i < p.M * c4; i += kCompute) {
                const int m = i / c4, k4 = i - m * c4;
                cp_async16(xp + (size_t)m * xs + 4 * k4, sd->x + (int64_t)m * cols + 4 * k4);
            }
            cp_async_wait_all();
            named_sync(1, kCompute);
            const int nsbr = cols / 32, nsbk = p.M * nsbr;
            const int a = lane & 7;
            for (int base = warp * 4; base < nsbk; base += W * 4) {
                const int j = base + (lane >> 3);
                const bool valid = j < nsbk;
                const int m = valid ? j / nsbr : 0, sb = valid ? j - m * nsbr : 0;
                float* blk = xp + (size_t)m * xs + (size_t)sb * 32;
                float4 v = valid ? *reinterpret_cast<const float4*>(blk + 4 * a) : make_float4(0.f, 0.f, 0.f, 0.f);
                float sum = (v.x + v.y) + (v.z + v.w);
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                sum += __shfl_xor_sync(0xffffffffu, sum, 4);
                __syncwarp();   // the 8 lanes of a sub-block have read it before any writes
                if (valid) {
                    const int k0 = (sb & 7) * 32 + 4 * a;   // position in the super-block
                    blk[a] = v.x * q4k_xscale(k0);
                    blk[8 + a] = v.y * q4k_xscale(k0 + 1);
                    blk[16 + a] = v.z * q4k_xscale(k0 + 2);
                    blk[24 + a] = v.w * q4k_xscale(k0 + 3);
                    if (a == 0) sums[m * p.nsub + sb] = sum;
                }
            }
        } else {
            // each x goes to the byte position B = 34b + 2 + i of its weight in
            // the 272-byte period; 128 * sum(x) per block
            for (int job = warp; job < p.M * units; job += W) {
                const int m = job / units, u = job - m * units;
                const float* src = sd->x + (int64_t)m * cols + (int64_t)u * 256;
                float* reg = xp + (size_t)m * xs + (size_t)u * U::kXp;
                float v[8];
#pragma unroll
                for (int b = 0; b < 8; ++b) v[b] = __ldcg(src + 32 * b + lane);
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    const int B = 34 * b + 2 + lane;
                    reg[B] = v[b] * q8_xscale(B);
                }
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    const float sum = warp_sum(v[b]);
                    if (lane == 0) sums[m * p.nsub + u * 8 + b] = 128.0f * sum;
                }
            }
        }
        named_sync(1, kCompute);

        if (gg < sd->ngroups) {
            const long long t0 = run_start(sd, gg), t1 = run_start(sd, gg + 1);
            const int n = (int)(t1 - t0);
            float acc[R][MMAX];     // the current row block
            float first[R][MMAX];   // the run's first row block when the run entered it mid-way
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < MMAX; ++m) acc[r][m] = first[r][m] = 0.0f;
            const int gr_first = (int)(t0 < 0x7fffffffll ? (int)((uint32_t)t0 / (uint32_t)units) : t0 / units);
            int gr = gr_first;
            int u = (int)(t0 - (long long)gr * units);
            bool covered_from_start = u == 0;
            bool have_first = false;

            // sum of the group's warps (G > 1): returns true in the warp that holds it
            auto group_sum = [&](float (&v)[R][MMAX]) -> bool {
                if constexpr (G > 1) {
                    float* mine = red + ((size_t)((grp * 2 + (nflush & 1)) * G + wig) * R * MMAX) * 32;
#pragma unroll
                    for (int r = 0; r < R; ++r)
#pragma unroll
                        for (int m = 0; m < MMAX; ++m) mine[(r * MMAX + m) * 32 + lane] = v[r][m];
                    named_sync(2 + grp, 32 * G);
                    const float* all = red + ((size_t)(grp * 2 + (nflush & 1)) * G * R * MMAX) * 32;
                    ++nflush;
                    if (wig != 0) return false;
#pragma unroll
                    for (int r = 0; r < R; ++r)
#pragma unroll
                        for (int m = 0; m < MMAX; ++m) {
                            float t = all[(r * MMAX + m) * 32 + lane];
#pragma unroll
                            for (int w = 1; w < G; ++w) t += all[((size_t)w * R * MMAX + r * MMAX + m) * 32 + lane];
                            v[r][m] = t;
                        }
                }
                return true;
            };
            auto store_y = [&](int cur, const float (&v)[R][MMAX]) {
                const int sg = seg_of(sd, cur);
                const int row0 = (cur - sd->rb0[sg]) * U::kTileRows + lane;
                const int rows = sd->rows[sg];
                float* ys = sd->y[sg];
#pragma unroll
                for (int r = 0; r < R; ++r)
                    if (row0 + 32 * r < rows)
#pragma unroll
                        for (int m = 0; m < MMAX; ++m)
                            if (m < p.M) ys[(int64_t)m * rows + row0 + 32 * r] = v[r][m];
            };
            auto deposit = [&](int pslot, const float (&v)[R][MMAX]) {
                float* part = p.partials + ((gg * 2 + pslot) * kMaxM) * 32;
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int m = 0; m < MMAX; ++m) part[(r * MMAX + m) * 32 + lane] = v[r][m];
            };
            // contributors of row block `cur`: groups lo..hi
            auto contributors = [&](int cur, long long& lo, long long& hi) {
                lo = group_of(sd, (long long)cur * units);
                hi = group_of(sd, (long long)(cur + 1) * units - 1);
            };
            // the last contributor: add every contributor's partial in group order
            // (deterministic), store y, reset the row block's counter
            auto finish = [&](int cur, long long lo, long long hi) {
                // only the first contributor can have started its run before this row block
                const bool lo_starts_before = run_start(sd, lo) < (long long)cur * units;
                float v[R][MMAX];
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int m = 0; m < MMAX; ++m) v[r][m] = 0.0f;
                for (long long c0 = lo; c0 <= hi; c0 += 8) {
                    float q[8][R * MMAX];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const long long c = c0 + j;
                        if (c <= hi) {
                            const int cs = (c == lo && lo_starts_before) ? 1 : 0;
                            const float* src = p.partials + ((c * 2 + cs) * kMaxM) * 32 + lane;
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
                store_y(cur, v);
                if (lane == 0) st_relaxed(&p.counters[kRbCounter0 + cur], 0);
            };

            for (int i = 0; i < n; ++i) {
                if (i > 0 && u == 0) {
                    // the run passed the end of row block gr - 1
                    if (covered_from_start) {
                        if (group_sum(acc)) store_y(gr - 1, acc);
                    } else {
                        // entered mid-way: its fixup waits for the end of the run, so
                        // no round trip stalls the tile loop
#pragma unroll
                        for (int r = 0; r < R; ++r)
#pragma unroll
                            for (int m = 0; m < MMAX; ++m) first[r][m] = acc[r][m];
                        have_first = true;
                    }
                    covered_from_start = true;
#pragma unroll
                    for (int r = 0; r < R; ++r)
#pragma unroll
                        for (int m = 0; m < MMAX; ++m) acc[r][m] = 0.0f;
                }
                wait_full(&full[grp * p.ring + slot], parity, p.status);
                const uint8_t* rp = ring + (size_t)slot * U::kTile + lane * U::kRowBytes;
                if constexpr (Q4K) {
                    if constexpr (G == 4)
                        q4k_chunk_rows<MMAX, R>(rp, 32 * U::kRowBytes, wig, xp + (size_t)u * 256, xs, sums + u * 8,
                                                p.nsub, acc);
                    else
                        q4k_tile_rows<MMAX, R>(rp, 32 * U::kRowBytes, xp + (size_t)u * 256, xs, sums + u * 8, p.nsub,
                                               acc);
                } else {
                    q8_tile_row<MMAX>(rp, xp + (size_t)u * U::kXp, xs, sums + u * 8, p.nsub, acc[0]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[grp * p.ring + slot]);   // buffer free for the producer
                if (++u == units) { u = 0; ++gr; }
                if (++slot == p.ring) { slot = 0; parity ^= 1u; }
            }

            // the run's last row block, and the deferred first one
            const int last = u == 0 ? gr - 1 : gr;
            const bool last_whole = u == 0 && covered_from_start;
            bool mine = true;
            if (have_first) mine = group_sum(first);
            mine = group_sum(acc) && mine;
            if (mine) {
                if (last_whole) store_y(last, acc);
                else deposit(last == gr_first ? 0 : 1, acc);
                if (have_first) deposit(0, first);
                if (have_first || !last_whole) {
                    // one acq_rel add per split row block publishes this warp's partials
                    // (ordered by the warp barrier) and, for the last contributor, makes
                    // the others' visible
                    __syncwarp();
                    int prev_first = -1, prev_last = -1;
                    if (lane == 0) {
                        if (have_first) prev_first = atom_acq_rel_add(&p.counters[kRbCounter0 + gr_first], 1);
                        if (!last_whole) prev_last = atom_acq_rel_add(&p.counters[kRbCounter0 + last], 1);
                    }
                    long long lo_f = 0, hi_f = 0, lo_l = 0, hi_l = 0;
                    if (have_first) contributors(gr_first, lo_f, hi_f);
                    if (!last_whole) contributors(last, lo_l, hi_l);
                    prev_first = __shfl_sync(0xffffffffu, prev_first, 0);
                    prev_last = __shfl_sync(0xffffffffu, prev_last, 0);
                    __syncwarp();
                    if (have_first && prev_first == (int)(hi_f - lo_f)) finish(gr_first, lo_f, hi_f);
                    if (!last_whole && prev_last == (int)(hi_l - lo_l)) finish(last, lo_l, hi_l);
                }
            }
        }

        // stage s done in this CTA: publish it (the CTA barrier orders every
        // warp's stores before thread 0's release); the last CTA to finish the
        // chain resets the counter for the next launch
        if (p.nstages > 1) {
            named_sync(1, kCompute);
            if (tid == 0) {
                if (s + 1 < p.nstages) {
                    red_release_add(p.counters, 1);
                } else if (atom_acq_rel_add(p.counters, 1) == p.nstages * (int)gridDim.x - 1) {
                    st_relaxed(p.counters, 0);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ host ----

struct Workspace {
    float* partials = nullptr;
    int* counters = nullptr;
    int max_groups = 0;
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
// (and grown if a later call needs more).
int get_workspace(cudaStream_t stream, int groups, int rb, Workspace** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace& ws = g_ws[{dev, stream}];
    if (ws.max_groups < groups) {
        if (ws.partials) cudaFree(ws.partials);
        ws.partials = nullptr;
        const int want = std::max(groups, 152 * 16);
        e = cudaMalloc(&ws.partials, (size_t)want * 2 * kMaxM * 32 * sizeof(float));
        if (e != cudaSuccess) { ws.max_groups = 0; return cuda_fail(e, "workspace allocation"); }
        ws.max_groups = want;
    }
    if (ws.max_rb < rb) {
        if (ws.counters) cudaFree(ws.counters);
        ws.counters = nullptr;
        const int want = std::max(rb, 1 << 17);
        e = cudaMalloc(&ws.counters, (size_t)(want + kRbCounter0) * sizeof(int));
        if (e != cudaSuccess) { ws.max_rb = 0; return cuda_fail(e, "workspace allocation"); }
        e = cudaMemsetAsync(ws.counters, 0, (size_t)(want + kRbCounter0) * sizeof(int), stream);
        if (e != cudaSuccess) return cuda_fail(e, "workspace clear");
        ws.max_rb = want;
    }
    *out = &ws;
    return GGQ_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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
    return fn;
}

int encode_map(CUtensorMap* map, const void* W, int64_t rows, int64_t row_bytes, bool q4k, int box_rows) {
    auto fn = tensor_map_encoder();
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

// Launch shape: compute warps per CTA, warps per tile group, rows per lane.
// GGQ_STREAM_SHAPE="warps,group,rows" overrides the default (a tuning aid).
struct Shape {
    int warps;
    int group;
    int rows;
};

int mmax_of(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : 4; }

// Register budget: registers are split between the four SM sub-partitions, so
// a CTA of 4k+1 warps gets the budget of 4k+4 warps; 12 compute warps plus the
// producer keep 128 registers per thread, 16 plus the producer only 96 (M = 4
// needs more than 128: 8 compute warps).
Shape stream_shape(bool q4k, int mmax) {
    Shape sh = q4k ? (mmax == 1 ? Shape{12, 4, 2} : mmax == 2 ? Shape{12, 4, 1} : Shape{8, 4, 1}) : Shape{8, 1, 1};
    static const Shape env = [] {   // read once: a chain's tiles are laid out with the shape of its creation
        Shape e = {0, 0, 0};
        if (const char* v = getenv("GGQ_STREAM_SHAPE")) {
            if (sscanf(v, "%d,%d,%d", &e.warps, &e.group, &e.rows) != 3) e = {0, 0, 0};
        }
        return e;
    }();
    const bool ok = q4k ? mmax == 1 && env.group == 4 && (env.warps == 12 || env.warps == 16) &&
                              (env.rows == 1 || env.rows == 2)
                        : mmax == 1 && env.group == 1 && env.warps == 8 && env.rows == 1;
    if (ok) sh = env;
    return sh;
}

size_t chain_smem(bool q4k, int mmax, int ring, int64_t cols_max) {
    const Shape sh = stream_shape(q4k, mmax);
    const int ng = sh.warps / sh.group;
    const int tile = kRows * sh.rows * (q4k ? 144 : 272);
    const int64_t xs = q4k ? cols_max : cols_max / 256 * 272;
    const size_t red = sh.group > 1 ? (size_t)ng * 2 * sh.group * sh.rows * mmax * 32 * 4 : 0;
    return (size_t)ng * ring * tile + (size_t)mmax * xs * 4 + (size_t)mmax * (cols_max / 32) * 4 + red +
           (size_t)(2 * ng * ring) * 8;
}

int chain_ring(bool q4k, int mmax, int64_t cols_max) {
    int ring = 8;
    while (ring > 1 && chain_smem(q4k, mmax, ring, cols_max) > kSmemLimit) --ring;
    return chain_smem(q4k, mmax, ring, cols_max) <= kSmemLimit ? ring : 0;
}

int groups_in_grid(bool q4k, int mmax) {
    const Shape sh = stream_shape(q4k, mmax);
    return num_sms() * (sh.warps / sh.group);
}

// Fill one stage descriptor (tensor maps, row blocks, tiles, groups with work).
int make_stage(int type, int M, int n, const void* const* W, const int64_t* rows, int64_t cols, const float* x,
               float* const* y, StageDesc* sd) {
    const bool q4k = type == GGQ_Q4_K;
    const int trows = kRows * stream_shape(q4k, mmax_of(M)).rows;
    const int64_t units = cols / 256;
    const int64_t row_bytes = q4k ? units * 144 : units * 272;
    memset(sd, 0, sizeof(*sd));
    int rb = 0;
    for (int s = 0; s < n; ++s) {
        int rc = encode_map(&sd->maps[s], W[s], rows[s], row_bytes, q4k, trows);
        if (rc) return rc;
        sd->y[s] = y[s];
        sd->rows[s] = (int)rows[s];
        sd->rb0[s] = rb;
        rb += (int)((rows[s] + trows - 1) / trows);
    }
    sd->rb0[n] = rb;
    sd->nseg = n;
    sd->x = x;
    sd->cols = (int)cols;
    sd->units = (int)units;
    sd->tiles = (long long)rb * units;
    sd->ngroups = (int)std::max<long long>(1, std::min<long long>(groups_in_grid(q4k, mmax_of(M)), sd->tiles));
    sd->quot = sd->tiles / sd->ngroups;
    sd->rem = (int)(sd->tiles % sd->ngroups);
    return GGQ_OK;
}

template <bool Q4K, int MMAX, int R, int W, int G>
int launch_t(const StageDesc& inl, const ChainParams& p, cudaStream_t stream, size_t smem) {
    auto kernel = chain_kernel<Q4K, MMAX, R, W, G>;
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
    cfg.blockDim = dim3(32 * (W + 1));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1].id = cudaLaunchAttributeCooperative;   // stage boundaries need every CTA resident
    attrs[1].val.cooperative = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kernel, inl, p);
    if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
    return GGQ_OK;
}

// Launch the chain kernel: `table` (device) holds nstages stages, or is null and
// `inl` is the only stage.
int launch_chain(int type, int M, const StageDesc& inl, const StageDesc* table, int nstages, int64_t cols_max,
                 float* partials, int* counters, cudaStream_t stream) {
    const bool q4k = type == GGQ_Q4_K;
    const int mmax = mmax_of(M);
    const Shape sh = stream_shape(q4k, mmax);
    ChainParams p = {};
    p.table = table;
    p.nstages = nstages;
    p.M = M;
    p.ring = chain_ring(q4k, mmax, cols_max);
    if (p.ring == 0) return fail(GGQ_EINVAL, "shape needs too much shared memory");
    p.xs = (int)(q4k ? cols_max : cols_max / 256 * 272);
    p.nsub = (int)(cols_max / 32);
    p.partials = partials;
    p.counters = counters;
    p.status = device_status_word();
    if (!p.status) return fail(GGQ_ECUDA, "device status word unavailable");
    const size_t smem = chain_smem(q4k, mmax, p.ring, cols_max);
    if (q4k) {
        if (mmax == 1) {
            if (sh.warps == 16) return sh.rows == 2 ? launch_t<true, 1, 2, 16, 4>(inl, p, stream, smem)
                                                    : launch_t<true, 1, 1, 16, 4>(inl, p, stream, smem);
            return sh.rows == 2 ? launch_t<true, 1, 2, 12, 4>(inl, p, stream, smem)
                                : launch_t<true, 1, 1, 12, 4>(inl, p, stream, smem);
        }
        if (mmax == 2) return launch_t<true, 2, 1, 12, 4>(inl, p, stream, smem);
        return launch_t<true, 4, 1, 8, 4>(inl, p, stream, smem);
    }
    if (mmax == 1) return launch_t<false, 1, 1, 8, 1>(inl, p, stream, smem);
    if (mmax == 2) return launch_t<false, 2, 1, 8, 1>(inl, p, stream, smem);
    return launch_t<false, 4, 1, 8, 1>(inl, p, stream, smem);
}

}  // namespace

// After a kernel's wait has run out, the counters of the workspaces on this
// device may be left non-zero: clear them (synchronous; called when the status
// word is read and found set).
void reset_stream_workspaces() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    for (auto& kv : g_ws)
        if (kv.first.first == dev && kv.second.counters)
            cudaMemset(kv.second.counters, 0, (size_t)(kv.second.max_rb + kRbCounter0) * sizeof(int));
}

bool stream_gemv_supported(int type, int64_t cols, int M, int nseg, const int64_t* rows) {
    if (M > kMaxM || nseg < 1 || nseg > kMaxSeg || cols % 256 || cols > (1 << 20)) return false;
    const bool q4k = type == GGQ_Q4_K;
    const int trows = kRows * stream_shape(q4k, mmax_of(M)).rows;
    int64_t rb = 0;
    for (int s = 0; s < nseg; ++s) rb += (rows[s] + trows - 1) / trows;
    if (rb > (1 << 22)) return false;
    return chain_ring(q4k, mmax_of(M), cols) > 0;
}

int launch_gemv_stream(int type, int nseg, const void* const* W, const int64_t* rows, int64_t cols, const float* x,
                       float* const* y, int M, cudaStream_t stream) {
    StageDesc sd;
    int rc = make_stage(type, M, nseg, W, rows, cols, x, y, &sd);
    if (rc) return rc;
    Workspace* ws = nullptr;
    rc = get_workspace(stream, groups_in_grid(type == GGQ_Q4_K, mmax_of(M)), sd.rb0[nseg], &ws);
    if (rc) return rc;
    return launch_chain(type, M, sd, nullptr, 1, cols, ws->partials, ws->counters, stream);
}

// Same launch with caller-provided scratch instead of the per-stream workspace:
// `partials` holds max_groups * 2 * kMaxM * 32 floats and `counters`
// 32 + max_row_blocks ints.  The counters this call uses are cleared first
// (cudaMemsetAsync on `stream`); nothing is allocated.
int launch_gemv_stream_scratch(int type, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int M,
                               cudaStream_t stream, float* partials, int max_groups, int* counters,
                               int max_row_blocks) {
    const bool q4k = type == GGQ_Q4_K;
    if (groups_in_grid(q4k, mmax_of(M)) > max_groups)
        return fail(GGQ_EINVAL, "this GPU needs more warp groups than the built-in scratch holds");
    StageDesc sd;
    int rc = make_stage(type, M, 1, &W, &rows, cols, x, &y, &sd);
    if (rc) return rc;
    const int rb = sd.rb0[1];
    if (rb > max_row_blocks)
        return fail(GGQ_EINVAL, "rows %lld exceed the %lld rows the built-in scratch can finish", (long long)rows,
                    (long long)max_row_blocks * ((rows + rb - 1) / rb));
    cudaError_t e = cudaMemsetAsync(counters, 0, (size_t)(rb + kRbCounter0) * sizeof(int), stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the scratch counters");
    return launch_chain(type, M, sd, nullptr, 1, cols, partials, counters, stream);
}

}  // namespace ggq

// ------------------------------------------------------------ chain ABI ----

using namespace ggq;

struct ggq_chain {
    int type = 0;
    int M = 0;
    int nstages = 0;
    int64_t cols_max = 0;
    int rb_max = 0;
    int device = -1;
    StageDesc* table = nullptr;   // device memory
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
    int rb_max = 0;
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
    }
    for (int s = 0; s < nstages; ++s) {   // all stages valid: encode them
        const ggq_chain_stage& st = stages[s];
        int rc = make_stage(type, M, st.n, st.W, st.rows, st.cols, st.x, st.y, &host[(size_t)s]);
        if (rc) return rc;
        cols_max = std::max<int64_t>(cols_max, st.cols);
        rb_max = std::max(rb_max, host[(size_t)s].rb0[st.n]);
    }
    if (chain_ring(type == GGQ_Q4_K, mmax_of(M), cols_max) == 0)
        return fail(GGQ_EINVAL, "ggq_chain_create: widest stage needs too much shared memory");
    ggq_chain* c = new (std::nothrow) ggq_chain();
    if (!c) return fail(GGQ_ENOMEM, "host allocation failed");
    cudaGetDevice(&c->device);
    cudaError_t e = cudaMalloc(&c->table, sizeof(StageDesc) * (size_t)nstages);
    if (e != cudaSuccess) {
        delete c;
        return cuda_fail(e, "ggq_chain_create: stage table");
    }
    e = cudaMemcpy(c->table, host.data(), sizeof(StageDesc) * (size_t)nstages, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cudaFree(c->table);
        delete c;
        return cuda_fail(e, "ggq_chain_create: stage table copy");
    }
    c->type = type;
    c->M = M;
    c->nstages = nstages;
    c->cols_max = cols_max;
    c->rb_max = rb_max;
    *out = c;
    return GGQ_OK;
}

extern "C" int ggq_chain_run(const ggq_chain* c, void* stream) {
    clear_error();
    if (!c) return fail(GGQ_EINVAL, "ggq_chain_run: NULL chain");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Workspace* ws = nullptr;
    int rc = get_workspace(s, groups_in_grid(c->type == GGQ_Q4_K, mmax_of(c->M)), c->rb_max, &ws);
    if (rc) return rc;
    StageDesc dummy;
    memset(&dummy, 0, sizeof(dummy));
    return launch_chain(c->type, c->M, dummy, c->table, c->nstages, c->cols_max, ws->partials, ws->counters, s);
}

extern "C" void ggq_chain_free(ggq_chain* c) {
    if (!c) return;
    if (c->table) cudaFree(c->table);
    delete c;
}
