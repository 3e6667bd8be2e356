// Persistent row-partitioned GEMV over a chain of dependent stages.
//
// A stage is up to four weight matrices of one type and width that share their
// input x (e.g. the q, k and v projections of a layer): y_i = W_i x.  A chain is
// a list of stages run in order; stage s+1 reads its x only after every output
// of stage s is written, so the x of a later stage may be the y of an earlier
// one.  A single GEMV is a chain of one stage.
//
// Work unit: one 256-column block of one row (SB) -- a Q4_K super-block
// (144 B), a Q8_0 period of 8 blocks (272 B), a Q4_0 period of 8 blocks
// (144 B) or a Q6_K super-block (210 B) -- split into four 64-column chunks.
// A launch decodes one weight kind, or Q6_K and one other kind stage by stage.  Each matrix's rows form groups of 16 (the last may be shorter),
// numbered across the stage's matrices.
//
//   * CTA b (one per SM) owns groups [GT*b/G, GT*(b+1)/G) of the stage's GT:
//     whole rows, so no output is ever split between CTAs and no cross-CTA
//     reduction exists.
//   * Its (group, SB) tiles are cut into W - 1 equal contiguous runs, one per
//     consumer warp.  Each consumer has a ring of 2-D bulk tensor copies (16
//     rows x up to NSB SBs); the CTA's last warp issues them all, lane w for
//     consumer w (its copy cursor), the lanes stepping together and each
//     refilling its consumer's slots as they are freed.  Weights do not depend
//     on earlier stages, so the rings run ahead into the next stages while the
//     chain waits at a stage boundary.
//   * Lane (r, c) = (lane / 4, lane % 4) decodes chunk c of rows r and r + 8 of
//     each SB in registers against x', the pre-scaled activations (each x' value
//     loaded once for both rows).  The 8 lanes of one
//     chunk read the same x' address (a broadcast), and chunks are padded so
//     that the four addresses of one load sit in different banks.  Two
//     shuffles add a row's chunks; a group that a warp sees over all its SBs is
//     stored directly, a group cut between warps is finished in shared memory
//     by the warp where it starts, adding the others' parts in warp order
//     (deterministic).
//   * Stage boundary: every CTA adds one to a device counter with release
//     semantics after its outputs are stored; CTAs wait (acquire, bounded) for
//     the count of all CTAs before reading the next stage's x.
//   * Fused steps (optional, per stage): RMSNorm or SiLU(gate) * up applied to
//     x while x' is built, a residual added as each output row is stored.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstddef>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "gemv_tile.cuh"
#include "ggq_internal.h"
#include "ptx.cuh"

namespace ggq {

namespace {

constexpr int kMaxSeg = 4;
constexpr int kMaxM = 4;
constexpr size_t kSmemLimit = 227 * 1024;

constexpr int kRowsPerLane = 2;                 // rows r and r + 8 of a group
constexpr int kGroupRows = 8 * kRowsPerLane;

// The fields of a stage other than its tensor maps.  A CTA keeps those of the
// next stages in shared memory (kInfoSlots slots, stage s in slot s mod
// kInfoSlots): read from global memory after a stage barrier, whose acquire
// leaves the L1 cold, each would wait an L2 round trip.
struct StageInfo {
    float* y[kMaxSeg];          // [M][rows]
    const float* x;             // [M][cols]
    const float* norm_w;        // x_op RMSNORM: [cols]
    const float* up;            // x_op SILU_MUL: [M][cols]
    const float* res[kMaxSeg];  // null, or [M][rows]: added to y
    int rows[kMaxSeg];
    int gstart[kMaxSeg + 1];    // first row group of each matrix in the stage's numbering; gstart[nseg] = groups
    int nseg;
    int cols;
    int units;                  // U = cols / 256
    int x_op;                   // GGQ_X_PLAIN / RMSNORM / SILU_MUL
    float eps;                  // RMSNORM
    int kind;                   // Kind of the stage's weights
    int pad_[3];
};
constexpr int kInfoVec = sizeof(StageInfo) / 16;   // 16-byte pieces
// While stage s runs, slots hold stages s .. s + kInfoSlots - 2; stage
// s + kInfoSlots - 1 is being fetched into the slot stage s - 1 used.
constexpr int kInfoSlots = 8;
// Group ranges of the CTA in the first kPartMax stages, worked out once at the
// start of a launch (two integer divisions each) and kept in shared memory.
constexpr int kPartMax = 128;
static_assert(sizeof(StageInfo) % 16 == 0, "StageInfo is copied in 16-byte pieces");

// One stage of a chain (device-visible: kernel parameter or global table).
struct StageDesc {
    CUtensorMap maps[kMaxSeg];  // per matrix: 8-byte elements, box of 16 rows x (NSB SBs + pad)
    StageInfo info;
};
static_assert(offsetof(StageDesc, info) % 16 == 0, "StageInfo is copied in 16-byte pieces");

struct ChainParams {
    const StageDesc* table;     // the stages in device memory, or null: the inline stage only
    int nstages;
    int M;
    int ring;                   // tiles per warp ring
    int xs;                     // x' floats per activation row (kXsb per SB of the widest stage)
    int nsub;                   // x sums per activation row (8 per SB of the widest stage)
    int* counter;               // stage counter (chains of > 1 stage); zero between launches
    int* status;
};

// Weight layouts the kernel streams: the copy geometry and the decode.
enum Kind { kKQ8 = 0, kKQ4K = 1, kKQ40 = 2, kKQ6 = 3 };

// Tile of one bulk tensor copy: 16 rows x NSB SBs, each row padded so that
// rows r and r+1 of one chunk fall in different banks.  Copies of a few KB:
// much smaller ones cost more per copy than the bytes they bring.
// Q6_K: an SB is 210 bytes, so it starts on 16 bytes only every 8 SBs; its copy
// starts at the 16-byte boundary below it and takes 240 bytes a row (224 cover
// any start, 16 more stagger the rows across banks).
template <int K>
struct Blk {
    static constexpr int kBytes = K == kKQ8 ? 272 : K == kKQ6 ? 210 : 144;   // one SB
    static constexpr int kElems = kBytes / 8;                 // 8-byte elements per SB (not Q6_K)
    static constexpr int kNsb = (K == kKQ8 || K == kKQ6) ? 1 : 2;   // SBs per copy
    static constexpr int kPad = K == kKQ8 ? 0 : 2;            // elements of padding per row
    static constexpr int kRow = K == kKQ6 ? 240 : (kElems * kNsb + kPad) * 8;    // smem bytes per row
    // first 8-byte element of the copy of SB u, and where the SB starts in it
    __host__ __device__ static constexpr int coord(int u) { return K == kKQ6 ? ((210 * u) & ~15) / 8 : u * kElems; }
    __host__ __device__ static constexpr int skew(int u) { return K == kKQ6 ? (210 * u) & 15 : 0; }
    static constexpr int kCopy = kGroupRows * kRow;            // bytes per copy
    static constexpr int kTile = (kCopy + 127) / 128 * 128;    // smem stride: 128-byte aligned
    // x' floats per SB: Q4_K four chunks of 64 padded to 68; Q8_0 one per byte
    // of the period; Q4_0 two per byte of its four 36-byte chunks
    static constexpr int kXsb = K == kKQ40 ? 288 : 272;
};

// The weight kinds one kernel instance decodes: a bit mask over Kind.  With one
// kind every stage is that kind; with several, a stage's kind is read from its
// fields (StageInfo::kind) and the copy geometry is chosen per stage.  Ring
// slots are as large as the largest kind's tile.
template <int KM>
struct KindSet {
    static_assert(KM > 0 && KM < 16, "kind mask");
    static constexpr bool kMixed = (KM & (KM - 1)) != 0;
    static constexpr int kFirst = (KM & 1) ? 0 : (KM & 2) ? 1 : (KM & 4) ? 2 : 3;
    static constexpr int cmax(int a, int b) { return a > b ? a : b; }
    static constexpr int kTile = cmax(cmax((KM & 1) ? Blk<kKQ8>::kTile : 0, (KM & 2) ? Blk<kKQ4K>::kTile : 0),
                                      cmax((KM & 4) ? Blk<kKQ40>::kTile : 0, (KM & 8) ? Blk<kKQ6>::kTile : 0));
    static __device__ __forceinline__ bool has(int k) { return (KM >> k) & 1; }
    // SBs per copy, bytes per copy and the first 8-byte element of SB u's copy
    static __device__ __forceinline__ int nsb(int k) {
        if constexpr (!kMixed) return Blk<kFirst>::kNsb;
        return (k == kKQ4K || k == kKQ40) ? 2 : 1;
    }
    static __device__ __forceinline__ int copy(int k) {
        if constexpr (!kMixed) return Blk<kFirst>::kCopy;
        return k == kKQ8 ? Blk<kKQ8>::kCopy : k == kKQ4K ? Blk<kKQ4K>::kCopy : k == kKQ40 ? Blk<kKQ40>::kCopy
                                                                                   : Blk<kKQ6>::kCopy;
    }
    static __device__ __forceinline__ int coord(int k, int u) {
        if constexpr (!kMixed) return Blk<kFirst>::coord(u);
        return k == kKQ6 ? Blk<kKQ6>::coord(u) : u * (k == kKQ8 ? Blk<kKQ8>::kElems : Blk<kKQ4K>::kElems);
    }
};
static_assert(Blk<kKQ4K>::kElems == Blk<kKQ40>::kElems, "Q4_K and Q4_0 super-blocks are both 144 bytes");

template <int K>
struct KindTag {
    static constexpr int value = K;
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

// Row groups: each matrix's rows in groups of 16 (its last group may be
// shorter), numbered across the stage's matrices.  CTA b (of nb) takes groups
// [GT*b/nb, GT*(b+1)/nb) of the stage's GT: whole groups, so a CTA whose range
// crosses a matrix boundary gets no extra partial group.
struct Groups {
    int g0;   // first group (stage numbering)
    int n;    // groups
};

__device__ __forceinline__ int cta_part(int GT, int b, int nb) {
    // GT * b / nb; 32-bit division whenever the product fits (every realistic stage)
    const unsigned long long gb = (unsigned long long)(unsigned)GT * (unsigned)b;
    if (gb <= 0xFFFFFFFFull) return (int)((unsigned)gb / (unsigned)nb);
    return (int)(gb / (unsigned)nb);
}

// Groups [g0, g1) of CTA b in a stage
__device__ __forceinline__ int2 cta_span(const StageInfo* sd, int b, int nb) {
    const int GT = sd->gstart[sd->nseg];
    return make_int2(cta_part(GT, b, nb), cta_part(GT, b + 1, nb));
}

__device__ __forceinline__ Groups cta_groups(int2 span) { return Groups{span.x, span.y - span.x}; }

// The CTA's group gi: matrix, first row (in the matrix), rows in the group.
__device__ __forceinline__ void group_at(const StageInfo* sd, const Groups& G, int gi, int& seg, int& row, int& nrows) {
    const int g = G.g0 + gi;
    seg = 0;
#pragma unroll
    for (int s = 1; s < kMaxSeg; ++s)
        if (s < sd->nseg && g >= sd->gstart[s]) seg = s;
    row = (g - sd->gstart[seg]) * kGroupRows;
    nrows = min(kGroupRows, sd->rows[seg] - row);
}

// The tile run [t0, t1) of warp w (of NW): tile t = group * U + SB.  A CTA
// holds fewer than 2^28 tiles (the stage holds fewer than 2^31 SBs, so fewer
// than 2^27 + 4U group-SBs, and a CTA at most all of them), so T * w fits 32
// bits.
template <int NW>
__device__ __forceinline__ void warp_run(const Groups& G, int U, int w, int& t0, int& t1) {
    const unsigned T = (unsigned)G.n * (unsigned)U;
    t0 = (int)(T * (unsigned)w / NW);
    t1 = (int)(T * (unsigned)(w + 1) / NW);
}

template <int KM, int MMAX, int W>
__global__ void __launch_bounds__(32 * W, 1) rows_kernel(const __grid_constant__ StageDesc inl, const ChainParams p) {
    using KSet = KindSet<KM>;
    constexpr int kTileK = KSet::kTile;   // ring slot stride
    constexpr int kThreads = 32 * W;
    // warps 0 .. WC-1 decode (consumers); warp WC issues every weight copy of
    // the CTA, lane w for consumer warp w (its copy cursor, its ring)
    constexpr int WC = W - 1;
    constexpr int kCThreads = 32 * WC;
    static_assert(WC >= 1 && WC <= 31, "one producer lane per consumer warp");
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = lane >> 2, c = lane & 3;   // row of the group, chunk of the SB
    const int D = p.ring;

    // shared memory: [consumer rings][stage info slots][group ranges][x'][sums][cut-group parts][barriers]
    StageInfo* infos = reinterpret_cast<StageInfo*>(smem + (size_t)WC * D * kTileK);
    int2* part = reinterpret_cast<int2*>(infos + kInfoSlots);   // [kPartMax]
    float* xp = reinterpret_cast<float*>(part + kPartMax);
    float* sums = xp + (size_t)MMAX * p.xs;
    float* cut_val = sums + (size_t)MMAX * p.nsub;                                 // [2][WC][16][MMAX]
    int* cut_grp = reinterpret_cast<int*>(cut_val + 2 * WC * kGroupRows * MMAX);   // [2][WC]
    uint64_t* full_all = reinterpret_cast<uint64_t*>(cut_grp + 2 * WC);            // [WC][D]; 8-byte aligned: all sizes even
    uint64_t* empty_all = full_all + WC * D;                                       // [WC][D]
    // consumer-only CTA barrier (the producer warp runs on its own)
    auto csync = [] { asm volatile("bar.sync 1, %0;" ::"n"(kCThreads) : "memory"); };

    if (warp < WC && lane == 0) {
        for (int i = 0; i < D; ++i) {
            mbar_init(&full_all[warp * D + i], 1);    // the producer's expect_tx; the copy's bytes
            mbar_init(&empty_all[warp * D + i], 1);   // the consumer warp, done with the slot
        }
        fence_mbar_init();
    }
    // stages 0 .. kInfoSlots - 2, and the row ranges
    for (int i = tid; i < min(p.nstages, kInfoSlots - 1) * kInfoVec; i += kThreads)
        reinterpret_cast<int4*>(infos)[i] =
            reinterpret_cast<const int4*>(p.table ? &p.table[i / kInfoVec].info : &inl.info)[i % kInfoVec];
    for (int i = tid; i < min(p.nstages, kPartMax); i += kThreads)
        part[i] = cta_span(p.table ? &p.table[i].info : &inl.info, blockIdx.x, gridDim.x);
    __syncthreads();
    pdl_launch_dependents();

    if (warp == WC) {
        // ---- producer: lane w walks consumer warp w's tiles of every stage, in
        // order, one copy per (group, up to NSB consecutive SBs), into ring
        // slots as the consumer frees them.  Stage fields are read from the
        // stage table (global memory, L2): the consumers' window moves with
        // their stage, not with this cursor, which runs ahead.
        const int w = lane;
        if (w < WC) {
            uint8_t* ring = smem + (size_t)w * D * kTileK;
            uint64_t* full = full_all + w * D;
            uint64_t* empty = empty_all + w * D;
            // stage, next tile, end of the run; (group, SB) of the next tile and
            // the group's matrix and first row, advanced without dividing
            int cs = -1, ct = 0, ct1 = 0, cU = 1, cgi = 0, cu = 0, cseg = 0, crow = 0;
            int cnext = 0;                   // first local group of matrix cseg + 1
            int ckind = KSet::kFirst;        // weight kind of stage cs
            const StageDesc* csd = &inl;
            const StageInfo* cinf = &inl.info;
            Groups cg{};
            auto next_seg_start = [&]() {
                return cseg + 1 < cinf->nseg ? cinf->gstart[cseg + 1] - cg.g0 : 0x7fffffff;
            };
            // the next stage in which warp w has tiles; false past the last
            auto next_stage = [&]() {
                while (ct == ct1) {
                    if (++cs >= p.nstages) return false;
                    csd = p.table ? p.table + cs : &inl;
                    cinf = &csd->info;
                    cg = cta_groups(cs < kPartMax ? part[cs] : cta_span(cinf, blockIdx.x, gridDim.x));
                    warp_run<WC>(cg, cinf->units, w, ct, ct1);
                }
                cU = cinf->units;
                if constexpr (KSet::kMixed) ckind = cinf->kind;
                cgi = ct / cU;
                cu = ct - cgi * cU;
                int nrows;
                group_at(cinf, cg, cgi, cseg, crow, nrows);
                cnext = next_seg_start();
                return true;
            };
            const uint64_t wpol = l2_evict_first_policy();   // weights are read once per pass
            // The previous kernel in the stream may still be writing what this
            // one reads (x, and W too if a caller rewrites weights in place), so
            // every copy is issued after the wait.  Before it, only L2 is warmed
            // with warp w's first tiles of stage 0 (a prefetch never decides what
            // a copy reads).
            {
                const StageDesc* d0 = p.table ? p.table : &inl;
                const Groups g0 = cta_groups(part[0]);
                const int U0 = infos[0].units;
                const int k0 = KSet::kMixed ? infos[0].kind : KSet::kFirst;
                int t, tend;
                warp_run<WC>(g0, U0, w, t, tend);
                for (int k = 0; k < D && t < tend; ++k) {
                    const int gi = t / U0, u = t - gi * U0;
                    int seg, row, nrows;
                    group_at(&infos[0], g0, gi, seg, row, nrows);
                    tma_prefetch_2d(&d0->maps[seg], KSet::coord(k0, u), row);
                    t += min(min(KSet::nsb(k0), U0 - u), tend - t);
                }
            }
            pdl_wait();
            int eslot = 0;
            uint32_t ephase = 0;
            // The lanes step together: each round, every lane whose consumer has
            // freed its next slot issues that copy, under predication, so one
            // pass through this code serves up to WC copies.  A lane ends after
            // its last copy; a slot that stays busy beyond the wait limit ends
            // its lane with the timeout bit set.
            bool live = ct < ct1 || next_stage();
            unsigned long long t_wait = 0;   // when this lane began to wait, 0: not waiting
            for (uint32_t it = 0;; ++it) {
                const bool ready = live && mbar_try_wait(&empty[eslot], ephase ^ 1u);
                if (ready) {
                    t_wait = 0;
                    const int nv = min(min(KSet::nsb(ckind), cU - cu), ct1 - ct);
                    tma_issue_2d(true, ring + (size_t)eslot * kTileK, &csd->maps[cseg], &full[eslot],
                                 KSet::coord(ckind, cu), crow, KSet::copy(ckind), wpol);
                    ct += nv;
                    cu += nv;
                    if (cu == cU && ct < ct1) {   // next group of this run: same matrix, 16 rows on, or the next matrix
                        cu = 0;
                        ++cgi;
                        if (cgi == cnext) {
                            ++cseg;
                            crow = 0;
                            cnext = next_seg_start();
                        } else {
                            crow += kGroupRows;
                        }
                    }
                    if (++eslot == D) {
                        eslot = 0;
                        ephase ^= 1u;
                    }
                    live = ct < ct1 || next_stage();
                } else if (live && (it & 63u) == 0) {
                    const unsigned long long now = globaltimer_ns();
                    if (t_wait == 0) {
                        t_wait = now;
                    } else {
                        const unsigned long long limit = ld_relaxed(p.status) != 0 ? kDrainNs : kWaitLimitNs;
                        if (now - t_wait > limit) {
                            atomicOr(p.status, kStatusTimeout);
                            live = false;
                        }
                    }
                }
                const unsigned busy = __ballot_sync((1u << WC) - 1u, live);   // the WC producer lanes
                if (busy == 0) break;
            }
        }
        return;
    }

    // ---- consumers
    uint8_t* ring = smem + (size_t)warp * D * kTileK;
    uint64_t* full = full_all + warp * D;
    uint64_t* empty = empty_all + warp * D;
    pdl_wait();

    int cslot = 0;          // ring slot of the next copy to consume
    uint32_t cphase = 0;    // its barrier phase

    for (int s = 0; s < p.nstages; ++s) {
        const StageInfo* sd = infos + s % kInfoSlots;
        // this CTA's row groups and this warp's tile run: independent of x, so
        // worked out before the stage barrier
        const Groups G = cta_groups(s < kPartMax ? part[s] : cta_span(sd, blockIdx.x, gridDim.x));
        int t0, t1;
        warp_run<WC>(G, sd->units, warp, t0, t1);
        // the fields of stage s + kInfoSlots - 1, to the slot of stage s - 1
        // (free: every consumer warp has passed the end of stage s - 1);
        // waited for before the end of stage s
        if (s + kInfoSlots - 1 < p.nstages && warp == WC - 1 && lane < kInfoVec)
            cp_async_16(reinterpret_cast<int4*>(infos + (s + kInfoSlots - 1) % kInfoSlots) + lane,
                        reinterpret_cast<const int4*>(&p.table[s + kInfoSlots - 1].info) + lane);
        if (s > 0) {
            // every CTA has finished stage s-1 (its outputs are visible)
            if (tid == 0) wait_count(p.counter, s * (int)gridDim.x, p.status);
            csync();
        }
        const int cols = sd->cols, U = sd->units;
        const int xs = p.xs, nsub = p.nsub;

        // ---- the stage's work for its weight kind KS: x' and sums, this warp's
        // tiles, groups cut between warps
        auto stage_body = [&](auto ktag) {
            constexpr int KS = decltype(ktag)::value;
            using BS = Blk<KS>;
            constexpr bool Q4K = KS == kKQ4K;
            // x' placement of the lane's 4 consecutive columns 4l .. 4l+3 of a
            // 128-column half of an SB (the other half adds kXsb / 2 floats).  Q4_K:
            // chunk l/16 (68 floats each), byte positions b = 0..3 of word l%8, low or
            // high nibble ((l/8) odd: high) at q4k_xslot, stride 16.  Q8_0: byte
            // positions of the period, 34 per block of 32 after its 2-byte scale.
            // Q4_0: block l/8 of the half (chunk l/16, block (l/8)%2 of the chunk),
            // weights 4(l%8) .. +3 of the block: byte positions 2 + 4(l%4) .. +3 after
            // the block's start, high nibble when l%8 >= 4, at 2B + hi, stride 2.
            int xoff;
            float4 xsc;
            {
                const int hi = (lane >> 3) & 1;
                if (Q4K) {
                    xoff = (lane >> 4) * 68 + 2 * (lane & 7) + hi;
                    const int k = 4 * lane;
                    xsc = make_float4(q4k_xscale(k), q4k_xscale(k + 1), q4k_xscale(k + 2), q4k_xscale(k + 3));
                } else if (KS == kKQ6) {
                    // chunk (h, gp) with gp = (l/8) % 2, pair slot l/16, word l % 8
                    xoff = ((lane >> 3) & 1) * 68 + 2 * (lane & 7) + (lane >> 4);
                    xsc = make_float4(pow2f(53), pow2f(45), pow2f(37), (lane >> 4) ? pow2f(37) : pow2f(53));
                } else if (KS == kKQ40) {
                    const int b4 = lane >> 3;
                    xoff = (b4 >> 1) * 72 + 2 * (18 * (b4 & 1) + 2 + 4 * (lane & 3)) + ((lane >> 2) & 1);
                    xsc = make_float4(q40_xscale(xoff), q40_xscale(xoff + 2), q40_xscale(xoff + 4), q40_xscale(xoff + 6));
                } else {
                    xoff = 34 * (lane >> 3) + 2 + 4 * (lane & 7);
                    xsc = make_float4(q8_xscale(xoff), q8_xscale(xoff + 1), q8_xscale(xoff + 2), q8_xscale(xoff + 3));
                }
            }

            // ---- x' and the 32-column sums of this stage: kXsb floats per SB (Q4_K:
            // four chunks of 64 in the q4k_xslot order, each padded by 4; Q8_0: one
            // float per byte position of the period; Q4_0: two per byte position).
            // x may have been written by other CTAs: read it from L2.
            {
                // Lane l of a warp step takes 4 consecutive values (one float4) of x:
                // 8 lanes cover a 32-column sub-block, whose sum takes 3 shuffles.
                // A warp step covers 128 columns of one activation row (cols is a
                // multiple of 256), half of an SB: the lane's place in it and the
                // scales of its 4 values are the lane constants xoff and xsc.
                // Every load of a batch is issued before any is used (one L2 round
                // trip per batch of kBatch float4 per lane).
                const int c4 = cols / 4;          // float4 per activation row
                const int n4 = p.M * c4;
                const float4* x4 = reinterpret_cast<const float4*>(sd->x);
                // place the float4 v of warp step qb (the lane's 4 columns): x', and
                // the sub-block sum from 8 lanes
                auto place = [&](int qb, float4 v) {
                    float sum = (v.x + v.y) + (v.z + v.w);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                    const float sum16 = sum;   // Q6_K: 16 columns
                    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
                    const int m = MMAX == 1 ? 0 : qb / c4;
                    const int h = qb - m * c4;          // first float4 of the step within the row
                    const int u = h >> 6;               // SB
                    float* dst = xp + (size_t)m * xs + u * BS::kXsb + ((h & 32) ? BS::kXsb / 2 : 0) + xoff;
                    const float4 e = make_float4(v.x * xsc.x, v.y * xsc.y, v.z * xsc.z, v.w * xsc.w);
                    if (Q4K || KS == kKQ6) {
                        dst[0] = e.x;
                        dst[16] = e.y;
                        dst[32] = e.z;
                        dst[48] = e.w;
                    } else if (KS == kKQ40) {
                        dst[0] = e.x;
                        dst[2] = e.y;
                        dst[4] = e.z;
                        dst[6] = e.w;
                    } else {
                        dst[0] = e.x;
                        dst[1] = e.y;
                        dst[2] = e.z;
                        dst[3] = e.w;
                    }
                    // the code offsets: Q8_0 bytes are stored XOR 0x80 (128), Q4_0 codes are q + 8,
                    // Q6_K codes q + 32 (sums per 16 columns: slot 8 half + 4 gp + 2 (l >= 16) + g / 2)
                    if constexpr (KS == kKQ6) {
                        if ((lane & 3) == 0)
                            sums[m * nsub + u * 16 + ((h & 32) >> 2) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) +
                                 (lane >> 4)] = 32.0f * sum16;
                    } else if ((lane & 7) == 0) {
                        sums[m * nsub + u * 8 + ((h & 32) >> 3) + (lane >> 3)] =
                            Q4K ? sum : (KS == kKQ40 ? 8.0f : 128.0f) * sum;
                    }
                };
                const int xop = sd->x_op;
                if (xop == GGQ_X_PLAIN) {
                    constexpr int kBatch = 8;
                    for (int q0 = warp * 32; q0 < n4; q0 += kCThreads * kBatch) {
                        float4 v[kBatch];
    #pragma unroll
                        for (int i = 0; i < kBatch; ++i) {
                            const int q = q0 + i * kCThreads + lane;
                            v[i] = q < n4 ? __ldcg(x4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
    #pragma unroll
                        for (int i = 0; i < kBatch; ++i) {
                            const int qb = q0 + i * kCThreads;   // warp-uniform, a multiple of 32
                            if (qb >= n4) break;
                            place(qb, v[i]);
                        }
                    }
                } else {
                    // fused step on x ("GGUF Inferencer in R" section 4).  RMSNORM: the
                    // sum of squares of each activation row first (a CTA reduction
                    // through the cut-group scratch, free until the tiles), then
                    // norm_w * x / sqrt(mean + eps).  SILU_MUL: silu(x) * up.
                    const float4* o4 = reinterpret_cast<const float4*>(xop == GGQ_X_RMSNORM ? sd->norm_w : sd->up);
                    constexpr int kBatch = 4;   // two float4 a step: x and norm_w / up
                    float* red = cut_val;       // [WC][MMAX]: per-warp sums of squares
                    float rs[MMAX];
                    auto load2 = [&](int q0, float4 (&v)[kBatch], float4 (&o)[kBatch]) {
    #pragma unroll
                        for (int i = 0; i < kBatch; ++i) {
                            const int q = q0 + i * kCThreads + lane;
                            const int qb = q0 + i * kCThreads;
                            const int m = MMAX == 1 ? 0 : qb / c4;
                            v[i] = q < n4 ? __ldcg(x4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
                            o[i] = q < n4 ? __ldcg(o4 + (xop == GGQ_X_RMSNORM ? q - m * c4 : q))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    };
                    // sums of squares per activation row (ss from this thread) -> rs
                    auto reduce_rs = [&](float (&ss)[MMAX]) {
    #pragma unroll
                        for (int m = 0; m < MMAX; ++m) {
                            const float t = warp_sum(ss[m]);
                            if (lane == 0) red[warp * MMAX + m] = t;
                        }
                        csync();
    #pragma unroll
                        for (int m = 0; m < MMAX; ++m) {
                            float t = 0.0f;
                            for (int w2 = 0; w2 < WC; ++w2) t += red[w2 * MMAX + m];   // same order in every thread
                            rs[m] = 1.0f / sqrtf(t / (float)cols + sd->eps);
                        }
                    };
                    auto transform = [&](int qb, float4 t, float4 o) {
                        if (xop == GGQ_X_RMSNORM) {
                            float r = rs[0];
    #pragma unroll
                            for (int m = 1; m < MMAX; ++m)
                                if (qb >= m * c4) r = rs[m];
                            return make_float4(o.x * (t.x * r), o.y * (t.y * r), o.z * (t.z * r), o.w * (t.w * r));
                        }
                        return make_float4(t.x / (1.0f + expf(-t.x)) * o.x, t.y / (1.0f + expf(-t.y)) * o.y,
                                           t.z / (1.0f + expf(-t.z)) * o.z, t.w / (1.0f + expf(-t.w)) * o.w);
                    };
                    if (MMAX <= 2 && xop == GGQ_X_RMSNORM && n4 <= kCThreads * kBatch) {
                        // one batch a thread: the squares come from the registers the
                        // values are placed from (one L2 round trip; up to 2 activation
                        // rows, where the registers allow it)
                        float4 v[kBatch], o[kBatch];
                        const int q0 = warp * 32;
                        load2(q0, v, o);
                        float ss[MMAX];
    #pragma unroll
                        for (int m = 0; m < MMAX; ++m) ss[m] = 0.0f;
    #pragma unroll
                        for (int i = 0; i < kBatch; ++i) {
                            const int qb = q0 + i * kCThreads;
                            const float e = fmaf(v[i].x, v[i].x, fmaf(v[i].y, v[i].y, fmaf(v[i].z, v[i].z, v[i].w * v[i].w)));
    #pragma unroll
                            for (int m = 0; m < MMAX; ++m)
                                if (qb >= m * c4 && qb < (m + 1) * c4) ss[m] += e;   // zero beyond n4
                        }
                        reduce_rs(ss);
    #pragma unroll
                        for (int i = 0; i < kBatch; ++i) {
                            const int qb = q0 + i * kCThreads;
                            if (qb >= n4) break;
                            place(qb, transform(qb, v[i], o[i]));
                        }
                    } else {
                        if (xop == GGQ_X_RMSNORM) {
                            // x too long for one batch: a first pass for the squares
                            float ss[MMAX];
    #pragma unroll
                            for (int m = 0; m < MMAX; ++m) {
                                ss[m] = 0.0f;
                                if (m < p.M) {
    #pragma unroll 4
                                    for (int q = tid; q < c4; q += kCThreads) {
                                        const float4 v = __ldcg(x4 + (size_t)m * c4 + q);
                                        ss[m] = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss[m]))));
                                    }
                                }
                            }
                            reduce_rs(ss);
                        }
                        for (int q0 = warp * 32; q0 < n4; q0 += kCThreads * kBatch) {
                            float4 v[kBatch], o[kBatch];
                            load2(q0, v, o);
    #pragma unroll
                            for (int i = 0; i < kBatch; ++i) {
                                const int qb = q0 + i * kCThreads;
                                if (qb >= n4) break;
                                place(qb, transform(qb, v[i], o[i]));
                            }
                        }
                    }
                }
            }
            if (tid < 2 * WC) cut_grp[tid] = -1;
            csync();

            // ---- this warp's tiles
            constexpr int R = kRowsPerLane;
            float acc[R][MMAX];     // rows r + 8i of the group
            float2 acc2[R][MMAX];   // Q4_K: (low-nibble part, high-nibble part)
    #pragma unroll
            for (int i = 0; i < R; ++i)
    #pragma unroll
                for (int m = 0; m < MMAX; ++m) {
                    acc[i][m] = 0.0f;
                    acc2[i][m] = make_float2(0.0f, 0.0f);
                }
            int cur = -1;   // group being accumulated
            // the residual of the group's rows (lanes c == 0), read when the warp
            // starts a group whose first tile is in its run: that warp's part of
            // the group is the one that carries it (deterministic sum order)
            float resv[R][MMAX];
    #pragma unroll
            for (int i = 0; i < R; ++i)
    #pragma unroll
                for (int m = 0; m < MMAX; ++m) resv[i][m] = 0.0f;
            auto load_res = [&](int gi) {
                if (c != 0 || gi * U < t0) return;
                int seg, row, nrows;
                group_at(sd, G, gi, seg, row, nrows);
                const float* rp = sd->res[seg];
                if (!rp) return;
                const int rows = sd->rows[seg];
    #pragma unroll
                for (int i = 0; i < R; ++i)
    #pragma unroll
                    for (int m = 0; m < MMAX; ++m)
                        resv[i][m] = (r + 8 * i < nrows && m < p.M) ? __ldcg(rp + (int64_t)m * rows + row + r + 8 * i) : 0.0f;
            };

            // finish group gi: add each row's four chunks, then store the group's
            // rows if this warp saw all of its SBs, else keep this warp's part
            auto flush = [&](int gi) {
    #pragma unroll
                for (int i = 0; i < R; ++i)
    #pragma unroll
                    for (int m = 0; m < MMAX; ++m) {
                        if constexpr (Q4K) {
                            acc[i][m] = acc2[i][m].x + acc2[i][m].y;
                            acc2[i][m] = make_float2(0.0f, 0.0f);
                        }
                        acc[i][m] += __shfl_xor_sync(0xffffffffu, acc[i][m], 1);
                        acc[i][m] += __shfl_xor_sync(0xffffffffu, acc[i][m], 2);
                    }
                const bool started = gi * U >= t0;
                const bool whole = started && (gi + 1) * U <= t1;
                if (started && c == 0) {
    #pragma unroll
                    for (int i = 0; i < R; ++i)
    #pragma unroll
                        for (int m = 0; m < MMAX; ++m) {
                            acc[i][m] += resv[i][m];
                            resv[i][m] = 0.0f;
                        }
                }
                if (whole) {
                    int seg, row, nrows;
                    group_at(sd, G, gi, seg, row, nrows);
                    if (c == 0) {
                        const int rows = sd->rows[seg];
    #pragma unroll
                        for (int i = 0; i < R; ++i)
                            if (r + 8 * i < nrows) {
                                float* ys = sd->y[seg] + row + r + 8 * i;
    #pragma unroll
                                for (int m = 0; m < MMAX; ++m)
                                    if (m < p.M) ys[(int64_t)m * rows] = acc[i][m];
                            }
                    }
                } else {
                    // part of a group that started before this run (slot 0) or that
                    // goes on past it (slot 1)
                    const int k = started ? 1 : 0;
                    if (c == 0) {
    #pragma unroll
                        for (int i = 0; i < R; ++i)
    #pragma unroll
                            for (int m = 0; m < MMAX; ++m)
                                cut_val[((k * WC + warp) * kGroupRows + r + 8 * i) * MMAX + m] = acc[i][m];
                    }
                    if (lane == 0) cut_grp[k * WC + warp] = gi;
                }
    #pragma unroll
                for (int i = 0; i < R; ++i)
    #pragma unroll
                    for (int m = 0; m < MMAX; ++m) acc[i][m] = 0.0f;
            };

            int gi = t0 / U, u = t0 - (t0 / U) * U;   // (group, SB) of tile t, advanced without dividing
            for (int t = t0; t < t1;) {
                const int nv = min(min(BS::kNsb, U - u), t1 - t);
                if (gi != cur) {
                    if (cur >= 0) flush(cur);
                    load_res(gi);
                    cur = gi;
                }
                wait_full(&full[cslot], cphase, p.status);
                const int slot = cslot;
                const uint8_t* rowp = ring + (size_t)slot * kTileK + r * BS::kRow;
    #pragma unroll
                for (int j = 0; j < BS::kNsb; ++j) {
                    if (j < nv) {
                        const int uj = u + j;
                        if constexpr (Q4K) {
                            q4k_chunk_rows<MMAX, R>(rowp + j * BS::kBytes, 8 * BS::kRow, c, xp + uj * BS::kXsb, xs,
                                                    sums + uj * 8, nsub, acc2, 68);
                        } else if constexpr (KS == kKQ6) {
                            q6k_chunk_rows<MMAX, R>(rowp, BS::skew(uj), 8 * BS::kRow, c, xp + uj * BS::kXsb + 68 * c, xs,
                                                    sums + uj * 16 + 8 * (c >> 1) + 4 * (c & 1), nsub, acc);
                        } else if constexpr (KS == kKQ40) {
                            q40_chunk_rows<MMAX, R>(rowp + j * BS::kBytes + 36 * c, 8 * BS::kRow, xp + uj * BS::kXsb + 72 * c,
                                                    xs, sums + uj * 8 + 2 * c, nsub, acc);
                        } else {
    #pragma unroll
                            for (int i = 0; i < R; ++i)
                                q8_chunk<MMAX>(rowp + 8 * i * BS::kRow + j * BS::kBytes + 68 * c, xp + uj * BS::kXsb + 68 * c,
                                               xs, sums + uj * 8 + 2 * c, nsub, acc[i]);
                        }
                    }
                }
                __syncwarp();   // every lane is done with the buffer: the producer may refill it
                if (lane == 0) mbar_arrive(&empty[cslot]);
                if (++cslot == D) {
                    cslot = 0;
                    cphase ^= 1u;
                }
                t += nv;
                u += nv;
                if (u == U) {
                    u = 0;
                    ++gi;
                }
            }
            if (cur >= 0) flush(cur);
            csync();

            // ---- groups cut between warps: the warp where the group starts adds the
            // later warps' parts in order and stores it (lane r: row r)
            if (cut_grp[WC + warp] >= 0 && lane < kGroupRows) {
                const int gi = cut_grp[WC + warp];
                float tsum[MMAX];
    #pragma unroll
                for (int m = 0; m < MMAX; ++m) tsum[m] = cut_val[((WC + warp) * kGroupRows + lane) * MMAX + m];
                // the other parts: the later warps whose (non-empty) run starts
                // inside this group, told from the run bounds alone so that every
                // load is independent; added in warp order
                const int g0 = gi * U, g1 = g0 + U;
    #pragma unroll
                for (int w2 = 1; w2 < WC; ++w2) {
                    int a2, b2;
                    warp_run<WC>(G, U, w2, a2, b2);
                    const bool part = w2 > warp && a2 < b2 && a2 > g0 && a2 < g1;
    #pragma unroll
                    for (int m = 0; m < MMAX; ++m) {
                        const float v = cut_val[(w2 * kGroupRows + lane) * MMAX + m];
                        if (part) tsum[m] += v;
                    }
                }
                int seg, row, nrows;
                group_at(sd, G, gi, seg, row, nrows);
                if (lane < nrows) {
                    const int rows = sd->rows[seg];
                    float* ys = sd->y[seg] + row + lane;
    #pragma unroll
                    for (int m = 0; m < MMAX; ++m)
                        if (m < p.M) ys[(int64_t)m * rows] = tsum[m];
                }
            }
        };
        if constexpr (!KSet::kMixed) {
            stage_body(KindTag<KSet::kFirst>{});
        } else {
            const int kd = sd->kind;
            if (kd == kKQ4K) {
                if constexpr ((KM >> kKQ4K) & 1) stage_body(KindTag<kKQ4K>{});
            } else if (kd == kKQ6) {
                if constexpr ((KM >> kKQ6) & 1) stage_body(KindTag<kKQ6>{});
            } else if (kd == kKQ40) {
                if constexpr ((KM >> kKQ40) & 1) stage_body(KindTag<kKQ40>{});
            } else {
                if constexpr ((KM >> kKQ8) & 1) stage_body(KindTag<kKQ8>{});
            }
        }

        // ---- stage s done in this CTA: publish it (the consumer barrier orders
        // every consumer warp's stores before thread 0's release); the last CTA of the chain
        // resets the counter for the next launch
        if (p.nstages > 1) {
            if (warp == WC - 1) cp_async_wait_all();
            csync();
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
    static std::atomic<int> sms[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 1;
    int n = sms[dev].load(std::memory_order_relaxed);
    if (!n) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        sms[dev].store(n, std::memory_order_relaxed);
    }
    return n > 0 ? n : 1;
}

int mmax_of(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : 4; }

// Warps per CTA (one of them issues the copies): 16, or 12 where four
// activation rows need the registers
int warps_of(int mmax) { return mmax == 4 ? 12 : 16; }

int kind_of(int type) {
    return type == GGQ_Q4_K ? kKQ4K : type == GGQ_Q4_0 ? kKQ40 : type == GGQ_Q6_K ? kKQ6 : kKQ8;
}

constexpr int kMaxRing = 8;

size_t tile_bytes(int kind) {
    return kind == kKQ8 ? (size_t)Blk<kKQ8>::kTile : kind == kKQ4K ? (size_t)Blk<kKQ4K>::kTile
         : kind == kKQ6 ? (size_t)Blk<kKQ6>::kTile : (size_t)Blk<kKQ40>::kTile;
}
int row_box(int kind) {   // 8-byte elements per row of a copy box
    return kind == kKQ8 ? Blk<kKQ8>::kRow / 8 : kind == kKQ4K ? Blk<kKQ4K>::kRow / 8
         : kind == kKQ6 ? Blk<kKQ6>::kRow / 8 : Blk<kKQ40>::kRow / 8;
}
int xsb_of(int kind) { return kind == kKQ40 ? Blk<kKQ40>::kXsb : kind == kKQ4K ? Blk<kKQ4K>::kXsb : Blk<kKQ8>::kXsb; }
int64_t sb_bytes(int kind) { return kind == kKQ8 ? 272 : kind == kKQ6 ? 210 : 144; }
int sums_per_sb(int kind) { return kind == kKQ6 ? 16 : 8; }

// The kernel instance that runs the kinds of a chain: one kind, or Q6_K with
// Q4_K (Q4_K_M / Q4_K_S files) or with Q4_0 (a Q6_K output head); 0: no
// instance.  (An instance decoding all four kinds is one kernel function large
// enough that building it with line info overflowed the compiler's stack.)
constexpr int kMixQ4K = (1 << kKQ4K) | (1 << kKQ6);
constexpr int kMixQ40 = (1 << kKQ40) | (1 << kKQ6);
int mask_of(int kinds) {
    if (kinds > 0 && (kinds & (kinds - 1)) == 0) return kinds;
    if ((kinds & ~kMixQ4K) == 0) return kMixQ4K;
    if ((kinds & ~kMixQ40) == 0) return kMixQ40;
    return 0;
}

// the largest per-kind size over the kinds of a mask
template <typename F>
int64_t max_over(int kmask, F f) {
    int64_t v = 0;
    for (int k = 0; k < 4; ++k)
        if ((kmask >> k) & 1) v = std::max<int64_t>(v, (int64_t)f(k));
    return v;
}

// Shared memory of a launch over stages of the kinds in `kinds`: ring slots
// of the instance's size, x' and sums for the kinds present
size_t rows_smem(int kinds, int mmax, int ring, int64_t cols_max) {
    const int WC = warps_of(mmax) - 1;   // consumer warps (one more warp issues the copies)
    const int64_t U = cols_max / 256;
    const size_t cut = (size_t)2 * WC * kGroupRows * mmax * 4 + (size_t)2 * WC * 4;
    return (size_t)WC * ring * max_over(mask_of(kinds), tile_bytes) + kInfoSlots * sizeof(StageInfo) +
           kPartMax * sizeof(int2) + (size_t)mmax * U * max_over(kinds, xsb_of) * 4 +
           (size_t)mmax * U * max_over(kinds, sums_per_sb) * 4 + cut + (size_t)2 * WC * ring * 8;
}

int rows_ring(int kinds, int mmax, int64_t cols_max) {
    int ring = kMaxRing;
    while (ring > 1 && rows_smem(kinds, mmax, ring, cols_max) > kSmemLimit) --ring;
    return rows_smem(kinds, mmax, ring, cols_max) <= kSmemLimit ? ring : 0;
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

// Tensor map of one matrix: rows of `row_bytes` as 8-byte elements, box of
// 16 rows x (NSB SBs + pad).  Out-of-range parts of a box read as zeros.
int encode_map(CUtensorMap* map, const void* W, int64_t rows, int64_t row_bytes, int kind) {
    auto fn = tensor_map_encoder();
    if (!fn) return fail(GGQ_ECUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 8), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)row_box(kind), (cuuint32_t)kGroupRows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(W), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GGQ_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return GGQ_OK;
}

int make_stage(int type, int n, const void* const* W, const int64_t* rows, int64_t cols, const float* x,
               float* const* y, StageDesc* sd) {
    const int kind = kind_of(type);
    memset(sd, 0, sizeof(*sd));
    int g = 0;
    for (int s = 0; s < n; ++s) {
        const int64_t row_bytes = cols / 256 * sb_bytes(kind);
        int rc = encode_map(&sd->maps[s], W[s], rows[s], row_bytes, kind);
        if (rc) return rc;
        sd->info.y[s] = y[s];
        sd->info.rows[s] = (int)rows[s];
        sd->info.gstart[s] = g;
        g += (int)((rows[s] + kGroupRows - 1) / kGroupRows);
    }
    sd->info.gstart[n] = g;
    sd->info.nseg = n;
    sd->info.x = x;
    sd->info.cols = (int)cols;
    sd->info.units = (int)(cols / 256);
    sd->info.kind = kind;
    return GGQ_OK;
}

template <int KM, int MMAX, int W>
int launch_t(const StageDesc& inl, const ChainParams& p, cudaStream_t stream, size_t smem, bool cooperative) {
    auto kernel = rows_kernel<KM, MMAX, W>;
    // largest dynamic smem set so far, per device; host threads may launch
    // concurrently, so the check is atomic and the update serialised
    static std::atomic<int> configured[64] = {};
    static std::mutex update;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t e = cudaSuccess;
    if (dev < 0 || dev >= 64 || configured[dev].load(std::memory_order_acquire) < (int)smem) {
        std::lock_guard<std::mutex> lock(update);
        if (dev < 0 || dev >= 64 || configured[dev].load(std::memory_order_relaxed) < (int)smem) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
            if (dev >= 0 && dev < 64) configured[dev].store((int)smem, std::memory_order_release);
        }
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
// `inl` is the only stage; `kinds` is the mask of their weight kinds.
int launch_rows(int kinds, int M, const StageDesc& inl, const StageDesc* table, int nstages, int64_t cols_max,
                int* counter, cudaStream_t stream) {
    const int km = mask_of(kinds);
    const int mmax = mmax_of(M);
    ChainParams p = {};
    p.table = table;
    p.nstages = nstages;
    p.M = M;
    p.ring = rows_ring(kinds, mmax, cols_max);
    if (p.ring == 0) return fail(GGQ_EINVAL, "shape needs too much shared memory");
    p.xs = (int)(cols_max / 256 * max_over(kinds, xsb_of));
    p.nsub = (int)(cols_max / 256 * max_over(kinds, sums_per_sb));
    p.counter = counter;
    p.status = device_status_word();
    if (!p.status) return fail(GGQ_ECUDA, "device status word unavailable");
    const size_t smem = rows_smem(kinds, mmax, p.ring, cols_max);
    const bool coop = nstages > 1;
    switch (km * 8 + mmax) {
#define GGQ_ROWS_CASE(KM)                                                                         \
    case (KM) * 8 + 1: return launch_t<(KM), 1, 16>(inl, p, stream, smem, coop);                \
    case (KM) * 8 + 2: return launch_t<(KM), 2, 16>(inl, p, stream, smem, coop);                \
    case (KM) * 8 + 4: return launch_t<(KM), 4, 12>(inl, p, stream, smem, coop);
        GGQ_ROWS_CASE(1 << kKQ8)
        GGQ_ROWS_CASE(1 << kKQ4K)
        GGQ_ROWS_CASE(1 << kKQ40)
        GGQ_ROWS_CASE(1 << kKQ6)
        GGQ_ROWS_CASE(kMixQ4K)
        GGQ_ROWS_CASE(kMixQ40)
#undef GGQ_ROWS_CASE
        default: return fail(GGQ_EINVAL, "no kernel instance for kinds %d, M %d", kinds, M);
    }
}

}  // namespace

bool stream_gemv_supported(int type, int64_t cols, int M, int nseg, const int64_t* rows) {
    if (M > kMaxM || nseg < 1 || nseg > kMaxSeg || cols % 256 || cols > (1 << 20)) return false;
    if (type != GGQ_Q8_0 && type != GGQ_Q4_K && type != GGQ_Q4_0 && type != GGQ_Q6_K) return false;
    // a Q4_K / Q4_0 copy box (2 SBs + pad) must not be wider than a row
    if (type != GGQ_Q8_0 && cols < 768) return false;
    // Q6_K rows (210 bytes per SB) are a multiple of 16 bytes only when cols % 2048 == 0
    if (type == GGQ_Q6_K && cols % 2048) return false;
    int64_t r = 0;
    for (int s = 0; s < nseg; ++s) r += rows[s];
    if (r * (cols / 256) >= (1ll << 31)) return false;   // SB indices are 32-bit
    return rows_ring(1 << kind_of(type), mmax_of(M), cols) > 0;
}

int launch_gemv_stream(int type, int nseg, const void* const* W, const int64_t* rows, int64_t cols, const float* x,
                       float* const* y, int M, cudaStream_t stream) {
    StageDesc sd;
    int rc = make_stage(type, nseg, W, rows, cols, x, y, &sd);
    if (rc) return rc;
    return launch_rows(1 << kind_of(type), M, sd, nullptr, 1, cols, nullptr, stream);
}

}  // namespace ggq

// ------------------------------------------------------------ chain ABI ----

using namespace ggq;

struct ggq_chain {
    int kinds = 0;   // mask of the stages' weight kinds
    int M = 0;
    int nstages = 0;
    int64_t cols_max = 0;
    int device = -1;
    StageDesc* table = nullptr;   // device memory
    int* counter = nullptr;       // device memory, zero between runs
};

extern "C" int ggq_chain_create(int type, int M, int nstages, const ggq_chain_stage* stages, ggq_chain** out) {
    return ggq_chain_create_ops(type, M, nstages, stages, nullptr, out);
}

extern "C" int ggq_chain_create_ops(int type, int M, int nstages, const ggq_chain_stage* stages,
                                    const ggq_chain_ops* ops, ggq_chain** out) {
    clear_error();
    if (!out) return fail(GGQ_EINVAL, "ggq_chain_create: out is NULL");
    *out = nullptr;
    if (nstages < 1 || nstages > 65536 || !stages) return fail(GGQ_EINVAL, "ggq_chain_create: bad stage list");
    std::vector<int> types((size_t)nstages, type);
    return ggq_chain_create_typed(M, nstages, types.data(), stages, ops, out);
}

extern "C" int ggq_chain_create_typed(int M, int nstages, const int* types, const ggq_chain_stage* stages,
                                      const ggq_chain_ops* ops, ggq_chain** out) {
    clear_error();
    if (!out) return fail(GGQ_EINVAL, "ggq_chain_create: out is NULL");
    *out = nullptr;
    if (M < 1 || M > kMaxM) return fail(GGQ_EINVAL, "ggq_chain_create: M %d outside 1..%d", M, kMaxM);
    if (nstages < 1 || nstages > 65536 || !stages || !types)
        return fail(GGQ_EINVAL, "ggq_chain_create: bad stage list");
    std::vector<StageDesc> host((size_t)nstages);
    int64_t cols_max = 0;
    int kinds = 0;
    for (int s = 0; s < nstages; ++s) {
        const int type = types[s];
        if (type != GGQ_Q8_0 && type != GGQ_Q4_K && type != GGQ_Q4_0 && type != GGQ_Q6_K)
            return fail(GGQ_ETYPE, "ggq_chain_create: stage %d type %d not supported", s, type);
        kinds |= 1 << kind_of(type);
        if (mask_of(kinds) == 0)
            return fail(GGQ_ETYPE, "ggq_chain_create: stage %d type %d: a chain mixes Q6_K with one other type at most",
                        s, type);
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
        if (ops) {
            const ggq_chain_ops& o = ops[s];
            if (o.x_op == GGQ_X_RMSNORM) {
                if (!o.norm_w || (reinterpret_cast<uintptr_t>(o.norm_w) & 15) != 0)
                    return fail(GGQ_EINVAL, "ggq_chain_create: stage %d norm_w missing or not 16-byte aligned", s);
                if (!(o.eps >= 0.0f) || !(o.eps < INFINITY))
                    return fail(GGQ_EINVAL, "ggq_chain_create: stage %d eps must be finite and >= 0", s);
            } else if (o.x_op == GGQ_X_SILU_MUL) {
                if (!o.up || (reinterpret_cast<uintptr_t>(o.up) & 15) != 0)
                    return fail(GGQ_EINVAL, "ggq_chain_create: stage %d up missing or not 16-byte aligned", s);
            } else if (o.x_op != GGQ_X_PLAIN) {
                return fail(GGQ_EINVAL, "ggq_chain_create: stage %d x_op %d unknown", s, o.x_op);
            }
            for (int i = 0; i < st.n; ++i)
                if ((reinterpret_cast<uintptr_t>(o.res[i]) & 3) != 0)
                    return fail(GGQ_EINVAL, "ggq_chain_create: stage %d res[%d] misaligned", s, i);
        }
        cols_max = std::max<int64_t>(cols_max, st.cols);
    }
    if (rows_ring(kinds, mmax_of(M), cols_max) == 0)
        return fail(GGQ_EINVAL, "ggq_chain_create: widest stage needs too much shared memory");
    for (int s = 0; s < nstages; ++s) {   // all stages valid: encode them
        const ggq_chain_stage& st = stages[s];
        int rc = make_stage(types[s], st.n, st.W, st.rows, st.cols, st.x, st.y, &host[(size_t)s]);
        if (rc) return rc;
        if (ops) {
            StageInfo& si = host[(size_t)s].info;
            si.x_op = ops[s].x_op;
            si.eps = ops[s].eps;
            si.norm_w = ops[s].norm_w;
            si.up = ops[s].up;
            for (int i = 0; i < st.n; ++i) si.res[i] = ops[s].res[i];
        }
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
    c->kinds = kinds;
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
    return launch_rows(c->kinds, c->M, none, c->table, c->nstages, c->cols_max, c->counter,
                       static_cast<cudaStream_t>(stream));
}

extern "C" int ggq_chain_reset(ggq_chain* c) {
    clear_error();
    if (!c) return fail(GGQ_EINVAL, "ggq_chain_reset: NULL chain");
    int prev = -1;
    cudaGetDevice(&prev);
    if (c->device >= 0 && c->device != prev) {
        cudaError_t e = cudaSetDevice(c->device);
        if (e != cudaSuccess) return cuda_fail(e, "ggq_chain_reset: set device");
    }
    // the counter, and the device status word: while it is set, every bounded
    // wait of this device gives up after a few polls, so a run after a reset
    // that left it set would read stage inputs before they are written
    int rc = GGQ_OK;
    cudaError_t e = cudaMemset(c->counter, 0, sizeof(int));
    if (e != cudaSuccess) rc = cuda_fail(e, "ggq_chain_reset");
    int status = 0;
    if (rc == GGQ_OK) rc = read_and_clear_status(&status);
    if (c->device >= 0 && c->device != prev && prev >= 0) cudaSetDevice(prev);
    return rc;
}

extern "C" void ggq_chain_free(ggq_chain* c) {
    if (!c) return;
    if (c->table) cudaFree(c->table);
    if (c->counter) cudaFree(c->counter);
    delete c;
}
