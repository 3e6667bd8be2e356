// Small-batch dequant-GEMM on the tcgen05 tensor cores: Y[M, rows] = X[M, cols] W^T
// for a few activation rows (M <= 16), W in Q8_0, Q4_K or Q4_0 ("GGUF: The File
// Format...", "How a Q8_0 block is stored": w = d*q; k-quant paragraph:
// w = d*sc_j*q - dmin*m_j; Q4_0 the Q8_0 layout with 4-bit codes, w = d*(u - 8)).
// Each decoded block is used for all M rows of X.
//
// Tiles that would leave SMs idle are split along K (whole 256-column blocks)
// between two CTAs, as halves or, when the tiles fill more than half of the SMs
// in one wave, as a big part (one CTA a tile) and a small part (several tiles'
// small parts a CTA).  The call then zeroes Y first and both parts of a split
// tile add into it (red.global.add): two terms, the same fp32 sum in either
// order; nothing is shared between launches.
//
// A CTA computes its parts one after another; for each, a 128-row tile of W
// against all M activation rows
// (UMMA M = 128 W rows, N = 16 activation rows padded with zeros, K = 16):
//   warp 0      TMA producer: raw blocks of 128 W rows x 256 columns;
//   warps 1, 18 (19, 20) one thread each issues MMAs (warp 1 also allocates
//               the TMEM columns): warp 1 those into accumulator columns 0-31,
//               warp 18 those into 32-47, and with four issuers warps 1 and 18
//               take the even stages and 19, 20 the odd ones (columns 64-111);
//               each commits its MMAs of a stage back to the stage's "empty"
//               barrier, which counts the two that use the stage;
//   warps 2..17 decoders: four threads a W row, 16 columns each per 64-column
//               stage (packed f32x2 arithmetic).  A weight is decoded exactly in fp32 and split into two
//               bf16 parts, hi = bf16(w) and lo = bf16(w - hi); X is split the
//               same way.  The three products hi*hi + hi*lo + lo*hi keep each
//               term to ~2^-16 relative with fp32 accumulation, and every
//               operand keeps the fp32 exponent range.  They take two MMAs per
//               16 columns: X_hi and X_lo, adjacent in shared memory, are one
//               N = 32 operand for W_hi (accumulator columns 0-15 and 16-31),
//               and W_lo * X_hi (N = 16) goes to columns 32-47.  At these
//               small N an issuing thread's MMA rate sets the pace, so the
//               products have threads of their own (one thread for both: 37.5
//               us on Q8_0 14336 x 4096 at M = 8; two: 34.1; four: 32.1).
//   epilogue    warps 2..5 read the three 128 x 16 accumulators (tcgen05.ld; a
//               warp reaches only its own quarter of the 128 TMEM lanes), add
//               them and store Y (or add it, for a split tile).
// Every wait is bounded (ptx.cuh: mbar_wait); a timeout is recorded in the device
// status word and the kernel runs to completion without the data.
#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "ggq_internal.h"
#include "ptx.cuh"

namespace ggq {

namespace {

constexpr int kTileRows = 128;   // UMMA M (W rows)
constexpr int kN = 16;           // UMMA N (activation rows, zero padded)
constexpr int kKStage = 64;      // columns per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr int kRawStages = 2;
constexpr int kDecoders = 512;
constexpr int kLoWarp = 2 + kDecoders / 32;   // the further MMA-issuing warps, after the decoders

constexpr int kAPiece = kTileRows * kKStage * 2;   // 16 KB: one bf16 part of a W tile
constexpr int kBPiece = kN * kKStage * 2;          // 2 KB: one bf16 part of an X tile
constexpr int kStageBytes = 2 * kAPiece + 2 * kBPiece;   // [A hi][A lo][B hi][B lo], 1024-aligned parts
constexpr int kRawMax = kTileRows * 272;                  // Q8_0: 8 blocks a row; Q4_K uses 144 of it

constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + (size_t)kRawStages * kRawMax + 1024 + 256;

// weight layouts: Q8_0 periods of 8 blocks (272 bytes), Q4_K super-blocks and
// Q4_0 runs of 8 blocks (144 bytes), Q6_K super-blocks (210 bytes: copied from
// the 16-byte boundary below them, 240 bytes a row), each 256 columns of a row
enum SmKind { kSmQ8 = 0, kSmQ4K = 1, kSmQ40 = 2, kSmQ6 = 3 };

// MMA-issuing threads: two (the W_hi and the W_lo product) or four (each of
// those for the even and for the odd stages, into their own accumulators).
// Four for Q8_0, Q4_K and Q4_0; Q6_K, whose decoders set the pace, keeps two
// (the extra warps cost its decoders more than they gain).
template <int K>
struct Iss {
    static constexpr int kN = K == kSmQ6 ? 2 : 4;
    static constexpr int kThreads = 64 + kDecoders + 32 * (kN - 1);
    // D[0:32] = A_hi [X_hi; X_lo]^T, D[32:48] = A_lo X_hi^T; with four issuers
    // the odd stages' products at D[64:112]
    static constexpr int kTmemCols = kN == 4 ? 128 : 64;
};

// TMA x coordinate (elements of the tensor map) of 256-column block sb
template <int K>
__device__ __forceinline__ int raw_x(int sb) {
    if constexpr (K == kSmQ8) return sb * 136;            // 2-byte elements
    if constexpr (K == kSmQ6) return (210 * sb) & ~15;    // bytes, 16-byte aligned
    return sb * 144;                                      // bytes
}
constexpr int kMaxPieces = 8;

struct SmallParams {
    const float* x;   // [M, cols]
    float* y;         // [M, rows]; zeroed by the call when tiles are split
    int rows;
    int cols;
    int M;
    int full_tiles;   // tiles computed whole (CTAs 0 .. full_tiles-1)
    int nsplit;       // split tiles after them
    int sb_big;       // big/small layout: 256-column blocks of the big part (0: halves)
    int k_small;      // big/small layout: small parts a CTA
    int* status;
};

// The parts a CTA computes: tile, 256-column blocks [sb0, sb1), split or not
struct Piece {
    int tile, sb0, sb1;
    bool split;
};

__device__ __forceinline__ int pieces_of(const SmallParams& p, int cta) {
    if (cta < p.full_tiles || p.sb_big == 0) return 1;
    const int c = cta - p.full_tiles;
    if (c < p.nsplit) return 1;
    return min(p.k_small, p.nsplit - (c - p.nsplit) * p.k_small);
}

__device__ __forceinline__ Piece piece_of(const SmallParams& p, int cta, int i, int nsb_all) {
    if (cta < p.full_tiles) return Piece{cta, 0, nsb_all, false};
    const int c = cta - p.full_tiles;
    if (p.sb_big == 0) {   // halves: CTAs 2j, 2j + 1 of split tile j
        const int j = c >> 1, part = c & 1;
        return Piece{p.full_tiles + j, part ? nsb_all / 2 : 0, part ? nsb_all : nsb_all / 2, true};
    }
    if (c < p.nsplit) return Piece{p.full_tiles + c, 0, p.sb_big, true};
    const int j = (c - p.nsplit) * p.k_small + i;
    return Piece{p.full_tiles + j, p.sb_big, nsb_all, true};
}

// *p += v at the memory, no value returned
__device__ __forceinline__ void red_add_f32(float* p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 x bf16 -> fp32
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// K-major, 128-byte swizzle: 8-row groups 1024 B apart, descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// kind::f16: D fp32, A and B bf16, both K-major, N = 16, M = 128.
constexpr uint32_t kIdesc =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kTileRows >> 4) << 24);
// the same with N = 32: B is X_hi and X_lo stacked (their 16-row pieces are
// adjacent, so they form one 32-row K-major operand)
constexpr uint32_t kIdesc32 =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)((2 * kN) >> 3) << 17) | ((uint32_t)(kTileRows >> 4) << 24);

// w -> bf16 pairs hi = bf16(w), lo = bf16(w - hi) (w - hi is exact in fp32)
__device__ __forceinline__ void split_bf16x2(float2 w, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __float22bfloat162_rn(w);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __float22bfloat162_rn(__ffma2_rn(hf, make_float2(-1.0f, -1.0f), w));
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// 6-bit scale and min of sub-block j from the 12 packed bytes (three words)
__device__ __forceinline__ void q4k_sm(uint32_t s0, uint32_t s1, uint32_t s2, int j, int& sc, int& m) {
    if (j < 4) {
        sc = (s0 >> (8 * j)) & 63;
        m = (s1 >> (8 * j)) & 63;
    } else {
        const int k = j - 4;
        sc = ((s2 >> (8 * k)) & 15) | (((s0 >> (8 * k + 6)) & 3) << 4);
        m = ((s2 >> (8 * k + 4)) & 15) | (((s1 >> (8 * k + 6)) & 3) << 4);
    }
}

template <int K>
__global__ void __launch_bounds__(Iss<K>::kThreads, 1) smallm_kernel(const __grid_constant__ CUtensorMap wmap,
                                                             const SmallParams p) {
    constexpr bool Q4K = K == kSmQ4K;
    constexpr int NI = Iss<K>::kN;   // MMA-issuing threads
    constexpr int kRowBytes = K == kSmQ8 ? 272 : K == kSmQ6 ? 240 : 144;   // raw bytes of one W row per 256 columns
    constexpr int kRawBytes = kTileRows * kRowBytes;
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsb_all = p.cols / 256;
    const int npc = pieces_of(p, blockIdx.x);

    const uint32_t base_u32 = smem_u32(smem_raw);
    uint8_t* base = smem_raw + (((base_u32 + 1023u) & ~1023u) - base_u32);
    uint8_t* sStage = base;                                          // kStages x [A hi][A lo][B hi][B lo]
    uint8_t* sRaw = sStage + (size_t)kStages * kStageBytes;         // kRawStages x kRawMax
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRaw + (size_t)kRawStages * kRawMax);
    uint64_t* full = bars;                          // [kStages]  decoders -> MMA
    uint64_t* empty = bars + kStages;               // [kStages]  MMA -> decoders
    uint64_t* full_raw = bars + 2 * kStages;        // [kRawStages]  TMA -> decoders
    uint64_t* empty_raw = full_raw + kRawStages;    // [kRawStages]  decoders -> TMA
    uint64_t* acc_full = empty_raw + kRawStages;    // MMA -> epilogue, once a part
    uint64_t* acc_empty = acc_full + 1;             // epilogue -> MMA: the accumulator has been read
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 1);

    if (threadIdx.x == 0) {
        prefetch_tensormap(&wmap);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], kDecoders);
            mbar_init(&empty[s], 2);   // a commit from each MMA-issuing thread
        }
        for (int r = 0; r < kRawStages; ++r) {
            mbar_init(&full_raw[r], 1);
            mbar_init(&empty_raw[r], kDecoders);
        }
        mbar_init(acc_full, NI);   // a commit from each issuing thread
        mbar_init(acc_empty, 128);   // the four epilogue warps
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, Iss<K>::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // the previous kernel in the stream may still be writing W (a caller
            // that rewrites weights in place): warm L2 with the first raw stages,
            // then wait before any copy
            {
                const Piece p0 = piece_of(p, blockIdx.x, 0, nsb_all);
                for (int sb = p0.sb0; sb < p0.sb1 && sb < p0.sb0 + kRawStages; ++sb)
                    tma_prefetch_2d(&wmap, raw_x<K>(sb), p0.tile * kTileRows);
            }
            pdl_wait();
            int gsb = 0;   // raw stages issued (all parts)
            for (int pc = 0; pc < npc; ++pc) {
                const Piece pi = piece_of(p, blockIdx.x, pc, nsb_all);
                for (int sb = pi.sb0; sb < pi.sb1; ++sb, ++gsb) {
                    const int r = gsb % kRawStages;
                    mbar_wait(&empty_raw[r], ((gsb / kRawStages) & 1) ^ 1, p.status);
                    mbar_arrive_expect_tx(&full_raw[r], kRawBytes);
                    tma_load_2d(sRaw + (size_t)r * kRawMax, &wmap, &full_raw[r], raw_x<K>(sb), pi.tile * kTileRows);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp >= kLoWarp) {
        if (lane == 0) {
            // NI issuing threads, each into accumulator columns of its own: warp
            // 1 issues W_hi x [X_hi; X_lo] (columns 0-31), warp kLoWarp W_lo x
            // X_hi (columns 32-47); with four, these for the even stages and
            // warps kLoWarp + 1, + 2 the same for the odd ones (columns 64 on).
            // Each commits its own MMAs; the barriers count the commits.
            const int iss = warp == 1 ? 0 : warp - kLoWarp + 1;
            const bool lo = iss & 1;
            const int par = NI == 4 ? iss >> 1 : 0;
            // a descriptor's address field is (address >> 4): descriptors of the
            // other parts and offsets are the stage-0 one plus (offset >> 4)
            const uint64_t d0 = sw128_desc(smem_u32(sStage));
            constexpr uint32_t kLo = kAPiece >> 4, kBhi = (2 * kAPiece) >> 4;   // X_lo follows X_hi: one N = 32 operand
            const uint64_t a_off = lo ? kLo : 0;
            const uint32_t d_col = (lo ? 2 * kN : 0) + 64 * par;
            const uint32_t idesc = lo ? kIdesc : kIdesc32;
            // one loop over the stages of all parts (this thread's issue rate
            // sets the pace, so the loop is kept as plain as for one part);
            // at a part's end: its accumulator to the epilogue, and the next
            // part starts once the epilogue has read it
            int nks = 0;   // stages of all parts
            for (int pc = 0; pc < npc; ++pc) {
                const Piece pi = piece_of(p, blockIdx.x, pc, nsb_all);
                nks += 4 * (pi.sb1 - pi.sb0);
            }
            const Piece p0 = piece_of(p, blockIdx.x, 0, nsb_all);
            int pc = 0, pstart = 0, pend = 4 * (p0.sb1 - p0.sb0);
            for (int ks = 0; ks < nks; ++ks) {
                if (ks == pend) {
                    umma_commit(acc_full);
                    mbar_wait(acc_empty, pc & 1, p.status);
                    tc_fence_after();
                    ++pc;
                    const Piece pi = piece_of(p, blockIdx.x, pc, nsb_all);
                    pstart = ks;
                    pend = ks + 4 * (pi.sb1 - pi.sb0);
                }
                if (NI == 4 && (ks & 1) != par) continue;   // the other parity's stage
                const int s = ks % kStages;
                mbar_wait(&full[s], (ks / kStages) & 1, p.status);
                tc_fence_after();
                const uint64_t ds = d0 + (uint64_t)((s * kStageBytes) >> 4);
                // this thread's first stage of the part (a part has at least 4)
                const int first = ks == pstart + (NI == 4 ? ((par ^ pstart) & 1) : 0);
#pragma unroll
                for (int kk = 0; kk < kKStage / 16; ++kk) {
                    const uint64_t a = ds + 2 * kk;   // 16 bf16 = 32 bytes further along the swizzled rows
                    umma_bf16(tmem + d_col, a + a_off, a + kBhi, idesc, !(first && kk == 0));
                }
                umma_commit(&empty[s]);
            }
            umma_commit(acc_full);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- decoders (warps 2..17)
        const int t = threadIdx.x - 64;
        const int row = t & (kTileRows - 1);   // W row within the tile
        const int qt = t >> 7;                 // which 16 columns of a 64-column stage
        // X part of a stage: activation row t / 32, columns 2*(t % 32), +1
        const int xt = t >> 5, xk = 2 * (t & 31);
        const bool xv = xt < p.M;
        const float* xrow = p.x + (size_t)(xv ? xt : 0) * p.cols + xk;
        pdl_wait();   // X may come from the previous kernel in the stream
        int gsb = 0;   // raw stages consumed (all parts): the rings' position
        for (int pc = 0; pc < npc; ++pc) {
            const Piece pi = piece_of(p, blockIdx.x, pc, nsb_all);
            const int nks = 4 * (pi.sb1 - pi.sb0);
            const float* xp = xrow + (size_t)pi.sb0 * 256;
            // X of the next 4 stages in registers, so its loads are in flight early
            float2 xb[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                xb[c] = (xv && c < nks) ? __ldg(reinterpret_cast<const float2*>(xp + kKStage * c))
                                        : make_float2(0.f, 0.f);
            for (int lsb = 0; lsb < pi.sb1 - pi.sb0; ++lsb, ++gsb) {
                const int r = gsb % kRawStages;
                mbar_wait(&full_raw[r], (gsb / kRawStages) & 1, p.status);
                const uint8_t* rp = sRaw + (size_t)r * kRawMax + (size_t)row * kRowBytes +
                                    (K == kSmQ6 ? ((210 * (pi.sb0 + lsb)) & 15) : 0);   // the super-block's start
                uint4 hdr = make_uint4(0, 0, 0, 0);
                if constexpr (Q4K) hdr = *reinterpret_cast<const uint4*>(rp);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int lks = lsb * 4 + c;   // stage within the part
                    const int ks = gsb * 4 + c;    // ring position
                    const int s = ks % kStages;
                    // 16 weights of this thread, exact in fp32, as 8 pairs
                    float2 w[8];
                    if constexpr (K == kSmQ4K) {
                        // columns 64c + 16qt .. +15: sub-block 2c + qt/2, qs bytes 32c + 16(qt&1) ..
                        int sc, m;
                        q4k_sm(hdr.y, hdr.z, hdr.w, 2 * c + (qt >> 1), sc, m);
                        const float a = half_bits_to_float(hdr.x) * (float)sc;
                        const float bm = half_bits_to_float(hdr.x >> 16) * (float)m;
                        const uint4 q = *reinterpret_cast<const uint4*>(rp + 16 + 32 * c + 16 * (qt & 1));
                        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
                        const int ns = 4 * (qt >> 1);   // low or high nibbles
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            // 0x4B000000 | q is the float 2^23 + q
                            const uint32_t n0 = (qw[i >> 1] >> (16 * (i & 1) + ns)) & 15u;
                            const uint32_t n1 = (qw[i >> 1] >> (16 * (i & 1) + 8 + ns)) & 15u;
                            const float2 f = make_float2(__uint_as_float(0x4B000000u | n0), __uint_as_float(0x4B000000u | n1));
                            const float2 qf = __fadd2_rn(f, make_float2(-8388608.0f, -8388608.0f));
                            w[i] = __ffma2_rn(qf, make_float2(a, a), make_float2(-bm, -bm));
                        }
                    } else if constexpr (K == kSmQ6) {
                        // weights k = 64c + 16qt + i (i < 16): half h = c/2, quarter
                        // g = 2(c%2) + qt/2, l = 16(qt%2) + i; low bits in ql[64h +
                        // 32(g%2) + l] at bit 4(g/2), high bits in qh[32h + l] at bit
                        // 2g; one scale, sc[4c + qt].  The super-block starts on 2 bytes
                        // (rp even): words are read aligned and realigned.
                        const int h = c >> 1, g = 2 * (c & 1) + (qt >> 1), l0 = 16 * (qt & 1);
                        const int lo_off = 64 * h + 32 * (g & 1) + l0, hi_off = 128 + 32 * h + l0;
                        const int sh = 8 * ((int)(reinterpret_cast<uintptr_t>(rp)) & 3);   // 0 or 16
                        const uint32_t* wl = reinterpret_cast<const uint32_t*>(
                            reinterpret_cast<uintptr_t>(rp + lo_off) & ~(uintptr_t)3);
                        const uint32_t* wh = reinterpret_cast<const uint32_t*>(
                            reinterpret_cast<uintptr_t>(rp + hi_off) & ~(uintptr_t)3);
                        uint32_t a[5], b[5];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            a[i] = wl[i];
                            b[i] = wh[i];
                        }
                        a[4] = sh ? wl[4] : 0u;
                        b[4] = sh ? wh[4] : 0u;
                        uint32_t u[4];   // the 16 six-bit codes q + 32, four a word
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t qlw = __funnelshift_r(a[i], a[i + 1], sh);
                            const uint32_t qhw = __funnelshift_r(b[i], b[i + 1], sh);
                            u[i] = ((qlw >> (4 * (g >> 1))) & 0x0F0F0F0Fu) | (((qhw >> (2 * g)) & 0x03030303u) << 4);
                        }
                        const float d = half_bits_to_float(*reinterpret_cast<const uint16_t*>(rp + 208));
                        const float dsc = d * (float)(int)reinterpret_cast<const int8_t*>(rp + 192)[4 * c + qt];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            // 0x4B0000 | u is the float 2^23 + u; minus 2^23 + 32: q exactly
                            const uint32_t f0 = __byte_perm(u[i >> 1], 0x4B000000u, 0x7650u | (uint32_t)(2 * (i & 1)));
                            const uint32_t f1 = __byte_perm(u[i >> 1], 0x4B000000u, 0x7650u | (uint32_t)(2 * (i & 1) + 1));
                            const float2 qf = __fadd2_rn(make_float2(__uint_as_float(f0), __uint_as_float(f1)),
                                                         make_float2(-8388640.0f, -8388640.0f));
                            w[i] = __fmul2_rn(qf, make_float2(dsc, dsc));
                        }
                    } else {
                        // block 2c + qt/2 of the row's 256 columns: fp16 d at its start,
                        // then its codes; Q8_0: q bytes 16(qt&1) .. +15 of its 32 (34-byte
                        // blocks); Q4_0: the low (qt even) or high nibbles of its 16 code
                        // bytes (18-byte blocks: weight l low nibble, weight 16 + l high)
                        constexpr int kBlk = K == kSmQ8 ? 34 : 18;
                        const int off = kBlk * (2 * c + (qt >> 1));
                        const uint16_t dh = *reinterpret_cast<const uint16_t*>(rp + off);
                        const int qo = off + 2 + (K == kSmQ8 ? 16 * (qt & 1) : 0);   // 2-byte aligned
                        const uint32_t* wp = reinterpret_cast<const uint32_t*>(rp + (qo & ~3));
                        const int sh = 8 * (qo & 3);   // 0 or 16
                        uint32_t v[5];
#pragma unroll
                        for (int i = 0; i < 4; ++i) v[i] = wp[i];
                        v[4] = sh ? wp[4] : 0u;   // only a misaligned start reaches a fifth word
                        uint32_t u[4];   // the 16 codes, four a word, as unsigned bytes
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t wv = __funnelshift_r(v[i], v[i + 1], sh);
                            if constexpr (K == kSmQ8) u[i] = wv ^ 0x80808080u;   // q + 128
                            else u[i] = (qt & 1) ? ((wv >> 4) & 0x0F0F0F0Fu) : (wv & 0x0F0F0F0Fu);   // u = q + 8
                        }
                        const float d = half_bits_to_float(dh);
                        // 0x4B0000 | byte is the float 2^23 + byte; minus 2^23 + the offset: q
                        constexpr float kOff = K == kSmQ8 ? -8388736.0f : -8388616.0f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint32_t f0 = __byte_perm(u[i >> 1], 0x4B000000u, 0x7650u | (uint32_t)(2 * (i & 1)));
                            const uint32_t f1 = __byte_perm(u[i >> 1], 0x4B000000u, 0x7650u | (uint32_t)(2 * (i & 1) + 1));
                            const float2 qf = __fadd2_rn(make_float2(__uint_as_float(f0), __uint_as_float(f1)),
                                                         make_float2(kOff, kOff));
                            w[i] = __fmul2_rn(qf, make_float2(d, d));
                        }
                    }
                    mbar_wait(&empty[s], ((ks / kStages) & 1) ^ 1, p.status);
                    uint8_t* sA = sStage + (size_t)s * kStageBytes;
                    uint8_t* ahi = sA + (size_t)row * 128;
                    uint8_t* alo = ahi + kAPiece;
                    const int sw = row & 7;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {   // 16-byte chunk 2qt + j of the row: columns 16qt + 8j .. +7
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) split_bf16x2(w[4 * j + e], hi[e], lo[e]);
                        const int ch = ((2 * qt + j) ^ sw) << 4;
                        *reinterpret_cast<uint4*>(ahi + ch) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4*>(alo + ch) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                    {
                        // X: activation row xt, columns xk, xk+1 of this stage
                        uint32_t hi, lo;
                        split_bf16x2(xb[c], hi, lo);
                        uint8_t* bhi = sA + 2 * kAPiece + (size_t)xt * 128;
                        const int ch = (((xk >> 3) ^ (xt & 7)) << 4) + 4 * ((xk >> 1) & 3);
                        *reinterpret_cast<uint32_t*>(bhi + ch) = hi;
                        *reinterpret_cast<uint32_t*>(bhi + kBPiece + ch) = lo;
                        // next use of this register: stage lks + 4 of the part
                        xb[c] = (xv && lks + 4 < nks) ? __ldg(reinterpret_cast<const float2*>(xp + kKStage * (lks + 4)))
                                                      : make_float2(0.f, 0.f);
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&full[s]);
                }
                mbar_arrive(&empty_raw[r]);
            }

            // -------------------------------------------------------- epilogue
            if (warp < 6) {   // warps 2..5 cover the four TMEM lane quarters
                mbar_wait(acc_full, pc & 1, p.status);
                tc_fence_after();
                const int q = warp & 3;   // TMEM lane quarter of this warp
                const int yrow = pi.tile * kTileRows + 32 * q + lane;
                float v[16], vl[16], vh[16];
                const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
                tmem_ld16(tq, v);               // hi * hi
                tmem_ld16(tq + kN, vl);         // hi * lo
                tmem_ld16(tq + 2 * kN, vh);     // lo * hi
                if constexpr (NI == 4) {        // the same for the odd stages
                    float v2[16], vl2[16], vh2[16];
                    tmem_ld16(tq + 64, v2);
                    tmem_ld16(tq + 64 + kN, vl2);
                    tmem_ld16(tq + 64 + 2 * kN, vh2);
#pragma unroll
                    for (int i = 0; i < kN; ++i) v[i] = (v[i] + vl[i] + vh[i]) + (v2[i] + vl2[i] + vh2[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < kN; ++i) v[i] += vl[i] + vh[i];
                }
                tc_fence_before();
                mbar_arrive(acc_empty);   // the accumulator may take the next part's products
                if (yrow < p.rows) {
#pragma unroll
                    for (int i = 0; i < kN; ++i) {
                        if (i < p.M) {
                            float* yp = p.y + (size_t)i * p.rows + yrow;
                            if (pi.split) red_add_f32(yp, v[i]);
                            else *yp = v[i];
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Iss<K>::kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

template <int K>
int launch_t(const CUtensorMap& wmap, const SmallParams& p, int grid, cudaStream_t stream) {
    static std::atomic<int> configured[64] = {};   // set once per device; the value set never changes
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(smallm_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        if (dev >= 0 && dev < 64) configured[dev].store(1, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Iss<K>::kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, smallm_kernel<K>, wmap, p);
    if (e != cudaSuccess) return cuda_fail(e, "small-M launch");
    return GGQ_OK;
}

}  // namespace

bool smallm_supported(int type, int64_t rows, int64_t cols, int M) {
    // Q6_K rows (210 bytes per 256 columns) start on 16 bytes only when cols % 2048 == 0
    if (type == GGQ_Q6_K && cols % 2048) return false;
    return (type == GGQ_Q8_0 || type == GGQ_Q4_K || type == GGQ_Q4_0 || type == GGQ_Q6_K) && M >= 1 && M <= kN &&
           cols >= 256 && cols % 256 == 0 && cols <= (1 << 24) && rows >= 1 && rows <= 0x7fffffff;
}

int launch_smallm(int type, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int M,
                  cudaStream_t stream) {
    auto enc = encoder();
    if (!enc) return fail(GGQ_ECUDA, "cuTensorMapEncodeTiled unavailable");
    const int kind = type == GGQ_Q4_K ? kSmQ4K : type == GGQ_Q4_0 ? kSmQ40 : type == GGQ_Q6_K ? kSmQ6 : kSmQ8;
    const bool bytes = kind != kSmQ8;   // 144- and 210-byte units as bytes; Q8_0 periods as 2-byte elements
    const int64_t row_bytes = cols / 256 * (kind == kSmQ8 ? 272 : kind == kSmQ6 ? 210 : 144);
    CUtensorMap wmap;
    cuuint64_t dims[2] = {(cuuint64_t)(bytes ? row_bytes : row_bytes / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    // Q6_K: 240 bytes from the 16-byte boundary below each super-block cover its
    // 210 (a box past the row's end reads zeros)
    cuuint32_t box[2] = {(cuuint32_t)(kind == kSmQ8 ? 136 : kind == kSmQ6 ? 240 : 144), (cuuint32_t)kTileRows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(&wmap, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                     const_cast<void*>(W), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GGQ_ECUDA, "tensor map (W) failed (%d)", (int)r);
    SmallParams p = {};
    p.x = x;
    p.y = y;
    p.rows = (int)rows;
    p.cols = (int)cols;
    p.M = M;
    p.status = device_status_word();
    if (!p.status) return fail(GGQ_ECUDA, "device status word unavailable");
    // Split tiles of a partly filled wave along K: halves when they fit the SMs
    // twice over, else (one wave of more than half the SMs) a big part of sb_big
    // 256-column blocks a tile and small parts, k_small a CTA, with sb_big the
    // least for which R + ceil(R / k_small) CTAs fit the SMs.
    int dev = 0, nsm = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int T = (int)((rows + kTileRows - 1) / kTileRows);
    const int S = (int)(cols / 256);
    const int R = T > nsm ? T % nsm : T;
    int grid = T;
    if (R > 0 && S >= 2) {
        if (2 * R <= nsm) {
            p.nsplit = R;
            grid = T + R;
        } else if (R == T) {
            for (int B = (S * R + nsm - 1) / nsm; B <= S - 1; ++B) {
                const int k = std::min(B / (S - B), kMaxPieces);
                if (k >= 1 && R + (R + k - 1) / k <= nsm) {
                    p.nsplit = R;
                    p.sb_big = B;
                    p.k_small = k;
                    grid = R + (R + k - 1) / k;
                    break;
                }
            }
        }
    }
    p.full_tiles = T - p.nsplit;
    if (p.nsplit > 0) {   // split tiles add both parts into a zeroed y
        cudaError_t e = cudaMemsetAsync(y, 0, sizeof(float) * (size_t)M * (size_t)rows, stream);
        if (e != cudaSuccess) return cuda_fail(e, "small-M: zero y");
    }
    if (kind == kSmQ4K) return launch_t<kSmQ4K>(wmap, p, grid, stream);
    if (kind == kSmQ40) return launch_t<kSmQ40>(wmap, p, grid, stream);
    if (kind == kSmQ6) return launch_t<kSmQ6>(wmap, p, grid, stream);
    return launch_t<kSmQ8>(wmap, p, grid, stream);
}

}  // namespace ggq
