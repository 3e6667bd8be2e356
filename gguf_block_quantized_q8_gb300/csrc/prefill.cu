// Prefill dequant-GEMM on the tcgen05 tensor cores:  Y[M, rows] = X[M, cols] * W^T.
//
// "GGUF Inferencer in R" section 4: prefill takes the whole prompt through each
// weight matrix as one large matrix product.  W is Q4_K ("GGUF: The File
// Format...", k-quant paragraph of "How a Q8_0 block is stored"): 256 weights per
// 144-byte super-block, w = d*sc_j*q - dmin*m_j; or Q8_0 (same section): 34-byte
// blocks of an fp16 d and 32 int8 q, w = d*q, staged 8 blocks (272 bytes, 256
// columns) at a time like a super-block.  X is bf16.
//
// One CTA computes a 128 (W rows) x 256 TH (tokens) tile of Y^T in tensor
// memory, TH = 2 for Q4_K when M is a multiple of 512 (each decoded W tile then
// feeds both token halves: every weight is decoded once for 512 tokens), else 1
// (tiles of the last, partly filled wave as two halves along K, see
// g_split_sync):
//   warp 0      TMA producer: raw Q4_K super-blocks [128 rows x 144 B] and X tiles
//               [256 tokens x 64 k] per token half (128-byte swizzle) into
//               shared-memory rings;
//   warp 1      allocates 256 TH TMEM columns; one thread issues tcgen05.mma
//               (kind::f16, bf16 x bf16 -> fp32, M=128, N=256, K=16) per 16 k and
//               token half, and commits each stage back to its "empty" barrier;
//   warps 2..   decoders (4 or 8 warps, see Dec): one or two threads per W row;
//               each 64-k stage decodes the row's weights exactly in fp32,
//               rounds them to bf16 and writes them in the canonical K-major
//               128-byte-swizzle layout the MMA reads; afterwards the same warps
//               read the accumulator (tcgen05.ld) and store Y (each warp may only
//               reach its own quarter of the 128 TMEM lanes).
// Every wait is bounded (ptx.cuh: mbar_wait); a timeout is recorded in the device
// status word and the kernel runs to completion without the data.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ggq_internal.h"
#include "ptx.cuh"

namespace ggq {

namespace {

constexpr int kTileRows = 128;        // UMMA M (W rows)
constexpr int kTileTok = 256;         // UMMA N (tokens): one token half of a tile
constexpr int kKStage = 64;           // k per stage of one-half tiles: one 128-byte swizzle row of bf16
constexpr int kRawStages = 2;
template <bool Q4K>
struct Raw {   // one 256-column block column of a 128-row tile: Q4_K super-blocks or Q8_0 periods
    static constexpr int kRowBytes = Q4K ? 144 : 272;
    static constexpr int kBytes = kTileRows * kRowBytes;
};
constexpr int kRawBytes = Raw<false>::kBytes;            // the larger of the two: the ring's slot
// Decoder warps 2 .. 2 + kDecWarps - 1: kParts threads per W row, each
// decoding its share of a stage's 64 k (kParts = 2: the low- or high-nibble
// half of Q4_K, one of the two Q8_0 blocks), then reading their TMEM lane
// quarter's share of the accumulator columns in the epilogue.  Eight warps
// where the decode sets the pace (Q8_0; tiles of 256 tokens), four for Q4_K
// tiles of 512 tokens (measured faster there).
template <bool Q4K, int TH>
struct Dec {
    static constexpr int kDecWarps = Q4K && TH == 2 ? 4 : 8;
    static constexpr int kDecoders = 32 * kDecWarps;
    static constexpr int kParts = kDecWarps / 4;
    static constexpr int kThreads = 64 + kDecoders;
};

// A tile is 128 W rows x TH token halves of 256 (TH = 1 or 2).  With TH = 2
// each decoded W tile feeds two MMAs (one per half) into a 512-column TMEM
// accumulator: every weight is decoded once for 512 tokens.  Its B stages take
// 64 KB, so the ring is two stages deep (three for TH = 1); the raw weight
// ring holds Q4_K super-blocks (18 KB a slot), so TH = 2 is for Q4_K (Q8_0's
// 34 KB periods leave no room: it keeps TH = 1).
template <bool Q4K, int TH>
struct Tile {
    static constexpr int kTok = kTileTok * TH;
    static constexpr int kKS = kKStage;                      // k per stage
    static constexpr int kSPS = 256 / kKS;                   // stages per 256-column block
    static constexpr int kRowB = kKS * 2;                    // bytes of a swizzled A / B row
    static constexpr int kStages = TH == 2 ? 2 : 3;
    static constexpr int kABytes = kTileRows * kRowB;
    static constexpr int kHalfBBytes = kTileTok * kRowB;
    static constexpr int kBBytes = kHalfBBytes * TH;
    static constexpr int kTmemCols = kTileTok * TH;
    static constexpr int kRawSlot = TH == 2 ? Raw<true>::kBytes : kRawBytes;
    static constexpr size_t kSmemBytes = (size_t)kStages * (kABytes + kBBytes) + (size_t)kRawStages * kRawSlot +
                                         1024 /* alignment */ + 256 /* barriers */;
};
static_assert(Tile<true, 2>::kSmemBytes <= 227 * 1024, "two-half Q4_K tiles fit shared memory");

// The last, partly filled wave of tiles is split in two along K (whole
// super-block columns): two CTAs compute halves of one tile.  The first to
// finish stores its half and raises the tile's flag; the second waits for the
// flag (its partner is already storing), adds its half to Y and resets the
// tile's counter and flag for the next launch.  Two terms: the same fp32 sum
// whichever finishes first.
constexpr int kMaxSplit = 256;
__device__ int g_split_sync[2 * kMaxSplit];   // [counter, flag] per split tile, zero between launches

struct PrefillParams {
    float* Y;
    int* split;      // g_split_sync
    int full_tiles;  // tiles computed whole (CTAs 0 .. full_tiles-1); the rest as halves
    int rows;        // W rows (Y columns)
    int cols;        // K
    int M;           // tokens
    int tok_tiles;   // M / (256 * TH) (rounded up)
    int* status;
};

// ------------------------------------------------------------- tcgen05 wrappers

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

// D[tmem] (+)= A[smem desc] * B[smem desc]^T
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive on `bar` once every tcgen05 operation issued so far by this thread is done
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 TMEM lanes x 16 consecutive 32-bit columns -> 16 registers per thread
// 64 accumulator columns of the warp's 32 TMEM lanes: one load, one wait
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B
// apart (stride byte offset), leading byte offset unused for this layout (1),
// descriptor version 1, base offset 0 (tiles are 1024-byte aligned).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTileTok >> 3) << 17) |
                            ((uint32_t)(kTileRows >> 4) << 24);

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// 6-bit scale and min of sub-block j from the 12 packed bytes (three words)
__device__ __forceinline__ void q4k_scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int j, int& sc, int& m) {
    if (j < 4) {
        sc = (s0 >> (8 * j)) & 63;
        m = (s1 >> (8 * j)) & 63;
    } else {
        const int k = j - 4;
        sc = ((s2 >> (8 * k)) & 15) | (((s0 >> (8 * k + 6)) & 3) << 4);
        m = ((s2 >> (8 * k + 4)) & 15) | (((s1 >> (8 * k + 6)) & 3) << 4);
    }
}

// ------------------------------------------------------------------- kernel

__device__ __forceinline__ void st_relaxed_i32(int* p, int v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_add_i32(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_i32(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait (bounded) until *flag != 0: the partner half of a split tile has stored.
__device__ __forceinline__ void wait_flag(const int* flag, int* status) {
    if (ld_acquire_i32(flag)) return;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ld_acquire_i32(flag)) return;
        if ((it & 15u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, kStatusTimeout);
            return;
        }
    }
}

template <bool Q4K, int TH>
__global__ void __launch_bounds__(Dec<Q4K, TH>::kThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap wmap,
                                                              const __grid_constant__ CUtensorMap xmap,
                                                              const PrefillParams p) {
    using RB = Raw<Q4K>;
    using TL = Tile<Q4K, TH>;
    constexpr int kDecoders = Dec<Q4K, TH>::kDecoders, kParts = Dec<Q4K, TH>::kParts;
    static_assert(Q4K || TH == 1, "two token halves per tile for Q4_K only");
    constexpr int kRawSlot = TL::kRawSlot;
    constexpr int kKS = TL::kKS, kSPS = TL::kSPS, kABytes = TL::kABytes, kHalfBBytes = TL::kHalfBBytes;
    auto desc = [](uint32_t addr) { return sw128_desc(addr); };
    constexpr int kStages = TL::kStages;
    constexpr int kBBytes = TL::kBBytes;
    constexpr int kTmemCols = TL::kTmemCols;
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // work item: a whole tile, or half of one (super-blocks [sb0, sb1))
    const int nsb_all = p.cols / 256;
    const bool split = (int)blockIdx.x >= p.full_tiles;
    const int part = split ? ((int)blockIdx.x - p.full_tiles) & 1 : 0;
    const int split_idx = split ? ((int)blockIdx.x - p.full_tiles) >> 1 : 0;
    const int tile = split ? p.full_tiles + split_idx : (int)blockIdx.x;
    const int sb0 = split && part ? nsb_all / 2 : 0;
    const int sb1 = split && !part ? nsb_all / 2 : nsb_all;
    const int row_tile = tile / p.tok_tiles;
    const int tok_tile = tile % p.tok_tiles;
    const int row0 = row_tile * kTileRows;
    const int tok0 = tok_tile * TL::kTok;
    const int ks0 = kSPS * sb0;
    const int nks = kSPS * (sb1 - sb0);   // k stages of this item (local index i: global stage ks0 + i)
    const int nsb = sb1 - sb0;            // super-blocks of this item

    // 1024-aligned carve-out
    const uint32_t base_u32 = smem_u32(smem_raw);
    uint8_t* base = smem_raw + (((base_u32 + 1023u) & ~1023u) - base_u32);
    uint8_t* sB = base;                                      // kStages x TH x (16 or 32 KB)
    uint8_t* sA = sB + (size_t)kStages * kBBytes;            // kStages x (8 or 16 KB)
    uint8_t* sRaw = sA + (size_t)kStages * kABytes;          // kRawStages x 18 KB
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRaw + (size_t)kRawStages * kRawSlot);
    // B (X) stages are filled and freed per token half: the MMAs of half 0 of a
    // stage are issued and committed before those of half 1, so its half-0
    // buffer is refilled half a stage earlier (the next X load has that much
    // more time to arrive)
    uint64_t* full_b = bars;                     // [kStages][TH]
    uint64_t* empty_b = bars + kStages * TH;     // [kStages][TH]
    uint64_t* full_a = bars + 2 * kStages * TH;  // [kStages]
    uint64_t* empty = full_a + kStages;          // [kStages]: the A (decoded W) slot
    uint64_t* full_raw = empty + kStages;        // [kRawStages]
    uint64_t* empty_raw = full_raw + kRawStages; // [kRawStages]
    uint64_t* acc_full = empty_raw + kRawStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

    if (threadIdx.x == 0) {
        prefetch_tensormap(&wmap);
        prefetch_tensormap(&xmap);
        for (int s = 0; s < kStages; ++s) {
            for (int h = 0; h < TH; ++h) {
                mbar_init(&full_b[s * TH + h], 1);
                mbar_init(&empty_b[s * TH + h], 1);
            }
            mbar_init(&full_a[s], kDecoders);
            mbar_init(&empty[s], 1);
        }
        for (int r = 0; r < kRawStages; ++r) {
            mbar_init(&full_raw[r], 1);
            mbar_init(&empty_raw[r], kDecoders);
        }
        mbar_init(acc_full, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            pdl_wait();   // X may come from the previous kernel in the stream
            for (int ks = 0; ks < nks; ++ks) {   // local stage index
                if (ks % kSPS == 0) {
                    const int sb = ks / kSPS, r = sb % kRawStages;
                    mbar_wait(&empty_raw[r], ((sb / kRawStages) & 1) ^ 1, p.status);
                    mbar_arrive_expect_tx(&full_raw[r], RB::kBytes);
                    // Q4_K map: 1-byte elements; Q8_0 map: 2-byte elements (136 a period)
                    tma_load_2d(sRaw + (size_t)r * kRawSlot, &wmap, &full_raw[r], (sb0 + sb) * (Q4K ? 144 : 136),
                                row0);
                }
                const int s = ks % kStages;
#pragma unroll
                for (int h = 0; h < TH; ++h) {   // tokens beyond M read as zeros
                    mbar_wait(&empty_b[s * TH + h], ((ks / kStages) & 1) ^ 1, p.status);
                    mbar_arrive_expect_tx(&full_b[s * TH + h], kHalfBBytes);
                    tma_load_2d(sB + (size_t)s * kBBytes + (size_t)h * kHalfBBytes, &xmap, &full_b[s * TH + h],
                                (ks0 + ks) * kKS, tok0 + h * kTileTok);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            for (int ks = 0; ks < nks; ++ks) {
                const int s = ks % kStages;
                const uint32_t ph = (ks / kStages) & 1;
                mbar_wait(&full_a[s], ph, p.status);
                const uint32_t a_addr = smem_u32(sA + (size_t)s * kABytes);
                const uint32_t b_addr = smem_u32(sB + (size_t)s * kBBytes);
#pragma unroll
                for (int h = 0; h < TH; ++h) {   // token half h: accumulator columns 256 h ..
                    mbar_wait(&full_b[s * TH + h], ph, p.status);
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kKS / 16; ++kk)   // 16 bf16 = 32 bytes further along the swizzled rows
                        umma_bf16(tmem + (uint32_t)(h * kTileTok), desc(a_addr + 32 * kk),
                                  desc(b_addr + (uint32_t)(h * kHalfBBytes) + 32 * kk), kIdesc, (ks | kk) != 0);
                    umma_commit(&empty_b[s * TH + h]);
                }
                umma_commit(&empty[s]);
            }
            umma_commit(acc_full);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ decoders (warps 2..)
        const int t = (threadIdx.x - 64) & (kTileRows - 1);   // W row within the tile
        const int part = (threadIdx.x - 64) >> 7;             // share of the row's k (kParts > 1)
        for (int sb = 0; sb < nsb; ++sb) {
            const int r = sb % kRawStages;
            mbar_wait(&full_raw[r], (sb / kRawStages) & 1, p.status);
            const uint8_t* rp = sRaw + (size_t)r * kRawSlot + (size_t)t * RB::kRowBytes;
            if constexpr (Q4K) {
            const uint4 h = *reinterpret_cast<const uint4*>(rp);
            const float d = half_bits_to_float(h.x), dmin = half_bits_to_float(h.x >> 16);
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                int sc_lo, m_lo, sc_hi, m_hi;
                q4k_scale_min(h.y, h.z, h.w, 2 * c, sc_lo, m_lo);
                q4k_scale_min(h.y, h.z, h.w, 2 * c + 1, sc_hi, m_hi);
                const float a_lo = d * (float)sc_lo, b_lo = dmin * (float)m_lo;
                const float a_hi = d * (float)sc_hi, b_hi = dmin * (float)m_hi;
                const uint4 q0 = *reinterpret_cast<const uint4*>(rp + 16 + 32 * c);
                const uint4 q1 = *reinterpret_cast<const uint4*>(rp + 32 + 32 * c);
                const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                // chunk j (k = 8j .. 8j+7 of the 64): low nibbles, sub-block 2c;
                // high nibbles, sub-block 2c+1, are k = 32 + 8j ..  Four nibbles
                // of a word are masked at once; byte b then goes under 0x4B0000
                // (the float 2^23 + q), and pairs take packed arithmetic:
                // w = a * q - b, exactly as one fma each.
                uint32_t lo[4][4], hi[4][4];
                auto four = [](uint32_t n4, float a, float nb, uint32_t& p01, uint32_t& p23) {
                    const float2 k = make_float2(-8388608.0f, -8388608.0f);
                    const float2 a2 = make_float2(a, a), nb2 = make_float2(nb, nb);
                    const float2 f01 = __ffma2_rn(__fadd2_rn(make_float2(__uint_as_float(__byte_perm(n4, 0x4B000000u, 0x7650)),
                                                                         __uint_as_float(__byte_perm(n4, 0x4B000000u, 0x7651))), k),
                                                  a2, nb2);
                    const float2 f23 = __ffma2_rn(__fadd2_rn(make_float2(__uint_as_float(__byte_perm(n4, 0x4B000000u, 0x7652)),
                                                                         __uint_as_float(__byte_perm(n4, 0x4B000000u, 0x7653))), k),
                                                  a2, nb2);
                    p01 = pack_bf16x2(f01.x, f01.y);
                    p23 = pack_bf16x2(f23.x, f23.y);
                };
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const uint32_t w = qw[2 * j + half];
                        if (kParts == 1 || part == 0)
                            four(w & 0x0F0F0F0Fu, a_lo, -b_lo, lo[j][2 * half], lo[j][2 * half + 1]);
                        if (kParts == 1 || part == 1)
                            four((w >> 4) & 0x0F0F0F0Fu, a_hi, -b_hi, hi[j][2 * half], hi[j][2 * half + 1]);
                    }
                }
                // one 64-k stage: a 128-byte row, chunk position j ^ (row % 8)
                const int ks = sb * 4 + c;
                const int s = ks % kStages;
                mbar_wait(&empty[s], ((ks / kStages) & 1) ^ 1, p.status);
                uint8_t* arow = sA + (size_t)s * kABytes + (size_t)t * 128;
                const int sw = t & 7;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (kParts == 1 || part == 0)
                        *reinterpret_cast<uint4*>(arow + ((j ^ sw) << 4)) =
                            make_uint4(lo[j][0], lo[j][1], lo[j][2], lo[j][3]);
                    if (kParts == 1 || part == 1)
                        *reinterpret_cast<uint4*>(arow + (((j + 4) ^ sw) << 4)) =
                            make_uint4(hi[j][0], hi[j][1], hi[j][2], hi[j][3]);
                }
                fence_proxy_async_smem();
                mbar_arrive(&full_a[s]);
            }
            } else {
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                // Q8_0: stage c holds blocks 2c (k = 0..31) and 2c+1 (k = 32..63) of
                // the row's 272-byte period, each an fp16 d and 32 int8 q; w = d*q
                // is exact in fp32, then rounded to bf16
                const int ks = sb * 4 + c;
                const int s = ks % kStages;
                uint32_t u[2][8];   // the 32 q bytes of each block, four a word
                float d[2];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    if (kParts == 2 && h2 != part) continue;
                    const int off = 34 * (2 * c + h2);   // 2-byte aligned; q bytes at off + 2
                    d[h2] = half_bits_to_float(*reinterpret_cast<const uint16_t*>(rp + off));
                    const int qo = off + 2;
                    const uint32_t* wp = reinterpret_cast<const uint32_t*>(rp + (qo & ~3));
                    const int sh = 8 * (qo & 3);        // 0 or 16
                    uint32_t v[9];
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = wp[i];
                    v[8] = sh ? wp[8] : 0u;             // only a misaligned start reaches a ninth word
#pragma unroll
                    for (int i = 0; i < 8; ++i) u[h2][i] = __funnelshift_r(v[i], v[i + 1], sh);
                }
                mbar_wait(&empty[s], ((ks / kStages) & 1) ^ 1, p.status);
                uint8_t* arow = sA + (size_t)s * kABytes + (size_t)t * 128;
                const int sw = t & 7;
#pragma unroll
                for (int j = 0; j < 8; ++j) {   // chunk j: k = 8j..8j+7 (block 2c + j/4)
                    const int h2 = j >> 2;
                    if (kParts == 2 && h2 != part) continue;
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        // q + 128 under 0x4B0000 is the float 2^23 + 128 + q: q
                        // exactly after one subtraction, then w = d * q
                        const uint32_t w = u[h2][2 * (j & 3) + (e >> 1)] ^ 0x80808080u;
                        const uint32_t b0 = 2 * (e & 1);
                        const float2 qf = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7650u | b0)),
                                                                 __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7651u | b0))),
                                                     make_float2(-8388736.0f, -8388736.0f));
                        const float2 f = __fmul2_rn(qf, make_float2(d[h2], d[h2]));
                        o[e] = pack_bf16x2(f.x, f.y);
                    }
                    *reinterpret_cast<uint4*>(arow + ((j ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                fence_proxy_async_smem();
                mbar_arrive(&full_a[s]);
            }
            }
            mbar_arrive(&empty_raw[r]);
        }

        // ------------------------------------------------------------ epilogue
        mbar_wait(acc_full, 0, p.status);
        tc_fence_after();
        const int q = warp & 3;                  // TMEM lane quarter of this warp
        constexpr int kCols = TL::kTok / kParts;  // accumulator columns this warp reads
        const int col0 = ((warp - 2) >> 2) * kCols;
        const int row = row0 + 32 * q + lane;
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16);
        // half of a split tile: the first half done stores, the second adds
        // (after the first's stores are visible: flag, release / acquire)
        bool add = false;
        int* cnt = p.split + 2 * split_idx;
        __shared__ int s_role;
        if (split) {
            if (threadIdx.x == 64) s_role = atomicAdd(cnt, 1);
            asm volatile("bar.sync 1, %0;" ::"n"(kDecoders) : "memory");   // the epilogue threads
            add = s_role != 0;
            if (add) {
                if (threadIdx.x == 64) wait_flag(cnt + 1, p.status);
                asm volatile("bar.sync 1, %0;" ::"n"(kDecoders) : "memory");
            }
        }
        static_assert(kCols % 64 == 0, "the epilogue reads 64 accumulator columns at a time");
        for (int col = col0; col < col0 + kCols; col += 64) {
            float v[64];
            tmem_ld64(taddr + (uint32_t)col, v);
            if (add) {
                // every old value of the 64 tokens is read before any is written
                // (one L2 round trip a step, not one per token)
                float old[64];
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const int tok = tok0 + col + i;
                    old[i] = tok < p.M ? __ldcg(p.Y + (size_t)tok * p.rows + row) : 0.0f;
                }
#pragma unroll
                for (int i = 0; i < 64; ++i) v[i] += old[i];
            }
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const int tok = tok0 + col + i;
                if (tok < p.M) p.Y[(size_t)tok * p.rows + row] = v[i];
            }
        }
        if (split) {
            asm volatile("bar.sync 1, %0;" ::"n"(kDecoders) : "memory");
            if (threadIdx.x == 64) {
                if (add) {   // both halves done: reset for the next launch
                    st_relaxed_i32(cnt, 0);
                    st_relaxed_i32(cnt + 1, 0);
                } else {
                    red_release_add_i32(cnt + 1, 1);   // this half's stores, then the flag
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

}  // namespace

int launch_prefill(int type, const void* W, int64_t rows, int64_t cols, const uint16_t* X, float* Y, int M,
                   cudaStream_t stream) {
    const bool q4k = type == GGQ_Q4_K;
    auto enc = encoder();
    if (!enc) return fail(GGQ_ECUDA, "cuTensorMapEncodeTiled unavailable");
    CUtensorMap wmap, xmap;
    {
        // Q4_K: 144-byte super-blocks as bytes; Q8_0: 272-byte periods of 8 blocks
        // as 2-byte elements (136 a period)
        const int64_t rb = cols / 256 * (q4k ? 144 : 272);
        cuuint64_t dims[2] = {(cuuint64_t)(q4k ? rb : rb / 2), (cuuint64_t)rows};
        cuuint64_t strides[1] = {(cuuint64_t)rb};
        cuuint32_t box[2] = {(cuuint32_t)(q4k ? 144 : 136), kTileRows};
        cuuint32_t es[2] = {1, 1};
        CUresult r = enc(&wmap, q4k ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                         const_cast<void*>(W), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(GGQ_ECUDA, "tensor map (W) failed (%d)", (int)r);
    }
    // two token halves per tile (each weight decoded once for 512 tokens)
    // when M is a multiple of 512, else one
    const int th = q4k && M % (2 * kTileTok) == 0 ? 2 : 1;
    {
        cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)M};
        cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
        cuuint32_t box[2] = {(cuuint32_t)kKStage, kTileTok};
        cuuint32_t es[2] = {1, 1};
        CUresult r = enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(X), dims, strides, box,
                         es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(GGQ_ECUDA, "tensor map (X) failed (%d)", (int)r);
    }
    PrefillParams p = {};
    p.Y = Y;
    p.rows = (int)rows;
    p.cols = (int)cols;
    p.M = M;
    p.tok_tiles = (M + th * kTileTok - 1) / (th * kTileTok);
    p.status = device_status_word();
    if (!p.status) return fail(GGQ_ECUDA, "device status word unavailable");
    {
        void* sp = nullptr;
        cudaError_t e2 = cudaGetSymbolAddress(&sp, g_split_sync);
        if (e2 != cudaSuccess) return cuda_fail(e2, "split-tile sync words");
        p.split = static_cast<int*>(sp);
    }
    // tiles in the last, partly filled wave (all tiles if they fill at most half
    // of the SMs) are computed as two halves along K when the halves fit one wave
    int dev = 0, nsm = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int T = (int)(rows / kTileRows) * p.tok_tiles;
    const int R = T > nsm ? T % nsm : T;
    const int nsplit = (R > 0 && 2 * R <= nsm && R <= kMaxSplit && cols >= 512) ? R : 0;
    p.full_tiles = T - nsplit;

    auto kernel = q4k ? (th == 2 ? prefill_kernel<true, 2> : prefill_kernel<true, 1>) : prefill_kernel<false, 1>;
    const size_t smem = q4k ? (th == 2 ? Tile<true, 2>::kSmemBytes : Tile<true, 1>::kSmemBytes)
                            : Tile<false, 1>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.full_tiles + 2 * nsplit));
    cfg.blockDim = dim3(q4k && th == 2 ? Dec<true, 2>::kThreads : q4k ? Dec<true, 1>::kThreads
                                                                     : Dec<false, 1>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, wmap, xmap, p);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return GGQ_OK;
}

// Zero the split-tile counters and flags (after a timeout left them set).
int reset_prefill_sync() {
    static const int zero[2 * kMaxSplit] = {};
    cudaError_t e = cudaMemcpyToSymbol(g_split_sync, zero, sizeof(zero));
    return e == cudaSuccess ? GGQ_OK : cuda_fail(e, "reset split-tile sync words");
}

}  // namespace ggq
