// Fused prefill: out = x . W + bias with W read packed (4 bits per weight)
// and dequantized in shared memory inside the main loop; the dense matrix is
// never written to HBM ("GPTQ's 'Exllama Kernel Not Installed' Warning",
// "What the fallback actually does": the fused route reads packed weights and
// never materializes the dequantized matrix).  fp32 accumulation, bias added
// to the fp32 sum before the single rounding to fp16 ("Inference Backends",
// "Numeric epilogues and input gradients").
//
// Persistent kernel, one CTA per SM.  Work: BM x BN output tiles taken round
// robin (m fastest, so the CTAs working at the same time share weight tiles
// in L2) when there are enough of them; otherwise stream-K (cooperative
// launch, bounded waits): every tile cut into equal k ranges, one CTA each,
// whose CTAs each finish a share of its rows after the main loop; or every
// CTA one contiguous range of the tiles x k-blocks space, each tile cut at
// range ends finished by the CTA holding its first k blocks, which keeps
// them in tensor memory and adds the other pieces after its main loop.
// Roles, for BN = 256 (BM = 128 or 256):
//
//   warp 0       one thread: TMA loads of the packed-word stages (8 KB of
//                packed words per 64 rows) with their scale pairs and zero
//                words, a 4-slot ring
//   warp 1       allocates TMEM (two 128x256 fp32 accumulators at BM = 128,
//                one 256x256 pair at BM = 256); one thread issues tcgen05.mma
//                M=128 N=256 K=16 (two per k step at BM = 256, sharing the B
//                tile) and commits each stage back to the x producer and the
//                dequantizers
//   warp 2       one thread: TMA loads of the x tiles (BM x 64 fp16, 128-byte
//                swizzle), a 5-slot ring at BM = 128, 3 at BM = 256
//   warp 3       waits for each stage's x and B tiles and hands the stage to
//                warp 1 through a named barrier
//   warps 4-19   dequantize each packed stage into the fp16 B ring (3 slots
//                at BM = 128, 2 at BM = 256; K-major, 128-byte swizzle: the
//                UMMA operand layout), w16 = fp16(s * (q - z - 1)) rounded
//                once, unpacked and scaled before its B slot is free; at
//                BM = 256 every warp takes one n16 tile of every stage, at
//                BM = 128 two groups of eight warps take alternate stages,
//                two n16 tiles per warp
//   warps 20-23  epilogue: tcgen05.ld an accumulator, add bias, round to fp16,
//                store (or write a stream-K piece's fp32 partial); then hand
//                the accumulator back, so the epilogue of one tile overlaps
//                the main loop of the next.
//
// Up to 64 rows of x a stage is 128 rows of K instead of 64 (two 64-row
// chunks; x tiles of 64 rows, whose shared memory pays for the 64 KB B
// stages), and every dequantizer takes one n16 tile of both chunks.
//
// Every mbarrier wait is bounded (~2 s); a wait that runs out records an
// error bit in the handle's status word, the CTA lets its copies land, frees
// its TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>
#include <cstdint>

#include "q4_internal.cuh"
#include "q4_tc.cuh"

// Ring depths (stages): x tiles, packed words, fp16 B tiles, per tile height.
#ifndef Q4_PF_SX128
#define Q4_PF_SX128 5
#endif
#ifndef Q4_PF_SB128
#define Q4_PF_SB128 3
#endif
#ifndef Q4_PF_SX256
#define Q4_PF_SX256 3
#endif
#ifndef Q4_PF_SB256
#define Q4_PF_SB256 2
#endif
#ifndef Q4_PF_SP
#define Q4_PF_SP 4
#endif
// most rows of x for which 128-row stages are used, and their x and packed rings
#ifndef Q4_PF_BK128_MAXM
#define Q4_PF_BK128_MAXM 64
#endif
#ifndef Q4_PF_SXK128
#define Q4_PF_SXK128 2
#endif
#ifndef Q4_PF_SPK128
#define Q4_PF_SPK128 3
#endif

namespace q4 {

cudaError_t encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *ptr, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

namespace {

using namespace tc;

constexpr int kEpiWarps = 4;
// Stream-K pieces.  With one range per CTA over the tiles x k-blocks space,
// a tile is cut into at most three pieces, and all but piece 0 (the tile's
// first k blocks, the last unit of its CTA's range) are the first units of
// their CTAs' ranges, written as soon as they are done (mid-loop unless the
// range ends inside the same tile): the CTA holding piece 0 keeps it in
// tensor memory and finishes the tile, adding the others
// (8192 x 28672 at M = 256-512, 4096 x 11008 and 8192 x 10240 at M = 1024:
// 5-12 % faster than every piece's CTA summing a share of the rows).  With
// the even K split every piece ends at the same time, one reader per tile is
// slower (4096 x 4096 at M = 1024: 43.3 against 39.6 us), and the pieces'
// CTAs share the sum.
constexpr int kFinishMax = 3;

// Per tile BM x BN: BN = 256, or 128 where 256-wide tiles leave SMs idle (one
// dequant warp per 16 columns); BM = 128, or 256 (two M = 128 MMAs per k step
// on the same fp16 B tile, halving the dequantization per flop, with the one
// accumulator pair filling tensor memory) when there are tiles enough.
// Three rings, per stage of BK rows of K (64, or 128 up to 64 rows of x): x
// tiles (BM x 64 fp16 per 64-row chunk, 128-byte swizzle), packed-word stages
// {packed words BN*32 B per chunk, scale pairs of up to BK/32 groups (BN*2 B
// each), their zero words (BN/2 B each)}, and fp16 B tiles (K-major, 128-byte
// swizzle, one BN x 64 sub-tile per chunk).
template <int BM_, int BN_, int BK_ = 64>
struct PfCfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_;
    static_assert(BK == 64 || (BK == 128 && BM == 128), "128-row stages: 128-row tiles only");
    static constexpr int kKC = BK / 64;                // 64-row chunks per stage
    static constexpr int kBlk = BK / 32;               // 32-row blocks per stage
    // 128-row stages serve M <= 64: x tiles of 64 rows (the MMA's rows 64..127
    // read whatever follows in shared memory and are never stored)
    static constexpr int kXRows = BK == 128 ? 64 : BM;
    static constexpr int kHalves = BM / 128;           // M = 128 MMAs per k step
    static constexpr int kAccBufs = BM == 128 ? 2 : 1; // accumulator sets (double-buffered when they fit)
    static constexpr int kSX = BK == 128 ? Q4_PF_SXK128 : (BM == 128 ? Q4_PF_SX128 : Q4_PF_SX256);   // x-tile ring (released by the MMAs)
    static constexpr int kSP = BK == 128 ? Q4_PF_SPK128 : Q4_PF_SP;   // packed-word ring (released by the dequantizers)
    static constexpr int kSB = BK == 128 ? 2 : (BM == 128 ? Q4_PF_SB128 : Q4_PF_SB256);   // fp16 B ring
    static constexpr int kXStage = kXRows * BK * 2;    // kKC sub-tiles of kXRows x 64
    static constexpr int kMaxG = kBlk;                 // groups a stage can touch (a group is whole blocks)
    static constexpr int kSGroup = BN * 2, kZGroup = BN / 2;
    static constexpr int kSzOff = BN * 32 * kKC;       // within a packed stage
    static constexpr int kZOff = kMaxG * kSGroup;      // zero words after all groups' scales
    static constexpr int kPStage = (kSzOff + kMaxG * (kSGroup + kZGroup) + 127) / 128 * 128;
    static constexpr int kBStage = BN * BK * 2;        // kKC sub-tiles of BN x 64
    static constexpr int kRingP = kSX * kXStage;
    static constexpr int kRingB = (kRingP + kSP * kPStage + 1023) / 1024 * 1024;
    static constexpr int kBarOff = kRingB + kSB * kBStage;
    static constexpr int kNumBars = 2 * kSX + 2 * kSP + 2 * kSB + 5;
    static constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + 1024;
    static constexpr int kDqWarps = BN / 16;
    // 128-row tiles: two dequant groups on alternate stages, two n16 tiles
    // per warp (measured 5-7 % faster there, 3 % slower with 256-row tiles);
    // 128-row stages: every warp one n16 tile of every stage, both chunks
    static constexpr int kDqGroups = BM == 128 && BK == 64 ? 2 : 1;
    static constexpr int kUnits = BK == 128 ? 2 : kDqGroups;   // (n16 tile, chunk) pairs per warp and stage
    static constexpr int kDqHalf = kDqWarps / kDqGroups;   // warps per dequant group
    static constexpr int kDq0 = 4;                     // first dequant warp
    static constexpr int kThreads = 32 * (kDq0 + kDqWarps + kEpiWarps);
    static constexpr uint32_t kTmemCols = kAccBufs * kHalves * BN;
    static_assert(kSmem <= 227 * 1024, "shared memory");
    static_assert(kTmemCols == 256 || kTmemCols == 512, "tensor memory");
};

struct PfArgs {
    int M, N, K;
    const uint16_t *bias;
    uint16_t *out;
    int *status;
    const uint32_t *s2;      // scale pairs [G][N/16][8]
    const uint32_t *zeros;   // zero words [G][N/8]
    int bpg;                 // 32-row blocks per group
    int tiles_m, tiles_n;
    int zero_offset;         // effective zero = stored + zero_offset
    int zsplit;              // groups [0, zsplit) take zero offset 0
    const float *rowscale;   // epilogue: y = acc * rowscale[m] + bias (NULL: 1)
    int out_bf16;            // output rounded to bf16 instead of fp16
    int sk;                  // 1: stream-K (every CTA one contiguous range of the (tile, k
                             // block) space, cooperative launch); 0: whole tiles round robin
    int pmax;                // stream-K: most pieces (CTAs) any tile is cut into
    int fin0;                // stream-K: piece 0's CTA finishes each cut tile (else all pieces' CTAs)
    float *ws;               // stream-K: fp32 partial tiles [tile][piece][BM][BN]
    int *tickets;            // one per tile, zero between calls
};

// One unit of a CTA's work: tile t, k blocks [kb0, kb1), piece p of the np
// pieces the tile is cut into (np = 1: the whole tile).
struct PfUnit {
    int t, kb0, kb1, p, np;
};

// The i-th unit of CTA c (false past the last).  Round robin: tile c + i G.
// Stream-K: the CTA's range [c W / G, (c + 1) W / G) of the W = tiles x KB
// (tile, k block) pairs, tile by tile; piece p of tile t is the CTA's index
// minus that of the first CTA whose range touches t.
__device__ __forceinline__ bool pf_unit(const PfArgs &a, int KB, int i, PfUnit &u) {
    const int G = gridDim.x, c = blockIdx.x;
    const int ntiles = a.tiles_m * a.tiles_n;
    if (!a.sk) {
        u.t = c + i * G;
        u.kb0 = 0;
        u.kb1 = KB;
        u.p = 0;
        u.np = 1;
        return u.t < ntiles;
    }
    const long long W = static_cast<long long>(ntiles) * KB;
    const long long w0 = c * W / G, w1 = (c + 1) * W / G;
    const int t = static_cast<int>(w0 / KB) + i;
    const long long tb = static_cast<long long>(t) * KB;
    if (tb >= w1 || w0 >= w1) return false;
    u.t = t;
    u.kb0 = static_cast<int>(w0 > tb ? w0 - tb : 0);
    u.kb1 = static_cast<int>(w1 < tb + KB ? w1 - tb : KB);
    auto owner = [&](long long w) { return static_cast<int>(((w + 1) * G - 1) / W); };
    const int f = owner(tb);
    u.p = c - f;
    u.np = owner(tb + KB - 1) - f + 1;
    return true;
}

__device__ __forceinline__ void fail(int *status, int bit, int *abort_flag) {
    if (status) atomicOr(status, bit);
    atomicExch(abort_flag, 1);
}
__device__ __forceinline__ bool aborted(int *abort_flag) { return *reinterpret_cast<volatile int *>(abort_flag) != 0; }

// 32 consecutive accumulator columns of one output row (one lane's share of
// a tensor-memory load), the first at column n: the row scale, bias and one
// rounding to fp16 or bf16, or the raw fp32 sums; columns at or past N are
// skipped.
template <bool BF>
__device__ __forceinline__ void store_row32_t(const PfArgs &a, int row, int n, const uint32_t (&r)[32]) {
    const float rs = BF && a.rowscale ? a.rowscale[row] : 1.f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int nv = n + 8 * v;
        if (nv < a.N) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pk[e] = out_pair_t<BF>(__uint_as_float(r[8 * v + 2 * e]), __uint_as_float(r[8 * v + 2 * e + 1]), rs,
                                       a.bias, nv + 2 * e);
            *reinterpret_cast<uint4 *>(a.out + static_cast<size_t>(row) * a.N + nv) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
    }
}
__device__ __forceinline__ void store_row32(const PfArgs &a, int row, int n, const uint32_t (&r)[32]) {
    if (a.out_bf16 == kOutF32) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int nv = n + 8 * v;
            if (nv < a.N) {
                float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.out) + static_cast<size_t>(row) * a.N + nv);
                dst[0] = make_float4(__uint_as_float(r[8 * v]), __uint_as_float(r[8 * v + 1]), __uint_as_float(r[8 * v + 2]),
                                     __uint_as_float(r[8 * v + 3]));
                dst[1] = make_float4(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]),
                                     __uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
            }
        }
    } else if (a.out_bf16) {
        store_row32_t<true>(a, row, n, r);
    } else {
        store_row32_t<false>(a, row, n, r);
    }
}
// The same for a warp's 32 rows (lane = row row0 + lane) through 2 KB of the
// warp's shared memory (16-byte slots XOR-swizzled by row pair: no bank
// conflicts either way), so that each store instruction writes 8 rows x 64
// contiguous bytes instead of 32 rows x 16 bytes: measured faster where many
// warps write at once (the stream-K finish), slower for the epilogue's four.
template <bool BF>
__device__ __forceinline__ void store_block16_t(const PfArgs &a, int row0, int n, const uint32_t (&r)[32], uint8_t *stage,
                                                int lane) {
    const int row = row0 + lane;
    const float rs = BF && a.rowscale && row < a.M ? a.rowscale[row] : 1.f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = n + 8 * v + 2 * e;
            pk[e] = c < a.N ? out_pair_t<BF>(__uint_as_float(r[8 * v + 2 * e]), __uint_as_float(r[8 * v + 2 * e + 1]), rs,
                                             a.bias, c)
                            : 0u;
        }
        *reinterpret_cast<uint4 *>(stage + lane * 64 + 16 * (v ^ ((lane >> 1) & 3))) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int rr = 8 * it + (lane >> 2), sg = lane & 3;
        const uint4 val = *reinterpret_cast<const uint4 *>(stage + rr * 64 + 16 * (sg ^ ((rr >> 1) & 3)));
        if (row0 + rr < a.M && n + 8 * sg < a.N)
            *reinterpret_cast<uint4 *>(a.out + static_cast<size_t>(row0 + rr) * a.N + n + 8 * sg) = val;
    }
    __syncwarp();
}
__device__ __forceinline__ void store_block(const PfArgs &a, int row0, int n, const uint32_t (&r)[32], uint8_t *stage,
                                            int lane) {
    if (a.out_bf16 == kOutF32) {
        float *out = reinterpret_cast<float *>(a.out);
#pragma unroll
        for (int h = 0; h < 2; ++h) {               // 16 columns (64 bytes) per round
#pragma unroll
            for (int v = 0; v < 4; ++v)
                *reinterpret_cast<uint4 *>(stage + lane * 64 + 16 * (v ^ ((lane >> 1) & 3))) =
                    make_uint4(r[16 * h + 4 * v], r[16 * h + 4 * v + 1], r[16 * h + 4 * v + 2], r[16 * h + 4 * v + 3]);
            __syncwarp();
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int rr = 8 * it + (lane >> 2), sg = lane & 3;
                const uint4 val = *reinterpret_cast<const uint4 *>(stage + rr * 64 + 16 * (sg ^ ((rr >> 1) & 3)));
                const int c = n + 16 * h + 4 * sg;
                if (row0 + rr < a.M && c < a.N)
                    *reinterpret_cast<uint4 *>(out + static_cast<size_t>(row0 + rr) * a.N + c) = val;
            }
            __syncwarp();
        }
    } else if (a.out_bf16) {
        store_block16_t<true>(a, row0, n, r, stage, lane);
    } else {
        store_block16_t<false>(a, row0, n, r, stage, lane);
    }
}

// Ring position: slot and the parity of its current phase.
struct RingPos {
    int s = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next(int n) {
        if (++s == n) {
            s = 0;
            ph ^= 1;
        }
    }
};

template <int BMT, int BNT, int BKT>
__global__ void __launch_bounds__(PfCfg<BMT, BNT, BKT>::kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, PfArgs a) {
    using P = PfCfg<BMT, BNT, BKT>;
    constexpr int BK = P::BK, kKC = P::kKC, kBlk = P::kBlk, kXRows = P::kXRows, kUnits = P::kUnits;
    constexpr int BM = P::BM, BN = P::BN, kSzOff = P::kSzOff, kZOff = P::kZOff;
    constexpr int kSX = P::kSX, kSP = P::kSP, kSB = P::kSB, kHalves = P::kHalves, kAccBufs = P::kAccBufs;
    constexpr int kXStage = P::kXStage, kPStage = P::kPStage, kBStage = P::kBStage;
    constexpr int kRingP = P::kRingP, kRingB = P::kRingB, kBarOff = P::kBarOff;
    constexpr int kNumBars = P::kNumBars, kDqWarps = P::kDqWarps, kDq0 = P::kDq0, kDqHalf = P::kDqHalf;
    constexpr int kDqGroups = P::kDqGroups;
    constexpr uint32_t kTmemCols = P::kTmemCols;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + kBarOff;
    auto fullX = [&](int s) { return bar0 + 8u * s; };
    auto emptyX = [&](int s) { return bar0 + 8u * (kSX + s); };
    auto fullP = [&](int s) { return bar0 + 8u * (2 * kSX + s); };
    auto emptyP = [&](int s) { return bar0 + 8u * (2 * kSX + kSP + s); };
    auto fullB = [&](int s) { return bar0 + 8u * (2 * kSX + 2 * kSP + s); };
    auto emptyB = [&](int s) { return bar0 + 8u * (2 * kSX + 2 * kSP + kSB + s); };
    auto accF = [&](int i) { return bar0 + 8u * (2 * kSX + 2 * kSP + 2 * kSB + i); };
    auto accE = [&](int i) { return bar0 + 8u * (2 * kSX + 2 * kSP + 2 * kSB + 2 + i); };
    const uint32_t stageB = bar0 + 8u * (2 * kSX + 2 * kSP + 2 * kSB + 4);   // stream-K pieces staged after the loop
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + kBarOff + kNumBars * 8);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = a.K / BK;
    const int NT16 = a.N >> 4;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSX; ++s) {
            mbar_init(fullX(s), 1);
            mbar_init(emptyX(s), 1);                 // the MMAs that read it
        }
        for (int s = 0; s < kSP; ++s) {
            mbar_init(fullP(s), 1);
            mbar_init(emptyP(s), kDqHalf);           // every warp of the stage's dequant group has read it
        }
        for (int s = 0; s < kSB; ++s) {
            mbar_init(fullB(s), kDqHalf);
            mbar_init(emptyB(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(accF(i), 1);
            mbar_init(accE(i), kEpiWarps);
        }
        mbar_init(stageB, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------ producer: packed words, scales, zeros
        if (lane == 0) {
            RingPos r;
            int issued = 0;
            bool ok = true;
            PfUnit un;
            for (int ui = 0; ok && pf_unit(a, KB, ui, un); ++ui) {
                const int t = un.t;
                const int kbeg = un.kb0, kend = un.kb1;
                const int nt0 = (t / a.tiles_m) * (BN / 16);
                const int tiles16 = min(BN / 16, NT16 - nt0);
                const uint32_t sbytes = tiles16 * 32u, zbytes = tiles16 * 8u;
                // group of the first 32-row block and the blocks left in it (itself included)
                int gcur = (kBlk * kbeg) / a.bpg, left = a.bpg - (kBlk * kbeg - gcur * a.bpg);
                for (int kb = kbeg; kb < kend; ++kb) {
                    if (aborted(abort_flag)) { ok = false; break; }
                    if (!mbar_wait(emptyP(r.s), r.ph ^ 1)) { fail(a.status, 0x10, abort_flag); ok = false; break; }
                    int g_first = gcur;
#pragma unroll
                    for (int b = 0; b < kBlk; ++b) {
                        if (left == 0) { ++gcur; left = a.bpg; }
                        if (b == 0) g_first = gcur;
                        --left;
                    }
                    const int ng = gcur - g_first + 1;
                    const uint32_t st = base + kRingP + r.s * kPStage;
                    mbar_arrive_expect_tx(fullP(r.s), BN * 32u * kKC + ng * (sbytes + zbytes));
                    tma_load_2d(st, &tmW, fullP(r.s), kb * 128 * kKC, nt0);
                    for (int gi = 0; gi < ng; ++gi) {
                        const size_t gr = static_cast<size_t>(g_first + gi);
                        bulk_load(st + kSzOff + gi * P::kSGroup, a.s2 + (gr * NT16 + nt0) * 8, sbytes, fullP(r.s));
                        bulk_load(st + kSzOff + kZOff + gi * P::kZGroup, a.zeros + gr * (a.N >> 3) + nt0 * 2, zbytes,
                                  fullP(r.s));
                    }
                    ++issued;
                    r.next(kSP);
                }
            }
            if (aborted(abort_flag))
                for (int j = issued > kSP ? issued - kSP : 0; j < issued; ++j) mbar_wait(fullP(j % kSP), (j / kSP) & 1);
        }
    } else if (warp == 2) {
        // ------------------------------------------ producer: x tiles
        if (lane == 0) {
            RingPos r;
            int issued = 0;
            bool ok = true;
            PfUnit un;
            for (int ui = 0; ok && pf_unit(a, KB, ui, un); ++ui) {
                const int t = un.t;
                const int kbeg = un.kb0, kend = un.kb1;
                const int m0 = (t % a.tiles_m) * BM;
                for (int kb = kbeg; kb < kend; ++kb) {
                    if (aborted(abort_flag)) { ok = false; break; }
                    if (!mbar_wait(emptyX(r.s), r.ph ^ 1)) { fail(a.status, 0x10, abort_flag); ok = false; break; }
                    mbar_arrive_expect_tx(fullX(r.s), static_cast<uint32_t>(kXStage));
#pragma unroll
                    for (int j = 0; j < kKC; ++j)
                        tma_load_2d(base + r.s * kXStage + j * kXRows * 128, &tmA, fullX(r.s), kb * BK + j * 64, m0);
                    ++issued;
                    r.next(kSX);
                }
            }
            if (aborted(abort_flag))
                for (int j = issued > kSX ? issued - kSX : 0; j < issued; ++j) mbar_wait(fullX(j % kSX), (j / kSX) & 1);
        }
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------- MMA issuer (warp 1) and its poller (warp 3)
        // One thread issues every tcgen05.mma, and the tensor core queues only
        // about two of them, so whatever that thread does between stages
        // leaves the tensor pipe idle.  An mbarrier poll right after an MMA
        // measured ~200 cycles on sm_103a, a named-barrier hand-off ~45: warp
        // 3 waits for each stage's x and B tiles and hands the stage over
        // through named barrier 1 (a reduction that also carries either
        // side's failure, so both leave the loop at the same point); warp 1
        // issues its MMAs and commits.  The operand descriptors are formed
        // once (slot 0 of each ring) and advanced by constant address offsets
        // (the descriptor's low field is the shared address / 16; every
        // address here is below 256 KB, so the field never carries).
        const bool issuer = warp == 1;
        constexpr uint32_t idesc = idesc_f16(128, BN, false);
        const uint64_t dA0 = smem_desc_sw128(base, 16, 1024);
        const uint64_t dB0 = smem_desc_sw128(base + kRingB, 16, 1024);
        RingPos rx, rb;
        int lt = 0;
        bool ok = true;
        PfUnit un;
        for (int ui = 0; ok && pf_unit(a, KB, ui, un); ++ui, ++lt) {
            const int kbeg = un.kb0, kend = un.kb1;
            const int acc = lt % kAccBufs;
            const uint32_t aph = (lt / kAccBufs) & 1;
            // the issuer needs the accumulator set drained by the epilogue
            bool mine = true;
            if (issuer && lane == 0) mine = !aborted(abort_flag) && mbar_wait(accE(acc), aph ^ 1);
            const uint32_t d = tmem + static_cast<uint32_t>(acc * kHalves * BN);
            for (int kb = kbeg; kb < kend; ++kb) {
                if (!issuer && lane == 0) mine = mbar_wait(fullX(rx.s), rx.ph) && mbar_wait(fullB(rb.s), rb.ph);
                __syncwarp();
                if (!bar_and(1, 64, mine)) {
                    if (lane == 0) fail(a.status, 0x20, abort_flag);
                    ok = false;
                    break;
                }
                if (issuer && lane == 0) {
                    tc_fence_after();
                    const uint64_t da = dA0 + static_cast<uint32_t>((rx.s * kXStage) >> 4);
                    const uint64_t db = dB0 + static_cast<uint32_t>((rb.s * kBStage) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
#pragma unroll
                        for (int hm = 0; hm < kHalves; ++hm)    // rows 128*hm.. of the x tile, same B tile
                            umma_f16(d + hm * BN, da + ((hm * 16384 + (kk / 4) * kXRows * 128 + (kk % 4) * 32) >> 4),
                                     db + (((kk / 4) * BN * 128 + (kk % 4) * 32) >> 4), idesc, (kb != kbeg) || (kk != 0));
                    umma_commit(emptyX(rx.s));
                    umma_commit(emptyB(rb.s));
                }
                __syncwarp();
                mine = true;
                rx.next(kSX);
                rb.next(kSB);
            }
            if (ok && issuer && lane == 0) umma_commit(accF(acc));
        }
    } else if (warp < kDq0 + kDqWarps) {
        // ------------------------------------------------------ dequantizers
        // kDqGroups groups of kDqHalf warps take the stages in turn, and warp
        // wg of a group owns kDqGroups n16 tiles of its stages: every stage
        // costs its warps two barrier waits and two arrivals whatever its
        // work, so with 128-row tiles (half the MMA work per stage) two
        // groups on alternate stages keep up better than all sixteen warps
        // on every stage.
        // Lane -> packed-word assignment: in every 8-lane phase (p = lane >> 3)
        // the lanes take columns gq in {p, p ^ 5} and all four tq, so the
        // 16-byte loads of packed words and the 16-byte stores into the
        // swizzled B tile both hit eight distinct bank groups per phase.
        const int wl = warp - kDq0;
        const int grp = wl / kDqHalf, wg = wl % kDqHalf;
        const int pq = lane >> 3;
        const int gq = ((lane >> 2) & 1) ? (pq ^ 5) : pq;
        const int tq = lane & 3;
        const int ls = 4 * gq + tq;
        const uint32_t sw0 = static_cast<uint32_t>((tq ^ gq) << 4);
        const uint32_t sw1 = static_cast<uint32_t>(((4 + tq) ^ gq) << 4);
        // one n16 tile and 64-row chunk kc of a stage: the constants of the
        // chunk's one or two groups (global group g0, stage slot s0; gl1: the
        // second 32-row block starts the next group), the words, and the
        // scaled fp16 pairs (four 16-byte vectors)
        auto dequant_tile = [&](const uint8_t *st, int nt, int kc, int g0, int s0, bool gl1, uint4 (&bv)[4]) {
            const uint8_t *sz = st + kSzOff;
            uint32_t c_s[2][2], c_nl[2][2], c_nh[2][2];   // [group slot][column gq / gq+8]
#pragma unroll
            for (int gl = 0; gl < 2; ++gl) {
                if (gl == 1 && !gl1) break;
                const int g = g0 + gl;
                const uint32_t sp = *reinterpret_cast<const uint32_t *>(sz + (s0 + gl) * P::kSGroup + (nt * 8 + gq) * 4);
                const uint2 zw = *reinterpret_cast<const uint2 *>(sz + kZOff + (s0 + gl) * P::kZGroup + nt * 8);
                c_s[gl][0] = __byte_perm(sp, sp, 0x1010);
                c_s[gl][1] = __byte_perm(sp, sp, 0x3232);
                // effective zero points minus one (stored + zero offset - 1)
                const uint32_t zoff = g < a.zsplit ? 0u : static_cast<uint32_t>(a.zero_offset);
                const uint32_t z0 = ((zw.x >> (4 * gq)) & 0xFu) + zoff - 1u;
                const uint32_t z1 = ((zw.y >> (4 * gq)) & 0xFu) + zoff - 1u;
                c_nl[gl][0] = neg_zlo(z0);
                c_nh[gl][0] = neg_zhi(z0);
                c_nl[gl][1] = neg_zlo(z1);
                c_nh[gl][1] = neg_zhi(z1);
            }
            const uint4 wv = *reinterpret_cast<const uint4 *>(st + ((nt * kKC + kc) * 32 + ls) * 16);
            const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int J = j >> 1, jj = j & 1;     // J: the 32-row block
                const uint32_t sp = (J && gl1) ? c_s[1][jj] : c_s[0][jj];
                const uint32_t nl = (J && gl1) ? c_nl[1][jj] : c_nl[0][jj];
                const uint32_t nh = (J && gl1) ? c_nh[1][jj] : c_nh[0][jj];
                uint32_t q[4];
                unpack_qz(w[j], nl, nh, q);
                bv[j] = make_uint4(hmul2(q[0], sp), hmul2(q[1], sp), hmul2(q[2], sp), hmul2(q[3], sp));
            }
        };
        RingPos rp, rb;
        bool ok = true;
        int si = 0;                                   // stage index over the CTA's units
        PfUnit un;
        for (int ui = 0; ok && pf_unit(a, KB, ui, un); ++ui) {
            const int kbeg = un.kb0, kend = un.kb1;
            // group of the unit's first 32-row block (a slice may start inside a
            // group) and the blocks left in it, itself included
            int gcur = (kBlk * kbeg) / a.bpg, left = a.bpg - (kBlk * kbeg - gcur * a.bpg);
            for (int kb = kbeg; kb < kend; ++kb, ++si) {
                // the stage's first group and each block's group slot (as the producer loads them)
                int g_first = gcur, gsl[kBlk];
#pragma unroll
                for (int b = 0; b < kBlk; ++b) {
                    if (left == 0) { ++gcur; left = a.bpg; }
                    if (b == 0) g_first = gcur;
                    gsl[b] = gcur - g_first;
                    --left;
                }
                if (si % kDqGroups == grp) {
                    if (aborted(abort_flag)) { ok = false; break; }
                    // The B slot is freed only when the MMAs of the stage kSB back
                    // complete, so that wait is on the tensor pipe's critical loop:
                    // everything that needs only the packed stage runs before it,
                    // leaving the stores, the proxy fence and the arrival after it.
                    if (!mbar_wait(fullP(rp.s), rp.ph)) {
                        fail(a.status, 0x40, abort_flag);
                        ok = false;
                        break;
                    }
                    const uint8_t *st = sbase + kRingP + rp.s * kPStage;
                    uint4 bv[kUnits][4];
#pragma unroll
                    for (int u = 0; u < kUnits; ++u) {
                        const int nt = BK == 128 ? wg : kDqGroups * wg + u, kc = BK == 128 ? u : 0;
                        dequant_tile(st, nt, kc, g_first + gsl[2 * kc], gsl[2 * kc], gsl[2 * kc + 1] != gsl[2 * kc], bv[u]);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(emptyP(rp.s));   // every value read from it is in registers
                    if (!mbar_wait(emptyB(rb.s), rb.ph ^ 1)) {
                        fail(a.status, 0x40, abort_flag);
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int u = 0; u < kUnits; ++u) {
                        const int nt = BK == 128 ? wg : kDqGroups * wg + u, kc = BK == 128 ? u : 0;
                        uint8_t *brow = sbase + kRingB + rb.s * kBStage + kc * BN * 128 + 2 * nt * 1024 + gq * 128;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            *reinterpret_cast<uint4 *>(brow + (j & 1) * 1024 + ((j >> 1) ? sw1 : sw0)) = bv[u][j];
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(fullB(rb.s));
                }
                rp.next(kSP);
                rb.next(kSB);
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        const int quad = warp & 3;                  // TMEM lanes 32*quad .. +31
        int lt = 0;
        PfUnit un;
        for (int ui = 0; pf_unit(a, KB, ui, un); ++ui, ++lt) {
            const int t = un.t;
            const int acc = lt % kAccBufs;
            const uint32_t aph = (lt / kAccBufs) & 1;
            bool ok = !aborted(abort_flag) && mbar_wait(accF(acc), aph);
            __syncwarp();
            ok = bar_and(2, 32 * kEpiWarps, ok);        // the four epilogue warps agree
            if (!ok) {
                if (lane == 0) fail(a.status, 0x80, abort_flag);
                break;
            }
            tc_fence_after();
            // With fin0, piece 0 of a tile cut into 2..kFinishMax pieces (its
            // first k blocks; always the CTA's last unit) stays in tensor
            // memory: the CTA finishes that tile after the main loop.
            PfUnit nx;
            if (a.fin0 && un.np > 1 && un.np <= kFinishMax && un.p == 0 && !pf_unit(a, KB, ui + 1, nx)) break;
            const int m0 = (t % a.tiles_m) * BM;
            const int n0 = (t / a.tiles_m) * BN;
#pragma unroll 1
            for (int hc = 0; hc < kHalves * BN; hc += 32) {
                const int hm = hc / BN, c0 = hc % BN;
                const int row = m0 + 128 * hm + 32 * quad + lane;
                uint32_t r[32];
                tmem_ld_x32(tmem + static_cast<uint32_t>(acc * kHalves * BN + hc) + (static_cast<uint32_t>(32 * quad) << 16),
                            r);
                if (un.np > 1) {
                    // the fp32 partial of this piece, whole tile, lane-major so that
                    // each warp store is 512 contiguous bytes: slot sl = t pmax + p,
                    // float4 index (((sl * (kHalves*BN/32) + hc/32) * 4 + quad) * 8 + v) * 32 + lane
                    const size_t sl = static_cast<size_t>(t) * a.pmax + un.p;
                    float4 *dst = reinterpret_cast<float4 *>(a.ws) +
                                  ((sl * (kHalves * BN / 32) + hc / 32) * 4 + quad) * 8 * 32 + lane;
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        dst[v * 32] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                                  __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                } else if (row < a.M) {
                    store_row32(a, row, n0 + c0, r);
                }
            }
            tc_fence_before();
            if (un.np > 1) {
                // this piece's partial is written: count it for the CTAs that
                // finish the tile
                __threadfence();
                __syncwarp();
                bar_and(2, 32 * kEpiWarps, true);
                if (quad == 0 && lane == 0) atomicAdd(a.tickets + t, 1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(accE(acc));
        }
    }

    tc_fence_before();
    __syncthreads();
    // Stream-K.  Every piece of a tile cut into pieces is counted in the
    // tile's ticket as soon as its CTA's epilogue has written it, and no CTA
    // waits before writing its pieces, so no wait below depends on another
    // (bounded waits all the same; the cooperative launch keeps every CTA
    // resident).
    //
    // (a) With fin0, when this CTA's last unit is piece 0 of a tile cut into
    // at most kFinishMax pieces (still in tensor memory): wait for the tile's
    // other pieces, stage them through the idle ring memory (one bulk copy
    // per piece and pass) and add them in piece order, all warps at once
    // (warp w reads TMEM lanes 32 (w % 4) ..), then add bias and round once.
    constexpr int CP = kHalves * BN / 32;              // 32-column chunks of a tile, 16 KB of fp32 each
    constexpr int kStage = kBarOff / 16384;            // chunks the ring memory holds
    const bool fin = a.sk && a.fin0 != 0;
    PfUnit un;
    if (fin) {
        PfUnit last{};
        int nu = 0;
        for (; pf_unit(a, KB, nu, un); ++nu) last = un;
        if (nu > 0 && last.np > 1 && last.np <= kFinishMax && last.p == 0) {
            const int t = last.t, quad = warp & 3, nw = static_cast<int>(blockDim.x) / 128;
            const int m0 = (t % a.tiles_m) * BM, n0 = (t / a.tiles_m) * BN;
            const uint32_t tacc = tmem + static_cast<uint32_t>(((nu - 1) % kAccBufs) * kHalves * BN) +
                                  (static_cast<uint32_t>(32 * quad) << 16);
            const int S = last.np;
            __shared__ int s_ready;
            if (threadIdx.x == 0) {
                bool ready = !aborted(abort_flag) && S - 1 <= kStage;
                const uint64_t t0 = globaltimer();
                while (ready && atomicAdd(a.tickets + t, 0) < S - 1) {
                    if (aborted(abort_flag) || globaltimer() - t0 > 2000000000ull) ready = false;
                    else __nanosleep(128);
                }
                __threadfence();
                if (ready) a.tickets[t] = 0;            // every other piece has arrived: ready for the next call
                else fail(a.status, 0x100, abort_flag);
                s_ready = ready;
            }
            __syncthreads();
            if (s_ready) {
                tc_fence_after();
                const int C = kStage / (S - 1);            // chunks per pass
                // piece j of tile t: float4 ((t pmax + j) CP + chunk) 1024 + (quad 8 + v) 32 + lane
                const float4 *ws4 = reinterpret_cast<const float4 *>(a.ws) + static_cast<size_t>(t) * a.pmax * CP * 1024;
                float4 *st4 = reinterpret_cast<float4 *>(sbase);
                for (int c0 = 0, pass = 0; c0 < CP; c0 += C, ++pass) {
                    const int nc = min(C, CP - c0), per = nc * 1024;
                    // one bulk copy per piece (its chunks [c0, c0 + nc) are contiguous),
                    // after every thread's last reads of this memory (barrier above);
                    // the pieces were published by other CTAs' plain stores
                    if (threadIdx.x == 0) {
                        asm volatile("fence.proxy.async.global;\n\tfence.proxy.async.shared::cta;" ::: "memory");
                        mbar_arrive_expect_tx(stageB, static_cast<uint32_t>((S - 1) * nc) * 16384u);
                        for (int j = 0; j < S - 1; ++j)
                            bulk_load(base + static_cast<uint32_t>(j * per) * 16u,
                                      ws4 + (static_cast<size_t>(j + 1) * CP + c0) * 1024, static_cast<uint32_t>(nc) * 16384u,
                                      stageB);
                    }
                    if (!__syncthreads_and(mbar_wait(stageB, pass & 1))) {
                        if (threadIdx.x == 0) fail(a.status, 0x100, abort_flag);
                        break;
                    }
                    for (int ch = c0 + (warp >> 2); ch < c0 + nc; ch += nw) {
                        uint32_t r[32];
                        tmem_ld_x32(tacc + static_cast<uint32_t>(32 * ch), r);
                        for (int j = 0; j < S - 1; ++j) {
                            const float4 *src = st4 + j * per + ((ch - c0) * 4 + quad) * 256 + lane;
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                const float4 q = src[v * 32];
                                r[4 * v] = __float_as_uint(__uint_as_float(r[4 * v]) + q.x);
                                r[4 * v + 1] = __float_as_uint(__uint_as_float(r[4 * v + 1]) + q.y);
                                r[4 * v + 2] = __float_as_uint(__uint_as_float(r[4 * v + 2]) + q.z);
                                r[4 * v + 3] = __float_as_uint(__uint_as_float(r[4 * v + 3]) + q.w);
                            }
                        }
                        // this warp's slice of the first staged piece, read only by this warp
                        __syncwarp();
                        const int row0 = m0 + 128 * ((32 * ch) / BN) + 32 * quad;
                        if (row0 < a.M)
                            store_block(a, row0, n0 + (32 * ch) % BN, r,
                                        reinterpret_cast<uint8_t *>(st4 + ((ch - c0) * 4 + quad) * 256), lane);
                    }
                    __syncthreads();                       // before the next pass overwrites the stage
                }
            }
        }
    }
    if (a.sk) {
        // (b) Otherwise (the even K split: S equal k ranges, one CTA each):
        // once all S are counted, every piece's CTA finishes rows
        // [p BM / S, (p + 1) BM / S) of the tile, summing the pieces in order,
        // adding bias, rounding once; the second round of counts lets the
        // last of the 2 S reset the ticket for the next call.
        for (int ui = 0; pf_unit(a, KB, ui, un); ++ui) {
            if (un.np == 1 || (fin && un.np <= kFinishMax)) continue;
            const int t = un.t, S = un.np, ks = un.p;
            __shared__ int s_all;
            if (threadIdx.x == 0) {
                bool ready = true;
                const uint64_t t0 = globaltimer();
                while (atomicAdd(a.tickets + t, 0) < S) {
                    if (aborted(abort_flag) || globaltimer() - t0 > 2000000000ull) {
                        ready = false;
                        break;
                    }
                    __nanosleep(256);
                }
                __threadfence();
                s_all = ready;
                if (!ready) fail(a.status, 0x100, abort_flag);
            }
            __syncthreads();
            if (s_all) {
                const int m0 = (t % a.tiles_m) * BM, n0 = (t / a.tiles_m) * BN;
                const int r0 = (BM * ks) / S, r1 = (BM * (ks + 1)) / S, rows = r1 - r0;
                const float4 *ws4 = reinterpret_cast<const float4 *>(a.ws);
                // consecutive threads take consecutive rows of one 8-column group: their
                // loads of the lane-major partials are contiguous
                for (int i = threadIdx.x; i < rows * (BN / 8); i += blockDim.x) {
                    const int rl = r0 + i % rows, c = 8 * (i / rows);
                    const int row = m0 + rl, n = n0 + c;
                    if (row >= a.M || n >= a.N) continue;
                    const int hm = rl / 128, q = (rl % 128) / 32, ln = rl % 32;
                    const int hc = hm * BN + c;
                    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    for (int j = 0; j < S; ++j) {
                        const size_t sl = static_cast<size_t>(t) * a.pmax + j;
                        const float4 *src = ws4 + ((sl * CP + hc / 32) * 4 + q) * 8 * 32 + ((hc % 32) / 4) * 32 + ln;
                        const float4 p0 = __ldcg(src), p1 = __ldcg(src + 32);
                        v[0] += p0.x; v[1] += p0.y; v[2] += p0.z; v[3] += p0.w;
                        v[4] += p1.x; v[5] += p1.y; v[6] += p1.z; v[7] += p1.w;
                    }
                    if (a.out_bf16 == kOutF32) {
                        float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.out) +
                                                                 static_cast<size_t>(row) * a.N + n);
                        dst[0] = make_float4(v[0], v[1], v[2], v[3]);
                        dst[1] = make_float4(v[4], v[5], v[6], v[7]);
                        continue;
                    }
                    uint32_t pk[4];
                    const float rs = a.rowscale ? a.rowscale[row] : 1.f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) pk[e] = out_pair(v[2 * e], v[2 * e + 1], rs, a.bias, n + 2 * e, a.out_bf16);
                    *reinterpret_cast<uint4 *>(a.out + static_cast<size_t>(row) * a.N + n) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            }
            __syncthreads();
            if (threadIdx.x == 0 && atomicAdd(a.tickets + t, 1) == 2 * S - 1) atomicExch(a.tickets + t, 0);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

int sm_count() {
    static int n = -1;
    if (n < 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            n = v;
        else
            n = kSMs;
    }
    return n;
}


template <int BM, int BN, int BKS>
cudaError_t launch_prefill_tile(const HandleView &h, const PrefillPlan &p, float *ws, int *tickets,
                                const uint16_t *x, int M, uint16_t *out, cudaStream_t s) {
    using P = PfCfg<BM, BN, BKS>;
    // 128-row stages load 64 rows of x: M <= 64 only; their k blocks are whole
    if ((BKS == 128 && M > P::kXRows) || h.K % BKS) return cudaErrorInvalidValue;
    CUtensorMap tmA, tmW;
    cudaError_t e;
    const int KC = h.K / 64;
    if ((e = encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, h.K, M, static_cast<uint64_t>(h.K) * 2, 64, P::kXRows,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, h.wp, static_cast<uint64_t>(KC) * 128, h.N / 16,
                       static_cast<uint64_t>(KC) * 512, 128 * P::kKC, BN / 16, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
        cudaSuccess)
        return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = dyn_smem_optin(reinterpret_cast<const void *>(prefill_kernel<BM, BN, BKS>), dev, P::kSmem, nullptr)) !=
        cudaSuccess)
        return e;
    PfArgs args{M, h.N, h.K, h.bias, out, h.status, h.s2, h.zeros, h.geff / 32, (M + BM - 1) / BM,
                (h.N + BN - 1) / BN, h.zero_offset, h.zsplit, h.rowscale, h.out_bf16, p.sk, p.pmax, p.fin0, ws, tickets};
    const int ntiles = args.tiles_m * args.tiles_n;
    const int grid = p.sk ? p.grid : (ntiles < sm_count() ? ntiles : sm_count());
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(P::kThreads);
    cfg.dynamicSmemBytes = P::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeCooperative;         // split units wait on each other: all resident
    at.val.cooperative = 1;
    cfg.attrs = &at;
    cfg.numAttrs = p.sk ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, prefill_kernel<BM, BN, BKS>, tmA, tmW, args);
}

}  // namespace

// Tile shape and work split by tile count (c = SMs), measured on GB300:
//   - 256 x 256 tiles round robin when there are enough of them to give
//     every SM at least three quarters of a tile's work;
//   - else, when that gives at least two pieces per tile, every 256 x 256
//     tile cut into S = floor(c / tiles) <= 8 equal k ranges, one CTA each
//     (the stream-K walk below with S CTAs per tile);
//   - else stream-K over 256 x 256 tiles: one CTA per SM (fewer when that
//     would leave a CTA under 8 k blocks), each a contiguous range of the
//     tiles x k-blocks space, tiles cut into pieces at the range ends and
//     summed after the main loop.  256-row tiles let one dequantized B tile
//     feed two M = 128 MMAs; up to 128 rows take 128 x 256 tiles instead.
PrefillPlan plan_prefill(int M, int K, int N, int sms) {
    PrefillPlan p{};
    const long long c = sms > 0 ? sms : sm_count();
    const long long n256 = (N + 255) / 256;
    const long long t256x256 = static_cast<long long>((M + 255) / 256) * n256;
    p.bm = 256, p.bn = 256, p.bk = 64;
    // whole 256 x 256 tiles round robin while the rounds are at least three
    // quarters full; stream-K when the last round would leave SMs idle
    // (8192 x 10240 at M = 1024: 160 tiles, 186 -> 134 us; at M = 2048: 293
    // -> 247 us; with fuller rounds round robin measured as fast or faster)
    const long long rounds = (t256x256 + c - 1) / c;
    if (4 * t256x256 >= 3 * rounds * c) return p;
    // up to 128 rows: one 128-row tile holds them all (256-row MMAs would
    // spend half or more of the tensor pipe on rows that do not exist)
    if (M <= 128) p.bm = 128;
    // up to 64 rows: 128-row stages (twice the weights per stage hand-off;
    // x tiles of 64 rows leave the shared memory for it)
    if (M <= Q4_PF_BK128_MAXM && K % 128 == 0) p.bk = 128;
    const long long tiles = static_cast<long long>((M + p.bm - 1) / p.bm) * n256;
    // the split is decided in 64-row blocks, the work walked in stages
    const int KB64 = K / 64, KB = K / p.bk;
    const long long W = tiles * KB;
    p.sk = 1;
    if (c / tiles >= 2 && KB64 / 2 >= 8) {
        int S = static_cast<int>(std::min<long long>(8, c / tiles));
        while (S > 2 && KB64 / S < 8) --S;
        p.grid = static_cast<int>(tiles) * S;
    } else {
        // (measured against round robin over 128-row tiles, the choice before
        // stream-K: 1.4x-1.9x faster on 8192 x 28672 at M <= 256, 8192 x 10240
        // and 4096 x 11008 at M = 512, the same elsewhere)
        p.grid = static_cast<int>(std::max<long long>(1, std::min<long long>(c, tiles * KB64 / 8)));
        p.fin0 = 1;
    }
    auto owner = [&](long long w) { return static_cast<int>(((w + 1) * p.grid - 1) / W); };
    p.pmax = 1;
    for (long long t = 0; t < tiles; ++t)
        p.pmax = std::max(p.pmax, owner(t * KB + KB - 1) - owner(t * KB) + 1);
    if (p.pmax > 1) {
        p.ws_floats = static_cast<size_t>(tiles) * p.pmax * p.bm * p.bn;
        p.n_tickets = static_cast<int>(tiles);
    }
    return p;
}

cudaError_t launch_prefill(const HandleView &h, const PrefillPlan &p, float *ws, int *tickets, const uint16_t *x,
                           int M, uint16_t *out, cudaStream_t s) {
    if (p.bn != 256) return cudaErrorInvalidValue;
    if (p.bm == 128 && p.bk == 128) return launch_prefill_tile<128, 256, 128>(h, p, ws, tickets, x, M, out, s);
    if (p.bm == 128) return launch_prefill_tile<128, 256, 64>(h, p, ws, tickets, x, M, out, s);
    return launch_prefill_tile<256, 256, 64>(h, p, ws, tickets, x, M, out, s);
}

// Rows from which the fused prefill beats the decode kernels, measured on
// GB300 (CUDA-graph replays over more weights than L2): 17 in general; 9 with
// 32-row groups (8192x28672 M = 9-16: 75 against 112-125 us), and with 64-row
// groups on layers of 100 Mi weights or more (69 against 74-78 us), where the
// decode kernels' per-group step weighs most.
int prefill_default_min_m(int K, int N, int geff) {
    const size_t weights = static_cast<size_t>(K) * N;
    if (geff <= 32 || (geff <= 64 && weights >= (size_t{100} << 20))) return 9;
    return 17;
}

}  // namespace q4
