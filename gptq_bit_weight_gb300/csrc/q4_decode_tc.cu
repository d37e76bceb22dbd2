// Decode (M <= 16) GPTQ W4A16 matmul on the 5th-generation tensor cores.
//
// "GPTQ's 'Exllama Kernel Not Installed' Warning", "What the fallback
// actually does": weight-bound decoding is limited by memory bandwidth; the
// fused kernel reads packed weights, dequantizes them on chip and never
// writes a dequantized matrix.  "Inference Backends", "Numeric epilogues and
// input gradients": fp32 accumulation, bias added to the fp32 sum before one
// cast, split reductions in fp32.
//
// Formulation: D[n][m] = sum_k W[k][n] x[m][k] with a 128-column weight tile
// as the UMMA A operand (M = 128 rows = output columns n, K-major) and the
// x tile as B (N = 16 rows of x, zero-filled past M).  A holds the exact
// integers (q - z - 1) in fp16; the scale is not applied per weight.  Each
// quantization group accumulates into its own 16-column slice of tensor
// memory (up to 32 groups, 512 columns), and the epilogue forms
//     y[m][n] = sum_g s[g][n] * D_g[n][m]
// in fp32.  Per packed word the dequantizing threads spend one shift, four
// LOP3 and four fp16x2 subtractions (all exact) and one 16-byte shared store;
// no fp16 multiply and no legacy mma.sync.
//
// CTA = one 128-column tile x one K slice (the slices of a tile form a
// thread-block cluster and are summed through distributed shared memory).
//   warp 0       one thread: TMA loads into an 8-stage ring of {x tile 16x64
//                fp16 (128-byte swizzle), packed-word tile 128x64 (4 KB)};
//                the slice's scales and zero words once, up front
//   warp 1       allocates 512 TMEM columns; one thread issues
//                tcgen05.mma M=128 N=16 K=16 into the group's columns
//   warps 2-9    dequantize into an 8-stage ring of fp16 A tiles (K-major,
//                128-byte swizzle); afterwards warps 2-5 run the epilogue
// Every mbarrier wait is bounded (~2 s); a wait that runs out records an
// error bit in the handle's status word, the CTA lets its copies land, frees
// its TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdint>

#include "q4_internal.cuh"
#include "q4_tc.cuh"

namespace q4 {

cudaError_t encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *ptr, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

namespace {

using namespace tc;

constexpr int BN = 128;                              // output columns per CTA (UMMA M)
constexpr int MP = 16;                               // x rows per CTA (UMMA N)
constexpr int BK = 64;                               // rows of W per stage
constexpr int kSP = 8;                               // TMA ring stages
constexpr int kSA = 8;                               // fp16 A ring stages
constexpr int kXOff = 0, kPOff = 2048;               // within a TMA stage
constexpr int kPStage = 6144;                        // 2 KB x + 4 KB packed
constexpr int kAStage = BN * BK * 2;                 // 16 KB
constexpr int kMaxGroups = 512 / MP;                 // TMEM columns / group width
constexpr int kSzGroupBytes = 8 * 8 * 4 + 16 * 4;    // scale pairs (8 n16 tiles) + zero words
constexpr int kRingA = kSP * kPStage;
constexpr int kSzOff = kRingA + kSA * kAStage;
constexpr int kRedOff = kSzOff + kMaxGroups * kSzGroupBytes;
constexpr int kBarOff = kRedOff + BN * MP * 4;
constexpr int kNumBars = 2 * kSP + 2 * kSA + 2;
constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + 1024;
constexpr int kDqWarps = 8;
constexpr int kThreads = 32 * (2 + kDqWarps);
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxCluster = 8;

struct DtArgs {
    int M, N, K;
    const uint16_t *bias;
    uint16_t *out;
    int *status;
    const uint32_t *s2;
    const uint32_t *zeros;
    int geff;
    int slice_kb;        // k-blocks per slice
    int splits;
    int zero_offset;     // effective zero = stored + zero_offset
};

__device__ __forceinline__ void fail(int *status, int bit, int *abort_flag) {
    if (status) atomicOr(status, bit);
    atomicExch(abort_flag, 1);
}
__device__ __forceinline__ bool aborted(int *abort_flag) { return *reinterpret_cast<volatile int *>(abort_flag) != 0; }

__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, DtArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + kBarOff;
    auto fullP = [&](int s) { return bar0 + 8u * s; };
    auto emptyP = [&](int s) { return bar0 + 8u * (kSP + s); };
    auto fullA = [&](int s) { return bar0 + 8u * (2 * kSP + s); };
    auto emptyA = [&](int s) { return bar0 + 8u * (2 * kSP + kSA + s); };
    const uint32_t szBar = bar0 + 8u * (2 * kSP + 2 * kSA);
    const uint32_t accBar = szBar + 8u;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + kBarOff + kNumBars * 8);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    float *red = reinterpret_cast<float *>(sbase + kRedOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT16 = a.N >> 4;
    const int nt0 = blockIdx.x * (BN / 16);
    const int n0 = blockIdx.x * BN;
    const int split = blockIdx.y;
    const int m0 = blockIdx.z * MP;
    const int KB = a.K / BK;
    const int kb_beg = split * a.slice_kb;
    const int kb_end = min(KB, kb_beg + a.slice_kb);
    const int nkb = kb_end - kb_beg;
    const int bpg = a.geff / 32;                     // 32-row blocks per group
    const int g_beg = (kb_beg * 2) / bpg;
    const int g_end = (kb_end * 2 - 1) / bpg + 1;
    const int ng = g_end - g_beg;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSP; ++s) {
            mbar_init(fullP(s), 1);
            mbar_init(emptyP(s), 1 + kDqWarps);      // MMA commit + each dequantizing warp's release
        }
        for (int s = 0; s < kSA; ++s) {
            mbar_init(fullA(s), kDqWarps);
            mbar_init(emptyA(s), 1);
        }
        mbar_init(szBar, 1);
        mbar_init(accBar, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            // scales and zero words of the slice's groups, for this CTA's 8 n16 tiles
            // (a last tile of 64 columns copies only its 4 valid n16 tiles)
            const uint32_t szb = base + kSzOff;
            const int tv = min(8, NT16 - nt0);
            mbar_arrive_expect_tx(szBar, static_cast<uint32_t>(ng) * tv * 40u);
            for (int gl = 0; gl < ng; ++gl) {
                const size_t gr = static_cast<size_t>(g_beg + gl);
                bulk_load(szb + gl * kSzGroupBytes, a.s2 + (gr * NT16 + nt0) * 8, tv * 32u, szBar);
                bulk_load(szb + gl * kSzGroupBytes + 256, a.zeros + gr * (a.N >> 3) + nt0 * 2, tv * 8u, szBar);
            }
            int issued = 0;
            for (int i = 0; i < nkb; ++i, ++issued) {
                const int s = i % kSP;
                if (aborted(abort_flag)) break;
                if (!mbar_wait(emptyP(s), ((i / kSP) & 1) ^ 1)) { fail(a.status, 0x100, abort_flag); break; }
                const uint32_t st = base + s * kPStage;
                mbar_arrive_expect_tx(fullP(s), 2048u + 4096u);
                tma_load_2d(st + kXOff, &tmX, fullP(s), (kb_beg + i) * BK, m0);
                tma_load_2d(st + kPOff, &tmW, fullP(s), (kb_beg + i) * 128, nt0);
            }
            if (aborted(abort_flag)) {
                mbar_wait(szBar, 0);
                for (int j = issued > kSP ? issued - kSP : 0; j < issued; ++j) mbar_wait(fullP(j % kSP), (j / kSP) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(BN, MP, false);
            bool ok = true;
            for (int i = 0; i < nkb; ++i) {
                const int s = i % kSP, sa = i % kSA;
                if (aborted(abort_flag) || !mbar_poll(fullP(s), (i / kSP) & 1) || !mbar_poll(fullA(sa), (i / kSA) & 1)) {
                    fail(a.status, 0x200, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sx = base + s * kPStage + kXOff;
                const uint32_t sA = base + kRingA + sa * kAStage;
                const int blk0 = 2 * (kb_beg + i);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const int blk = blk0 + (kk >> 1);            // 32-row block of this K=16 step
                    const int g = blk / bpg;
                    const bool first = (blk % bpg == 0) && !(kk & 1);
                    const uint32_t d = tmem + static_cast<uint32_t>((g - g_beg) * MP);
                    // a group's first step also starts the slice: a group cut by the slice
                    // start begins fresh at this slice's first block
                    const bool fresh = first || (i == 0 && kk == 0);
                    umma_f16(d, smem_desc_sw128(sA + kk * 32, 16, 1024), smem_desc_sw128(sx + kk * 32, 16, 1024),
                             idesc, fresh ? 0u : 1u);
                }
                umma_commit(emptyP(s));
                umma_commit(emptyA(sa));
            }
            if (ok) umma_commit(accBar);
        }
    } else {
        // ------------------------------------------------------ dequantizers
        const int wl = warp - 2;                      // 0..7: the n16 tile of this warp
        const int pq = lane >> 3;
        const int gq = ((lane >> 2) & 1) ? (pq ^ 5) : pq;
        const int tq = lane & 3;
        const int ls = 4 * gq + tq;
        const uint32_t sw0 = static_cast<uint32_t>((tq ^ gq) << 4);
        const uint32_t sw1 = static_cast<uint32_t>(((4 + tq) ^ gq) << 4);
        const uint32_t szb = base + kSzOff;
        bool ok = mbar_wait(szBar, 0);
        if (!ok) fail(a.status, 0x400, abort_flag);
        uint32_t nzl[2][2], nzh[2][2];                // [half J][column gq / gq+8]
        int cached_g = -1;
        auto load_zero = [&](int gl, int J) {
            uint32_t z0w, z1w;
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                         : "=r"(z0w), "=r"(z1w)
                         : "r"(szb + gl * kSzGroupBytes + 256 + wl * 8));
            // effective zero points minus one (stored + zero_offset - 1)
            const uint32_t z0 = ((z0w >> (4 * gq)) & 0xFu) + a.zero_offset - 1u;
            const uint32_t z1 = ((z1w >> (4 * gq)) & 0xFu) + a.zero_offset - 1u;
            nzl[J][0] = neg_zlo(z0);
            nzh[J][0] = neg_zhi(z0);
            nzl[J][1] = neg_zlo(z1);
            nzh[J][1] = neg_zhi(z1);
        };
        for (int i = 0; ok && i < nkb; ++i) {
            const int s = i % kSP, sa = i % kSA;
            if (aborted(abort_flag)) break;
            if (!mbar_wait(fullP(s), (i / kSP) & 1) || !mbar_wait(emptyA(sa), ((i / kSA) & 1) ^ 1)) {
                fail(a.status, 0x800, abort_flag);
                break;
            }
            const int blk0 = 2 * (kb_beg + i);
            const int g0 = blk0 / bpg, g1 = (blk0 + 1) / bpg;
            if (g0 != cached_g) {
                load_zero(g0 - g_beg, 0);
                cached_g = g0;
            }
            if (g1 != g0) load_zero(g1 - g_beg, 1);
            uint32_t w[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(base + s * kPStage + kPOff + (wl * 32 + ls) * 16));
            const uint32_t arow = base + kRingA + sa * kAStage + static_cast<uint32_t>(2 * wl * 1024 + gq * 128);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int J = j >> 1, jj = j & 1;
                const uint32_t nl = (J && g1 != g0) ? nzl[1][jj] : nzl[0][jj];
                const uint32_t nh = (J && g1 != g0) ? nzh[1][jj] : nzh[0][jj];
                uint32_t q[4];
                unpack_qz(w[j], nl, nh, q);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(arow + jj * 1024 + (J ? sw1 : sw0)),
                             "r"(q[0]), "r"(q[1]), "r"(q[2]), "r"(q[3])
                             : "memory");
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(fullA(sa));
                mbar_arrive(emptyP(s));                   // this warp no longer reads the packed words
            }
        }
        // ------------------------------------------------------ epilogue
        // Warps 2-5 own TMEM lanes 32*(warp%4): one output column n per thread.
        if (warp < 6) {
            bool okw = !aborted(abort_flag) && mbar_wait(accBar, 0);
            okw = __all_sync(0xffffffffu, okw);
            if (okw) {
                tc_fence_after();
                const int quad = warp & 3;
                const int nl = 32 * quad + lane;                 // column within the tile
                const int ntl = nl >> 4, c16 = nl & 15;
                float y[MP];
#pragma unroll
                for (int m = 0; m < MP; ++m) y[m] = 0.f;
                for (int gl = 0; gl < ng; ++gl) {
                    uint32_t r[16];
                    tmem_ld_x16(tmem + static_cast<uint32_t>(gl * MP) + (static_cast<uint32_t>(32 * quad) << 16), r);
                    const uint32_t sp = *reinterpret_cast<const uint32_t *>(
                        sbase + kSzOff + gl * kSzGroupBytes + (ntl * 8 + (c16 & 7)) * 4);
                    const float sc = __half2float(__ushort_as_half(
                        static_cast<unsigned short>((c16 < 8) ? (sp & 0xFFFFu) : (sp >> 16))));
#pragma unroll
                    for (int m = 0; m < MP; ++m) y[m] = fmaf(sc, __uint_as_float(r[m]), y[m]);
                }
                if (a.splits == 1) {
                    const bool col_ok = n0 + nl < a.N;
                    const float b = (a.bias && col_ok) ? __half2float(__ushort_as_half(a.bias[n0 + nl])) : 0.f;
#pragma unroll
                    for (int m = 0; m < MP; ++m)
                        if (col_ok && m0 + m < a.M)
                            a.out[static_cast<size_t>(m0 + m) * a.N + n0 + nl] =
                                __half_as_ushort(__float2half_rn(y[m] + b));
                } else {
#pragma unroll
                    for (int m = 0; m < MP; ++m) red[m * BN + nl] = y[m];
                }
            } else if (lane == 0) {
                fail(a.status, 0x1000, abort_flag);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }

    if (a.splits > 1) {
        // The K slices of this tile form one cluster: sum the slices' partial
        // tiles in slice order out of each other's shared memory.  Rank r
        // finishes rows m with m % splits == r.
        cluster_sync();
        if (!aborted(abort_flag)) {
            const uint32_t red_local = base + kRedOff;
            for (int e = threadIdx.x; e < MP * BN; e += kThreads) {
                const int m = e / BN, nl = e % BN;
                if (m % a.splits != split || m0 + m >= a.M || n0 + nl >= a.N) continue;
                float v = 0.f;
                for (int r = 0; r < a.splits; ++r) v += ld_dsmem_f32(red_local + e * 4, r);
                if (a.bias) v += __half2float(__ushort_as_half(a.bias[n0 + nl]));
                a.out[static_cast<size_t>(m0 + m) * a.N + n0 + nl] = __half_as_ushort(__float2half_rn(v));
            }
        }
        cluster_sync();
    }
}

}  // namespace

// Slices: at most 32 groups (tensor-memory columns) and at most 8 per tile
// (cluster size); among those, the count whose grid best fills whole waves
// of one CTA per SM.
DecodeTcPlan plan_decode_tc(int M, int K, int N, int geff, int sms) {
    DecodeTcPlan p{};
    const int KB = K / BK;
    const int bpg = geff / 32;
    const int tiles = (N + BN - 1) / BN;
    const int zdim = (M + MP - 1) / MP;
    // largest slice (in k-blocks) whose groups fit the 32 tensor-memory slices
    int max_slice = KB;
    while (max_slice > 1) {
        const int worst = (max_slice * 2 + bpg - 1) / bpg + 1;   // groups a slice can touch
        if (worst <= kMaxGroups) break;
        --max_slice;
    }
    const int min_splits = (KB + max_slice - 1) / max_slice;
    int best = -1;
    double best_eff = -1.0;
    for (int sp = min_splits; sp <= std::min(kMaxCluster, KB); ++sp) {
        const int slice = (KB + sp - 1) / sp;
        if ((KB + slice - 1) / slice != sp) continue;
        const long long ctas = static_cast<long long>(tiles) * sp * zdim;
        const long long waves = (ctas + sms - 1) / sms;
        const double eff = static_cast<double>(ctas) / static_cast<double>(waves * sms);
        if (eff > best_eff + 0.02) {
            best_eff = eff;
            best = sp;
        }
    }
    if (best < 0) {
        p.ok = 0;
        return p;
    }
    p.ok = 1;
    p.splits = best;
    p.slice_kb = (KB + best - 1) / best;
    p.tiles = tiles;
    p.zdim = zdim;
    return p;
}

bool decode_tc_supported(int M, int K, int N, int geff) {
    if (M < 1 || M > MP || N % 64 != 0 || K % BK != 0) return false;
    return plan_decode_tc(M, K, N, geff, kSMs).ok != 0;
}

cudaError_t launch_decode_tc(const HandleView &h, const uint16_t *x, int M, uint16_t *out, cudaStream_t s) {
    CUtensorMap tmX, tmW;
    cudaError_t e;
    const int KC = h.K / 64;
    if ((e = encode_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, h.K, M, static_cast<uint64_t>(h.K) * 2, BK, MP,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, h.wp, static_cast<uint64_t>(KC) * 128, h.N / 16,
                       static_cast<uint64_t>(KC) * 512, 128, 8, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
        return e;
    static cudaError_t attr = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (attr != cudaSuccess) return attr;
    int dev = 0, sms = kSMs;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const DecodeTcPlan p = plan_decode_tc(M, h.K, h.N, h.geff, sms);
    if (!p.ok) return cudaErrorInvalidValue;
    DtArgs args{M, h.N, h.K, h.bias, out, h.status, h.s2, h.zeros, h.geff, p.slice_kb, p.splits, h.zero_offset};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.tiles, p.splits, p.zdim);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[1];
    int na = 0;
    if (p.splits > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 1;
        attrs[na].val.clusterDim.y = static_cast<unsigned>(p.splits);
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, decode_tc_kernel, tmX, tmW, args);
}

}  // namespace q4
