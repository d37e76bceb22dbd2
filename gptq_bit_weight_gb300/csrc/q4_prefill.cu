// Fused prefill: out = x . W + bias with W read packed (4 bits per weight)
// and dequantized in shared memory inside the main loop; the dense matrix is
// never written to HBM ("GPTQ's 'Exllama Kernel Not Installed' Warning",
// "What the fallback actually does": the fused route reads packed weights and
// never materializes the dequantized matrix).  fp32 accumulation, bias added
// to the fp32 sum before the single rounding to fp16 ("Inference Backends",
// "Numeric epilogues and input gradients").
//
// Persistent kernel, one CTA per SM, 128 x BN output tiles taken round-robin
// (m fastest, so the CTAs working at the same time share weight tiles in L2);
// BN = 256, or 128 when 256-wide tiles would leave SMs idle (small M).  The
// roles below are for BN = 256 (BN = 128: 8 dequant warps, 256 TMEM columns).
//
//   warp 0       one thread: TMA loads into a 6-stage ring of {x tile 128x64
//                fp16 (128-byte swizzle), packed-word tile 256x64 (8 KB), the
//                stage's scale pairs and zero words}
//   warp 1       allocates 512 TMEM columns (two 128x256 fp32 accumulators);
//                one thread issues tcgen05.mma M=128 N=256 K=16 and commits
//                stages back to the producer and the dequantizers
//   warps 2-17   dequantize each stage's packed words into a 2-stage ring of
//                fp16 B tiles (K-major, 128-byte swizzle: the UMMA operand
//                layout), w16 = fp16(s * (q - z - 1)) rounded once; each
//                thread one 16-byte vector (four words) per stage
//   warps 18-21  epilogue: tcgen05.ld an accumulator, add bias, round to fp16,
//                store; then hand the accumulator back, so the epilogue of
//                one tile overlaps the main loop of the next.
//
// Only the 24 KB of x and packed words per 64-row stage travel through TMA
// (the 32 KB fp16 tile is made on chip), so six stages keep ~150 KB in flight
// per SM, enough to cover the L2 round trip at the tensor-core rate.
// Every mbarrier wait is bounded (~2 s); a wait that runs out records an
// error bit in the handle's status word, the CTA lets its copies land, frees
// its TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "q4_internal.cuh"
#include "q4_tc.cuh"

namespace q4 {

cudaError_t encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *ptr, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

namespace {

using namespace tc;

constexpr int BM = 128, BK = 64;
#ifndef Q4_PREFILL_SA
#define Q4_PREFILL_SA 6
#endif
#ifndef Q4_PREFILL_SB
#define Q4_PREFILL_SB 2
#endif
constexpr int kSA = Q4_PREFILL_SA;                   // TMA ring stages
constexpr int kSB = Q4_PREFILL_SB;                   // fp16 B ring stages
constexpr int kEpiWarps = 4;

// Per tile width BN (256, or 128 where 256-wide tiles leave SMs idle): one
// dequant warp per 16 columns; a stage holds {x 16 KB, packed words BN*32 B,
// scale pairs of up to two groups (BN*2 B each), their zero words (BN/2 B
// each)}, padded to 1 KB so every x tile keeps the 128-byte swizzle atom.
template <int BN_>
struct PfCfg {
    static constexpr int BN = BN_;
    static constexpr int kAOff = 0, kPOff = 16384;
    static constexpr int kSGroup = BN * 2, kZGroup = BN / 2;
    static constexpr int kSzOff = kPOff + BN * 32;
    static constexpr int kZOff = 2 * kSGroup;           // zero words after both groups' scales
    static constexpr int kAStage = ((kSzOff + 2 * kSGroup + 2 * kZGroup) + 1023) / 1024 * 1024;
    static constexpr int kBStage = BN * BK * 2;
    static constexpr int kRingB = kSA * kAStage;
    static constexpr int kBarOff = kRingB + kSB * kBStage;
    static constexpr int kNumBars = 2 * kSA + 2 * kSB + 4;
    static constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + 1024;
    static constexpr int kDqWarps = BN / 16;
    static constexpr int kThreads = 32 * (2 + kDqWarps + kEpiWarps);
    static constexpr uint32_t kTmemCols = 2 * BN;
    static_assert(kSmem <= 227 * 1024, "shared memory");
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
};

__device__ __forceinline__ void fail(int *status, int bit, int *abort_flag) {
    if (status) atomicOr(status, bit);
    atomicExch(abort_flag, 1);
}
__device__ __forceinline__ bool aborted(int *abort_flag) { return *reinterpret_cast<volatile int *>(abort_flag) != 0; }

template <int BNT>
__global__ void __launch_bounds__(PfCfg<BNT>::kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, PfArgs a) {
    using P = PfCfg<BNT>;
    constexpr int BN = P::BN, kAOff = P::kAOff, kPOff = P::kPOff, kSzOff = P::kSzOff, kZOff = P::kZOff;
    constexpr int kAStage = P::kAStage, kBStage = P::kBStage, kRingB = P::kRingB, kBarOff = P::kBarOff;
    constexpr int kNumBars = P::kNumBars, kDqWarps = P::kDqWarps;
    constexpr uint32_t kTmemCols = P::kTmemCols;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + kBarOff;
    auto fullA = [&](int s) { return bar0 + 8u * s; };
    auto emptyA = [&](int s) { return bar0 + 8u * (kSA + s); };
    auto fullB = [&](int s) { return bar0 + 8u * (2 * kSA + s); };
    auto emptyB = [&](int s) { return bar0 + 8u * (2 * kSA + kSB + s); };
    auto accF = [&](int i) { return bar0 + 8u * (2 * kSA + 2 * kSB + i); };
    auto accE = [&](int i) { return bar0 + 8u * (2 * kSA + 2 * kSB + 2 + i); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + kBarOff + kNumBars * 8);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = a.K / BK;
    const int NT16 = a.N >> 4;
    const int ntiles = a.tiles_m * a.tiles_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSA; ++s) {
            mbar_init(fullA(s), 1);
            mbar_init(emptyA(s), 1 + kDqWarps);
        }
        for (int s = 0; s < kSB; ++s) {
            mbar_init(fullB(s), kDqWarps);
            mbar_init(emptyB(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(accF(i), 1);
            mbar_init(accE(i), kEpiWarps);
        }
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
            int it = 0, s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
                const int m0 = (t % a.tiles_m) * BM;
                const int nt0 = (t / a.tiles_m) * (BN / 16);
                const int tiles16 = min(BN / 16, NT16 - nt0);
                const uint32_t sbytes = tiles16 * 32u, zbytes = tiles16 * 8u;
                int gcur = -1, left = 0;                 // group of the next 32-row block, blocks left in it
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    if (aborted(abort_flag)) { ok = false; break; }
                    if (!mbar_wait(emptyA(s), ph ^ 1)) { fail(a.status, 0x10, abort_flag); ok = false; break; }
                    if (left == 0) { ++gcur; left = a.bpg; }
                    const int g_first = gcur;
                    --left;
                    if (left == 0) { ++gcur; left = a.bpg; }
                    --left;
                    const int ng = gcur - g_first + 1;
                    const uint32_t st = base + s * kAStage;
                    mbar_arrive_expect_tx(fullA(s), 16384u + BN * 32u + ng * (sbytes + zbytes));
                    tma_load_2d(st + kAOff, &tmA, fullA(s), kb * BK, m0);
                    tma_load_2d(st + kPOff, &tmW, fullA(s), kb * 128, nt0);
                    for (int gi = 0; gi < ng; ++gi) {
                        const size_t gr = static_cast<size_t>(g_first + gi);
                        bulk_load(st + kSzOff + gi * P::kSGroup, a.s2 + (gr * NT16 + nt0) * 8, sbytes, fullA(s));
                        bulk_load(st + kSzOff + kZOff + gi * P::kZGroup, a.zeros + gr * (a.N >> 3) + nt0 * 2, zbytes,
                                  fullA(s));
                    }
                    if (++s == kSA) { s = 0; ph ^= 1; }
                }
            }
            if (aborted(abort_flag))
                for (int j = it > kSA ? it - kSA : 0; j < it; ++j) mbar_wait(fullA(j % kSA), (j / kSA) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(BM, BN, false);
            int it = 0, lt = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x, ++lt) {
                const int acc = lt & 1;
                const uint32_t aph = (lt >> 1) & 1;
                if (aborted(abort_flag) || !mbar_wait(accE(acc), aph ^ 1)) {
                    fail(a.status, 0x20, abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % kSA, sb = it % kSB;
                    if (aborted(abort_flag) || !mbar_poll(fullA(s), (it / kSA) & 1) ||
                        !mbar_poll(fullB(sb), (it / kSB) & 1)) {
                        fail(a.status, 0x20, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + s * kAStage + kAOff;
                    const uint32_t sbb = base + kRingB + sb * kBStage;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_f16(d, smem_desc_sw128(sa + kk * 32, 16, 1024), smem_desc_sw128(sbb + kk * 32, 16, 1024),
                                 idesc, (kb | kk) != 0);
                    umma_commit(emptyA(s));
                    umma_commit(emptyB(sb));
                }
                if (ok) umma_commit(accF(acc));
            }
        }
    } else if (warp < 2 + kDqWarps) {
        // ------------------------------------------------------ dequantizers
        // Lane -> packed-word assignment: in every 8-lane phase (p = lane >> 3)
        // the lanes take columns gq in {p, p ^ 5} and all four tq, so the
        // 16-byte loads of packed words and the 16-byte stores into the
        // swizzled B tile both hit eight distinct bank groups per phase.
        // Warp wl owns n16 tile wl of the 256-column tile.
        const int wl = warp - 2;
        const int pq = lane >> 3;
        const int gq = ((lane >> 2) & 1) ? (pq ^ 5) : pq;
        const int tq = lane & 3;
        const int ls = 4 * gq + tq;
        const uint32_t sw0 = static_cast<uint32_t>((tq ^ gq) << 4);
        const uint32_t sw1 = static_cast<uint32_t>(((4 + tq) ^ gq) << 4);
        uint32_t c_s[2][2], c_nl[2][2], c_nh[2][2];   // [half J][column gq / gq+8]
        auto load_consts = [&](const uint8_t *sz, int gl, int J) {
            const uint32_t sp = *reinterpret_cast<const uint32_t *>(sz + gl * P::kSGroup + (wl * 8 + gq) * 4);
            const uint2 zw = *reinterpret_cast<const uint2 *>(sz + kZOff + gl * P::kZGroup + wl * 8);
            c_s[J][0] = __byte_perm(sp, sp, 0x1010);
            c_s[J][1] = __byte_perm(sp, sp, 0x3232);
            const uint32_t z0 = (zw.x >> (4 * gq)) & 0xFu, z1 = (zw.y >> (4 * gq)) & 0xFu;
            c_nl[J][0] = neg_zlo(z0);
            c_nh[J][0] = neg_zhi(z0);
            c_nl[J][1] = neg_zlo(z1);
            c_nh[J][1] = neg_zhi(z1);
        };
        int s = 0, sb = 0;
        uint32_t ph = 0, phb = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
            int left = 0;                             // 32-row blocks left in the current group
            for (int kb = 0; kb < KB; ++kb) {
                if (aborted(abort_flag)) { ok = false; break; }
                if (!mbar_wait(fullA(s), ph) || !mbar_wait(emptyB(sb), phb ^ 1)) {
                    fail(a.status, 0x40, abort_flag);
                    ok = false;
                    break;
                }
                const uint8_t *st = sbase + s * kAStage;
                const uint8_t *sz = st + kSzOff;
                // first block: a new group starts here (slot 0) or continues from the
                // previous stage's second block, whose constants are already in slot 0
                if (left == 0) { load_consts(sz, 0, 0); left = a.bpg; }
                --left;
                const bool gl1 = left == 0;           // the second block starts a new group (slot 1)
                if (gl1) { load_consts(sz, 1, 1); left = a.bpg; }
                --left;
                const uint4 wv = *reinterpret_cast<const uint4 *>(st + kPOff + (wl * 32 + ls) * 16);
                const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
                uint8_t *brow = sbase + kRingB + sb * kBStage + 2 * wl * 1024 + gq * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int J = j >> 1, jj = j & 1;
                    const uint32_t sp = (J && gl1) ? c_s[1][jj] : c_s[0][jj];
                    const uint32_t nl = (J && gl1) ? c_nl[1][jj] : c_nl[0][jj];
                    const uint32_t nh = (J && gl1) ? c_nh[1][jj] : c_nh[0][jj];
                    uint32_t q[4];
                    unpack_qz(w[j], nl, nh, q);
                    *reinterpret_cast<uint4 *>(brow + jj * 1024 + (J ? sw1 : sw0)) =
                        make_uint4(hmul2(q[0], sp), hmul2(q[1], sp), hmul2(q[2], sp), hmul2(q[3], sp));
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(fullB(sb));
                    mbar_arrive(emptyA(s));
                }
                if (gl1) {                            // that group continues into the next stage
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        c_s[0][c] = c_s[1][c];
                        c_nl[0][c] = c_nl[1][c];
                        c_nh[0][c] = c_nh[1][c];
                    }
                }
                if (++s == kSA) { s = 0; ph ^= 1; }
                if (++sb == kSB) { sb = 0; phb ^= 1; }
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        const int quad = warp & 3;                  // TMEM lanes 32*quad .. +31
        int lt = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++lt) {
            const int acc = lt & 1;
            const uint32_t aph = (lt >> 1) & 1;
            bool ok = !aborted(abort_flag) && mbar_wait(accF(acc), aph);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) fail(a.status, 0x80, abort_flag);
                break;
            }
            tc_fence_after();
            const int m0 = (t % a.tiles_m) * BM;
            const int n0 = (t / a.tiles_m) * BN;
            const int row = m0 + 32 * quad + lane;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t r[32];
                tmem_ld_x32(tmem + static_cast<uint32_t>(acc * BN + c0) + (static_cast<uint32_t>(32 * quad) << 16), r);
                if (row < a.M) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int n = n0 + c0 + 8 * v;
                        if (n < a.N) {
                            uint32_t pk[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float lo = __uint_as_float(r[8 * v + 2 * e]);
                                float hi = __uint_as_float(r[8 * v + 2 * e + 1]);
                                if (a.bias) {
                                    lo += __half2float(__ushort_as_half(a.bias[n + 2 * e]));
                                    hi += __half2float(__ushort_as_half(a.bias[n + 2 * e + 1]));
                                }
                                pk[e] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(lo))) |
                                        (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(hi))) << 16);
                            }
                            *reinterpret_cast<uint4 *>(a.out + static_cast<size_t>(row) * a.N + n) =
                                make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(accE(acc));
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


template <int BN>
cudaError_t launch_prefill_bn(const HandleView &h, const uint16_t *x, int M, uint16_t *out, cudaStream_t s) {
    using P = PfCfg<BN>;
    CUtensorMap tmA, tmW;
    cudaError_t e;
    const int KC = h.K / 64;
    if ((e = encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, h.K, M, static_cast<uint64_t>(h.K) * 2, BK, BM,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, h.wp, static_cast<uint64_t>(KC) * 128, h.N / 16,
                       static_cast<uint64_t>(KC) * 512, 128, BN / 16, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
        return e;
    static cudaError_t attr =
        cudaFuncSetAttribute(prefill_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, P::kSmem);
    if (attr != cudaSuccess) return attr;
    PfArgs args{M, h.N, h.K, h.bias, out, h.status, h.s2, h.zeros, h.geff / 32, (M + BM - 1) / BM, (h.N + BN - 1) / BN};
    const int ntiles = args.tiles_m * args.tiles_n;
    const int grid = ntiles < sm_count() ? ntiles : sm_count();
    prefill_kernel<BN><<<grid, P::kThreads, P::kSmem, s>>>(tmA, tmW, args);
    return cudaGetLastError();
}

}  // namespace

// 256-column tiles unless they leave more than a quarter of the SMs without a
// tile (small M): then 128-column tiles, at the same cost per flop, twice as
// many of them.
cudaError_t launch_prefill(const HandleView &h, const uint16_t *x, int M, uint16_t *out, cudaStream_t s) {
    const long long tiles256 = static_cast<long long>((M + BM - 1) / BM) * ((h.N + 255) / 256);
    if (4 * tiles256 < 3LL * sm_count()) return launch_prefill_bn<128>(h, x, M, out, s);
    return launch_prefill_bn<256>(h, x, M, out, s);
}

int prefill_default_min_m() { return 64; }

}  // namespace q4
