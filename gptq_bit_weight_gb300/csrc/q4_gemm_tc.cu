// Dense fp16 GEMM on the 5th-generation tensor cores (tcgen05 / TMEM / TMA),
// sm_103a:  out = a . b + bias,  a [M][K] fp16 (K-major), b [K][N] fp16
// (N-major), fp32 accumulation, one rounding to fp16.  The matmul on the
// dequantized matrix temp_dq "during prefill" ("Implementation: Predibase
// Lorax GPTQ Exllama V1", "Description"): the unfused comparison route.  The
// fused route is in q4_prefill.cu.
//
// One CTA computes a 128 x 256 output tile with fp32 accumulators in tensor
// memory (256 TMEM columns).  Warp roles:
//   warp 0       one thread issues TMA loads (128-byte swizzle) of the a and b
//                tiles into a 4-stage ring of shared-memory stages
//   warp 1       allocates TMEM; one thread issues tcgen05.mma (M=128,
//                N=256, K=16) and commits each stage back to the producer
//   warps 2..5   read TMEM (tcgen05.ld), add bias in fp32, round once to fp16
//                and store.
// Every wait on an mbarrier is bounded (about two seconds of global time);
// a wait that runs out records an error bit in the caller's status word,
// stops its role, and the CTA still frees its TMEM before returning.
#include <cuda.h>
#include <cuda_fp16.h>

#include <climits>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "q4_internal.cuh"
#include "q4_tc.cuh"

namespace q4 {

namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kABytes = BM * BK * 2;         // 16 KB activation tile
constexpr int kBBytes = BN * BK * 2;         // 32 KB weight tile (fp16)
constexpr uint32_t kTmemCols = 256;

struct Cfg {
    static constexpr int kStages = 4;
    static constexpr int kAOff = 0;
    static constexpr int kBOff = kABytes;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kWorkerWarps = 4;
    static constexpr int kThreads = 64 + 32 * kWorkerWarps;
    static constexpr int kBarBytes = 8 * (2 * kStages + 1) + 16;
    static constexpr int kSmem = kStages * kStageBytes + kBarBytes + 1024;
};


struct TcArgs {
    int M, N, K;
    const uint16_t *bias;
    uint16_t *out;
    int *status;
    const uint32_t *s2;      // fused: scale pairs [G][N/16][8]
    const uint32_t *zeros;   // fused: zero words [G][N/8]
    int bpg;                 // fused: 32-row blocks per group
    const float *rowscale;   // epilogue: y = acc * rowscale[m] + bias (NULL: 1)
    int out_bf16;            // output rounded to bf16 instead of fp16
};

__device__ __forceinline__ void record_error(int *status, int bit, int *abort_flag) {
    if (status) atomicOr(status, bit);
    atomicExch(abort_flag, 1);
}

__global__ void __launch_bounds__(Cfg::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, TcArgs a) {
    using C = Cfg;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + S * C::kStageBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    const uint32_t done_bar = bar0 + 8u * (2 * S);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + S * C::kStageBytes + 8 * (2 * S + 1));
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int KB = a.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < KB; ++kb) {
                const int s = kb % S;
                const uint32_t ph = (kb / S) & 1;
                if (*reinterpret_cast<volatile int *>(abort_flag)) break;
                if (!mbar_wait(empty_bar(s), ph ^ 1)) {
                    record_error(a.status, 0x1, abort_flag);
                    break;
                }
                const uint32_t st = base + s * C::kStageBytes;
                const int nb = min(4, (a.N - n0) / 64);
                mbar_arrive_expect_tx(full_bar(s), kABytes + nb * (BK * 64 * 2));
                tma_load_2d(st + C::kAOff, &tmA, full_bar(s), kb * BK, m0);
                for (int j = 0; j < nb; ++j)
                    tma_load_2d(st + C::kBOff + j * (BK * 64 * 2), &tmB, full_bar(s), n0 + 64 * j, kb * BK);
                ++issued;
            }
            if (*reinterpret_cast<volatile int *>(abort_flag)) {
                // Let copies already in flight land before the CTA can exit.
                for (int kb = issued > S ? issued - S : 0; kb < issued; ++kb)
                    mbar_wait(full_bar(kb % S), (kb / S) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(BM, BN, true);
            bool ok = true;
            for (int kb = 0; kb < KB; ++kb) {
                const int s = kb % S;
                const uint32_t ph = (kb / S) & 1;
                if (*reinterpret_cast<volatile int *>(abort_flag) ||
                    !mbar_wait(full_bar(s), ph)) {
                    record_error(a.status, 0x2, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t st = base + s * C::kStageBytes;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint64_t ad = smem_desc_sw128(st + C::kAOff + kk * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(st + C::kBOff + kk * 2048, BK * 64 * 2, 1024);
                    umma_f16(tmem, ad, bd, idesc, (kb | kk) != 0);
                }
                umma_commit(empty_bar(s));
            }
            if (ok) umma_commit(done_bar);
        }
    } else {
        const int wi = warp - 2;
        // ------------------------------------------------ epilogue
        const bool have = !*reinterpret_cast<volatile int *>(abort_flag);
        bool ok = have && mbar_wait(done_bar, 0);
        if (have && !ok) record_error(a.status, 0x8, abort_flag);
        __syncwarp();
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            const int quad = warp & 3;
            constexpr int kColsPerWarp = BN * 4 / C::kWorkerWarps;
            const int c_beg = (wi >> 2) * kColsPerWarp;
            const int row = m0 + 32 * quad + lane;
#pragma unroll 1
            for (int c0 = c_beg; c0 < c_beg + kColsPerWarp; c0 += 32) {
                uint32_t r[32];
                tmem_ld_x32(tmem + (static_cast<uint32_t>(32 * quad) << 16) + c0, r);
                if (row < a.M) {
                    // one branch per 32 columns into fp16-only or bf16-only code
                    auto store = [&](auto bf16c) {
                        constexpr bool BF = decltype(bf16c)::value;
                        const float rs = BF && a.rowscale ? a.rowscale[row] : 1.f;
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int n = n0 + c0 + 8 * v;
                            if (n < a.N) {
                                uint32_t pk[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    pk[e] = out_pair_t<BF>(__uint_as_float(r[8 * v + 2 * e]),
                                                           __uint_as_float(r[8 * v + 2 * e + 1]), rs, a.bias, n + 2 * e);
                                *reinterpret_cast<uint4 *>(a.out + static_cast<size_t>(row) * a.N + n) =
                                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            }
                        }
                    };
                    if (a.out_bf16 == kOutF32) {
                        // raw fp32 sums, 32 bytes per 8 columns
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int n = n0 + c0 + 8 * v;
                            if (n < a.N) {
                                float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.out) +
                                                                         static_cast<size_t>(row) * a.N + n);
                                dst[0] = make_float4(__uint_as_float(r[8 * v]), __uint_as_float(r[8 * v + 1]),
                                                     __uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                                dst[1] = make_float4(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]),
                                                     __uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                            }
                        }
                    } else if (a.out_bf16) store(std::true_type{});
                    else store(std::false_type{});
                }
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
}

cudaError_t ensure_smem_attr() {
    static cudaError_t st = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 Cfg::kSmem);
    return st;
}

}  // namespace

// ----------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

cudaError_t encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *ptr, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_gemm_f16(const uint16_t *a, const uint16_t *b, const uint16_t *bias, int M, int K, int N,
                            uint16_t *out, int *status, cudaStream_t s, const float *rowscale, int out_bf16) {
    CUtensorMap tmA, tmB;
    cudaError_t e;
    if ((e = encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a, K, M, static_cast<uint64_t>(K) * 2, BK, BM,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, b, N, K, static_cast<uint64_t>(N) * 2, 64, BK,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = ensure_smem_attr()) != cudaSuccess) return e;
    TcArgs args{M, N, K, bias, out, status, nullptr, nullptr, 1, rowscale, out_bf16};
    dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
    tc_gemm_kernel<<<grid, Cfg::kThreads, Cfg::kSmem, s>>>(tmA, tmB, args);
    return cudaGetLastError();
}


}  // namespace q4
