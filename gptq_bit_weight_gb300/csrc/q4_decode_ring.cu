// Decode (M <= 16) GPTQ W4A16 matmul fed by a TMA ring.
//
// "GPTQ's 'Exllama Kernel Not Installed' Warning", "What the fallback
// actually does": weight-bound decoding is limited by memory bandwidth; the
// fused kernel reads packed weights, dequantizes them on chip and never
// writes a dequantized matrix.  "Inference Backends", "Numeric epilogues and
// input gradients": fp32 accumulation, bias added to the fp32 sum before one
// cast, split reductions in fp32 in a fixed order.
//
// CTA = one 128-column tile x one K slice; the K slices of a tile form a
// thread-block cluster and are summed through distributed shared memory.
//   warp 4      one thread: the slice's scale pairs and zero words once (bulk
//               copies), then a ring of kStages stages, each {x tile of 8*MT
//               rows x 64 fp16 (128-byte swizzle), packed-word tile 128
//               columns x 64 rows (4 KB)}, by TMA.  The first kStages weight
//               tiles are requested before the preceding grid has finished
//               (programmatic dependent launch): they are handle constants.
//   warps 0-3   warp w owns the 32 columns 32w..32w+31 (two n16 tiles) for
//               the whole slice; no reduction across the warps of a CTA.
//
// Arithmetic per packed word: one LOP3 per code pair gives the fp16 pair
// (1024 + q) for rows with even nibble index and (1024 + 16 q) for the
// others (the 0x6400 exponent pattern; Kim et al. 2022, "Who Says Elephants
// Can't Run").  No fp16 subtraction follows: the two kinds go to two
// m16n8k16 MMA accumulators, Dlo and Dhi, and one more MMA per kind with an
// all-ones A operand accumulates the sums of x that met them, Slo and Shi.
// At the end of a quantization group, per column (zero point z, scale s):
//     sum_k x (q - z - 1) = Dlo - (1025 + z) Slo + (Dhi - (1040 + 16 z) Shi) / 16
// and acc += s * that, in fp32.  Products on the tensor cores are exact; the
// only rounding is fp32 accumulation.
// Group slots (M <= 4): an m16n8k16 MMA has 8 B columns and M rows of x use
// only MP of them (MP = M rounded up to a power of two).  The other columns
// then carry the next groups: B column c holds x row c % MP while the
// slice is in its (c / MP)-th group of the current batch of 8 / MP groups,
// and zeros otherwise.  So D, Slo and Shi keep each group of a batch apart,
// and the per-group step above runs once per batch instead of once per
// group.  At the end the slots of each row are summed across the lanes.  The stage is released once the MMAs
// have consumed every register loaded from it, so no load of it can still
// be outstanding when the producer refills it.
// Every mbarrier wait is bounded (~2 s); a wait that runs out records an
// error bit in the handle's status word and the CTA lets its copies land and
// returns.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdlib>
#include <cstdint>

#include "q4_internal.cuh"
#include "q4_tc.cuh"

namespace q4 {

cudaError_t encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *ptr, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

namespace {

using namespace tc;

constexpr int BN = 128;                              // columns per CTA (8 n16 tiles)
constexpr int BK = 64;                               // rows per stage
#ifndef Q4_RING_TPW
#define Q4_RING_TPW 2
#endif
constexpr int kTPW = Q4_RING_TPW;                    // n16 tiles per consumer warp
constexpr int kCW = (BN / 16) / kTPW;                // consumer warps
constexpr int kThreads = 32 * (kCW + 1);
#ifndef Q4_RING_STAGES
#define Q4_RING_STAGES 8
#endif
constexpr int kStages = Q4_RING_STAGES;
constexpr int kWBytes = BN * BK / 2;                 // packed words per stage (4 KB)
constexpr int kMaxGroups = 48;                       // groups a slice may touch
constexpr int kSzGroupBytes = 8 * 8 * 4 + 16 * 4;    // scale pairs (8 n16 tiles) + zero words
constexpr int kMaxCluster = 8;

template <int MT>
struct RingCfg {
    static constexpr int kXBytes = 8 * MT * 128;     // x tile, 128-byte rows
    static constexpr int kStage = kXBytes + kWBytes; // multiple of 1024: x tiles stay swizzle-aligned
    static constexpr int kSzOff = kStages * kStage;
    static constexpr int kRedOff = kSzOff + kMaxGroups * kSzGroupBytes;
    static constexpr int kBarOff = kRedOff + 8 * MT * BN * 4;
    static constexpr int kNumBars = 2 * kStages + 1;
    static constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + 1024;   // + base alignment slack
    static_assert(kStage % 1024 == 0, "stage size must keep 1024-byte alignment");
};

struct RingArgs {
    int M, N, K;
    const uint16_t *bias;
    uint16_t *out;
    int *status;
    const uint32_t *s2;
    const uint32_t *zeros;
    int bpg;             // 32-row blocks per group
    int zero_offset;     // effective zero = stored + zero_offset
    int zsplit;          // groups [0, zsplit) take zero offset 0
    const float *rowscale;   // epilogue: y = acc * rowscale[m] + bias (NULL: 1)
    int out_bf16;            // output rounded to bf16 instead of fp16
    int slice_kb;        // stages per slice
    int splits;
};

__device__ __forceinline__ void fail(int *status, int bit, int *abort_flag) {
    if (status) atomicOr(status, bit);
    atomicExch(abort_flag, 1);
}
__device__ __forceinline__ bool aborted(int *abort_flag) { return *reinterpret_cast<volatile int *>(abort_flag) != 0; }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
template <int MT, int MP>
__global__ void __launch_bounds__(kThreads, 3)
    decode_ring_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, RingArgs a) {
    static_assert(MP == 8 || (MT == 1 && (MP == 1 || MP == 2 || MP == 4)), "group slots need one m tile");
    constexpr int kSlots = 8 / MP;                   // groups per batch
    using C = RingCfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + C::kBarOff;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
    const uint32_t szBar = bar0 + 8u * (2 * kStages);
    int *abort_flag = reinterpret_cast<int *>(sbase + C::kBarOff + C::kNumBars * 8);
    const uint32_t szb = base + C::kSzOff;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT16 = a.N >> 4;
    const int nt0 = blockIdx.x * (BN / 16);
    const int n0 = blockIdx.x * BN;
    const int split = blockIdx.y;
    const int m0 = blockIdx.z * 8 * MT;
    const int mrows = min(8 * MT, a.M - m0);
    const int KB = a.K / BK;
    const int kb_beg = split * a.slice_kb;
    const int kb_end = min(KB, kb_beg + a.slice_kb);
    const int nkb = kb_end - kb_beg;
    const int g_beg = (2 * kb_beg) / a.bpg;
    const int ng = (2 * kb_end - 1) / a.bpg + 1 - g_beg;

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kCW);                // each consumer warp releases the stage once
        }
        mbar_init(szBar, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();

    float acc[kTPW][MT][4];
#pragma unroll
    for (int t = 0; t < kTPW; ++t)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[t][mt][i] = 0.f;

    if (warp == kCW) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            // scale pairs and zero words of the slice's groups for this tile's
            // n16 tiles (a last tile of 64 columns copies only its 4 valid ones)
            const int tv = min(8, NT16 - nt0);
            mbar_arrive_expect_tx(szBar, static_cast<uint32_t>(ng) * tv * 40u);
            for (int gl = 0; gl < ng; ++gl) {
                const size_t gr = static_cast<size_t>(g_beg + gl);
                bulk_load(szb + gl * kSzGroupBytes, a.s2 + (gr * NT16 + nt0) * 8, tv * 32u, szBar);
                bulk_load(szb + gl * kSzGroupBytes + 256, a.zeros + gr * (a.N >> 3) + nt0 * 2, tv * 8u, szBar);
            }
            constexpr uint32_t kTx = C::kXBytes + kWBytes;
            const int pre = min(kStages, nkb);
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(full(i), kTx);
                tma_load_2d(base + i * C::kStage + C::kXBytes, &tmW, full(i), (kb_beg + i) * 128, nt0);
            }
            griddep_wait();                          // x may be written by the preceding grid
            for (int i = 0; i < pre; ++i)
                tma_load_2d(base + i * C::kStage, &tmX, full(i), (kb_beg + i) * BK, m0);
            int issued = pre;
            int s = 0;
            uint32_t ph = 1;                         // parity of the empty phase a refill waits for
            if (pre == kStages) {
                for (int i = pre; i < nkb; ++i) {
                    if (aborted(abort_flag)) break;
                    if (!mbar_wait(empty(s), ph ^ 1)) {
                        fail(a.status, 0x100, abort_flag);
                        break;
                    }
                    const uint32_t st = base + s * C::kStage;
                    mbar_arrive_expect_tx(full(s), kTx);
                    tma_load_2d(st + C::kXBytes, &tmW, full(s), (kb_beg + i) * 128, nt0);
                    tma_load_2d(st, &tmX, full(s), (kb_beg + i) * BK, m0);
                    ++issued;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (aborted(abort_flag)) {               // let every requested copy land before exiting
                mbar_wait(szBar, 0);
                for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
                    mbar_wait(full(j % kStages), (j / kStages) & 1);
            }
        }
    } else {
        // ---------------------------------------------------------- consumers
        const int gq = lane >> 2, tq = lane & 3;
        const bool wactive = nt0 + kTPW * warp < NT16; // a 64-column last tile idles warps 2-3
        bool ok = mbar_wait(szBar, 0);
        if (!ok) fail(a.status, 0x400, abort_flag);
        float dlo[kTPW][MT][4], dhi[kTPW][MT][4], slo[MT][4], shi[MT][4];
        auto clear_partials = [&]() {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    slo[mt][i] = 0.f;
                    shi[mt][i] = 0.f;
#pragma unroll
                    for (int t = 0; t < kTPW; ++t) dlo[t][mt][i] = dhi[t][mt][i] = 0.f;
                }
        };
        clear_partials();
        // The batch's groups start at slice group gb0.  Accumulator element
        // i of a lane sits in B column 2 tq + (i & 1), i.e. slot
        // (2 tq + (i & 1)) / MP; with MP >= 2 both elements of a lane share
        // one slot, with MP = 1 they are two.  Per slot and column (gq,
        // gq + 8): scale s, -(1024 + z), -(64 + z).  A slot past the slice's
        // last group has all-zero partials; it reads the last group's
        // constants (finite), so it adds exactly zero.
        int gb0 = 0;
        auto flush = [&]() {
            constexpr int kLaneSlots = MP == 1 ? 2 : 1;
#pragma unroll
            for (int t = 0; t < kTPW; ++t) {
                const int nt = kTPW * warp + t;
#pragma unroll
                for (int j = 0; j < kLaneSlots; ++j) {
                    const int gle = min(gb0 + (2 * tq + j) / MP, ng - 1);
                    const uint32_t gb = szb + gle * kSzGroupBytes;
                    const uint32_t sp = ld_shared_u32(gb + (nt * 8 + gq) * 4);
                    const uint32_t zw0 = ld_shared_u32(gb + 256 + nt * 8);
                    const uint32_t zw1 = ld_shared_u32(gb + 256 + nt * 8 + 4);
                    float sc[2], czl[2], czh[2];
                    sc[0] = __half2float(__ushort_as_half(static_cast<unsigned short>(sp & 0xFFFFu)));
                    sc[1] = __half2float(__ushort_as_half(static_cast<unsigned short>(sp >> 16)));
                    // effective zero points (stored + zero offset) of columns gq, gq + 8
                    const uint32_t zoff = g_beg + gle < a.zsplit ? 0u : static_cast<uint32_t>(a.zero_offset);
                    const float z0 = static_cast<float>(((zw0 >> (4 * gq)) & 0xFu) + zoff);
                    const float z1 = static_cast<float>(((zw1 >> (4 * gq)) & 0xFu) + zoff);
                    czl[0] = -(1024.f + z0);
                    czl[1] = -(1024.f + z1);
                    czh[0] = -(64.f + z0);
                    czh[1] = -(64.f + z1);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            if (kLaneSlots == 2 && (i & 1) != j) continue;
                            const int c = i >> 1;
                            float p = fmaf(czl[c], slo[mt][i], dlo[t][mt][i]);
                            p = fmaf(0.0625f, dhi[t][mt][i], p);
                            p = fmaf(czh[c], shi[mt][i], p);
                            acc[t][mt][i] = fmaf(sc[c], p, acc[t][mt][i]);
                        }
                }
            }
            clear_partials();
        };
        // this lane's x row in each m tile and its 16-byte chunk of each
        // 32-row block inside the 128-byte swizzled row (0xFFFFFFFF: row >= M);
        // with group slots, lane gq serves row gq % MP in slot gq / MP
        uint32_t xoff[2][MT];
        const int my_slot = gq / MP;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int r = mt * 8 + (MP == 8 ? gq : gq % MP);
                xoff[hh][mt] = r < mrows ? static_cast<uint32_t>(r * 128 + ((((hh << 2) | tq) ^ (r & 7)) << 4))
                                         : 0xFFFFFFFFu;
            }
        constexpr uint32_t kOnes = 0x3C003C00u;
        const uint32_t ones[4] = {kOnes, kOnes, kOnes, kOnes};
        int gl = 0;
        int slot = 0;                                       // slot of group gl in its batch
        int left = a.bpg - (2 * kb_beg - g_beg * a.bpg);   // 32-row blocks left in the current group
        int s = 0;
        uint32_t ph = 0;
        for (int i = 0; ok && i < nkb; ++i) {
            if (!mbar_wait(full(s), ph)) {
                fail(a.status, 0x800, abort_flag);
                break;
            }
            if (wactive) {
                const uint32_t st = base + s * C::kStage;
                uint4 wv[kTPW];
#pragma unroll
                for (int t = 0; t < kTPW; ++t) wv[t] = ld_shared_v4(st + C::kXBytes + (kTPW * warp + t) * 512 + lane * 16);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (left == 0) {
                        ++gl;
                        if (++slot == kSlots) {
                            flush();
                            gb0 = gl;
                            slot = 0;
                        }
                        left = a.bpg;
                    }
                    --left;
                    uint4 xb[MT];
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        xb[mt] = xoff[hh][mt] != 0xFFFFFFFFu && (MP == 8 || my_slot == slot)
                                     ? ld_shared_v4(st + xoff[hh][mt])
                                     : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        mma_16816(slo[mt], ones, xb[mt].x, xb[mt].z);
                        mma_16816(shi[mt], ones, xb[mt].y, xb[mt].w);
                    }
#pragma unroll
                    for (int t = 0; t < kTPW; ++t) {
                        uint32_t al[4], ah[4];
                        unpack_raw(hh ? wv[t].z : wv[t].x, al);      // column 16nt + gq
                        unpack_raw(hh ? wv[t].w : wv[t].y, ah);      // column 16nt + gq + 8
                        const uint32_t alo[4] = {al[0], ah[0], al[2], ah[2]};
                        const uint32_t ahi[4] = {al[1], ah[1], al[3], ah[3]};
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            mma_16816(dlo[t][mt], alo, xb[mt].x, xb[mt].z);
                            mma_16816(dhi[t][mt], ahi, xb[mt].y, xb[mt].w);
                        }
                    }
                }
            }
            // every register loaded from the stage has been consumed above
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
            if (++s == kStages) {
                s = 0;
                ph ^= 1;
            }
        }
        if (wactive) {
            flush();
            if (MP < 8) {
                // sum each row's slots: element i of lane tq is column
                // 2 tq + (i & 1) = slot * MP + row
#pragma unroll
                for (int t = 0; t < kTPW; ++t) {
                    float v[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] = acc[t][0][i] + (MP == 1 ? acc[t][0][i ^ 1] : 0.f);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (MP <= 2) v[i] += __shfl_xor_sync(0xFFFFFFFFu, v[i], 1);
                        v[i] += __shfl_xor_sync(0xFFFFFFFFu, v[i], 2);
                        acc[t][0][i] = v[i];            // valid where 2 tq + (i & 1) < MP
                    }
                }
            }
        }
    }

    // ------------------------------------------------------------ epilogue
    // out may still be read by the preceding grid: wait for it before the
    // first store.
    griddep_wait();
    const int gq = lane >> 2, tq = lane & 3;
    if (a.splits == 1) {
        if (warp < kCW && !aborted(abort_flag)) {
#pragma unroll
            for (int t = 0; t < kTPW; ++t)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int n = n0 + 16 * (kTPW * warp + t) + gq + 8 * (i >> 1);
                        const int m = m0 + mt * 8 + 2 * tq + (i & 1);
                        if (m < a.M && n < a.N) {
                            if (a.out_bf16 == kOutF32)
                                reinterpret_cast<float *>(a.out)[static_cast<size_t>(m) * a.N + n] = acc[t][mt][i];
                            else
                                a.out[static_cast<size_t>(m) * a.N + n] =
                                    out_one(acc[t][mt][i], a.rowscale ? a.rowscale[m] : 1.f, a.bias, n, a.out_bf16);
                        }
                    }
        }
        return;
    }
    // The K slices of this tile form one cluster: sum the slices' partial
    // tiles in slice order out of each other's shared memory.  Rank r
    // finishes the elements e of the 8*MT x 128 tile with e % splits == r.
    float *red = reinterpret_cast<float *>(sbase + C::kRedOff);
    if (warp < kCW) {
#pragma unroll
        for (int t = 0; t < kTPW; ++t)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    red[(mt * 8 + 2 * tq + (i & 1)) * BN + 16 * (kTPW * warp + t) + gq + 8 * (i >> 1)] = acc[t][mt][i];
    }
    cluster_sync();
    if (!aborted(abort_flag)) {
        const uint32_t red_local = base + C::kRedOff;
        for (int e = threadIdx.x; e < 8 * MT * BN; e += kThreads) {
            const int ml = e / BN, nl = e % BN;
            if (e % a.splits != split || ml >= mrows || n0 + nl >= a.N) continue;
            float v = 0.f;
            for (int r = 0; r < a.splits; ++r) v += ld_dsmem_f32(red_local + e * 4, r);
            if (a.out_bf16 == kOutF32)
                reinterpret_cast<float *>(a.out)[static_cast<size_t>(m0 + ml) * a.N + n0 + nl] = v;
            else
                a.out[static_cast<size_t>(m0 + ml) * a.N + n0 + nl] =
                    out_one(v, a.rowscale ? a.rowscale[m0 + ml] : 1.f, a.bias, n0 + nl, a.out_bf16);
        }
    }
    cluster_sync();                                   // partials stay alive until all are read
}

template <int MT, int MP>
cudaError_t ensure_attr() {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return dyn_smem_optin(reinterpret_cast<const void *>(decode_ring_kernel<MT, MP>), dev, RingCfg<MT>::kSmem,
                          nullptr);
}

// Rows of x per group slot for M rows (8: no slots)
int slot_rows(int M, int mt) {
    static const bool on = [] {
        const char *v = getenv("GPTQ_Q4_RING_SLOTS");
        return !(v && v[0] == '0');
    }();
    if (!on || mt != 1 || M > 4) return 8;
    return M == 1 ? 1 : (M == 2 ? 2 : 4);
}

template <int MT, int MP>
cudaError_t launch_variant(cudaLaunchConfig_t &cfg, const CUtensorMap &tmX, const CUtensorMap &tmW,
                           const RingArgs &args) {
    cudaError_t e;
    if ((e = ensure_attr<MT, MP>()) != cudaSuccess) return e;
    cfg.dynamicSmemBytes = RingCfg<MT>::kSmem;
    return cudaLaunchKernelEx(&cfg, decode_ring_kernel<MT, MP>, tmX, tmW, args);
}

}  // namespace

// Co-resident clusters of `sp` CTAs (one K slice each) the device can hold
// for the MT variant, from the occupancy calculator; queried once per MT on
// the first device that asks.
template <int MT>
int max_active_clusters(int sp) {
    static int table[kMaxCluster + 1] = {};
    static bool done = false;
    if (!done) {
        done = true;
        if (ensure_attr<MT, 8>() == cudaSuccess) {
            for (int c = 1; c <= kMaxCluster; ++c) {
                cudaLaunchConfig_t cfg{};
                cfg.gridDim = dim3(1, c, 1);
                cfg.blockDim = dim3(kThreads);
                cfg.dynamicSmemBytes = RingCfg<MT>::kSmem;
                cudaLaunchAttribute attr;
                attr.id = cudaLaunchAttributeClusterDimension;
                attr.val.clusterDim.x = 1;
                attr.val.clusterDim.y = static_cast<unsigned>(c);
                attr.val.clusterDim.z = 1;
                cfg.attrs = &attr;
                cfg.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, decode_ring_kernel<MT, 8>, &cfg) != cudaSuccess) n = 0;
                table[c] = n;
            }
        }
        cudaGetLastError();                          // a failed query leaves no sticky error
    }
    return table[sp];
}

// Slices: whole stages, at most kMaxGroups groups and at most 8 per tile
// (portable cluster size).  The split count is the largest one whose
// clusters (one per 128-column tile) can all be resident at once, so the
// grid is a single wave; when even one slice per tile needs more than one
// wave, one slice per tile.
DecodeRingPlan plan_decode_ring(int M, int K, int N, int geff, int sms) {
    DecodeRingPlan p{};
    if (M < 1 || M > 16 || K % BK != 0 || N % 64 != 0 || geff % 32 != 0) return p;
    const int mt = M > 8 ? 2 : 1;
    const int KB = K / BK;
    const int bpg = geff / 32;
    const int tiles = (N + BN - 1) / BN;
    int best = -1;
    for (int sp = 1; sp <= std::min(kMaxCluster, KB); ++sp) {
        const int slice = (KB + sp - 1) / sp;
        if ((KB + slice - 1) / slice != sp) continue;  // no empty slice
        if ((slice * 2 + bpg - 1) / bpg + 1 > kMaxGroups) continue;
        int fit = mt == 1 ? max_active_clusters<1>(sp) : max_active_clusters<2>(sp);
        if (fit <= 0) fit = (3 * sms) / sp;            // occupancy query unavailable: three CTAs per SM
        if (best < 0 || tiles <= fit) best = sp;       // first feasible, then the largest that fits one wave
    }
    if (best < 0) return p;
    p.ok = 1;
    p.mt = mt;
    p.splits = best;
    p.slice_kb = (KB + best - 1) / best;
    p.tiles = tiles;
    return p;
}

int device_sm_count() {
    static const int sms = [] {
        int dev = 0, n = kSMs;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n;
    }();
    return sms;
}

cudaError_t launch_decode_ring(const HandleView &h, const DecodeRingPlan &p, const uint16_t *x, int M, uint16_t *out,
                               cudaStream_t s) {
    if (!p.ok || p.splits < 1 || p.splits > kMaxCluster || M < 1 || M > 8 * p.mt) return cudaErrorInvalidValue;
    CUtensorMap tmX, tmW;
    cudaError_t e;
    const int KC = h.K / 64;
    if ((e = encode_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, h.K, M, static_cast<uint64_t>(h.K) * 2, BK,
                       8 * p.mt, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = encode_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, h.wp, static_cast<uint64_t>(KC) * 128, h.N / 16,
                       static_cast<uint64_t>(KC) * 512, 128, 8, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
        return e;
    RingArgs args{M, h.N, h.K, h.bias, out, h.status, h.s2, h.zeros, h.geff / 32, h.zero_offset, h.zsplit,
                  h.rowscale, h.out_bf16, p.slice_kb, p.splits};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.tiles, p.splits, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (p.splits > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 1;
        attrs[na].val.clusterDim.y = static_cast<unsigned>(p.splits);
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl_enabled()) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    if (p.mt == 2) return launch_variant<2, 8>(cfg, tmX, tmW, args);
    switch (slot_rows(M, p.mt)) {
        case 1: return launch_variant<1, 1>(cfg, tmX, tmW, args);
        case 2: return launch_variant<1, 2>(cfg, tmX, tmW, args);
        case 4: return launch_variant<1, 4>(cfg, tmX, tmW, args);
        default: return launch_variant<1, 8>(cfg, tmX, tmW, args);
    }
}

}  // namespace q4
