// Decode (M <= 8) GPTQ W4A16 matmul with a stream-K split and group slots.
//
// "GPTQ's 'Exllama Kernel Not Installed' Warning", "What the fallback
// actually does": weight-bound decoding is limited by memory bandwidth; the
// fused kernel reads the packed weights once, dequantizes them on chip and
// never writes a dequantized matrix.  "Inference Backends", "Numeric
// epilogues and input gradients": fp32 accumulation, fp32 split reductions in
// a fixed order (no atomic partial-output reduction), bias added to the fp32
// sum before the one final cast.
//
// Work split (stream-K).  The layer is cut into units of 32 output columns
// (two n16 tiles) x 64 rows (one chunk), numbered tile by tile along K:
// u = tile * KC + chunk.  Every warp of the grid is an independent worker and
// takes one contiguous run of floor(U / W) or ceil(U / W) units, so each warp
// streams the same number of weight bytes (to one chunk) whatever the shape:
// no wave of CTAs is left half full.  A run covers the end of one tile and
// the start of the next (or more); each piece is a "segment".  A tile cut
// into several segments is finished by the last of its workers to arrive
// (an atomic ticket; nobody waits), which sums the segments' fp32 partials
// in segment order, so the result does not depend on arrival order.
//
// Ring.  Each warp owns a ring of slots in shared memory (8, or 4 with eight
// rows of x), each holding one unit's packed words (16 bytes per lane and
// n16 tile) and its x fragments (MP rows x 64 fp16), filled by asynchronous
// copies, one commit group per unit, all but one slot in flight.  The unit
// loop is not unrolled: its body stays small enough for the instruction
// cache (an unrolled body measured slower, stalled on instruction fetch).  The first units' weights are requested
// before the preceding grid has finished (programmatic dependent launch; they
// are handle constants); x, the workspace, tickets and out only after.
//
// Arithmetic per packed word, as in the other decode kernels: one LOP3 per
// code pair gives the fp16 pair 1024 + q (rows of even nibble index) or
// 1024 + 16 q (odd), exact (the 0x6400 exponent pattern of 1024; Kim et al.
// 2022, "Who Says Elephants Can't Run"); m16n8k16 MMAs accumulate, per kind,
// the products with x (Dlo, Dhi) and the sums of x that met them (Slo, Shi,
// from an all-ones A operand).  At the end of a group, per column (zero point
// z, scale s):  sum_k x (q - z - 1) = Dlo - (1024 + z + 1) Slo
// + (Dhi - 16 (64 + z + 1) Shi) / 16, and acc += s * that, in fp32.
//
// Group slots.  An m16n8k16 MMA has 8 B columns and the M rows of x fill MP
// of them (MP = 2 for one or two rows, else M rounded up to a power of two,
// so that a lane's two accumulator columns always share one slot).  The other columns carry the
// next groups: B column c holds x row c % MP while the run is in group
// c / MP of the current batch of 8 / MP groups, and zeros otherwise, so the
// per-group step above runs once per batch instead of once per group; at the
// end of a segment the slots of each row are summed across the lanes.
#include <cuda_fp16.h>

#include <algorithm>

#include "q4_internal.cuh"

#ifndef Q4_SK_NTW
#define Q4_SK_NTW 2
#endif

namespace q4 {

namespace {

#ifndef Q4_SK_WARPS
#define Q4_SK_WARPS 8
#endif
constexpr int kWarps = Q4_SK_WARPS;
constexpr int kThreads = 32 * kWarps;
// ring slots per warp (depth - 1 units in flight), a power of two: 8, or 4
// with eight rows of x per slot (two CTAs per SM must fit in shared memory)
#ifndef Q4_SK_DEPTH
#define Q4_SK_DEPTH 8
#endif
#ifndef Q4_SK_CTAS
#define Q4_SK_CTAS 2
#endif
constexpr int depth_for(int mp) { return mp == 8 ? (Q4_SK_DEPTH < 4 ? Q4_SK_DEPTH : 4) : Q4_SK_DEPTH; }
constexpr int kCtasPerSm = Q4_SK_CTAS;
constexpr int kMinUnits = 4;            // fewest units per worker

// Ring slot: the unit's packed words (NTW x 512 bytes) and its x fragments
// (MP rows x 128 bytes).  After the ring, per warp: the segment's fp32
// accumulators, NTW x 16 bytes per lane (touched only when a batch of groups
// is flushed), and 128 bytes of zeros that lanes outside the current group
// slot read instead of x (so no select is needed per MMA).
template <int MP, int NTW>
struct SkCfg {
    static constexpr int kDepth = depth_for(MP);
    static constexpr int kXOff = NTW * 512;
    static constexpr int kSlot = kXOff + MP * 128;    // multiple of 16
    static constexpr int kAccOff = kDepth * kSlot;
    static constexpr int kZeroOff = kAccOff + NTW * 512;
    static constexpr int kWarpBytes = kZeroOff + 128;
    static constexpr int kSmem = kWarps * kWarpBytes;
};

struct SkArgs {
    const uint16_t *x;
    uint16_t *out;
    float *ws;              // [T][smax][8 rows][16 NTW columns] fp32 partials
    int *tickets;           // [T], zero between calls
    int M;
    int T;                  // tiles of 16 NTW columns
    int KC;                 // 64-row chunks per tile
    long long U;            // units = T * KC
    int workers;            // active warps, <= U
    int smax;               // workspace slots per tile
};

// D += A . B, m16n8k16, fp16 inputs, fp32 accumulators; no side effects, so
// the compiler may schedule it freely among the loop's other instructions.
__device__ __forceinline__ void mma_f32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Worker owning unit u (workers take [floor(w U / W), floor((w + 1) U / W))).
__device__ __forceinline__ int owner(long long u, long long U, int W) {
    return static_cast<int>(((u + 1) * W - 1) / U);
}

template <int MP, int NTW>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_sk_kernel(HandleView h, SkArgs a) {
    static_assert(MP == 2 || MP == 4 || MP == 8, "rows per slot");
    constexpr int S = 8 / MP;                         // group slots per batch
    constexpr int kCols = 16 * NTW;                   // columns per tile
    constexpr int kPart = 8 * kCols;                  // partial floats per segment
    using C = SkCfg<MP, NTW>;
    constexpr int kDepth = C::kDepth;
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    const int wid = blockIdx.x * kWarps + warp;

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (wid >= a.workers) return;

    const int K = h.K, N = h.N, KC = a.KC, NT16 = N >> 4;
    const long long u0 = static_cast<long long>(wid) * a.U / a.workers;
    const long long u1 = static_cast<long long>(wid + 1) * a.U / a.workers;
    const int n_units = static_cast<int>(u1 - u0);
    unsigned char *ring = smem + warp * C::kWarpBytes;
    // the warp's zero area
    if (lane < 8) *reinterpret_cast<uint4 *>(ring + C::kZeroOff + lane * 16) = make_uint4(0, 0, 0, 0);
    __syncwarp();

    // Fill cursor: word offset (in 16-byte vectors) of the next unit's first
    // n16 tile, (NTW t KC + c) 32, and its chunk c.
    const int t_first = static_cast<int>(u0 / KC);
    int fc = static_cast<int>(u0 - static_cast<long long>(t_first) * KC);
    uint32_t fw = (static_cast<uint32_t>(NTW * t_first) * KC + fc) * 32u;
    const uint32_t tile_stride = static_cast<uint32_t>(KC) * 32u;    // between n16 tiles of one unit
    const uint4 *wsrc = h.wp + lane;
    const bool xcopy = gq < MP && gq < a.M;           // this lane copies x row gq
    const uint16_t *xsrc = a.x + static_cast<size_t>(xcopy ? gq : 0) * K + 8 * tq;
    unsigned char *const wdst = ring + lane * 16;
    unsigned char *const xdst = ring + C::kXOff + gq * 128 + tq * 16;
    auto copy_w = [&](int slot) {
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) cp_async_16(wdst + slot * C::kSlot + nt * 512, wsrc + fw + nt * tile_stride);
    };
    auto copy_x = [&](int slot, int c) {
        if (xcopy) {
            cp_async_16(xdst + slot * C::kSlot, xsrc + c * 64);
            cp_async_16(xdst + slot * C::kSlot + 64, xsrc + c * 64 + 32);
        }
    };
    auto advance = [&]() {
        fw += 32u;
        if (++fc == KC) {
            fc = 0;
            fw += static_cast<uint32_t>(NTW - 1) * tile_stride;
        }
    };

    // ---- prologue: weights of the first kDepth - 1 units (one group each),
    //      then, once the preceding grid is done, their x (one more group)
    const int pre = min(kDepth - 1, n_units);
    {
        const int c0 = fc;
#pragma unroll
        for (int i = 0; i < kDepth - 1; ++i) {
            if (i < pre) {
                copy_w(i);
                advance();
            }
            cp_async_commit();
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int cc = c0;
#pragma unroll
        for (int i = 0; i < kDepth - 1; ++i) {
            if (i < pre) copy_x(i, cc);
            if (++cc == KC) cc = 0;
        }
        cp_async_commit();
    }

    constexpr uint32_t kOnes = 0x3C003C00u;
    const uint32_t ones[4] = {kOnes, kOnes, kOnes, kOnes};
    const int bpg = h.geff >> 5;                      // 32-row blocks per group
    const int G = h.G;

    // per-segment state
    float dlo[NTW][4], dhi[NTW][4], slo[4], shi[4];
    float4 *const accs = reinterpret_cast<float4 *>(ring + C::kAccOff) + lane;     // [nt][lane]
    // the current batch's constants, per lane slot j and n16 tile: scale
    // pair, zero words of columns gq (word 0) and gq + 8 (word 1)
    uint32_t csc[NTW], cz0[NTW], cz1[NTW];
    uint32_t gzoff;
    int seg_t = 0, gb0 = 0, slot = 0, left = 0;
    // lanes whose B column belongs to the current slot read x (at this offset
    // within a ring slot), the others the warp's zero area
    const int x_real = C::kXOff + (gq % MP) * 128 + tq * 16;
    const unsigned char *const xzero = ring + C::kZeroOff + tq * 16;
    bool xuse = true;
    auto set_xoff = [&]() { xuse = (S == 1 || gq / MP == slot) && (gq % MP) < a.M; };
    auto clear_partials = [&]() {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            slo[i] = 0.f;
            shi[i] = 0.f;
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) dlo[nt][i] = dhi[nt][i] = 0.f;
        }
    };
    // the lane's accumulators hold B columns 2 tq and 2 tq + 1: slot 2 tq / MP,
    // group gb0 + 2 tq / MP
    auto load_batch = [&]() {
        const int gr = min(gb0 + (2 * tq) / MP, G - 1);
        gzoff = gr < h.zsplit ? 0u : static_cast<uint32_t>(h.zero_offset);
        const uint32_t *sp = h.s2 + (static_cast<size_t>(gr) * NT16 + NTW * seg_t) * 8 + gq;
        const uint32_t *zw = h.zeros + static_cast<size_t>(gr) * (N >> 3) + NTW * seg_t * 2;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
            csc[nt] = __ldg(sp + nt * 8);
            cz0[nt] = __ldg(zw + nt * 2);
            cz1[nt] = __ldg(zw + nt * 2 + 1);
        }
    };
    auto flush = [&]() {
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
            float4 a4 = accs[nt * 32];
            float acc[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t sp = csc[nt];
                const uint32_t zw = (i >> 1) ? cz1[nt] : cz0[nt];
                const float s = __half2float(__ushort_as_half(static_cast<unsigned short>((i >> 1) ? sp >> 16 : sp & 0xFFFFu)));
                const float z = static_cast<float>(((zw >> (4 * gq)) & 0xFu) + gzoff);
                float p = fmaf(-(1024.f + z), slo[i], dlo[nt][i]);
                p = fmaf(0.0625f, dhi[nt][i], p);
                p = fmaf(-(64.f + z), shi[i], p);
                acc[i] = fmaf(s, p, acc[i]);
            }
            accs[nt * 32] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        }
        clear_partials();
    };
    // next group of the run: a new slot of the batch, or, past the last slot,
    // flush the batch and start the next one
    auto next_group = [&]() {
        if (++slot == S) {
            flush();
            gb0 += S;
            slot = 0;
            load_batch();
        }
        set_xoff();
        left = bpg;
    };
    auto begin_segment = [&](int t, int c) {
        seg_t = t;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) accs[nt * 32] = make_float4(0.f, 0.f, 0.f, 0.f);
        clear_partials();
        const int blk = 2 * c;
        gb0 = blk / bpg;
        left = bpg - (blk - gb0 * bpg);
        slot = 0;
        set_xoff();
        load_batch();
    };
    // Segment done: flush, sum the slots of each row, then write out or hand
    // the partial to the tile's last worker.
    auto end_segment = [&]() {
        flush();
        float v[NTW][4];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
            const float4 a4 = accs[nt * 32];
            v[nt][0] = a4.x;
            v[nt][1] = a4.y;
            v[nt][2] = a4.z;
            v[nt][3] = a4.w;
        }
        if (MP < 8) {
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (MP <= 2) v[nt][i] += __shfl_xor_sync(0xFFFFFFFFu, v[nt][i], 1);
                    v[nt][i] += __shfl_xor_sync(0xFFFFFFFFu, v[nt][i], 2);
                }
        }
        // element (nt, i): row 2 tq + (i & 1), column 16 nt + gq + 8 (i >> 1) of the tile
        const long long tu0 = static_cast<long long>(seg_t) * KC;
        const int wf = owner(tu0, a.U, a.workers), wl = owner(tu0 + KC - 1, a.U, a.workers);
        const int n0 = kCols * seg_t;
        auto store = [&](int row, int col, float val) {
            if (h.out_bf16 == kOutF32) reinterpret_cast<float *>(a.out)[static_cast<size_t>(row) * N + n0 + col] = val;
            else
                a.out[static_cast<size_t>(row) * N + n0 + col] =
                    out_one(val, h.rowscale ? h.rowscale[row] : 1.f, h.bias, n0 + col, h.out_bf16);
        };
        if (wf == wl) {
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = 2 * tq + (i & 1);
                    if (row < MP && row < a.M) store(row, 16 * nt + gq + 8 * (i >> 1), v[nt][i]);
                }
            return;
        }
        const int seg = wid - wf, nseg = wl - wf + 1;
        float *tile_ws = a.ws + static_cast<size_t>(seg_t) * a.smax * kPart;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = 2 * tq + (i & 1);
                if (row < MP && row < a.M)
                    __stcg(tile_ws + seg * kPart + row * kCols + 16 * nt + gq + 8 * (i >> 1), v[nt][i]);
            }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(a.tickets + seg_t, 1) == nseg - 1;
        last = __shfl_sync(0xFFFFFFFFu, last, 0);
        if (!last) return;
        __threadfence();
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = 2 * tq + (i & 1);
                const int col = 16 * nt + gq + 8 * (i >> 1);
                if (row < MP && row < a.M) {
                    float sum = 0.f;
                    for (int sg = 0; sg < nseg; ++sg) sum += __ldcg(tile_ws + sg * kPart + row * kCols + col);
                    store(row, col, sum);
                }
            }
        if (lane == 0) a.tickets[seg_t] = 0;          // ready for the next call on this stream
    };

    // ---- main loop over this worker's units (kept compact: the loop body
    //      stays small enough for the instruction cache)
    int t = t_first, c = static_cast<int>(u0 - static_cast<long long>(t_first) * KC);
    begin_segment(t, c);
    cp_async_wait<0>();
    int s = 0;                                        // ring slot of unit i
#pragma unroll 1
    for (int i = 0; i < n_units; ++i) {
        cp_async_wait<kDepth - 2>();
        __syncwarp();                                 // every lane's x copy of unit i has landed
        const unsigned char *slot_base = ring + s * C::kSlot;
        uint4 w[NTW];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) w[nt] = *reinterpret_cast<const uint4 *>(slot_base + lane * 16 + nt * 512);
        // refill the slot consumed by unit i - 1 with unit i + kDepth - 1
        if (i + kDepth - 1 < n_units) {
            const int fs = s == 0 ? kDepth - 1 : s - 1;
            copy_w(fs);
            copy_x(fs, fc);
            advance();
        }
        cp_async_commit();
        // one 32-row block: the sums of x for the zero point, then per n16
        // tile the A fragments straight from the code pairs (rows (0,1),
        // (4,5) as 1024 + q, rows (2,3), (6,7) as 1024 + 16 q) into the MMAs
        auto block = [&](int hh) {
            const uint4 xb = *reinterpret_cast<const uint4 *>((xuse ? slot_base + x_real : xzero) + hh * 64);
            mma_f32(slo, ones, xb.x, xb.z);
            mma_f32(shi, ones, xb.y, xb.w);
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) {
                const uint32_t lo = hh ? w[nt].z : w[nt].x;     // column 16 nt + gq
                const uint32_t hi = hh ? w[nt].w : w[nt].y;     // column 16 nt + gq + 8
                const uint32_t lo8 = lo >> 8, hi8 = hi >> 8;
                const uint32_t alo[4] = {lop3_and_or(lo, 0x000F000Fu, 0x64006400u),
                                         lop3_and_or(hi, 0x000F000Fu, 0x64006400u),
                                         lop3_and_or(lo8, 0x000F000Fu, 0x64006400u),
                                         lop3_and_or(hi8, 0x000F000Fu, 0x64006400u)};
                const uint32_t ahi[4] = {lop3_and_or(lo, 0x00F000F0u, 0x64006400u),
                                         lop3_and_or(hi, 0x00F000F0u, 0x64006400u),
                                         lop3_and_or(lo8, 0x00F000F0u, 0x64006400u),
                                         lop3_and_or(hi8, 0x00F000F0u, 0x64006400u)};
                mma_f32(dlo[nt], alo, xb.x, xb.z);
                mma_f32(dhi[nt], ahi, xb.y, xb.w);
            }
        };
        // group bookkeeping once per unit (a group is a whole number of
        // 32-row blocks; with an even number, groups change only between units)
        if (left == 0) next_group();
        if (left >= 2) {
            left -= 2;
            block(0);
            block(1);
        } else {                                      // the group ends after the first block
            block(0);
            next_group();
            --left;
            block(1);
        }
        if (++c == KC || i == n_units - 1) {
            end_segment();
            if (c == KC && i + 1 < n_units) {
                c = 0;
                ++t;
                begin_segment(t, 0);
            }
        }
        if (++s == kDepth) s = 0;
    }
    cp_async_wait<0>();
}

}  // namespace

DecodeSkPlan plan_decode_sk(int M, int K, int N, int sms) {
    DecodeSkPlan p{};
    if (M < 1 || M > 8 || K % 64 || N % 64) return p;
    // one row takes the two-row layout (B columns 2 s, 2 s + 1 for slot s, the
    // second empty): each lane's accumulators then belong to one slot
    p.mp = M <= 2 ? 2 : (M <= 4 ? 4 : 8);
    p.ntw = Q4_SK_NTW;
    p.T = N / (16 * p.ntw);
    p.KC = K / 64;
    p.U = static_cast<long long>(p.T) * p.KC;
    // every resident warp a worker, but at least kMinUnits units each (a
    // segment's partial write and ticket cost about one unit)
    const long long want = static_cast<long long>(sms) * kCtasPerSm * kWarps;
    p.workers = static_cast<int>(std::max<long long>(1, std::min<long long>(want, p.U / kMinUnits)));
    p.ctas = (p.workers + kWarps - 1) / kWarps;
    // segments of a tile: the owners of its first and last unit and all
    // between (workers take [floor(w U / W), floor((w + 1) U / W)))
    auto own = [&](long long u) { return static_cast<int>(((u + 1) * p.workers - 1) / p.U); };
    p.smax = 1;
    for (int t = 0; t < p.T; ++t) {
        const long long a0 = static_cast<long long>(t) * p.KC;
        p.smax = std::max(p.smax, own(a0 + p.KC - 1) - own(a0) + 1);
    }
    p.ws_floats = static_cast<size_t>(p.T) * p.smax * 8 * 16 * p.ntw;
    p.n_tickets = p.T;
    p.ok = 1;
    return p;
}

template <int MP, int NTW>
static cudaError_t launch_sk_mp(const HandleView &h, const DecodeSkPlan &p, const SkArgs &args, cudaStream_t s) {
    using C = SkCfg<MP, NTW>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = dyn_smem_optin(reinterpret_cast<const void *>(decode_sk_kernel<MP, NTW>), dev, C::kSmem, nullptr);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (pdl_enabled()) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, decode_sk_kernel<MP, NTW>, h, args);
}

cudaError_t launch_decode_sk(const HandleView &h, const DecodeSkPlan &p, float *ws, int *tickets, const uint16_t *x,
                             int M, uint16_t *out, cudaStream_t s) {
    if (!p.ok || M < 1 || M > 8 || p.ntw != Q4_SK_NTW) return cudaErrorInvalidValue;
    const SkArgs args{x, out, ws, tickets, M, p.T, p.KC, p.U, p.workers, p.smax};
    switch (p.mp) {
        case 2: return launch_sk_mp<2, Q4_SK_NTW>(h, p, args, s);
        case 4: return launch_sk_mp<4, Q4_SK_NTW>(h, p, args, s);
        default: return launch_sk_mp<8, Q4_SK_NTW>(h, p, args, s);
    }
}

}  // namespace q4
