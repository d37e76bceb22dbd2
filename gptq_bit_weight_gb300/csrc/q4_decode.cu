// Decode (small-M) fused GPTQ W4A16 matmul.
//
// "GPTQ's 'Exllama Kernel Not Installed' Warning", "What the fallback
// actually does": the fused kernel reads packed 4-bit weights from memory,
// unpacks and dequantizes them in registers and multiplies against fp16
// activations without ever writing a dequantized matrix; weight-bound
// decoding is limited by memory bandwidth.
// "Inference Backends", "Numeric epilogues and input gradients": fp32
// accumulation, fp32 split reductions, bias added to the fp32 sum before the
// one final cast, and no atomic partial-output reduction.
//
// Work split.  A CTA (8 warps) owns 32 output columns (two 16-column tiles),
// up to 8*MT rows of x, and one K slice.  Its warps split the slice into
// contiguous runs of 64-row chunks; for each chunk a lane needs one 16-byte
// vector per column tile.  Two ways to keep those in flight:
//   shared ring (SR, M <= 4): each warp owns a ring of kDepth chunk slots in
//     shared memory, filled by asynchronous copies (one commit group per
//     chunk); a lane reads back exactly the vectors it copied, so no barrier
//     is needed.  The first kDepth - 1 chunks are requested before the
//     preceding grid has finished (they are handle constants), and x comes in
//     with plain loads so that waiting for x does not wait for the weights.
//   register ring (larger M, whose x slice takes the shared memory): each
//     warp keeps kRegDepth chunks of loads in flight in registers.
// Groups are tracked with counters along the warp's run (no division in
// the loop).
//
// Arithmetic.  Each packed word gives, with one LOP3 and one HFMA2 per pair,
// the exact integers (q - z - 1) of eight consecutive rows of one column as
// four half2 registers.  Those are the A operand of m16n8k16 tensor-core MMAs
// (rows = output columns n, k = weight rows) against x as the B operand
// (columns = rows of x), accumulating in fp32.  The K index inside a 32-row
// block is permuted identically for A and B (lane tq owns rows 8tq..8tq+7),
// which lets both operands come from single 16-byte loads; a sum does not
// depend on the order of its terms beyond rounding.  The scale is factored
// out of each group: a fresh fp32 partial per group, then acc += s * partial.
// The raw-pair variant (RAW) enters the code pairs as raw 1024 + q / 1024 +
// 16 q, removes the zero points per group from MMA-accumulated sums of x, and
// puts successive groups in the spare B columns of its MMAs (group slots), so
// that its per-group step runs once per batch of 8 / MP groups.
//
// Reduction.  Warps of a CTA are summed in a fixed order through shared
// memory.  With more than one K slice, each CTA writes its fp32 partial tile
// to the workspace, and the last CTA of a column tile to arrive (an atomic
// ticket; nobody waits) adds the slices in slice order, adds bias and rounds
// once to fp16.  The result is deterministic.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "q4_internal.cuh"

namespace q4 {

// Per (kernel, device, size): set a kernel's dynamic shared-memory limit.
// The attribute belongs to the device that is current, so every device the
// library runs on gets its own set-up; each is done once.  bytes < 0: the
// largest the device allows beside the kernel's static shared memory.  The
// limit set is returned in *set.
cudaError_t dyn_smem_optin(const void *fn, int dev, int bytes, int *set) {
    struct Entry {
        const void *fn;
        int dev;
        int want;
        int bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry &en : done)
        if (en.fn == fn && en.dev == dev && en.want == bytes) {
            if (set) *set = en.bytes;
            return cudaSuccess;
        }
    int val = bytes;
    cudaError_t e = cudaSuccess;
    if (bytes < 0) {
        int optin = 0;
        cudaFuncAttributes fa{};
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, fn);
        val = optin - static_cast<int>(fa.sharedSizeBytes);
    }
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, val);
    if (e != cudaSuccess) return e;
    done.push_back(Entry{fn, dev, bytes, val});
    if (set) *set = val;
    return cudaSuccess;
}

namespace {

// Tuning parameters (compile-time; the defaults are the measured choice).
#ifndef Q4_DECODE_WARPS
#define Q4_DECODE_WARPS 8
#endif
#ifndef Q4_DECODE_NTW
#define Q4_DECODE_NTW 2
#endif
#ifndef Q4_DECODE_DEPTH
#define Q4_DECODE_DEPTH 3
#endif
constexpr int kWarps = Q4_DECODE_WARPS;
constexpr int kThreads = 32 * kWarps;
constexpr int kNTW = Q4_DECODE_NTW;             // 16-column tiles per CTA
constexpr int kNB = 16 * kNTW;      // columns per CTA
constexpr int kDepth = Q4_DECODE_DEPTH;         // shared ring: slots per warp (kDepth - 1 chunks in flight)
// A shared-ring slot: the chunk's packed words (16 bytes per lane and tile)
// and its x fragments (8 rows x 64 fp16, 128 bytes per row).
constexpr int kSlotBytes = kNTW * 512 + 8 * 128;
constexpr int kRingWarpBytes = kDepth * kSlotBytes;
constexpr int kRegDepth = 4;                    // register ring: chunks in flight per warp
#ifndef Q4_DECODE_XSTAGE_BYTES
#define Q4_DECODE_XSTAGE_BYTES 16384
#endif
constexpr long long kXStageBytes = Q4_DECODE_XSTAGE_BYTES;   // largest staged x slice with the shared ring
constexpr int kMaxCluster = 8;      // portable thread-block cluster size
// Shared words staged per group: kNTW*8 scale pairs, then kNTW*2 zero words,
// padded to a multiple of 4 so every group's copies start 16-byte aligned.
constexpr int kGszStride = ((kNTW * 10 + 3) / 4) * 4;

struct DecodeArgs {
    const uint16_t *x;
    uint16_t *out;
    float *ws;
    int *tickets;
    int M;
    int splits;
    int slice_chunks;
    int xrows;          // rows of x staged per CTA: min(8*MT, M)
    int cluster;        // slices reduce through distributed shared memory
};

__host__ __device__ inline int x_row_stride(int slice_chunks) { return slice_chunks * 64 + 32; }

// Bytes per warp of the first shared region: the weight ring (shared ring)
// or the warp partials alone (register ring); the ring holds the partials
// at the end.
__host__ __device__ constexpr int warp_region_bytes(int mt, bool sr) {
    return sr ? kRingWarpBytes : kNTW * mt * 512;
}
// Shared memory: the warps' regions, the staged x slice (none when the
// shared ring carries x per chunk), the slice's scale pairs and zero words.
__host__ __device__ inline size_t smem_bytes_for(int mt, bool sr, bool xr, int xrows, int slice_chunks, int max_groups) {
    return static_cast<size_t>(kWarps) * warp_region_bytes(mt, sr) +
           (xr ? 0 : static_cast<size_t>(xrows) * x_row_stride(slice_chunks) * 2) +
           static_cast<size_t>(max_groups) * kGszStride * 4;
}

__host__ __device__ inline int max_groups_in_slice(int slice_chunks, int geff) {
    return (slice_chunks * 64 + geff - 1) / geff + 1;
}

// Resident-CTA target per SM for the register budget: 24, 16 and 8 warps
// (16 for the raw-pair arithmetic at MT = 1, whose partial sums take more
// registers).
constexpr int min_warps(int mt, bool raw) { return mt == 1 ? (raw ? 16 : 24) : (mt == 2 ? 16 : 8); }
constexpr int min_blocks(int mt, bool raw) { return min_warps(mt, raw) / kWarps > 0 ? min_warps(mt, raw) / kWarps : 1; }

// RAW: code pairs enter the MMAs as raw 1024 + q / 1024 + 16 q (one LOP3 per
// pair) and the zero point is removed per group from MMA-accumulated sums of
// x; otherwise each pair is turned into the exact fp16 (q - z - 1) first (one
// LOP3 and one HFMA2).  Same result up to fp32 rounding.
template <int MT, bool RAW, bool SR, bool XR>
__global__ void __launch_bounds__(kThreads, min_blocks(MT, RAW)) decode_kernel(HandleView h, DecodeArgs a) {
    static_assert(!XR || SR, "x rides in the shared ring only");
    static_assert(!RAW || MT == 1, "raw pairs: one m tile");
    constexpr int kRegion = warp_region_bytes(MT, SR);
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    const int K = h.K, N = h.N, KC = K >> 6, NT16 = N >> 4;
    const int nt0 = blockIdx.x * kNTW;
    const int split = blockIdx.y;
    const int m0 = blockIdx.z * (8 * MT);
    const int mrows = min(8 * MT, a.M - m0);
    const int c_beg = split * a.slice_chunks;
    const int c_end = min(KC, c_beg + a.slice_chunks);
    const int nch = c_end - c_beg;
    const int XS = x_row_stride(a.slice_chunks);
    const int geff = h.geff;

    static_assert(kDepth >= 2 && kRegion >= kNTW * MT * 128 * 4, "a warp's region holds its partials at the end");
    static_assert(!SR || MT == 1, "the shared ring serves one m tile");
    unsigned char *wring = smem;
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem + kWarps * kRegion);
    uint32_t *gsz = reinterpret_cast<uint32_t *>(smem + kWarps * kRegion + (XR ? 0 : static_cast<size_t>(a.xrows) * XS * 2));

    // Let the next kernel in the stream start its own prologue as soon as
    // every CTA of this grid is resident (programmatic dependent launch).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // This warp's run of 64-row chunks within the CTA's slice.
    const int wc_beg = c_beg + (nch * warp) / kWarps;
    const int wn = c_beg + (nch * (warp + 1)) / kWarps - wc_beg;
    auto chunk_of = [&](int c) { return wc_beg + c; };
    const int g_base = (c_beg * 64) / geff;

    // ---- the slice's scale pairs / zero words (constant), then the first
    //      chunks of this warp's packed weights (handle-owned constant data,
    //      so both go out before the preceding grid has finished), then x
    //      once it has.
    {
        const int g_beg = (c_beg * 64) / geff;
        const int g_end = (c_end * 64 - 1) / geff + 1;
        // per group: kNTW*8 scale-pair words, then kNTW*2 zero words
        for (int gl = threadIdx.x; gl < g_end - g_beg; gl += kThreads) {
            const size_t gr = static_cast<size_t>(g_beg + gl);
            uint32_t *dst = gsz + gl * kGszStride;      // 16-byte aligned (stride % 4 == 0)
            const uint32_t *s2src = h.s2 + (gr * NT16 + nt0) * 8;
#pragma unroll
            for (int v = 0; v < kNTW * 2; ++v) cp_async_16(dst + 4 * v, s2src + 4 * v);
            // zero words: 8 * kNTW bytes at a source offset that is a multiple
            // of 8 * kNTW bytes; 16-byte copies while they fit, then one of 8.
            const uint32_t *zsrc = h.zeros + gr * (N >> 3) + nt0 * 2;
#pragma unroll
            for (int v = 0; v < kNTW / 2; ++v) cp_async_16(dst + kNTW * 8 + 4 * v, zsrc + 4 * v);
            if (kNTW & 1) cp_async_8(dst + kNTW * 8 + 4 * (kNTW / 2), zsrc + 4 * (kNTW / 2));
        }
        cp_async_commit();
    }
    // Shared ring: slot s of this warp holds at  s * kSlotBytes
    //   + nt * 512 + lane * 16                      the lane's packed words of tile nt
    //   + kNTW * 512 + gq * 128 + hh * 64 + tq * 16 its x fragment of row gq, half hh
    //                                               (XR: x carried per chunk)
    // Every lane copies exactly the pieces it later reads, so the ring needs
    // no barrier; each chunk is one commit group.  Without XR the CTA stages
    // its whole x slice once instead: better when that slice is short, since
    // with XR every CTA asks for the same x line of a chunk at about the same
    // time.
    unsigned char *myring = wring + warp * kRingWarpBytes;
    unsigned char *myw = myring + lane * 16;
    unsigned char *myx = myring + kNTW * 512 + gq * 128 + tq * 16;
    const bool xrow = gq < mrows;                       // this lane's x row exists
    const uint16_t *xsrc = a.x + static_cast<size_t>(m0 + (xrow ? gq : 0)) * K + 8 * tq;
    auto copy_x = [&](int slot, int chunk) {
        if (xrow) {
            cp_async_16(myx + slot * kSlotBytes, xsrc + chunk * 64);
            cp_async_16(myx + slot * kSlotBytes + 64, xsrc + chunk * 64 + 32);
        }
    };
    const uint4 *wsrc[kNTW];
#pragma unroll
    for (int nt = 0; nt < kNTW; ++nt) wsrc[nt] = h.wp + static_cast<size_t>(nt0 + nt) * KC * 32 + lane;
    uint4 buf[SR ? 1 : kRegDepth][kNTW];               // register ring
    if (SR) {
#pragma unroll
        for (int i = 0; i < kDepth - 1; ++i) {
            if (i < wn)
#pragma unroll
                for (int nt = 0; nt < kNTW; ++nt)
                    cp_async_16(myw + i * kSlotBytes + nt * 512, wsrc[nt] + static_cast<size_t>(chunk_of(i)) * 32);
            cp_async_commit();
        }
    } else {
#pragma unroll
        for (int i = 0; i < kRegDepth; ++i)
            if (i < wn)
#pragma unroll
                for (int nt = 0; nt < kNTW; ++nt)
                    buf[SR ? 0 : i][nt] = ldg_stream(wsrc[nt] + static_cast<size_t>(chunk_of(i)) * 32);
    }
    {
        // x, the workspace, the tickets and out may belong to the preceding
        // grid: wait for it (a no-op without programmatic dependent launch).
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int vpr = nch * 8;                        // 16-byte vectors per row
        if (XR) {
            // x of the first kDepth - 1 chunks: one more group
#pragma unroll
            for (int i = 0; i < kDepth - 1; ++i)
                if (i < wn) copy_x(i, chunk_of(i));
            cp_async_commit();
            cp_async_wait<kDepth>();                    // the scale/zero copies: the oldest group
        } else if (SR) {
            // plain L2 loads, eight per thread in flight, so that waiting for
            // x does not wait for the weight copies
            const int total = mrows * vpr;
            for (int v0 = threadIdx.x; v0 < total; v0 += 8 * kThreads) {
                uint4 xv8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int v = v0 + u * kThreads;
                    if (v < total) {
                        const int r = v / vpr, cv = v - r * vpr;
                        xv8[u] = __ldcg(reinterpret_cast<const uint4 *>(a.x + static_cast<size_t>(m0 + r) * K + c_beg * 64) + cv);
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int v = v0 + u * kThreads;
                    if (v < total) {
                        const int r = v / vpr, cv = v - r * vpr;
                        *reinterpret_cast<uint4 *>(xs + r * XS + cv * 8) = xv8[u];
                    }
                }
            }
            cp_async_wait<kDepth - 1>();                // the scale/zero copies: the oldest group
        } else {
            for (int r = 0; r < mrows; ++r) {
                const uint16_t *src = a.x + static_cast<size_t>(m0 + r) * K + c_beg * 64;
                for (int c = threadIdx.x; c < vpr; c += kThreads) cp_async_16(xs + r * XS + c * 8, src + c * 8);
            }
            cp_async_commit();
            cp_async_wait<0>();
        }
    }
    __syncthreads();

    float acc[kNTW][MT][4];
#pragma unroll
    for (int nt = 0; nt < kNTW; ++nt)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][mt][i] = 0.f;

    if (wn > 0) {
        // per group: products of x with the raw pairs (dlo: 1024 + q rows,
        // dhi: 1024 + 16 q rows) and the sums of x that met them (slo, shi);
        // exact arithmetic: dlo alone holds sum x (q - z - 1)
        float dlo[kNTW][MT][4], dhi[kNTW][MT][4], slo[MT][4], shi[MT][4];
        auto clear_partials = [&]() {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    slo[mt][i] = 0.f;
                    shi[mt][i] = 0.f;
#pragma unroll
                    for (int nt = 0; nt < kNTW; ++nt) dlo[nt][mt][i] = dhi[nt][mt][i] = 0.f;
                }
        };
        clear_partials();

        // The current group's scales, and per pair kind either the unpack_qz
        // constants (exact pairs) or -(1024 + z), -(64 + z) (raw pairs), z
        // the effective zero point of columns gq, gq + 8.
        float sc[kNTW][2], czl[kNTW][2], czh[kNTW][2];
        uint32_t nzlo[kNTW][2], nzhi[kNTW][2];
        // neg_zlo / neg_zhi of (stored zero + zero offset - 1) = stored zero
        // times the pair stride plus these (32-bit wrap-around included); the
        // groups below h.zsplit take zero offset 0
        const uint32_t lo_base1 = neg_zlo(static_cast<uint32_t>(h.zero_offset) - 1u);
        const uint32_t hi_base1 = neg_zhi(static_cast<uint32_t>(h.zero_offset) - 1u);
        const uint32_t lo_base0 = neg_zlo(0xFFFFFFFFu), hi_base0 = neg_zhi(0xFFFFFFFFu);
        // Group slots (raw pairs).  An m16n8k16 MMA has 8 B columns and the
        // rows of x fill MP of them (MP = 2 for one or two rows, else M rounded
        // up to a power of two); the others carry the next groups: B column c
        // holds x row c % MP while the run is in group c / MP of the current
        // batch of S = 8 / MP groups, zeros otherwise.  Each group then
        // accumulates in its own columns and the per-group step (zero point,
        // scale) runs once per batch; a lane's two accumulator columns belong
        // to slot 2 tq / MP, whose group's constants it loads.  The slots of
        // each row are summed across the lanes at the end.
        const int MP = mrows <= 2 ? 2 : (mrows <= 4 ? 4 : 8);
        const int S = 8 / MP;
        const int lslot = (2 * tq) / MP;
        const int ng_slice = (c_end * 64 - 1) / geff + 1 - g_base;   // groups staged for the slice
        int slot = 0;
        auto load_group = [&](int gl) {
            if (RAW) gl = min(gl + lslot, ng_slice - 1);   // past the run's last group: zero sums
            const uint32_t *base = gsz + gl * kGszStride;
            const bool z0grp = g_base + gl < h.zsplit;
            const uint32_t zoff = z0grp ? 0u : static_cast<uint32_t>(h.zero_offset);
            const uint32_t lo_base = z0grp ? lo_base0 : lo_base1, hi_base = z0grp ? hi_base0 : hi_base1;
#pragma unroll
            for (int nt = 0; nt < kNTW; ++nt) {
                const uint32_t sp = base[nt * 8 + gq];
                const uint32_t zw0 = base[kNTW * 8 + nt * 2], zw1 = base[kNTW * 8 + nt * 2 + 1];
                sc[nt][0] = __half2float(__ushort_as_half(static_cast<unsigned short>(sp & 0xFFFFu)));
                sc[nt][1] = __half2float(__ushort_as_half(static_cast<unsigned short>(sp >> 16)));
                const uint32_t z0s = (zw0 >> (4 * gq)) & 0xFu, z1s = (zw1 >> (4 * gq)) & 0xFu;   // stored
                const uint32_t z0 = z0s + zoff, z1 = z1s + zoff;
                if (RAW) {
                    czl[nt][0] = -(1024.f + static_cast<float>(z0));
                    czl[nt][1] = -(1024.f + static_cast<float>(z1));
                    czh[nt][0] = -(64.f + static_cast<float>(z0));
                    czh[nt][1] = -(64.f + static_cast<float>(z1));
                } else {
                    // unpack_qz constants of (effective zero) - 1, one multiply-add each
                    nzlo[nt][0] = z0s * 0x00010001u + lo_base;
                    nzhi[nt][0] = z0s * 0x00100010u + hi_base;
                    nzlo[nt][1] = z1s * 0x00010001u + lo_base;
                    nzhi[nt][1] = z1s * 0x00100010u + hi_base;
                }
            }
        };
        // sum_k x (q - z - 1) = dlo - (1025 + z) slo + (dhi - (1040 + 16 z) shi) / 16
        auto flush = [&]() {
#pragma unroll
            for (int nt = 0; nt < kNTW; ++nt)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int c = i >> 1;
                        float p = dlo[nt][mt][i];
                        if (RAW) {
                            p = fmaf(czl[nt][c], slo[mt][i], p);
                            p = fmaf(0.0625f, dhi[nt][mt][i], p);
                            p = fmaf(czh[nt][c], shi[mt][i], p);
                        }
                        acc[nt][mt][i] = fmaf(sc[nt][c], p, acc[nt][mt][i]);
                    }
            clear_partials();
        };
        constexpr uint32_t kOnes = 0x3C003C00u;
        const uint32_t ones[4] = {kOnes, kOnes, kOnes, kOnes};

        // Group of the warp's first 32-row block and the blocks left in it;
        // the run's blocks are consecutive, so counters track the rest.
        const int bpg = geff >> 5;
        const int blk0 = 2 * wc_beg;
        int gl = blk0 / bpg - g_base;
        int left = bpg - (blk0 - (gl + g_base) * bpg);
        load_group(gl);

        // This lane's x row in each m tile and its 16-byte piece of the first
        // 32-row block of the run.
        const uint16_t *xp[MT];
        bool xv[MT];
        const int rraw = gq & (MP - 1);                // raw pairs: the lane's x row in its slot
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int r = mt * 8 + (RAW ? rraw : gq);
            xv[mt] = r < mrows && (!RAW || gq / MP == slot);
            xp[mt] = xs + (r < mrows ? r : 0) * XS + 2 * (wc_beg - c_beg) * 32 + 8 * tq;
        }
        // shared ring: offset from the lane's own x row to the row it reads
        const int xring_off = RAW ? (rraw - gq) * 128 : 0;
        bool xsel = RAW ? xv[0] : xrow;

        const unsigned char *xcur = myx;               // shared ring: x fragments of the current chunk
        auto run_chunk = [&](int c, const uint4 (&w)[kNTW]) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                if (left == 0) {
                    if (RAW) {
                        if (++slot == S) {
                            flush();
                            gl += S;
                            slot = 0;
                            load_group(gl);
                        }
                        xsel = gq / MP == slot && rraw < mrows;
                        xv[0] = xsel;
                    } else {
                        flush();
                        load_group(++gl);
                    }
                    left = bpg;
                }
                --left;
                uint4 xb[MT];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    if (XR)
                        xb[mt] = xsel ? *reinterpret_cast<const uint4 *>(xcur + xring_off + hh * 64)
                                      : make_uint4(0u, 0u, 0u, 0u);
                    else
                        xb[mt] = xv[mt] ? *reinterpret_cast<const uint4 *>(xp[mt] + (2 * c + hh) * 32)
                                        : make_uint4(0u, 0u, 0u, 0u);
                }
                if (RAW) {
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        mma_16816(slo[mt], ones, xb[mt].x, xb[mt].z);
                        mma_16816(shi[mt], ones, xb[mt].y, xb[mt].w);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < kNTW; ++nt) {
                    const uint32_t lo = hh ? w[nt].z : w[nt].x;    // column 16nt + gq
                    const uint32_t hi = hh ? w[nt].w : w[nt].y;    // column 16nt + gq + 8
                    uint32_t al[4], ah[4];
                    if (RAW) {
                        unpack_raw(lo, al);
                        unpack_raw(hi, ah);
                        const uint32_t alo[4] = {al[0], ah[0], al[2], ah[2]};
                        const uint32_t ahi[4] = {al[1], ah[1], al[3], ah[3]};
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            mma_16816(dlo[nt][mt], alo, xb[mt].x, xb[mt].z);
                            mma_16816(dhi[nt][mt], ahi, xb[mt].y, xb[mt].w);
                        }
                    } else {
                        unpack_qz(lo, nzlo[nt][0], nzhi[nt][0], al);
                        unpack_qz(hi, nzlo[nt][1], nzhi[nt][1], ah);
                        const uint32_t A0[4] = {al[0], ah[0], al[1], ah[1]};
                        const uint32_t A1[4] = {al[2], ah[2], al[3], ah[3]};
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            mma_16816(dlo[nt][mt], A0, xb[mt].x, xb[mt].y);
                            mma_16816(dlo[nt][mt], A1, xb[mt].z, xb[mt].w);
                        }
                    }
                }
            }
        };
        if (SR) {
            // sources of the next chunk to request, c + kDepth - 1
            const uint4 *wnext[kNTW];
#pragma unroll
            for (int nt = 0; nt < kNTW; ++nt) wnext[nt] = wsrc[nt] + static_cast<size_t>(chunk_of(kDepth - 1)) * 32;
            const uint16_t *xnext = xsrc + chunk_of(kDepth - 1) * 64;
            for (int base = 0; base < wn; base += kDepth) {
#pragma unroll
                for (int i = 0; i < kDepth; ++i) {       // chunk c sits in slot i = c % kDepth
                    const int c = base + i;
                    if (c < wn) {
                        // chunk c has landed: the first waits for the prologue's
                        // x group as well (the most recent one)
                        if (XR && c == 0) cp_async_wait<0>();
                        else cp_async_wait<kDepth - 2>();
                        uint4 w[kNTW];
#pragma unroll
                        for (int nt = 0; nt < kNTW; ++nt)
                            w[nt] = *reinterpret_cast<const uint4 *>(myw + i * kSlotBytes + nt * 512);
                        if (XR) xcur = myx + i * kSlotBytes;
                        // refill the slot of chunk c - 1 (consumed) with chunk c + kDepth - 1
                        const int fs = (i + kDepth - 1) % kDepth;
                        if (c + kDepth - 1 < wn) {
#pragma unroll
                            for (int nt = 0; nt < kNTW; ++nt) {
                                cp_async_16(myw + fs * kSlotBytes + nt * 512, wnext[nt]);
                                wnext[nt] += 32;
                            }
                            if (XR && xrow) {
                                cp_async_16(myx + fs * kSlotBytes, xnext);
                                cp_async_16(myx + fs * kSlotBytes + 64, xnext + 32);
                            }
                            xnext += 64;
                        }
                        cp_async_commit();
                        run_chunk(c, w);
                    }
                }
            }
        } else {
            for (int base = 0; base < wn; base += kRegDepth) {
#pragma unroll
                for (int i = 0; i < kRegDepth; ++i) {
                    const int c = base + i;
                    if (c < wn) {
                        run_chunk(c, buf[SR ? 0 : i]);
                        if (c + kRegDepth < wn)
#pragma unroll
                            for (int nt = 0; nt < kNTW; ++nt)
                                buf[SR ? 0 : i][nt] = ldg_stream(wsrc[nt] + static_cast<size_t>(chunk_of(c + kRegDepth)) * 32);
                    }
                }
            }
        }
        flush();
    }
    if (RAW && mrows <= 4) {
        // raw pairs: sum each row's group slots across the lanes (xor 1 and 2
        // with two slot columns per row set of four lanes, xor 2 with four rows)
#pragma unroll
        for (int nt = 0; nt < kNTW; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float v = acc[nt][0][i];
                if (mrows <= 2) v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
                acc[nt][0][i] = v;
            }
    }

    // ---- fixed-order reduction over the CTA's warps; warp w's partials go to
    //      its own (drained) ring, so no warp waits before writing them
    constexpr int E = kNTW * MT * 128;                 // partial elements per CTA
    constexpr int RW = kRegion / 4;                     // floats between two warps' partials
    float *red = reinterpret_cast<float *>(wring);
    cp_async_wait<0>();
#pragma unroll
    for (int nt = 0; nt < kNTW; ++nt)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            *reinterpret_cast<float4 *>(red + warp * RW + (nt * MT + mt) * 128 + lane * 4) =
                make_float4(acc[nt][mt][0], acc[nt][mt][1], acc[nt][mt][2], acc[nt][mt][3]);
    __syncthreads();

    auto element_mn = [&](int e, int &m, int &n) {
        const int ntm = e >> 7, l = (e >> 2) & 31, i = e & 3;
        const int nt = ntm / MT, mt = ntm - nt * MT;
        n = 16 * (nt0 + nt) + (l >> 2) + 8 * (i >> 1);
        m = m0 + mt * 8 + 2 * (l & 3) + (i & 1);
    };
    auto store_out = [&](int e, float v) {
        int m, n;
        element_mn(e, m, n);
        if (m < a.M) {
            if (h.out_bf16 == kOutF32) reinterpret_cast<float *>(a.out)[static_cast<size_t>(m) * N + n] = v;
            else a.out[static_cast<size_t>(m) * N + n] = out_one(v, h.rowscale ? h.rowscale[m] : 1.f, h.bias, n, h.out_bf16);
        }
    };

    // CTA partial: the warps' partials summed in warp order, kept in red[0, E)
    // (each thread reads its own elements of every warp before writing one).
    for (int e = threadIdx.x; e < E; e += kThreads) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += red[w * RW + e];
        if (a.splits == 1) store_out(e, v);
        else red[e] = v;
    }
    if (a.splits == 1) return;

    if (a.cluster) {
        // The K slices of a column tile form one thread-block cluster: sum the
        // slices' partials in slice order straight out of each other's shared
        // memory.  Cluster rank r finishes elements [r E / S, (r + 1) E / S).
        cluster_sync();
        const int S = a.splits;
        const int e0 = (split * E) / S, e1 = ((split + 1) * E) / S;
        for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += kThreads) {
            const uint32_t local = shared_addr(red + e);
            float v = 0.f;
            for (int r = 0; r < S; ++r) v += ld_dsmem_f32(local, r);
            store_out(e, v);
        }
        cluster_sync();                                 // partials stay alive until all are read
        return;
    }

    // Too many slices for one cluster: the partial goes to the workspace and
    // the last CTA of the column tile to arrive (an atomic ticket; nobody
    // waits) adds the slices in slice order.
    const int tile_id = blockIdx.z * gridDim.x + blockIdx.x;
    float *my_ws = a.ws + (static_cast<size_t>(tile_id) * a.splits + split) * E;
    for (int e = threadIdx.x; e < E; e += kThreads) __stcg(my_ws + e, red[e]);
    __threadfence();
    __syncthreads();
    __shared__ int s_last;
    if (threadIdx.x == 0) {
        const int prev = atomicAdd(a.tickets + tile_id, 1);
        s_last = (prev == a.splits - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const float *tile_ws = a.ws + static_cast<size_t>(tile_id) * a.splits * E;
    for (int e = threadIdx.x; e < E; e += kThreads) {
        float v = 0.f;
        for (int sl = 0; sl < a.splits; ++sl) v += __ldcg(tile_ws + static_cast<size_t>(sl) * E + e);
        store_out(e, v);
    }
    if (threadIdx.x == 0) a.tickets[tile_id] = 0;     // ready for the next call on this stream
}

template <int MT, bool RAW, bool SR, bool XR>
cudaError_t launch_mt(const HandleView &h, const DecodePlan &p, const DecodeWork &w, const uint16_t *x, int M,
                      uint16_t *out, cudaStream_t s) {
    const int xrows = M < 8 * MT ? M : 8 * MT;
    const size_t smem = smem_bytes_for(MT, SR, XR, xrows, p.slice_chunks, max_groups_in_slice(p.slice_chunks, h.geff));
    // Opt in, once per device, to the largest dynamic shared memory the
    // device allows next to the kernel's static shared memory.
    int max_dyn = 0;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess)
            e = dyn_smem_optin(reinterpret_cast<const void *>(decode_kernel<MT, RAW, SR, XR>), dev, -1, &max_dyn);
        if (e != cudaSuccess) return e;
    }
    if (smem > static_cast<size_t>(max_dyn)) return cudaErrorInvalidConfiguration;
    DecodeArgs a{x, out, w.ws, w.tickets, M, p.splits, p.slice_chunks, xrows, p.cluster};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.ctas_n, p.splits, p.zdim);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (p.cluster) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = static_cast<unsigned>(p.splits);
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl_enabled()) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, decode_kernel<MT, RAW, SR, XR>, h, a);
}

}  // namespace

// Programmatic dependent launch is on unless GPTQ_Q4_PDL=0.
bool pdl_enabled() {
    static const bool on = [] {
        const char *e = getenv("GPTQ_Q4_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

// Resident CTAs per SM for a variant: registers (the launch bounds) and
// shared memory, whichever is tighter.
int resident_ctas(int mt, bool raw, size_t smem) {
    const int by_regs = min_blocks(mt, raw);
    const size_t per_sm = 228 * 1024;                   // shared memory per SM
    const int by_smem = static_cast<int>(per_sm / (smem + 1024));
    return std::max(1, std::min(by_regs, by_smem));
}

// Split count.  Every slice fits the 64 KB x staging.  When the grid fits in
// one wave of resident CTAs, take the most splits that still fit (the most
// bytes in flight while the whole grid is one DRAM round trip deep); when it
// does not, fill whole waves as closely as possible (fewer splits on a tie).
static DecodePlan plan_decode_arith(int M, int K, int N, int geff, bool raw, bool sr) {
    DecodePlan p{};
    p.raw = raw ? 1 : 0;
    p.sr = sr ? 1 : 0;
    p.mt = M <= 8 ? 1 : (M <= 16 ? 2 : 4);
    p.zdim = (M + 8 * p.mt - 1) / (8 * p.mt);
    p.ctas_n = N / kNB;
    const int KC = K / 64;
    const int xrows = std::min(M, 8 * p.mt);
    // register ring: the x slice is staged, xrows * slice * 64 fp16 <= 64 KB.
    // Shared ring: x is staged when its slice takes at most kXStageBytes
    // (half that with at most one column tile per SM, where fewer CTAs share
    // each x line and carrying x per chunk measured faster), else carried
    // per chunk.
    const int max_slice = sr ? KC : std::min(KC, std::max(8, std::min(64, 512 / xrows)));
    // Also carried per chunk when staging it would cost a resident CTA per SM
    // (small groups stage more scale words: 8192x10240 g32 M = 1 measured
    // 22.2 -> 18.7 us at three CTAs per SM instead of two).
    auto xr_for = [&](int slice) {
        const long long xb = static_cast<long long>(xrows) * slice * 128;
        if (!sr) return false;
        if (xb > kXStageBytes || (p.ctas_n * p.zdim <= kSMs && xb > kXStageBytes / 2)) return true;
        const int mg = max_groups_in_slice(slice, geff);
        return resident_ctas(p.mt, raw, smem_bytes_for(p.mt, sr, false, xrows, slice, mg)) <
               resident_ctas(p.mt, raw, smem_bytes_for(p.mt, sr, true, xrows, slice, mg));
    };
    const int base = p.ctas_n * p.zdim;
    const int min_splits = (KC + max_slice - 1) / max_slice;
    const int max_splits = std::max(min_splits, KC / 16);   // at least two chunks per warp
    auto slots_for = [&](int sp) {
        const int slice = (KC + sp - 1) / sp;
        const size_t smem = smem_bytes_for(p.mt, sr, xr_for(slice), xrows, slice, max_groups_in_slice(slice, geff));
        return static_cast<long long>(kSMs) * resident_ctas(p.mt, raw, smem);
    };
    auto valid = [&](int sp) {
        const int slice = (KC + sp - 1) / sp;
        return (KC + slice - 1) / slice == sp;             // no empty slices
    };
    int best = min_splits;
    if (static_cast<long long>(base) * min_splits <= slots_for(min_splits)) {
        for (int sp = min_splits; sp <= max_splits; ++sp)
            if (valid(sp) && static_cast<long long>(base) * sp <= slots_for(sp)) best = sp;
    } else {
        double best_eff = -1.0;
        for (int sp = min_splits; sp <= max_splits; ++sp) {
            if (!valid(sp)) continue;
            const long long slots = slots_for(sp);
            const long long ctas = static_cast<long long>(base) * sp;
            const long long waves = (ctas + slots - 1) / slots;
            const double eff = static_cast<double>(ctas) / static_cast<double>(waves * slots);
            if (eff > best_eff + 1e-9) {
                best_eff = eff;
                best = sp;
            }
            if (waves > 4) break;
        }
    }
    p.slice_chunks = (KC + best - 1) / best;
    p.splits = (KC + p.slice_chunks - 1) / p.slice_chunks;
    p.xr = xr_for(p.slice_chunks) ? 1 : 0;
    p.cluster = (p.splits > 1 && p.splits <= kMaxCluster) ? 1 : 0;
    p.n_tickets = base;
    p.ws_floats = (p.splits > 1 && !p.cluster) ? static_cast<size_t>(base) * p.splits * kNTW * p.mt * 128 : 0;
    p.one_wave = static_cast<long long>(base) * p.splits <=
                 static_cast<long long>(kSMs) *
                     resident_ctas(p.mt, raw, smem_bytes_for(p.mt, sr, p.xr != 0, std::min(M, 8 * p.mt), p.slice_chunks,
                                                             max_groups_in_slice(p.slice_chunks, geff)));
    return p;
}

// Weight and x ring in shared memory for M <= Q4_DECODE_SR_MAX_M rows (one
// m tile), in registers otherwise.
#ifndef Q4_DECODE_SR_MAX_M
#define Q4_DECODE_SR_MAX_M 8
#endif
// M <= 8: the raw-pair arithmetic (fewer instructions, 2 CTAs per SM) when its
// grid is a single wave, else the exact-pair arithmetic at 3 CTAs per SM,
// which keeps mid-size layers in one wave.  Larger M: exact pairs.
DecodePlan plan_decode(int M, int K, int N, int geff) {
    const bool sr = M <= Q4_DECODE_SR_MAX_M;
    if (M <= 8) {
        const DecodePlan r = plan_decode_arith(M, K, N, geff, true, sr);
        if (r.one_wave) return r;
    }
    return plan_decode_arith(M, K, N, geff, false, sr);
}

size_t decode_ws_floats_for(int M, int K, int N, int geff) { return plan_decode(M, K, N, geff).ws_floats; }

cudaError_t launch_decode(const HandleView &h, const DecodePlan &p, const DecodeWork &w, const uint16_t *x, int M,
                          uint16_t *out, cudaStream_t s) {
    switch (p.mt) {
        case 1:
            if (p.raw) {
                if (!p.sr) return launch_mt<1, true, false, false>(h, p, w, x, M, out, s);
                return p.xr ? launch_mt<1, true, true, true>(h, p, w, x, M, out, s)
                            : launch_mt<1, true, true, false>(h, p, w, x, M, out, s);
            }
            if (!p.sr) return launch_mt<1, false, false, false>(h, p, w, x, M, out, s);
            return p.xr ? launch_mt<1, false, true, true>(h, p, w, x, M, out, s)
                        : launch_mt<1, false, true, false>(h, p, w, x, M, out, s);
        case 2: return launch_mt<2, false, false, false>(h, p, w, x, M, out, s);
        default: return launch_mt<4, false, false, false>(h, p, w, x, M, out, s);
    }
}

}  // namespace q4
