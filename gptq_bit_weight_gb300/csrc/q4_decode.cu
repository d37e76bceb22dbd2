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
// contiguous runs of 64-row chunks.  For each chunk a lane issues one 16-byte
// streaming load per column tile; a ring of DEPTH chunks keeps loads in
// flight while earlier chunks are computed.
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
//
// Reduction.  Warps of a CTA are summed in a fixed order through shared
// memory.  With more than one K slice, each CTA writes its fp32 partial tile
// to the workspace, and the last CTA of a column tile to arrive (an atomic
// ticket; nobody waits) adds the slices in slice order, adds bias and rounds
// once to fp16.  The result is deterministic.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdlib>

#include "q4_internal.cuh"

namespace q4 {

namespace {

// Tuning parameters (compile-time; the defaults are the measured choice).
#ifndef Q4_DECODE_WARPS
#define Q4_DECODE_WARPS 8
#endif
#ifndef Q4_DECODE_NTW
#define Q4_DECODE_NTW 2
#endif
#ifndef Q4_DECODE_DEPTH
#define Q4_DECODE_DEPTH 4
#endif
// 0: each warp streams one contiguous run of 64-row chunks; 1: the warps of a
// CTA take consecutive chunk pairs, so a CTA reads one contiguous span per step.
#ifndef Q4_DECODE_INTERLEAVE
#define Q4_DECODE_INTERLEAVE 0
#endif
constexpr int kWarps = Q4_DECODE_WARPS;
constexpr int kThreads = 32 * kWarps;
constexpr int kNTW = Q4_DECODE_NTW;             // 16-column tiles per CTA
constexpr int kNB = 16 * kNTW;      // columns per CTA
constexpr int kDepth = Q4_DECODE_DEPTH;         // chunks in the load ring
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
    uint64_t inv_bpg;   // ceil(2^32 / blocks-per-group): group of 32-row block b = (b * inv_bpg) >> 32
};

__host__ __device__ inline int x_row_stride(int slice_chunks) { return slice_chunks * 64 + 32; }

template <int MT>
__host__ __device__ inline size_t smem_bytes(int xrows, int slice_chunks, int max_groups) {
    return static_cast<size_t>(xrows) * x_row_stride(slice_chunks) * 2      // x slice
           + static_cast<size_t>(kWarps) * kNTW * MT * 128 * 4              // warp partials
           + static_cast<size_t>(max_groups) * kGszStride * 4;             // scale pairs + zero words
}

__host__ __device__ inline size_t smem_bytes_for(int mt, int xrows, int slice_chunks, int max_groups) {
    return static_cast<size_t>(xrows) * x_row_stride(slice_chunks) * 2 +
           static_cast<size_t>(kWarps) * kNTW * mt * 128 * 4 + static_cast<size_t>(max_groups) * kGszStride * 4;
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
template <int MT, bool RAW>
__global__ void __launch_bounds__(kThreads, min_blocks(MT, RAW)) decode_kernel(HandleView h, DecodeArgs a) {
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

    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);
    float *red = reinterpret_cast<float *>(smem + static_cast<size_t>(a.xrows) * XS * 2);
    uint32_t *gsz = reinterpret_cast<uint32_t *>(red + kWarps * kNTW * MT * 128);

    // Let the next kernel in the stream start its own prologue as soon as
    // every CTA of this grid is resident (programmatic dependent launch).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // This warp's sequence of 64-row chunks within the CTA's slice.
#if Q4_DECODE_INTERLEAVE
    const int full_steps = nch / (2 * kWarps);
    const int rem = nch - full_steps * 2 * kWarps;
    const int extra = min(2, max(0, rem - 2 * warp));
    const int wn = 2 * full_steps + extra;
    auto chunk_of = [&](int c) { return c_beg + 2 * kWarps * (c >> 1) + 2 * warp + (c & 1); };
#else
    const int wc_beg = c_beg + (nch * warp) / kWarps;
    const int wn = c_beg + (nch * (warp + 1)) / kWarps - wc_beg;
    auto chunk_of = [&](int c) { return wc_beg + c; };
#endif
    const int g_base = (c_beg * 64) / geff;

    // ---- first kDepth chunks of packed weights: handle-owned constant data,
    //      so the loads may be issued before the preceding grid has finished.
    const uint4 *wbase[kNTW];
#pragma unroll
    for (int nt = 0; nt < kNTW; ++nt) wbase[nt] = h.wp + static_cast<size_t>(nt0 + nt) * KC * 32 + lane;
    uint4 buf[kDepth][kNTW];
#pragma unroll
    for (int i = 0; i < kDepth; ++i)
        if (i < wn)
#pragma unroll
            for (int nt = 0; nt < kNTW; ++nt) buf[i][nt] = ldg_stream(wbase[nt] + static_cast<size_t>(chunk_of(i)) * 32);

    // ---- stage the slice's scale pairs / zero words (constant) and, once
    //      the preceding grid is done, x[m0 : m0 + mrows][slice], with
    //      asynchronous global->shared copies: together with the weight loads
    //      above they form a single round trip to memory.  Lanes whose x row
    //      is past M use zeros without reading shared memory.
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
        // x, the workspace, the tickets and out may belong to the preceding
        // grid: wait for it (a no-op without programmatic dependent launch).
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int vpr = nch * 8;                        // 16-byte vectors per row
        for (int r = 0; r < mrows; ++r) {
            const uint16_t *src = a.x + static_cast<size_t>(m0 + r) * K + c_beg * 64;
            for (int c = threadIdx.x; c < vpr; c += kThreads) cp_async_16(xs + r * XS + c * 8, src + c * 8);
        }
        cp_async_wait_all();
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
        uint32_t nzlo[kNTW][2], nzhi[kNTW][2];
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
        float sc[kNTW][2], czl[kNTW][2], czh[kNTW][2];   // scale, -(1025 + z), -(65 + z)
        int grp = -1;

        auto load_group = [&](int g) {
            const uint32_t *base = gsz + (g - g_base) * kGszStride;
#pragma unroll
            for (int nt = 0; nt < kNTW; ++nt) {
                const uint32_t sp = base[nt * 8 + gq];
                const uint32_t zw0 = base[kNTW * 8 + nt * 2], zw1 = base[kNTW * 8 + nt * 2 + 1];
                sc[nt][0] = __half2float(__ushort_as_half(static_cast<unsigned short>(sp & 0xFFFFu)));
                sc[nt][1] = __half2float(__ushort_as_half(static_cast<unsigned short>(sp >> 16)));
                // effective zero points (stored + zero_offset) of columns gq, gq + 8
                const float z0 = static_cast<float>(((zw0 >> (4 * gq)) & 0xFu) + h.zero_offset);
                const float z1 = static_cast<float>(((zw1 >> (4 * gq)) & 0xFu) + h.zero_offset);
                czl[nt][0] = -(1024.f + z0);
                czl[nt][1] = -(1024.f + z1);
                czh[nt][0] = -(64.f + z0);
                czh[nt][1] = -(64.f + z1);
                if (!RAW) {
                    const uint32_t zi0 = ((zw0 >> (4 * gq)) & 0xFu) + h.zero_offset - 1u;
                    const uint32_t zi1 = ((zw1 >> (4 * gq)) & 0xFu) + h.zero_offset - 1u;
                    nzlo[nt][0] = neg_zlo(zi0);
                    nzhi[nt][0] = neg_zhi(zi0);
                    nzlo[nt][1] = neg_zlo(zi1);
                    nzhi[nt][1] = neg_zhi(zi1);
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

        for (int base = 0; base < wn; base += kDepth) {
#pragma unroll
            for (int i = 0; i < kDepth; ++i) {
                const int c = base + i;
                if (c < wn) {
                    const int chunk = chunk_of(c);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int g = static_cast<int>((static_cast<uint64_t>(2 * chunk + hh) * a.inv_bpg) >> 32);
                        if (g != grp) {
                            if (grp >= 0) flush();
                            load_group(g);
                            grp = g;
                        }
                        const int kk = (2 * (chunk - c_beg) + hh) * 32 + 8 * tq;
                        uint4 xb[MT];
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            xb[mt] = make_uint4(0u, 0u, 0u, 0u);
                            if (mt * 8 + gq < mrows)
                                xb[mt] = *reinterpret_cast<const uint4 *>(xs + (mt * 8 + gq) * XS + kk);
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
                            const uint32_t lo = hh ? buf[i][nt].z : buf[i][nt].x;    // column 16nt + gq
                            const uint32_t hi = hh ? buf[i][nt].w : buf[i][nt].y;    // column 16nt + gq + 8
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
                    if (c + kDepth < wn)
#pragma unroll
                        for (int nt = 0; nt < kNTW; ++nt)
                            buf[i][nt] = ldg_stream(wbase[nt] + static_cast<size_t>(chunk_of(c + kDepth)) * 32);
                }
            }
        }
        flush();
    }

    // ---- fixed-order reduction over the CTA's warps
    constexpr int E = kNTW * MT * 128;                 // partial elements per CTA
#pragma unroll
    for (int nt = 0; nt < kNTW; ++nt)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            *reinterpret_cast<float4 *>(red + warp * E + (nt * MT + mt) * 128 + lane * 4) =
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
            if (h.bias) v += __half2float(__ushort_as_half(h.bias[n]));
            a.out[static_cast<size_t>(m) * N + n] = __half_as_ushort(__float2half_rn(v));
        }
    };

    // CTA partial: the warps' partials summed in warp order, kept in red[0, E)
    // (each thread reads its own elements of every warp before writing one).
    for (int e = threadIdx.x; e < E; e += kThreads) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += red[w * E + e];
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

template <int MT, bool RAW>
cudaError_t launch_mt(const HandleView &h, const DecodePlan &p, const DecodeWork &w, const uint16_t *x, int M,
                      uint16_t *out, cudaStream_t s) {
    const int xrows = M < 8 * MT ? M : 8 * MT;
    const size_t smem = smem_bytes<MT>(xrows, p.slice_chunks, max_groups_in_slice(p.slice_chunks, h.geff));
    // Opt in once to the largest dynamic shared memory the device allows
    // next to the kernel's static shared memory.
    static int max_dyn = -1;
    if (max_dyn < 0) {
        int dev = 0, optin = 0;
        cudaFuncAttributes fa{};
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, decode_kernel<MT, RAW>);
        const int want = optin - static_cast<int>(fa.sharedSizeBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_kernel<MT, RAW>, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
        if (e != cudaSuccess) return e;
        max_dyn = want;
    }
    if (smem > static_cast<size_t>(max_dyn)) return cudaErrorInvalidConfiguration;
    // exact floor(b / bpg) for b * bpg < 2^32 (b <= K / 32)
    const uint64_t bpg = static_cast<uint64_t>(h.geff / 32);
    const uint64_t inv_bpg = (0x100000000ull + bpg - 1) / bpg;
    DecodeArgs a{x, out, w.ws, w.tickets, M, p.splits, p.slice_chunks, xrows, p.cluster, inv_bpg};
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
    return cudaLaunchKernelEx(&cfg, decode_kernel<MT, RAW>, h, a);
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
static DecodePlan plan_decode_arith(int M, int K, int N, int geff, bool raw) {
    DecodePlan p{};
    p.raw = raw ? 1 : 0;
    p.mt = M <= 8 ? 1 : (M <= 16 ? 2 : 4);
    p.zdim = (M + 8 * p.mt - 1) / (8 * p.mt);
    p.ctas_n = N / kNB;
    const int KC = K / 64;
    const int xrows = std::min(M, 8 * p.mt);
    // x staging: xrows * slice * 64 fp16 <= 64 KB
    const int max_slice = std::min(KC, std::max(8, std::min(64, 512 / xrows)));
    const int base = p.ctas_n * p.zdim;
    const int min_splits = (KC + max_slice - 1) / max_slice;
    const int max_splits = std::max(min_splits, KC / 16);   // at least two chunks per warp
    auto slots_for = [&](int sp) {
        const int slice = (KC + sp - 1) / sp;
        const size_t smem = smem_bytes_for(p.mt, xrows, slice, max_groups_in_slice(slice, geff));
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
    p.cluster = (p.splits > 1 && p.splits <= kMaxCluster) ? 1 : 0;
    p.n_tickets = base;
    p.ws_floats = (p.splits > 1 && !p.cluster) ? static_cast<size_t>(base) * p.splits * kNTW * p.mt * 128 : 0;
    p.one_wave = static_cast<long long>(base) * p.splits <=
                 static_cast<long long>(kSMs) *
                     resident_ctas(p.mt, raw, smem_bytes_for(p.mt, std::min(M, 8 * p.mt), p.slice_chunks,
                                                             max_groups_in_slice(p.slice_chunks, geff)));
    return p;
}

// M <= 8: the raw-pair arithmetic (fewer instructions, 2 CTAs per SM) when its
// grid is a single wave, else the exact-pair arithmetic at 3 CTAs per SM,
// which keeps mid-size layers in one wave.  Larger M: exact pairs.
DecodePlan plan_decode(int M, int K, int N, int geff) {
    if (M <= 8) {
        const DecodePlan r = plan_decode_arith(M, K, N, geff, true);
        if (r.one_wave) return r;
    }
    return plan_decode_arith(M, K, N, geff, false);
}

size_t decode_ws_floats_for(int M, int K, int N, int geff) { return plan_decode(M, K, N, geff).ws_floats; }

cudaError_t launch_decode(const HandleView &h, const DecodePlan &p, const DecodeWork &w, const uint16_t *x, int M,
                          uint16_t *out, cudaStream_t s) {
    switch (p.mt) {
        case 1: return p.raw ? launch_mt<1, true>(h, p, w, x, M, out, s) : launch_mt<1, false>(h, p, w, x, M, out, s);
        case 2: return launch_mt<2, false>(h, p, w, x, M, out, s);
        default: return launch_mt<4, false>(h, p, w, x, M, out, s);
    }
}

}  // namespace q4
