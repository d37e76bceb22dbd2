// One-time repack of a GPTQ checkpoint into the private execution layout,
// and the read-back kernels (codes, dequantized weights) plus the act-order
// activation gather.
//
// "Inference Backends", "Packing, conversion, and runtime initialization":
// runtime initialization repacks loaded tensors into a kernel's private
// layout and shuffles scales/zeros.  "Implementation: Predibase Lorax GPTQ
// Exllama V1", "Description": temp_state reorders activations for act-order
// and temp_dq receives dequantized weights.
#include <cuda_fp16.h>

#include <algorithm>

#include "q4_internal.cuh"

namespace q4 {

// ---------------------------------------------------------------- codes
// One thread per private word.  Each of its eight rows (permuted order) is
// looked up in the checkpoint through P, its nibble extracted and placed at
// nib_pos(r).  Rows of one act-order word come from different checkpoint
// words, so the codes are unpacked and repacked one by one.  P[j] = -1 marks
// a padding row (groups of unequal size padded to a common length): code 0.
__global__ void repack_codes_kernel(const int32_t *__restrict__ qweight, const int32_t *__restrict__ perm,
                                    int K, int N, uint32_t *__restrict__ wp) {
    const int KC = K / 64;
    const size_t total = static_cast<size_t>(N / 16) * KC * 128;
    for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int j = static_cast<int>(idx & 3);
        const int lane = static_cast<int>((idx >> 2) & 31);
        const size_t tile = idx >> 7;
        const int kc = static_cast<int>(tile % KC);
        const int nt = static_cast<int>(tile / KC);
        const int gq = lane >> 2, tq = lane & 3;
        const int n = 16 * nt + gq + 8 * (j & 1);
        const int kb = 64 * kc + 32 * (j >> 1) + 8 * tq;
        uint32_t out = 0;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int k = perm ? perm[kb + r] : kb + r;
            if (k < 0) continue;                        // a padding row: code 0 (x is 0 there)
            const uint32_t word = static_cast<uint32_t>(qweight[static_cast<size_t>(k >> 3) * N + n]);
            const uint32_t code = (word >> (4 * (k & 7))) & 0xFu;
            out |= code << (4 * nib_pos(r));
        }
        wp[idx] = out;
    }
}

cudaError_t launch_repack_codes(const int32_t *qweight, const int32_t *perm, int K, int N, uint32_t *wp,
                                cudaStream_t s) {
    const size_t total = static_cast<size_t>(N / 16) * (K / 64) * 128;
    const int threads = 256;
    const size_t want = (total + threads - 1) / threads;
    const int blocks = static_cast<int>(want < 65535u * 16u ? want : 65535u * 16u);
    repack_codes_kernel<<<blocks, threads, 0, s>>>(qweight, perm, K, N, wp);
    return cudaGetLastError();
}

// --------------------------------------------------------------- scales
__global__ void repack_scales_kernel(const uint16_t *__restrict__ scales, int G, int N, uint32_t *__restrict__ s2) {
    const size_t total = static_cast<size_t>(G) * (N / 16) * 8;
    for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int gq = static_cast<int>(idx & 7);
        const size_t rest = idx >> 3;
        const int nt = static_cast<int>(rest % (N / 16));
        const int gr = static_cast<int>(rest / (N / 16));
        const size_t base = static_cast<size_t>(gr) * N + 16 * nt + gq;
        s2[idx] = static_cast<uint32_t>(scales[base]) | (static_cast<uint32_t>(scales[base + 8]) << 16);
    }
}

cudaError_t launch_repack_scales(const uint16_t *scales, int G, int N, uint32_t *s2, cudaStream_t s) {
    const size_t total = static_cast<size_t>(G) * (N / 16) * 8;
    const int threads = 256;
    const size_t want = (total + threads - 1) / threads;
    const int blocks = static_cast<int>(want < 65535u * 16u ? want : 65535u * 16u);
    repack_scales_kernel<<<blocks, threads, 0, s>>>(scales, G, N, s2);
    return cudaGetLastError();
}

// -------------------------------------------------- unpack (read-back)
// q[k][n] in original row order from the private words; z from the zeros.
__global__ void debug_unpack_kernel(HandleView h, uint8_t *__restrict__ q, uint8_t *__restrict__ z) {
    const int K = h.K, N = h.N, KC = K / 64;
    const uint32_t *wp = reinterpret_cast<const uint32_t *>(h.wp);
    const size_t total_words = static_cast<size_t>(N / 16) * KC * 128;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    const size_t tid = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
    if (q) {
        for (size_t idx = tid; idx < total_words; idx += stride) {
            const int j = static_cast<int>(idx & 3);
            const int lane = static_cast<int>((idx >> 2) & 31);
            const size_t tile = idx >> 7;
            const int kc = static_cast<int>(tile % KC);
            const int nt = static_cast<int>(tile / KC);
            const int n = 16 * nt + (lane >> 2) + 8 * (j & 1);
            const int kb = 64 * kc + 32 * (j >> 1) + 8 * (lane & 3);
            const uint32_t w = wp[idx];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int k = h.perm ? h.perm[kb + r] : kb + r;
                if (k >= 0) q[static_cast<size_t>(k) * N + n] = static_cast<uint8_t>((w >> (4 * nib_pos(r))) & 0xFu);
            }
        }
    }
    if (z) {
        const size_t total_z = static_cast<size_t>(h.G) * N;
        for (size_t idx = tid; idx < total_z; idx += stride) {
            const int n = static_cast<int>(idx % N);
            const size_t gr = idx / N;
            const uint32_t w = h.zeros[gr * (N / 8) + n / 8];
            z[idx] = static_cast<uint8_t>((w >> (4 * (n & 7))) & 0xFu);
        }
    }
}

cudaError_t launch_debug_unpack(const HandleView &h, uint8_t *q, uint8_t *z, cudaStream_t s) {
    debug_unpack_kernel<<<kSMs * 8, 256, 0, s>>>(h, q, z);
    return cudaGetLastError();
}

// -------------------------------------------------------------- dequant
// temp_dq[k][n] = fp16(s * (q - (z + zero_offset))), original row order.
// A CTA takes 64 columns x 64 (permuted) rows at a time: 256 threads each
// dequantize two private words (16 values) into a shared tile, then the tile
// is written out one 128-byte row per 8 threads, each row to its original
// position P[j].  The product s * (q - z - 1) is exact in fp32 (11-bit times
// 5-bit integer), so __float2half_rn rounds it exactly once.
__global__ void __launch_bounds__(256) dequant_kernel(HandleView h, uint16_t *__restrict__ out) {
    constexpr int kPad = 8;
    __shared__ __align__(16) uint16_t tile[64][64 + kPad];
    const int K = h.K, N = h.N, KC = K / 64, NT64 = N / 64;
    const int tid = threadIdx.x;
    const int bpg = h.geff / 32;
    const uint32_t *wp = reinterpret_cast<const uint32_t *>(h.wp);
    const size_t ntiles = static_cast<size_t>(NT64) * KC;
    for (size_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int kc = static_cast<int>(t % KC);
        const int n64 = static_cast<int>(t / KC);
#pragma unroll
        for (int rep = 0; rep < 2; ++rep) {
            const int widx = tid + 256 * rep;          // 0..511 within the 64x64 tile
            const int j = widx & 3;
            const int lane = (widx >> 2) & 31;
            const int ntl = widx >> 7;                 // n16 tile within the 64 columns
            const int nt = 4 * n64 + ntl;
            const int gq = lane >> 2, tq = lane & 3;
            const int n = 16 * nt + gq + 8 * (j & 1);
            const int kl = 32 * (j >> 1) + 8 * tq;     // local row of r = 0
            const int gr = (64 * kc + kl) / 32 / bpg;  // group of these eight rows
            const uint32_t w = wp[wp_index(nt, kc, lane, j, KC)];
            const uint32_t zw = h.zeros[static_cast<size_t>(gr) * (N / 8) + n / 8];
            const int zeff = static_cast<int>((zw >> (4 * (n & 7))) & 0xFu) + (gr < h.zsplit ? 0 : h.zero_offset);
            const uint32_t sp = h.s2[(static_cast<size_t>(gr) * (N / 16) + nt) * 8 + gq];
            const uint16_t sbits = static_cast<uint16_t>((j & 1) ? (sp >> 16) : (sp & 0xFFFFu));
            const float s = __half2float(__ushort_as_half(sbits));
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int code = static_cast<int>((w >> (4 * nib_pos(r))) & 0xFu);
                const float v = s * static_cast<float>(code - zeff);
                tile[kl + r][n - 64 * n64] = __half_as_ushort(__float2half_rn(v));
            }
        }
        __syncthreads();
#pragma unroll
        for (int rep = 0; rep < 2; ++rep) {
            const int row = (tid >> 3) + 32 * rep;
            const int c8 = tid & 7;
            const int jrow = 64 * kc + row;
            const int k = h.perm ? h.perm[jrow] : jrow;
            const uint4 v = *reinterpret_cast<const uint4 *>(&tile[row][8 * c8]);
            if (k >= 0) *reinterpret_cast<uint4 *>(out + static_cast<size_t>(k) * N + 64 * n64 + 8 * c8) = v;
        }
        __syncthreads();
    }
}

cudaError_t launch_dequant(const HandleView &h, uint16_t *temp_dq, cudaStream_t s) {
    const size_t ntiles = static_cast<size_t>(h.N / 64) * (h.K / 64);
    const size_t want = ntiles;
    const int blocks = static_cast<int>(want < static_cast<size_t>(kSMs) * 8 ? want : static_cast<size_t>(kSMs) * 8);
    dequant_kernel<<<blocks, 256, 0, s>>>(h, temp_dq);
    return cudaGetLastError();
}

// Programmatic dependent launch for the activation kernels: the dependent
// decode / prefill grid may launch at once (its weight prefetch needs nothing
// from here), while these kernels wait for the preceding grid before they
// read x or overwrite temp_state, which that grid may still be reading.
// Used when the register-streaming decode follows (early), where it measured
// 10-30 % faster per call at M <= 8; before the TMA-ring decode (M = 16) it
// measured slower.
// (early: let the dependent grid launch now; otherwise it launches when this
// grid ends, which keeps a TMA-ring decode from holding SM slots the gather
// still needs.)
__device__ __forceinline__ void pdl_enter(bool early) {
    if (early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl(bool pdl, Kern kern, int grid, int block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl && pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ------------------------------------------------------------- xreorder
// temp_state[m][j] = x[m][P[j]] (0 where P[j] = -1, a padding row): eight
// consecutive j per thread, written as one 16-byte store; the gathered reads
// come from the small x (L2-resident).  x rows hold Kx values, temp_state
// rows K >= Kx.
__device__ __forceinline__ uint32_t gather2(const uint16_t *xr, int pa, int pb) {
    const uint32_t a = pa >= 0 ? xr[pa] : 0u, b = pb >= 0 ? xr[pb] : 0u;
    return a | (b << 16);
}

__global__ void xreorder_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ perm, int M, int Kx,
                                int K, uint16_t *__restrict__ ts, bool early) {
    if (early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const size_t total = static_cast<size_t>(M) * (K / 8);
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
    // The permutation is a handle constant: the thread's first vectors of it
    // are read before the preceding grid has finished, leaving only the
    // gather from x on the path after it.
    int4 p0 = make_int4(-1, -1, -1, -1), p1 = p0;
    if (idx < total) {
        const int j0 = static_cast<int>(idx % (K / 8)) * 8;
        p0 = *reinterpret_cast<const int4 *>(perm + j0);
        p1 = *reinterpret_cast<const int4 *>(perm + j0 + 4);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (bool first = true; idx < total; idx += stride, first = false) {
        const size_t m = idx / (K / 8);
        const int j0 = static_cast<int>(idx % (K / 8)) * 8;
        const uint16_t *xr = x + m * Kx;
        if (!first) {
            p0 = *reinterpret_cast<const int4 *>(perm + j0);
            p1 = *reinterpret_cast<const int4 *>(perm + j0 + 4);
        }
        uint4 v;
        v.x = gather2(xr, p0.x, p0.y);
        v.y = gather2(xr, p0.z, p0.w);
        v.z = gather2(xr, p1.x, p1.y);
        v.w = gather2(xr, p1.z, p1.w);
        *reinterpret_cast<uint4 *>(ts + m * K + j0) = v;
    }
}

// Many rows: the permutation is staged once per CTA and each row of x is
// staged in shared memory with 16-byte loads, so that both the reads and the
// gathered 16-byte writes are coalesced (the gather itself hits shared
// memory).  Rows are taken round-robin by the CTAs.  Each thread's loads of a
// row are all issued before any is stored, and rows wide enough to leave one
// CTA per SM get 1024 threads, so that a row costs about one memory round
// trip (with 256 threads and one load at a time a 28672-wide row took ~14:
// Llama-70B act-order prefill at M = 2048 on 28672 x 8192 1.31 -> 1.42
// PFLOP/s).
__global__ void __launch_bounds__(1024) xreorder_rows_kernel(const uint16_t *__restrict__ x,
                                                              const int32_t *__restrict__ perm, int M, int Kx, int K,
                                                              uint16_t *__restrict__ ts, bool early) {
    extern __shared__ __align__(16) unsigned char sm[];
    pdl_enter(early);
    int32_t *sp = reinterpret_cast<int32_t *>(sm);
    uint16_t *sx = reinterpret_cast<uint16_t *>(sm + static_cast<size_t>(K) * 4);
    const int nvx = Kx / 8, nv = K / 8;                    // 16-byte vectors per x row / temp_state row
    for (int i = threadIdx.x; i < K / 4; i += blockDim.x)
        reinterpret_cast<int4 *>(sp)[i] = reinterpret_cast<const int4 *>(perm)[i];
    constexpr int kBatch = 4;                              // loads in flight per thread
    for (int m = blockIdx.x; m < M; m += gridDim.x) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(m) * Kx);
        __syncthreads();                                   // the previous row's gathers are done
        for (int i0 = threadIdx.x; i0 < nvx; i0 += kBatch * blockDim.x) {
            uint4 v[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int i = i0 + b * blockDim.x;
                if (i < nvx) v[b] = xr[i];
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int i = i0 + b * blockDim.x;
                if (i < nvx) reinterpret_cast<uint4 *>(sx)[i] = v[b];
            }
        }
        __syncthreads();
        uint4 *out = reinterpret_cast<uint4 *>(ts + static_cast<size_t>(m) * K);
        for (int i = threadIdx.x; i < nv; i += blockDim.x) {
            const int4 p0 = reinterpret_cast<const int4 *>(sp)[2 * i];
            const int4 p1 = reinterpret_cast<const int4 *>(sp)[2 * i + 1];
            uint4 v;
            v.x = gather2(sx, p0.x, p0.y);
            v.y = gather2(sx, p0.z, p0.w);
            v.z = gather2(sx, p1.x, p1.y);
            v.w = gather2(sx, p1.z, p1.w);
            out[i] = v;
        }
    }
}

cudaError_t launch_xreorder(const uint16_t *x, const int32_t *perm, int M, int Kx, int K, uint16_t *temp_state,
                            cudaStream_t s, bool early) {
    const size_t rows_smem = static_cast<size_t>(K) * 4 + static_cast<size_t>(Kx) * 2;   // permutation + one row
    if (M >= 32 && rows_smem <= 200 * 1024) {
        static cudaError_t attr =
            cudaFuncSetAttribute(xreorder_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (attr != cudaSuccess) return attr;
        const int per_sm = static_cast<int>((228 * 1024) / (rows_smem + 1024));
        // one CTA per SM (a wide row and its permutation fill shared memory):
        // 1024 threads; else 256 threads and several CTAs per SM (measured
        // faster on 4096- and 11008-wide rows)
        const int threads = per_sm <= 1 ? 1024 : 256;
        const int ctas = std::min(M, kSMs * std::max(1, std::min(per_sm, 8)));
        return launch_pdl(early, xreorder_rows_kernel, ctas, threads, rows_smem, s, x, perm, M, Kx, K, temp_state,
                          early);
    }
    const size_t total = static_cast<size_t>(M) * (K / 8);
    const int threads = 256;
    const size_t want = (total + threads - 1) / threads;
    const int blocks = static_cast<int>(want < static_cast<size_t>(kSMs) * 16 ? want : static_cast<size_t>(kSMs) * 16);
    return launch_pdl(early, xreorder_kernel, blocks > 0 ? blocks : 1, threads, size_t{0}, s, x, perm, M, Kx, K,
                      temp_state, early);
}

// --------------------------------------------------- bf16 activations
// One CTA per row: the largest magnitude of the row picks a power of two
// 2^e with max|x| * 2^-e in [2^14, 2^15); each value times 2^-e (exact in
// fp32) is rounded once to fp16.  A bf16 value has an 8-bit significand, so
// the fp16 value is exact unless it lies more than ~2^28 below the row's
// largest.  The kernels' epilogues multiply the fp32 sums by 2^e (exact).
__global__ void __launch_bounds__(1024) xprep_bf16_kernel(const uint16_t *__restrict__ x,
                                                         const int32_t *__restrict__ perm, int M, int Kx, int K,
                                                         uint16_t *__restrict__ ts, float *__restrict__ rowscale,
                                                         bool early) {
    __shared__ float wmax[32];
    pdl_enter(early);
    const int nw = blockDim.x >> 5;
    for (int m = blockIdx.x; m < M; m += gridDim.x) {
        const uint16_t *xr = x + static_cast<size_t>(m) * Kx;
        float mx = 0.f;
        for (int k = threadIdx.x; k < Kx; k += blockDim.x)
            mx = fmaxf(mx, fabsf(__uint_as_float(static_cast<uint32_t>(xr[k]) << 16)));
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
        __syncthreads();
        mx = wmax[0];
        for (int w = 1; w < nw; ++w) mx = fmaxf(mx, wmax[w]);
        __syncthreads();                               // wmax is reused by the next row
        // e = ilogb(max) - 14, kept where 2^-e and 2^e are normal fp32 values
        int e = 0;
        if (mx > 0.f && mx <= 3.402823466e38f) e = min(max(ilogbf(mx) - 14, -110), 113);
        const float down = __int_as_float((127 - e) << 23);   // 2^-e
        if (threadIdx.x == 0) rowscale[m] = __int_as_float((127 + e) << 23);
        uint16_t *tr = ts + static_cast<size_t>(m) * K;
        for (int j = threadIdx.x; j < K; j += blockDim.x) {
            const int k = perm ? perm[j] : j;
            const float v = k >= 0 ? __uint_as_float(static_cast<uint32_t>(xr[k]) << 16) * down : 0.f;
            tr[j] = __half_as_ushort(__float2half_rn(v));
        }
    }
}

cudaError_t launch_xprep_bf16(const uint16_t *x, const int32_t *perm, int M, int Kx, int K, uint16_t *temp_state,
                              float *rowscale, cudaStream_t s, bool early) {
    // one CTA per row; wide CTAs when there are few rows
    const int ctas = std::min(M, kSMs * 8);
    const int threads = M <= kSMs ? 1024 : 256;
    return launch_pdl(early, xprep_bf16_kernel, ctas > 0 ? ctas : 1, threads, size_t{0}, s, x, perm, M, Kx, K,
                      temp_state, rowscale, early);
}

// --------------------------------------------------- fp32 activations
// One CTA per row.  As for bf16, the row's largest magnitude picks 2^e with
// max|x| * 2^-e in [2^14, 2^15); v = x * 2^-e is exact in fp32.  hi = v
// rounded once to fp16; v - hi is exact in fp32 (hi is within half an fp16
// unit of v), and lo = that residual rounded once to fp16.  hi + lo carries
// v to about 2^-22 of itself, so the fp16 kernels run on 2M rows (hi rows,
// then lo rows) and the two results of each row are summed afterwards.
__global__ void __launch_bounds__(1024) xprep_f32_kernel(const float *__restrict__ x, const int32_t *__restrict__ perm,
                                                        int M, int Kx, int K, uint16_t *__restrict__ ts,
                                                        float *__restrict__ rowscale) {
    __shared__ float wmax[32];
    pdl_enter(false);
    const int nw = blockDim.x >> 5;
    for (int m = blockIdx.x; m < M; m += gridDim.x) {
        const float *xr = x + static_cast<size_t>(m) * Kx;
        float mx = 0.f;
        for (int k = threadIdx.x; k < Kx; k += blockDim.x) mx = fmaxf(mx, fabsf(xr[k]));
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
        __syncthreads();
        mx = wmax[0];
        for (int w = 1; w < nw; ++w) mx = fmaxf(mx, wmax[w]);
        __syncthreads();                               // wmax is reused by the next row
        // e = ilogb(max) - 14, kept where 2^-e and 2^e are normal fp32 values
        int e = 0;
        if (mx > 0.f && mx <= 3.402823466e38f) e = min(max(ilogbf(mx) - 14, -110), 113);
        const float down = __int_as_float((127 - e) << 23);   // 2^-e
        if (threadIdx.x == 0) rowscale[m] = __int_as_float((127 + e) << 23);
        uint16_t *hi_row = ts + static_cast<size_t>(m) * K;
        uint16_t *lo_row = ts + static_cast<size_t>(M + m) * K;
        for (int j = threadIdx.x; j < K; j += blockDim.x) {
            const int k = perm ? perm[j] : j;
            const float v = k >= 0 ? xr[k] * down : 0.f;
            const __half hi = __float2half_rn(v);
            const float r = v - __half2float(hi);
            hi_row[j] = __half_as_ushort(hi);
            lo_row[j] = __half_as_ushort(__float2half_rn(r));
        }
    }
}

cudaError_t launch_xprep_f32(const float *x, const int32_t *perm, int M, int Kx, int K, uint16_t *temp_state,
                             float *rowscale, cudaStream_t s) {
    const int ctas = std::min(M, kSMs * 8);
    const int threads = M <= kSMs ? 1024 : 256;
    return launch_pdl(false, xprep_f32_kernel, ctas > 0 ? ctas : 1, threads, size_t{0}, s, x, perm, M, Kx, K,
                      temp_state, rowscale);
}

// y[m][n] = (part[m][n] + part[M + m][n]) * rowscale[m] + bias[n]: the hi and
// lo results of a row summed in fp32, the row's power of two restored
// (exact), bias added; no rounding beyond fp32.  Four columns per thread.
__global__ void combine_f32_kernel(const float *__restrict__ part, const float *__restrict__ rowscale,
                                   const uint16_t *__restrict__ bias, int M, int N, float *__restrict__ y) {
    pdl_enter(false);
    const size_t total = static_cast<size_t>(M) * (N / 4);
    for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t m = idx / (N / 4);
        const int n = static_cast<int>(idx % (N / 4)) * 4;
        const float4 a = *reinterpret_cast<const float4 *>(part + m * N + n);
        const float4 b = *reinterpret_cast<const float4 *>(part + (m + M) * N + n);
        const float rs = rowscale[m];
        float4 o = make_float4((a.x + b.x) * rs, (a.y + b.y) * rs, (a.z + b.z) * rs, (a.w + b.w) * rs);
        if (bias) {
            o.x += __half2float(__ushort_as_half(bias[n]));
            o.y += __half2float(__ushort_as_half(bias[n + 1]));
            o.z += __half2float(__ushort_as_half(bias[n + 2]));
            o.w += __half2float(__ushort_as_half(bias[n + 3]));
        }
        *reinterpret_cast<float4 *>(y + m * N + n) = o;
    }
}

cudaError_t launch_combine_f32(const float *part, const float *rowscale, const uint16_t *bias, int M, int N, float *y,
                               cudaStream_t s) {
    const size_t total = static_cast<size_t>(M) * (N / 4);
    const int threads = 256;
    const size_t want = (total + threads - 1) / threads;
    const int blocks = static_cast<int>(std::min<size_t>(want, static_cast<size_t>(kSMs) * 16));
    return launch_pdl(false, combine_f32_kernel, blocks > 0 ? blocks : 1, threads, size_t{0}, s, part, rowscale, bias,
                      M, N, y);
}

}  // namespace q4
