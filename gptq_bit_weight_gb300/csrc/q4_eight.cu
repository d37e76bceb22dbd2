// 8-bit GPTQ layers held as two 4-bit halves along K.
//
// "Inference Backends", "GPTQ kernel contract": 8-bit codes pack four to an
// int32 word along K (qweight [K/4][N], lowest byte first) and four zero
// points to a word along N (qzeros [G][N/4]); w = s * (q - (z + 1)).
// With q = 16 qh + ql and z = 16 zh + zl (nibbles),
//     s (q - z - 1) = 16 s (qh - zh) + s (ql - zl - 1)
// exactly, so an 8-bit layer is a 4-bit layer over 2K rows: rows [0, K) hold
// the high nibbles with scale 16 s and zero offset 0, rows [K, 2K) the low
// nibbles with scale s and the format's zero offset, and both halves read the
// same column of x.  Every 4-bit kernel then serves 8-bit layers unchanged;
// the read-back kernels here rebuild the 8-bit codes and the dequantized
// matrix from the two halves.
#include <cuda_fp16.h>

#include "q4_internal.cuh"

namespace q4 {

namespace {

// One thread per 4-bit output word of the split layer.
__global__ void split8_codes_kernel(const int32_t *__restrict__ qw8, int K, int N, int32_t *__restrict__ qw4) {
    const size_t total = static_cast<size_t>(2 * K / 8) * N;
    for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(idx % N);
        const int r8 = static_cast<int>(idx / N);           // 8-row block of the 2K rows
        const bool hi = r8 < K / 8;
        const int k0 = 8 * (hi ? r8 : r8 - K / 8);           // first original row
        const uint32_t a = static_cast<uint32_t>(qw8[static_cast<size_t>(k0 / 4) * N + n]);
        const uint32_t b = static_cast<uint32_t>(qw8[static_cast<size_t>(k0 / 4 + 1) * N + n]);
        uint32_t out = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t code = ((i < 4 ? a : b) >> (8 * (i & 3))) & 0xFFu;
            out |= (hi ? code >> 4 : code & 0xFu) << (4 * i);
        }
        qw4[idx] = static_cast<int32_t>(out);
    }
}

// Zero points: [2G][N/8] words; scales: [2G][N], 16 s for the high half.
__global__ void split8_meta_kernel(const int32_t *__restrict__ qz8, const uint16_t *__restrict__ sc, int G, int N,
                                   int32_t *__restrict__ qz4, uint16_t *__restrict__ sc4) {
    const size_t tz = static_cast<size_t>(2 * G) * (N / 8);
    const size_t ts = static_cast<size_t>(2 * G) * N;
    for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < tz + ts;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        if (idx < tz) {
            const int c8 = static_cast<int>(idx % (N / 8));
            const int g2 = static_cast<int>(idx / (N / 8));
            const bool hi = g2 < G;
            const int g = hi ? g2 : g2 - G;
            const uint32_t a = static_cast<uint32_t>(qz8[static_cast<size_t>(g) * (N / 4) + 2 * c8]);
            const uint32_t b = static_cast<uint32_t>(qz8[static_cast<size_t>(g) * (N / 4) + 2 * c8 + 1]);
            uint32_t out = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t z = ((i < 4 ? a : b) >> (8 * (i & 3))) & 0xFFu;
                out |= (hi ? z >> 4 : z & 0xFu) << (4 * i);
            }
            qz4[idx] = static_cast<int32_t>(out);
        } else {
            const size_t j = idx - tz;
            const int n = static_cast<int>(j % N);
            const int g2 = static_cast<int>(j / N);
            const bool hi = g2 < G;
            const uint16_t s = sc[static_cast<size_t>(hi ? g2 : g2 - G) * N + n];
            // 16 s: the exponent moves up by 4, exact unless it overflows
            sc4[j] = hi ? __half_as_ushort(__hmul(__ushort_as_half(s), __float2half(16.0f))) : s;
        }
    }
}

// Code of private row j, column n of the 4-bit layout.
__device__ __forceinline__ uint32_t code_at(const uint32_t *wp, int KC, int j, int n) {
    const int kc = j >> 6, jr = j & 63;
    const int hh = jr >> 5, tq = (jr & 31) >> 3, r = jr & 7;
    const int nt = n >> 4, gq = n & 7, half = (n >> 3) & 1;
    const uint32_t w = wp[wp_index(nt, kc, 4 * gq + tq, 2 * hh + half, KC)];
    return (w >> (4 * nib_pos(r))) & 0xFu;
}

// q[k][n] (8-bit codes) and z[g][n] (8-bit zero points) from the two halves.
__global__ void unpack8_kernel(HandleView h, const int32_t *__restrict__ inv, int K8, int G8,
                               uint8_t *__restrict__ q, uint8_t *__restrict__ z) {
    const int N = h.N, KC = h.K / 64;
    const uint32_t *wp = reinterpret_cast<const uint32_t *>(h.wp);
    const size_t tq_ = q ? static_cast<size_t>(K8) * N : 0;
    const size_t tz = z ? static_cast<size_t>(G8) * N : 0;
    for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < tq_ + tz;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        if (idx < tq_) {
            const int n = static_cast<int>(idx % N);
            const int k = static_cast<int>(idx / N);
            q[idx] = static_cast<uint8_t>(16u * code_at(wp, KC, inv[k], n) + code_at(wp, KC, inv[K8 + k], n));
        } else {
            const size_t j = idx - tq_;
            const int n = static_cast<int>(j % N);
            const int g = static_cast<int>(j / N);
            const uint32_t zh = (h.zeros[static_cast<size_t>(g) * (N / 8) + n / 8] >> (4 * (n & 7))) & 0xFu;
            const uint32_t zl = (h.zeros[static_cast<size_t>(G8 + g) * (N / 8) + n / 8] >> (4 * (n & 7))) & 0xFu;
            z[j] = static_cast<uint8_t>(16u * zh + zl);
        }
    }
}

// temp_dq[k][n] = fp16(s * (q - (z + zero_offset))): the integer
// 16 (qh - zh) + (ql - zl - zero_offset) times s is exact in fp32 (11-bit
// scale, 9-bit integer), rounded once.  s comes from the low half's scales.
__global__ void dequant8_kernel(HandleView h, const int32_t *__restrict__ inv, int K8, uint16_t *__restrict__ out) {
    const int N = h.N, KC = h.K / 64, gpad = h.geff;
    const uint32_t *wp = reinterpret_cast<const uint32_t *>(h.wp);
    const size_t total = static_cast<size_t>(K8) * N;
    for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int n = static_cast<int>(idx % N);
        const int k = static_cast<int>(idx / N);
        const int jh = inv[k], jl = inv[K8 + k];
        const int gh = jh / gpad, gl = jl / gpad;              // groups of the two private rows
        const int qh = static_cast<int>(code_at(wp, KC, jh, n)), ql = static_cast<int>(code_at(wp, KC, jl, n));
        const int zh = static_cast<int>((h.zeros[static_cast<size_t>(gh) * (N / 8) + n / 8] >> (4 * (n & 7))) & 0xFu);
        const int zl = static_cast<int>((h.zeros[static_cast<size_t>(gl) * (N / 8) + n / 8] >> (4 * (n & 7))) & 0xFu);
        const uint32_t sp = h.s2[(static_cast<size_t>(gl) * (N / 16) + n / 16) * 8 + (n & 7)];
        const uint16_t sb = static_cast<uint16_t>((n & 8) ? (sp >> 16) : (sp & 0xFFFFu));
        const float s = __half2float(__ushort_as_half(sb));
        const int v = 16 * (qh - zh) + (ql - zl - h.zero_offset);
        out[idx] = __half_as_ushort(__float2half_rn(s * static_cast<float>(v)));
    }
}

int grid_for(size_t total) {
    const size_t want = (total + 255) / 256;
    const size_t cap = static_cast<size_t>(kSMs) * 16;
    return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_split8(const int32_t *qw8, const int32_t *qz8, const uint16_t *sc, int K, int N, int G,
                          int32_t *qw4, int32_t *qz4, uint16_t *sc4, cudaStream_t s) {
    split8_codes_kernel<<<grid_for(static_cast<size_t>(2 * K / 8) * N), 256, 0, s>>>(qw8, K, N, qw4);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    split8_meta_kernel<<<grid_for(static_cast<size_t>(2 * G) * (N / 8 + N)), 256, 0, s>>>(qz8, sc, G, N, qz4, sc4);
    return cudaGetLastError();
}

cudaError_t launch_unpack8(const HandleView &h, const int32_t *inv, int K8, int G8, uint8_t *q, uint8_t *z,
                           cudaStream_t s) {
    const size_t total = (q ? static_cast<size_t>(K8) * h.N : 0) + (z ? static_cast<size_t>(G8) * h.N : 0);
    unpack8_kernel<<<grid_for(total), 256, 0, s>>>(h, inv, K8, G8, q, z);
    return cudaGetLastError();
}

cudaError_t launch_dequant8(const HandleView &h, const int32_t *inv, int K8, uint16_t *temp_dq, cudaStream_t s) {
    dequant8_kernel<<<grid_for(static_cast<size_t>(K8) * h.N), 256, 0, s>>>(h, inv, K8, temp_dq);
    return cudaGetLastError();
}

}  // namespace q4
