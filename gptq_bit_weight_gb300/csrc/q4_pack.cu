// GPU packer: float weights plus the quantizer's scales and zero points into
// a GPTQ checkpoint (qweight, qzeros).  "Inference Backends", "Packing,
// conversion, and runtime initialization": packing takes the original
// linear layer's weights, scales, zeros and optional act-order index, and a
// GPU packing path accelerates the packing math; symmetric modules without
// zeros use 2^(bits-1).
//
// Code of w[k][n]: the nearest integer (ties to even) to the IEEE binary32
// quotient w / s, plus the effective zero point z, clamped to [0, 15]
// (0/0 gives z).  qweight [K/8][N]: eight codes along K per word, lowest
// nibble first.  qzeros [G][N/8]: eight stored zeros along N per word,
// lowest nibble first; stored = (z - zero_offset) mod 16 (GPTQ: z - 1,
// GPTQ_V2: z).
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdint>

#include "q4_internal.cuh"

namespace q4 {
namespace {

// One thread per checkpoint word: column n = blockIdx.x * blockDim.x + tid,
// word row kw = blockIdx.y (eight rows of w, coalesced across the warp).
__global__ void pack_qweight_kernel(const uint16_t *__restrict__ w, const uint16_t *__restrict__ scales,
                                    const int32_t *__restrict__ zeros, const int32_t *__restrict__ g_idx, int K,
                                    int N, int geff, int32_t *__restrict__ qweight) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    const int kw = blockIdx.y;
    if (n >= N) return;
    uint32_t word = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int k = 8 * kw + r;
        const int g = g_idx ? g_idx[k] : k / geff;
        const size_t gi = static_cast<size_t>(g) * N + n;
        const float wf = __half2float(__ushort_as_half(w[static_cast<size_t>(k) * N + n]));
        const float sf = __half2float(__ushort_as_half(scales[gi]));
        const float qf = rintf(__fdiv_rn(wf, sf));
        const int z = zeros ? zeros[gi] : 8;
        float v = (qf != qf) ? static_cast<float>(z) : qf + static_cast<float>(z);
        v = fminf(fmaxf(v, 0.0f), 15.0f);
        word |= static_cast<uint32_t>(v) << (4 * r);
    }
    qweight[static_cast<size_t>(kw) * N + n] = static_cast<int32_t>(word);
}

__global__ void pack_qzeros_kernel(const int32_t *__restrict__ zeros, int G, int N, int zero_offset,
                                   int32_t *__restrict__ qzeros) {
    const size_t total = static_cast<size_t>(G) * (N / 8);
    for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int g = static_cast<int>(idx / (N / 8)), c = static_cast<int>(idx % (N / 8));
        uint32_t word = 0;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int z = zeros ? zeros[static_cast<size_t>(g) * N + 8 * c + r] : 8;
            word |= (static_cast<uint32_t>(z - zero_offset) & 0xFu) << (4 * r);
        }
        qzeros[idx] = static_cast<int32_t>(word);
    }
}

}  // namespace

cudaError_t launch_pack(const uint16_t *w, const uint16_t *scales, const int32_t *zeros, const int32_t *g_idx,
                        int K, int N, int geff, int G, int zero_offset, int32_t *qweight, int32_t *qzeros,
                        cudaStream_t s) {
    const int threads = 256;
    const size_t nz = static_cast<size_t>(G) * (N / 8);
    const int bz = static_cast<int>(std::min<size_t>((nz + threads - 1) / threads, static_cast<size_t>(kSMs) * 32));
    pack_qweight_kernel<<<dim3((N + threads - 1) / threads, K / 8), threads, 0, s>>>(w, scales, zeros, g_idx, K, N,
                                                                                  geff, qweight);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    pack_qzeros_kernel<<<bz > 0 ? bz : 1, threads, 0, s>>>(zeros, G, N, zero_offset, qzeros);
    return cudaGetLastError();
}

}  // namespace q4
