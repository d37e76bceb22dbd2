// Internal definitions shared by the kernels and the C-ABI layer.
//
// Private execution layout of the packed weights ("Inference Backends",
// "Packing, conversion, and runtime initialization": runtime init may repack
// into a private layout).  Rows are taken in act-order permutation order P
// (identity when there is no act-order), so that every group is a contiguous
// run of rows and groups never need gathering at run time.
//
//   Wp word (nt, kc, lane, j), nt = n/16, kc = k/64, lane = 4*gq + tq:
//     column  n = 16*nt + gq + 8*(j & 1)
//     rows    j' = 64*kc + 32*(j >> 1) + 8*tq + r,  r = 0..7   (permuted order)
//     code of row r sits in nibble  pos(r) = (r >> 1) + 4*(r & 1),
//     i.e. nibbles 0..7 hold rows r = 0,2,4,6,1,3,5,7.
//   Word index ((nt*KC + kc)*32 + lane)*4 + j: each lane owns one aligned
//   16-byte vector per (nt, kc), and a warp reads one contiguous 512-byte run.
//
// Why this shape: (1) one 16-byte load gives a lane exactly the A-operand
// codes of two m16n8k16 MMAs for rows n = gq and gq+8 over 64 values of k;
// (2) one word holds eight consecutive k of one column, which is one 16-byte
// row segment of a K-major fp16 operand tile for the prefill tensor cores;
// (3) the nibble order lets the 0x6400 fp16 "magic number" (the exponent
// pattern of 1024) turn two codes into a half2 with one LOP3: codes of rows r
// and r+1 land in the low and high half of the same 32-bit register
// (Kim et al. 2022, "Who Says Elephants Can't Run", fast int4 -> fp16).
//
// Scales: S2 word (gr, nt, gq) = half2(scales[gr][16nt+gq], scales[gr][16nt+gq+8]).
// Zero points keep the checkpoint layout [G][N/8].
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace q4 {

constexpr int kSMs = 152;

__host__ __device__ inline int nib_pos(int r) { return (r >> 1) + 4 * (r & 1); }

__host__ __device__ inline size_t wp_index(int nt, int kc, int lane, int j, int KC) {
    return ((static_cast<size_t>(nt) * KC + kc) * 32 + lane) * 4 + j;
}

// ----------------------------------------------------------- device helpers
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
    return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Streaming 16-byte load of packed weights: read once per call, so it skips
// L1 allocation.
__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Four codes pairs of one packed word -> four half2 registers holding
// (q - z - 1) exactly for rows (0,1), (2,3), (4,5), (6,7) of the word.
//   nzlo = half2 splat of -(1025 + z)  : (1024 + q) - (1025 + z)
//   nzhi = half2 splat of -(65 + z)    : (1024 + 16 q) / 16 - (65 + z)
// Every intermediate is a small integer, so each fp16 step is exact.
__device__ __forceinline__ void unpack_qz(uint32_t w, uint32_t nzlo, uint32_t nzhi, uint32_t (&a)[4]) {
    const uint32_t kLo = 0x000F000Fu, kHi = 0x00F000F0u, kMagic = 0x64006400u;
    const uint32_t kOne = 0x3C003C00u, kSixteenth = 0x2C002C00u;
    uint32_t t0 = lop3_and_or(w, kLo, kMagic);
    uint32_t t1 = lop3_and_or(w, kHi, kMagic);
    uint32_t w8 = w >> 8;
    uint32_t t2 = lop3_and_or(w8, kLo, kMagic);
    uint32_t t3 = lop3_and_or(w8, kHi, kMagic);
    a[0] = hfma2(t0, kOne, nzlo);
    a[1] = hfma2(t1, kSixteenth, nzhi);
    a[2] = hfma2(t2, kOne, nzlo);
    a[3] = hfma2(t3, kSixteenth, nzhi);
}

// Code pairs of one packed word as raw fp16 pairs, no zero point: rows
// (0,1) and (4,5) as 1024 + q, rows (2,3) and (6,7) as 1024 + 16 q (nibble
// order of the packed layout: nibbles 0..7 hold rows 0,2,4,6,1,3,5,7).  One
// LOP3 per pair; the decode kernels remove 1024 + z + 1 (16 (64 + z + 1) for
// the second kind) per group from MMA-accumulated sums of x.
__device__ __forceinline__ void unpack_raw(uint32_t w, uint32_t (&t)[4]) {
    const uint32_t kLo = 0x000F000Fu, kHi = 0x00F000F0u, kMagic = 0x64006400u;
    const uint32_t w8 = w >> 8;
    t[0] = lop3_and_or(w, kLo, kMagic);
    t[1] = lop3_and_or(w, kHi, kMagic);
    t[2] = lop3_and_or(w8, kLo, kMagic);
    t[3] = lop3_and_or(w8, kHi, kMagic);
}

// Zero-point constants for unpack_qz from zm1 = (effective zero) - 1, i.e.
// the stored zero for GPTQ (v1) checkpoints and the stored zero minus one
// for GPTQ_V2 (zm1 = 0xFFFFFFFF for a stored 0: the 32-bit sums below then
// wrap to -1024 and -64 exactly).
__device__ __forceinline__ uint32_t neg_zlo(uint32_t z) { return (0xE401u + z) * 0x00010001u; }
__device__ __forceinline__ uint32_t neg_zhi(uint32_t z) { return (0xD410u + 16u * z) * 0x00010001u; }

// D += A . B on the tensor cores, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared-memory (CTA window) address of a generic pointer.
__device__ __forceinline__ uint32_t shared_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Asynchronous global -> shared copies (no register round trip).
__device__ __forceinline__ void cp_async_4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(shared_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_8(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(shared_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(shared_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most N of this thread's most recent copy groups are pending
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Hardware barrier over every thread of every CTA of the cluster, with
// release/acquire ordering of shared-memory writes across the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// fp32 load from the shared memory of CTA `rank` of this cluster, at the
// address that `local` has in this CTA's shared memory.
__device__ __forceinline__ float ld_dsmem_f32(uint32_t local, int rank) {
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// ------------------------------------------------------------ launchers
struct HandleView {
    int K, N, G, geff, groupsize;
    const uint4 *wp;        // private packed codes
    const uint32_t *s2;     // scale pairs
    const uint32_t *zeros;  // checkpoint-layout zero points
    const int32_t *perm;    // P (device) or nullptr
    const uint16_t *bias;   // device fp16 [N] or nullptr
    int *status;            // device status word
    int zero_offset;        // effective zero = stored + zero_offset (1: GPTQ, 0: GPTQ_V2)
    int zsplit;             // groups [0, zsplit) take zero offset 0 instead (the high-nibble
                            // half of an 8-bit layer), the rest zero_offset
    // output epilogue of this call (out_bf16 is the output mode):
    //   kOutF16  y = acc * rowscale[m] + bias, rounded once to fp16
    //   kOutBF16 the same rounded once to bf16 (rowscale NULL: 1)
    //   kOutF32  the fp32 sum acc itself, no bias and no row scale, stored as
    //            float (out points to M x N floats); the fp32-activation route
    //            combines two such rows per output row afterwards
    const float *rowscale;
    int out_bf16;
};
constexpr int kOutF16 = 0, kOutBF16 = 1, kOutF32 = 2;

// One output value / pair of the epilogue above.
__device__ __forceinline__ uint32_t out_bits(float v, bool bf16) {
    return bf16 ? static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)))
                : static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v)));
}
// Two values rounded to nearest-even in one packed conversion (lo in the low
// 16 bits): the same bits as two out_bits calls, one instruction instead of
// several on an epilogue's critical path.
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi, bool bf16) {
    if (bf16) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&v);
    }
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ uint16_t out_one(float acc, float rs, const uint16_t *bias, int n, bool bf16) {
    float v = acc * rs;
    if (bias) v += __half2float(__ushort_as_half(bias[n]));
    return static_cast<uint16_t>(out_bits(v, bf16));
}
// The same with the output type fixed at compile time (fp16: no row scale),
// for epilogues on a kernel's critical path.
template <bool BF16>
__device__ __forceinline__ uint32_t out_pair_t(float lo, float hi, float rs, const uint16_t *bias, int n) {
    if (BF16) {
        lo *= rs;
        hi *= rs;
    }
    if (bias) {
        lo += __half2float(__ushort_as_half(bias[n]));
        hi += __half2float(__ushort_as_half(bias[n + 1]));
    }
    return pack_pair(lo, hi, BF16);
}
__device__ __forceinline__ uint32_t out_pair(float lo, float hi, float rs, const uint16_t *bias, int n, bool bf16) {
    lo *= rs;
    hi *= rs;
    if (bias) {
        lo += __half2float(__ushort_as_half(bias[n]));
        hi += __half2float(__ushort_as_half(bias[n + 1]));
    }
    return pack_pair(lo, hi, bf16);
}

struct DecodeWork {
    float *ws;              // split-K partials
    size_t ws_floats;
    int *tickets;           // one per output tile, all zero between calls
    int n_tickets;
};

// repack / unpack / dequant / reorder (q4_repack.cu)
cudaError_t launch_repack_codes(const int32_t *qweight, const int32_t *perm, int K, int N,
                                uint32_t *wp, cudaStream_t s);
cudaError_t launch_repack_scales(const uint16_t *scales, int G, int N, uint32_t *s2, cudaStream_t s);
cudaError_t launch_debug_unpack(const HandleView &h, uint8_t *q, uint8_t *z, cudaStream_t s);
cudaError_t launch_dequant(const HandleView &h, uint16_t *temp_dq, cudaStream_t s);
// temp_state[m][j] = x[m][perm[j]] (0 where perm[j] = -1); x rows hold Kx
// values, temp_state rows K
// (early: launched so that the next grid, a register-streaming decode, may
// start now; only measured faster before that kernel)
cudaError_t launch_xreorder(const uint16_t *x, const int32_t *perm, int M, int Kx, int K,
                            uint16_t *temp_state, cudaStream_t s, bool early = false);
// bf16 activations: per row m, e_m with max|x[m]| * 2^-e_m in [2^14, 2^15),
// temp_state[m][j] = fp16(x[m][perm[j]] * 2^-e_m) (perm NULL: j; -1: 0) and
// rowscale[m] = 2^e_m
cudaError_t launch_xprep_bf16(const uint16_t *x, const int32_t *perm, int M, int Kx, int K, uint16_t *temp_state,
                              float *rowscale, cudaStream_t s, bool early = false);

// fp32 activations: per row m, e_m with max|x[m]| * 2^-e_m in [2^14, 2^15);
// v = x[m][perm[j]] * 2^-e_m (perm NULL: j; -1: 0), temp_state[m][j] =
// fp16(v) (hi) and temp_state[M + m][j] = fp16(v - hi) (lo, exact residual
// rounded once); rowscale[m] = 2^e_m
cudaError_t launch_xprep_f32(const float *x, const int32_t *perm, int M, int Kx, int K, uint16_t *temp_state,
                             float *rowscale, cudaStream_t s);
// y[m][n] = (part[m][n] + part[M + m][n]) * rowscale[m] + bias[n] in fp32
cudaError_t launch_combine_f32(const float *part, const float *rowscale, const uint16_t *bias, int M, int N, float *y,
                               cudaStream_t s);
// decode (q4_decode.cu)
struct DecodePlan {
    int mt;            // 8-row m tiles per CTA (1, 2 or 4)
    int zdim;          // row blocks
    int ctas_n;        // column tiles of 32
    int splits;        // K slices
    int slice_chunks;  // 64-row chunks per slice
    int cluster;       // 1: the slices of a column tile form a cluster and reduce through DSMEM
    size_t ws_floats;  // workspace needed (slices reduced through global memory)
    int n_tickets;
    int raw;           // 1: raw code pairs + sums of x (M <= 8); 0: exact (q - z - 1) pairs
    int sr;            // 1: weight ring in shared memory; 0: in registers
    int xr;            // shared ring: 1 x carried per chunk in the ring; 0 x slice staged once
    int one_wave;      // every CTA of the grid is resident at once
};
DecodePlan plan_decode(int M, int K, int N, int geff);
size_t decode_ws_floats_for(int M, int K, int N, int geff);
cudaError_t launch_decode(const HandleView &h, const DecodePlan &plan, const DecodeWork &w,
                          const uint16_t *x, int M, uint16_t *out, cudaStream_t s);

// decode on the tcgen05 tensor cores (q4_decode_tc.cu), M <= 16
struct DecodeTcPlan {
    int ok;            // 0: shape not supported by this kernel
    int splits;        // K slices (one cluster per column tile)
    int slice_kb;      // 64-row blocks per slice
    int tiles;         // 128-column tiles
    int zdim;          // 16-row blocks of x
};
DecodeTcPlan plan_decode_tc(int M, int K, int N, int geff, int sms);
bool decode_tc_supported(int M, int K, int N, int geff);
cudaError_t launch_decode_tc(const HandleView &h, const uint16_t *x, int M, uint16_t *out, cudaStream_t s);
// decode fed by a TMA ring, register dequantization, mma.sync (q4_decode_ring.cu), M <= 16
struct DecodeRingPlan {
    int ok;            // 0: shape not supported by this kernel
    int mt;            // 8-row m tiles (1 or 2)
    int splits;        // K slices (one cluster per column tile)
    int slice_kb;      // 64-row stages per slice
    int tiles;         // 128-column tiles
};
DecodeRingPlan plan_decode_ring(int M, int K, int N, int geff, int sms);
cudaError_t launch_decode_ring(const HandleView &h, const DecodeRingPlan &plan, const uint16_t *x, int M,
                               uint16_t *out, cudaStream_t s);
// stream-K decode with group slots (q4_decode_sk.cu), M <= 8
struct DecodeSkPlan {
    int ok;            // 0: shape not supported
    int mp;            // rows per group slot (M rounded up to a power of two)
    int ntw;           // n16 tiles per unit
    int T, KC;         // tiles of 16 ntw columns, 64-row chunks per tile
    long long U;       // units (tile, chunk)
    int workers;       // warps with work
    int ctas;
    int smax;          // most segments of one tile
    size_t ws_floats;  // fp32 partials [T][smax][8][16 ntw]
    int n_tickets;     // one per tile
};
DecodeSkPlan plan_decode_sk(int M, int K, int N, int sms);
cudaError_t launch_decode_sk(const HandleView &h, const DecodeSkPlan &p, float *ws, int *tickets, const uint16_t *x,
                             int M, uint16_t *out, cudaStream_t s);
// Dynamic shared-memory limit of kernel fn on device dev, set once per
// (fn, dev, bytes); bytes < 0 asks for the device's largest (q4_decode.cu)
cudaError_t dyn_smem_optin(const void *fn, int dev, int bytes, int *set);
// SMs of the current device (queried once)
int device_sm_count();
// programmatic dependent launch switch (GPTQ_Q4_PDL=0 turns it off)
bool pdl_enabled();
// fused prefill (q4_prefill.cu): tile shape, K split and split workspace
struct PrefillPlan {
    int bm, bn;        // tile
    int bk;            // rows of K per pipeline stage (64, or 128 for M <= 64)
    int sk;            // 1: stream-K over the tiles x k-blocks space (cooperative launch)
    int grid;          // stream-K: CTAs
    int pmax;          // stream-K: most pieces of one tile
    int fin0;          // stream-K, one range per CTA: piece 0's CTA finishes each cut tile
    size_t ws_floats;  // fp32 partial tiles when tiles are cut into pieces
    int n_tickets;     // one per tile when tiles are cut into pieces
};
// sms: SMs to plan for (0: this device's)
PrefillPlan plan_prefill(int M, int K, int N, int sms = 0);
cudaError_t launch_prefill(const HandleView &h, const PrefillPlan &p, float *ws, int *tickets, const uint16_t *x,
                           int M, uint16_t *out, cudaStream_t s);
// float weights + scales + zero points -> GPTQ checkpoint words (q4_pack.cu)
cudaError_t launch_pack(const uint16_t *w, const uint16_t *scales, const int32_t *zeros, const int32_t *g_idx,
                        int K, int N, int geff, int G, int zero_offset, int32_t *qweight, int32_t *qzeros,
                        cudaStream_t s);
// 8-bit layers as two 4-bit halves along K (q4_eight.cu): the split of the
// checkpoint, and the read-back of codes / dequantized weights through the
// inverse row map inv[k'] (private row of split row k')
cudaError_t launch_split8(const int32_t *qw8, const int32_t *qz8, const uint16_t *sc, int K, int N, int G,
                          int32_t *qw4, int32_t *qz4, uint16_t *sc4, cudaStream_t s);
cudaError_t launch_unpack8(const HandleView &h, const int32_t *inv, int K8, int G8, uint8_t *q, uint8_t *z,
                           cudaStream_t s);
cudaError_t launch_dequant8(const HandleView &h, const int32_t *inv, int K8, uint16_t *temp_dq, cudaStream_t s);
// test hook: a bounded mbarrier wait that runs out (q4_debug.cu)
cudaError_t launch_wait_probe(int *status, uint64_t limit_ns, cudaStream_t s);

}  // namespace q4
