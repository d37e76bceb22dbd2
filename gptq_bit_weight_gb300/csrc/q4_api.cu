// C ABI of the fused GPTQ W4A16 linear layer: argument checks, the handle
// (the Q4Matrix of "Implementation: Predibase Lorax GPTQ Exllama V1",
// "Description"), act-order permutation, path selection and status
// reporting.  Every failure returns a status with the specific reason kept
// for gptq_q4_last_error ("Inference Backends", "Hardware, dependency, and
// format requirements": validation errors keep their specific reason); there
// is no fallback route.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/gptq_q4.h"
#include "q4_internal.cuh"

namespace q4 {
cudaError_t launch_gemm_f16(const uint16_t *a, const uint16_t *b, const uint16_t *bias, int M, int K, int N,
                            uint16_t *out, int *status, cudaStream_t s, const float *rowscale = nullptr,
                            int out_bf16 = 0);
int prefill_default_min_m(int K, int N, int geff);
}  // namespace q4

#include "q4_handle.h"

namespace {

thread_local int t_status = GPTQ_Q4_OK;
thread_local char t_msg[512] = "";
std::atomic<uint64_t> g_launches{0};

int set_status(int code, const char *fmt, ...) {
    t_status = code;
    if (fmt) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
        va_end(ap);
    } else {
        t_msg[0] = '\0';
    }
    return code;
}

int ok() { return set_status(GPTQ_Q4_OK, nullptr); }

int cuda_fail(cudaError_t e, const char *what) {
    cudaGetLastError();   // clear a sticky-free error so the next call starts clean
    if (e == cudaErrorMemoryAllocation)
        return set_status(GPTQ_Q4_OUT_OF_MEMORY, "%s: %s", what, cudaGetErrorString(e));
    return set_status(GPTQ_Q4_CUDA_ERROR, "%s: %s", what, cudaGetErrorString(e));
}

#define Q4_CUDA(expr, what)                               \
    do {                                                  \
        cudaError_t e_ = (expr);                          \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device memory of the current device (or managed)?
int check_device_ptr(const void *p, int dev, const char *name) {
    cudaPointerAttributes attr{};
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "%s is not a CUDA pointer", name);
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "%s is not device memory", name);
    if (attr.type == cudaMemoryTypeDevice && attr.device != dev)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "%s lives on device %d, current device is %d", name,
                          attr.device, dev);
    return GPTQ_Q4_OK;
}

int check_device_sm103(int *dev_out) {
    int dev = 0;
    Q4_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    int major = 0, minor = 0;
    Q4_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "cudaDeviceGetAttribute");
    Q4_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
        return set_status(GPTQ_Q4_UNSUPPORTED,
                          "kernels are built for sm_103a only; device %d has compute capability %d.%d", dev,
                          major, minor);
    *dev_out = dev;
    return GPTQ_Q4_OK;
}

template <typename T>
int dev_alloc(T **p, size_t count, gptq_q4_s *h, const char *what) {
    if (count == 0) {
        *p = nullptr;
        return GPTQ_Q4_OK;
    }
    void *v = nullptr;
    cudaError_t e = cudaMalloc(&v, count * sizeof(T));
    if (e != cudaSuccess) return cuda_fail(e, what);
    *p = static_cast<T *>(v);
    if (h) h->device_bytes += count * sizeof(T);
    return GPTQ_Q4_OK;
}

void release(gptq_q4_s *h) {
    if (!h) return;
    int cur = -1;
    cudaGetDevice(&cur);
    if (h->device >= 0) cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    cudaFree(h->wp);
    cudaFree(h->s2);
    cudaFree(h->zeros);
    cudaFree(h->perm);
    cudaFree(h->inv8);
    cudaFree(h->bias);
    cudaFree(h->status);
    cudaFree(h->ws);
    cudaFree(h->tickets);
    cudaFree(h->temp_state);
    cudaFree(h->rowscale);
    cudaFree(h->part);
    if (cur >= 0) cudaSetDevice(cur);
    delete h;
}

q4::HandleView view(const gptq_q4_s *h) {
    q4::HandleView v{};
    v.K = h->K;
    v.N = h->N;
    v.G = h->G;
    v.geff = h->geff;
    v.groupsize = h->groupsize;
    v.wp = reinterpret_cast<const uint4 *>(h->wp);
    v.s2 = h->s2;
    v.zeros = h->zeros;
    v.zero_offset = h->zero_offset;
    v.zsplit = h->zsplit;
    v.perm = h->act_order ? h->perm : nullptr;
    v.bias = h->bias;
    v.status = h->status;
    return v;
}

int check_handle(gptq_q4_handle h) {
    if (!h) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "handle is NULL");
    int dev = -1;
    Q4_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev != h->device)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "handle was made on device %d, current device is %d",
                          h->device, dev);
    return GPTQ_Q4_OK;
}

// Grow the split-K workspace / tickets (stream-ordered when a stream is given).
int ensure_decode_work(gptq_q4_s *h, size_t ws_floats, int n_tickets, cudaStream_t s, bool sync_alloc) {
    if (ws_floats > h->ws_floats) {
        if (h->ws) {
            if (sync_alloc) cudaFree(h->ws);
            else Q4_CUDA(cudaFreeAsync(h->ws, s), "cudaFreeAsync(workspace)");
            h->device_bytes -= h->ws_floats * sizeof(float);
            h->ws = nullptr;
            h->ws_floats = 0;
        }
        void *v = nullptr;
        cudaError_t e = sync_alloc ? cudaMalloc(&v, ws_floats * sizeof(float))
                                   : cudaMallocAsync(&v, ws_floats * sizeof(float), s);
        if (e != cudaSuccess) return cuda_fail(e, "allocating split-K workspace");
        h->ws = static_cast<float *>(v);
        h->ws_floats = ws_floats;
        h->device_bytes += ws_floats * sizeof(float);
    }
    if (n_tickets > h->n_tickets) {
        if (h->tickets) {
            if (sync_alloc) cudaFree(h->tickets);
            else Q4_CUDA(cudaFreeAsync(h->tickets, s), "cudaFreeAsync(tickets)");
            h->device_bytes -= static_cast<size_t>(h->n_tickets) * sizeof(int);
            h->tickets = nullptr;
            h->n_tickets = 0;
        }
        void *v = nullptr;
        cudaError_t e = sync_alloc ? cudaMalloc(&v, n_tickets * sizeof(int))
                                   : cudaMallocAsync(&v, n_tickets * sizeof(int), s);
        if (e != cudaSuccess) return cuda_fail(e, "allocating split-K tickets");
        h->tickets = static_cast<int *>(v);
        h->n_tickets = n_tickets;
        h->device_bytes += static_cast<size_t>(n_tickets) * sizeof(int);
        if (sync_alloc) Q4_CUDA(cudaMemset(h->tickets, 0, n_tickets * sizeof(int)), "cudaMemset(tickets)");
        else Q4_CUDA(cudaMemsetAsync(h->tickets, 0, n_tickets * sizeof(int), s), "cudaMemsetAsync(tickets)");
    }
    return GPTQ_Q4_OK;
}

int ensure_temp_state(gptq_q4_s *h, int M, cudaStream_t s, bool sync_alloc) {
    const size_t need = static_cast<size_t>(M) * h->K;
    if ((h->act_bf16 || h->act_f32) && static_cast<size_t>(M) > h->rowscale_elems) {
        if (h->rowscale) {
            if (sync_alloc) cudaFree(h->rowscale);
            else Q4_CUDA(cudaFreeAsync(h->rowscale, s), "cudaFreeAsync(rowscale)");
            h->device_bytes -= h->rowscale_elems * sizeof(float);
            h->rowscale = nullptr;
            h->rowscale_elems = 0;
        }
        void *v = nullptr;
        cudaError_t e = sync_alloc ? cudaMalloc(&v, M * sizeof(float)) : cudaMallocAsync(&v, M * sizeof(float), s);
        if (e != cudaSuccess) return cuda_fail(e, "allocating row scales");
        h->rowscale = static_cast<float *>(v);
        h->rowscale_elems = static_cast<size_t>(M);
        h->device_bytes += M * sizeof(float);
    }
    if (!(h->act_order || h->act_bf16 || h->act_f32) || need <= h->temp_state_elems) return GPTQ_Q4_OK;
    if (h->temp_state) {
        if (sync_alloc) cudaFree(h->temp_state);
        else Q4_CUDA(cudaFreeAsync(h->temp_state, s), "cudaFreeAsync(temp_state)");
        h->device_bytes -= h->temp_state_elems * 2;
        h->temp_state = nullptr;
        h->temp_state_elems = 0;
    }
    void *v = nullptr;
    cudaError_t e = sync_alloc ? cudaMalloc(&v, need * 2) : cudaMallocAsync(&v, need * 2, s);
    if (e != cudaSuccess) return cuda_fail(e, "allocating temp_state");
    h->temp_state = static_cast<uint16_t *>(v);
    h->temp_state_elems = need;
    h->device_bytes += need * 2;
    return GPTQ_Q4_OK;
}

// fp32 activations: room for the raw fp32 sums of 2M rows
int ensure_part(gptq_q4_s *h, size_t elems, cudaStream_t s, bool sync_alloc) {
    if (elems <= h->part_elems) return GPTQ_Q4_OK;
    if (h->part) {
        if (sync_alloc) cudaFree(h->part);
        else Q4_CUDA(cudaFreeAsync(h->part, s), "cudaFreeAsync(partial rows)");
        h->device_bytes -= h->part_elems * sizeof(float);
        h->part = nullptr;
        h->part_elems = 0;
    }
    void *v = nullptr;
    cudaError_t e = sync_alloc ? cudaMalloc(&v, elems * sizeof(float)) : cudaMallocAsync(&v, elems * sizeof(float), s);
    if (e != cudaSuccess) return cuda_fail(e, "allocating the fp32 partial rows");
    h->part = static_cast<float *>(v);
    h->part_elems = elems;
    h->device_bytes += elems * sizeof(float);
    return GPTQ_Q4_OK;
}

int decode_max_ws_rows() { return 16; }

}  // namespace

extern "C" {

gptq_q4_handle gptq_q4_make(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                            const int32_t *g_idx, int K, int N, int groupsize) {
    if (!qweight || !qzeros || !scales) {
        set_status(GPTQ_Q4_INVALID_ARGUMENT, "qweight, qzeros and scales must not be NULL");
        return nullptr;
    }
    if (K <= 0 || N <= 0 || K % 8 || N % 8) {
        set_status(GPTQ_Q4_INVALID_ARGUMENT, "K=%d and N=%d must be positive multiples of 8 (eight codes per word)",
                   K, N);
        return nullptr;
    }
    if (!(groupsize == -1 || (groupsize > 0 && K % groupsize == 0))) {
        set_status(GPTQ_Q4_INVALID_ARGUMENT, "groupsize=%d must be -1 or a positive divisor of K=%d", groupsize, K);
        return nullptr;
    }
    const int geff = groupsize == -1 ? K : groupsize;
    const int G = K / geff;
    int dev = -1;
    if (check_device_sm103(&dev) != GPTQ_Q4_OK) return nullptr;
    if (check_device_ptr(qweight, dev, "qweight") || check_device_ptr(qzeros, dev, "qzeros") ||
        check_device_ptr(scales, dev, "scales") || (g_idx && check_device_ptr(g_idx, dev, "g_idx")))
        return nullptr;
    if (!aligned(qweight, 4) || !aligned(qzeros, 4) || !aligned(scales, 2) || (g_idx && !aligned(g_idx, 4))) {
        set_status(GPTQ_Q4_INVALID_ARGUMENT, "misaligned input pointer");
        return nullptr;
    }

    // act-order: one stable argsort of g_idx (a counting sort by group keeps
    // the original order inside each group), identity -> no act-order.
    // Groups of unequal size, or of a size that is not whole 32-row blocks,
    // are each padded to gpad rows (the largest group rounded up to 32-row
    // blocks): padding rows carry code 0 and perm = -1, and the x gather
    // writes 0 there, so they add nothing.
    std::vector<int32_t> perm;
    bool act = false;
    int gpad = geff;           // rows per group in the private layout
    int Kp = K;                // rows of the private layout
    if (g_idx || geff % 32) {
        std::vector<int32_t> gi(K);
        if (g_idx) {
            cudaError_t e = cudaMemcpy(gi.data(), g_idx, sizeof(int32_t) * K, cudaMemcpyDeviceToHost);
            if (e != cudaSuccess) {
                cuda_fail(e, "copying g_idx to the host");
                return nullptr;
            }
        } else {
            for (int k = 0; k < K; ++k) gi[k] = k / geff;
        }
        std::vector<int> count(G + 1, 0);
        for (int k = 0; k < K; ++k) {
            if (gi[k] < 0 || gi[k] >= G) {
                set_status(GPTQ_Q4_INVALID_ARGUMENT, "g_idx[%d]=%d is outside [0, %d)", k, gi[k], G);
                return nullptr;
            }
            ++count[gi[k] + 1];
        }
        bool uniform = true;
        int largest = 0;
        for (int g = 0; g < G; ++g) {
            uniform = uniform && count[g + 1] == geff;
            largest = std::max(largest, count[g + 1]);
        }
        if (!uniform || geff % 32) {
            gpad = (largest + 31) / 32 * 32;
            if ((static_cast<long long>(G) * gpad) % 64) gpad += 32;     // whole 64-row chunks
            if (static_cast<long long>(G) * gpad > 4LL * K) {
                set_status(GPTQ_Q4_UNSUPPORTED,
                           "groups of unequal size (largest %d rows of %d) padded to %d rows each would make the "
                           "packed layout more than 4x the checkpoint",
                           largest, K, gpad);
                return nullptr;
            }
            Kp = G * gpad;
        }
        // first padded row of each group, then the rows of each group in order
        std::vector<int> next(G);
        for (int g = 0; g < G; ++g) next[g] = g * gpad;
        perm.assign(Kp, -1);
        for (int k = 0; k < K; ++k) perm[next[gi[k]]++] = k;
        act = Kp != K;
        for (int j = 0; j < K && !act; ++j) act = perm[j] != j;
    }
    if (K % 64 || N % 64 || gpad % 32) {
        set_status(GPTQ_Q4_UNSUPPORTED,
                   "the GPU kernels need K %% 64 == 0, N %% 64 == 0 and a group size that is a multiple of 32 "
                   "(K=%d N=%d group=%d)",
                   K, N, gpad);
        return nullptr;
    }

    gptq_q4_s *h = new (std::nothrow) gptq_q4_s();
    if (!h) {
        set_status(GPTQ_Q4_OUT_OF_MEMORY, "host allocation of the handle failed");
        return nullptr;
    }
    h->device = dev;
    h->K = Kp;
    h->Kx = K;
    h->N = N;
    h->groupsize = groupsize;
    h->geff = gpad;
    h->G = G;
    h->act_order = act ? 1 : 0;
    h->prefill_min_m = q4::prefill_default_min_m(Kp, N, gpad);

    cudaStream_t s = nullptr;
    auto fail = [&](int) -> gptq_q4_handle {
        int code = t_status;
        char msg[512];
        std::memcpy(msg, t_msg, sizeof(msg));
        if (s) cudaStreamDestroy(s);
        release(h);
        t_status = code;
        std::memcpy(t_msg, msg, sizeof(msg));
        return nullptr;
    };
    const size_t words = static_cast<size_t>(Kp / 8) * N;
    if (dev_alloc(&h->wp, words, h, "allocating packed weights") ||
        dev_alloc(&h->s2, static_cast<size_t>(G) * (N / 16) * 8, h, "allocating scales") ||
        dev_alloc(&h->zeros, static_cast<size_t>(G) * (N / 8), h, "allocating zeros") ||
        dev_alloc(&h->status, 1, h, "allocating status word") ||
        (act && dev_alloc(&h->perm, static_cast<size_t>(Kp), h, "allocating permutation")))
        return fail(0);
    cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return fail(cuda_fail(e, "cudaStreamCreate"));
    if ((e = cudaMemsetAsync(h->status, 0, sizeof(int), s)) != cudaSuccess) return fail(cuda_fail(e, "memset"));
    if (act && (e = cudaMemcpyAsync(h->perm, perm.data(), sizeof(int32_t) * Kp, cudaMemcpyHostToDevice, s)) !=
                   cudaSuccess)
        return fail(cuda_fail(e, "copying the permutation"));
    if ((e = cudaMemcpyAsync(h->zeros, qzeros, sizeof(uint32_t) * G * (N / 8), cudaMemcpyDeviceToDevice, s)) !=
        cudaSuccess)
        return fail(cuda_fail(e, "copying qzeros"));
    if ((e = q4::launch_repack_codes(qweight, act ? h->perm : nullptr, Kp, N, h->wp, s)) != cudaSuccess)
        return fail(cuda_fail(e, "repack launch"));
    if ((e = q4::launch_repack_scales(scales, G, N, h->s2, s)) != cudaSuccess)
        return fail(cuda_fail(e, "scale repack launch"));
    g_launches += 2;
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail(cuda_fail(e, "repack"));
    cudaStreamDestroy(s);
    s = nullptr;
    const q4::DecodePlan p = q4::plan_decode(decode_max_ws_rows(), Kp, N, gpad);
    const q4::DecodeSkPlan sp = q4::plan_decode_sk(1, Kp, N, q4::device_sm_count());
    if (ensure_decode_work(h, std::max(p.ws_floats, sp.ws_floats), std::max(p.n_tickets, sp.n_tickets), nullptr,
                           true))
        return fail(0);
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return fail(cuda_fail(e, "make"));
    ok();
    return h;
}

gptq_q4_handle gptq_q4_make8(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                             const int32_t *g_idx, int K, int N, int groupsize) {
    if (!qweight || !qzeros || !scales) {
        set_status(GPTQ_Q4_INVALID_ARGUMENT, "qweight, qzeros and scales must not be NULL");
        return nullptr;
    }
    if (K <= 0 || N <= 0 || K % 8 || N % 8) {
        set_status(GPTQ_Q4_INVALID_ARGUMENT, "K=%d and N=%d must be positive multiples of 8", K, N);
        return nullptr;
    }
    if (!(groupsize == -1 || (groupsize > 0 && K % groupsize == 0))) {
        set_status(GPTQ_Q4_INVALID_ARGUMENT, "groupsize=%d must be -1 or a positive divisor of K=%d", groupsize, K);
        return nullptr;
    }
    const int geff = groupsize == -1 ? K : groupsize;
    const int G = K / geff;
    if (K % 64 || N % 64) {   // the split layer has 2K rows, but x and the unfused route keep K
        set_status(GPTQ_Q4_UNSUPPORTED, "the GPU kernels need K %% 64 == 0 and N %% 64 == 0 (K=%d N=%d)", K, N);
        return nullptr;
    }
    int dev = -1;
    if (check_device_sm103(&dev) != GPTQ_Q4_OK) return nullptr;
    if (check_device_ptr(qweight, dev, "qweight") || check_device_ptr(qzeros, dev, "qzeros") ||
        check_device_ptr(scales, dev, "scales") || (g_idx && check_device_ptr(g_idx, dev, "g_idx")))
        return nullptr;
    if (!aligned(qweight, 4) || !aligned(qzeros, 4) || !aligned(scales, 2) || (g_idx && !aligned(g_idx, 4))) {
        set_status(GPTQ_Q4_INVALID_ARGUMENT, "misaligned input pointer");
        return nullptr;
    }
    // the groups of the split layer: row k -> g_idx[k], row K + k -> G + g_idx[k]
    std::vector<int32_t> gi(2 * static_cast<size_t>(K));
    if (g_idx) {
        cudaError_t e = cudaMemcpy(gi.data(), g_idx, sizeof(int32_t) * K, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) {
            cuda_fail(e, "copying g_idx to the host");
            return nullptr;
        }
        for (int k = 0; k < K; ++k)
            if (gi[k] < 0 || gi[k] >= G) {
                set_status(GPTQ_Q4_INVALID_ARGUMENT, "g_idx[%d]=%d is outside [0, %d)", k, gi[k], G);
                return nullptr;
            }
    } else {
        for (int k = 0; k < K; ++k) gi[k] = k / geff;
    }
    for (int k = 0; k < K; ++k) gi[K + k] = G + gi[k];

    // split checkpoint (temporary), then the ordinary 4-bit handle over 2K rows
    int32_t *qw4 = nullptr, *qz4 = nullptr, *gi4 = nullptr;
    uint16_t *sc4 = nullptr;
    auto cleanup = [&]() {
        cudaFree(qw4);
        cudaFree(qz4);
        cudaFree(sc4);
        cudaFree(gi4);
    };
    if (dev_alloc(&qw4, static_cast<size_t>(2 * K / 8) * N, nullptr, "allocating the split codes") ||
        dev_alloc(&qz4, static_cast<size_t>(2 * G) * (N / 8), nullptr, "allocating the split zeros") ||
        dev_alloc(&sc4, static_cast<size_t>(2 * G) * N, nullptr, "allocating the split scales") ||
        dev_alloc(&gi4, static_cast<size_t>(2 * K), nullptr, "allocating the split g_idx")) {
        cleanup();
        return nullptr;
    }
    cudaError_t e = cudaMemcpy(gi4, gi.data(), sizeof(int32_t) * 2 * K, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = q4::launch_split8(qweight, qzeros, scales, K, N, G, qw4, qz4, sc4, nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cuda_fail(e, "splitting the 8-bit checkpoint");
        cleanup();
        return nullptr;
    }
    g_launches += 2;
    gptq_q4_s *h = gptq_q4_make(qw4, qz4, sc4, gi4, 2 * K, N, geff);
    cleanup();
    if (!h) return nullptr;

    // Private row order of the 2K split rows (the identity when make found no
    // act-order), its inverse for the read-back kernels, and the column of x
    // each private row reads: both halves read column k.
    const int Kp = h->K;
    std::vector<int32_t> perm(Kp);
    if (h->act_order) e = cudaMemcpy(perm.data(), h->perm, sizeof(int32_t) * Kp, cudaMemcpyDeviceToHost);
    else
        for (int j = 0; j < Kp; ++j) perm[j] = j;
    std::vector<int32_t> inv(2 * static_cast<size_t>(K), -1), xcol(Kp);
    for (int j = 0; j < Kp; ++j) {
        if (perm[j] >= 0) inv[perm[j]] = j;
        xcol[j] = perm[j] < 0 ? -1 : perm[j] % K;
    }
    if (e == cudaSuccess && !h->act_order &&
        dev_alloc(&h->perm, static_cast<size_t>(Kp), h, "allocating the activation gather") != GPTQ_Q4_OK) {
        release(h);
        return nullptr;
    }
    if (e == cudaSuccess && dev_alloc(&h->inv8, static_cast<size_t>(2 * K), h, "allocating the row map") != GPTQ_Q4_OK) {
        release(h);
        return nullptr;
    }
    if (e == cudaSuccess) e = cudaMemcpy(h->perm, xcol.data(), sizeof(int32_t) * Kp, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(h->inv8, inv.data(), sizeof(int32_t) * 2 * K, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cuda_fail(e, "building the 8-bit row maps");
        release(h);
        return nullptr;
    }
    h->act_order = 1;
    h->Kx = K;
    h->groupsize = groupsize;
    h->bits = 8;
    h->zsplit = G;
    ok();
    return h;
}

gptq_q4_handle gptq_q4_make_fused(int parts, const int32_t *const *qweight, const int32_t *const *qzeros,
                                  const uint16_t *const *scales, const int32_t *g_idx, int K, const int *N,
                                  int groupsize) {
    if (parts < 1 || parts > GPTQ_Q4_MAX_FUSED_PARTS || !qweight || !qzeros || !scales || !N) {
        set_status(GPTQ_Q4_INVALID_ARGUMENT, "parts=%d must be in [1, %d] with non-NULL arrays", parts,
                   GPTQ_Q4_MAX_FUSED_PARTS);
        return nullptr;
    }
    if (K <= 0 || K % 8 || !(groupsize == -1 || (groupsize > 0 && K % groupsize == 0))) {
        set_status(GPTQ_Q4_INVALID_ARGUMENT, "K=%d must be a positive multiple of 8 and groupsize=%d -1 or a divisor",
                   K, groupsize);
        return nullptr;
    }
    long long ntot = 0;
    for (int i = 0; i < parts; ++i) {
        if (!qweight[i] || !qzeros[i] || !scales[i] || N[i] <= 0 || N[i] % 8) {
            set_status(GPTQ_Q4_INVALID_ARGUMENT, "part %d: NULL tensor or N=%d not a positive multiple of 8", i,
                       N[i]);
            return nullptr;
        }
        ntot += N[i];
    }
    if (ntot > INT_MAX / 8) {
        set_status(GPTQ_Q4_INVALID_ARGUMENT, "total N=%lld too large", ntot);
        return nullptr;
    }
    const int Nt = static_cast<int>(ntot);
    const int G = groupsize == -1 ? 1 : K / groupsize;
    int dev = -1;
    if (check_device_sm103(&dev) != GPTQ_Q4_OK) return nullptr;
    for (int i = 0; i < parts; ++i)
        if (check_device_ptr(qweight[i], dev, "qweight part") || check_device_ptr(qzeros[i], dev, "qzeros part") ||
            check_device_ptr(scales[i], dev, "scales part"))
            return nullptr;
    // Concatenate the parts along N into temporaries in the checkpoint layout,
    // then make one handle from them (make copies what it keeps).
    int32_t *qw = nullptr, *qz = nullptr;
    uint16_t *sc = nullptr;
    gptq_q4_handle h = nullptr;
    if (dev_alloc(&qw, static_cast<size_t>(K / 8) * Nt, nullptr, "fused qweight") == GPTQ_Q4_OK &&
        dev_alloc(&qz, static_cast<size_t>(G) * (Nt / 8), nullptr, "fused qzeros") == GPTQ_Q4_OK &&
        dev_alloc(&sc, static_cast<size_t>(G) * Nt, nullptr, "fused scales") == GPTQ_Q4_OK) {
        bool copied = true;
        size_t off = 0;
        for (int i = 0; i < parts && copied; ++i) {
            const size_t n = static_cast<size_t>(N[i]);
            cudaError_t e = cudaMemcpy2D(qw + off, Nt * 4, qweight[i], n * 4, n * 4, K / 8, cudaMemcpyDeviceToDevice);
            if (e == cudaSuccess)
                e = cudaMemcpy2D(qz + off / 8, (Nt / 8) * 4, qzeros[i], (n / 8) * 4, (n / 8) * 4, G,
                                 cudaMemcpyDeviceToDevice);
            if (e == cudaSuccess)
                e = cudaMemcpy2D(sc + off, Nt * 2, scales[i], n * 2, n * 2, G, cudaMemcpyDeviceToDevice);
            if (e != cudaSuccess) {
                cuda_fail(e, "concatenating the fused parts");
                copied = false;
            }
            off += n;
        }
        if (copied) h = gptq_q4_make(qw, qz, sc, g_idx, K, Nt, groupsize);
    }
    const int status = t_status;
    char msg[sizeof(t_msg)];
    memcpy(msg, t_msg, sizeof(t_msg));
    cudaDeviceSynchronize();
    cudaFree(qw);
    cudaFree(qz);
    cudaFree(sc);
    t_status = status;                                 // keep make's status and message
    memcpy(t_msg, msg, sizeof(t_msg));
    return h;
}

int gptq_q4_set_bias(gptq_q4_handle h, const uint16_t *bias) {
    if (int r = check_handle(h)) return r;
    if (!bias) {
        cudaDeviceSynchronize();
        cudaFree(h->bias);
        if (h->bias) h->device_bytes -= static_cast<size_t>(h->N) * 2;
        h->bias = nullptr;
        return ok();
    }
    if (int r = check_device_ptr(bias, h->device, "bias")) return r;
    if (!aligned(bias, 2)) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "misaligned bias");
    if (!h->bias && dev_alloc(&h->bias, static_cast<size_t>(h->N), h, "allocating bias")) return t_status;
    Q4_CUDA(cudaMemcpy(h->bias, bias, static_cast<size_t>(h->N) * 2, cudaMemcpyDeviceToDevice), "copying bias");
    Q4_CUDA(cudaDeviceSynchronize(), "set_bias");
    return ok();
}

int gptq_q4_reserve(gptq_q4_handle h, int max_m) {
    if (int r = check_handle(h)) return r;
    if (max_m < 0) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "max_m=%d < 0", max_m);
    Q4_CUDA(cudaDeviceSynchronize(), "reserve");
    size_t ws = 0;
    int nt = 0;
    for (int m = 1; m <= std::min(max_m, 64); ++m) {
        const q4::DecodePlan p = q4::plan_decode(m, h->K, h->N, h->geff);
        ws = std::max(ws, p.ws_floats);
        nt = std::max(nt, p.n_tickets);
    }
    if (max_m >= 1) {       // the stream-K decode: the same workspace at every M <= 8
        const q4::DecodeSkPlan sp = q4::plan_decode_sk(1, h->K, h->N, q4::device_sm_count());
        ws = std::max(ws, sp.ws_floats);
        nt = std::max(nt, sp.n_tickets);
    }
    if (max_m > 64) {
        const q4::DecodePlan p = q4::plan_decode(max_m, h->K, h->N, h->geff);
        ws = std::max(ws, p.ws_floats);
        nt = std::max(nt, p.n_tickets);
    }
    if (int r = ensure_decode_work(h, ws, nt, nullptr, true)) return r;
    if (int r = ensure_temp_state(h, max_m, nullptr, true)) return r;
    Q4_CUDA(cudaDeviceSynchronize(), "reserve");
    return ok();
}

// The kernels a call can run.
enum class Kern { Prefill = 0, Reg = 1, Stream = 2, Ring = 3, Tc = 4 };

// Which kernel run_path launches for `path` on M rows (host logic only):
// the requested kernel where its planner accepts the shape, else the
// register-streaming decode.  tc_ok: fp16 output and GPTQ zero points, the
// tcgen05 decode's only case.  The plan of the chosen stream-K or TMA-ring
// kernel is returned through sk / rp.
static Kern kernel_for(int path, int M, int K, int N, int geff, bool tc_ok, bool small_layer, int sms,
                       q4::DecodeSkPlan *sk, q4::DecodeRingPlan *rp) {
    if (path == GPTQ_Q4_PATH_PREFILL) return Kern::Prefill;
    if (path == GPTQ_Q4_PATH_DECODE_TC && tc_ok && q4::decode_tc_supported(M, K, N, geff)) return Kern::Tc;
    if (path == GPTQ_Q4_PATH_DECODE_STREAM && M <= 8) {
        *sk = q4::plan_decode_sk(M, K, N, sms);
        if (sk->ok) return Kern::Stream;
    }
    if ((path == GPTQ_Q4_PATH_DECODE && !small_layer) || path == GPTQ_Q4_PATH_DECODE_RING) {
        *rp = q4::plan_decode_ring(M, K, N, geff, sms);
        if (rp->ok) return Kern::Ring;
    }
    return Kern::Reg;
}

// One of the kernels on prepared fp16 rows xin [M][K] (K the private
// layout's rows), epilogue as v says.
static int run_path(gptq_q4_handle h, const q4::HandleView &v, const uint16_t *xin, int M, uint16_t *out,
                    cudaStream_t stream, int path, bool small_layer) {
    q4::DecodeSkPlan sp{};
    q4::DecodeRingPlan rp{};
    const bool tc_ok = h->zsplit == 0 && v.out_bf16 == q4::kOutF16;
    switch (kernel_for(path, M, h->K, h->N, h->geff, tc_ok, small_layer, q4::device_sm_count(), &sp, &rp)) {
        case Kern::Prefill: {
            const q4::PrefillPlan pp = q4::plan_prefill(M, h->K, h->N);
            if (int r = ensure_decode_work(h, pp.ws_floats, pp.n_tickets, stream, false)) return r;
            Q4_CUDA(q4::launch_prefill(v, pp, h->ws, h->tickets, xin, M, out, stream), "prefill launch");
            break;
        }
        case Kern::Tc:
            Q4_CUDA(q4::launch_decode_tc(v, xin, M, out, stream), "decode launch");
            break;
        case Kern::Stream:
            if (int r = ensure_decode_work(h, sp.ws_floats, sp.n_tickets, stream, false)) return r;
            Q4_CUDA(q4::launch_decode_sk(v, sp, h->ws, h->tickets, xin, M, out, stream), "decode launch");
            break;
        case Kern::Ring:
            Q4_CUDA(q4::launch_decode_ring(v, rp, xin, M, out, stream), "decode launch");
            break;
        case Kern::Reg: {
            const q4::DecodePlan p = q4::plan_decode(M, h->K, h->N, h->geff);
            if (int r = ensure_decode_work(h, p.ws_floats, p.n_tickets, stream, false)) return r;
            q4::DecodeWork w{h->ws, h->ws_floats, h->tickets, h->n_tickets};
            Q4_CUDA(q4::launch_decode(v, p, w, xin, M, out, stream), "decode launch");
            break;
        }
    }
    ++g_launches;
    return ok();
}

// GPTQ_Q4_PATH_DECODE: where the stream-K kernel is ahead, measured on GB300
// over the Llama-7B and Llama-70B projection layers at M = 1, 2, 4, 8
// (CUDA-graph replays over more weights than L2): only on a large tall layer
// whose 32-column tiles cannot fill the GPU (K >= 2 N, fewer than two tiles
// per SM, 100 Mi weights or more: 28672 x 8192; on 11008 x 4096 the
// register-streaming kernel is ahead, M = 1 9.4 against 12.7 us), where the
// other kernels leave SMs short of warps: at one row with groups of at most
// 128 rows, at two rows with 32-row groups, and at 3-8 rows with groups of
// 128 rows or more (28672 x 8192 g128 M = 8: 42.1 against 45.8 us).
static bool prefer_stream(int K, int N, int geff, int M, int sms) {
    const long long tiles = N / 32;
    const bool tall = K >= 2LL * N && tiles < 2LL * sms && static_cast<size_t>(K) * N >= (size_t{100} << 20);
    if (!tall || M > 8) return false;
    if (M == 1) return geff <= 128;
    if (M == 2) return geff <= 32;
    return geff >= 128;
}

// Which decode kernel: measured on GB300 (CUDA-graph replays over more
// weights than L2), the register-streaming kernel (with its shared weight
// ring at M <= 8) is ahead at M <= 4 on every layer, at M <= 8 on layers
// below 64 Mi weights or with groups of at most 64 rows (8192 x 28672 g32
// M = 8: 45.0 against 89.3 us) and at any M on layers below 24 Mi weights;
// the TMA-ring kernel is ahead everywhere else it applies.
static bool small_layer_for(int K, int N, int geff, int M) {
    const size_t weights = static_cast<size_t>(K) * N;
    return M <= 4 || weights < (size_t{24} << 20) || (M <= 8 && (weights < (size_t{64} << 20) || geff <= 64));
}

static int run_matmul(gptq_q4_handle h, const void *x, int M, void *out, cudaStream_t stream, int path) {
    // fp32 activations: the kernels see 2M fp16 rows (each row's hi and lo
    // parts) and write raw fp32 sums; a last pass adds each row's two parts
    const int Mk = h->act_f32 ? 2 * M : M;
    if (path == GPTQ_Q4_PATH_DECODE && prefer_stream(h->K, h->N, h->geff, Mk, q4::device_sm_count()))
        path = GPTQ_Q4_PATH_DECODE_STREAM;
    const bool small_layer = small_layer_for(h->K, h->N, h->geff, Mk);
    // the activation kernel lets the decode grid start early when that grid
    // is the register-streaming kernel at M <= 8, or the stream-K kernel at
    // one row (28672x8192 act-order M = 1: 39.0 -> 37.0 us; measured slower
    // elsewhere, 1-3 % for the stream-K kernel at two rows)
    const bool early = Mk <= 8 && (path == GPTQ_Q4_PATH_DECODE_MMA || (path == GPTQ_Q4_PATH_DECODE_STREAM && Mk == 1) ||
                                   (path == GPTQ_Q4_PATH_DECODE && small_layer));
    const uint16_t *xin = static_cast<const uint16_t *>(x);
    q4::HandleView v = view(h);
    if (h->act_f32) {
        if (int r = ensure_temp_state(h, Mk, stream, false)) return r;
        if (int r = ensure_part(h, static_cast<size_t>(Mk) * h->N, stream, false)) return r;
        Q4_CUDA(q4::launch_xprep_f32(static_cast<const float *>(x), h->act_order ? h->perm : nullptr, M, h->Kx, h->K,
                                     h->temp_state, h->rowscale, stream),
                "fp32 preparation launch");
        ++g_launches;
        xin = h->temp_state;
        v.out_bf16 = q4::kOutF32;
        v.bias = nullptr;
        if (int r = run_path(h, v, xin, Mk, reinterpret_cast<uint16_t *>(h->part), stream, path, small_layer))
            return r;
        Q4_CUDA(q4::launch_combine_f32(h->part, h->rowscale, h->bias, M, h->N, static_cast<float *>(out), stream),
                "fp32 combine launch");
        ++g_launches;
        return ok();
    }
    if (h->act_bf16) {
        // bf16 x: scaled by a power of two per row and rounded once to fp16
        // (gathered at the same time under act-order); the epilogues undo the scale
        if (int r = ensure_temp_state(h, M, stream, false)) return r;
        Q4_CUDA(q4::launch_xprep_bf16(xin, h->act_order ? h->perm : nullptr, M, h->Kx, h->K, h->temp_state,
                                      h->rowscale, stream, early),
                "bf16 preparation launch");
        ++g_launches;
        xin = h->temp_state;
        v.rowscale = h->rowscale;
        v.out_bf16 = q4::kOutBF16;
    } else if (h->act_order) {
        if (int r = ensure_temp_state(h, M, stream, false)) return r;
        Q4_CUDA(q4::launch_xreorder(xin, h->perm, M, h->Kx, h->K, h->temp_state, stream, early), "xreorder launch");
        ++g_launches;
        xin = h->temp_state;
    }
    return run_path(h, v, xin, M, static_cast<uint16_t *>(out), stream, path, small_layer);
}

static int check_matmul_args(gptq_q4_handle h, const void *x, int M, const void *out) {
    if (int r = check_handle(h)) return r;
    if (M < 0) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "M=%d < 0", M);
    if (M == 0) return GPTQ_Q4_OK;
    if (!x || !out) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "x and out must not be NULL when M > 0");
    if (!aligned(x, 16) || !aligned(out, 16))
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "x and out must be 16-byte aligned");
    return GPTQ_Q4_OK;
}

int gptq_q4_matmul(gptq_q4_handle h, const void *x, int M, void *out, cudaStream_t stream) {
    if (int r = check_matmul_args(h, x, M, out)) return r;
    if (M == 0) return ok();
    int path = h->path;
    const int Mk = h->act_f32 ? 2 * M : M;            // rows the kernels see
    if (path == GPTQ_Q4_PATH_AUTO) path = (Mk >= h->prefill_min_m) ? GPTQ_Q4_PATH_PREFILL : GPTQ_Q4_PATH_DECODE;
    return run_matmul(h, x, M, out, stream, path);
}

int gptq_q4_dequant(gptq_q4_handle h, uint16_t *temp_dq, cudaStream_t stream) {
    if (int r = check_handle(h)) return r;
    if (!temp_dq) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "temp_dq must not be NULL");
    if (!aligned(temp_dq, 16)) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "temp_dq must be 16-byte aligned");
    if (h->bits == 8) Q4_CUDA(q4::launch_dequant8(view(h), h->inv8, h->Kx, temp_dq, stream), "dequant launch");
    else Q4_CUDA(q4::launch_dequant(view(h), temp_dq, stream), "dequant launch");
    ++g_launches;
    return ok();
}

int gptq_q4_debug_unpack(gptq_q4_handle h, uint8_t *q, uint8_t *z, cudaStream_t stream) {
    if (int r = check_handle(h)) return r;
    if (!q && !z) return ok();
    if (h->bits == 8) Q4_CUDA(q4::launch_unpack8(view(h), h->inv8, h->Kx, h->zsplit, q, z, stream), "unpack launch");
    else Q4_CUDA(q4::launch_debug_unpack(view(h), q, z, stream), "unpack launch");
    ++g_launches;
    return ok();
}

int gptq_q4_gemm_f16(const uint16_t *a, const uint16_t *b, const uint16_t *bias, int M, int K, int N,
                     uint16_t *out, cudaStream_t stream) {
    if (M < 0 || K <= 0 || N <= 0) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "bad sizes M=%d K=%d N=%d", M, K, N);
    if (K % 64 || N % 64)
        return set_status(GPTQ_Q4_UNSUPPORTED, "the tensor-core GEMM needs K %% 64 == 0 and N %% 64 == 0");
    if (M == 0) return ok();
    if (!a || !b || !out) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "a, b and out must not be NULL");
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(out, 16) || (bias && !aligned(bias, 2)))
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "a, b and out must be 16-byte aligned");
    Q4_CUDA(q4::launch_gemm_f16(a, b, bias, M, K, N, out, nullptr, stream), "gemm launch");
    ++g_launches;
    return ok();
}

int gptq_q4_matmul_unfused(gptq_q4_handle h, const void *x, int M, uint16_t *temp_dq, void *out,
                           cudaStream_t stream) {
    if (int r = check_matmul_args(h, x, M, out)) return r;
    if (M == 0) return ok();
    if (!temp_dq || !aligned(temp_dq, 16))
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "temp_dq must be a 16-byte aligned device buffer");
    if (h->bits == 8) Q4_CUDA(q4::launch_dequant8(view(h), h->inv8, h->Kx, temp_dq, stream), "dequant launch");
    else Q4_CUDA(q4::launch_dequant(view(h), temp_dq, stream), "dequant launch");
    ++g_launches;
    const uint16_t *xa = static_cast<const uint16_t *>(x);
    if (h->act_f32) {    // x in original order, split into hi and lo fp16 rows
        if (int r = ensure_temp_state(h, 2 * M, stream, false)) return r;
        if (int r = ensure_part(h, static_cast<size_t>(2 * M) * h->N, stream, false)) return r;
        Q4_CUDA(q4::launch_xprep_f32(static_cast<const float *>(x), nullptr, M, h->Kx, h->Kx, h->temp_state,
                                     h->rowscale, stream),
                "fp32 preparation launch");
        Q4_CUDA(q4::launch_gemm_f16(h->temp_state, temp_dq, nullptr, 2 * M, h->Kx, h->N,
                                    reinterpret_cast<uint16_t *>(h->part), h->status, stream, nullptr, q4::kOutF32),
                "gemm launch");
        Q4_CUDA(q4::launch_combine_f32(h->part, h->rowscale, h->bias, M, h->N, static_cast<float *>(out), stream),
                "fp32 combine launch");
        g_launches += 3;
        return ok();
    }
    if (h->act_bf16) {   // x in original order, scaled per row and rounded once to fp16
        if (int r = ensure_temp_state(h, M, stream, false)) return r;
        Q4_CUDA(q4::launch_xprep_bf16(xa, nullptr, M, h->Kx, h->Kx, h->temp_state, h->rowscale, stream),
                "bf16 preparation launch");
        ++g_launches;
        xa = h->temp_state;
    }
    Q4_CUDA(q4::launch_gemm_f16(xa, temp_dq, h->bias, M, h->Kx, h->N, static_cast<uint16_t *>(out), h->status, stream,
                                h->act_bf16 ? h->rowscale : nullptr, h->act_bf16),
            "gemm launch");
    ++g_launches;
    return ok();
}

int gptq_q4_set_path(gptq_q4_handle h, int path) {
    if (!h) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "handle is NULL");
    if (path < GPTQ_Q4_PATH_AUTO || path > GPTQ_Q4_PATH_DECODE_STREAM)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "unknown path %d", path);
    h->path = path;
    return ok();
}

int gptq_q4_set_prefill_min_m(gptq_q4_handle h, int min_m) {
    if (!h) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "handle is NULL");
    if (min_m < 0) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "min_m=%d < 0", min_m);
    h->prefill_min_m = min_m;
    return ok();
}

int gptq_q4_pack(const uint16_t *w, const uint16_t *scales, const int32_t *zeros, const int32_t *g_idx, int K,
                 int N, int groupsize, int format, int32_t *qweight, int32_t *qzeros, cudaStream_t stream) {
    if (!w || !scales || !qweight || !qzeros)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "w, scales, qweight and qzeros must not be NULL");
    if (K <= 0 || N <= 0 || K % 8 || N % 8)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "K=%d and N=%d must be positive multiples of 8", K, N);
    if (!(groupsize == -1 || (groupsize > 0 && K % groupsize == 0)))
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "groupsize=%d must be -1 or a positive divisor of K=%d",
                          groupsize, K);
    if (format != GPTQ_Q4_FORMAT_GPTQ && format != GPTQ_Q4_FORMAT_GPTQ_V2)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "format=%d is neither GPTQ nor GPTQ_V2", format);
    if (K / 8 > 65535) return set_status(GPTQ_Q4_UNSUPPORTED, "K=%d: the packer takes K <= 524280", K);
    const int geff = groupsize == -1 ? K : groupsize;
    const int G = K / geff;
    int dev = -1;
    Q4_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    if (int r = check_device_ptr(w, dev, "w")) return r;
    if (int r = check_device_ptr(scales, dev, "scales")) return r;
    if (zeros)
        if (int r = check_device_ptr(zeros, dev, "zeros")) return r;
    if (g_idx)
        if (int r = check_device_ptr(g_idx, dev, "g_idx")) return r;
    if (int r = check_device_ptr(qweight, dev, "qweight")) return r;
    if (int r = check_device_ptr(qzeros, dev, "qzeros")) return r;
    if (g_idx) {   // every row's group must exist: checked on the host before any kernel reads it
        std::vector<int32_t> gi(K);
        Q4_CUDA(cudaMemcpy(gi.data(), g_idx, sizeof(int32_t) * K, cudaMemcpyDeviceToHost), "copying g_idx");
        for (int k = 0; k < K; ++k)
            if (gi[k] < 0 || gi[k] >= G)
                return set_status(GPTQ_Q4_INVALID_ARGUMENT, "g_idx[%d]=%d outside [0, %d)", k, gi[k], G);
    }
    Q4_CUDA(q4::launch_pack(w, scales, zeros, g_idx, K, N, geff, G, format == GPTQ_Q4_FORMAT_GPTQ ? 1 : 0, qweight,
                            qzeros, stream),
            "pack launch");
    g_launches += 2;
    return ok();
}

int gptq_q4_debug_wait_probe(int *status, unsigned limit_us, cudaStream_t stream) {
    if (!status) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "status must not be NULL");
    if (limit_us == 0 || limit_us > 2000000u)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "limit_us=%u outside [1, 2000000]", limit_us);
    Q4_CUDA(q4::launch_wait_probe(status, static_cast<uint64_t>(limit_us) * 1000ull, stream), "wait probe launch");
    ++g_launches;
    return ok();
}

int gptq_q4_debug_dispatch(int M, int K, int N, int groupsize, int path, int sms, int *kernel) {
    if (!kernel) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "kernel must not be NULL");
    const int geff = groupsize == -1 ? K : groupsize;
    if (M < 1 || K <= 0 || N <= 0 || K % 64 || N % 64 || sms < 1 || geff <= 0 || geff % 32 || K % geff)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT,
                          "M=%d K=%d N=%d groupsize=%d sms=%d: need M >= 1, K and N positive multiples of 64, a "
                          "group size that is -1 or a multiple of 32 dividing K, sms >= 1",
                          M, K, N, groupsize, sms);
    if (path < GPTQ_Q4_PATH_AUTO || path > GPTQ_Q4_PATH_DECODE_STREAM)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "path=%d is not a GPTQ_Q4_PATH_* value", path);
    if (path == GPTQ_Q4_PATH_AUTO)
        path = M >= q4::prefill_default_min_m(K, N, geff) ? GPTQ_Q4_PATH_PREFILL : GPTQ_Q4_PATH_DECODE;
    if (path == GPTQ_Q4_PATH_DECODE && prefer_stream(K, N, geff, M, sms)) path = GPTQ_Q4_PATH_DECODE_STREAM;
    q4::DecodeSkPlan sp{};
    q4::DecodeRingPlan rp{};
    *kernel = static_cast<int>(kernel_for(path, M, K, N, geff, true, small_layer_for(K, N, geff, M), sms, &sp, &rp));
    return ok();
}

int gptq_q4_debug_prefill_plan(int M, int K, int N, int sms, int *out) {
    if (!out) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "out must not be NULL");
    if (M < 1 || K <= 0 || N <= 0 || K % 64 || N % 64 || sms < 1)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "M=%d K=%d N=%d sms=%d: need M >= 1, K and N positive multiples of 64, sms >= 1",
                          M, K, N, sms);
    const q4::PrefillPlan p = q4::plan_prefill(M, K, N, sms);
    out[0] = p.bm;
    out[1] = p.bn;
    out[2] = p.sk;
    out[3] = p.sk ? p.grid : 0;
    out[4] = p.sk ? p.pmax : 1;
    out[5] = p.fin0;
    out[6] = p.bk;
    return ok();
}

int gptq_q4_set_act_dtype(gptq_q4_handle h, int dtype) {
    if (!h) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "handle is NULL");
    if (dtype != GPTQ_Q4_DTYPE_FP16 && dtype != GPTQ_Q4_DTYPE_BF16 && dtype != GPTQ_Q4_DTYPE_FP32)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT,
                          "dtype=%d is none of GPTQ_Q4_DTYPE_FP16, GPTQ_Q4_DTYPE_BF16, GPTQ_Q4_DTYPE_FP32", dtype);
    h->act_bf16 = dtype == GPTQ_Q4_DTYPE_BF16 ? 1 : 0;
    h->act_f32 = dtype == GPTQ_Q4_DTYPE_FP32 ? 1 : 0;
    return ok();
}

int gptq_q4_set_format(gptq_q4_handle h, int format) {
    if (!h) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "handle is NULL");
    if (format != GPTQ_Q4_FORMAT_GPTQ && format != GPTQ_Q4_FORMAT_GPTQ_V2)
        return set_status(GPTQ_Q4_INVALID_ARGUMENT, "format=%d is neither GPTQ_Q4_FORMAT_GPTQ nor GPTQ_Q4_FORMAT_GPTQ_V2",
                          format);
    h->zero_offset = format == GPTQ_Q4_FORMAT_GPTQ ? 1 : 0;
    return ok();
}

int gptq_q4_info(gptq_q4_handle h, int *K, int *N, int *groupsize, int *G, int *act_order, size_t *device_bytes) {
    if (!h) return set_status(GPTQ_Q4_INVALID_ARGUMENT, "handle is NULL");
    if (K) *K = h->Kx;
    if (N) *N = h->N;
    if (groupsize) *groupsize = h->groupsize;
    if (G) *G = h->bits == 8 ? h->zsplit : h->G;
    if (act_order) *act_order = h->act_order;
    if (device_bytes) *device_bytes = h->device_bytes;
    return ok();
}

int gptq_q4_device_error(gptq_q4_handle h) {
    if (int r = check_handle(h)) return r;
    Q4_CUDA(cudaDeviceSynchronize(), "synchronize");
    int flag = 0;
    Q4_CUDA(cudaMemcpy(&flag, h->status, sizeof(int), cudaMemcpyDeviceToHost), "reading status word");
    if (flag) {
        Q4_CUDA(cudaMemset(h->status, 0, sizeof(int)), "clearing status word");
        return set_status(GPTQ_Q4_DEVICE_FAULT, "a kernel reported status 0x%x", flag);
    }
    return ok();
}

void gptq_q4_free(gptq_q4_handle h) {
    release(h);
    ok();
}

int gptq_q4_last_status(void) { return t_status; }
const char *gptq_q4_last_error(void) { return t_msg; }
uint64_t gptq_q4_launch_count(void) { return g_launches.load(); }

}  // extern "C"

namespace q4 {
int api_set_status(int code, const char *msg) { return set_status(code, msg ? "%s" : nullptr, msg); }
int api_cuda_fail(cudaError_t e, const char *what) { return cuda_fail(e, what); }
int api_check_matmul_args(gptq_q4_handle h, const void *x, int M, const void *out) {
    return check_matmul_args(h, x, M, out);
}
HandleView api_view(const gptq_q4_s *h) { return view(h); }
void api_count_launches(int n) { g_launches += static_cast<uint64_t>(n); }
}  // namespace q4
