// gptq_q4_matmul_noalloc: the decode matmul with no device allocation.
//
// Who needs it.  Some callers cannot allocate device memory when they run a
// layer: a plugin inside a host framework that owns all device memory and
// hands the plugin only the tensors it works on; a service whose device
// memory is budgeted in full before the first request, so any later
// cudaMalloc could fail; a latency-critical loop that must never hit
// cudaMalloc/cudaFree, which can synchronize the whole device.  gptq_q4_matmul
// may grow its handle's work buffers on demand, so it is not for them.
//
// What it does.  The same decode kernel as gptq_q4_matmul's decode path,
// with its scratch -- the per-tile arrival tickets, the split-K fp32 partial
// sums and, for act-order, the gathered activations (temp_state) -- carved
// out of one fixed array, g_noalloc_scratch below, a file-scope static
// __device__ variable of GPTQ_Q4_NOALLOC_SCRATCH_BYTES bytes.  Every GPU
// that loads this library holds that array until the process exits.  The
// caller still passes x and out; nothing is allocated and nothing is freed.
//
// The weights of the handle were copied at gptq_q4_make time, which does
// allocate: only the per-call work is allocation-free.  This entry point has
// no counterpart on the web pages the rest of the library follows.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "q4_handle.h"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(GPTQ_Q4_NOALLOC_SCRATCH_BYTES);

// One array per device, shared by every call on that device; each call
// leaves its contents behind for the next.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// In host code the name g_noalloc_scratch is only a host-side stand-in, not a
// device address: a kernel handed it would fault or touch the wrong memory.
// The device address comes from cudaGetSymbolAddress, called with the device
// current.  The address belongs to the CUDA context that is current, not
// just to the device: a host framework may run this library inside a context
// of its own, and a context destroyed by cudaDeviceReset takes its mapping
// with it.  So the set-up runs once per context, and the cache is keyed by the
// context's process-unique ID (cuCtxGetId; IDs are never reused, so a context
// made after a reset never finds a stale entry).
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

struct ScratchEntry {
    unsigned long long ctx_id;
    void *ptr;
};
constexpr int kMaxContexts = 64;
std::mutex g_setup_mutex;
ScratchEntry g_entries[kMaxContexts] = {};
int g_used = 0, g_next_evict = 0;

bool driver_fns(CtxGetCurrentFn *get_current, CtxGetIdFn *get_id) {
    static CtxGetCurrentFn cur = nullptr;
    static CtxGetIdFn id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            cur = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            id = reinterpret_cast<CtxGetIdFn>(p);
        cudaGetLastError();
    });
    *get_current = cur;
    *get_id = id;
    return cur && id;
}

// The array's device address in the current context (the caller has made the
// handle's device current).  The first call in each context looks it up.
cudaError_t scratch_address(void **out) {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
    if (!driver_fns(&get_current, &get_id)) return cudaErrorNotSupported;
    CUcontext ctx = nullptr;
    unsigned long long ctx_id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &ctx_id) != CUDA_SUCCESS)
        return cudaErrorDeviceUninitialized;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    for (int i = 0; i < g_used; ++i)
        if (g_entries[i].ctx_id == ctx_id) {
            *out = g_entries[i].ptr;
            return cudaSuccess;
        }
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    int slot = g_used < kMaxContexts ? g_used++ : (g_next_evict++ % kMaxContexts);
    g_entries[slot] = ScratchEntry{ctx_id, p};
    *out = p;
    return cudaSuccess;
}

size_t round_up_256(size_t bytes) { return (bytes + 255) & ~static_cast<size_t>(255); }

}  // namespace

extern "C" int gptq_q4_matmul_noalloc(gptq_q4_handle h, const uint16_t *x, int M, uint16_t *out,
                                      cudaStream_t stream) {
    if (int r = q4::api_check_matmul_args(h, x, M, out)) return r;
    if (M == 0) return q4::api_set_status(GPTQ_Q4_OK, nullptr);
    if (h->act_f32)
        return q4::api_set_status(GPTQ_Q4_UNSUPPORTED,
                                  "gptq_q4_matmul_noalloc does not take fp32 activations (its scratch holds no "
                                  "partial rows); use gptq_q4_matmul");

    // Carve the scratch: tickets | split-K partials | temp_state.
    const q4::DecodePlan p = q4::plan_decode(M, h->K, h->N, h->geff);
    const size_t ticket_bytes = round_up_256(static_cast<size_t>(p.n_tickets) * sizeof(int));
    const size_t ws_bytes = round_up_256(p.ws_floats * sizeof(float));
    const size_t ts_bytes =
        (h->act_order || h->act_bf16) ? round_up_256(static_cast<size_t>(M) * h->K * sizeof(uint16_t)) : 0;
    const size_t rs_bytes = h->act_bf16 ? round_up_256(static_cast<size_t>(M) * sizeof(float)) : 0;
    const size_t need = ticket_bytes + ws_bytes + ts_bytes + rs_bytes;
    if (need > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "M=%d on this %dx%d layer needs %zu bytes of scratch; the static scratch of "
                 "gptq_q4_matmul_noalloc holds %zu bytes",
                 M, h->K, h->N, need, kScratchBytes);
        return q4::api_set_status(GPTQ_Q4_INVALID_ARGUMENT, msg);
    }
    void *base = nullptr;
    cudaError_t e;
    if ((e = scratch_address(&base)) != cudaSuccess)
        return q4::api_cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    unsigned char *scratch = static_cast<unsigned char *>(base);
    int *tickets = reinterpret_cast<int *>(scratch);
    float *ws = reinterpret_cast<float *>(scratch + ticket_bytes);
    uint16_t *temp_state = reinterpret_cast<uint16_t *>(scratch + ticket_bytes + ws_bytes);
    float *rowscale = reinterpret_cast<float *>(scratch + ticket_bytes + ws_bytes + ts_bytes);

    // The tickets must start at zero; the array keeps whatever the last
    // call (on any handle) left in it.
    if ((e = cudaMemsetAsync(tickets, 0, ticket_bytes, stream)) != cudaSuccess)
        return q4::api_cuda_fail(e, "clearing the scratch tickets");

    const uint16_t *xin = x;
    if (h->act_bf16) {
        if ((e = q4::launch_xprep_bf16(x, h->act_order ? h->perm : nullptr, M, h->Kx, h->K, temp_state, rowscale,
                                       stream, M <= 8)) != cudaSuccess)
            return q4::api_cuda_fail(e, "bf16 preparation launch");
        q4::api_count_launches(1);
        xin = temp_state;
    } else if (h->act_order) {
        if ((e = q4::launch_xreorder(x, h->perm, M, h->Kx, h->K, temp_state, stream, M <= 8)) != cudaSuccess)
            return q4::api_cuda_fail(e, "xreorder launch");
        q4::api_count_launches(1);
        xin = temp_state;
    }
    const q4::DecodeWork w{ws, p.ws_floats, tickets, p.n_tickets};
    q4::HandleView v = q4::api_view(h);
    if (h->act_bf16) {
        v.rowscale = rowscale;
        v.out_bf16 = 1;
    }
    if ((e = q4::launch_decode(v, p, w, xin, M, out, stream)) != cudaSuccess)
        return q4::api_cuda_fail(e, "decode launch");
    q4::api_count_launches(1);
    return q4::api_set_status(GPTQ_Q4_OK, nullptr);
}
