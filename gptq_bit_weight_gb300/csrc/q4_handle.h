// The handle behind gptq_q4_handle, shared by the C-ABI translation units.
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/gptq_q4.h"
#include "q4_internal.cuh"

struct gptq_q4_s {
    int device = -1;
    int K = 0, N = 0, groupsize = 0, geff = 0, G = 0;   // K, geff: rows and rows per group of the private layout
    int Kx = 0;             // the caller's K (columns of x); K > Kx when groups are padded
    int act_order = 0;
    uint32_t *wp = nullptr;
    uint32_t *s2 = nullptr;
    uint32_t *zeros = nullptr;
    int32_t *perm = nullptr;
    int32_t *inv8 = nullptr;    // 8-bit: private row of each split row (2 Kx entries)
    uint16_t *bias = nullptr;
    int *status = nullptr;
    float *ws = nullptr;
    size_t ws_floats = 0;
    int *tickets = nullptr;
    int n_tickets = 0;
    uint16_t *temp_state = nullptr;
    size_t temp_state_elems = 0;
    int path = GPTQ_Q4_PATH_AUTO;
    int prefill_min_m = 0;
    int zero_offset = 1;    // GPTQ_Q4_FORMAT_GPTQ: effective zero = stored + 1
    int bits = 4;           // 8: the handle holds an 8-bit layer as two 4-bit halves along K
    int zsplit = 0;         // groups [0, zsplit) take zero offset 0 (8-bit: the high-nibble half)
    int act_bf16 = 0;       // x and out are bf16 (GPTQ_Q4_DTYPE_BF16)
    int act_f32 = 0;        // x and out are fp32 (GPTQ_Q4_DTYPE_FP32)
    float *rowscale = nullptr;  // bf16 / fp32: 2^e per row of the current call
    size_t rowscale_elems = 0;
    float *part = nullptr;      // fp32: the raw sums of the hi and lo rows, [2M][N]
    size_t part_elems = 0;
    size_t device_bytes = 0;
};

namespace q4 {
// Status reporting and argument checks of the C ABI (q4_api.cu).
int api_set_status(int code, const char *msg);
int api_cuda_fail(cudaError_t e, const char *what);
int api_check_matmul_args(gptq_q4_handle h, const void *x, int M, const void *out);
HandleView api_view(const gptq_q4_s *h);
void api_count_launches(int n);
}  // namespace q4
