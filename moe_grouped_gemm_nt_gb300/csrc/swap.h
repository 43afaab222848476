// swap.h -- the swapped-operand path (gemm_swap_kernel.cuh) as seen by the
// library's dispatch in fp8gemm.cu; implemented in swap.cu.
#pragma once

#include "host_common.cuh"

namespace fgh {

// Plan of a swapped call: tokens per tile (128 or 256) and split-K cluster size.
struct SwapPlan {
    int bt = 128;
    int split = 1;
};

// Whether a call of this layout (fg::KIND_DENSE or fg::KIND_MASKED) with
// `rows` rows per group (dense m, masked M_cap) takes the swapped path under
// the current mode (fg_set_swap_mode), and its plan.
bool swap_applies(int kind, int rows, int G, int n, int k, int sms, SwapPlan *plan);

// Launch of a swapped call whose arguments the caller has checked.
fg_status launch_swap(int kind, bool f32out, const SwapPlan &plan, const void *A, int a_fmt, const float *sA,
                      int ld_sA, const void *B, int b_fmt, const float *sB, void *D, const int32_t *masked_m,
                      int rows, int G, int n, int k, int sms, const DeviceInfo *dev, cudaStream_t stream);

}  // namespace fgh
