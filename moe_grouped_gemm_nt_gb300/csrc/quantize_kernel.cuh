// quantize_kernel.cuh -- per-token (1 x 128) FP8 quantization of BF16
// activations into the GEMM's LHS: the FP8 matrix A and its MN-major scales sA.
//
// What it computes (page "DeepSeek开源周第三天DeepGEMM", section "基本用法": the
// LHS is FP8 with one FP32 scale per row and 128-wide K block, its scales
// transposed so that each K block's scales of all rows are contiguous; page
// "企业官网建设流程全解析", section 5.2: a scale comes from a scan of the group
// for its largest magnitude).  For row r of batch b and K block kb, over the
// block's columns inside k:
//
//   amax = max |x|,  s = amax / fmax  (1 when amax == 0),  q = fp8_rn_sat(x / s)
//
// with fmax = 448 (E4M3) or 57344 (E5M2), IEEE float32 division for both
// quotients, and round-to-nearest-even, saturating conversion to FP8.
//
// The work is bound by HBM bandwidth: 2 bytes read and 1 + 4/128 bytes written
// per element.  One CTA of 256 threads covers 32 rows x one 128-column K
// block; each row is handled by 8 consecutive lanes of one warp, 16 columns
// (two 16-byte loads, one 16-byte store) per lane, so a warp reads 4 rows x
// 256 contiguous bytes and the group maximum needs three butterfly shuffles.
// The 32 scales of the CTA form one contiguous 128-byte run of sA.
#pragma once

#include <cstdint>

#include "gemm_kernel.cuh"  // device status codes
#include "ptx.cuh"

namespace fg {

struct QuantParams {
    const uint16_t *x;         // bfloat16 bits [batches][rows][ld_x]
    uint8_t *a;                // FP8 codes [batches][rows][k]
    float *sa;                 // [batches][kb][ld_sa]
    const int32_t *masked_m;   // [batches] valid rows per batch, or null (all rows)
    uint32_t *status;          // per-device status word ([0] code, [1] detail)
    long long ld_x;            // elements between rows of x
    int ld_sa;                 // floats between K blocks of sa
    int rows;                  // rows per batch
    int k;                     // columns (multiple of 16)
    int kb;                    // ceil(k / 128)
};

constexpr int QUANT_ROWS = 32;      // rows per CTA
constexpr int QUANT_THREADS = 256;  // 8 lanes per row, 16 columns per lane
constexpr int QUANT_COLS_PER_LANE = 16;

// Two floats to two FP8 codes, round to nearest even, saturating to the finite
// range; `lo` lands in the low byte.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi) {
    uint16_t r;
    if constexpr (FMT == 0)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int FMT>
__global__ void __launch_bounds__(QUANT_THREADS) quantize_per_token_kernel(QuantParams p) {
    const int lane_row = threadIdx.x >> 3;  // 0..31
    const int seg = threadIdx.x & 7;        // which 16 columns of the K block
    const int row0 = blockIdx.x * QUANT_ROWS;
    const int kbi = blockIdx.y;
    const size_t b = blockIdx.z;

    // With programmatic dependent launch the previous kernel of the stream may
    // still be writing x or masked_m: wait for it before the first read.
    griddep_wait();

    int limit = p.rows;
    if (p.masked_m != nullptr) {
        const int c = __ldg(p.masked_m + b);
        if (c < 0 || c > p.rows) {
            if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 &&
                atomicCAS(p.status, 0u, (uint32_t)DEV_ERR_CHECK) == 0u)
                atomicExch(p.status + 1, (uint32_t)b);
            limit = c < 0 ? 0 : p.rows;
        } else {
            limit = c;
        }
    }
    if (row0 >= limit) return;  // uniform over the CTA

    const int row = row0 + lane_row;
    const int col = kbi * 128 + seg * QUANT_COLS_PER_LANE;
    const bool active = row < limit && col < p.k;  // k % 16 == 0: a lane's 16 columns are all in or all out

    float v[QUANT_COLS_PER_LANE];
    if (active) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (b * (size_t)p.rows + (size_t)row) * (size_t)p.ld_x +
                                                           (size_t)col);
        const uint4 w0 = __ldcs(src);      // streamed: x is read once, keep L2 for A and the weights
        const uint4 w1 = __ldcs(src + 1);
        const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < QUANT_COLS_PER_LANE; ++i) v[i] = 0.f;
    }

    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < QUANT_COLS_PER_LANE; ++i) amax = fmaxf(amax, fabsf(v[i]));
    // the 8 lanes of a row are 8 consecutive lanes: xor 1, 2, 4 stays inside them
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));

    if (!active) return;
    constexpr float kFmax = FMT == 0 ? 448.f : 57344.f;
    const float scale = amax > 0.f ? __fdiv_rn(amax, kFmax) : 1.f;

    uint32_t packed[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = cvt_fp8x2<FMT>(__fdiv_rn(v[4 * i], scale), __fdiv_rn(v[4 * i + 1], scale));
        const uint32_t hi = cvt_fp8x2<FMT>(__fdiv_rn(v[4 * i + 2], scale), __fdiv_rn(v[4 * i + 3], scale));
        packed[i] = lo | (hi << 16);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(p.a + (b * (size_t)p.rows + (size_t)row) * (size_t)p.k + (size_t)col);
    *dst = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if (seg == 0) p.sa[(b * (size_t)p.kb + (size_t)kbi) * (size_t)p.ld_sa + (size_t)row] = scale;
}

}  // namespace fg
