// quantize_kernel.cuh -- per-token (1 x 128) FP8 quantization of BF16 or FP32
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
// The work is bound by HBM bandwidth: 2 bytes (FP32 input: 4) read and
// 1 + 4/128 bytes written per element.  A unit of work is 32 rows x one
// 128-column K block (8 KB of BF16 X, 16 KB of FP32).  CTAs are persistent (as many as fit on the SMs: seven per SM, by registers);
// each takes a contiguous range of units, walked along K.  One producer
// thread loads each unit with a single 3-D TMA box (columns past k and rows
// past the batch read as zeros) into the CTA's shared-memory stage; four
// consumer warps copy it to registers and release it at once, so the next
// unit's load overlaps their arithmetic and stores.  (Rings of two to four
// stages per CTA, and 64-row units with eight consumer warps, measured
// slower: more small CTAs per SM keep HBM busier than deeper rings.)  Each
// row is handled by 4 consecutive lanes with 32 columns each (four 16-byte
// chunks; odd rows take the chunks in the other order, so every quarter-
// warp's shared loads hit 32 distinct banks; FP32 rows are 512 bytes, so odd
// rows instead read the two 16-byte halves of each 32-byte piece in the other
// order); the group maximum runs on BF16 pairs (max.xorsign.abs: the larger
// magnitude of each half) or on FP32 magnitudes and needs two butterfly
// shuffles.  A consumer warp writes its codes (8-byte stores, 32
// contiguous bytes per row and store) and the row's scale (8 rows of a warp:
// 32 contiguous bytes of sA).  Every wait is bounded by a %globaltimer
// watchdog: on expiry the CTA records FG_ERR_TIMEOUT, stops, and waits (again
// bounded) for the copies it issued before it exits.
//
// The division by the group scale dominates the arithmetic.  It is computed
// from one correctly rounded reciprocal y = 1/s per group and fused
// multiply-adds on FP32 pairs (fma.rn.f32x2): q0 = x*y, then two corrections
// q <- q + (x - s*q)*y with an exact FMA residual.  After the first
// correction q is within one ulp of x/s; the second then gives the correctly
// rounded quotient (Markstein's theorem on quotient correction: P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990; see also Muller et al., "Handbook
// of Floating-Point Arithmetic", division by fused multiply-add), so the codes
// equal those of an IEEE division.  The theorem needs intermediates clear of
// underflow: with s >= 2^-40 every element whose quotient is large enough to
// give a nonzero FP8 code (|x/s| >= 2^-20) keeps them there, and smaller
// quotients round to a zero code either way.  Groups with s < 2^-40 take the
// plain IEEE division.  The sequence runs on the negated quotient p = -q
// (p0 = x*(-y), residual x + s*p, p <- p + residual*(-y)): every step is then
// an FMA with constant pair operands, rounding to nearest is symmetric so p
// is exactly -RN(x/s), and flipping the sign bits of the packed codes gives
// RN(x/s)'s codes, zeros of either sign included.  The scale itself,
// amax / fmax, is computed the same way from a reciprocal of fmax (IEEE
// division for amax < 2^-100).
#pragma once

#include <cstdint>

#include "gemm_kernel.cuh"  // device status codes
#include "ptx.cuh"

namespace fg {

struct QuantParams {
    const void *x;             // bfloat16 bits or float32 [batches][rows][ld_x]
    uint8_t *a;                // FP8 codes [batches][rows][k]
    float *sa;                 // [batches][kb][ld_sa]
    const int32_t *masked_m;   // [batches] valid rows per batch, or null (all rows)
    uint32_t *status;          // per-device status word ([0] code, [1] detail)
    unsigned long long timeout_ns;  // watchdog limit of each wait
    long long ld_x;            // elements between rows of x
    int ld_sa;                 // floats between K blocks of sa
    int rows;                  // rows per batch
    int k;                     // columns (multiple of 16)
    int kb;                    // ceil(k / 128)
    int row_blocks;            // ceil(rows / QUANT_ROWS)
    int units;                 // batches * row_blocks * kb
    int debug_skip_unit;       // producers leave their unit with this index unfilled (-1: never)
};

constexpr int QUANT_ROWS = 32;                              // rows per unit
constexpr int QUANT_CONSUMER_WARPS = QUANT_ROWS / 8;        // 8 rows each, 4 lanes per row
constexpr int QUANT_THREADS = (QUANT_CONSUMER_WARPS + 1) * 32;  // + the producer warp
constexpr int QUANT_STAGES = 1;  // measured best: many small CTAs beat deep rings
constexpr int QUANT_IN_BF16 = 0, QUANT_IN_F32 = 1;  // element type of X
// one unit of X: 8 KB of BF16 or 16 KB of FP32
__host__ __device__ constexpr int quant_stage_bytes(int in) { return QUANT_ROWS * 128 * (in == QUANT_IN_F32 ? 4 : 2); }
__host__ __device__ constexpr int quant_smem_bytes(int in) {
    return QUANT_STAGES * quant_stage_bytes(in) + 2 * QUANT_STAGES * 8 + 16;
}
constexpr float QUANT_MIN_FAST_SCALE = 0x1p-40f;
constexpr float QUANT_MIN_FAST_AMAX = 0x1p-100f;
constexpr uint32_t QUANT_ROLE_PRODUCER = 1, QUANT_ROLE_CONSUMER = 3;

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

__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f32x2_split(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// a / b rounded to nearest for one float, given yb = 1/b rounded to nearest
// (same construction; a >= 2^-100, b a normal power-of-two multiple such as
// an FP8 maximum).
__device__ __forceinline__ float div_by_const(float a, float b, float yb) {
    float q = __fmul_rn(a, yb);
    q = __fmaf_rn(__fmaf_rn(-q, b, a), yb, q);
    return __fmaf_rn(__fmaf_rn(-q, b, a), yb, q);
}

// A walk over consecutive units (K block fastest, then 32-row block, then
// batch) with the batch's valid rows.  next() is only called while units
// remain, so the batch index never passes the last batch.
struct QuantWalk {
    int b, rb, kbi, limit;

    __device__ __forceinline__ void start(const QuantParams &p, int u) {
        const int r = u / p.kb;
        kbi = u - r * p.kb;
        b = r / p.row_blocks;
        rb = r - b * p.row_blocks;
        load_limit(p);
    }
    __device__ __forceinline__ void next(const QuantParams &p) {
        if (++kbi == p.kb) {
            kbi = 0;
            if (++rb == p.row_blocks) {
                rb = 0;
                ++b;
                load_limit(p);
            }
        }
    }
    // valid rows of batch b; a count outside [0, rows] is clamped and reported
    // once per batch, by the consumer thread 0 of the CTA whose walk starts at
    // or enters the batch's first unit
    __device__ __forceinline__ void load_limit(const QuantParams &p) {
        limit = p.rows;
        if (p.masked_m == nullptr) return;
        const int c = __ldg(p.masked_m + b);
        if (c >= 0 && c <= p.rows) {
            limit = c;
            return;
        }
        limit = c < 0 ? 0 : p.rows;
        if (threadIdx.x == 0 && rb == 0 && kbi == 0 && atomicCAS(p.status, 0u, (uint32_t)DEV_ERR_CHECK) == 0u)
            atomicExch(p.status + 1, (uint32_t)b);
    }
};

// Bounded wait on an mbarrier phase; false on expiry (recorded, abort raised)
// or when another warp of the CTA aborted.
__device__ __noinline__ bool quant_wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                             const QuantParams &p, uint32_t role);

__device__ __forceinline__ bool quant_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                           const QuantParams &p, uint32_t role) {
    if (mbar_try_wait(bar, parity)) return true;
    return quant_wait_slow(bar, parity, abort_flag, p, role);
}

__device__ __noinline__ bool quant_wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                        const QuantParams &p, uint32_t role) {
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if ((++spins & 31u) == 0u && global_timer_ns() - t0 > p.timeout_ns) {
            if (atomicCAS(p.status, 0u, (uint32_t)DEV_ERR_TIMEOUT) == 0u)
                atomicExch(p.status + 1, (role << 24) | (bar & 0xFFFFu));
            *abort_flag = 1u;
            return false;
        }
    }
    return true;
}

// max(|a|, |b|) of each BF16 half (sign bit: the XOR of the inputs' signs)
__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// the pair of floats held by one BF16 pair
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
    return f32x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

template <int FMT, int IN>
__global__ void __launch_bounds__(QUANT_THREADS)
    quantize_per_token_kernel(const __grid_constant__ CUtensorMap tmap_x, QuantParams p) {
    constexpr int QUANT_STAGE_BYTES = quant_stage_bytes(IN);
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full0 = sbase + QUANT_STAGES * QUANT_STAGE_BYTES;  // full[s] = full0 + 8 s
    const uint32_t empty0 = full0 + QUANT_STAGES * 8;                 // empty[s] = empty0 + 8 s
    volatile uint32_t *abort_flag =
        reinterpret_cast<volatile uint32_t *>(smem + QUANT_STAGES * QUANT_STAGE_BYTES + 2 * QUANT_STAGES * 8);
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    // this CTA's units: a contiguous, balanced share
    const int u_begin = (int)(((long long)p.units * blockIdx.x) / gridDim.x);
    const int u_end = (int)(((long long)p.units * (blockIdx.x + 1)) / gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < QUANT_STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);                     // the producer's arrive.expect_tx
            mbar_init(empty0 + 8 * s, QUANT_CONSUMER_WARPS);  // one arrival per consumer warp
        }
        *abort_flag = 0u;
        fence_mbarrier_init();
    }
    if (threadIdx.x == QUANT_CONSUMER_WARPS * 32) prefetch_tensormap(&tmap_x);
    __syncthreads();

    // With programmatic dependent launch the previous kernel of the stream may
    // still be writing x or masked_m: wait for it before the first read.  The
    // next kernel may start its own set-up as CTAs of this one finish (it
    // waits for this grid's completion before it reads anything).
    griddep_wait();
    griddep_launch_dependents();
    if (u_begin >= u_end) return;

    if (warp == QUANT_CONSUMER_WARPS) {
        // ---------------------------------------------------------- producer
        if (lane != 0) return;
        QuantWalk w;
        w.start(p, u_begin);
        int j = 0;  // units of this CTA passed so far
        for (int u = u_begin; u < u_end; ++u, ++j, (u < u_end ? w.next(p) : (void)0)) {
            const int s = j % QUANT_STAGES;
            if (j >= QUANT_STAGES &&
                !quant_wait(empty0 + 8 * s, ((j / QUANT_STAGES) - 1) & 1, abort_flag, p, QUANT_ROLE_PRODUCER))
                break;
            if (j == p.debug_skip_unit) continue;  // test hook: this stage's consumers' wait runs out
            const int row0 = w.rb * QUANT_ROWS;
            if (row0 >= w.limit) {
                mbar_arrive(full0 + 8 * s);  // no valid row: nothing to load
            } else {
                mbar_arrive_expect_tx(full0 + 8 * s, QUANT_STAGE_BYTES);
                tma_load_3d(sbase + s * QUANT_STAGE_BYTES, &tmap_x, full0 + 8 * s, w.kbi * 128, row0, w.b);
            }
        }
        // Normally the consumers have waited for every copy; after an abort,
        // let the copies already issued land before the CTA's shared memory
        // goes away (bounded).
        if (*abort_flag) {
            for (int s = 0; s < QUANT_STAGES && s < j; ++s) {
                const int uses = (j - 1 - s) / QUANT_STAGES + 1;  // units passed through stage s
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(full0 + 8 * s, (uses - 1) & 1))
                    if (global_timer_ns() - t0 > p.timeout_ns) break;
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int lrow = warp * 8 + (lane >> 2);  // row of the unit, 0..QUANT_ROWS-1
    const int jq = lane & 3;                  // columns 32 c' + 8 jq .. + 7 for chunks c' = c ^ (lrow & 1)
    const int flip = lrow & 1;
    constexpr float kFmax = FMT == 0 ? 448.f : 57344.f;
    constexpr float kRcpFmax = FMT == 0 ? 0x1.24924ap-9f : 0x1.24924ap-16f;  // 1/fmax rounded to nearest
    QuantWalk w;
    w.start(p, u_begin);
    int j = 0;
    for (int u = u_begin; u < u_end; ++u, ++j, (u < u_end ? w.next(p) : (void)0)) {
        const int s = j % QUANT_STAGES;
        const bool ok = quant_wait(full0 + 8 * s, (j / QUANT_STAGES) & 1, abort_flag, p, QUANT_ROLE_CONSUMER);
        if (!__all_sync(0xffffffffu, ok)) break;  // warp-uniform exit
        const int row = w.rb * QUANT_ROWS + lrow;
        const bool act_row = row < w.limit;
        // this lane's 32 values (columns 32 c' + 8 jq .. + 7 of chunks c = 0..3):
        // BF16 pairs wd[4c .. 4c+3], or FP32 xf[8c .. 8c+7]
        uint32_t wd[IN == QUANT_IN_F32 ? 1 : 16];
        float xf[IN == QUANT_IN_F32 ? 32 : 1];
        if constexpr (IN == QUANT_IN_F32) {
            const uint8_t *srow = smem + s * QUANT_STAGE_BYTES + lrow * 512 + 32 * jq;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                // odd rows take the second 16 bytes first: the quarter-warp's two
                // rows then cover all 32 banks in each load
                const float4 v0 = *reinterpret_cast<const float4 *>(srow + 128 * (c ^ flip) + 16 * flip);
                const float4 v1 = *reinterpret_cast<const float4 *>(srow + 128 * (c ^ flip) + 16 * (flip ^ 1));
                const float4 lo = flip ? v1 : v0, hi = flip ? v0 : v1;
                xf[8 * c] = lo.x;
                xf[8 * c + 1] = lo.y;
                xf[8 * c + 2] = lo.z;
                xf[8 * c + 3] = lo.w;
                xf[8 * c + 4] = hi.x;
                xf[8 * c + 5] = hi.y;
                xf[8 * c + 6] = hi.z;
                xf[8 * c + 7] = hi.w;
            }
        } else {
            const uint8_t *srow = smem + s * QUANT_STAGE_BYTES + lrow * 256 + 16 * jq;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 v = *reinterpret_cast<const uint4 *>(srow + 64 * (c ^ flip));
                wd[4 * c] = v.x;
                wd[4 * c + 1] = v.y;
                wd[4 * c + 2] = v.z;
                wd[4 * c + 3] = v.w;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);  // the stage may be refilled now

        float amax;
        if constexpr (IN == QUANT_IN_F32) {
            amax = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(xf[i]));
        } else {
            uint32_t m2 = 0u;
#pragma unroll
            for (int i = 0; i < 16; ++i) m2 = bf16x2_max_abs(m2, wd[i]);
            amax = fmaxf(__uint_as_float((m2 << 16) & 0x7FFFFFFFu), __uint_as_float(m2 & 0x7FFF0000u));
        }
        // the 4 lanes of a row are 4 consecutive lanes: xor 1, 2 stays inside them
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        if (!act_row) continue;

        const float scale = amax >= QUANT_MIN_FAST_AMAX ? div_by_const(amax, kFmax, kRcpFmax)
                                                        : (amax > 0.f ? __fdiv_rn(amax, kFmax) : 1.f);
        uint32_t codes[8];  // chunk c: codes[2c] (columns +0..3), codes[2c+1] (+4..7); codes of -x/s
        if (scale >= QUANT_MIN_FAST_SCALE) {
            const float y = __frcp_rn(scale);
            const uint64_t ny2 = f32x2(-y, -y), s2 = f32x2(scale, scale);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t half[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint64_t x2;
                    if constexpr (IN == QUANT_IN_F32)
                        x2 = f32x2(xf[4 * i + 2 * h], xf[4 * i + 2 * h + 1]);
                    else
                        x2 = bf16x2_to_f32x2(wd[2 * i + h]);
                    uint64_t q = f32x2_mul(x2, ny2);
                    q = f32x2_fma(f32x2_fma(q, s2, x2), ny2, q);
                    q = f32x2_fma(f32x2_fma(q, s2, x2), ny2, q);
                    float lo, hi;
                    f32x2_split(q, lo, hi);
                    half[h] = cvt_fp8x2<FMT>(lo, hi);
                }
                codes[i] = half[0] | (half[1] << 16);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t half[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float x0, x1;
                    if constexpr (IN == QUANT_IN_F32) {
                        x0 = xf[4 * i + 2 * h];
                        x1 = xf[4 * i + 2 * h + 1];
                    } else {
                        x0 = __uint_as_float(wd[2 * i + h] << 16);
                        x1 = __uint_as_float(wd[2 * i + h] & 0xFFFF0000u);
                    }
                    half[h] = cvt_fp8x2<FMT>(__fdiv_rn(-x0, scale), __fdiv_rn(-x1, scale));
                }
                codes[i] = half[0] | (half[1] << 16);
            }
        }
        uint8_t *arow = p.a + ((size_t)w.b * (size_t)p.rows + (size_t)row) * (size_t)p.k + (size_t)w.kbi * 128;
        const int len = min(128, p.k - w.kbi * 128);  // valid columns of this block (multiple of 16)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int col = 32 * (c ^ flip) + 8 * jq;
            if (col < len)  // the sign flip turns the codes of -x/s into those of x/s
                *reinterpret_cast<uint2 *>(arow + col) =
                    make_uint2(codes[2 * c] ^ 0x80808080u, codes[2 * c + 1] ^ 0x80808080u);
        }
        if (jq == 0) p.sa[((size_t)w.b * (size_t)p.kb + (size_t)w.kbi) * (size_t)p.ld_sa + (size_t)row] = scale;
    }
}

}  // namespace fg
