// fp8gemm.cu -- C ABI of the FP8 NT GEMM library (declared in include/fp8gemm.h):
// argument checks, TMA tensor-map encoding, kernel selection and launch, and the
// per-device status word written by the kernels' watchdogs and range checks.
#include "host_common.cuh"
#include "gemm_pair_kernel.cuh"
#include "quantize_kernel.cuh"
#include "swap.h"

namespace fg {

// Row-major [batches][rows][kb] -> MN-major [batches][kb][ld] (zero padding).
__global__ void scales_to_mn_major_kernel(const float *__restrict__ src, float *__restrict__ dst, int rows,
                                          int kb, int ld) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    const int j = blockIdx.y;
    const size_t b = blockIdx.z;
    if (r >= ld) return;
    const float v = r < rows ? src[(b * rows + r) * kb + j] : 0.f;
    dst[(b * kb + j) * ld + r] = v;
}

}  // namespace fg

namespace fgh {

// [0] first error code, [1] detail; one copy per device (module globals are per context)
__device__ uint32_t g_status[2];

std::atomic<int> g_num_sms_override{0};
std::atomic<uint32_t> g_watchdog_ms{kDefaultWatchdogMs};
std::atomic<int> g_debug_skip_iter{-1};
std::atomic<int> g_force_bn{0};
std::atomic<int> g_pdl{1};
std::atomic<int> g_force_split{0};
std::atomic<int> g_pair_mode{-1};
std::atomic<int> g_swap_mode{-1};
std::atomic<int> g_debug_bad_coord{-1};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

fg_status device_info(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cuda_fail();
    DeviceInfo &d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int sms = 0;
            void *st = nullptr;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return cuda_fail();
            if (cudaGetSymbolAddress(&st, g_status) != cudaSuccess) return cuda_fail();
            d.status = static_cast<uint32_t *>(st);
            d.num_sms = sms;
            d.ready.store(1, std::memory_order_release);
        }
    }
    *out = &d;
    return FG_OK;
}

}  // namespace fgh

namespace {

using namespace fgh;

// Operand stages of the one-CTA kernel: 4 of 16 + 32 KB for 256-wide tiles, 6
// of 16 + 16 KB for 128-wide ones (what fits beside the staging buffers).  The
// debug build (FG_DEBUG) runs every pipeline on as few stages as it can: one,
// or for split-K the fewest whose ring holds the FP32 partial tile (3 and 2),
// so that a result which changes with the pipeline depth points at a missing
// wait (the single-buffer bisection of the pages' debugging method).
template <int BN, bool SPLITK>
constexpr int one_cta_stages() {
    if (fg::kDebugBuild) return SPLITK ? (BN == 256 ? 3 : 2) : 1;
    return BN == 256 ? 4 : 6;
}

template <int BN, int KIND, bool SPLITK, bool F32OUT = false>
using Kernel = Launcher<fg::fp8_gemm_kernel<BN, one_cta_stages<BN, SPLITK>(), KIND, SPLITK, F32OUT>,
                        fg::SmemLayout<BN, one_cta_stages<BN, SPLITK>()>::BYTES, SPLITK>;

// 256 x 256 tiles on CTA pairs: operand stages of 16 + 16 KB per CTA, and a
// scale ring at least as deep (the producer issues both in the same iteration)
constexpr int kPairStages = fg::kDebugBuild ? 1 : 5;
constexpr int kPairScaleStages = 8;
template <int KIND, bool F32OUT = false>
using PairKernel = Launcher<fg::fp8_gemm_pair_kernel<KIND, kPairStages, kPairScaleStages, F32OUT>,
                            fg::PairSmemLayout<kPairStages, kPairScaleStages>::BYTES, true>;
// deferred stores (BF16 output): the staging holds a whole tile, bought with
// one operand stage less
constexpr int kPairDeferStages = fg::kDebugBuild ? 1 : 4;
template <int KIND>
using PairDeferKernel = Launcher<fg::fp8_gemm_pair_kernel<KIND, kPairDeferStages, kPairScaleStages, false, true>,
                                 fg::PairSmemLayout<kPairDeferStages, kPairScaleStages, true>::BYTES, true,
                                 fg::PAIR_DEFER_THREADS>;
// -1: deferred stores for dense (and masked) tiles of at most kPairDeferMaxKb
// K blocks and for K-grouped segments of kKgDeferMinKb to kKgDeferMaxKb K
// blocks on average; 0 never; 1 always.  Measured on CTA pairs (graph-timed,
// without -> with the store warp, which costs the fifth operand stage): dense
// 4096 x 24576 x 1536 135.5 -> 120.7 us, 4096 x 7168 x 2048 51.9 -> 49.1,
// 4096 x 7168 x 4096 89.6 -> 87.1, 4096 x 4096 x 7168 99.4 -> 98.1, 4096 x 7168
// x 7168 146.7 -> 144.6; 8192^3 385.6 -> 386.8, 4096 x 7168 x 16384 324.6 ->
// 329.1.  K-grouped, 8 groups of 4096 x 7168: 1024 tokens each 244.8 -> 228.6,
// 1536: 323.5 -> 322.1, 1792: 362.9 -> 365.1, 2048: 401.4 -> 411.8; segments of
// 2 K blocks: 32 groups of 4096 x 7168 with 256 tokens 371.3 -> 394.5.
std::atomic<int> g_pair_defer{-1};
constexpr int kPairDeferMaxKb = 56;
constexpr int kKgDeferMinKb = 4;
constexpr int kKgDeferMaxKb = 12;

// Tile plan of one call: output tile width and split-K factor.
struct Plan {
    int bn = 256;
    int split = 1;  // CTAs per output tile (one cluster); 1 = persistent walk
};

// ---- plan of a call with `m_blocks` 128-row blocks (grouped layouts: all
// groups; masked: the capacity, as the counts live on the device) and at most
// `rows` valid rows per 128-row block.  Persistent 128 x 256 tiles when they
// fill the GPU.  Otherwise (few output tiles, e.g. m <= 128) the tile width
// and split-K cluster size with the lowest estimated time:
//   start-up + max(HBM time, K blocks per CTA x K-block time) x waves
//   + (split-K) cluster barrier + partial exchange through distributed smem.
// The constants were measured on GB300 (per-phase timestamps in the kernel,
// a distributed-shared-memory microbenchmark) and rank the measured plans of
// the small-m problems correctly.
constexpr double kStartUs = 3.5;         // launch to first operand bytes
constexpr double kKBlockUs256 = 0.50;    // one 128 x 256 x 128 K block, promotion included
constexpr double kKBlockUs128 = 0.35;    // one 128 x 128 x 128 K block
constexpr double kHbmBytesPerUs = 6.5e6; // sustained HBM bandwidth
constexpr double kDsmemBytesPerUs = 3.4e4;  // per-SM distributed shared memory bandwidth
constexpr double kReduceSyncUs = 1.0;    // the cluster barriers around the exchange

double plan_cost(long long m_blocks, int rows, int n, int k, int bn, int split, long long cap_ctas) {
    const long long kb = cdiv(k, fg::BLOCK_K);
    const long long tiles = m_blocks * cdiv(n, bn);
    const long long ctas = tiles * split;
    const long long waves = (ctas + cap_ctas - 1) / cap_ctas;
    const double kb_per_cta = (double)((kb + split - 1) / split) * (double)waves;
    const double rows_total = (double)(rows < m_blocks * fg::BLOCK_M ? rows : m_blocks * fg::BLOCK_M);
    const double hbm_us = (rows_total * k + (double)n * k + rows_total * n * 2.0) / kHbmBytesPerUs;
    const double main_us = std::max(hbm_us, kb_per_cta * (bn == 256 ? kKBlockUs256 : kKBlockUs128));
    double red_us = 0.0;
    if (split > 1) {
        const double tile_rows = rows < fg::BLOCK_M ? rows : fg::BLOCK_M;
        red_us = kReduceSyncUs + tile_rows * bn * 4.0 * (split - 1) / split / kDsmemBytesPerUs;
    }
    return kStartUs + main_us + red_us;
}

Plan choose_plan(long long m_blocks, int rows, int n, int k, int sms) {
    Plan plan;
    const int fbn = g_force_bn.load(), fsplit = g_force_split.load();
    if (fbn != 0 || fsplit != 0) {
        plan.bn = fbn == 128 ? 128 : 256;
        plan.split = fsplit > 0 ? fsplit : 1;
        return plan;
    }
    const int num_kb = cdiv(k, fg::BLOCK_K);
    const long long tiles256 = m_blocks * cdiv(n, 256);
    if (tiles256 * 4 >= (long long)sms * 3) return plan;
    double best = 1e30;
    for (int bn : {256, 128}) {
        for (int sp = 1; sp <= 8; ++sp) {
            if (sp > 1 && num_kb < 2 * sp) break;  // at least two K blocks per rank
            long long cap = sms;
            if (sp > 1) {
                const int clusters = bn == 256 ? Kernel<256, fg::KIND_DENSE, true>::max_active_clusters(sp)
                                               : Kernel<128, fg::KIND_DENSE, true>::max_active_clusters(sp);
                cap = (long long)sp * clusters;
                if (cap > (long long)(sms / sp) * sp) cap = (long long)(sms / sp) * sp;  // the SM limit
                // a second wave of clusters would pay start-up and exchange again
                if (cap <= 0 || m_blocks * cdiv(n, bn) * sp > cap) continue;
            }
            const double c = plan_cost(m_blocks, rows, n, k, bn, sp, cap);
            if (c < best) {
                best = c;
                plan.bn = bn;
                plan.split = sp;
            }
        }
    }
    return plan;
}

bool fmt_ok(int f) { return f == FG_E4M3 || f == FG_E5M2; }

// M blocks per raster group: as many as keep the group's A rows (128 x k bytes
// per block) within about 48 MiB of L2, so B is streamed once per group while
// A stays resident.  Masked problems walk N fastest (raster groups of one M
// block): a CTA's tiles then visit the valid M blocks in increasing order, so
// each role finds a tile's group with a forward scan over the counts, and a
// group's weights, read once per M block, are still in L2 for its next one.
int raster_group_m(int kind, int m_blocks, int k) {
    if (kind == fg::KIND_MASKED) return 1;
    const long long per_block = (long long)fg::BLOCK_M * k;
    long long g = (48ll << 20) / (per_block > 0 ? per_block : 1);
    if (g < 1) g = 1;
    if (g > m_blocks) g = m_blocks;
    return (int)(g > 0 ? g : 1);
}

// Whether a call runs on CTA pairs (256 x 256 tiles): by default, persistent
// 256-wide dense plans with at least 256 rows, unless a tile plan is forced;
// with the pair mode at 1, every persistent 256-wide plan.  The contiguous
// layout keeps 128-row tiles by default: on pairs (a tile whose two 128-row
// blocks belong to different groups runs once per group) it measured within
// 2% of them either way (graph-timed, one CTA / pairs / pairs with the store
// warp: 4 groups of 8192 rows x 4096 x 7168 715.2 / 698.8 / 700.3 us, 8 groups
// 1433.5 / 1454.8 / 1494.9, 8 x 8192 rows x 7168 x 2048 807.7 / 821.2 / 805.0)
// and 21% slower when every pair holds two groups (64 groups of 128 rows x
// 7168 x 2048: 176.4 / 212.9 / 218.0).  The masked layout keeps them by default: a group's valid rows rarely fill 256,
// and a 256-row tile computes and loads its empty lower half where a 128-row
// block past the count is skipped (measured on the masked workloads with
// capacity 256: 16 groups take 108 us on 128-row tiles against 133 us on
// pairs for n = 4096, 63 against 72 us for n = 7168).
bool use_pair(int kind, const Plan &plan, int rows) {
    if (plan.split != 1 || plan.bn != 256) return false;
    const int mode = g_pair_mode.load();
    if (mode == 0) return false;
    if (mode == 1) return true;
    if (kind == fg::KIND_MASKED || kind == fg::KIND_CONTIGUOUS) return false;
    if (g_force_bn.load() != 0 || g_force_split.load() != 0) return false;
    return rows >= fg::PAIR_ROWS;
}

// Shared part of the GEMM entry points (BF16 or, with F32OUT, FP32 output).
//   a_rows: rows of the 2-D A / D row space; b_rows: G * n.
template <int KIND, bool F32OUT = false>
fg_status run(const void *A, int a_fmt, const float *sA, int ld_sA, const void *B, int b_fmt, const float *sB,
              void *D, const int32_t *m_indices, const int32_t *masked_m, int rows, int G, int n, int k,
              cudaStream_t stream) {
    if (!A || !B || !sA || !sB || !D) return FG_ERR_INVALID_ARG;
    if (!fmt_ok(a_fmt) || !fmt_ok(b_fmt)) return FG_ERR_INVALID_ARG;
    if (rows < 0 || n < 1 || k < 1 || G < 1) return FG_ERR_INVALID_ARG;
    if (ld_sA < rows || ld_sA < 1) return FG_ERR_INVALID_ARG;
    if (KIND == fg::KIND_CONTIGUOUS && !m_indices) return FG_ERR_INVALID_ARG;
    if (KIND == fg::KIND_MASKED && !masked_m) return FG_ERR_INVALID_ARG;
    if (k % 16 != 0 || n % 8 != 0) return FG_ERR_UNSUPPORTED;
    if (KIND == fg::KIND_CONTIGUOUS && rows % fg::BLOCK_M != 0) return FG_ERR_UNSUPPORTED;
    if (ld_sA % 4 != 0) return FG_ERR_MISALIGNED;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || !aligned16(sA) || !aligned4(sB))
        return FG_ERR_MISALIGNED;
    const long long a_rows_total = (KIND == fg::KIND_MASKED) ? (long long)G * rows : rows;
    if ((long long)G * n > INT32_MAX || a_rows_total > INT32_MAX) return FG_ERR_UNSUPPORTED;
    if (rows == 0) return FG_OK;

    DeviceInfo *dev = nullptr;
    if (fg_status st = device_info(&dev); st != FG_OK) return st;

    int sms = dev->num_sms;
    const int ovr = g_num_sms_override.load();
    if (ovr > 0 && ovr < sms) sms = ovr;
    if constexpr (KIND != fg::KIND_CONTIGUOUS) {
        // few rows per group: the weights in the MMA's 128-row role (swap.cu)
        SwapPlan sp;
        if (swap_applies(KIND, rows, G, n, k, sms, &sp))
            return launch_swap(KIND, F32OUT, sp, A, a_fmt, sA, ld_sA, B, b_fmt, sB, D, masked_m, rows, G, n, k, sms,
                               dev, stream);
    }
    const int num_kb = cdiv(k, fg::BLOCK_K);
    const long long m_blocks_total = (long long)cdiv(rows, fg::BLOCK_M) * (KIND == fg::KIND_MASKED ? G : 1);
    const Plan plan = choose_plan(m_blocks_total, KIND == fg::KIND_DENSE ? rows : INT32_MAX, n, k, sms);
    const int BN = plan.bn;
    const bool pair = use_pair(KIND, plan, rows) && sms >= 2;

    CUtensorMap ta, tb, td, tsa;
    if (!encode_scales_a(&tsa, sA, ld_sA, rows, cdiv(k, fg::BLOCK_K), G, KIND == fg::KIND_MASKED) ||
        !encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, (uint64_t)k, (uint64_t)a_rows_total, (uint64_t)k,
                   fg::BLOCK_K, fg::BLOCK_M) ||
        !encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, (uint64_t)k, (uint64_t)G * n, (uint64_t)k, fg::BLOCK_K,
                   (uint32_t)(pair ? fg::PAIR_BN / 2 : BN)) ||
        !(F32OUT ? encode_2d(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D, (uint64_t)n, (uint64_t)a_rows_total,
                             (uint64_t)n * 4, 32, 32)
                 : encode_2d(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)n, (uint64_t)a_rows_total,
                             (uint64_t)n * 2, 64, 32)))
        return cuda_fail();

    GemmParams p{};
    p.rows = rows;
    p.n = n;
    p.k = k;
    p.num_groups = G;
    p.num_kb = num_kb;
    p.num_nb = cdiv(n, 128);
    p.num_n_blocks = cdiv(n, BN);
    p.num_m_blocks = cdiv(rows, fg::BLOCK_M);
    p.group_m = raster_group_m(KIND, p.num_m_blocks * (KIND == fg::KIND_MASKED ? G : 1), k);
    p.idesc = fg::make_idesc_f8f6f4(fg::BLOCK_M, BN, (uint32_t)a_fmt, (uint32_t)b_fmt);
    p.sB = sB;
    p.m_indices = m_indices;
    p.masked_m = masked_m;
    p.D = D;
    p.status = dev->status;
    p.timeout_ns = (unsigned long long)g_watchdog_ms.load() * 1000000ull;
    p.debug_skip_iter = g_debug_skip_iter.exchange(-1);
    p.a_rows_total = (int)a_rows_total;
    p.b_rows_total = G * n;
    p.debug_bad_coord = g_debug_bad_coord.exchange(-1);

    {
        if (pair) {
            // 256 x 256 tiles on CTA pairs: the raster counts 256-row blocks
            // (whose A rows take twice the bytes of a 128-row block)
            const long long pblocks = (long long)cdiv(rows, fg::PAIR_ROWS) * (KIND == fg::KIND_MASKED ? G : 1);
            p.num_n_blocks = cdiv(n, fg::PAIR_BN);
            p.group_m = raster_group_m(KIND, (int)pblocks, 2 * k);
            p.idesc = fg::make_idesc_f8f6f4(fg::PAIR_ROWS, fg::PAIR_BN, (uint32_t)a_fmt, (uint32_t)b_fmt);
            const long long tiles = pblocks * p.num_n_blocks;
            const int dmode = g_pair_defer.load();
            const bool defer = !F32OUT && (dmode == 1 || (dmode < 0 && num_kb <= kPairDeferMaxKb));
            long long clusters = defer ? PairDeferKernel<KIND>::max_active_clusters(2)
                                       : PairKernel<KIND, F32OUT>::max_active_clusters(2);
            if (clusters < 1) return cuda_fail();
            if (clusters > sms / 2) clusters = sms / 2;  // the SM limit (fg_set_num_sms); sms >= 2 here
            if (clusters > tiles) clusters = tiles;
            if constexpr (!F32OUT) {
                if (defer) return PairDeferKernel<KIND>::launch(ta, tb, td, tsa, p, (int)(2 * clusters), 2, stream);
            }
            return PairKernel<KIND, F32OUT>::launch(ta, tb, td, tsa, p, (int)(2 * clusters), 2, stream);
        }
    }
    const long long max_tiles = m_blocks_total * p.num_n_blocks;
    {
        if (plan.split > 1) {
            // one cluster of `split` CTAs per output tile
            const long long grid = max_tiles * plan.split;
            if (grid > INT32_MAX) return FG_ERR_UNSUPPORTED;
            if (BN == 256)
                return Kernel<256, KIND, true, F32OUT>::launch(ta, tb, td, tsa, p, (int)grid, plan.split,
                                                                  stream);
            return Kernel<128, KIND, true, F32OUT>::launch(ta, tb, td, tsa, p, (int)grid, plan.split, stream);
        }
        if (BN == 128) {
            const int grid = (int)(max_tiles < sms ? max_tiles : sms);
            return Kernel<128, KIND, false, F32OUT>::launch(ta, tb, td, tsa, p, grid, 1, stream);
        }
    }
    const int grid = (int)(max_tiles < sms ? max_tiles : sms);
    return Kernel<256, KIND, false, F32OUT>::launch(ta, tb, td, tsa, p, grid, 1, stream);
}

// K-grouped entry points: G groups, each an NT product over its own segment of
// K (segment lengths on the device), all sharing A [M][K] and B [N][K]; output
// planes D [G][M][N].  Persistent tiles, no split-K: 256 x 256 on CTA pairs
// (BF16 output, M >= 256, the 256-wide tiles filling the SMs; the store warp
// for segments of 4 to 12 K blocks on average), else one-CTA 128 x 256 (or
// 128 x 128 when the 256-wide tiles would leave SMs idle).
struct KgPlan {
    int bn = 256;
    bool pair = false;
    bool defer = false;  // CTA pairs with the store warp (BF16 output only)
};
KgPlan kgrouped_plan(int G, int M, int N, int K, int sms, bool f32out) {
    KgPlan kp;
    // 256-wide tiles unless they fill less than three quarters of the SMs
    // four times over and 128-wide ones have more tiles (or the width is forced)
    const long long tiles256 = (long long)G * cdiv(M, fg::BLOCK_M) * cdiv(N, 256);
    const int fbn = g_force_bn.load();
    if (fbn == 128 || (fbn == 0 && tiles256 * 4 < (long long)sms * 3)) kp.bn = 128;
    // CTA pairs for BF16 output with M >= 256, whatever the segment lengths,
    // with the store warp when the segments average kKgDeferMinKb to
    // kKgDeferMaxKb K blocks.  Measured (graph-timed; one CTA / pairs / pairs
    // with the store warp): 4 groups of 4096 x 7168 with 8192 tokens each
    // 728.5 / 690.4 / 792.5 us; 8 of 7168 x 2048 with 8192 tokens 753.6 /
    // 711.9 / 822.9; 8 of 4096 x 7168 with 2048 tokens 417.6 / 404.9 / 414.5,
    // with 1024 tokens 253.4 / 248.3 / 230.8; 32 of 4096 x 7168 with 512 tokens
    // 629.2 / 637.3 / 519.7, with 256 tokens 395.0 / 371.3 / 394.5.
    const long long kb_total = cdiv(K, fg::BLOCK_K);
    const int pmode = g_pair_mode.load();
    kp.pair = sms >= 2 && kp.bn == 256 && pmode != 0 &&
              (pmode == 1 || (fbn == 0 && M >= fg::PAIR_ROWS && !f32out));
    const int dmode = g_pair_defer.load();
    const bool defer_len = kb_total >= (long long)kKgDeferMinKb * G && kb_total <= (long long)kKgDeferMaxKb * G;
    kp.defer = kp.pair && !f32out && (dmode == 1 || (dmode < 0 && defer_len));
    return kp;
}

template <bool F32OUT>
fg_status run_kgrouped(const void *A, int a_fmt, const float *sA, int ld_sA, const void *B, int b_fmt,
                       const float *sB, void *D, const int32_t *k_sizes, int G, int M, int N, int K,
                       cudaStream_t stream) {
    if (!A || !B || !sA || !sB || !D || !k_sizes) return FG_ERR_INVALID_ARG;
    if (!fmt_ok(a_fmt) || !fmt_ok(b_fmt)) return FG_ERR_INVALID_ARG;
    if (M < 0 || N < 1 || K < 1 || G < 1 || ld_sA < M || ld_sA < 1) return FG_ERR_INVALID_ARG;
    if (K % 16 != 0 || N % 8 != 0) return FG_ERR_UNSUPPORTED;
    if (ld_sA % 4 != 0) return FG_ERR_MISALIGNED;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || !aligned16(sA) || !aligned4(sB)) return FG_ERR_MISALIGNED;
    const long long tiles256 = (long long)G * cdiv(M, fg::BLOCK_M) * cdiv(N, 256);
    if ((long long)G * M > INT32_MAX || tiles256 * 2 > INT32_MAX || G > 65535) return FG_ERR_UNSUPPORTED;
    if (M == 0) return FG_OK;

    DeviceInfo *dev = nullptr;
    if (fg_status st = device_info(&dev); st != FG_OK) return st;
    int sms = dev->num_sms;
    const int ovr = g_num_sms_override.load();
    if (ovr > 0 && ovr < sms) sms = ovr;
    const KgPlan kp = kgrouped_plan(G, M, N, K, sms, F32OUT);
    const int BN = kp.bn;
    const bool pair = kp.pair;

    const int num_kb = cdiv(K, fg::BLOCK_K);
    CUtensorMap ta, tb, td, tsa;
    const uint64_t ddims[3] = {(uint64_t)N, (uint64_t)M, (uint64_t)G};
    const uint64_t dstrides[2] = {(uint64_t)N * (F32OUT ? 4 : 2), (uint64_t)N * (F32OUT ? 4 : 2) * (uint64_t)M};
    const uint32_t dbox[3] = {F32OUT ? 32u : 64u, 32u, 1u};
    if (!encode_scales_a(&tsa, sA, ld_sA, M, num_kb, 1, false) ||
        !encode_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, (uint64_t)K, (uint64_t)M, (uint64_t)K, fg::BLOCK_K,
                   fg::BLOCK_M) ||
        !encode_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, (uint64_t)K, (uint64_t)N, (uint64_t)K, fg::BLOCK_K,
                   (uint32_t)(pair ? fg::PAIR_BN / 2 : BN)) ||
        !encode(&td, F32OUT ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, 3, ddims,
                dstrides, dbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return cuda_fail();

    GemmParams p{};
    p.rows = M;
    p.n = N;
    p.k = K;
    p.num_groups = G;
    p.num_kb = num_kb;
    p.num_nb = cdiv(N, 128);
    p.num_n_blocks = cdiv(N, BN);
    p.num_m_blocks = cdiv(M, fg::BLOCK_M);
    // the raster sizes its L2 working set by the K that one tile reads: the
    // segments' average length (the lengths stay on the device)
    const int k_seg = (int)std::max<long long>(fg::BLOCK_K, (long long)cdiv(K, fg::BLOCK_K) * fg::BLOCK_K / G);
    p.group_m = raster_group_m(fg::KIND_KGROUPED, p.num_m_blocks, k_seg);
    p.idesc = fg::make_idesc_f8f6f4(fg::BLOCK_M, BN, (uint32_t)a_fmt, (uint32_t)b_fmt);
    p.sB = sB;
    p.k_sizes = k_sizes;
    p.D = D;
    p.status = dev->status;
    p.timeout_ns = (unsigned long long)g_watchdog_ms.load() * 1000000ull;
    p.debug_skip_iter = g_debug_skip_iter.exchange(-1);
    p.a_rows_total = M;
    p.b_rows_total = N;
    p.debug_bad_coord = g_debug_bad_coord.exchange(-1);
    if (pair) {
        // the raster counts 256-row blocks within each group's plane
        const int pblocks = cdiv(M, fg::PAIR_ROWS);
        p.num_n_blocks = cdiv(N, fg::PAIR_BN);
        p.group_m = raster_group_m(fg::KIND_KGROUPED, pblocks, 2 * k_seg);
        p.idesc = fg::make_idesc_f8f6f4(fg::PAIR_ROWS, fg::PAIR_BN, (uint32_t)a_fmt, (uint32_t)b_fmt);
        const long long tiles = (long long)G * pblocks * p.num_n_blocks;
        const bool defer = kp.defer;
        long long clusters = defer ? PairDeferKernel<fg::KIND_KGROUPED>::max_active_clusters(2)
                                   : PairKernel<fg::KIND_KGROUPED, F32OUT>::max_active_clusters(2);
        if (clusters < 1) return cuda_fail();
        if (clusters > sms / 2) clusters = sms / 2;
        if (clusters > tiles) clusters = tiles;
        if constexpr (!F32OUT) {
            if (defer)
                return PairDeferKernel<fg::KIND_KGROUPED>::launch(ta, tb, td, tsa, p, (int)(2 * clusters), 2, stream);
        }
        return PairKernel<fg::KIND_KGROUPED, F32OUT>::launch(ta, tb, td, tsa, p, (int)(2 * clusters), 2, stream);
    }
    const long long tiles = (long long)G * p.num_m_blocks * p.num_n_blocks;
    const int grid = (int)(tiles < sms ? tiles : sms);
    if (BN == 128)
        return Kernel<128, fg::KIND_KGROUPED, false, F32OUT>::launch(ta, tb, td, tsa, p, grid, 1, stream);
    return Kernel<256, fg::KIND_KGROUPED, false, F32OUT>::launch(ta, tb, td, tsa, p, grid, 1, stream);
}

}  // namespace

namespace {
// The quantization kernel of one FP8 format and input type.
using QuantKernel = void (*)(const CUtensorMap, fg::QuantParams);
QuantKernel quantize_kernel(int fmt, int in) {
    if (in == fg::QUANT_IN_F32)
        return fmt == FG_E4M3 ? fg::quantize_per_token_kernel<0, fg::QUANT_IN_F32>
                              : fg::quantize_per_token_kernel<1, fg::QUANT_IN_F32>;
    return fmt == FG_E4M3 ? fg::quantize_per_token_kernel<0, fg::QUANT_IN_BF16>
                          : fg::quantize_per_token_kernel<1, fg::QUANT_IN_BF16>;
}

// Dynamic shared memory attribute of the quantization kernel and its resident
// CTAs per SM (occupancy query), once per device, format and input type; 0 on
// failure.
int quantize_blocks_per_sm(int fmt, int in) {
    static std::atomic<int> cache[kMaxDevices][2][2];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    const int v = cache[dev][fmt][in].load();
    if (v > 0) return v;
    const QuantKernel kernel = quantize_kernel(fmt, in);
    const int smem = fg::quant_smem_bytes(in);
    int n = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, fg::QUANT_THREADS, smem) != cudaSuccess ||
        n <= 0) {
        cudaGetLastError();
        return 0;
    }
    cache[dev][fmt][in].store(n);
    return n;
}

// Shared part of the quantization entry points; `in`: element type of X.
fg_status quantize(int in, const void *X, int ld_x, int fmt, void *A, float *sA, int ld_sA, const int32_t *masked_m,
                   int batches, int rows, int k, void *stream) {
    if (!X || !A || !sA || batches < 1 || rows < 0 || k < 1 || ld_x < k || ld_sA < rows || ld_sA < 1)
        return FG_ERR_INVALID_ARG;
    if (fmt != FG_E4M3 && fmt != FG_E5M2) return FG_ERR_INVALID_ARG;
    const int esize = in == fg::QUANT_IN_F32 ? 4 : 2;
    if (!aligned16(X) || !aligned16(A) || !aligned16(sA) || (ld_x * esize) % 16 != 0 || ld_sA % 4 != 0)
        return FG_ERR_MISALIGNED;
    if (k % 16 != 0) return FG_ERR_UNSUPPORTED;
    const int kb = cdiv(k, 128);
    if (kb > 65535 || batches > 65535) return FG_ERR_UNSUPPORTED;
    if (rows == 0) return FG_OK;
    const long long units = (long long)batches * cdiv(rows, fg::QUANT_ROWS) * kb;
    if (units > 0x7FFFFFFFLL - (1LL << 20)) return FG_ERR_UNSUPPORTED;  // unit index + grid stays in int
    DeviceInfo *dev = nullptr;
    if (fg_status st = device_info(&dev); st != FG_OK) return st;
    const int per_sm = quantize_blocks_per_sm(fmt, in);
    if (per_sm <= 0) return cuda_fail();
    int sms = dev->num_sms;
    const int ovr = g_num_sms_override.load();
    if (ovr > 0 && ovr < sms) sms = ovr;

    fg::QuantParams p{};
    p.x = X;
    p.a = static_cast<uint8_t *>(A);
    p.sa = sA;
    p.masked_m = masked_m;
    p.status = dev->status;
    p.ld_x = ld_x;
    p.ld_sa = ld_sA;
    p.rows = rows;
    p.k = k;
    p.kb = kb;
    p.timeout_ns = (unsigned long long)g_watchdog_ms.load() * 1000000ull;
    p.debug_skip_unit = g_debug_skip_iter.exchange(-1);
    p.row_blocks = cdiv(rows, fg::QUANT_ROWS);
    p.units = (int)units;

    // persistent CTAs: as many as are resident at once, each walks the units
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)std::min<long long>(units, (long long)sms * per_sm), 1, 1);
    cfg.blockDim = dim3(fg::QUANT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = fg::quant_smem_bytes(in);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute at[1];
    if (g_pdl.load() != 0) {
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
    }
    // X as a 3-D tensor {k, rows, batches}; one box = one unit (128 columns x 32 rows)
    CUtensorMap tx;
    {
        const uint64_t dims[3] = {(uint64_t)k, (uint64_t)rows, (uint64_t)batches};
        const uint64_t strides[2] = {(uint64_t)ld_x * esize, (uint64_t)ld_x * esize * (uint64_t)rows};
        const uint32_t box[3] = {128, (uint32_t)fg::QUANT_ROWS, 1};
        if (!encode(&tx, in == fg::QUANT_IN_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X,
                    3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cuda_fail();
    }
    const cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_kernel(fmt, in), tx, p);
    if (e != cudaSuccess) return cuda_fail();
    return cudaPeekAtLastError() == cudaSuccess ? FG_OK : cuda_fail();
}
}  // namespace

extern "C" {

fg_status fg_gemm_fp8_nt(const void *A, int a_fmt, const float *sA, int ld_sA, const void *B, int b_fmt,
                         const float *sB, void *D, int m, int n, int k, void *stream) {
    return run<fg::KIND_DENSE>(A, a_fmt, sA, ld_sA, B, b_fmt, sB, D, nullptr, nullptr, m, 1, n, k,
                               static_cast<cudaStream_t>(stream));
}

fg_status fg_grouped_gemm_fp8_contiguous(const void *A, int a_fmt, const float *sA, int ld_sA, const void *B,
                                         int b_fmt, const float *sB, void *D, const int32_t *m_indices, int M,
                                         int n, int k, int G, void *stream) {
    return run<fg::KIND_CONTIGUOUS>(A, a_fmt, sA, ld_sA, B, b_fmt, sB, D, m_indices, nullptr, M, G, n, k,
                                    static_cast<cudaStream_t>(stream));
}

fg_status fg_grouped_gemm_fp8_masked(const void *A, int a_fmt, const float *sA, int ld_sA, const void *B,
                                     int b_fmt, const float *sB, void *D, const int32_t *masked_m, int G,
                                     int M_cap, int n, int k, void *stream) {
    return run<fg::KIND_MASKED>(A, a_fmt, sA, ld_sA, B, b_fmt, sB, D, nullptr, masked_m, M_cap, G, n, k,
                                static_cast<cudaStream_t>(stream));
}

fg_status fg_gemm_fp8_nt_f32out(const void *A, int a_fmt, const float *sA, int ld_sA, const void *B, int b_fmt,
                                const float *sB, float *D, int m, int n, int k, void *stream) {
    return run<fg::KIND_DENSE, true>(A, a_fmt, sA, ld_sA, B, b_fmt, sB, D, nullptr, nullptr, m, 1, n, k,
                                     static_cast<cudaStream_t>(stream));
}

fg_status fg_grouped_gemm_fp8_contiguous_f32out(const void *A, int a_fmt, const float *sA, int ld_sA,
                                                const void *B, int b_fmt, const float *sB, float *D,
                                                const int32_t *m_indices, int M, int n, int k, int G,
                                                void *stream) {
    return run<fg::KIND_CONTIGUOUS, true>(A, a_fmt, sA, ld_sA, B, b_fmt, sB, D, m_indices, nullptr, M, G, n, k,
                                          static_cast<cudaStream_t>(stream));
}

fg_status fg_grouped_gemm_fp8_masked_f32out(const void *A, int a_fmt, const float *sA, int ld_sA, const void *B,
                                            int b_fmt, const float *sB, float *D, const int32_t *masked_m, int G,
                                            int M_cap, int n, int k, void *stream) {
    return run<fg::KIND_MASKED, true>(A, a_fmt, sA, ld_sA, B, b_fmt, sB, D, nullptr, masked_m, M_cap, G, n, k,
                                      static_cast<cudaStream_t>(stream));
}

fg_status fg_k_grouped_gemm_fp8_nt(const void *A, int a_fmt, const float *sA, int ld_sA, const void *B, int b_fmt,
                                   const float *sB, void *D, const int32_t *k_sizes, int G, int M, int N, int K,
                                   void *stream) {
    return run_kgrouped<false>(A, a_fmt, sA, ld_sA, B, b_fmt, sB, D, k_sizes, G, M, N, K,
                               static_cast<cudaStream_t>(stream));
}

fg_status fg_k_grouped_gemm_fp8_nt_f32out(const void *A, int a_fmt, const float *sA, int ld_sA, const void *B,
                                          int b_fmt, const float *sB, float *D, const int32_t *k_sizes, int G,
                                          int M, int N, int K, void *stream) {
    return run_kgrouped<true>(A, a_fmt, sA, ld_sA, B, b_fmt, sB, D, k_sizes, G, M, N, K,
                              static_cast<cudaStream_t>(stream));
}

fg_status fg_scales_a_to_mn_major(const float *src, float *dst, int batches, int rows, int kb, int ld_dst,
                                  void *stream) {
    if (!src || !dst || batches < 1 || rows < 0 || kb < 1 || ld_dst < rows || ld_dst < 1) return FG_ERR_INVALID_ARG;
    if (ld_dst % 4 != 0) return FG_ERR_MISALIGNED;
    if (kb > 65535 || batches > 65535) return FG_ERR_UNSUPPORTED;
    dim3 grid((unsigned)cdiv(ld_dst, 256), (unsigned)kb, (unsigned)batches);
    fg::scales_to_mn_major_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(src, dst, rows, kb, ld_dst);
    return cudaPeekAtLastError() == cudaSuccess ? FG_OK : FG_ERR_CUDA;
}

fg_status fg_quantize_fp8_per_token(const void *X, int ld_x, int fmt, void *A, float *sA, int ld_sA,
                                    const int32_t *masked_m, int batches, int rows, int k, void *stream) {
    return quantize(fg::QUANT_IN_BF16, X, ld_x, fmt, A, sA, ld_sA, masked_m, batches, rows, k, stream);
}

fg_status fg_quantize_fp8_per_token_f32in(const float *X, int ld_x, int fmt, void *A, float *sA, int ld_sA,
                                          const int32_t *masked_m, int batches, int rows, int k, void *stream) {
    return quantize(fg::QUANT_IN_F32, X, ld_x, fmt, A, sA, ld_sA, masked_m, batches, rows, k, stream);
}

int fg_scales_a_ld(int rows) { return rows <= 0 ? 4 : (rows + 3) / 4 * 4; }

fg_status fg_get_device_status(void *stream, uint32_t *detail) {
    DeviceInfo *dev = nullptr;
    if (fg_status st = device_info(&dev); st != FG_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FG_ERR_CUDA;
    uint32_t host[2] = {0, 0};
    if (cudaMemcpyFromSymbol(host, g_status, sizeof(host)) != cudaSuccess) return FG_ERR_CUDA;
    const uint32_t zero[2] = {0, 0};
    if (cudaMemcpyToSymbol(g_status, zero, sizeof(zero)) != cudaSuccess) return FG_ERR_CUDA;
    if (detail) *detail = host[1];
    return static_cast<fg_status>(host[0]);
}

fg_status fg_set_num_sms(int num_sms) {
    if (num_sms < 0) return FG_ERR_INVALID_ARG;
    g_num_sms_override.store(num_sms);
    return FG_OK;
}

fg_status fg_query_dense_plan(int m, int n, int k, int *block_n, int *split_k) {
    if (m < 1 || n < 1 || k < 1 || !block_n || !split_k) return FG_ERR_INVALID_ARG;
    DeviceInfo *dev = nullptr;
    if (fg_status st = device_info(&dev); st != FG_OK) return st;
    int sms = dev->num_sms;
    const int ovr = g_num_sms_override.load();
    if (ovr > 0 && ovr < sms) sms = ovr;
    const Plan plan = choose_plan(cdiv(m, fg::BLOCK_M), m, n, k, sms);
    *block_n = plan.bn;
    *split_k = plan.split;
    return FG_OK;
}

fg_status fg_query_dense_plan_ex(int m, int n, int k, int *block_n, int *split_k, int *cta_pair) {
    if (!cta_pair) return FG_ERR_INVALID_ARG;
    const fg_status st = fg_query_dense_plan(m, n, k, block_n, split_k);
    if (st != FG_OK) return st;
    Plan plan;
    plan.bn = *block_n;
    plan.split = *split_k;
    *cta_pair = use_pair(fg::KIND_DENSE, plan, m) && g_num_sms_override.load() != 1 ? 1 : 0;
    return FG_OK;
}

fg_status fg_query_plan(int kind, int rows, int G, int n, int k, int *plan) {
    if (!plan || rows < 1 || G < 1 || n < 1 || k < 1 || kind < fg::KIND_DENSE || kind > fg::KIND_KGROUPED)
        return FG_ERR_INVALID_ARG;
    if (kind == fg::KIND_DENSE && G != 1) return FG_ERR_INVALID_ARG;
    DeviceInfo *dev = nullptr;
    if (fg_status st = device_info(&dev); st != FG_OK) return st;
    int sms = dev->num_sms;
    const int ovr = g_num_sms_override.load();
    if (ovr > 0 && ovr < sms) sms = ovr;
    if (kind == fg::KIND_KGROUPED) {
        const KgPlan kp = kgrouped_plan(G, rows, n, k, sms, false);
        plan[0] = kp.bn;
        plan[1] = 1;
        plan[2] = kp.pair ? 1 : 0;
        plan[3] = 0;
        plan[4] = kp.defer ? 1 : 0;
        return FG_OK;
    }
    SwapPlan sp;
    plan[4] = 0;
    if (kind != fg::KIND_CONTIGUOUS && swap_applies(kind, rows, G, n, k, sms, &sp)) {
        plan[0] = sp.bt;
        plan[1] = sp.split;
        plan[2] = 0;
        plan[3] = 1;
        return FG_OK;
    }
    const long long m_blocks = (long long)cdiv(rows, fg::BLOCK_M) * (kind == fg::KIND_MASKED ? G : 1);
    const Plan p = choose_plan(m_blocks, kind == fg::KIND_DENSE ? rows : INT32_MAX, n, k, sms);
    plan[0] = p.bn;
    plan[1] = p.split;
    plan[2] = use_pair(kind, p, rows) && sms >= 2 ? 1 : 0;
    plan[3] = 0;
    const int dmode = g_pair_defer.load();
    plan[4] = plan[2] && (dmode == 1 || (dmode < 0 && cdiv(k, fg::BLOCK_K) <= kPairDeferMaxKb)) ? 1 : 0;
    return FG_OK;
}

fg_status fg_set_pair_mode(int mode) {
    if (mode < -1 || mode > 1) return FG_ERR_INVALID_ARG;
    g_pair_mode.store(mode);
    return FG_OK;
}

fg_status fg_set_swap_mode(int mode) {
    if (mode < -1 || mode > 1) return FG_ERR_INVALID_ARG;
    g_swap_mode.store(mode);
    return FG_OK;
}

fg_status fg_set_programmatic_launch(int enable) {
    g_pdl.store(enable ? 1 : 0);
    return FG_OK;
}

fg_status fg_set_config_override(int block_n, int split_k) {
    if ((block_n != 0 && block_n != 128 && block_n != 256) || split_k < 0 || split_k > 8)
        return FG_ERR_INVALID_ARG;
    g_force_bn.store(block_n);
    g_force_split.store(split_k);
    return FG_OK;
}

fg_status fg_set_watchdog_ms(uint32_t ms) {
    g_watchdog_ms.store(ms == 0 ? kDefaultWatchdogMs : ms);
    return FG_OK;
}

// Test hook of the debug build (not part of the public header): in the next
// GEMM call, the producer of every CTA moves the A load of its K iteration
// `iter` past K; the debug build's bounds check catches it before the load is
// issued (records FG_ERR_DEVICE_CHECK, tag 0x41).  The release build ignores
// the hook (FG_ERR_UNSUPPORTED).
fg_status fg_debug_bad_coordinate(int iter) {
    if (!fg::kDebugBuild) return FG_ERR_UNSUPPORTED;
    g_debug_bad_coord.store(iter);
    return FG_OK;
}

// Whether this library is the debug build (FG_DEBUG): 1 or 0.
int fg_debug_build(void) { return fg::kDebugBuild ? 1 : 0; }

// Test hook (not part of the public header): in the next GEMM call, the
// producer of every CTA leaves its K iteration `iter` unarmed, so the MMA
// warp's bounded wait expires and the call reports FG_ERR_TIMEOUT; in the next
// quantization call, every CTA's producer leaves its unit number `iter`
// unfilled, with the same outcome for the consumer warps.
// Test and measurement hook (not part of the public header): CTA-pair tiles
// with BF16 output stage a whole tile and let an eleventh warp issue its
// stores (1), stage box by box and store from the promotion warps (0), or
// choose by the number of K blocks (-1, the default).
fg_status fg_debug_set_pair_defer(int mode) {
    if (mode < -1 || mode > 1) return FG_ERR_INVALID_ARG;
    g_pair_defer.store(mode);
    return FG_OK;
}

fg_status fg_debug_skip_producer_iteration(int iter) {
    g_debug_skip_iter.store(iter);
    return FG_OK;
}

const char *fg_status_string(int status) {
    switch (status) {
        case FG_OK: return "FG_OK";
        case FG_ERR_INVALID_ARG: return "FG_ERR_INVALID_ARG";
        case FG_ERR_MISALIGNED: return "FG_ERR_MISALIGNED";
        case FG_ERR_UNSUPPORTED: return "FG_ERR_UNSUPPORTED";
        case FG_ERR_CUDA: return "FG_ERR_CUDA";
        case FG_ERR_TIMEOUT: return "FG_ERR_TIMEOUT";
        case FG_ERR_DEVICE_CHECK: return "FG_ERR_DEVICE_CHECK";
        default: return "FG_ERR_UNKNOWN";
    }
}

int fg_version(void) { return 100; }

}  // extern "C"
