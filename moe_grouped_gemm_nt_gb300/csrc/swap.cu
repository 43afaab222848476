// swap.cu -- plan and launch of the swapped-operand FP8 NT GEMM
// (gemm_swap_kernel.cuh): the weights take the MMA's 128-row role and the few
// rows of A (tokens) its N role, for the dense layout with at most 256 rows and
// the masked layout with a capacity of at most 256 rows per group.
#include "swap.h"

#include "gemm_swap_kernel.cuh"

namespace fgh {

namespace {

// Operand stages: 6 of 16 + 16 KB for 128-token tiles, 3 of 16 + 32 KB for
// 256-token tiles (with the staging buffers and the 4-deep scale ring, the
// most that fits in 227 KB of shared memory).  The debug build: one stage, or
// for split-K the fewest that hold the FP32 partial tile.
template <int BT, bool SPLITK>
constexpr int swap_stages() {
    if (fg::kDebugBuild) return SPLITK ? (BT == 256 ? 3 : 2) : 1;
    return BT == 256 ? 3 : 6;
}

template <int BT, int KIND, bool SPLITK, bool F32OUT>
using SwapKernel = Launcher<fg::fp8_gemm_swap_kernel<BT, swap_stages<BT, SPLITK>(), KIND, SPLITK, F32OUT>,
                            fg::SwapSmemLayout<BT, swap_stages<BT, SPLITK>()>::BYTES, SPLITK>;

// Estimated time (us) of a swapped plan, in the form of the one-CTA plan model
// (start-up + the larger of HBM time and per-SM operand intake + split-K
// exchange through distributed shared memory).
double swap_cost(int kind_rows, int G, int n, int k, int bt, int split) {
    const double kb = (double)((k + 127) / 128);
    const double rows = kind_rows < bt ? kind_rows : bt;
    const double hbm_us = ((double)G * n * k + (double)G * kind_rows * k + (double)G * kind_rows * n * 2.0) / 6.5e6;
    const double intake_us = std::ceil(kb / split) * (16384.0 + 128.0 * bt) / 9.0e4;
    const double red_us = split > 1 ? 1.0 + 128.0 * rows * 4.0 * (split - 1) / split / 3.4e4 : 0.0;
    return 3.5 + std::max(hbm_us, intake_us) + red_us;
}

template <int BT, int KIND>
int max_clusters(int split, bool f32out) {
    return f32out ? SwapKernel<BT, KIND, true, true>::max_active_clusters(split)
                  : SwapKernel<BT, KIND, true, false>::max_active_clusters(split);
}

template <int KIND>
SwapPlan plan_for(int rows, int G, int n, int k, int sms) {
    SwapPlan plan;
    plan.bt = rows <= 128 ? 128 : 256;
    const long long tiles = (long long)G * ((rows + plan.bt - 1) / plan.bt) * ((n + 127) / 128);
    const int num_kb = (k + 127) / 128;
    const int forced = g_force_split.load();
    if (forced > 0) {
        plan.split = forced;
        return plan;
    }
    if (tiles * 4 >= (long long)sms * 3) return plan;  // enough tiles: persistent, no split
    double best = swap_cost(rows, G, n, k, plan.bt, 1);
    for (int sp = 2; sp <= 8; ++sp) {
        if (num_kb < 2 * sp) break;  // at least two K blocks per rank
        const int clusters = plan.bt == 256 ? max_clusters<256, KIND>(sp, false) : max_clusters<128, KIND>(sp, false);
        long long cap = (long long)sp * clusters;
        if (cap > (long long)(sms / sp) * sp) cap = (long long)(sms / sp) * sp;
        if (cap <= 0 || tiles * sp > cap) continue;  // one wave of clusters
        const double c = swap_cost(rows, G, n, k, plan.bt, sp);
        if (c < best) {
            best = c;
            plan.split = sp;
        }
    }
    return plan;
}

template <int BT, int KIND, bool F32OUT>
fg_status launch(const SwapPlan &plan, const CUtensorMap &tw, const CUtensorMap &tt, const CUtensorMap &td,
                 const CUtensorMap &tts, const GemmParams &p, long long tiles, int sms, cudaStream_t stream) {
    if (plan.split > 1) {
        const long long grid = tiles * plan.split;
        if (grid > INT32_MAX) return FG_ERR_UNSUPPORTED;
        return SwapKernel<BT, KIND, true, F32OUT>::launch(tw, tt, td, tts, p, (int)grid, plan.split, stream);
    }
    const int grid = (int)(tiles < sms ? tiles : sms);
    return SwapKernel<BT, KIND, false, F32OUT>::launch(tw, tt, td, tts, p, grid, 1, stream);
}

}  // namespace

bool swap_applies(int kind, int rows, int G, int n, int k, int sms, SwapPlan *plan) {
    if (kind != fg::KIND_DENSE && kind != fg::KIND_MASKED) return false;
    if (rows < 1 || rows > 256) return false;
    // automatic choice (-1): never.  Measured on the dense sweep's m <= 128
    // problems and the masked workloads (capacity 256, 1..16 groups), the
    // swapped path is 10-100% slower than the one-CTA plans on every problem:
    // a tile covers 128 weight rows (the MMA's M), so the rows of A are read
    // again for every 128 weights instead of every 256, and the per-column
    // scales cost promotion instructions; only mode 1 selects it.
    if (g_swap_mode.load() != 1) return false;
    *plan = kind == fg::KIND_MASKED ? plan_for<fg::KIND_MASKED>(rows, G, n, k, sms)
                                    : plan_for<fg::KIND_DENSE>(rows, G, n, k, sms);
    return true;
}

fg_status launch_swap(int kind, bool f32out, const SwapPlan &plan, const void *A, int a_fmt, const float *sA,
                      int ld_sA, const void *B, int b_fmt, const float *sB, void *D, const int32_t *masked_m,
                      int rows, int G, int n, int k, int sms, const DeviceInfo *dev, cudaStream_t stream) {
    const bool masked = kind == fg::KIND_MASKED;
    const int bt = plan.bt;
    const int num_kb = cdiv(k, fg::BLOCK_K);
    const uint64_t rows_total = masked ? (uint64_t)G * rows : (uint64_t)rows;
    CUtensorMap tw, tt, td, tts;
    // token scales, MN-major: 2-D {rows, kb} (dense) or 3-D {M_cap, kb, G}; box of bt rows
    const uint64_t sdims[3] = {(uint64_t)rows, (uint64_t)num_kb, (uint64_t)G};
    const uint64_t sstrides[2] = {(uint64_t)ld_sA * 4, (uint64_t)ld_sA * 4 * (uint64_t)num_kb};
    const uint32_t sbox[3] = {(uint32_t)bt, 1, 1};
    // D: [rows_total][n], boxes of 32 columns x 32 rows, written token-major
    const uint64_t ddims[2] = {(uint64_t)n, rows_total};
    const uint64_t dstrides[1] = {(uint64_t)n * (f32out ? 4 : 2)};
    const uint32_t dbox[2] = {32, 32};
    if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, (uint64_t)k, (uint64_t)G * n, (uint64_t)k, fg::BLOCK_K,
                   fg::BLOCK_M) ||
        !encode_2d(&tt, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, (uint64_t)k, rows_total, (uint64_t)k, fg::BLOCK_K,
                   (uint32_t)bt) ||
        !encode(&tts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sA, masked ? 3 : 2, sdims, sstrides, sbox,
                CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode(&td, f32out ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, 2, ddims,
                dstrides, dbox, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cuda_fail();

    GemmParams p{};
    p.rows = rows;
    p.n = n;
    p.k = k;
    p.num_groups = G;
    p.num_kb = num_kb;
    p.num_nb = cdiv(n, 128);
    p.num_n_blocks = cdiv(n, fg::BLOCK_M);  // 128-row weight blocks
    p.num_m_blocks = cdiv(rows, bt);        // token blocks per group
    p.group_m = 1;
    // the MMA's A operand is the weights (B's format), its B operand the tokens
    p.idesc = fg::make_idesc_f8f6f4(fg::BLOCK_M, bt, (uint32_t)b_fmt, (uint32_t)a_fmt);
    p.sB = sB;
    p.masked_m = masked_m;
    p.D = D;
    p.status = dev->status;
    p.timeout_ns = (unsigned long long)g_watchdog_ms.load() * 1000000ull;
    p.debug_skip_iter = g_debug_skip_iter.exchange(-1);
    const long long tiles = (long long)(masked ? G : 1) * p.num_m_blocks * p.num_n_blocks;

    if (bt == 256) {
        if (masked)
            return f32out ? launch<256, fg::KIND_MASKED, true>(plan, tw, tt, td, tts, p, tiles, sms, stream)
                          : launch<256, fg::KIND_MASKED, false>(plan, tw, tt, td, tts, p, tiles, sms, stream);
        return f32out ? launch<256, fg::KIND_DENSE, true>(plan, tw, tt, td, tts, p, tiles, sms, stream)
                      : launch<256, fg::KIND_DENSE, false>(plan, tw, tt, td, tts, p, tiles, sms, stream);
    }
    if (masked)
        return f32out ? launch<128, fg::KIND_MASKED, true>(plan, tw, tt, td, tts, p, tiles, sms, stream)
                      : launch<128, fg::KIND_MASKED, false>(plan, tw, tt, td, tts, p, tiles, sms, stream);
    return f32out ? launch<128, fg::KIND_DENSE, true>(plan, tw, tt, td, tts, p, tiles, sms, stream)
                  : launch<128, fg::KIND_DENSE, false>(plan, tw, tt, td, tts, p, tiles, sms, stream);
}

}  // namespace fgh
