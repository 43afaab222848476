// gemm_pair_kernel.cuh -- the persistent FP8 NT GEMM on CTA pairs (cta_group::2).
//
// Same method as gemm_kernel.cuh (page "DeepSeek开源周第三天DeepGEMM",
// "两级精度累加与细粒度缩放": one 128-deep K block on the tensor cores into a
// fresh FP32 partial, scaled by sA * sB and added on the CUDA cores), on output
// tiles of 256 x 256 shared by the two CTAs (two SMs) of a cluster:
//
//   * CTA rank r holds rows [r*128, r*128+128) of the tile's A block and rows
//     [r*128, r*128+128) of the tile's 256 B rows, so each SM brings in 32 KB
//     per K block instead of 48 KB for a 128 x 256 tile; the same shared memory
//     then holds more stages (five, with an eight-deep scale ring: the
//     producer issues both in the same iteration, so its lookahead is the
//     shallower of the two).
//   * The even CTA's MMA warp issues tcgen05.mma.cta_group::2 (M = 256,
//     N = 256, K = 32); each CTA's TMEM receives its 128 rows x 256 columns.
//     Both CTAs' operand loads signal the even CTA's `full[s]`; its commits
//     arrive on `empty[s]` and `tmem_full[b]` of both CTAs (multicast).
//   * Each CTA's promotion warps promote and store their own 128 rows exactly
//     like the one-CTA kernel; they hand the TMEM buffer back by arriving on
//     the even CTA's `tmem_empty[b]` (16 arrivals: 8 warps per CTA).
//
// Dense, masked, K-grouped and contiguous layouts (the masked walk pairs
// 128-row blocks inside a group; rows past a group's count are loaded but
// never stored).  Contiguous layout: a pair tile covers 128-row blocks 2p and
// 2p + 1, which may belong to different groups (segments are 128-aligned) and
// one MMA multiplies both by one group's weights, so a tile takes one pass per
// group present: the group of block 2p, then that of block 2p + 1 if it is
// another; a pass stores only the rows of its group (the group id of each row
// decides, which also leaves the -1 padding rows untouched).  Every wait
// is bounded by the same watchdog as the one-CTA kernel; both CTAs always
// reach the final cluster barrier, so neither leaves while the other (or the
// even CTA's MMAs) may still use its shared memory or TMEM.
#pragma once

#include "gemm_kernel.cuh"

namespace fg {

constexpr int PAIR_BN = 256;         // N of the pair tile = columns of each CTA's accumulator
constexpr int PAIR_ROWS = 2 * BLOCK_M;  // M of the pair tile

// Deferred stores (DEFER): an eleventh warp issues the epilogue's TMA stores, so
// the promotion warps stage a whole tile (both 64-column boxes of each warp)
// and go straight on to the next tile.
constexpr int STORE_WARP = 10;
constexpr int PAIR_DEFER_THREADS = 352;

template <int STAGES, int SS, bool DEFER = false>
struct PairSmemLayout {
    static constexpr int HB_STAGE_BYTES = (PAIR_BN / 2) * BLOCK_K;  // this CTA's half of B
    static constexpr int STG_PER_WARP = DEFER ? 2 * STAGING_BYTES_PER_WARP : STAGING_BYTES_PER_WARP;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = A_OFF + STAGES * A_STAGE_BYTES;
    static constexpr int STG_OFF = B_OFF + STAGES * HB_STAGE_BYTES;
    static constexpr int SA_OFF = STG_OFF + NUM_EPI_WARPS * STG_PER_WARP;
    static constexpr int SB_OFF = SA_OFF + SS * SA_STAGE_BYTES;
    static constexpr int BAR_OFF = SB_OFF + SS * SB_STAGE_BYTES;
    static constexpr int NUM_TBUF = 2;
    // full, empty, scale_full, scale_empty, tmem_full, tmem_empty, drain
    // (DEFER: + staging_full, staging_empty)
    static constexpr int NUM_BARS = 2 * STAGES + 2 * SS + 2 * NUM_TBUF + 1 + (DEFER ? 2 : 0);
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    // TMEM address, abort flag, DEFER: one byte per promotion warp (1 = its rows
    // of the tile are staged for the store warp, 0 = stored row by row)
    static constexpr int BYTES = MISC_OFF + 8 + NUM_EPI_WARPS;
    static constexpr int TMEM_COLS = 512;
};

struct PairTile {
    int valid;
    int group;
    int n_blk;      // 256-column block
    int a_row;      // first row of this CTA's half in the 2-D row space of A and D
    int sa_row;     // same, as the row coordinate of the scale tensor map
    int b_row;      // first row of this CTA's half of B in the 2-D row space [G*n][k]
    int row_limit;  // rows of this CTA's half below the bound (<= 0: none)
    int kb_lo, kb_hi;  // K-grouped layout: the tile's K blocks (its group's segment)
    int own_group;     // contiguous layout: group id of the first row of this CTA's block (-2: past M)
    int own_pass;      // contiguous layout: this pass is the one of this CTA's block
};

// Passes per pair tile: the contiguous layout may need one per group of its
// two 128-row blocks; the walk runs over v = tile * PASSES + pass.
template <int KIND>
__host__ __device__ constexpr int pair_passes() { return KIND == KIND_CONTIGUOUS ? 2 : 1; }

// 256-row blocks of the whole walk (masked: of all groups' counts).
template <int KIND>
__device__ __forceinline__ int total_pair_blocks(const GemmParams &p) {
    if constexpr (KIND == KIND_MASKED) {
        int pb = 0;
        for (int g = 0; g < p.num_groups; ++g)
            pb += (clamp_count(__ldg(p.masked_m + g), p.rows) + PAIR_ROWS - 1) / PAIR_ROWS;
        return pb;
    } else {
        return (p.rows + PAIR_ROWS - 1) / PAIR_ROWS;
    }
}

// Pass v of the walk: pair tile t = v / pair_passes<KIND>() (cluster c takes
// tiles c, c + clusters, ...), the half of CTA `rank`; the raster is that of
// get_tile() over 256-row blocks.  K-grouped layout: the tiles of group g
// (every 256-row block of its output plane) before those of group g + 1, the K
// range from the forward scan of get_tile().
template <int KIND>
__device__ __forceinline__ PairTile get_pair_tile(const GemmParams &p, int v, int pblocks, uint32_t rank,
                                                  GroupScan &scan) {
    PairTile ti;
    ti.kb_lo = 0;
    ti.kb_hi = p.num_kb;
    ti.group = 0;
    ti.own_group = 0;
    ti.own_pass = 1;
    int t = v, pass = 0;
    if constexpr (KIND == KIND_CONTIGUOUS) {
        t = v >> 1;
        pass = v & 1;
    }
    if constexpr (KIND == KIND_KGROUPED) {
        const int per_g = pblocks * p.num_n_blocks;
        const int g = t / per_g;
        t -= g * per_g;
        if (g < scan.g) scan = GroupScan{};
        while (scan.g < g) scan.first += k_segment_blocks(p, scan.g++);
        ti.kb_lo = min(scan.first, p.num_kb);
        ti.kb_hi = min(scan.first + k_segment_blocks(p, g), p.num_kb);
        ti.group = g;
    }
    const int per_group = p.group_m * p.num_n_blocks;
    const int grp = t / per_group;
    const int rem = t - grp * per_group;
    const int m0 = grp * p.group_m;
    const int gm = min(p.group_m, pblocks - m0);
    const int pb_lin = m0 + rem % gm;
    ti.n_blk = rem / gm;
    const int half = (int)rank * BLOCK_M;
    if constexpr (KIND == KIND_MASKED) {
        // the group holding valid 256-row block pb_lin, by the role's forward scan
        if (pb_lin < scan.first) scan = GroupScan{};
        int g = scan.g, acc = scan.first, cnt = 0;
        for (; g < p.num_groups; ++g) {
            cnt = clamp_count(__ldg(p.masked_m + g), p.rows);
            const int nb = (cnt + PAIR_ROWS - 1) / PAIR_ROWS;
            if (pb_lin < acc + nb) break;
            acc += nb;
        }
        scan.g = g;
        scan.first = acc;
        ti.valid = g < p.num_groups;
        ti.group = g;
        const int row0 = (pb_lin - acc) * PAIR_ROWS + half;  // within the group
        ti.a_row = g * p.rows + row0;
        ti.sa_row = row0;
        ti.b_row = g * p.n + ti.n_blk * PAIR_BN + half;
        ti.row_limit = min(BLOCK_M, cnt - row0);
    } else if constexpr (KIND == KIND_CONTIGUOUS) {
        // the groups of the tile's two 128-row blocks (first rows); pass 0 runs
        // with the first block's group, pass 1 with the second's when it differs
        const int blk0 = pb_lin * 2;
        const int g0 = __ldg(p.m_indices + (size_t)blk0 * BLOCK_M);
        const int g1 = (blk0 + 1) * BLOCK_M < p.rows ? __ldg(p.m_indices + (size_t)(blk0 + 1) * BLOCK_M) : -2;
        const bool v0 = g0 >= 0 && g0 < p.num_groups;
        const bool v1 = g1 >= 0 && g1 < p.num_groups && g1 != g0;
        const int g = pass == 0 ? g0 : g1;
        ti.valid = pass == 0 ? v0 : v1;
        ti.group = g;
        ti.own_group = rank == 0 ? g0 : g1;
        ti.own_pass = pass == (int)rank;
        const int row0 = pb_lin * PAIR_ROWS + half;
        ti.a_row = row0;
        ti.sa_row = row0;
        ti.b_row = (ti.valid ? g : 0) * p.n + ti.n_blk * PAIR_BN + half;
        ti.row_limit = min(BLOCK_M, p.rows - row0);
    } else {
        // dense, or K-grouped (A and B shared by the groups; the group picks
        // the K range and the output plane)
        ti.valid = 1;
        const int row0 = pb_lin * PAIR_ROWS + half;
        ti.a_row = row0;
        ti.sa_row = row0;
        ti.b_row = ti.n_blk * PAIR_BN + half;
        ti.row_limit = min(BLOCK_M, p.rows - row0);
    }
    return ti;
}

// Tensor maps: A [rows][k] u8 (box 128 rows), B [G*n][k] u8 (box 128 rows: one
// CTA's half of the pair tile's 256), D [rows][n] bf16 or (F32OUT) fp32, SA as
// for the one-CTA kernel.  Launched with clusters of 2 CTAs (DEFER: 352
// threads per CTA, the eleventh warp issuing the epilogue's stores).
template <int KIND, int STAGES, int SS, bool F32OUT, bool DEFER = false>
__global__ void __launch_bounds__(DEFER ? PAIR_DEFER_THREADS : NUM_THREADS, 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ CUtensorMap tmap_sa,
                         const GemmParams p) {
    // rows of D past the bound are clipped by the tensor map (no per-row stores)
    constexpr bool CLIPPED = KIND == KIND_DENSE || KIND == KIND_KGROUPED;
    constexpr int PASSES = pair_passes<KIND>();
    static_assert((SS & (SS - 1)) == 0, "scale ring size");
    static_assert(!(DEFER && F32OUT), "deferred stores: BF16 output");
    using L = PairSmemLayout<STAGES, SS, DEFER>;
    constexpr int BN = PAIR_BN;
    constexpr int COLS = BN / 2;  // columns per promotion warp
    // TMEM columns loaded per tcgen05.wait::ld: the warp's whole share, so a K
    // block's partial reaches registers behind one wait and its buffer goes back
    // to the MMA warp sooner (dense: 162 registers, no spills; 1.6% less time
    // over the dense m = 4096 problems than four waits of 32 columns, bitwise the
    // same).  The debug build keeps 32 (its finite-value check on every loaded
    // column would otherwise spill).
    constexpr int LD_COLS = kDebugBuild ? TMEM_LD_COLS : COLS;
    constexpr uint32_t NTB = L::NUM_TBUF;
    // bytes of one stage of both CTAs, all signalled on the even CTA's full[s]
    constexpr uint32_t PAIR_TX = 2u * (A_STAGE_BYTES + L::HB_STAGE_BYTES);
    constexpr uint16_t BOTH = 0x3;

    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);

    const uint32_t bar0 = sbase + L::BAR_OFF;
    auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (STAGES + s); };
    auto sfull_bar = [&](uint32_t q) { return bar0 + 8u * (2 * STAGES + q); };
    auto sempty_bar = [&](uint32_t q) { return bar0 + 8u * (2 * STAGES + SS + q); };
    auto tfull_bar = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + 2 * SS + b); };
    auto tempty_bar = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + 2 * SS + NTB + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * SS + 2 * NTB);
    const uint32_t stg_full_bar = drain_bar + 8u;    // DEFER: the tile's boxes are staged
    const uint32_t stg_empty_bar = drain_bar + 16u;  // DEFER: their stores have read the staging
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + L::MISC_OFF + 4);
    volatile uint8_t *staged = smem + L::MISC_OFF + 8;  // DEFER, not CLIPPED: per promotion warp

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    // Both CTAs run the same code on the same layout, so both see the same
    // alignment and either both return here or neither does.
    if (sbase & 1023u) {
        if (threadIdx.x == 0) record_error(p, DEV_ERR_CHECK, (ROLE_SETUP << 24) | (sbase & 0xFFFFu));
        return;
    }

    // ------------------------------------------------------------- set-up
    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            prefetch_tensormap(&tmap_a);
            prefetch_tensormap(&tmap_b);
            prefetch_tensormap(&tmap_sa);
            prefetch_tensormap(&tmap_d);
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(full_bar(s), 1);   // the even CTA's expect_tx arrival (+ both CTAs' bytes)
                mbar_init(empty_bar(s), 1);  // one multicast commit
            }
            for (int q = 0; q < SS; ++q) {
                mbar_init(sfull_bar(q), 2);
                mbar_init(sempty_bar(q), NUM_EPI_WARPS);
            }
            for (uint32_t b = 0; b < NTB; ++b) {
                mbar_init(tfull_bar(b), 1);
                mbar_init(tempty_bar(b), 2 * NUM_EPI_WARPS);  // both CTAs' promotion warps
            }
            mbar_init(drain_bar, 1);
            if constexpr (DEFER) {
                mbar_init(stg_full_bar, NUM_EPI_WARPS);
                mbar_init(stg_empty_bar, 1);
            }
            *abort_flag = 0u;
            fence_mbarrier_init();
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        tmem_alloc_pair(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish_pair();
    }
    // barriers initialized and TMEM allocated in both CTAs before any use
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    griddep_wait();
    griddep_launch_dependents();
    if constexpr (KIND == KIND_MASKED) {
        if (blockIdx.x == 0 && warp == 0) {
            for (int g = lane; g < p.num_groups; g += 32) {
                const int c = __ldg(p.masked_m + g);
                if (c < 0 || c > p.rows) record_error(p, DEV_ERR_CHECK, (uint32_t)g);
            }
        }
    }
    if constexpr (KIND == KIND_KGROUPED) {
        // segment lengths: multiples of 128 that fit in K (others are reported)
        if (blockIdx.x == 0 && warp == 0 && lane == 0) {
            long long total = 0;
            for (int g = 0; g < p.num_groups; ++g) {
                const int c = __ldg(p.k_sizes + g);
                if (c < 0 || c % BLOCK_K != 0) record_error(p, DEV_ERR_CHECK, (uint32_t)g);
                total += c > 0 ? c : 0;
            }
            if (total > p.k) record_error(p, DEV_ERR_CHECK, (uint32_t)p.num_groups);
        }
    }

    const int pblocks = total_pair_blocks<KIND>(p);
    const int num_tiles = pblocks * p.num_n_blocks * (KIND == KIND_KGROUPED ? p.num_groups : 1);
    const int t_begin = (int)(blockIdx.x >> 1), t_step = (int)(gridDim.x >> 1);
    // the walk: passes v = t * PASSES + pass of this cluster's tiles t
    const int v_begin = t_begin * PASSES, v_end = num_tiles * PASSES;
    auto next_v = [&](int v) { return (v % PASSES == PASSES - 1) ? v + 1 + (t_step - 1) * PASSES : v + 1; };

    if (warp == PRODUCER_WARP) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            GroupScan scan;
            for (int v = v_begin; v < v_end && ok; v = next_v(v)) {
                const PairTile ti = get_pair_tile<KIND>(p, v, pblocks, rank, scan);
                if (!ti.valid) continue;
                const int nb0 = min((ti.n_blk * BN) / 128, p.num_nb - 1);
                const int nb1 = min((ti.n_blk * BN + BN / 2) / 128, p.num_nb - 1);
                const int bgroup = KIND == KIND_KGROUPED ? 0 : ti.group;  // K-grouped: one B for all groups
                const float *sb0 = p.sB + ((size_t)bgroup * p.num_nb + nb0) * p.num_kb;
                const float *sb1 = p.sB + ((size_t)bgroup * p.num_nb + nb1) * p.num_kb;
                for (int kb = ti.kb_lo; kb < ti.kb_hi; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    const uint32_t q = it % SS, qph = (it / SS) & 1u;
                    if (!wait_phase_call(empty_bar(s), ph ^ 1u, abort_flag, p, ROLE_PRODUCER) ||
                        !wait_phase_call(sempty_bar(q), qph ^ 1u, abort_flag, p, ROLE_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    if ((int)it == p.debug_skip_iter) continue;
                    int ax = kb * BLOCK_K;
                    if constexpr (kDebugBuild) {
                        if ((int)it == p.debug_bad_coord) ax += p.num_kb * BLOCK_K;
                        const int sa_rows = KIND == KIND_MASKED ? p.rows : p.a_rows_total;
                        if (!(dbg_ok(p, s < (uint32_t)STAGES && q < (uint32_t)SS, DBG_RING, (int)it) &&
                              dbg_box(p, ax, p.k, ti.a_row, load_row_limit(p.a_rows_total), DBG_TMA_A) &&
                              dbg_box(p, kb * BLOCK_K, p.k, ti.b_row, load_row_limit(p.b_rows_total), DBG_TMA_B) &&
                              dbg_box(p, kb, p.num_kb, ti.sa_row, load_row_limit(sa_rows), DBG_TMA_A) &&
                              dbg_ok(p, ti.group >= 0 && ti.group < p.num_groups, DBG_TMA_B, ti.group))) {
                            *abort_flag = 1u;
                            ok = false;
                            break;
                        }
                    }
                    if (leader) mbar_arrive_expect_tx(full_bar(s), PAIR_TX);
                    const uint32_t lead_full = map_shared_rank(full_bar(s), 0);
                    tma_load_2d_pair(sbase + L::A_OFF + s * A_STAGE_BYTES, &tmap_a, lead_full, ax, ti.a_row);
                    tma_load_2d_pair(sbase + L::B_OFF + s * L::HB_STAGE_BYTES, &tmap_b, lead_full, kb * BLOCK_K,
                                     ti.b_row);
                    mbar_arrive_expect_tx(sfull_bar(q), SA_STAGE_BYTES);
                    if constexpr (KIND == KIND_MASKED)
                        tma_load_3d(sbase + L::SA_OFF + q * SA_STAGE_BYTES, &tmap_sa, sfull_bar(q), ti.sa_row, kb,
                                    ti.group);
                    else
                        tma_load_2d(sbase + L::SA_OFF + q * SA_STAGE_BYTES, &tmap_sa, sfull_bar(q), ti.sa_row, kb);
                    cp_async_4(sbase + L::SB_OFF + q * SB_STAGE_BYTES, sb0 + kb);
                    cp_async_4(sbase + L::SB_OFF + q * SB_STAGE_BYTES + 4, sb1 + kb);
                    cp_async_mbar_arrive_noinc(sfull_bar(q));
                }
            }
            if (!ok) {
                // Let copies in flight land before the CTA exits.  The operand
                // loads of both CTAs complete on the even CTA's full barriers,
                // which only it can wait on; the odd CTA's copies were issued
                // at least one bounded wait (the watchdog limit) ago.
                if (leader) {
                    const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
                    for (uint32_t j = first; j < it; ++j) {
                        if ((int)j == p.debug_skip_iter) continue;
                        drain_phase(full_bar(j % STAGES), (j / STAGES) & 1u, p.timeout_ns);
                    }
                }
                const uint32_t firstq = it > (uint32_t)SS ? it - SS : 0u;
                for (uint32_t j = firstq; j < it; ++j) {
                    if ((int)j == p.debug_skip_iter) continue;
                    drain_phase(sfull_bar(j % SS), (j / SS) & 1u, p.timeout_ns);
                }
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // -------------------------------------------- MMA issuer (even CTA)
        if (leader && lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            GroupScan scan;
            for (int v = v_begin; v < v_end && ok; v = next_v(v)) {
                const PairTile ti = get_pair_tile<KIND>(p, v, pblocks, rank, scan);
                if (!ti.valid) continue;
                for (int kb = ti.kb_lo; kb < ti.kb_hi; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    const uint32_t b = it & (NTB - 1u), bph = (it / NTB) & 1u;
                    if (!wait_phase_call(tempty_bar(b), bph ^ 1u, abort_flag, p, ROLE_MMA) ||
                        !wait_phase_call(full_bar(s), ph, abort_flag, p, ROLE_MMA)) {
                        ok = false;
                        break;
                    }
                    if constexpr (kDebugBuild) {
                        if (!dbg_ok(p, s < (uint32_t)STAGES && b < NTB && (int)(b + 1) * BN <= L::TMEM_COLS, DBG_TMEM,
                                    (int)it)) {
                            *abort_flag = 1u;
                            ok = false;
                            break;
                        }
                    }
                    tc_fence_after();
                    const uint64_t adesc = make_desc_kmajor_sw128(sbase + L::A_OFF + s * A_STAGE_BYTES);
                    const uint64_t bdesc = make_desc_kmajor_sw128(sbase + L::B_OFF + s * L::HB_STAGE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BLOCK_K / MMA_K; ++kk) {
                        const uint64_t koff = (uint64_t)((kk * MMA_K) >> 4);
                        mma_f8f6f4_pair(tmem_base + b * BN, adesc + koff, bdesc + koff, p.idesc, kk > 0 ? 1u : 0u);
                    }
                    mma_commit_pair(empty_bar(s), BOTH);
                    mma_commit_pair(tfull_bar(b), BOTH);
                }
            }
            if (!ok) {
                // every MMA issued so far (they write both CTAs' TMEM) must finish
                mma_commit_pair(drain_bar, 0x1);
                drain_phase(drain_bar, 0u, p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp < NUM_EPI_WARPS) {
        // ------------------------------------------ promotion + epilogue warps
        const int sub = warp & 3;
        const int half = warp >> 2;
        const int r = sub * 32 + lane;
        const uint32_t stg = sbase + L::STG_OFF + warp * L::STG_PER_WARP;
        const uint32_t t_lane = (uint32_t)(sub * 32) << 16;
        const uint32_t sa_addr = sbase + L::SA_OFF + r * 4;
        const uint32_t sb_addr = sbase + L::SB_OFF + half * 4;
        const uint32_t t_base = tmem_base + t_lane + half * COLS;
        uint32_t b = 0, bph = 0, q = 0, qph = 0;
        uint32_t ep = 0;  // DEFER: tiles staged so far (parity of the staging barriers)
        bool ok = true;
        GroupScan scan;
        for (int v = v_begin; v < v_end && ok; v = next_v(v)) {
            const PairTile ti = get_pair_tile<KIND>(p, v, pblocks, rank, scan);
            if (!ti.valid) {
                if constexpr (KIND == KIND_CONTIGUOUS) {
                    // this CTA's block, in the pass of its own group and once per
                    // block (first column block): a first row out of range
                    // breaks the layout, and a block whose first row is -1 must
                    // be all padding (a group id elsewhere in it breaks the
                    // 128-row alignment contract)
                    if (ti.own_pass && ti.n_blk == 0 && ti.own_group != -2 &&
                        !(ti.own_group >= 0 && ti.own_group < p.num_groups)) {
                        if (ti.own_group != -1) {
                            if (warp == 0 && lane == 0) record_error(p, DEV_ERR_CHECK, (uint32_t)ti.a_row);
                        } else if (half == 0) {
                            const int gid = __ldg(p.m_indices + ti.a_row + r);
                            if (gid != -1) record_error(p, DEV_ERR_CHECK, (uint32_t)(ti.a_row + r));
                        }
                    }
                }
                continue;
            }
            // which rows of this warp are written
            bool row_ok;
            if constexpr (KIND == KIND_CONTIGUOUS) {
                // the rows of the pass's group (-1 padding rows and the other
                // block's group stay untouched); in the pass of this CTA's own
                // block any other valid id breaks the alignment contract
                const int gid = r < ti.row_limit ? __ldg(p.m_indices + ti.a_row + r) : -1;
                row_ok = gid == ti.group;
                if (ti.group == ti.own_group && gid != ti.group && gid != -1 && half == 0)
                    record_error(p, DEV_ERR_CHECK, (uint32_t)(ti.a_row + r));
            } else {
                row_ok = r < ti.row_limit;
            }
            const int col0 = ti.n_blk * BN + half * COLS;

            uint64_t acc2[COLS / 2];
#pragma unroll
            for (int j = 0; j < COLS / 2; ++j) acc2[j] = 0ull;

            // (K-grouped: an empty segment leaves the sums at zero, and zeros are stored)
            for (int kb = ti.kb_lo; kb < ti.kb_hi; ++kb) {
                const bool got = wait_phase_call(sfull_bar(q), qph, abort_flag, p, ROLE_EPILOGUE) &&
                                 wait_phase_call(tfull_bar(b), bph, abort_flag, p, ROLE_EPILOGUE);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                if constexpr (kDebugBuild) {
                    const bool in = dbg_ok(p,
                                           b < NTB && q < (uint32_t)SS &&
                                               (int)b * BN + half * COLS + COLS <= L::TMEM_COLS,
                                           DBG_TMEM, kb);
                    if (!__all_sync(0xffffffffu, in)) {
                        *abort_flag = 1u;
                        ok = false;
                        break;
                    }
                }
                tc_fence_after();
                const float sc = ld_shared_f32(sa_addr + q * SA_STAGE_BYTES) *
                                 ld_shared_f32(sb_addr + q * SB_STAGE_BYTES);
                __syncwarp();
                if (lane == 0) mbar_arrive(sempty_bar(q));
                const uint64_t sc2 = pack_f32x2(sc, sc);
                const uint32_t taddr = t_base + b * BN;
#pragma unroll
                for (int c = 0; c < COLS / LD_COLS; ++c) {
                    uint32_t v[LD_COLS];
#pragma unroll
                    for (int u = 0; u < LD_COLS / 8; ++u)
                        tmem_ld_32x32b_x8(taddr + c * LD_COLS + 8 * u, *reinterpret_cast<uint32_t(*)[8]>(&v[8 * u]));
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < LD_COLS; ++j) reg_fence(v[j]);
                    if constexpr (kDebugBuild) {
                        bool fin = true;
#pragma unroll
                        for (int j = 0; j < LD_COLS; ++j) fin = fin && isfinite(__uint_as_float(v[j]));
                        dbg_ok(p, fin, DBG_NONFINITE, kb);
                    }
                    if (c == COLS / LD_COLS - 1) {
                        // the partial is in registers: hand the buffer back to the
                        // even CTA's MMA warp before the last FMAs
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_remote(map_shared_rank(tempty_bar(b), 0));
                    }
#pragma unroll
                    for (int j = 0; j < LD_COLS; j += 2)
                        ffma2(acc2[(c * LD_COLS + j) / 2], v[j], v[j + 1], sc2);
                }
                b = (b + 1u) & (NTB - 1u);
                bph ^= (b == 0u);
                q = (q + 1u) & (SS - 1u);
                qph ^= (q == 0u);
            }
            if (!ok) break;

            // ---------------------------------------------------- epilogue
            float acc[COLS];
#pragma unroll
            for (int j = 0; j < COLS / 2; ++j) unpack_f32x2(acc2[j], acc[2 * j], acc[2 * j + 1]);
            // first row of this warp's block in D (K-grouped: within the group's
            // output plane, the third coordinate of D's tensor map)
            const int d_row = ti.a_row + sub * 32;
            const bool rows_in = sub * 32 < ti.row_limit;  // some row of this warp is written
            bool use_tma;
            if constexpr (CLIPPED)
                use_tma = true;  // rows past m are clipped by the tensor map bounds
            else
                use_tma = __all_sync(0xffffffffu, row_ok);
            if constexpr (DEFER) {
                // the store warp has finished reading the previous tile's staging
                // (every warp waits, so none can be a tile ahead of the others)
                if (!__all_sync(0xffffffffu,
                                wait_phase_call(stg_empty_bar, (ep & 1u) ^ 1u, abort_flag, p, ROLE_EPILOGUE)))
                    break;
                ++ep;
                // tell the store warp whether this warp's boxes are staged (its
                // arrival on stg_full below orders this write before the read)
                if constexpr (!CLIPPED) {
                    if (lane == 0) staged[warp] = (use_tma && rows_in) ? 1 : 0;
                }
            }
            if (DEFER && use_tma) {
                // stage both 64-column boxes; the store warp issues their stores
#pragma unroll
                for (int bx = 0; bx < COLS / 64; ++bx) {
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const float *f = acc + bx * 64 + ch * 8;
                        const uint32_t off = (uint32_t)lane * 128u + ((uint32_t)(ch ^ (lane & 7)) << 4);
                        st_shared_v4(stg + bx * STAGING_BYTES_PER_WARP + off, pack_bf16x2(f[0], f[1]),
                                     pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                    }
                }
                fence_proxy_async_smem();
            } else if (use_tma) {
                if constexpr (F32OUT) {
                    // FP32 boxes: 32 rows x 32 columns (128 bytes per row, same swizzle)
#pragma unroll
                    for (int bx = 0; bx < COLS / 32; ++bx) {
                        const int x = col0 + bx * 32;
                        if (!rows_in || x >= p.n) continue;  // box entirely outside D: nothing to write
                        if (lane == 0) bulk_wait_group_read<0>();  // staging buffer free again
                        __syncwarp();
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            const float *f = acc + bx * 32 + ch * 4;
                            const uint32_t off = (uint32_t)lane * 128u + ((uint32_t)(ch ^ (lane & 7)) << 4);
                            st_shared_v4(stg + off, __float_as_uint(f[0]), __float_as_uint(f[1]),
                                         __float_as_uint(f[2]), __float_as_uint(f[3]));
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            store_d_box<KIND>(&tmap_d, stg, x, d_row, ti.group, p);
                            bulk_commit_group();
                        }
                    }
                } else {
#pragma unroll
                for (int bx = 0; bx < COLS / 64; ++bx) {
                    const int x = col0 + bx * 64;
                    if (!rows_in || x >= p.n) continue;  // box entirely outside D: nothing to write
                    if (lane == 0) bulk_wait_group_read<0>();  // staging buffer free again
                    __syncwarp();
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const float *f = acc + bx * 64 + ch * 8;
                        const uint32_t off = (uint32_t)lane * 128u + ((uint32_t)(ch ^ (lane & 7)) << 4);
                        st_shared_v4(stg + off, pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                     pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        store_d_box<KIND>(&tmap_d, stg, x, d_row, ti.group, p);
                        bulk_commit_group();
                    }
                }
                }
            } else if (row_ok) {
                if constexpr (F32OUT) {
                    float *drow = static_cast<float *>(p.D) + (size_t)(d_row + lane) * p.n;
#pragma unroll
                    for (int ch = 0; ch < COLS / 8; ++ch) {
                        const int c = col0 + ch * 8;
                        if (c < p.n) {
                            const float *f = acc + ch * 8;
                            st_global_v4(drow + c, __float_as_uint(f[0]), __float_as_uint(f[1]),
                                         __float_as_uint(f[2]), __float_as_uint(f[3]));
                            st_global_v4(drow + c + 4, __float_as_uint(f[4]), __float_as_uint(f[5]),
                                         __float_as_uint(f[6]), __float_as_uint(f[7]));
                        }
                    }
                } else {
                    __nv_bfloat16 *drow = static_cast<__nv_bfloat16 *>(p.D) + (size_t)(d_row + lane) * p.n;
#pragma unroll
                    for (int ch = 0; ch < COLS / 8; ++ch) {
                        const int c = col0 + ch * 8;
                        if (c < p.n) {
                            const float *f = acc + ch * 8;
                            st_global_v4(drow + c, pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                         pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                        }
                    }
                }
            }
            if constexpr (DEFER) {
                __syncwarp();
                if (lane == 0) mbar_arrive(stg_full_bar);  // this warp's part of the tile is staged (or stored)
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    } else if (DEFER && warp == STORE_WARP) {
        // ------------------------------------------------ store warp (DEFER)
        // Walks the same tiles; once all promotion warps have staged a tile it
        // issues the TMA stores of the boxes they would have stored (same
        // predicates), waits until the stores have read the staging and hands
        // it back.
        if (lane == 0) {
            uint32_t ep = 0;
            GroupScan scan;
            for (int v = v_begin; v < v_end; v = next_v(v)) {
                const PairTile ti = get_pair_tile<KIND>(p, v, pblocks, rank, scan);
                if (!ti.valid) continue;
                if (!wait_phase_call(stg_full_bar, ep & 1u, abort_flag, p, ROLE_EPILOGUE)) break;
                ++ep;
                for (int w = 0; w < NUM_EPI_WARPS; ++w) {
                    const int wsub = w & 3, whalf = w >> 2;
                    if constexpr (CLIPPED) {
                        if (wsub * 32 >= ti.row_limit) continue;  // no row of this warp in D
                    } else {
                        if (!staged[w]) continue;  // nothing staged: stored row by row, or no row written
                    }
                    const int d_row = ti.a_row + wsub * 32;
                    for (int bx = 0; bx < COLS / 64; ++bx) {
                        const int x = ti.n_blk * BN + whalf * COLS + bx * 64;
                        if (x >= p.n) continue;
                        store_d_box<KIND>(&tmap_d,
                                          sbase + L::STG_OFF + w * L::STG_PER_WARP + bx * STAGING_BYTES_PER_WARP, x,
                                          d_row, ti.group, p);
                    }
                }
                bulk_commit_group();
                bulk_wait_group_read<0>();
                mbar_arrive(stg_empty_bar);
            }
            bulk_wait_group<0>();
        }
        __syncwarp();
    }

    // ------------------------------------------------------------ teardown
    // Both CTAs: every MMA has completed (its partials were waited for, or the
    // drain above) and no arrival or load targets the other CTA any more.
    tc_fence_before();
    cluster_sync();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
    }
}

}  // namespace fg
