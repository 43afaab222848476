// gemm_swap_kernel.cuh -- the FP8 NT GEMM with the operand roles swapped, for
// problems with few rows per group ("swap-AB").
//
// Same method as gemm_kernel.cuh (page "DeepSeek开源周第三天DeepGEMM",
// "两级精度累加与细粒度缩放": one 128-deep K block on the tensor cores into a
// fresh FP32 partial, scaled by sA * sB and added on the CUDA cores), with the
// weights in the MMA's M = 128 role and the tokens (the rows of A, at most BT
// of them per tile) in its N = BT role:
//
//   P^T[w, t] = sum_{k in kb} B[n0 + w, k] * A[m0 + t, k]     (tcgen05.mma, TMEM)
//   D[m0 + t, n0 + w] += (sA[m0 + t, kb] * sB[n0 / 128, kb]) * P^T[w, t]
//
// A tile therefore covers 128 weight rows (one 128 x 128 scale block of B per K
// block, a single scalar) and BT token rows (a vector of BT scales of A per K
// block).  When a group has fewer than 128 valid rows, the one-CTA kernel
// multiplies (and loads, and promotes) a 128-row tile that is mostly empty,
// and with the masked layout it launches tiles for the rows past the counts
// too; here a tile holds up to BT = 256 tokens, so every launched tile of a
// group with rows does useful work and the tensor-core tile is never larger
// than the weight block it streams.
//
// Roles and pipeline as in the one-CTA kernel (warp 8 producer, warp 9 MMA
// issuer, warps 0..7 promotion + epilogue; warp w owns TMEM lanes 32*(w%4)..,
// i.e. weight rows, and token columns [(w/4)*BT/2, (w/4+1)*BT/2)).  The
// promotion multiplies each column by its own scale (token scale times the
// tile's weight scale, the same FP32 product as the one-CTA kernel forms).
// The epilogue transposes through shared memory: each warp's 32 weight columns
// x 32 tokens go out as one TMA box of D, or with per-element stores where a
// masked group's count ends inside the box.  Split-K (SPLITK): a cluster of S
// CTAs per tile shares its K blocks and reduces the FP32 partials through
// distributed shared memory in rank order, each rank a slice of the tokens.
// Every wait is bounded by the watchdog of gemm_kernel.cuh.
#pragma once

#include "gemm_kernel.cuh"

namespace fg {

template <int BT, int STAGES>
struct SwapSmemLayout {
    static constexpr int W_STAGE_BYTES = BLOCK_M * BLOCK_K;  // 128 weight rows of one K block
    static constexpr int T_STAGE_BYTES = BT * BLOCK_K;       // BT token rows of one K block
    static constexpr int W_OFF = 0;
    static constexpr int T_OFF = W_OFF + STAGES * W_STAGE_BYTES;
    static constexpr int STG_OFF = T_OFF + STAGES * T_STAGE_BYTES;
    static constexpr int TS_BYTES = BT * 4;  // token scales of one K block
    static constexpr int TS_OFF = STG_OFF + NUM_EPI_WARPS * STAGING_BYTES_PER_WARP;
    static constexpr int WS_OFF = TS_OFF + SCALE_STAGES * TS_BYTES;  // the weight block's scale (16-byte slot)
    static constexpr int BAR_OFF = WS_OFF + SCALE_STAGES * 16;
    static constexpr int TMEM_COLS = 512;
    static constexpr int NUM_TBUF = TMEM_COLS / BT;
    // full, empty, scale_full, scale_empty, tmem_full, tmem_empty, drain
    static constexpr int NUM_BARS = 2 * STAGES + 2 * SCALE_STAGES + 2 * NUM_TBUF + 1;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int BYTES = MISC_OFF + 16;
    // split-K partial (128 weight rows x BT tokens, FP32), aliased on the operand ring
    static constexpr int P_OFF = 0;
    static constexpr bool PARTIAL_FITS = BLOCK_M * BT * 4 <= STG_OFF;
};

struct SwapTile {
    int valid;
    int group;
    int w_blk;    // 128-row weight block (the output columns n0 = 128 * w_blk)
    int t_blk;    // BT-row token block within the group
    int w_row;    // first weight row in the 2-D row space of B ([G*n][k])
    int t_row;    // first token row in the 2-D row space of A and D
    int count;    // tokens of the tile that are written (<= BT)
};

// Token blocks of group g that hold rows (masked: from the device count).
template <int BT, int KIND>
__device__ __forceinline__ int swap_token_blocks(const GemmParams &p, int g) {
    const int rows = KIND == KIND_MASKED ? clamp_count(__ldg(p.masked_m + g), p.rows) : p.rows;
    return (rows + BT - 1) / BT;
}

template <int BT, int KIND>
__device__ __forceinline__ int total_swap_tiles(const GemmParams &p) {
    if constexpr (KIND == KIND_MASKED) {
        int t = 0;
        for (int g = 0; g < p.num_groups; ++g) t += swap_token_blocks<BT, KIND>(p, g);
        return t * p.num_n_blocks;
    } else {
        return swap_token_blocks<BT, KIND>(p, 0) * p.num_n_blocks;
    }
}

// Tile t: groups in order, token blocks of a group in order, weight blocks
// fastest (the tiles that run at the same time share their tokens, which stay
// in L2, while the weights stream once).
template <int BT, int KIND>
__device__ __forceinline__ SwapTile get_swap_tile(const GemmParams &p, int t) {
    SwapTile ti;
    const int nw = p.num_n_blocks;
    int g = 0, rows = p.rows;
    if constexpr (KIND == KIND_MASKED) {
        for (; g < p.num_groups; ++g) {
            rows = clamp_count(__ldg(p.masked_m + g), p.rows);
            const int tiles = ((rows + BT - 1) / BT) * nw;
            if (t < tiles) break;
            t -= tiles;
        }
    }
    ti.valid = g < p.num_groups;
    ti.group = g;
    ti.w_blk = t % nw;
    ti.t_blk = t / nw;
    ti.w_row = g * p.n + ti.w_blk * BLOCK_M;
    ti.t_row = g * p.rows + ti.t_blk * BT;  // masked: the group's rows start at g * M_cap
    ti.count = min(BT, rows - ti.t_blk * BT);
    return ti;
}

__device__ __forceinline__ float4 ld_shared_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<const uint16_t *>(&h);
}

// Tensor maps: tmap_w over the weights B [G*n][k] u8 (box 128 rows), tmap_t over
// the tokens A [rows][k] u8 (box BT rows), both 128-byte swizzled; tmap_d over
// D [rows][n] (bf16, or fp32 for F32OUT), box 32 columns x 32 rows, no swizzle;
// tmap_ts over the MN-major token scales (2-D {rows, kb}, masked 3-D {M_cap,
// kb, G}), box BT.
template <int BT, int STAGES, int KIND, bool SPLITK, bool F32OUT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fp8_gemm_swap_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_t,
                         const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ CUtensorMap tmap_ts,
                         const GemmParams p) {
    static_assert(BT == 128 || BT == 256, "token tile of 128 or 256");
    static_assert(KIND == KIND_DENSE || KIND == KIND_MASKED, "swap-AB: dense and masked layouts");
    using L = SwapSmemLayout<BT, STAGES>;
    static_assert(!SPLITK || L::PARTIAL_FITS, "split-K: the partial tile must fit in the operand ring");
    constexpr int COLS = BT / 2;  // token columns per promotion warp
    constexpr uint32_t STAGE_TX = L::W_STAGE_BYTES + L::T_STAGE_BYTES;
    constexpr uint32_t NTB = L::NUM_TBUF;
    static_assert((NTB & (NTB - 1)) == 0 && NTB >= 2, "TMEM buffer count");
    constexpr int ROW_BYTES = BT * 4;  // one weight row of the split-K partial

    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::BAR_OFF;
    auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (STAGES + s); };
    auto sfull_bar = [&](uint32_t q) { return bar0 + 8u * (2 * STAGES + q); };
    auto sempty_bar = [&](uint32_t q) { return bar0 + 8u * (2 * STAGES + SCALE_STAGES + q); };
    auto tfull_bar = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + 2 * SCALE_STAGES + b); };
    auto tempty_bar = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + 2 * SCALE_STAGES + NTB + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * SCALE_STAGES + 2 * NTB);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + L::MISC_OFF + 4);

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    if (sbase & 1023u) {
        if (threadIdx.x == 0) record_error(p, DEV_ERR_CHECK, (ROLE_SETUP << 24) | (sbase & 0xFFFFu));
        return;
    }

    // ------------------------------------------------------------- set-up
    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            prefetch_tensormap(&tmap_w);
            prefetch_tensormap(&tmap_t);
            prefetch_tensormap(&tmap_ts);
            prefetch_tensormap(&tmap_d);
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(full_bar(s), 1);
                mbar_init(empty_bar(s), 1);
            }
            for (int q = 0; q < SCALE_STAGES; ++q) {
                mbar_init(sfull_bar(q), 2);  // producer's expect_tx arrival + the cp.async arrival
                mbar_init(sempty_bar(q), NUM_EPI_WARPS);
            }
            for (uint32_t b = 0; b < NTB; ++b) {
                mbar_init(tfull_bar(b), 1);
                mbar_init(tempty_bar(b), NUM_EPI_WARPS);
            }
            mbar_init(drain_bar, 1);
            *abort_flag = 0u;
            fence_mbarrier_init();
        }
        __syncwarp();
        named_bar_arrive(1, NUM_THREADS);
    } else {
        if (warp == MMA_WARP) {
            tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
            tmem_relinquish();
        }
        tc_fence_before();
        named_bar_sync(1, NUM_THREADS);
        tc_fence_after();
    }
    const uint32_t tmem_base = warp == PRODUCER_WARP ? 0u : *tmem_slot;

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

    const int num_tiles = total_swap_tiles<BT, KIND>(p);
    int t_begin = blockIdx.x, t_step = gridDim.x, kb_begin = 0, kb_end = p.num_kb;
    uint32_t split = 1, rank = 0;
    if constexpr (SPLITK) {
        split = cluster_nctarank();
        rank = cluster_ctarank();
        t_begin = blockIdx.x / split;
        t_step = num_tiles > 0 ? num_tiles : 1;
        kb_begin = (int)(((long long)p.num_kb * rank) / split);
        kb_end = (int)(((long long)p.num_kb * (rank + 1)) / split);
    }

    if (warp == PRODUCER_WARP) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = t_begin; t < num_tiles && ok; t += t_step) {
                const SwapTile ti = get_swap_tile<BT, KIND>(p, t);
                if (!ti.valid) continue;
                const float *sw = p.sB + ((size_t)ti.group * p.num_nb + ti.w_blk) * p.num_kb;
                for (int kb = kb_begin; kb < kb_end; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    const uint32_t q = it % SCALE_STAGES, qph = (it / SCALE_STAGES) & 1u;
                    if (!wait_phase_call(empty_bar(s), ph ^ 1u, abort_flag, p, ROLE_PRODUCER) ||
                        !wait_phase_call(sempty_bar(q), qph ^ 1u, abort_flag, p, ROLE_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    if ((int)it == p.debug_skip_iter) continue;
                    mbar_arrive_expect_tx(full_bar(s), STAGE_TX);
                    tma_load_2d(sbase + L::W_OFF + s * L::W_STAGE_BYTES, &tmap_w, full_bar(s), kb * BLOCK_K,
                                ti.w_row);
                    tma_load_2d(sbase + L::T_OFF + s * L::T_STAGE_BYTES, &tmap_t, full_bar(s), kb * BLOCK_K,
                                ti.t_row);
                    mbar_arrive_expect_tx(sfull_bar(q), L::TS_BYTES);
                    if constexpr (KIND == KIND_MASKED)
                        tma_load_3d(sbase + L::TS_OFF + q * L::TS_BYTES, &tmap_ts, sfull_bar(q), ti.t_blk * BT, kb,
                                    ti.group);
                    else
                        tma_load_2d(sbase + L::TS_OFF + q * L::TS_BYTES, &tmap_ts, sfull_bar(q), ti.t_blk * BT, kb);
                    cp_async_4(sbase + L::WS_OFF + q * 16, sw + kb);
                    cp_async_mbar_arrive_noinc(sfull_bar(q));
                }
            }
            if (!ok) {
                const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
                for (uint32_t j = first; j < it; ++j) {
                    if ((int)j == p.debug_skip_iter) continue;
                    drain_phase(full_bar(j % STAGES), (j / STAGES) & 1u, p.timeout_ns);
                }
                const uint32_t firstq = it > (uint32_t)SCALE_STAGES ? it - SCALE_STAGES : 0u;
                for (uint32_t j = firstq; j < it; ++j) {
                    if ((int)j == p.debug_skip_iter) continue;
                    drain_phase(sfull_bar(j % SCALE_STAGES), (j / SCALE_STAGES) & 1u, p.timeout_ns);
                }
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = t_begin; t < num_tiles && ok; t += t_step) {
                const SwapTile ti = get_swap_tile<BT, KIND>(p, t);
                if (!ti.valid) continue;
                for (int kb = kb_begin; kb < kb_end; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    const uint32_t b = it & (NTB - 1u), bph = (it / NTB) & 1u;
                    if (!wait_phase_call(tempty_bar(b), bph ^ 1u, abort_flag, p, ROLE_MMA) ||
                        !wait_phase_call(full_bar(s), ph, abort_flag, p, ROLE_MMA)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t wdesc = make_desc_kmajor_sw128(sbase + L::W_OFF + s * L::W_STAGE_BYTES);
                    const uint64_t tdesc = make_desc_kmajor_sw128(sbase + L::T_OFF + s * L::T_STAGE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BLOCK_K / MMA_K; ++kk) {
                        const uint64_t koff = (uint64_t)((kk * MMA_K) >> 4);
                        mma_f8f6f4(tmem_base + b * BT, wdesc + koff, tdesc + koff, p.idesc, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(empty_bar(s));
                    mma_commit(tfull_bar(b));
                }
            }
            if (!ok) {
                mma_commit(drain_bar);
                drain_phase(drain_bar, 0u, p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp < NUM_EPI_WARPS) {
        // ------------------------------------------ promotion + epilogue warps
        const int sub = warp & 3;    // TMEM lane quarter: weight rows [32*sub, 32*sub+32)
        const int half = warp >> 2;  // token columns [half*COLS, half*COLS+COLS)
        const int wr = sub * 32 + lane;
        const uint32_t stg = sbase + L::STG_OFF + warp * STAGING_BYTES_PER_WARP;
        const uint32_t t_base = tmem_base + ((uint32_t)(sub * 32) << 16) + half * COLS;
        const uint32_t ts_base = sbase + L::TS_OFF + half * COLS * 4;
        uint32_t b = 0, bph = 0, q = 0, qph = 0;
        bool ok = true;
        for (int t = t_begin; t < num_tiles && ok; t += t_step) {
            const SwapTile ti = get_swap_tile<BT, KIND>(p, t);
            if (!ti.valid) continue;

            uint64_t acc2[COLS / 2];  // FP32 running sums of this weight row, pairs of token columns
#pragma unroll
            for (int j = 0; j < COLS / 2; ++j) acc2[j] = 0ull;

            for (int kb = kb_begin; kb < kb_end; ++kb) {
                const bool got = wait_phase_call(sfull_bar(q), qph, abort_flag, p, ROLE_EPILOGUE) &&
                                 wait_phase_call(tfull_bar(b), bph, abort_flag, p, ROLE_EPILOGUE);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float ws = ld_shared_f32(sbase + L::WS_OFF + q * 16);
                const uint32_t ts_addr = ts_base + q * L::TS_BYTES;
                const uint32_t taddr = t_base + b * BT;
#pragma unroll
                for (int c = 0; c < COLS / TMEM_LD_COLS; ++c) {
                    uint32_t v[TMEM_LD_COLS];
#pragma unroll
                    for (int u = 0; u < TMEM_LD_COLS / 8; ++u)
                        tmem_ld_32x32b_x8(taddr + c * TMEM_LD_COLS + 8 * u,
                                          *reinterpret_cast<uint32_t(*)[8]>(&v[8 * u]));
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < TMEM_LD_COLS; ++j) reg_fence(v[j]);
                    if (c == COLS / TMEM_LD_COLS - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(tempty_bar(b));
                    }
#pragma unroll
                    for (int u = 0; u < TMEM_LD_COLS / 4; ++u) {
                        // four token scales (the same for every lane: a broadcast read)
                        const float4 s4 = ld_shared_v4(ts_addr + (uint32_t)(c * TMEM_LD_COLS + 4 * u) * 4u);
                        const int j = c * TMEM_LD_COLS + 4 * u;
                        ffma2(acc2[j / 2], v[4 * u], v[4 * u + 1], pack_f32x2(s4.x * ws, s4.y * ws));
                        ffma2(acc2[j / 2 + 1], v[4 * u + 2], v[4 * u + 3], pack_f32x2(s4.z * ws, s4.w * ws));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sempty_bar(q));
                b = (b + 1u) & (NTB - 1u);
                bph ^= (b == 0u);
                q = (q + 1u) & (SCALE_STAGES - 1u);
                qph ^= (q == 0u);
            }
            if (!ok) break;

            if constexpr (SPLITK) {
                if (split > 1) {
                    // partial -> own shared memory (the operand ring is idle now):
                    // weight row wr, BT FP32 token columns, 16-byte chunks rotated by (wr & 7)
                    const uint32_t prow = sbase + L::P_OFF + (uint32_t)wr * ROW_BYTES;
#pragma unroll
                    for (int ch = 0; ch < COLS / 4; ++ch) {
                        const int cg = half * (COLS / 4) + ch;
                        float x0, x1, x2, x3;
                        unpack_f32x2(acc2[2 * ch], x0, x1);
                        unpack_f32x2(acc2[2 * ch + 1], x2, x3);
                        st_shared_v4(prow + (uint32_t)((cg ^ (wr & 7)) << 4), __float_as_uint(x0),
                                     __float_as_uint(x1), __float_as_uint(x2), __float_as_uint(x3));
                    }
                    continue;  // the cluster reduction below writes D
                }
            }

            // ------------------------------------------- epilogue (transposed)
            float acc[COLS];
#pragma unroll
            for (int j = 0; j < COLS / 2; ++j) unpack_f32x2(acc2[j], acc[2 * j], acc[2 * j + 1]);
            const int x = ti.w_blk * BLOCK_M + sub * 32;      // first output column of this warp
            const bool col_ok = x + lane < p.n;
#pragma unroll
            for (int bx = 0; bx < COLS / 32; ++bx) {
                const int c0 = half * COLS + bx * 32;          // first token of the box within the tile
                if (c0 >= ti.count || x >= p.n) continue;      // nothing of this box is written
                const int row0 = ti.t_row + c0;                // its first row of D
                if (ti.count - c0 >= 32 || KIND == KIND_DENSE) {
                    // whole box (dense rows past m and columns past n are clipped by
                    // the tensor map): stage token-major and store with TMA
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if constexpr (F32OUT)
                            st_shared_u32(stg + (uint32_t)(j * 32 + lane) * 4u, __float_as_uint(acc[bx * 32 + j]));
                        else
                            st_shared_u16(stg + (uint32_t)(j * 32 + lane) * 2u, bf16_bits(acc[bx * 32 + j]));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmap_d, stg, x, row0);
                        bulk_commit_group();
                    }
                } else if (col_ok) {
                    // a masked group's count ends inside the box: per-element stores
                    // of the valid tokens (32 lanes = 32 consecutive columns of a row)
                    const int nvalid = ti.count - c0;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (j < nvalid) {
                            const size_t off = (size_t)(row0 + j) * p.n + x + lane;
                            if constexpr (F32OUT)
                                static_cast<float *>(p.D)[off] = acc[bx * 32 + j];
                            else
                                static_cast<uint16_t *>(p.D)[off] = bf16_bits(acc[bx * 32 + j]);
                        }
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    if constexpr (SPLITK) {
        if (split > 1) {
            // every CTA of the cluster takes both barriers, whatever happened above
            cluster_sync();
            bool any_abort = false;
            for (uint32_t q = 0; q < split; ++q)
                any_abort |= ld_shared_cluster_u32(map_shared_rank(smem_u32((const void *)abort_flag), q)) != 0u;
            if (t_begin < num_tiles && !any_abort && warp < NUM_EPI_WARPS) {
                const SwapTile ti = get_swap_tile<BT, KIND>(p, t_begin);
                if (ti.valid && ti.count > 0) {
                    constexpr int MAX_SPLIT = 8;
                    constexpr int STRIDE = NUM_EPI_WARPS * 32;
                    // token chunks of 4 that hold written tokens, shared evenly by the ranks;
                    // an item is (chunk, weight row), weight rows fastest so that a warp
                    // writes 32 consecutive columns of each of its 4 rows of D
                    const int nch = (ti.count + 3) / 4;
                    const int c_lo = (int)((nch * rank) / split), c_hi = (int)((nch * (rank + 1)) / split);
                    const int items = (c_hi - c_lo) * BLOCK_M;
                    const int x0 = ti.w_blk * BLOCK_M;
                    for (int item = threadIdx.x; item < items; item += STRIDE) {
                        const int w = item % BLOCK_M;
                        const int ch = c_lo + item / BLOCK_M;
                        const uint32_t local = sbase + L::P_OFF + (uint32_t)w * ROW_BYTES +
                                               (uint32_t)((ch ^ (w & 7)) << 4);
                        float4 v[MAX_SPLIT];
#pragma unroll
                        for (int q = 0; q < MAX_SPLIT; ++q)
                            if (q < (int)split) v[q] = ld_shared_cluster_v4(map_shared_rank(local, q));
                        float4 sum = v[0];
#pragma unroll
                        for (int q = 1; q < MAX_SPLIT; ++q) {  // fixed rank (= K) order
                            if (q < (int)split) {
                                sum.x += v[q].x;
                                sum.y += v[q].y;
                                sum.z += v[q].z;
                                sum.w += v[q].w;
                            }
                        }
                        if (x0 + w >= p.n) continue;
                        const float s[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int tok = ch * 4 + e;
                            if (tok < ti.count) {
                                const size_t off = (size_t)(ti.t_row + tok) * p.n + x0 + w;
                                if constexpr (F32OUT)
                                    static_cast<float *>(p.D)[off] = s[e];
                                else
                                    static_cast<uint16_t *>(p.D)[off] = bf16_bits(s[e]);
                            }
                        }
                    }
                }
            }
            cluster_sync();  // peers may still be reading this CTA's partial until here
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

}  // namespace fg
