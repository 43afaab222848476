// gemm_kernel.cuh -- persistent, warp-specialized FP8 NT GEMM for sm_103a with
// fine-grained scaling and two-level accumulation, for the dense layout and the
// two MoE grouped layouts (contiguous and masked).
//
// Method (page "DeepSeek开源周第三天DeepGEMM"): each 128-wide K block is
// multiplied on the tensor cores into a fresh FP32 partial, which is then
// scaled by sA[row, kb] * sB[col/128, kb] and added to an FP32 running sum on
// the CUDA cores (promotion excerpt "两级精度累加与细粒度缩放"); BF16 output.
//
// Blackwell mapping (one CTA per SM, 320 threads):
//   warp 8      producer: one lane loads, per K block, the A tile (128 x 128 B)
//               and the B tile (BN x 128 B) into a STAGES-deep shared-memory
//               ring (TMA, 128-byte swizzle, `full[s]`), and the block's scales
//               into a SCALE_STAGES-deep scale ring: the tile's 128 LHS scales
//               by TMA from the MN-major sA (one 512-byte row, the reason the
//               layout is MN-major) and the two RHS block scales by cp.async
//               (`scale_full[q]`).
//   warp 9      MMA issuer: one lane issues 4 tcgen05.mma (K = 32 each) per K
//               block into one of 512/BN TMEM accumulators (128 lanes x BN
//               columns, FP32), then commits to `empty[s]` (smem stage free)
//               and `tmem_full[b]` (partial ready).
//   warps 0..7  promotion + epilogue: warp w owns TMEM lanes 32*(w%4).. (its
//               rows) and columns [(w/4)*BN/2, (w/4+1)*BN/2).  Per K block it
//               reads its scales from the scale ring (releasing the entry), reads
//               the partial in 32-column chunks of tcgen05.ld, hands the TMEM buffer back
//               (`tmem_empty[b]`) as soon as the last load has landed, and adds
//               sA*sB*partial into BN/2 FP32 registers per thread with packed
//               fma.rn.f32x2.  After the last K block a warp converts its
//               32 x BN/2 block to BF16, stages it in swizzled shared memory and
//               writes it with TMA stores, or with per-row predicated stores
//               when some of its rows must stay untouched (grouped layouts).
// The TMEM accumulators (two for BN = 256, four for BN = 128) let the tensor
// cores run the next K blocks while the promotion warps consume K block kb,
// and run the next tile's first K blocks while the previous tile's epilogue
// drains.
//
// Split-K (SPLITK = true, for problems with fewer output tiles than SMs): the
// grid is one cluster of S CTAs per output tile; CTA rank q runs K blocks
// [q*KB/S, (q+1)*KB/S) through the same pipeline, writes its FP32 partial tile
// into its own shared memory, and after a cluster barrier each rank sums one
// slice of rows over all S partials through distributed shared memory, in rank
// order (deterministic), and stores it as BF16.  No global scratch memory.
//
// Launch: programmatic dependent launch is enabled, so a grid may start while
// the previous grid of the stream drains; each CTA sets up its barriers, TMEM
// and tensor-map prefetches first and waits (griddepcontrol.wait) before its
// first access to global memory.
//
// Every wait is bounded by a %globaltimer watchdog: on expiry the kernel
// records FG_ERR_TIMEOUT in the status word, raises a CTA-wide abort flag,
// waits (bounded) for its own copies and MMAs in flight, frees TMEM and exits.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace fg {

enum : int { KIND_DENSE = 0, KIND_CONTIGUOUS = 1, KIND_MASKED = 2, KIND_KGROUPED = 3 };

// device-side status codes (same values as fg_status in fp8gemm.h)
enum : uint32_t { DEV_ERR_TIMEOUT = 5, DEV_ERR_CHECK = 6 };
enum : uint32_t { ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_EPILOGUE = 3, ROLE_SETUP = 4 };

constexpr int BLOCK_M = 128;
constexpr int BLOCK_K = 128;  // K block of the scales and of promotion
constexpr int MMA_K = 32;     // K of one tcgen05.mma kind::f8f6f4
constexpr int NUM_EPI_WARPS = 8;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int NUM_THREADS = 320;
constexpr int TMEM_LD_COLS = 32;  // columns per promotion TMEM load
constexpr int STAGING_BYTES_PER_WARP = 32 * 128;  // 32 rows x 64 BF16 columns
constexpr int A_STAGE_BYTES = BLOCK_M * BLOCK_K;
constexpr int SA_STAGE_BYTES = BLOCK_M * 4;      // 128 LHS scales of one K block
constexpr int SB_STAGE_BYTES = 16;               // the RHS scales of the two column halves
constexpr int SCALE_STAGES = 4;  // a power of two
static_assert((SCALE_STAGES & (SCALE_STAGES - 1)) == 0, "scale ring size");

struct GemmParams {
    int rows;          // rows of the A / D row space: dense m, contiguous M, masked M_cap
    int n, k;
    int num_groups;    // G (1 for dense)
    int num_kb;        // ceil(k / 128)
    int num_nb;        // ceil(n / 128): rows of sB per group
    int num_n_blocks;  // ceil(n / BN)
    int num_m_blocks;  // ceil(rows / 128) (per group for masked)
    int group_m;       // M blocks per raster group (tiles walk N inside a group of M blocks)
    uint32_t idesc;    // tcgen05 instruction descriptor (formats of A and B)
    const float *sB;
    const int32_t *m_indices;
    const int32_t *masked_m;
    const int32_t *k_sizes;  // K-grouped layout: [G] K-segment lengths (multiples of 128)
    void *D;           // bfloat16 [rows][n], or float [rows][n] for the FP32-output instantiations
                       // (K-grouped: [G][rows][n])
    uint32_t *status;  // [0] first error code, [1] its detail
    unsigned long long timeout_ns;
    int debug_skip_iter;  // producer leaves this K iteration unarmed (-1: never)
    // extents of the tensor maps' row spaces, for the debug build's checks
    int a_rows_total;     // rows of A and (2-D maps) of D: dense m, contiguous M, masked G * M_cap, K-grouped M
    int b_rows_total;     // rows of B: G * n (K-grouped: N)
    int debug_bad_coord;  // debug build: the A load of this K iteration is sent past K (-1: never)
};

template <int BN, int STAGES>
struct SmemLayout {
    static constexpr int B_STAGE_BYTES = BN * BLOCK_K;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = A_OFF + STAGES * A_STAGE_BYTES;
    static constexpr int STG_OFF = B_OFF + STAGES * B_STAGE_BYTES;
    static constexpr int SA_OFF = STG_OFF + NUM_EPI_WARPS * STAGING_BYTES_PER_WARP;
    static constexpr int SB_OFF = SA_OFF + SCALE_STAGES * SA_STAGE_BYTES;
    static constexpr int BAR_OFF = SB_OFF + SCALE_STAGES * SB_STAGE_BYTES;
    // TMEM: all 512 columns, as 512 / BN accumulator buffers of BN columns
    static constexpr int TMEM_COLS = 512;
    static constexpr int NUM_TBUF = TMEM_COLS / BN;
    // full, empty, scale_full, scale_empty, tmem_full, tmem_empty, drain
    static constexpr int NUM_BARS = 2 * STAGES + 2 * SCALE_STAGES + 2 * NUM_TBUF + 1;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int BYTES = MISC_OFF + 16;
    // split-K partial tile (128 x BN FP32), aliased on the operand ring
    static constexpr int P_OFF = 0;
    static constexpr bool PARTIAL_FITS = BLOCK_M * BN * 4 <= STG_OFF;
};

__device__ __forceinline__ int clamp_count(int c, int cap) { return c < 0 ? 0 : (c > cap ? cap : c); }

__device__ __forceinline__ void record_error(const GemmParams &p, uint32_t code, uint32_t detail) {
    if (atomicCAS(p.status, 0u, code) == 0u) atomicExch(p.status + 1, detail);
}

// Debug build (compiled with FG_DEBUG): every TMA box start, ring index and
// TMEM column is checked against what the launch allows before it is used.
// A failed check records FG_ERR_DEVICE_CHECK with a tag in bits 24..31 of the
// detail (the offending value in bits 0..23), raises the CTA's abort flag and
// skips the access; the other roles then leave through their bounded waits.
// The promotion warps also flag a non-finite K-block partial (finite inputs
// never give one).  In the release build the checks compile to nothing.
#ifdef FG_DEBUG
constexpr bool kDebugBuild = true;
#else
constexpr bool kDebugBuild = false;
#endif
enum : uint32_t {
    DBG_TMA_A = 0x41,  // A (or LHS scale) box start
    DBG_TMA_B = 0x42,  // B box start
    DBG_TMA_D = 0x43,  // D store box start
    DBG_RING = 0x44,   // operand / scale ring slot or TMEM buffer index
    DBG_TMEM = 0x45,   // TMEM column range of a load or an MMA
    DBG_NONFINITE = 0x46,  // a K-block partial holds Inf or NaN (detail: the K block)
};

__device__ __forceinline__ bool dbg_ok(const GemmParams &p, bool ok, uint32_t tag, int value) {
    if constexpr (kDebugBuild) {
        if (!ok) {
            record_error(p, DEV_ERR_CHECK, (tag << 24) | ((uint32_t)value & 0xFFFFFFu));
            return false;
        }
    }
    return true;
}

// A box starting at (x, y) in [0, x_end) x [0, y_end).  Stores pass the row
// extent; loads pass load_row_limit() of it: a load box may start up to one
// 256-row tile past the end (the missing rows of a partial tile are loaded as
// zeros, never stored).
__device__ __forceinline__ bool dbg_box(const GemmParams &p, int x, int x_end, int y, int y_end, uint32_t tag) {
    return dbg_ok(p, x >= 0 && x < x_end, tag, x) && dbg_ok(p, y >= 0 && y < y_end, tag, y);
}

__device__ __forceinline__ int load_row_limit(int rows) { return rows + 256; }

// TMA store of one staged box of D at column x, row d_row (K-grouped: of the
// group's output plane, the map's third coordinate).
template <int KIND>
__device__ __forceinline__ void store_d_box(const CUtensorMap *map, uint32_t src, int x, int d_row, int group,
                                            const GemmParams &p) {
    if constexpr (KIND == KIND_KGROUPED) {
        if (dbg_box(p, x, p.n, d_row, p.rows, DBG_TMA_D) && dbg_ok(p, group < p.num_groups, DBG_TMA_D, group))
            tma_store_3d(map, src, x, d_row, group);
    } else {
        if (dbg_box(p, x, p.n, d_row, p.a_rows_total, DBG_TMA_D)) tma_store_2d(map, src, x, d_row);
    }
}

struct Tile {
    int valid;
    int group;
    int m_blk;      // M block within the group (masked) or within the whole A
    int n_blk;
    int a_row;      // first row of the tile in the 2-D row space of A and D
    int b_row;      // first row of the tile in the 2-D row space of B ([G*n][k])
    int row_limit;  // rows of the tile below the bound (dense m, masked count)
    int kb_lo, kb_hi;  // K-grouped layout: the tile's K blocks (its group's segment)
};

// Position of a role's scan over the groups' device-side sizes: group g
// begins at block `first` (K-grouped layout: its first K block; masked
// layout: its first valid M block, or 256-row block on CTA pairs).  Every
// role visits its tiles in increasing order and the tiles of one group are
// consecutive, so the scan moves forward: O(G + tiles) loads per CTA, where a
// scan from group 0 for every tile would cost O(G) per tile.
struct GroupScan {
    int g = 0;
    int first = 0;
};

__device__ __forceinline__ int k_segment_blocks(const GemmParams &p, int g) {
    const int s = __ldg(p.k_sizes + g);
    return s > 0 ? s / BLOCK_K : 0;
}

// M blocks of the whole walk (masked: the valid blocks of all groups).
template <int KIND>
__device__ __forceinline__ int total_m_blocks(const GemmParams &p) {
    if constexpr (KIND == KIND_MASKED) {
        int mb = 0;
        for (int g = 0; g < p.num_groups; ++g)
            mb += (clamp_count(__ldg(p.masked_m + g), p.rows) + BLOCK_M - 1) / BLOCK_M;
        return mb;
    } else {
        return p.num_m_blocks;
    }
}

// Tile t of the persistent walk (CTA c takes tiles c, c + grid, ...).  The M
// blocks are cut into raster groups of `group_m`; the tiles of a group walk its
// N blocks with M varying fastest, so the CTAs running at the same time share
// the group's A rows (kept in L2) while B streams through once per group.
// group_m = 1 makes N vary fastest (B kept in L2, A streamed once).
// K-grouped layout: the tiles of group g (all M x N blocks of its output) come
// before those of group g + 1, each group walked like a dense problem.
template <int BN, int KIND>
__device__ __forceinline__ Tile get_tile(const GemmParams &p, int t, int mblocks, GroupScan &scan) {
    Tile ti;
    ti.kb_lo = 0;
    ti.kb_hi = p.num_kb;
    if constexpr (KIND == KIND_KGROUPED) {
        const int per_g = mblocks * p.num_n_blocks;
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
    const int gm = min(p.group_m, mblocks - m0);
    const int mb_lin = m0 + rem % gm;
    ti.n_blk = rem / gm;
    if constexpr (KIND == KIND_DENSE || KIND == KIND_KGROUPED) {
        // (K-grouped: A and B are shared by the groups; the group selects the
        // K range and the output plane)
        ti.valid = 1;
        if constexpr (KIND == KIND_DENSE) ti.group = 0;
        ti.m_blk = mb_lin;
        ti.a_row = mb_lin * BLOCK_M;
        ti.b_row = ti.n_blk * BN;
        ti.row_limit = min(BLOCK_M, p.rows - ti.a_row);
    } else if constexpr (KIND == KIND_CONTIGUOUS) {
        const int g = __ldg(p.m_indices + (size_t)mb_lin * BLOCK_M);
        ti.valid = (g >= 0 && g < p.num_groups);
        ti.group = g;
        ti.m_blk = mb_lin;
        ti.a_row = mb_lin * BLOCK_M;
        ti.b_row = g * p.n + ti.n_blk * BN;
        ti.row_limit = BLOCK_M;
    } else {
        // the group holding valid M block mb_lin, by the role's forward scan
        if (mb_lin < scan.first) scan = GroupScan{};
        int g = scan.g, acc = scan.first, cnt = 0;
        for (; g < p.num_groups; ++g) {
            cnt = clamp_count(__ldg(p.masked_m + g), p.rows);
            const int nb = (cnt + BLOCK_M - 1) / BLOCK_M;
            if (mb_lin < acc + nb) break;
            acc += nb;
        }
        scan.g = g;
        scan.first = acc;
        ti.valid = g < p.num_groups;
        ti.group = g;
        ti.m_blk = mb_lin - acc;
        ti.a_row = g * p.rows + ti.m_blk * BLOCK_M;
        ti.b_row = g * p.n + ti.n_blk * BN;
        ti.row_limit = min(BLOCK_M, cnt - ti.m_blk * BLOCK_M);
    }
    return ti;
}

// Spin part of a bounded mbarrier wait: polls until the phase completes, the
// CTA's abort flag rises (false) or the watchdog limit passes (records
// FG_ERR_TIMEOUT with the role, raises the abort flag, false).
__device__ __forceinline__ bool wait_phase_spin(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                                const GemmParams &p, uint32_t role) {
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if ((++spins & 31u) == 0u && global_timer_ns() - t0 > p.timeout_ns) {
            record_error(p, DEV_ERR_TIMEOUT, (role << 24) | (bar & 0xFFFFu));
            *abort_flag = 1u;
            return false;
        }
    }
    return true;
}

static __device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                                    const GemmParams &p, uint32_t role) {
    return wait_phase_spin(bar, parity, abort_flag, p, role);
}

// Bounded wait on an mbarrier phase.  Returns false on watchdog expiry (after
// recording it and raising the CTA abort flag) or when another role aborted.
// The first probe is inline in both forms.  wait_phase keeps the spin loop
// inline too; wait_phase_call makes it a call, which keeps the caller's loop
// smaller.  Measured on 4096 x 7168 x 8192: the one-CTA kernel's K-grouped
// form runs 5% faster with the inline spin (dense: the same), the CTA-pair
// kernel 4% slower, so the one-CTA kernel waits inline and the others call.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                           const GemmParams &p, uint32_t role) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_phase_spin(bar, parity, abort_flag, p, role);
}

__device__ __forceinline__ bool wait_phase_call(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                                const GemmParams &p, uint32_t role) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_phase_slow(bar, parity, abort_flag, p, role);
}

// Bounded wait that ignores the abort flag: used after an abort to let copies
// and MMAs already in flight land before the CTA frees its resources.
__device__ __forceinline__ bool drain_phase(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_global_v4(void *ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Tensor maps: A [rows][k] u8, B [G*n][k] u8, D [rows][n] bf16 or (F32OUT) fp32
// (all 2-D, 128-byte swizzle; D boxes of 32 rows x 128 bytes); SA over the
// MN-major LHS scales: 2-D {rows, kb} (dense, contiguous) or 3-D {M_cap, kb, G}
// (masked), fp32, no swizzle, box of 128 rows.
template <int BN, int STAGES, int KIND, bool SPLITK, bool F32OUT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ CUtensorMap tmap_sa,
                    const GemmParams p) {
    static_assert(BN == 128 || BN == 256, "BN must be 128 or 256");
    using L = SmemLayout<BN, STAGES>;
    static_assert(!SPLITK || L::PARTIAL_FITS, "split-K: the partial tile must fit in the operand ring");
    constexpr int COLS = BN / 2;  // columns per promotion warp
    // TMEM columns loaded per tcgen05.wait::ld.  Tensor-bound layouts load the
    // warp's whole share behind one wait (the buffer goes back to the MMA warp
    // sooner: 2% less time on the contiguous workloads, 0.8% on K-grouped ones,
    // bitwise the same); the masked layout measured 1-2% slower that way and the
    // debug build's finite-value check would spill, so both keep 32.
    constexpr int LD_COLS = (kDebugBuild || KIND == KIND_MASKED) ? TMEM_LD_COLS : COLS;
    constexpr uint32_t STAGE_TX = A_STAGE_BYTES + L::B_STAGE_BYTES;
    constexpr uint32_t NTB = L::NUM_TBUF;  // TMEM accumulator buffers (a power of two)
    static_assert((NTB & (NTB - 1)) == 0 && NTB >= 2, "TMEM buffer count");

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

    // warp index through a shuffle so the compiler knows it is warp-uniform
    // (TMEM addresses derived from it then stay in uniform registers)
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    // The 128-byte swizzled TMA tiles need a 1024-byte aligned base.
    if (sbase & 1023u) {
        if (threadIdx.x == 0) record_error(p, DEV_ERR_CHECK, (ROLE_SETUP << 24) | (sbase & 0xFFFFu));
        return;
    }

    // ------------------------------------------------------------- set-up
    // The producer warp initializes the barriers and starts loading right
    // away; the other warps wait (named barrier 1) for the barriers and for the
    // TMEM allocation, which only they need.
    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            prefetch_tensormap(&tmap_a);
            prefetch_tensormap(&tmap_b);
            prefetch_tensormap(&tmap_sa);
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
    const uint32_t tmem_base = warp == PRODUCER_WARP ? 0u : *tmem_slot;  // the producer never uses TMEM

    // Everything above touches only this CTA's own resources; global memory
    // may still be in use by the previous grid of the stream until here.
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
        // segment lengths must be multiples of 128 and fit in K; others are
        // reported (the walk rounds them down and clips them to K)
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

    const int m_blocks = total_m_blocks<KIND>(p);
    const int num_tiles = m_blocks * p.num_n_blocks * (KIND == KIND_KGROUPED ? p.num_groups : 1);
    // This CTA's work: persistent tiles t_begin, t_begin + t_step, ... over all
    // K blocks, or (split-K) the one tile of its cluster over its K range.
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
            GroupScan scan;
            for (int t = t_begin; t < num_tiles && ok; t += t_step) {
                const Tile ti = get_tile<BN, KIND>(p, t, m_blocks, scan);
                if (!ti.valid) continue;
                // RHS block scales of the two column halves of this tile
                const int nb0 = min((ti.n_blk * BN) / 128, p.num_nb - 1);
                const int nb1 = min((ti.n_blk * BN + BN / 2) / 128, p.num_nb - 1);
                const int bgroup = KIND == KIND_KGROUPED ? 0 : ti.group;  // K-grouped: one B for all groups
                const float *sb0 = p.sB + ((size_t)bgroup * p.num_nb + nb0) * p.num_kb;
                const float *sb1 = p.sB + ((size_t)bgroup * p.num_nb + nb1) * p.num_kb;
                const int kb_stop = KIND == KIND_KGROUPED ? ti.kb_hi : kb_end;
                for (int kb = KIND == KIND_KGROUPED ? ti.kb_lo : kb_begin; kb < kb_stop; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    const uint32_t q = it % SCALE_STAGES, qph = (it / SCALE_STAGES) & 1u;
                    if (!wait_phase(empty_bar(s), ph ^ 1u, abort_flag, p, ROLE_PRODUCER) ||
                        !wait_phase(sempty_bar(q), qph ^ 1u, abort_flag, p, ROLE_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    if ((int)it == p.debug_skip_iter) continue;
                    int ax = kb * BLOCK_K;
                    if constexpr (kDebugBuild) {
                        if ((int)it == p.debug_bad_coord) ax += p.num_kb * BLOCK_K;
                        const int sa_rows = KIND == KIND_MASKED ? p.rows : p.a_rows_total;
                        const int sa_row = KIND == KIND_MASKED ? ti.m_blk * BLOCK_M : ti.a_row;
                        if (!(dbg_ok(p, s < (uint32_t)STAGES && q < (uint32_t)SCALE_STAGES, DBG_RING, (int)it) &&
                              dbg_box(p, ax, p.k, ti.a_row, load_row_limit(p.a_rows_total), DBG_TMA_A) &&
                              dbg_box(p, kb * BLOCK_K, p.k, ti.b_row, load_row_limit(p.b_rows_total), DBG_TMA_B) &&
                              dbg_box(p, kb, p.num_kb, sa_row, load_row_limit(sa_rows), DBG_TMA_A) &&
                              dbg_ok(p, ti.group >= 0 && ti.group < p.num_groups, DBG_TMA_B, ti.group))) {
                            *abort_flag = 1u;
                            ok = false;
                            break;
                        }
                    }
                    mbar_arrive_expect_tx(full_bar(s), STAGE_TX);
                    tma_load_2d(sbase + L::A_OFF + s * A_STAGE_BYTES, &tmap_a, full_bar(s), ax, ti.a_row);
                    tma_load_2d(sbase + L::B_OFF + s * L::B_STAGE_BYTES, &tmap_b, full_bar(s), kb * BLOCK_K,
                                ti.b_row);
                    mbar_arrive_expect_tx(sfull_bar(q), SA_STAGE_BYTES);
                    if constexpr (KIND == KIND_MASKED)
                        tma_load_3d(sbase + L::SA_OFF + q * SA_STAGE_BYTES, &tmap_sa, sfull_bar(q),
                                    ti.m_blk * BLOCK_M, kb, ti.group);
                    else
                        tma_load_2d(sbase + L::SA_OFF + q * SA_STAGE_BYTES, &tmap_sa, sfull_bar(q), ti.a_row, kb);
                    cp_async_4(sbase + L::SB_OFF + q * SB_STAGE_BYTES, sb0 + kb);
                    cp_async_4(sbase + L::SB_OFF + q * SB_STAGE_BYTES + 4, sb1 + kb);
                    cp_async_mbar_arrive_noinc(sfull_bar(q));
                }
            }
            if (!ok) {
                // let the copies still in flight land before the CTA exits
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
            GroupScan scan;
            for (int t = t_begin; t < num_tiles && ok; t += t_step) {
                const Tile ti = get_tile<BN, KIND>(p, t, m_blocks, scan);
                if (!ti.valid) continue;
                const int kb_stop = KIND == KIND_KGROUPED ? ti.kb_hi : kb_end;
                for (int kb = KIND == KIND_KGROUPED ? ti.kb_lo : kb_begin; kb < kb_stop; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    const uint32_t b = it & (NTB - 1u), bph = (it / NTB) & 1u;
                    if (!wait_phase(tempty_bar(b), bph ^ 1u, abort_flag, p, ROLE_MMA) ||
                        !wait_phase(full_bar(s), ph, abort_flag, p, ROLE_MMA)) {
                        ok = false;
                        break;
                    }
                    if constexpr (kDebugBuild) {
                        if (!dbg_ok(p, s < (uint32_t)STAGES && b < NTB && (b + 1) * BN <= L::TMEM_COLS, DBG_TMEM,
                                    (int)it)) {
                            *abort_flag = 1u;
                            ok = false;
                            break;
                        }
                    }
                    tc_fence_after();
                    const uint64_t adesc = make_desc_kmajor_sw128(sbase + L::A_OFF + s * A_STAGE_BYTES);
                    const uint64_t bdesc = make_desc_kmajor_sw128(sbase + L::B_OFF + s * L::B_STAGE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BLOCK_K / MMA_K; ++kk) {
                        // advance the start address by kk * 32 bytes inside the swizzle atom
                        const uint64_t koff = (uint64_t)((kk * MMA_K) >> 4);
                        mma_f8f6f4(tmem_base + b * BN, adesc + koff, bdesc + koff, p.idesc, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(empty_bar(s));
                    mma_commit(tfull_bar(b));
                }
            }
            if (!ok) {
                // every MMA issued so far must finish before TMEM is freed
                mma_commit(drain_bar);
                drain_phase(drain_bar, 0u, p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp < NUM_EPI_WARPS) {
        // ------------------------------------------ promotion + epilogue warps
        const int sub = warp & 3;   // TMEM lane quarter: rows [32*sub, 32*sub+32)
        const int half = warp >> 2; // column half: [half*COLS, half*COLS+COLS)
        const int r = sub * 32 + lane;
        const uint32_t stg = sbase + L::STG_OFF + warp * STAGING_BYTES_PER_WARP;
        const uint32_t t_lane = (uint32_t)(sub * 32) << 16;
        const uint32_t sa_addr = sbase + L::SA_OFF + r * 4;
        const uint32_t sb_addr = sbase + L::SB_OFF + half * 4;
        const uint32_t t_base = tmem_base + t_lane + half * COLS;
        // ring positions, advanced incrementally: TMEM buffer b (phase bph) and
        // scale-ring entry q (phase qph) of the current K iteration
        uint32_t b = 0, bph = 0, q = 0, qph = 0;
        bool ok = true;
        GroupScan scan;
        for (int t = t_begin; t < num_tiles && ok; t += t_step) {
            const Tile ti = get_tile<BN, KIND>(p, t, m_blocks, scan);
            if (!ti.valid) {
                if constexpr (KIND == KIND_CONTIGUOUS) {
                    // a skipped block must be all padding (-1 rows); a group id
                    // elsewhere in it breaks the 128-row alignment contract
                    if (ti.group != -1) {
                        if (warp == 0 && lane == 0) record_error(p, DEV_ERR_CHECK, (uint32_t)t);
                    } else if (half == 0 && ti.n_blk == 0) {
                        const int gid = __ldg(p.m_indices + ti.a_row + r);
                        if (gid != -1) record_error(p, DEV_ERR_CHECK, (uint32_t)(ti.a_row + r));
                    }
                }
                continue;
            }
            // which rows of this warp are written
            bool row_ok;
            if constexpr (KIND == KIND_CONTIGUOUS) {
                // rows of the tile's group are written, -1 rows are padding; any
                // other id breaks the 128-row alignment contract (not written,
                // reported with the row index)
                const int gid = __ldg(p.m_indices + ti.a_row + r);
                row_ok = gid == ti.group;
                if (gid != ti.group && gid != -1 && half == 0)
                    record_error(p, DEV_ERR_CHECK, (uint32_t)(ti.a_row + r));
            } else {
                row_ok = r < ti.row_limit;
            }
            const int col0 = ti.n_blk * BN + half * COLS;

            uint64_t acc2[COLS / 2];  // FP32 running sums, packed in pairs of columns
#pragma unroll
            for (int j = 0; j < COLS / 2; ++j) acc2[j] = 0ull;

            // (K-grouped: an empty segment leaves the sums at zero, and zeros are stored)
            const int kb_stop = KIND == KIND_KGROUPED ? ti.kb_hi : kb_end;
            for (int kb = KIND == KIND_KGROUPED ? ti.kb_lo : kb_begin; kb < kb_stop; ++kb) {
                const bool got = wait_phase(sfull_bar(q), qph, abort_flag, p, ROLE_EPILOGUE) &&
                                 wait_phase(tfull_bar(b), bph, abort_flag, p, ROLE_EPILOGUE);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                if constexpr (kDebugBuild) {
                    const bool in = dbg_ok(p,
                                           b < NTB && q < (uint32_t)SCALE_STAGES &&
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
                        // all of this K block's partial is in registers: hand the
                        // TMEM buffer back to the MMA warp before the last FMAs
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(tempty_bar(b));
                    }
#pragma unroll
                    for (int j = 0; j < LD_COLS; j += 2)
                        ffma2(acc2[(c * LD_COLS + j) / 2], v[j], v[j + 1], sc2);
                }
                b = (b + 1u) & (NTB - 1u);
                bph ^= (b == 0u);
                q = (q + 1u) & (SCALE_STAGES - 1u);
                qph ^= (q == 0u);
            }
            if (!ok) break;

            if constexpr (SPLITK) {
                if (split > 1) {
                    // partial tile -> own shared memory (the operand ring is idle
                    // now: every MMA that read it has completed), rows of BN FP32
                    // with the 16-byte chunks of row r rotated by (r & 7)
                    const uint32_t prow = sbase + L::P_OFF + (uint32_t)r * (BN * 4);
#pragma unroll
                    for (int ch = 0; ch < COLS / 4; ++ch) {
                        const int cg = half * (COLS / 4) + ch;  // chunk index within the row
                        float x0, x1, x2, x3;
                        unpack_f32x2(acc2[2 * ch], x0, x1);
                        unpack_f32x2(acc2[2 * ch + 1], x2, x3);
                        st_shared_v4(prow + (uint32_t)((cg ^ (r & 7)) << 4), __float_as_uint(x0),
                                     __float_as_uint(x1), __float_as_uint(x2), __float_as_uint(x3));
                    }
                    continue;  // the cluster reduction below writes D
                }
            }

            // ---------------------------------------------------- epilogue
            float acc[COLS];
#pragma unroll
            for (int j = 0; j < COLS / 2; ++j) unpack_f32x2(acc2[j], acc[2 * j], acc[2 * j + 1]);
            // first row of this warp's block in D (K-grouped: within the group's
            // output plane, the third coordinate of D's tensor map)
            const int d_row = ti.a_row + sub * 32;
            constexpr bool CLIPPED = KIND == KIND_DENSE || KIND == KIND_KGROUPED;
            bool use_tma;
            if constexpr (CLIPPED)
                use_tma = true;  // rows past m are clipped by the tensor map bounds
            else
                use_tma = __all_sync(0xffffffffu, row_ok);
            if (use_tma) {
                const bool rows_in = !CLIPPED || (sub * 32 < ti.row_limit);
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
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    if constexpr (SPLITK) {
        if (split > 1) {
            // every CTA of the cluster takes both barriers, whatever happened above
            cluster_sync();
            // a rank whose watchdog fired left its partial incomplete: then no
            // rank writes D (the status word already records the timeout)
            bool any_abort = false;
            for (uint32_t q = 0; q < split; ++q)
                any_abort |= ld_shared_cluster_u32(map_shared_rank(smem_u32((const void *)abort_flag), q)) != 0u;
            const bool tile_ok = t_begin < num_tiles && !any_abort;
            if (tile_ok && warp < NUM_EPI_WARPS) {
                GroupScan scan;
                const Tile ti = get_tile<BN, KIND>(p, t_begin, m_blocks, scan);
                if (ti.valid) {
                    constexpr int CH = BN / 4;  // 16-byte chunks per partial row
                    constexpr int MAX_SPLIT = 8;
                    constexpr int STRIDE = NUM_EPI_WARPS * 32;
                    // rows of the tile that are written, shared evenly by the ranks
                    // (contiguous: all 128, the per-row group test below decides)
                    const int nrows = KIND == KIND_CONTIGUOUS ? BLOCK_M : max(0, min(BLOCK_M, ti.row_limit));
                    const int r0 = (int)((nrows * rank) / split), r1 = (int)((nrows * (rank + 1)) / split);
                    const int col_base = ti.n_blk * BN;
                    const int items = (r1 - r0) * CH;
                    // two chunks per thread per pass, all ranks' loads issued before any
                    // use so the distributed-shared-memory latency is paid once per pass
                    for (int base = threadIdx.x; base < items; base += 2 * STRIDE) {
                        float4 v[2][MAX_SPLIT];
                        bool live[2];
                        int row[2], col[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int item = base + u * STRIDE;
                            row[u] = r0 + item / CH;
                            const int ch = item % CH;
                            col[u] = col_base + ch * 4;
                            bool ok_row;
                            if (item >= items) {
                                ok_row = false;
                            } else if constexpr (KIND == KIND_CONTIGUOUS) {
                                ok_row = __ldg(p.m_indices + ti.a_row + row[u]) == ti.group;
                            } else {
                                ok_row = row[u] < ti.row_limit;
                            }
                            live[u] = ok_row && col[u] < p.n;
                            const uint32_t local = sbase + L::P_OFF + (uint32_t)row[u] * (BN * 4) +
                                                   (uint32_t)((ch ^ (row[u] & 7)) << 4);
#pragma unroll
                            for (int q = 0; q < MAX_SPLIT; ++q)
                                if (live[u] && q < (int)split) v[u][q] = ld_shared_cluster_v4(map_shared_rank(local, q));
                        }
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            if (!live[u]) continue;
                            float4 sum = v[u][0];
#pragma unroll
                            for (int q = 1; q < MAX_SPLIT; ++q) {  // fixed rank (= K) order
                                if (q < (int)split) {
                                    sum.x += v[u][q].x;
                                    sum.y += v[u][q].y;
                                    sum.z += v[u][q].z;
                                    sum.w += v[u][q].w;
                                }
                            }
                            const size_t d_off = (size_t)(ti.a_row + row[u]) * p.n + col[u];
                            if constexpr (F32OUT) {
                                *reinterpret_cast<float4 *>(static_cast<float *>(p.D) + d_off) = sum;
                            } else {
                                uint2 w;
                                w.x = pack_bf16x2(sum.x, sum.y);
                                w.y = pack_bf16x2(sum.z, sum.w);
                                *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.D) + d_off) = w;
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
