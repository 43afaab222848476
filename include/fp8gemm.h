/*
 * fp8gemm.h -- C ABI of the GB300 (sm_103a) FP8 NT GEMM library.
 *
 * The operation (page "DeepSeek开源周第三天DeepGEMM", sections "核心功能",
 * "基本用法" and the promotion excerpt "两级精度累加与细粒度缩放"):
 *
 *   D[m,n] = bf16( sum_kb sA[m,kb] * sB[n/128,kb] * sum_{k in kb} A[m,k] * B[n,k] )
 *
 * A (LHS) is an FP8 m x k matrix, B (RHS) an FP8 n x k matrix (both K-major:
 * the "NT" layout, B is stored transposed), sA holds one FP32 scale per row
 * and 128-wide K block (1x128 groups), sB one FP32 scale per 128x128 block.
 * kb runs over ceil(k/128) K blocks.  Each K block is multiplied on the tensor
 * cores into a fresh FP32 partial, which is then scaled by sA*sB and added to
 * an FP32 running sum on the CUDA cores (the page's two-level accumulation).
 * The output is BF16, rounded to nearest even.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All pointers named A, B, sA, sB, D, m_indices, masked_m are DEVICE
 *   pointers owned by the caller; the library keeps no reference after the
 *   call returns.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Calls are asynchronous on that stream: they allocate nothing, never
 *   synchronize the host and read no device data on the host, so they can be
 *   captured in a CUDA graph.
 * - FP8 formats: FG_E4M3 (float8 e4m3 "fn": max 448, no infinities) or
 *   FG_E5M2 (max 57344).  A and B may use different formats.
 * - Layouts (row-major, leading dimension = row length unless stated):
 *     A   [rows][k] bytes                      16-byte aligned, k % 16 == 0
 *     B   [G][n][k] bytes (dense: G = 1)       16-byte aligned
 *     sA  MN-major: [kb][ld_sA] floats, i.e. the scales of K block kb for all
 *         rows are contiguous (masked layout: [G][kb][ld_sA]);
 *         ld_sA >= rows (M_cap for masked), ld_sA % 4 == 0, sA 16-byte
 *         aligned (each K block's column is fetched by TMA).  Entries past
 *         the rows are never used.  fg_scales_a_to_mn_major() builds this
 *         layout from the row-major [rows][kb] one.
 *     sB  [G][ceil(n/128)][ceil(k/128)] floats, row-major
 *     D   [rows][n] bfloat16 (masked: [G][M_cap][n]), 16-byte aligned, n % 8 == 0
 * - A K block that runs past k (k % 128 != 0) contributes only its first
 *   k % 128 columns; the scale of that block still applies.
 * - Errors found on the host are returned at once (nothing is launched).
 *   Errors found by the kernel (a wait that exceeded the watchdog limit, a
 *   group id, count or segment length out of range) are recorded in a
 *   per-device status word and read with fg_get_device_status().
 * - The same ABI is exported by the FG_DEBUG build of the library
 *   (libfp8gemm_debug.so): single-stage pipelines and a device-side check of
 *   every TMA box start, ring index and TMEM column before use.  A failed
 *   check records FG_ERR_DEVICE_CHECK with a tag in bits 24..31 of the detail
 *   (0x41 A or LHS-scale box, 0x42 B box, 0x43 D box, 0x44 ring slot, 0x45
 *   TMEM columns, 0x46 a non-finite K-block partial) and the offending value
 *   in bits 0..23, and the access is skipped.  For bisecting races, not speed.
 */
#ifndef FP8GEMM_H_
#define FP8GEMM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fg_status {
    FG_OK = 0,
    FG_ERR_INVALID_ARG = 1,   /* null pointer, negative or inconsistent size, bad format  */
    FG_ERR_MISALIGNED = 2,    /* pointer or leading dimension breaks a 16-byte rule        */
    FG_ERR_UNSUPPORTED = 3,   /* shape outside what the kernels support (e.g. k % 16 != 0) */
    FG_ERR_CUDA = 4,          /* a CUDA runtime / driver call failed                       */
    FG_ERR_TIMEOUT = 5,       /* device: a pipeline wait exceeded the watchdog limit       */
    FG_ERR_DEVICE_CHECK = 6   /* device: group id or masked count out of range             */
} fg_status;

typedef enum fg_fp8 { FG_E4M3 = 0, FG_E5M2 = 1 } fg_fp8;

/* Dense NT GEMM ("普通密集GEMM"): D[m][n] = A[m][k] x B[n][k]^T with the
 * fine-grained scales above.  All m x n outputs are written.  m == 0 is a
 * no-op; n, k >= 1 are required. */
fg_status fg_gemm_fp8_nt(const void *A, int a_fmt, const float *sA, int ld_sA,
                         const void *B, int b_fmt, const float *sB,
                         void *D, int m, int n, int k, void *stream);

/* Contiguous-layout grouped GEMM ("连续布局分组GEMM": groups concatenated on
 * the M axis, each row tagged with its group).  A is [M][k]; B holds G weight
 * matrices [G][n][k]; m_indices[r] (int32, device) is the group of row r.
 * Segments are aligned to 128 rows: within each 128-row tile every row carries
 * either the group id of the tile's first row or -1 (padding).  Rows whose id
 * equals the tile's group are written with A[r] x B[g]^T; all other rows of D
 * are left untouched.  A tile whose first id is outside [0, G) is skipped (and
 * recorded as FG_ERR_DEVICE_CHECK unless it is -1).  Input that breaks the
 * alignment contract is reported, never computed: a row whose id is neither
 * -1 nor its tile's group, or a group id inside a tile whose first row is -1,
 * is left untouched and recorded as FG_ERR_DEVICE_CHECK with the row index as
 * the detail.  M % 128 == 0. */
fg_status fg_grouped_gemm_fp8_contiguous(const void *A, int a_fmt, const float *sA, int ld_sA,
                                         const void *B, int b_fmt, const float *sB, void *D,
                                         const int32_t *m_indices, int M, int n, int k, int G,
                                         void *stream);

/* Masked-layout grouped GEMM ("掩码布局分组GEMM": a fixed capacity per group
 * and a device-side count of valid rows, so the host needs no knowledge of the
 * counts and the call is CUDA-graph friendly).  A is [G][M_cap][k], sA is
 * [G][kb][ld_sA], D is [G][M_cap][n]; masked_m[g] (int32, device) rows of group
 * g are valid.  Rows r < masked_m[g] are written; all other rows are left
 * untouched.  A count outside [0, M_cap] is clamped into it and recorded as
 * FG_ERR_DEVICE_CHECK. */
fg_status fg_grouped_gemm_fp8_masked(const void *A, int a_fmt, const float *sA, int ld_sA,
                                     const void *B, int b_fmt, const float *sB, void *D,
                                     const int32_t *masked_m, int G, int M_cap, int n, int k,
                                     void *stream);

/* FP32-output forms of the three calls above (page whose first section is
 * "从一张“算力账单”说起", section 4.2 "基础矩阵乘法的调用与验证": the output is
 * BF16 by default, FP32 on request at some cost in speed).  Arguments,
 * layouts, written rows and errors are those of the BF16 calls; D is float
 * [rows][n] (masked: [G][M_cap][n]), 16-byte aligned, and receives the FP32
 * result of the two-level accumulation without the final rounding to BF16
 * (rounding it to BF16, nearest even, gives the BF16 call's result bit for
 * bit).  Tile plans are chosen as for BF16 output. */
fg_status fg_gemm_fp8_nt_f32out(const void *A, int a_fmt, const float *sA, int ld_sA,
                                const void *B, int b_fmt, const float *sB,
                                float *D, int m, int n, int k, void *stream);
fg_status fg_grouped_gemm_fp8_contiguous_f32out(const void *A, int a_fmt, const float *sA, int ld_sA,
                                                const void *B, int b_fmt, const float *sB, float *D,
                                                const int32_t *m_indices, int M, int n, int k, int G,
                                                void *stream);
fg_status fg_grouped_gemm_fp8_masked_f32out(const void *A, int a_fmt, const float *sA, int ld_sA,
                                            const void *B, int b_fmt, const float *sB, float *D,
                                            const int32_t *masked_m, int G, int M_cap, int n, int k,
                                            void *stream);

/* K-grouped GEMM: groups concatenated along K, one NT product per group over
 * its own segment of the K axis -- the weight-gradient step of MoE training,
 * which contracts over each expert's tokens (page "DeepSeek开源周第三天DeepGEMM",
 * section "DeepGEMM提供三种FP8GEMM实现", names the grouped kinds by the training
 * forward pass and inference; this is the same scaled product with the K range
 * restricted per group, the reading this library takes for the backward step).
 *
 *   D[g][m][n] = sum over the K blocks kb of segment g of
 *                sA[m,kb] * sB[n/128,kb] * sum_{k in kb} A[m,k] * B[n,k]
 *
 *   A   [M][K] FP8 (K-major: the token axis contiguous), shared by all groups
 *   B   [N][K] FP8 (K-major), shared by all groups
 *   sA  MN-major [ceil(K/128)][ld_sA] floats, ld_sA >= M, ld_sA % 4 == 0
 *   sB  [ceil(N/128)][ceil(K/128)] floats
 *   k_sizes [G] int32 on the device: group g covers K columns
 *       [k_sizes[0] + ... + k_sizes[g-1], ... + k_sizes[g]); every length a
 *       multiple of 128 (K blocks never straddle groups), their sum <= K.
 *       The host never reads them (graph-capturable); a length that is
 *       negative or not a multiple of 128, or a sum past K, is recorded as
 *       FG_ERR_DEVICE_CHECK (detail: the group, or G for the sum) and the
 *       walk rounds it down / clips it to K.
 *   D   [G][M][N] bfloat16 (the _f32out form: float), 16-byte aligned; every
 *       element is written (an empty segment gives zeros).
 * K % 16 == 0, N % 8 == 0; M == 0 is a no-op.  Tiles: for the BF16 form
 * with M >= 256, 256 x 256 on CTA pairs (with the store warp when the
 * segments average 4 to 12 K blocks, where it measured faster), else
 * 128 x 256 or, when those would leave SMs idle, 128 x 128 on one CTA;
 * fg_query_plan with kind 3 reports the choice. */
fg_status fg_k_grouped_gemm_fp8_nt(const void *A, int a_fmt, const float *sA, int ld_sA,
                                   const void *B, int b_fmt, const float *sB, void *D,
                                   const int32_t *k_sizes, int G, int M, int N, int K, void *stream);
fg_status fg_k_grouped_gemm_fp8_nt_f32out(const void *A, int a_fmt, const float *sA, int ld_sA,
                                          const void *B, int b_fmt, const float *sB, float *D,
                                          const int32_t *k_sizes, int G, int M, int N, int K,
                                          void *stream);

/* Layout helper (the page's "LHS scales must be TMA-aligned and transposed",
 * section "基本用法"): src is row-major [batches][rows][kb], dst receives
 * [batches][kb][ld_dst] with ld_dst >= rows, ld_dst % 4 == 0; padding entries
 * are set to 0.  Device pointers, asynchronous on `stream`. */
fg_status fg_scales_a_to_mn_major(const float *src, float *dst, int batches, int rows, int kb,
                                  int ld_dst, void *stream);

/* Per-token FP8 quantization of activations: the step that produces a GEMM
 * call's LHS (page "DeepSeek开源周第三天DeepGEMM", section "基本用法": FP8 LHS
 * with one FP32 scale per row and 128-wide K block, scales in the MN-major
 * layout; page "企业官网建设流程全解析", section 5.2: each scale comes from a
 * scan of its group for the largest magnitude).  For row r of batch b and K
 * block kb, over the block's columns inside k:
 *
 *   amax = max |X|,  sA = amax / fmax (1 when amax == 0),  A = fp8(X / sA)
 *
 * with fmax 448 (E4M3) or 57344 (E5M2), float32 IEEE divisions and round to
 * nearest even, saturating at +-fmax.
 *   X   [batches][rows][ld_x] bfloat16 (device), 16-byte aligned, ld_x >= k,
 *       ld_x % 8 == 0; finite values (codes for Inf/NaN inputs are unspecified)
 *   A   [batches][rows][k] FP8 bytes (device), 16-byte aligned, k % 16 == 0
 *   sA  [batches][ceil(k/128)][ld_sA] floats (device), 16-byte aligned,
 *       ld_sA >= rows, ld_sA % 4 == 0: the layout every GEMM call above takes
 *       (dense and contiguous: batches = 1; masked: batches = G, rows = M_cap)
 *   masked_m  NULL (all rows), or [batches] int32 counts on the device: rows
 *       r >= masked_m[b] of A and sA are left untouched; a count outside
 *       [0, rows] is clamped into it and recorded as FG_ERR_DEVICE_CHECK
 *       (detail: the batch index).
 * Entries of sA past `rows` are not written.  rows == 0 is a no-op.
 * Asynchronous on `stream`, no allocation, CUDA-graph capturable; launched
 * with programmatic dependent launch when that is on (it then waits for the
 * previous kernel of the stream before its first read). */
fg_status fg_quantize_fp8_per_token(const void *X, int ld_x, int fmt, void *A, float *sA, int ld_sA,
                                    const int32_t *masked_m, int batches, int rows, int k, void *stream);

/* fg_quantize_fp8_per_token with FP32 activations: X [batches][rows][ld_x]
 * float (device), 16-byte aligned, ld_x >= k, ld_x % 4 == 0; finite values.
 * The same per-group amax, scale and codes, computed on the FP32 values (the
 * usage walkthrough quantizes FP32 tensors with amax / 448 before the GEMM:
 * page whose first section is "从一张“算力账单”说起", section 4.2).  Every other
 * argument, contract and error as above. */
fg_status fg_quantize_fp8_per_token_f32in(const float *X, int ld_x, int fmt, void *A, float *sA, int ld_sA,
                                          const int32_t *masked_m, int batches, int rows, int k, void *stream);

/* Smallest valid ld_sA for `rows` rows: rows rounded up to a multiple of 4. */
int fg_scales_a_ld(int rows);

/* Synchronizes `stream`, then returns and clears the calling device's status
 * word (FG_OK when no kernel recorded an error).  `detail` (may be NULL)
 * receives a code saying where: for FG_ERR_TIMEOUT the role (1 producer,
 * 2 MMA, 3 epilogue) in bits 24..31; for FG_ERR_DEVICE_CHECK the offending
 * group or tile index. */
fg_status fg_get_device_status(void *stream, uint32_t *detail);

/* Tuning and testing knobs.  fg_set_num_sms, fg_set_config_override,
 * fg_set_pair_mode, fg_set_programmatic_launch and fg_set_watchdog_ms set
 * PROCESS-WIDE state: each applies to every later call from any thread, on any
 * device and stream, until it is set again.  Threads that want different
 * settings must serialize their set-and-call sequences themselves; a call
 * reads each setting once, when it starts. */

/* Limit the number of SMs (persistent CTAs) used by later calls on any device
 * ("SM资源控制"); 0 restores the default (all SMs). */
fg_status fg_set_num_sms(int num_sms);

/* Tuning / testing override of the tile plan of later calls: block_n
 * (output tile width, 128 or 256; 0 = automatic) and split_k (number of CTAs,
 * one thread-block cluster, that share the K blocks of one output tile and
 * reduce their partials through distributed shared memory in a fixed order;
 * 1 = no split, 0 = automatic, at most 8).  Results differ between plans only
 * by FP32 summation order. */
fg_status fg_set_config_override(int block_n, int split_k);

/* The tile plan a dense call of this shape would use on the current device:
 * output tile width (*block_n) and split-K cluster size (*split_k, 1 = none).
 * Host-only query (reads device attributes, launches nothing). */
fg_status fg_query_dense_plan(int m, int n, int k, int *block_n, int *split_k);

/* Same, plus whether the call runs on CTA pairs (*cta_pair = 1): 256 x 256
 * output tiles shared by the two CTAs (two SMs) of a cluster, one
 * tcgen05.mma.cta_group::2 per 32-deep K step, each CTA loading its 128 rows
 * of A and its 128 of the tile's 256 rows of B.  The pages' design has no
 * counterpart (Hopper has no paired tensor-core instruction). */
fg_status fg_query_dense_plan_ex(int m, int n, int k, int *block_n, int *split_k, int *cta_pair);

/* CTA-pair tiles for later calls: -1 (default) where they apply (persistent
 * 256-wide dense plans with at least 256 rows, K-grouped BF16 calls with at
 * least 256 rows; no forced plan), 0 never, 1 for every persistent 256-wide
 * plan of any layout.  The contiguous and masked layouts use 128-row tiles
 * unless the mode is 1.  Contiguous: a pair tile whose two 128-row blocks
 * belong to two groups runs once per group, each pass storing its group's
 * rows; measured within about 2% of 128-row tiles on the contiguous workloads
 * and 21% slower when every pair straddles two groups.  Masked: a 256-row tile
 * also computes a group's empty rows past its count; measured slower.  Results
 * differ between the modes only by FP32 summation order (measured bitwise
 * equal on the contiguous workloads); FG_ERR_INVALID_ARG for other values. */
fg_status fg_set_pair_mode(int mode);

/* Swapped operand roles ("swap-AB") for later calls: the weights (B) take the
 * tensor core's 128-row role and the rows of A (tokens, at most 256 per tile)
 * its N role, so a group with few rows multiplies, loads and promotes no empty
 * rows, and a masked call launches tiles only over the weights of the groups
 * that have rows.  The output, the scales and every other contract are those
 * of the unswapped call; each element still receives sum_kb (sA * sB) * P.
 * Applies to dense calls with m <= 256 and masked calls with M_cap <= 256.
 * -1 (default, automatic) and 0: never -- measured slower than the unswapped
 * plans on every problem of the dense sweep with m <= 128 and of the masked
 * workloads (a swapped tile covers 128 weight rows, so A is read once per 128
 * weights instead of once per 256); 1: wherever it applies (a forced split_k
 * then sets its split-K cluster size).  The pages' design has no counterpart
 * (their small-M path keeps the operand roles).  Results differ from the
 * unswapped path only by FP32 summation order. */
fg_status fg_set_swap_mode(int mode);

/* The tile plan a call of this layout and shape would use on the current
 * device.  kind: 0 dense (rows = m, G = 1), 1 contiguous (rows = M), 2 masked
 * (rows = M_cap), 3 K-grouped (rows = M, n = N, k = K).  plan[5] receives:
 * [0] the tile width (output columns per tile; with swapped roles, rows of A
 * per tile), [1] the split-K cluster size (1 = none), [2] 1 for CTA-pair
 * tiles, [3] 1 for swapped operand roles, [4] 1 when the CTA-pair tiles of a
 * BF16 call stage a whole tile and a store warp issues its stores (tiles of
 * at most 56 K blocks, K-grouped: 4 to 12 on average; the FP32 output forms
 * never do).  Host-only (reads device attributes, launches nothing). */
fg_status fg_query_plan(int kind, int rows, int G, int n, int k, int *plan);

/* Programmatic dependent launch of the GEMM kernels (default on): a call's
 * CTAs may start while the previous kernel of the stream finishes, set up
 * their shared memory, tensor memory and barriers, and wait for the previous
 * kernel to complete before their first global-memory access.  The results
 * are the same either way; 0 turns it off for later calls. */
fg_status fg_set_programmatic_launch(int enable);

/* Watchdog limit of each in-kernel pipeline wait, in milliseconds (default
 * 2000; 0 restores the default). */
fg_status fg_set_watchdog_ms(uint32_t ms);

/* Human-readable name of a status code (static storage). */
const char *fg_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int fg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8GEMM_H_ */
