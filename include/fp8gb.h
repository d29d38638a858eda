/*
 * fp8gb.h -- C ABI of the GB300 (sm_103a) FP8 linear-layer library.
 *
 * The library implements the hot path of FP8 mixed-precision training of a
 * linear layer:
 *   1. fp8_quantize            fused amax + scale + saturating cast of a bf16
 *                              matrix to FP8, rowwise and colwise-transposed
 *                              layouts from one kernel pass;
 *   2. fp8_update_amax_history the delayed-scaling history roll and scale
 *                              update for many tensors in one launch;
 *   3. fp8_scaled_gemm         FP8 x FP8 -> bf16 GEMM with per-tensor or
 *                              per-row / per-column scales in the epilogue
 *                              (fprop, dgrad and wgrad are all this call);
 *   4. fp8_grouped_gemm        the same over variable-size expert groups of a
 *                              Mixture-of-Experts layer.
 * Beyond those: fp8_quantize_rowwise_resident (the rowwise recipe in one
 * cooperative launch), the fused MoE prologues of the rowwise recipe
 * (fp8_permute_quantize, fp8_swiglu_quantize), the MXFP8 recipe (fp8_mx_quantize, fp8_mx_gemm,
 * fp8_mx_grouped_gemm, and the fused MoE prologues fp8_mx_permute_quantize
 * and fp8_mx_swiglu_quantize), and the blockwise recipe
 * (fp8_blockwise_quantize, whose scales feed fp8_mx_gemm).
 *
 * Method sources (page title, section):
 *   - "FP8 training for Flux models" (AMD Primus guide), Configuration >
 *     Key FP8 Parameters: fp8 format "e4m3" or "hybrid", fp8_recipe
 *     ("delayed", "tensorwise", ...), fp8_margin, fp8_amax_history_len,
 *     fp8_amax_compute_algo ("most_recent" or "max"), fp8_wgrad.
 *   - "FP8 Training on MI300X", "Discovered AMD FP8 dtype difference" and
 *     "Patched nanochat/fp8.py": E4M3 forward / E5M2 backward, e4m3fn max
 *     448, e4m3fnuz max 240.
 *   - "How PyTorch FP8 Optimizations on AMD GPUs Reduce LLM Cost ...", What
 *     Happened; "FP8 Training on AMD GPUs with TorchTitan and TorchAO":
 *     rowwise FP8, the colwise-scales kernel (transposed layout), grouped
 *     GEMM for MoE, fused quantize kernels, relaxed atomics.
 *
 * Conventions shared by every entry point
 *   - All pointers are caller-owned DEVICE memory unless the argument name
 *     starts with host_.  The library allocates nothing.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and never synchronises.
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns its status and launches nothing.
 *   - FP8_ERR_CUDA: a CUDA launch or runtime call failed (see
 *     fp8_last_cuda_error()).
 *   - Device-side waits are bounded.  A wait that gives up records an error
 *     word on the device; fp8_sync_status() synchronises the stream and
 *     returns FP8_ERR_TIMEOUT (clearing the word) if that happened.
 *   - Formats are explicit enums.  Nothing is auto-detected.
 */
#ifndef FP8GB_H
#define FP8GB_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP8GB_API __attribute__((visibility("default")))
#else
#define FP8GB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* FP8 formats.  e4m3fn: bias 7, max 448, NaN 0x7F/0xFF, no Inf.  e5m2: bias
 * 15, max 57344, IEEE-style Inf/NaN.  e4m3fnuz: bias 8, max 240; e5m2fnuz:
 * bias 16, max 57344; both fnuz formats have the single NaN 0x80, no Inf and
 * no negative zero -- the AMD formats ("FP8 Training on MI300X", "Discovered
 * AMD FP8 dtype difference": e4m3fnuz forward, e5m2fnuz backward).
 * fp8_quantize and fp8_update_amax_history accept all four; the GEMMs take
 * e4m3fn / e5m2 operands (FP8_ERR_UNSUPPORTED for fnuz). */
typedef enum { FP8_E4M3FN = 0, FP8_E5M2 = 1, FP8_E4M3FNUZ = 2, FP8_E5M2FNUZ = 3 } fp8_format_t;

/* Scaling recipes ("FP8 training for Flux models", fp8_recipe):
 *   DELAYED    cast with the stored per-tensor scale (from the amax history);
 *              the current amax is max-accumulated into the history slot.
 *   TENSORWISE one scale per tensor from the current amax.
 *   ROWWISE    current scaling with one scale per row for the row layout and
 *              one per column (per expert group and column when grouped) for
 *              the colwise-transposed layout. */
typedef enum { FP8_RECIPE_DELAYED = 0, FP8_RECIPE_TENSORWISE = 1, FP8_RECIPE_ROWWISE = 2 } fp8_recipe_kind_t;

/* fp8_amax_compute_algo: most_recent uses the current amax; max uses the
 * maximum over the history window. */
typedef enum { FP8_AMAX_MOST_RECENT = 0, FP8_AMAX_MAX = 1 } fp8_amax_algo_t;

/* The recipe knobs.  kind and margin drive fp8_quantize; history_len and
 * algo drive fp8_update_amax_history (they are carried here so a caller can
 * hold one struct per layer). */
typedef struct {
    int kind;        /* fp8_recipe_kind_t */
    int margin;      /* fp8_margin: scale = fp8_max / amax / 2^margin, 0..64 */
    int history_len; /* fp8_amax_history_len */
    int algo;        /* fp8_amax_algo_t */
} fp8_recipe_t;

typedef enum {
    FP8_OK = 0,
    FP8_ERR_INVALID_ARG = 1,
    FP8_ERR_UNSUPPORTED = 2,
    FP8_ERR_ALIGNMENT = 3,
    FP8_ERR_CUDA = 4,
    FP8_ERR_TIMEOUT = 5
} fp8_status_t;

enum { FP8_LAYOUT_ROW = 1, FP8_LAYOUT_COLT = 2 };      /* bitmask of layouts to emit */
enum { FP8_SCALE_TENSOR = 0, FP8_SCALE_PER_ROW = 1 };  /* GEMM operand scale granularity */
enum { FP8_GROUPED_M = 0, FP8_GROUPED_K = 1, FP8_GROUPED_M_BT = 2 };  /* grouped GEMM modes */

/*
 * fp8_quantize -- fused amax + scale + saturating round-to-nearest-even cast
 * of a bf16 matrix, emitting the row layout, the colwise-transposed layout,
 * or both from one read of x.
 *
 *   x_bf16        [rows][ld_x] bf16, row-major; 16-byte aligned, ld_x % 8 == 0.
 *   rows, cols    rows >= 0, cols >= 1, cols % 8 == 0.
 *   fmt           FP8_E4M3FN, FP8_E5M2, FP8_E4M3FNUZ or FP8_E5M2FNUZ.
 *   recipe        kind and margin are used (see fp8_recipe_t).
 *   layouts       FP8_LAYOUT_ROW | FP8_LAYOUT_COLT (at least one).
 *   scale_in      DELAYED only: device fp32 [1], the stored scale used for the
 *                 cast (NULL otherwise).
 *   amax_out      DELAYED: device fp32 [1] receiving max(amax_out, amax(x))
 *                 by one relaxed atomic per thread block -- pass the history
 *                 slot &hist[i*L + 0].  TENSORWISE: required, receives
 *                 amax(x) (it carries the amax between the reduction and the
 *                 cast).  ROWWISE: optional (NULL or [1]), receives amax(x).
 *   q_row         [rows][cols] u8 (if LAYOUT_ROW); q[r][c] = fp8(x[r][c] *
 *                 s_row(r)).  8-byte aligned.
 *   scale_inv_row [1] (DELAYED, TENSORWISE) or [rows] (ROWWISE): 1 / scale.
 *   q_colT        [cols][ld_colT] u8 (if LAYOUT_COLT); q_colT[c][j] =
 *                 fp8(x[r][c] * s_col(c)) with j = r when ungrouped.  Grouped:
 *                 group e's rows land at columns poff_e .. poff_e + m_e - 1,
 *                 poff_e = sum_{e'<e} roundup(m_e', 32); the padding columns up
 *                 to poff_{e+1} are written as 0.  ld_colT % 16 == 0 and
 *                 ld_colT >= rows (ungrouped) or >= poff_G (grouped).
 *   scale_inv_col [1] (DELAYED, TENSORWISE), [cols] (ROWWISE ungrouped) or
 *                 [num_groups][cols] (ROWWISE grouped).  An empty group, an
 *                 all-zero column or a non-finite amax gives scale 1.
 *   group_offsets NULL, or device int32 [num_groups + 1]: offsets[0] = 0,
 *                 non-decreasing, offsets[num_groups] = rows (the row range
 *                 of each expert group).  Not validated on the device beyond
 *                 bounds: rows outside [0, rows) are skipped.
 *   num_groups    with group_offsets: the number of groups (1 .. 4096).
 *                 Without (NULL): 0 for an ungrouped tensor, or num_groups
 *                 equal groups of rows / num_groups rows each (a stack of
 *                 expert weights), which must be a multiple of 64: the same
 *                 results as passing the offsets e * rows / num_groups (no
 *                 padding columns, since the groups are multiples of 32), on
 *                 the plain tensor's kernels.
 *   Scale arithmetic (fp32, IEEE): s = fp8_max / amax, s *= 2^-margin, an
 *   overflow to Inf becomes FLT_MAX, amax == 0 or non-finite gives s = 1;
 *   scale_inv = 1 / s.  NaN in x propagates into the amax.
 */
FP8GB_API fp8_status_t fp8_quantize(const void *x_bf16, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                          const fp8_recipe_t *recipe, int layouts, const float *scale_in, float *amax_out,
                          uint8_t *q_row, float *scale_inv_row, uint8_t *q_colT, int64_t ld_colT,
                          float *scale_inv_col, const int32_t *group_offsets, int num_groups, void *stream);

/*
 * fp8_quantize_rowwise_resident -- the ROWWISE recipe of fp8_quantize for a
 * plain (ungrouped) tensor in one cooperative launch, for callers that
 * cannot allocate device memory when they call.  The pages have no
 * counterpart to this entry point: it is an interface choice of this
 * library.
 *
 * Results: those of fp8_quantize with recipe kind FP8_RECIPE_ROWWISE, margin
 * `margin` and no groups, byte for byte -- q_row, q_colT, scale_inv_row
 * [rows], scale_inv_col [cols] and the optional amax_out [1] have the
 * meanings, layouts and alignment rules given there.  An empty tensor (rows
 * == 0) writes scale_inv_col = 1 and amax_out = 0, as fp8_quantize does.
 *
 * Why it exists.  One launch clears the amax accumulators, runs the row /
 * column amax pass, the cast pass and the scale_inv conversion, with
 * grid-wide barriers in between; for a tensor that fits in L2 (on GB300, up
 * to about 96 MB of bf16) the cast pass reads x back from L2.  The barriers
 * need a counter in global memory beyond the inputs and outputs.  A library
 * would normally take that from a workspace the caller allocates or allocate
 * it itself; this entry point does neither, because some callers cannot call
 * cudaMalloc: a framework whose caching allocator owns all device memory
 * (a cudaMalloc behind its back fragments its pool and can fail once the
 * pool has taken the free memory), an engine that reserves a fixed memory
 * budget up front, or a training step that must not stall, since cudaMalloc
 * and cudaFree can synchronise the device.  It calls no cudaMalloc, cudaFree
 * or allocating library routine.
 *
 * Scratch.  The counters live in a file-scope device array of the library:
 * 64 counters of 128 bytes (8 KB), present on every device that loads the
 * library until the process exits.  A call uses one counter whatever the
 * tensor size, so no tensor is refused for want of scratch; the size limits
 * are those of fp8_quantize (rows <= 2^40, cols <= 2^31, else
 * FP8_ERR_INVALID_ARG).  The first call on a device, made with that device
 * current, looks up the array's device address (cudaGetSymbolAddress) and
 * keeps it; make that first call before any stream capture on the device.
 * Every call shares the array, which keeps what the last call left: each
 * call takes the next counter in turn and clears it on `stream` before its
 * launch.  Calls that overlap on the GPU (on different streams) use
 * different counters while fewer than 64 are in flight at once; beyond
 * that, two overlapping calls share a counter and race.  Calls of every
 * other entry point are unaffected.
 *
 * Errors: FP8_ERR_INVALID_ARG / FP8_ERR_ALIGNMENT before any launch;
 * FP8_ERR_CUDA if the address lookup or the cooperative launch fails; a
 * barrier wait that gives up (about 2 s) is reported as FP8_ERR_TIMEOUT by
 * fp8_sync_status().
 */
FP8GB_API fp8_status_t fp8_quantize_rowwise_resident(const void *x_bf16, int64_t rows, int64_t cols, int64_t ld_x,
                                                     int fmt, int margin, int layouts, float *amax_out,
                                                     uint8_t *q_row, float *scale_inv_row, uint8_t *q_colT,
                                                     int64_t ld_colT, float *scale_inv_col, void *stream);

/*
 * Fused MoE prologues of the ROWWISE recipe ("FP8 Training on AMD GPUs with
 * TorchTitan and TorchAO", the question on fused Triton kernels: the
 * five-kernel eager chain in front of the MoE grouped GEMMs replaced by one
 * fused kernel; "How PyTorch FP8 Optimizations on AMD GPUs ...", What
 * Happened: rowwise FP8 with the colwise-scales kernel on the MoE path).
 * Each writes exactly what fp8_quantize with recipe kind FP8_RECIPE_ROWWISE,
 * margin `margin` and the given groups would write for the tensor its
 * prologue defines: q_row, scale_inv_row [rows], q_colT in the padded
 * grouped layout, scale_inv_col [num_groups][cols], the optional amax_out
 * [1].  Groups are required (1 <= num_groups <= 4096); the other limits,
 * alignments and errors are fp8_quantize's.
 *
 * They run the grouped rowwise passes of fp8_quantize (amax pass, cast
 * pass) with the prologue applied to what each pass reads, so neither the
 * gathered rows nor h is written to memory (except the optional copy of h).
 *
 * fp8_permute_quantize -- row r of the tensor is row src_rows[r] of x (the
 *   routed token rows in expert order; a token routed to k experts appears
 *   k times).
 *     x_bf16    [x_rows][ld_x] bf16 token rows.
 *     src_rows  device int32 [rows]; an index outside [0, x_rows) is read as
 *               a zero row and reported (fp8_sync_status: FP8_ERR_INVALID_ARG).
 *     rows      routed rows (= group_offsets[num_groups]).
 *
 * fp8_swiglu_quantize -- the tensor is h = bf16_rne(silu(g) * u), g and u
 *   the two halves of each row of gate_up_bf16 [rows][ld] (gate in columns
 *   [0, F), up in [F, 2F); ld >= 2F, ld % 8 == 0, F % 8 == 0), evaluated as
 *   in fp8_mx_swiglu_quantize (each h within one bf16 ulp of the exact
 *   value).  h_bf16: optional [rows][ld_h] bf16 copy of h (NULL: not
 *   written; ld_h % 8 == 0, 16-byte aligned).
 */
FP8GB_API fp8_status_t fp8_permute_quantize(const void *x_bf16, int64_t x_rows, int64_t cols, int64_t ld_x,
                                            const int32_t *src_rows, int64_t rows, int fmt, int margin, int layouts,
                                            float *amax_out, uint8_t *q_row, float *scale_inv_row, uint8_t *q_colT,
                                            int64_t ld_colT, float *scale_inv_col, const int32_t *group_offsets,
                                            int num_groups, void *stream);

FP8GB_API fp8_status_t fp8_swiglu_quantize(const void *gate_up_bf16, int64_t rows, int64_t F, int64_t ld, int fmt,
                                           int margin, int layouts, void *h_bf16, int64_t ld_h, float *amax_out,
                                           uint8_t *q_row, float *scale_inv_row, uint8_t *q_colT, int64_t ld_colT,
                                           float *scale_inv_col, const int32_t *group_offsets, int num_groups,
                                           void *stream);

/*
 * fp8_update_amax_history -- delayed-scaling update for n tensors in one
 * launch ("FP8 training for Flux models": fp8_amax_history_len,
 * fp8_amax_compute_algo, fp8_margin; its verification list names a "fused
 * delayed-scale update").
 *
 *   hist            fp32 [n][L] in place; hist[i][0] is the current step's
 *                   amax (filled by fp8_quantize with DELAYED).
 *   scale, scale_inv fp32 [n] in place.
 *   fmt             u8 [n] (fp8_format_t of each tensor; decides fp8_max).
 *   algo            most_recent: a = hist[i][0]; max: a = max_j hist[i][j]
 *                   (NaN anywhere in the window gives NaN).
 *   margin          0..64.
 *   nonfinite_count int32 [n] or NULL; incremented when a is not finite.
 *   Per tensor: if a is finite and > 0, scale = fp8_max / a * 2^-margin (Inf
 *   -> FLT_MAX) and scale_inv = 1 / scale; otherwise both are kept.  Then the
 *   row is shifted one slot towards the end (hist[j] = hist[j-1], the oldest
 *   value dropped) and hist[i][0] = 0.
 *   Limits: n >= 1, 1 <= L <= 32768.
 */
FP8GB_API fp8_status_t fp8_update_amax_history(float *hist, float *scale, float *scale_inv, const uint8_t *fmt, int n,
                                     int L, int algo, int margin, int32_t *nonfinite_count, void *stream);

/*
 * fp8_scaled_gemm -- C[m][n] = bf16( sum_k A[m][k] * B[n][k] * sa(m) * sb(n) )
 * with fp32 accumulation on the tcgen05 tensor cores ("TN": both operands
 * K-contiguous).
 *
 *   A  u8 [M][lda], format fa;  B  u8 [N][ldb], format fb  (E4M3FN or E5M2).
 *   M, N >= 1; K >= 16, K % 16 == 0; lda, ldb >= K, % 16 == 0; A, B 16-byte
 *   aligned.
 *   sa, sa_mode   FP8_SCALE_TENSOR: sa[0]; FP8_SCALE_PER_ROW: sa[m], [M].
 *   sb, sb_mode   FP8_SCALE_TENSOR: sb[0]; FP8_SCALE_PER_ROW: sb[n], [N].
 *   C_bf16        [M][ldc] bf16, ldc >= N, 2-byte aligned (16-byte vector
 *                 stores are used when C is 16-byte aligned and ldc % 8 == 0).
 *   The scales are the scale_inv outputs of fp8_quantize.  fprop Y = X W^T
 *   takes A = X row layout, B = W row layout; dgrad dX = dY W takes A = dY
 *   row layout, B = W colwise-transposed; wgrad dW = dY^T X takes A = dY
 *   colwise-transposed, B = X colwise-transposed.
 */
FP8GB_API fp8_status_t fp8_scaled_gemm(const uint8_t *A, int fa, int64_t lda, const uint8_t *B, int fb, int64_t ldb,
                             int64_t M, int64_t N, int64_t K, const float *sa, int sa_mode, const float *sb,
                             int sb_mode, void *C_bf16, int64_t ldc, void *stream);

/*
 * fp8_grouped_gemm -- per-expert GEMMs over variable-size row groups in one
 * launch (grouped GEMM for Mixture-of-Experts, "How PyTorch FP8
 * Optimizations on AMD GPUs ..." What Happened).
 *
 * group_offsets: device int32 [G+1] row ranges (offsets[0] = 0,
 * non-decreasing, offsets[G] = M_total).  Empty groups are allowed.
 *
 * FP8_GROUPED_M (fprop, dgrad): A u8 [M_total][K] (group rows stacked), B u8
 *   [G][N][K]; C[m][n] = sum_k A[m][k] B[e][n][k] sa(m) sb(e, n) for m in
 *   group e; C bf16 [M_total][N].  sa: [1] or [M_total]; sb: [1] or [G][N].
 * FP8_GROUPED_M_BT (dgrad with the weights' colwise-transposed layout): as
 *   FP8_GROUPED_M, but B u8 [N][ld_T] is the grouped colwise layout that
 *   fp8_quantize emits for a weight tensor [G*K][N] quantized with G equal
 *   groups of K rows: expert e's [N][K] matrix starts at column e * kpad,
 *   kpad = roundup(K, 32) (its padding columns are zero).  Requires
 *   ld_T >= G * kpad, ld_T % 16 == 0.  sb: [1] or [G][N] (that call's
 *   per-group column scales).
 * FP8_GROUPED_K (wgrad): A u8 [N][ld_T], B u8 [K][ld_T] in the padded
 *   grouped colwise layout of fp8_quantize (ld_T = that call's ld_colT);
 *   C[e][n][k] = sum_{r < m_e} A[n][poff_e + r] B[k][poff_e + r] sa(e, n)
 *   sb(e, k); C bf16 [G][N][K]; an empty group's block is written as 0.
 *   sa: [1] or [G][N]; sb: [1] or [G][K].
 * Limits: K % 16 == 0 (M mode), ld_T % 16 == 0 (K mode), 1 <= G <= 1024;
 * 16-byte aligned A and B; C 2-byte aligned.
 */
FP8GB_API fp8_status_t fp8_grouped_gemm(int mode, const uint8_t *A, int fa, const uint8_t *B, int fb,
                              const int32_t *group_offsets, int G, int64_t M_total, int64_t N, int64_t K,
                              const float *sa, int sa_mode, const float *sb, int sb_mode, void *C_bf16,
                              int64_t ld_T, void *stream);

/*
 * fp8_group_padded_offsets -- host helper for the grouped colwise layout.
 * host_offsets int32 [G+1] -> host_padded_out int64 [G+1] (may be NULL) with
 * poff_e = sum_{e'<e} roundup(m_e', align); returns poff_G (the ld_colT /
 * ld_T to allocate), or -1 for bad arguments (align must be a positive
 * multiple of 16; offsets non-decreasing).
 */
FP8GB_API int64_t fp8_group_padded_offsets(const int32_t *host_offsets, int G, int align, int64_t *host_padded_out);

/* ------------------------------------------------------------------------
 * MXFP8 -- the "mxfp8" recipe ("FP8 training for Flux models", Key FP8
 * Parameters, fp8_recipe) and the MXFP8 grouped GEMM ("FP8 Training on AMD
 * GPUs with TorchTitan and TorchAO", next work).  The pages name it without
 * a definition; this library follows the OCP Microscaling (MX) v1.0
 * specification: blocks of 32 consecutive elements along the contraction
 * dimension share one power-of-two scale X = 2^e stored as an E8M0 byte
 * (code e + 127; 255 = NaN), e = floor(log2(block amax)) - emax_elem
 * (emax_elem = 8 for E4M3, 15 for E5M2) clamped to [-127, 127], and each
 * element is sat_rne_fp8(v / X).  An all-zero block has code 0; a block
 * holding a NaN or Inf has code 255 and NaN elements.
 *
 * MX scale layout.  The E8M0 codes of an operand with R scale rows and KB
 * blocks per row are bytes [ceil(KB / 4)][R128][4] with R128 = roundup(R,
 * 128): a row's four blocks of one 128-element K tile form one 32-bit word,
 * and every 128 rows of a K tile are one 512-byte block in which row
 * 128 i + 32 j + L has word 4 L + j -- the order in which the tensor cores'
 * shared-to-tensor-memory copy (tcgen05.cp 32x128b) reads a 128-row block.
 * The scale of block b of row r is at byte 4 * ((b / 4) * R128 + 128 (r /
 * 128) + 4 (r % 32) + (r / 32) % 4) + b % 4, so the scales of a GEMM tile
 * are one contiguous copy that the GEMM uses as it lands.  Bytes of blocks
 * past KB and of rows past R are written as 0.  Grouped MX layouts pad every
 * group to FP8_MX_GROUP_ALIGN rows (fp8_group_padded_offsets with that align
 * gives the padded offsets and the total P).
 * ------------------------------------------------------------------------ */
#define FP8_MX_BLOCK 32
#define FP8_MX_GROUP_ALIGN 128

/* Bytes of an MX scale buffer for R scale rows and KB blocks per row. */
FP8GB_API int64_t fp8_mx_scale_bytes(int64_t scale_rows, int64_t blocks);

/*
 * fp8_mx_quantize -- MX quantize of a bf16 matrix, emitting the row layout
 * (blocks along each row), the transposed layout (blocks along each column,
 * stored column-major), or both, from one read of x.  The two layouts have
 * their own blocks, so q_colT is not the transpose of q_row.
 *
 *   x_bf16     [rows][ld_x] bf16; 16-byte aligned, ld_x % 8 == 0, ld_x >= cols.
 *              rows == 0 returns FP8_OK without touching any buffer.
 *   rows >= 0; cols >= 32, cols % 32 == 0.
 *   fmt        FP8_E4M3FN or FP8_E5M2 (FP8_ERR_UNSUPPORTED for the fnuz
 *              formats, which MX does not define).
 *   layouts    FP8_LAYOUT_ROW | FP8_LAYOUT_COLT (at least one).
 *   q_row      [rows][cols] u8, 16-byte aligned  (FP8_LAYOUT_ROW).
 *   s_row      MX scale layout, R = rows (grouped: the padded total P),
 *              KB = cols / 32; 4-byte aligned.  Grouped: row r of group e
 *              has scale row poff_e + (r - offsets[e]); padding rows are
 *              all-zero blocks (code 0).
 *   q_colT     [cols][ld_colT] u8, 16-byte aligned, ld_colT % 16 == 0
 *              (FP8_LAYOUT_COLT).  Ungrouped: rows % 32 == 0, ld_colT >=
 *              rows, column c holds x[0..rows)[c]; bytes past rows are left
 *              untouched.  Grouped: ld_colT >= P; group e's rows start at
 *              column poff_e and are followed by zero bytes up to poff_(e+1).
 *   s_col      MX scale layout, R = cols, KB = rows / 32 (grouped: P / 32).
 *   group_offsets  NULL, or device int32 [num_groups + 1] row ranges as for
 *              fp8_quantize (1 <= num_groups <= 4096).  Malformed offsets,
 *              or P > ld_colT, set the device error word (fp8_sync_status
 *              reports FP8_ERR_INVALID_ARG) and nothing is written.
 * Ownership: every buffer is caller-owned device memory; nothing is
 * allocated.  Errors: FP8_ERR_INVALID_ARG / FP8_ERR_UNSUPPORTED /
 * FP8_ERR_ALIGNMENT before any launch, FP8_ERR_CUDA on a launch failure.
 */
FP8GB_API fp8_status_t fp8_mx_quantize(const void *x_bf16, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                                       int layouts, uint8_t *q_row, uint8_t *s_row, uint8_t *q_colT,
                                       int64_t ld_colT, uint8_t *s_col, const int32_t *group_offsets,
                                       int num_groups, void *stream);

/*
 * fp8_blockwise_quantize -- the "blockwise" recipe ("FP8 training for Flux
 * models", Key FP8 Parameters; named there without a definition).  Blocks of
 * 128 elements along the contraction: block_rows = 1 gives 1 x 128 blocks
 * (activations, gradients; the transposed layout's blocks are 128 rows of one
 * column), block_rows = 128 gives 128 x 128 blocks (weights; one scale per
 * block serves both layouts).  Each block takes the largest power-of-two
 * scale s with amax * s <= fp8_max (amax 0 or non-finite: s = 1), q =
 * sat_rne(v * s) -- no finite element saturates -- and 1/s is stored as its
 * E8M0 code in the MX scale layout (the code in all four 32-element slots of
 * the block), so fp8_mx_gemm multiplies blockwise operands directly.
 *
 *   x_bf16   [rows][ld_x] bf16, 16-byte aligned, ld_x % 8 == 0; cols % 128 == 0;
 *            rows % 128 == 0 for the transposed layout or 128 x 128 blocks.
 *   fmt      FP8_E4M3FN or FP8_E5M2.
 *   q_row, s_row    [rows][cols] u8 and its scales (R = rows, KB = cols / 32).
 *   q_colT, s_col   [cols][ld_colT] u8 (ld_colT >= rows, % 16 == 0) and its
 *                   scales (R = cols, KB = rows / 32); s_col 8-byte aligned.
 * Errors as fp8_mx_quantize; nothing is allocated.
 */
FP8GB_API fp8_status_t fp8_blockwise_quantize(const void *x_bf16, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                                              int block_rows, int layouts, uint8_t *q_row, uint8_t *s_row,
                                              uint8_t *q_colT, int64_t ld_colT, uint8_t *s_col, void *stream);

/*
 * Fused MoE prologues ("FP8 Training on AMD GPUs with TorchTitan and TorchAO":
 * a five-kernel eager chain in front of the MoE grouped GEMMs replaced by one
 * fused kernel).  Each reads its bf16 input once and writes exactly what
 * fp8_mx_quantize would write for the tensor the prologue defines; same
 * layouts, grouping, limits and errors as fp8_mx_quantize.
 *
 * fp8_mx_permute_quantize -- gather, then MX quantize: output row r is input
 *   row src_rows[r] (the permutation of routed token rows into expert order;
 *   a token routed to k experts appears k times).
 *     x_bf16    [x_rows][ld_x] bf16 token rows; cols % 32 == 0.
 *     src_rows  device int32 [rows]; an index outside [0, x_rows) is read as a
 *               zero row and reported (fp8_sync_status: FP8_ERR_INVALID_ARG).
 *     rows      output rows (the routed rows, grouped by expert when
 *               group_offsets is given).
 *
 * fp8_mx_swiglu_quantize -- h = bf16(silu(g) * u), then MX quantize of h.
 *     gate_up_bf16  [rows][ld] bf16: gate in columns [0, F), up in [F, 2F);
 *                   ld >= 2F, ld % 8 == 0; F % 32 == 0.
 *     h_bf16        optional [rows][ld_h] bf16 copy of h (NULL: not written).
 *   h is bf16_rne(silu(g) * u), silu(g) = g / (1 + e^-g), evaluated in fp32
 *   with the fast exponential and divide; each element of h is within one
 *   bf16 ulp of the exact value rounded to bf16 (for |u| <= 2^110; NaN and
 *   +-Inf follow IEEE arithmetic, silu(-Inf) = -0).  The quantized bytes and
 *   scales are exactly fp8_mx_quantize's of that h.
 */
FP8GB_API fp8_status_t fp8_mx_permute_quantize(const void *x_bf16, int64_t x_rows, int64_t cols, int64_t ld_x,
                                               const int32_t *src_rows, int64_t rows, int fmt, int layouts,
                                               uint8_t *q_row, uint8_t *s_row, uint8_t *q_colT, int64_t ld_colT,
                                               uint8_t *s_col, const int32_t *group_offsets, int num_groups,
                                               void *stream);

FP8GB_API fp8_status_t fp8_mx_swiglu_quantize(const void *gate_up_bf16, int64_t rows, int64_t F, int64_t ld,
                                              int fmt, int layouts, void *h_bf16, int64_t ld_h, uint8_t *q_row,
                                              uint8_t *s_row, uint8_t *q_colT, int64_t ld_colT, uint8_t *s_col,
                                              const int32_t *group_offsets, int num_groups, void *stream);

/*
 * fp8_mx_gemm -- C[m][n] = bf16( sum_k A[m][k] X_A(m, k/32) B[n][k] X_B(n, k/32) )
 * on the tcgen05 block-scaled tensor cores (kind::mxf8f6f4, scales read by
 * the MMA from tensor memory), fp32 accumulation, "TN" operands.
 *
 *   A  u8 [M][lda] format fa, sA its MX scales (R = M, KB = K / 32);
 *   B  u8 [N][ldb] format fb, sB its MX scales (R = N, KB = K / 32);
 *   fa, fb: FP8_E4M3FN or FP8_E5M2.  M, N >= 1; K >= 32, K % 32 == 0;
 *   lda, ldb >= K, % 16 == 0; A, B 16-byte aligned; sA, sB 16-byte aligned.
 *   C_bf16 [M][ldc], ldc >= N, 2-byte aligned.
 * fprop takes A = X row layout, B = W row layout; dgrad A = dY row layout,
 * B = W transposed layout; wgrad A = dY transposed, B = X transposed, each
 * with the scales fp8_mx_quantize wrote beside it.
 */
FP8GB_API fp8_status_t fp8_mx_gemm(const uint8_t *A, int fa, int64_t lda, const uint8_t *sA, const uint8_t *B,
                                   int fb, int64_t ldb, const uint8_t *sB, int64_t M, int64_t N, int64_t K,
                                   void *C_bf16, int64_t ldc, void *stream);

/*
 * fp8_mx_grouped_gemm -- the MX counterpart of fp8_grouped_gemm (groups
 * padded to FP8_MX_GROUP_ALIGN in every padded layout).
 *
 * FP8_GROUPED_M: A u8 [M_total][K] (group rows stacked), sA the row-layout
 *   scales of a grouped fp8_mx_quantize (R = P, KB = K / 32); B u8 [G][N][K],
 *   sB its scales as one [G*N][K] operand (R = G * N); C bf16 [M_total][N].
 *   N % 128 == 0 (expert e's scale rows start at row e * N, which must begin
 *   a 128-row block of the MX scale layout), else FP8_ERR_ALIGNMENT.
 * FP8_GROUPED_K: A u8 [N][ld_T], B u8 [K][ld_T] the transposed layouts of
 *   grouped fp8_mx_quantize calls (ld_T their ld_colT), sA / sB their scales
 *   (R = N / K, KB = P / 32 with P the padded total); C[e] = A_e . B_e^T
 *   over group e's padded columns, C bf16 [G][N][K]; an empty group's block
 *   is 0.
 * FP8_GROUPED_M_BT (dgrad with the weights' transposed layout): as
 *   FP8_GROUPED_M, but B u8 [N][ld_T] is the transposed layout of a grouped
 *   fp8_mx_quantize of the weight stack [G*K][N] in G equal groups of K rows:
 *   expert e's [N][K] block starts at column e * kpad, kpad = roundup(K, 128)
 *   (ld_T >= G * kpad, ld_T % 16 == 0); sB its scales (R = N).
 * Limits: K % 32 == 0 (M modes); N % 4 == 0 (M modes); ld_T % 128 == 0
 * (K mode); 1 <= G <= 1024; A, B, sA, sB 16-byte aligned.
 */
FP8GB_API fp8_status_t fp8_mx_grouped_gemm(int mode, const uint8_t *A, int fa, const uint8_t *sA,
                                           const uint8_t *B, int fb, const uint8_t *sB,
                                           const int32_t *group_offsets, int G, int64_t M_total, int64_t N,
                                           int64_t K, void *C_bf16, int64_t ld_T, void *stream);

/* Synchronise `stream`, then report and clear a device-side timeout word:
 * FP8_OK, FP8_ERR_TIMEOUT, or FP8_ERR_CUDA. */
FP8GB_API fp8_status_t fp8_sync_status(void *stream);

/* Test support for the bounded-wait machinery: launches one thread block
 * that waits on a shared-memory barrier nothing will complete, giving up
 * after about `wait_ns` nanoseconds (1e3 .. 1e10).  The wait gives up,
 * records the device error word and the kernel returns; fp8_sync_status()
 * then reports FP8_ERR_TIMEOUT. */
FP8GB_API fp8_status_t fp8_selftest_bounded_wait(int64_t wait_ns, void *stream);

/* Human-readable name of a status; never NULL. */
FP8GB_API const char *fp8_status_string(fp8_status_t s);

/* Message of the last CUDA error seen by this library in this thread. */
FP8GB_API const char *fp8_last_cuda_error(void);

/* Library version, e.g. "fp8gb 0.1 sm_103a". */
FP8GB_API const char *fp8_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8GB_H */
