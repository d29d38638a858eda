// mxquant.cu -- MXFP8 quantize: blocks of 32 elements that share one E8M0
// (power-of-two) scale, emitting the row layout (blocks along rows) and the
// transposed layout (blocks along columns) from one read of the bf16 input.
//
// Method: the "mxfp8" recipe of "FP8 training for Flux models" (Configuration
// > Key FP8 Parameters) and the MXFP8 grouped GEMM of "FP8 Training on AMD
// GPUs with TorchTitan and TorchAO"; the block rule is the OCP Microscaling
// v1.0 one: X = 2^(floor(log2 amax) - emax_elem), element = sat_rne(v / X).
//
// Design (GB300): persistent 256-thread blocks looping over tiles of 64 rows
// x 128 columns (row-major; tall tensors in bands of eight column tiles);
// each block issues the next tile's loads before working on the current one.
//   Row layout: thread (row, block) loads its 32 bf16 (two 32-byte loads,
//     whole sectors, when the row blocks are 32-byte aligned; else four
//     16-byte loads),
//     takes the packed |bf16| maximum, derives the E8M0 code from the fp32
//     exponent bits, multiplies by 2^(127 - code) (exact) and converts with
//     cvt.rn.satfinite, writing its 32 codes with one 32-byte store (q_row
//     32-byte aligned); the four blocks of a row combine their codes into one
//     32-bit word of the scale layout by two shuffles.
//   Transposed layout: the tile is staged in shared memory (column pairs as
//     32-bit words, swizzled); a thread reads two columns x 16 rows, takes
//     the block maximum with its partner thread (the other 16 rows) and
//     writes 16 contiguous bytes per column of q_colT.
// One launch, no atomics, no scratch memory: every block's scale depends
// only on its own 32 elements.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8gb.h"
#include "fp8gb_device.cuh"
#include "fp8gb_host.h"

namespace fp8gb {

constexpr int MX_THREADS = 256;
constexpr int MX_ROWS = 64;             // rows per tile
constexpr int MX_COLS = 128;            // columns per tile: four blocks of a row
constexpr int MX_PITCH_W = 72;          // 32-bit words per shared-memory row (64 + two 4-word pads)
constexpr int MX_MAX_GROUPS = 4096;
constexpr int MX_BAND_TILES = 8;           // column tiles per band of the ungrouped tile walk
constexpr int64_t MX_BAND_MIN_ROWS = 65536;  // ... used from this many rows on

struct MxArgs {
    const uint16_t *x;
    int64_t rows, cols, ld_x;
    uint8_t *q_row, *s_row, *q_colT, *s_col;
    int64_t ld_colT;
    int64_t rs_row;       // scale rows of s_row, rows rounded up to 128 (ungrouped)
    int64_t cols128;      // scale rows of s_col, cols rounded up to 128
    int64_t n_row_tiles;  // grouped: an upper bound (tiles past the padded total exit)
    int64_t n_col_tiles;
    int band;  // ungrouped: tiles walked in bands of `band` column tiles (0: row-major)
    const int32_t *offsets;
    int G;
    int do_row, do_col;
    int ld32;  // every row block of the input starts on a 32-byte boundary: 32-byte loads
    int st32;  // q_row is 32-byte aligned: each row block's 32 codes in one 32-byte store
    unsigned int *err;
    // prologues (template parameter PRO of the kernel)
    const int32_t *src_rows;  // PRO_GATHER: output row r reads input row src_rows[r]
    int64_t x_rows;           // PRO_GATHER: rows of the input
    int64_t up_off;           // PRO_SWIGLU: column offset of `up` in each input row (= cols)
    uint16_t *h_out;          // PRO_SWIGLU: optional bf16 [rows][ld_h] copy of h
    int64_t ld_h;
};

enum { PRO_NONE = 0, PRO_GATHER = 1, PRO_SWIGLU = 2 };

// E8M0 code of a block from the fp32 bit pattern of its largest magnitude:
// floor(log2 amax) is the exponent field (normal) or the position of the top
// mantissa bit (subnormal), minus emax_elem, clamped to [-127, 127].
template <int FMT>
__device__ __forceinline__ uint32_t mx_code(uint32_t amax_bits)
{
    constexpr int emax = FMT == FP8_E5M2 ? 15 : 8;
    if (amax_bits >= 0x7F800000u) return 255u;  // Inf or NaN in the block
    if (amax_bits == 0u) return 0u;
    const int ex = (int)(amax_bits >> 23);
    const int fl = ex > 0 ? ex - 127 : (31 - __clz((int)amax_bits)) - 149;
    int e = fl - emax;
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
    return (uint32_t)(e + 127);
}

// 1 / X = 2^(127 - code) as an fp32 (a normal number for every code a bf16
// block can produce); NaN for the NaN scale, so the block's elements are NaN.
__device__ __forceinline__ float mx_inv_scale(uint32_t code)
{
    if (code == 255u) return __uint_as_float(0x7FC00000u);
    return code <= 253u ? __uint_as_float((254u - code) << 23) : __uint_as_float(0x00400000u);
}

// Exclusive prefix of roundup(m_e, FP8_MX_GROUP_ALIGN) over the groups, by
// warp 0 into shared memory poff[0 .. G], followed by a copy of the offsets
// (poff[G + 1 .. 2G + 1]) so tile lookups never wait on global memory; flags
// malformed offsets and a padded total that does not fit ld_colT.
__device__ void mx_padded_offsets(const MxArgs &a, int32_t *poff, int *bad)
{
    if (threadIdx.x >= 32) return;
    constexpr int AL = FP8_MX_GROUP_ALIGN;
    const int lane = threadIdx.x;
    const int G = a.G;
    const int per = (G + 31) / 32;
    const int g0 = min(G, lane * per), g1 = min(G, g0 + per);
    int64_t local = 0;
    int badl = 0;
    for (int e = g0; e < g1; e++) {
        const int m = a.offsets[e + 1] - a.offsets[e];
        if (m < 0) badl = 1;
        local += (int64_t)((max(m, 0) + AL - 1) / AL) * AL;
    }
    int64_t incl = local;
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    int64_t run = incl - local;
    int32_t *soff = poff + G + 1;
    for (int e = g0; e < g1; e++) {
        poff[e] = (int32_t)run;
        soff[e] = a.offsets[e];
        run += (int64_t)((max(a.offsets[e + 1] - a.offsets[e], 0) + AL - 1) / AL) * AL;
    }
    const int64_t total = __shfl_sync(0xffffffffu, incl, 31);
    badl = __any_sync(0xffffffffu, badl);
    if (lane == 0) {
        poff[G] = (int32_t)total;
        soff[G] = a.offsets[G];
        const int b = badl || a.offsets[0] != 0 || (int64_t)a.offsets[G] != a.rows ||
                      (a.do_col && total > a.ld_colT) || total > INT32_MAX;
        *bad = b;
        if (b) record_error(a.err, ERR_BAD_OFFSETS);
    }
}

// Geometry of tile t: its first row in the (padded) row space, first column,
// first input row and number of real rows.
struct MxTile {
    bool live;  // inside the (padded) row space
    int64_t rt, ct, pr0, c0, src0, nreal;
};

// `hint`: the group of the thread's previous tile.  A block's tiles advance
// through the row space, so the search steps forward from there (a few
// groups at most) before falling back to bisection.
__device__ __forceinline__ MxTile mx_tile(const MxArgs &a, int64_t t, int64_t prows, const int32_t *poff, int &hint)
{
    MxTile g;
    // tile counts stay far below 2^32 (rows and columns are at most 2^31):
    // a 32-bit division instead of a 64-bit one in every thread
    const uint32_t tt = (uint32_t)t, nct = (uint32_t)a.n_col_tiles;
    if (a.band) {
        // row-major inside bands of `band` column tiles (the last band narrower)
        const uint32_t per = (uint32_t)a.band * (uint32_t)a.n_row_tiles;
        const uint32_t bnd = tt / per, r = tt - bnd * per, c_lo = bnd * (uint32_t)a.band;
        const uint32_t w = nct - c_lo < (uint32_t)a.band ? nct - c_lo : (uint32_t)a.band;
        const uint32_t rt = r / w;
        g.rt = rt;
        g.ct = c_lo + (r - rt * w);
    } else {
        g.rt = tt / nct;
        g.ct = tt - (uint32_t)g.rt * nct;
    }
    g.pr0 = g.rt * MX_ROWS;
    g.c0 = g.ct * MX_COLS;
    // ungrouped: the row tiles run to the scale rows (rows rounded up to 128),
    // so the padding rows' scale words are written too (as 0)
    g.live = g.pr0 < (a.offsets ? prows : a.rs_row);
    g.src0 = g.pr0;
    g.nreal = a.rows - g.pr0 < MX_ROWS ? a.rows - g.pr0 : MX_ROWS;
    if (a.offsets && g.live) {
        // the tile lies inside one group (groups are padded to 128 rows)
        int lo = poff[hint] <= g.pr0 ? hint : 0;  // poff[lo] <= pr0
        int step = 0;
        while (step < 4 && lo + 1 < a.G && poff[lo + 1] <= g.pr0) {
            ++lo;
            ++step;
        }
        if (lo + 1 < a.G && poff[lo + 1] <= g.pr0) {
            int hi = a.G;  // poff[lo] <= pr0 < poff[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (poff[mid] <= g.pr0)
                    lo = mid;
                else
                    hi = mid;
            }
        }
        hint = lo;
        const int32_t *soff = poff + a.G + 1;  // the offsets, staged next to poff
        const int64_t local0 = g.pr0 - poff[lo];
        const int64_t m_e = (int64_t)soff[lo + 1] - soff[lo];
        g.src0 = soff[lo] + local0;
        g.nreal = m_e - local0 < MX_ROWS ? m_e - local0 : MX_ROWS;
    }
    if (g.nreal < 0) g.nreal = 0;
    return g;
}

// Raw input registers of one thread for one tile: the 32 bf16 of its row
// block, and for SwiGLU the 32 gate and 32 up values.
// 32 bytes (16 bf16) from a 32-byte-aligned address through the read-only
// path, as two 16-byte halves.
__device__ __forceinline__ void ld_nc_32b(const uint16_t *p, uint4 &lo, uint4 &hi)
{
    asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
                 : "l"(p));
}

// 32 bytes to a 32-byte-aligned address
__device__ __forceinline__ void st_32b(void *p, const uint32_t (&o)[8])
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(o[0]), "r"(o[1]),
                 "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                 : "memory");
}

template <int PRO>
struct MxRaw {
    uint4 v[PRO == PRO_SWIGLU ? 8 : 4];
};

// Thread (lr, blk) = (tid / 4, tid % 4) loads row lr, block blk of the tile
// (zeros outside the data).  Gather reads input row src_rows[r] for output
// row r (an index outside the input is reported and read as zeros); SwiGLU
// reads the gate block and the up block `up_off` columns further.
template <int PRO>
__device__ __forceinline__ void mx_load(const MxArgs &a, const MxTile &g, int tid, MxRaw<PRO> &raw)
{
    constexpr int NV = PRO == PRO_SWIGLU ? 8 : 4;
    const int lr = tid >> 2, blk = tid & 3;
    const uint16_t *row = nullptr;
    if (g.live && lr < g.nreal && g.c0 + 32 * blk < a.cols) {
        int64_t r = g.src0 + lr;
        if constexpr (PRO == PRO_GATHER) {
            r = __ldg(a.src_rows + r);
            if (r < 0 || r >= a.x_rows) {
                record_error(a.err, ERR_BAD_INDEX);
                r = -1;
            }
        }
        if (r >= 0) row = a.x + r * a.ld_x + g.c0 + 32 * blk;
    }
    if (row) {
        if (a.ld32) {
            // whole 32-byte sectors per load
            ld_nc_32b(row, raw.v[0], raw.v[1]);
            ld_nc_32b(row + 16, raw.v[2], raw.v[3]);
            if constexpr (PRO == PRO_SWIGLU) {
                ld_nc_32b(row + a.up_off, raw.v[4], raw.v[5]);
                ld_nc_32b(row + a.up_off + 16, raw.v[6], raw.v[7]);
            }
        } else {
            const uint4 *src = reinterpret_cast<const uint4 *>(row);
#pragma unroll
            for (int j = 0; j < 4; j++) raw.v[j] = __ldg(src + j);
            if constexpr (PRO == PRO_SWIGLU) {
                const uint4 *up = reinterpret_cast<const uint4 *>(row + a.up_off);
#pragma unroll
                for (int j = 0; j < 4; j++) raw.v[4 + j] = __ldg(up + j);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < NV; j++) raw.v[j] = make_uint4(0, 0, 0, 0);
    }
}

// The 32 bf16 the quantize sees: the raw values, or SwiGLU of gate and up
// (then also stored to h_out when requested).
template <int PRO>
__device__ __forceinline__ void mx_prologue(const MxArgs &a, const MxTile &g, int tid, const MxRaw<PRO> &raw,
                                            uint4 (&v)[4])
{
    if constexpr (PRO == PRO_SWIGLU) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const uint4 gg = raw.v[j], uu = raw.v[4 + j];
            v[j] = make_uint4(swiglu2(gg.x, uu.x), swiglu2(gg.y, uu.y), swiglu2(gg.z, uu.z), swiglu2(gg.w, uu.w));
        }
        const int lr = tid >> 2, blk = tid & 3;
        if (a.h_out && g.live && lr < g.nreal && g.c0 + 32 * blk < a.cols) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.h_out + (g.src0 + lr) * a.ld_h + g.c0 + 32 * blk);
#pragma unroll
            for (int j = 0; j < 4; j++) dst[j] = v[j];
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; j++) v[j] = raw.v[j];
    }
}

// Shared tile: 64 rows of MX_PITCH_W words.  The 32-bit word (column pair)
// index is XOR-swizzled by 16 in rows 16-31 of every 32, so the transposed
// phase's column-pair reads (rows r and r + 16 in one warp) hit all 32 banks;
// a 4-word gap after the first 32 words of a row and the row pitch of 72
// words (8 banks mod 32) make the row phase's 16-byte stores (two rows x four
// 32-column blocks per quarter warp) hit 32 distinct banks too.
__device__ __forceinline__ int mx_word(int row, int pair)
{
    const int pp = pair ^ (row & 16);
    return row * MX_PITCH_W + pp + 4 * (pp >> 5);
}

template <int FMT, int PRO>
__global__ void __launch_bounds__(MX_THREADS)
    mx_quantize_kernel(MxArgs a)
{
    __shared__ __align__(16) uint32_t tile[MX_ROWS * MX_PITCH_W];
    extern __shared__ int32_t poff[];  // grouped: padded offsets [G + 1], then the offsets [G + 1]
    __shared__ int s_bad;

    const int tid = threadIdx.x;
    int64_t prows = a.rows;  // rows of the (padded) row space
    if (a.offsets) {
        mx_padded_offsets(a, poff, &s_bad);
        __syncthreads();
        if (s_bad) return;
        prows = poff[a.G];
    }
    const int64_t total = a.n_row_tiles * a.n_col_tiles;
    const int64_t last_rt = prows > 0 ? (prows - 1) / MX_ROWS : -1;
    const int lr = tid >> 2, blk = tid & 3;

    // persistent loop; the next tile's loads are issued before this tile's work
    int64_t t = blockIdx.x;
    int hint = 0;
    MxTile g = mx_tile(a, t, prows, poff, hint);
    MxRaw<PRO> nraw;
    mx_load<PRO>(a, g, tid, nraw);
    for (; t < total; t += gridDim.x) {
        const MxTile cur = g;
        const MxRaw<PRO> raw = nraw;
        if (t + gridDim.x < total) {
            g = mx_tile(a, t + gridDim.x, prows, poff, hint);
            mx_load<PRO>(a, g, tid, nraw);
        }
        if (!cur.live) continue;  // grouped: beyond the padded total (block-uniform)
        uint4 v[4];
        mx_prologue<PRO>(a, cur, tid, raw, v);

        // ---- row layout ----
        if (a.do_row) {
            const bool row_real = lr < cur.nreal;
            const bool blk_ok = cur.c0 + 32 * blk < a.cols;
            uint32_t am = 0;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                am = absmax_bf16x2(am, v[j].x);
                am = absmax_bf16x2(am, v[j].y);
                am = absmax_bf16x2(am, v[j].z);
                am = absmax_bf16x2(am, v[j].w);
            }
            const uint32_t code = blk_ok ? mx_code<FMT>(fold_absmax(am)) : 0u;
            if (row_real && blk_ok) {
                const float inv = mx_inv_scale(code);
                uint32_t out[8];
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const uint2 b = cvt8_scaled<FMT>(v[j], inv);
                    out[2 * j] = b.x;
                    out[2 * j + 1] = b.y;
                }
                uint8_t *dst = a.q_row + (cur.src0 + lr) * a.cols + cur.c0 + 32 * blk;
                if (a.st32) {
                    st_32b(dst, out);
                } else {
                    reinterpret_cast<uint4 *>(dst)[0] = make_uint4(out[0], out[1], out[2], out[3]);
                    reinterpret_cast<uint4 *>(dst)[1] = make_uint4(out[4], out[5], out[6], out[7]);
                }
            }
            // the four blocks of the row (lanes 4i .. 4i+3) form one scale word
            uint32_t word = code << (8 * blk);
            word |= __shfl_xor_sync(0xffffffffu, word, 1);
            word |= __shfl_xor_sync(0xffffffffu, word, 2);
            const int64_t srow = cur.pr0 + lr;  // scale row (padded row space)
            const int64_t srows = a.offsets ? prows : a.rs_row;  // a multiple of 128 either way
            if (blk == 0 && srow < srows)
                *reinterpret_cast<uint32_t *>(a.s_row + mx_scale_word(cur.ct, srow, srows) * 4) = word;
        }

        // ---- transposed layout ----
        if (a.do_col) {
#pragma unroll
            for (int j = 0; j < 4; j++)
                *reinterpret_cast<uint4 *>(&tile[mx_word(lr, 16 * blk + 4 * j)]) = v[j];
            __syncthreads();
            // thread: column pair `pair`, 32-row block h, rows 16 s .. 16 s + 15
            // of it; the partner holding the other 16 rows is lane ^ 1
            const int s = tid & 1, pair = (tid >> 1) & 63, h = tid >> 7;
            const int64_t c = cur.c0 + 2 * pair;
            const int64_t kb = (cur.pr0 >> 5) + h;  // block index along the rows
            const bool blk_valid = cur.pr0 + 32 * h < prows;
            uint32_t w[16];
            uint32_t am = 0;
#pragma unroll
            for (int i = 0; i < 16; i++) {
                w[i] = tile[mx_word(32 * h + 16 * s + i, pair)];
                am = absmax_bf16x2(am, w[i]);
            }
            am = __vmaxu2(am, __shfl_xor_sync(0xffffffffu, am, 1));
            const bool real = c < a.cols && blk_valid;  // columns past cols: padding scale rows
            const uint32_t code0 = real ? mx_code<FMT>(am << 16) : 0u;
            const uint32_t code1 = real ? mx_code<FMT>(am & 0xFFFF0000u) : 0u;
            if (real) {
                const float inv0 = mx_inv_scale(code0), inv1 = mx_inv_scale(code1);
                uint32_t o0[4], o1[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const uint32_t x0 = w[4 * i], x1 = w[4 * i + 1], x2 = w[4 * i + 2], x3 = w[4 * i + 3];
                    float a0 = bf16lo(x0), a1 = bf16lo(x1), a2 = bf16lo(x2), a3 = bf16lo(x3);
                    float c0 = bf16hi(x0), c1 = bf16hi(x1), c2 = bf16hi(x2), c3 = bf16hi(x3);
                    mul2_rn(a0, a1, inv0, inv0);
                    mul2_rn(a2, a3, inv0, inv0);
                    mul2_rn(c0, c1, inv1, inv1);
                    mul2_rn(c2, c3, inv1, inv1);
                    o0[i] = cvt4<FMT>(a0, a1, a2, a3);
                    o1[i] = cvt4<FMT>(c0, c1, c2, c3);
                }
                const int64_t r0 = cur.pr0 + 32 * h + 16 * s;
                *reinterpret_cast<uint4 *>(a.q_colT + c * a.ld_colT + r0) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
                *reinterpret_cast<uint4 *>(a.q_colT + (c + 1) * a.ld_colT + r0) =
                    make_uint4(o1[0], o1[1], o1[2], o1[3]);
            }
            if (s == 0 && c < a.cols128) {
                // columns c and c + 1 are scale rows c and c + 1 of s_col
                uint8_t *sc0 = a.s_col + mx_scale_word(kb >> 2, c, a.cols128) * 4 + (kb & 3);
                uint8_t *sc1 = a.s_col + mx_scale_word(kb >> 2, c + 1, a.cols128) * 4 + (kb & 3);
                sc0[0] = (uint8_t)code0;
                sc1[0] = (uint8_t)code1;
                // the last word's blocks past the data are written as 0
                if (cur.rt == last_rt && (kb & 3) < 2) {
                    sc0[2] = 0;
                    sc1[2] = 0;
                }
            }
            __syncthreads();  // the tile is rewritten by the next iteration
        }
    }
}

template <int FMT, int PRO>
static fp8_status_t launch_mx(const MxArgs &a, cudaStream_t st)
{
    const size_t dyn = a.offsets ? 2 * (size_t)(a.G + 1) * sizeof(int32_t) : 0;  // poff + offsets
    if (dyn > 0 && cudaFuncSetAttribute(mx_quantize_kernel<FMT, PRO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)dyn) != cudaSuccess)
        return cuda_fail();
    const int64_t total = a.n_row_tiles * a.n_col_tiles;
    // persistent: as many blocks as fit at once, each looping over tiles
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mx_quantize_kernel<FMT, PRO>, MX_THREADS, dyn) !=
        cudaSuccess)
        return cuda_fail();
    const int64_t cap = (int64_t)num_sms() * (per_sm > 0 ? per_sm : 1);
    int64_t grid = total < cap ? total : cap;
    if (grid > INT32_MAX) grid = INT32_MAX;
    if (grid < 1) return FP8_OK;
    mx_quantize_kernel<FMT, PRO><<<(unsigned)grid, MX_THREADS, dyn, st>>>(a);
    return check_launch();
}

// Validation and launch shared by the three entry points: `rows` output rows
// of `cols` columns read from `x` (row stride ld_x) through the prologue.
static fp8_status_t mx_run(MxArgs a, int fmt, int layouts, int pro, cudaStream_t st)
{
    const int64_t rows = a.rows, cols = a.cols;
    if (rows < 0 || cols < 1 || a.ld_x < 1) return FP8_ERR_INVALID_ARG;
    if (fmt == FP8_E4M3FNUZ || fmt == FP8_E5M2FNUZ) return FP8_ERR_UNSUPPORTED;
    if (fmt != FP8_E4M3FN && fmt != FP8_E5M2) return FP8_ERR_INVALID_ARG;
    if (layouts < 1 || layouts > 3) return FP8_ERR_INVALID_ARG;
    if (rows == 0) return FP8_OK;  // nothing to read or write (an all-empty grouped tensor has P = 0)
    if (!a.x) return FP8_ERR_INVALID_ARG;
    const bool do_row = layouts & FP8_LAYOUT_ROW, do_col = layouts & FP8_LAYOUT_COLT;
    if (do_row && (!a.q_row || !a.s_row)) return FP8_ERR_INVALID_ARG;
    if (do_col && (!a.q_colT || !a.s_col)) return FP8_ERR_INVALID_ARG;
    if (a.offsets && (a.G < 1 || a.G > MX_MAX_GROUPS)) return FP8_ERR_INVALID_ARG;
    if (!a.offsets && a.G != 0) return FP8_ERR_INVALID_ARG;
    if (rows > INT32_MAX || cols > INT32_MAX) return FP8_ERR_INVALID_ARG;
    if (cols % FP8_MX_BLOCK != 0 || a.ld_x % 8 != 0 || !aligned(a.x, 16)) return FP8_ERR_ALIGNMENT;
    if (do_row && (!aligned(a.q_row, 16) || !aligned(a.s_row, 4))) return FP8_ERR_ALIGNMENT;
    if (do_col) {
        if (a.ld_colT < 16 || a.ld_colT % 16 != 0 || !aligned(a.q_colT, 16)) return FP8_ERR_ALIGNMENT;
        if (!a.offsets) {
            if (rows % FP8_MX_BLOCK != 0) return FP8_ERR_ALIGNMENT;
            if (a.ld_colT < rows) return FP8_ERR_INVALID_ARG;
        }
    }
    a.do_row = do_row;
    a.do_col = do_col;
    // row blocks start at x + r * ld_x + 32 k (+ up_off): 32-byte aligned
    // when the base is and the strides are multiples of 16 elements
    a.ld32 = aligned(a.x, 32) && a.ld_x % 16 == 0 && a.up_off % 16 == 0;
    a.st32 = a.q_row && aligned(a.q_row, 32);
    a.rs_row = round_up_128(rows);
    a.cols128 = round_up_128(cols);
    a.n_col_tiles = (cols + MX_COLS - 1) / MX_COLS;
    a.err = device_error_word();
    if (a.offsets) {
        // padded row space: at most 127 padding rows per group, and within ld_colT
        int64_t bound = rows + (int64_t)(FP8_MX_GROUP_ALIGN - 1) * a.G;
        if (do_col && a.ld_colT < bound) bound = a.ld_colT;
        a.n_row_tiles = (bound + MX_ROWS - 1) / MX_ROWS;
    } else {
        a.n_row_tiles = (a.rs_row + MX_ROWS - 1) / MX_ROWS;
    }
    if (a.n_row_tiles * a.n_col_tiles >= (1LL << 32)) return FP8_ERR_INVALID_ARG;  // tile indices are 32-bit
    // Tall tensors (q_colT rows of 64 KB and more) walk their tiles in column
    // bands, so the tiles in flight write runs of a few KB into a few
    // thousand q_colT rows rather than 512-byte pieces into all of them:
    // measured 9 % faster on a [1048576, 7168] expert-weight stack, 2 % slower
    // on [8192, 14336], where row-major order stays.
    a.band = !a.offsets && rows >= MX_BAND_MIN_ROWS && a.n_col_tiles > MX_BAND_TILES ? MX_BAND_TILES : 0;
    if (pro == PRO_GATHER) return fmt == FP8_E5M2 ? launch_mx<FP8_E5M2, PRO_GATHER>(a, st)
                                                  : launch_mx<FP8_E4M3FN, PRO_GATHER>(a, st);
    if (pro == PRO_SWIGLU) return fmt == FP8_E5M2 ? launch_mx<FP8_E5M2, PRO_SWIGLU>(a, st)
                                                  : launch_mx<FP8_E4M3FN, PRO_SWIGLU>(a, st);
    return fmt == FP8_E5M2 ? launch_mx<FP8_E5M2, PRO_NONE>(a, st) : launch_mx<FP8_E4M3FN, PRO_NONE>(a, st);
}

static MxArgs mx_args(const void *x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t *q_row, uint8_t *s_row,
                      uint8_t *q_colT, int64_t ld_colT, uint8_t *s_col, const int32_t *group_offsets, int num_groups)
{
    MxArgs a{};
    a.x = static_cast<const uint16_t *>(x);
    a.rows = rows;
    a.cols = cols;
    a.ld_x = ld_x;
    a.q_row = q_row;
    a.s_row = s_row;
    a.q_colT = q_colT;
    a.ld_colT = ld_colT;
    a.s_col = s_col;
    a.offsets = group_offsets;
    a.G = num_groups;
    return a;
}

}  // namespace fp8gb

using namespace fp8gb;

extern "C" int64_t fp8_mx_scale_bytes(int64_t scale_rows, int64_t blocks)
{
    if (scale_rows < 0 || blocks < 0) return -1;
    return (blocks + 3) / 4 * round_up_128(scale_rows) * 4;
}

extern "C" fp8_status_t fp8_mx_quantize(const void *x_bf16, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                                        int layouts, uint8_t *q_row, uint8_t *s_row, uint8_t *q_colT,
                                        int64_t ld_colT, uint8_t *s_col, const int32_t *group_offsets,
                                        int num_groups, void *stream)
{
    if (ld_x < cols) return FP8_ERR_INVALID_ARG;
    MxArgs a = mx_args(x_bf16, rows, cols, ld_x, q_row, s_row, q_colT, ld_colT, s_col, group_offsets, num_groups);
    return mx_run(a, fmt, layouts, PRO_NONE, static_cast<cudaStream_t>(stream));
}

extern "C" fp8_status_t fp8_mx_permute_quantize(const void *x_bf16, int64_t x_rows, int64_t cols, int64_t ld_x,
                                                const int32_t *src_rows, int64_t rows, int fmt, int layouts,
                                                uint8_t *q_row, uint8_t *s_row, uint8_t *q_colT, int64_t ld_colT,
                                                uint8_t *s_col, const int32_t *group_offsets, int num_groups,
                                                void *stream)
{
    if (x_rows < 0 || ld_x < cols) return FP8_ERR_INVALID_ARG;
    if (rows > 0 && (!src_rows || x_rows < 1)) return FP8_ERR_INVALID_ARG;
    MxArgs a = mx_args(x_bf16, rows, cols, ld_x, q_row, s_row, q_colT, ld_colT, s_col, group_offsets, num_groups);
    a.src_rows = src_rows;
    a.x_rows = x_rows;
    return mx_run(a, fmt, layouts, PRO_GATHER, static_cast<cudaStream_t>(stream));
}

extern "C" fp8_status_t fp8_mx_swiglu_quantize(const void *gate_up_bf16, int64_t rows, int64_t F, int64_t ld,
                                               int fmt, int layouts, void *h_bf16, int64_t ld_h, uint8_t *q_row,
                                               uint8_t *s_row, uint8_t *q_colT, int64_t ld_colT, uint8_t *s_col,
                                               const int32_t *group_offsets, int num_groups, void *stream)
{
    if (F < 1 || ld < 2 * F) return FP8_ERR_INVALID_ARG;
    if (h_bf16 && (ld_h < F)) return FP8_ERR_INVALID_ARG;
    if (h_bf16 && (ld_h % 8 != 0 || !aligned(h_bf16, 16))) return FP8_ERR_ALIGNMENT;
    MxArgs a = mx_args(gate_up_bf16, rows, F, ld, q_row, s_row, q_colT, ld_colT, s_col, group_offsets, num_groups);
    a.up_off = F;
    a.h_out = static_cast<uint16_t *>(h_bf16);
    a.ld_h = ld_h;
    return mx_run(a, fmt, layouts, PRO_SWIGLU, static_cast<cudaStream_t>(stream));
}
