// quantize.cu -- fused amax + scale + saturating cast of bf16 matrices to FP8,
// emitting the row layout and the colwise-transposed layout from one read.
//
// Method: "FP8 training for Flux models" (Configuration > Key FP8 Parameters:
// delayed / tensorwise recipes, fp8_margin); rowwise and colwise scales with
// the transposed layout and fused quantize kernels: "How PyTorch FP8
// Optimizations on AMD GPUs ..." (What Happened) and "FP8 Training on AMD
// GPUs with TorchTitan and TorchAO" (the colwise-scales kernel whose
// non-coalesced writes were the bottleneck; the five-kernel chain fused into
// one; relaxed atomics).
//
// Design (GB300): thread blocks of 256 threads work on tiles of 64 rows x 128
// columns for plain tensors (one tile per block); expert-grouped tensors are
// cast by persistent blocks on tiles of four padded 32-row blocks x 64
// columns (grouped_cast_kernel).  Each thread issues all of its 16-byte loads for a
// tile before touching the data, converts 8 elements at a time with
// cvt.rn.satfinite.{e4m3,e5m2}x2, stores the row layout directly (8-byte
// coalesced stores) and stages the bytes in shared memory; the transposed
// layout is then read back as 8x4 byte blocks, transposed in registers with
// byte permutes and written as 8-byte runs along the token dimension, so both
// layouts are written with coalesced stores.  Amax reductions use packed
// |bf16| maxima, warp shuffles and one relaxed atomic per block (tensor
// amax) or per tile row / column (rowwise / colwise amax).
//
// Kernels and passes:
//   DELAYED    : cast (stored scale) + fused amax            -> 1 launch
//   TENSORWISE : amax pass, cast pass                        -> 2 launches (+ a clear)
//   ROWWISE    : clear, amax pass (row + column amax), cast pass, scale_inv
//                (+ amax -> scale before the cast when grouped) -> 4 or 5 launches
//   fp8_quantize_rowwise_resident: the ROWWISE passes of a plain tensor in
//                one cooperative launch with grid-wide barriers
// The rowwise / colwise amax values are accumulated in the scale_inv output
// buffers themselves (as fp32 bit patterns), turned into the scales before
// the cast pass and into scale_inv after it, so the passes need no scratch
// memory; only the single-launch form keeps its barrier counters in a
// file-scope device array.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "fp8gb.h"
#include "fp8gb_device.cuh"
#include "fp8gb_host.h"

namespace fp8gb {

constexpr int QT_THREADS = 256;
constexpr int QT_COLS = 128;          // columns per tile
constexpr int QT_PITCH = QT_COLS + 4; // shared tile row pitch in bytes
constexpr int QT_MAX_GROUPS = 4096;

struct QArgs {
    const uint16_t *x;
    int64_t rows, cols, ld_x;
    uint8_t *q_row;
    uint8_t *q_colT;
    int64_t ld_colT;
    float *sinv_row;  // ROWWISE: amax bits during the passes
    float *sinv_col;
    const float *scale_in;
    float *amax_out;
    const int32_t *offsets;
    unsigned int *err;
    int G;
    int margin;
    int64_t n_row_blocks;
    int64_t n_col_chunks;
    int scales_ready;  // rowwise cast pass: the scale buffers already hold scales (else amaxes)
    int sup_blocks;  // rowwise amax pass: 32-row blocks per super tile (1..8)
    int sup_chunks;  // rowwise amax pass: 128-column chunks per super tile (1..8)
    int64_t group_rows;  // equal groups without offsets: rows per group (a multiple of 64); 0 = one group
    // fused MoE prologues of the grouped rowwise passes (template parameter PRO)
    const int32_t *src_rows;  // QPRO_GATHER: row r of the tensor is row src_rows[r] of x
    int64_t x_rows;           // QPRO_GATHER: rows of x
    int64_t up_off;           // QPRO_SWIGLU: column offset of `up` in each row of x
    uint16_t *h_out;          // QPRO_SWIGLU: optional bf16 copy of h, [rows][ld_h]
    int64_t ld_h;
};

// Prologues of the grouped rowwise passes: the tensor is x itself, the
// gathered rows x[src_rows[r]], or h = bf16(silu(gate) * up) of the two
// halves of each row of x.  Both passes apply the prologue to what they
// read, so neither the gathered tensor nor h is ever written to memory
// (except the optional copy of h).
enum { QPRO_NONE = 0, QPRO_GATHER = 1, QPRO_SWIGLU = 2 };

// input row of tensor row r: x's own row, or src_rows[r] (checked: an index
// outside x is reported and reads as a zero row, -1)
template <int PRO>
__device__ __forceinline__ int64_t pro_src_row(const QArgs &a, int64_t r)
{
    if constexpr (PRO == QPRO_GATHER) {
        const int64_t s = __ldg(a.src_rows + r);
        if (s < 0 || s >= a.x_rows) {
            record_error(a.err, ERR_BAD_INDEX);
            return -1;
        }
        return s;
    } else {
        return r;
    }
}

// eight bf16 of the tensor at input row `src` (-1: zeros), columns col .. col + 7
template <int PRO>
__device__ __forceinline__ uint4 pro_load8(const QArgs &a, int64_t src, int64_t col)
{
    if (src < 0) return make_uint4(0, 0, 0, 0);
    const uint16_t *p = a.x + src * a.ld_x + col;
    if constexpr (PRO == QPRO_SWIGLU) {
        const uint4 g = __ldg(reinterpret_cast<const uint4 *>(p)), u = __ldg(reinterpret_cast<const uint4 *>(p + a.up_off));
        return make_uint4(swiglu2(g.x, u.x), swiglu2(g.y, u.y), swiglu2(g.z, u.z), swiglu2(g.w, u.w));
    } else {
        return __ldg(reinterpret_cast<const uint4 *>(p));
    }
}

// Row-block geometry: which input rows a tile covers and where they land in
// the transposed layout.
struct RowBlock {
    bool skip;         // block lies beyond the padded total (grouped)
    int64_t in_row0;   // first input row
    int64_t out_col0;  // first column of q_colT
    int valid;         // number of real rows (<= RB)
    int group;         // expert group (0 when ungrouped)
};

// Exclusive prefix of roundup(m_e, 32) over groups, computed by warp 0 into
// shared memory poff[0 .. G], followed by a copy of the offsets themselves
// (poff[G + 1 .. 2G + 1]) so tile lookups never wait on global memory.
// Flags malformed offsets (negative group sizes, total beyond `rows`, padded
// total beyond ld_colT).
__device__ void compute_padded_offsets(const int32_t *off, int G, int64_t rows, int64_t ld_colT, int32_t *poff,
                                       int *bad, unsigned int *err)
{
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    const int per = (G + 31) / 32;
    const int g0 = min(G, lane * per), g1 = min(G, g0 + per);
    int64_t local = 0;
    int badl = 0;
    for (int e = g0; e < g1; e++) {
        int m = off[e + 1] - off[e];
        if (m < 0) badl = 1;
        local += (int64_t)((max(m, 0) + 31) / 32) * 32;
    }
    int64_t incl = local;
    for (int d = 1; d < 32; d <<= 1) {
        int64_t v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    int64_t run = incl - local;
    int32_t *soff = poff + G + 1;
    for (int e = g0; e < g1; e++) {
        poff[e] = (int32_t)run;
        soff[e] = off[e];
        int m = off[e + 1] - off[e];
        run += (int64_t)((max(m, 0) + 31) / 32) * 32;
    }
    int64_t total = __shfl_sync(0xffffffffu, incl, 31);
    badl = __any_sync(0xffffffffu, badl);
    if (lane == 0) {
        poff[G] = (int32_t)total;
        soff[G] = off[G];
        int b = badl || off[0] != 0 || (int64_t)off[G] != rows || (ld_colT > 0 && total > ld_colT);
        *bad = b;
        if (b) record_error(err, ERR_BAD_OFFSETS);
    }
}

// Equal groups: the group of row block b (group_rows is a multiple of RB),
// by a 32-bit division whenever b and the blocks per group fit 32 bits.
template <int RB>
__device__ __forceinline__ int equal_group_of(const QArgs &a, int64_t b)
{
    const int64_t gblk = a.group_rows / RB;
    if (((b | gblk) >> 32) == 0) return (int)((uint32_t)b / (uint32_t)gblk);
    return (int)(b / gblk);
}

// Advance the (row block, column chunk) coordinates of a tile walk by one
// step without dividing (ON): backwards by one tile, or forwards by db row
// blocks and dc chunks (a grid stride of db * ncc + dc tiles).
template <bool ON>
__device__ __forceinline__ void next_tile(int64_t &b, int64_t &ci, bool back, int64_t db, int64_t dc, int64_t ncc)
{
    if constexpr (ON) {
        if (back) {
            if (--ci < 0) {
                ci = ncc - 1;
                --b;
            }
        } else {
            ci += dc;
            b += db;
            if (ci >= ncc) {
                ci -= ncc;
                ++b;
            }
        }
    }
}

template <int RB>
// `hint` (optional): the group of the caller's previous block, when blocks
// are visited in increasing order; the search steps forward from it (a few
// groups at most) before falling back to bisection.
__device__ __forceinline__ RowBlock row_block(const QArgs &a, int64_t b, const int32_t *poff, int *hint = nullptr)
{
    RowBlock rb;
    rb.skip = false;
    if (a.offsets == nullptr) {
        rb.in_row0 = b * RB;
        rb.out_col0 = b * RB;
        rb.valid = (int)(a.rows - rb.in_row0 < RB ? a.rows - rb.in_row0 : RB);
        rb.group = a.group_rows ? equal_group_of<RB>(a, b) : 0;  // equal groups: a block lies in one
    } else {
        // padded block start p = b * RB (RB == 32): last group with poff <= p
        const int64_t p = b * RB;
        if (p >= poff[a.G]) {
            rb.skip = true;
            rb.in_row0 = rb.out_col0 = 0;
            rb.valid = 0;
            rb.group = 0;
            return rb;
        }
        int lo = hint && poff[*hint] <= p ? *hint : 0;  // poff[lo] <= p
        for (int step = 0; step < 4 && lo + 1 < a.G && poff[lo + 1] <= p; ++step) ++lo;
        if (lo + 1 < a.G && poff[lo + 1] <= p) {
            int hi = a.G;  // invariant: poff[lo] <= p < poff[hi]
            while (hi - lo > 1) {
                int mid = (lo + hi) >> 1;
                if (poff[mid] <= p)
                    lo = mid;
                else
                    hi = mid;
            }
        }
        if (hint) *hint = lo;
        const int e = lo;
        const int64_t within = p - poff[e];
        const int32_t *soff = poff + a.G + 1;  // the offsets, staged next to poff
        const int64_t m = (int64_t)soff[e + 1] - soff[e];
        rb.in_row0 = soff[e] + within;
        rb.out_col0 = p;
        rb.valid = (int)(m - within < RB ? (m - within > 0 ? m - within : 0) : RB);
        rb.group = e;
    }
    return rb;
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v)
{
    for (int d = 16; d > 0; d >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, d));
    return v;
}

// Block-wide max of a u32, then one relaxed atomic into `dst` (fp32 bits of a
// non-negative value or NaN).
__device__ __forceinline__ void block_amax_atomic(uint32_t v, float *dst, uint32_t *red)
{
    v = warp_max_u32(v);
    const int w = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t m = 0;
        for (int i = 0; i < QT_THREADS / 32; i++) m = max(m, red[i]);
        atomicMax(reinterpret_cast<unsigned int *>(dst), m);
    }
}

// ---------------------------------------------------------------------------
// Pass 1 (TENSORWISE and ROWWISE): amax only.
//   MODE 0: whole-tensor amax into amax_out.
//   MODE 1: per-row amax into sinv_row, per-(group, column) amax into
//           sinv_col (both as fp32 bits, buffers zeroed by the host), plus
//           the whole-tensor amax into amax_out when given.
// ---------------------------------------------------------------------------
template <int RB, int MODE>
__global__ void __launch_bounds__(QT_THREADS) amax_kernel(QArgs a)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    int32_t *poff = reinterpret_cast<int32_t *>(dsm);
    __shared__ uint32_t red[QT_THREADS / 32];
    __shared__ uint32_t colw[QT_THREADS / 32][16][4];  // per warp: 16 column groups x 4 packed words
    __shared__ int bad;
    if (a.offsets) {
        compute_padded_offsets(a.offsets, a.G, a.rows, 0, poff, &bad, a.err);
        __syncthreads();
        if (bad) return;
    }
    const int t = threadIdx.x, cg = t & 15, roff = t >> 4;
    const int64_t n_tiles = a.n_row_blocks * a.n_col_chunks;
    uint32_t tensor_acc = 0;
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int64_t b = tile / a.n_col_chunks;
        const int64_t c0 = (tile % a.n_col_chunks) * QT_COLS;
        const RowBlock rb = row_block<RB>(a, b, poff);
        if (rb.skip) continue;
        const int64_t col = c0 + cg * 8;
        const bool col_ok = col < a.cols;
        uint4 v[RB / 16];
#pragma unroll
        for (int i = 0; i < RB / 16; i++) {
            const int r = i * 16 + roff;
            if (col_ok && r < rb.valid)
                v[i] = __ldg(reinterpret_cast<const uint4 *>(a.x + (rb.in_row0 + r) * a.ld_x + col));
            else
                v[i] = make_uint4(0, 0, 0, 0);
        }
        uint32_t cacc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < RB / 16; i++) {
            uint32_t racc = 0;
            racc = absmax_bf16x2(racc, v[i].x);
            racc = absmax_bf16x2(racc, v[i].y);
            racc = absmax_bf16x2(racc, v[i].z);
            racc = absmax_bf16x2(racc, v[i].w);
            if constexpr (MODE == 1) {
                cacc[0] = absmax_bf16x2(cacc[0], v[i].x);
                cacc[1] = absmax_bf16x2(cacc[1], v[i].y);
                cacc[2] = absmax_bf16x2(cacc[2], v[i].z);
                cacc[3] = absmax_bf16x2(cacc[3], v[i].w);
                // row amax: reduce over the 16 threads sharing this row
                uint32_t rm = fold_absmax(racc);
                for (int d = 8; d > 0; d >>= 1) rm = max(rm, __shfl_xor_sync(0xffffffffu, rm, d));
                const int r = i * 16 + roff;
                if (cg == 0 && r < rb.valid && a.sinv_row)
                    atomicMax(reinterpret_cast<unsigned int *>(a.sinv_row) + rb.in_row0 + r, rm);
            }
            tensor_acc = max(tensor_acc, fold_absmax(racc));
        }
        if constexpr (MODE == 1) {
            if (a.sinv_col) {
                // column amax over the tile's rows: lanes t and t^16 share columns
#pragma unroll
                for (int k = 0; k < 4; k++) cacc[k] = __vmaxu2(cacc[k], __shfl_xor_sync(0xffffffffu, cacc[k], 16));
                const int w = t >> 5;
                if ((t & 31) < 16) {
#pragma unroll
                    for (int k = 0; k < 4; k++) colw[w][cg][k] = cacc[k];
                }
                __syncthreads();
                if (t < QT_COLS) {
                    const int g = t >> 3, j = t & 7;  // column c0 + 8g + j
                    uint32_t m = 0;
                    for (int ww = 0; ww < QT_THREADS / 32; ww++) {
                        const uint32_t word = colw[ww][g][j >> 1];
                        m = max(m, (j & 1) ? (word >> 16) : (word & 0xFFFFu));
                    }
                    const int64_t c = c0 + t;
                    if (c < a.cols && rb.valid > 0)
                        atomicMax(reinterpret_cast<unsigned int *>(a.sinv_col) + (int64_t)rb.group * a.cols + c,
                                  m << 16);
                }
                __syncthreads();
            }
        }
    }
    if (MODE == 0 || a.amax_out) block_amax_atomic(tensor_acc, a.amax_out, red);
}

// ---------------------------------------------------------------------------
// Pass 1 of the ROWWISE recipe on a plain (ungrouped) tensor: row amax and
// column amax in one read.
//
// Persistent blocks, each owning a contiguous run of tiles in row-major tile
// order, so consecutive tiles mostly belong to the same row block: the row
// maxima stay in registers across the run and are flushed (one relaxed
// atomic per row) only when the row block changes or the run ends.  The
// tile coordinates are stepped along the run (one division per run, none
// per tile), and an equal-groups tensor's group is looked up only when the
// row block changes.  The next
// tile's 16-byte loads are issued before the current tile is reduced, so
// every thread keeps loads in flight while it reduces.  Column maxima are
// reduced per tile (shuffles, then shared memory across the 8 warps) and
// flushed with one relaxed atomic per column per tile.
// ---------------------------------------------------------------------------
// L2 eviction-priority hints for the single-launch rowwise path: the amax
// pass marks x evict-last so the cast pass finds it in L2; the cast pass
// reads x for the last time and writes its outputs evict-first.
__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint4 ld_nc_hint(const void *ptr, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr), "l"(pol));
    return v;
}

__device__ __forceinline__ void st_hint(void *ptr, uint2 v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(ptr), "r"(v.x), "r"(v.y), "l"(pol)
                 : "memory");
}

template <int RB, bool HINTS = false>
__device__ __forceinline__ void dense_tile_load(const QArgs &a, int64_t b, int64_t chunk, int cg, int roff,
                                                uint4 (&v)[RB / 16])
{
    uint64_t pol = 0;
    if constexpr (HINTS) pol = l2_policy_evict_last();
    const int64_t col = chunk * QT_COLS + cg * 8;
    const int64_t row0 = b * RB;
#pragma unroll
    for (int i = 0; i < RB / 16; i++) {
        const int64_t r = row0 + i * 16 + roff;
        if (col < a.cols && r < a.rows) {
            if constexpr (HINTS)
                v[i] = ld_nc_hint(a.x + r * a.ld_x + col, pol);
            else
                v[i] = __ldg(reinterpret_cast<const uint4 *>(a.x + r * a.ld_x + col));
        } else
            v[i] = make_uint4(0, 0, 0, 0);
    }
}

// the run of tiles [first, last) of one block
template <int RB, bool HINTS = false>
__device__ __forceinline__ void dense_rowcol_amax_run(const QArgs &a, int64_t first, int64_t last)
{
    __shared__ uint32_t red[QT_THREADS / 32];
    __shared__ uint32_t colw[QT_THREADS / 32][16][4];  // per warp: 16 column groups x 4 packed words
    const int t = threadIdx.x, cg = t & 15, roff = t >> 4;
    uint32_t tensor_acc = 0;
    uint32_t racc[RB / 16];
#pragma unroll
    for (int i = 0; i < RB / 16; i++) racc[i] = 0;
    // coordinates of the tile being prefetched: one division per run, then increments
    int64_t nb = first < last ? first / a.n_col_chunks : -1;
    int64_t nc = first < last ? first - nb * a.n_col_chunks : 0;
    int64_t cur_b = nb;
    int grp = a.group_rows && nb >= 0 ? equal_group_of<RB>(a, nb) : 0;

    // row maxima of row block b: 16 threads share a row; one atomic per row
    auto flush_rows = [&](int64_t b) {
#pragma unroll
        for (int i = 0; i < RB / 16; i++) {
            uint32_t rm = racc[i];
            for (int d = 8; d > 0; d >>= 1) rm = max(rm, __shfl_xor_sync(0xffffffffu, rm, d));
            const int64_t r = b * RB + i * 16 + roff;
            if (cg == 0 && r < a.rows && a.sinv_row)
                atomicMax(reinterpret_cast<unsigned int *>(a.sinv_row) + r, rm);
            racc[i] = 0;
        }
    };

    uint4 nv[RB / 16];
    if (first < last) dense_tile_load<RB, HINTS>(a, nb, nc, cg, roff, nv);
    for (int64_t tile = first; tile < last; tile++) {
        uint4 v[RB / 16];
#pragma unroll
        for (int i = 0; i < RB / 16; i++) v[i] = nv[i];
        const int64_t b = nb, c0 = nc * QT_COLS;
        if (++nc == a.n_col_chunks) {
            nc = 0;
            ++nb;
        }
        if (tile + 1 < last) dense_tile_load<RB, HINTS>(a, nb, nc, cg, roff, nv);
        if (b != cur_b) {  // warp-uniform: the whole block moves to the next row block
            flush_rows(cur_b);
            cur_b = b;
            if (a.group_rows) grp = equal_group_of<RB>(a, b);
        }
        uint32_t cacc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < RB / 16; i++) {
            uint32_t rr = 0;
            rr = absmax_bf16x2(rr, v[i].x);
            rr = absmax_bf16x2(rr, v[i].y);
            rr = absmax_bf16x2(rr, v[i].z);
            rr = absmax_bf16x2(rr, v[i].w);
            cacc[0] = absmax_bf16x2(cacc[0], v[i].x);
            cacc[1] = absmax_bf16x2(cacc[1], v[i].y);
            cacc[2] = absmax_bf16x2(cacc[2], v[i].z);
            cacc[3] = absmax_bf16x2(cacc[3], v[i].w);
            const uint32_t f = fold_absmax(rr);
            racc[i] = max(racc[i], f);
            tensor_acc = max(tensor_acc, f);
        }
        if (a.sinv_col) {
            // column maxima over the tile's rows: lanes t and t^16 share columns
#pragma unroll
            for (int k = 0; k < 4; k++) cacc[k] = __vmaxu2(cacc[k], __shfl_xor_sync(0xffffffffu, cacc[k], 16));
            const int w = t >> 5;
            if ((t & 31) < 16) {
#pragma unroll
                for (int k = 0; k < 4; k++) colw[w][cg][k] = cacc[k];
            }
            __syncthreads();
            if (t < QT_COLS) {
                const int g = t >> 3, j = t & 7;  // column c0 + 8g + j
                uint32_t m = 0;
                for (int ww = 0; ww < QT_THREADS / 32; ww++) {
                    const uint32_t word = colw[ww][g][j >> 1];
                    m = max(m, (j & 1) ? (word >> 16) : (word & 0xFFFFu));
                }
                const int64_t c = c0 + t;
                // equal groups: the tile's rows lie in one group (group_rows is a multiple of RB)
                if (c < a.cols) atomicMax(reinterpret_cast<unsigned int *>(a.sinv_col) + (int64_t)grp * a.cols + c, m << 16);
            }
            __syncthreads();
        }
    }
    if (cur_b >= 0) flush_rows(cur_b);
    if (a.amax_out) block_amax_atomic(tensor_acc, a.amax_out, red);
}

template <int RB>
__global__ void __launch_bounds__(QT_THREADS) dense_rowcol_amax_kernel(QArgs a, int64_t tiles_per_block)
{
    const int64_t n_tiles = a.n_row_blocks * a.n_col_chunks;
    const int64_t first = (int64_t)blockIdx.x * tiles_per_block;
    const int64_t last = first + tiles_per_block < n_tiles ? first + tiles_per_block : n_tiles;
    dense_rowcol_amax_run<RB>(a, first, last);
}

// ---------------------------------------------------------------------------
// Pass 1 of the ROWWISE recipe: row amax and (group, column) amax.
//
// A thread block covers a super tile of up to 8 row blocks of 32 rows x up
// to 8 column chunks of 128 columns (smaller super tiles for smaller tensors,
// so that the grid still fills the GPU).  Column maxima are kept in registers
// across the row blocks of one group and reduced / flushed (one relaxed
// atomic per column) when the group changes or the chunk ends; row maxima are
// kept across the column chunks and flushed once per row per super tile.
// Both amaxes are accumulated as fp32 bit patterns in the scale_inv output
// buffers (zeroed by the host).
// ---------------------------------------------------------------------------
constexpr int SUP_BLOCKS = 8;   // at most 32-row blocks per super tile
constexpr int SUP_CHUNKS = 8;   // at most 128-column chunks per super tile

__device__ __forceinline__ void flush_col_amax(const QArgs &a, uint32_t (&cacc)[4], int group, int64_t c0,
                                               uint32_t (*colw)[16][4])
{
    const int t = threadIdx.x, cg = t & 15, w = t >> 5;
#pragma unroll
    for (int k = 0; k < 4; k++) cacc[k] = __vmaxu2(cacc[k], __shfl_xor_sync(0xffffffffu, cacc[k], 16));
    if ((t & 31) < 16) {
#pragma unroll
        for (int k = 0; k < 4; k++) colw[w][cg][k] = cacc[k];
    }
    __syncthreads();
    if (t < QT_COLS) {
        const int g = t >> 3, j = t & 7;  // column c0 + 8g + j
        uint32_t m = 0;
#pragma unroll
        for (int ww = 0; ww < QT_THREADS / 32; ww++) {
            const uint32_t word = colw[ww][g][j >> 1];
            m = max(m, (j & 1) ? (word >> 16) : (word & 0xFFFFu));
        }
        const int64_t c = c0 + t;
        if (c < a.cols && m != 0)
            atomicMax(reinterpret_cast<unsigned int *>(a.sinv_col) + (int64_t)group * a.cols + c, m << 16);
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 4; k++) cacc[k] = 0;
}

template <int PRO>
__global__ void __launch_bounds__(QT_THREADS) rowcol_amax_kernel(QArgs a)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    int32_t *poff = reinterpret_cast<int32_t *>(dsm);
    __shared__ uint32_t red[QT_THREADS / 32];
    __shared__ uint32_t colw[QT_THREADS / 32][16][4];
    __shared__ RowBlock srb[SUP_BLOCKS];
    __shared__ int64_t ssrc[PRO == QPRO_NONE ? 1 : SUP_BLOCKS * 32];  // input row of each row of the super tile
    __shared__ int bad;
    if (a.offsets) {
        compute_padded_offsets(a.offsets, a.G, a.rows, 0, poff, &bad, a.err);
        __syncthreads();
        if (bad) return;
    }
    const int t = threadIdx.x, cg = t & 15, roff = t >> 4;
    const int SB = a.sup_blocks, SC = a.sup_chunks;
    const int64_t n_sr = (a.n_row_blocks + SB - 1) / SB;
    const int64_t n_sc = (a.n_col_chunks + SC - 1) / SC;
    uint32_t tensor_acc = 0;
    for (int64_t st = blockIdx.x; st < n_sr * n_sc; st += gridDim.x) {
        const int64_t sr = st / n_sc, sc = st % n_sc;
        __syncthreads();
        if (t < SUP_BLOCKS) {
            const int64_t b = sr * SB + t;
            if (t < SB && b < a.n_row_blocks) {
                srb[t] = row_block<32>(a, b, poff);
            } else {
                srb[t].skip = true;
                srb[t].valid = 0;
            }
        }
        __syncthreads();
        if constexpr (PRO != QPRO_NONE) {
            if (t < SUP_BLOCKS * 32) {
                const RowBlock &rb = srb[t >> 5];
                const int r = t & 31;
                ssrc[t] = !rb.skip && r < rb.valid ? pro_src_row<PRO>(a, rb.in_row0 + r) : -1;
            }
            __syncthreads();
        }
        uint32_t rmax[SUP_BLOCKS][2];
#pragma unroll
        for (int kb = 0; kb < SUP_BLOCKS; kb++) rmax[kb][0] = rmax[kb][1] = 0;
        // step k: half k % 2 (row blocks 4 (k % 2) .. + 3) of column chunk k / 2;
        // the next step's loads are issued before this step is reduced
        auto load_step = [&](int k, uint4 (&v)[SUP_BLOCKS / 2][2]) {
            const int jj = k >> 1, hf = k & 1;
            const int64_t cc0 = (sc * SC + jj) * QT_COLS;
            const int64_t col = cc0 + cg * 8;
            const bool ok = jj < SC && hf * (SUP_BLOCKS / 2) < SB && col < a.cols;
#pragma unroll
            for (int kk = 0; kk < SUP_BLOCKS / 2; kk++) {
                const RowBlock &rb = srb[hf * (SUP_BLOCKS / 2) + kk];
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int r = h * 16 + roff;
                    if constexpr (PRO == QPRO_NONE) {
                        if (ok && !rb.skip && r < rb.valid)
                            v[kk][h] = __ldg(reinterpret_cast<const uint4 *>(a.x + (rb.in_row0 + r) * a.ld_x + col));
                        else
                            v[kk][h] = make_uint4(0, 0, 0, 0);
                    } else {
                        v[kk][h] = pro_load8<PRO>(a, ok ? ssrc[(hf * (SUP_BLOCKS / 2) + kk) * 32 + r] : -1, col);
                    }
                }
            }
        };
        uint4 nv[SUP_BLOCKS / 2][2];
        load_step(0, nv);
        uint32_t cacc[4] = {0, 0, 0, 0};
        int cur_group = -1;
        for (int j = 0; j < SC; j++) {
            const int64_t c0 = (sc * SC + j) * QT_COLS;
            if (c0 >= a.cols) break;  // uniform
#pragma unroll
            for (int half = 0; half < 2; half++) {
                const int k = 2 * j + half;
                if (half * (SUP_BLOCKS / 2) >= SB) continue;  // uniform: no second half
                uint4 v[SUP_BLOCKS / 2][2];
#pragma unroll
                for (int kk = 0; kk < SUP_BLOCKS / 2; kk++) {
                    v[kk][0] = nv[kk][0];
                    v[kk][1] = nv[kk][1];
                }
                // the next step that runs: half 1 exists only when SB > SUP_BLOCKS / 2
                const int kn = (k & 1) == 0 && SB <= SUP_BLOCKS / 2 ? k + 2 : k + 1;
                if (kn < 2 * SC) load_step(kn, nv);
#pragma unroll
                for (int kk = 0; kk < SUP_BLOCKS / 2; kk++) {
                    const int kb = half * (SUP_BLOCKS / 2) + kk;
                    const RowBlock &rb = srb[kb];
                    if (rb.skip) continue;  // uniform
                    if (a.sinv_col && cur_group >= 0 && rb.group != cur_group)
                        flush_col_amax(a, cacc, cur_group, c0, colw);
                    cur_group = rb.group;
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const uint4 w4 = v[kk][h];
                        uint32_t racc = 0;
                        racc = absmax_bf16x2(racc, w4.x);
                        racc = absmax_bf16x2(racc, w4.y);
                        racc = absmax_bf16x2(racc, w4.z);
                        racc = absmax_bf16x2(racc, w4.w);
                        cacc[0] = absmax_bf16x2(cacc[0], w4.x);
                        cacc[1] = absmax_bf16x2(cacc[1], w4.y);
                        cacc[2] = absmax_bf16x2(cacc[2], w4.z);
                        cacc[3] = absmax_bf16x2(cacc[3], w4.w);
                        rmax[kb][h] = max(rmax[kb][h], fold_absmax(racc));
                    }
                }
                const bool chunk_end = half == 1 || (SUP_BLOCKS / 2) >= SB;
                if (chunk_end) {
                    if (a.sinv_col && cur_group >= 0) flush_col_amax(a, cacc, cur_group, c0, colw);
                    cur_group = -1;
                }
            }
        }
        // row maxima: reduce over the 16 threads sharing a row, one atomic per row
#pragma unroll
        for (int kb = 0; kb < SUP_BLOCKS; kb++) {
#pragma unroll
            for (int h = 0; h < 2; h++) {
                uint32_t m = rmax[kb][h];
                for (int d = 8; d > 0; d >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, d));
                tensor_acc = max(tensor_acc, m);
                const RowBlock &rb = srb[kb];
                const int r = h * 16 + roff;
                if (cg == 0 && !rb.skip && r < rb.valid && a.sinv_row && m != 0)
                    atomicMax(reinterpret_cast<unsigned int *>(a.sinv_row) + rb.in_row0 + r, m);
            }
        }
    }
    if (a.amax_out) block_amax_atomic(tensor_acc, a.amax_out, red);
}

// ---------------------------------------------------------------------------
// Cast pass.
//   SMODE 0: one scale for the tensor (DELAYED: scale_in[0]; TENSORWISE:
//            from amax_out[0]).  DELAYED also max-accumulates the amax.
//   SMODE 1: ROWWISE -- row scales from the row amax, column scales from the
//            (group, column) amax.
// ---------------------------------------------------------------------------
// the tiles blockIdx.x, blockIdx.x + gridDim.x, ... , or with run_last >= 0
// the tiles run_last, run_last - 1, ..., run_first (a block's own run, newest
// first); dsm: the block's dynamic shared memory (RB * QT_PITCH bytes, then
// the grouped offsets)
template <int FMT, int RB, int SMODE, bool DELAYED, bool DO_ROW, bool DO_COLT, bool HINTS = false>
__device__ __forceinline__ void cast_run(const QArgs &a, unsigned char *dsm, int64_t run_first = 0,
                                         int64_t run_last = -1)
{
    uint64_t pol = 0;
    if constexpr (HINTS) pol = l2_policy_evict_first();
    uint8_t *tileT = dsm;                                                    // [RB][QT_PITCH]
    int32_t *poff = reinterpret_cast<int32_t *>(dsm + RB * QT_PITCH);       // grouped only
    __shared__ float srow[RB];
    __shared__ float scol[QT_COLS];
    __shared__ uint32_t red[QT_THREADS / 32];
    __shared__ int bad;
    const float fmax = fp8_max_of(FMT);
    if (a.offsets) {
        compute_padded_offsets(a.offsets, a.G, a.rows, DO_COLT ? a.ld_colT : 0, poff, &bad, a.err);
        __syncthreads();
        if (bad) return;
    }

    float s_tensor = 1.0f;
    if constexpr (SMODE == 0) {
        if constexpr (DELAYED)
            s_tensor = a.scale_in[0];
        else
            s_tensor = scale_from_amax(a.amax_out[0], fmax, a.margin);
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            const float sinv = recip_rn(s_tensor);
            if (DO_ROW) a.sinv_row[0] = sinv;
            if (DO_COLT) a.sinv_col[0] = sinv;
        }
    }

    const int t = threadIdx.x, cg = t & 15, roff = t >> 4;
    const int64_t n_tiles = a.n_row_blocks * a.n_col_chunks;
    uint32_t amax_acc = 0;
    const bool by_run = run_last >= 0;
    const int64_t ncc = a.n_col_chunks;
    const int64_t step = by_run ? -1 : (int64_t)gridDim.x;
    int64_t tile = by_run ? run_last : blockIdx.x;
    // Tile coordinates (row block, chunk).  The per-row / per-column scale
    // mode keeps them across tiles and steps them without dividing (its tile
    // body then needs 40 registers instead of 48: six blocks per SM instead
    // of five, measured 4-6 % faster on expert-weight stacks); the one-scale
    // mode divides per tile (the stepped form measured 1.5 % slower there).
    int64_t blk = 0, ci = 0, db = 0, dc = 0;
    if constexpr (SMODE == 1) {
        blk = tile / ncc;
        ci = tile - blk * ncc;
        if (!by_run && tile + step < n_tiles) {  // a second tile (plain tensors launch one block per tile)
            db = step / ncc;
            dc = step - db * ncc;
        }
    }
    for (; by_run ? tile >= run_first : tile < n_tiles; tile += step, next_tile<SMODE == 1>(blk, ci, by_run, db, dc, ncc)) {
        if constexpr (SMODE == 0) {
            blk = tile / ncc;
            ci = tile - blk * ncc;
        }
        const int64_t c0 = ci * QT_COLS;
        const RowBlock rb = row_block<RB>(a, blk, poff);
        if (rb.skip) continue;
        const int64_t col = c0 + cg * 8;
        const bool col_ok = col < a.cols;

        uint4 v[RB / 16];
#pragma unroll
        for (int i = 0; i < RB / 16; i++) {
            const int r = i * 16 + roff;
            if (col_ok && r < rb.valid) {
                if constexpr (HINTS)
                    v[i] = ld_nc_hint(a.x + (rb.in_row0 + r) * a.ld_x + col, pol);
                else
                    v[i] = __ldg(reinterpret_cast<const uint4 *>(a.x + (rb.in_row0 + r) * a.ld_x + col));
            } else {
                v[i] = make_uint4(0, 0, 0, 0);
            }
        }
        if constexpr (SMODE == 1) {
            // per-tile scales from the amax accumulated by pass 1
            // the scale buffers hold either the amaxes of pass 1 (turned into
            // scales here) or, when scales_ready, the scales themselves
            if (DO_ROW && t < RB) {
                const float v = t < rb.valid ? a.sinv_row[rb.in_row0 + t] : 0.0f;
                srow[t] = a.scales_ready ? (t < rb.valid ? v : 1.0f) : scale_from_amax(v, fmax, a.margin);
            }
            if (DO_COLT && t >= QT_THREADS - QT_COLS) {
                const int j = t - (QT_THREADS - QT_COLS);
                const float v = c0 + j < a.cols ? a.sinv_col[(int64_t)rb.group * a.cols + c0 + j] : 0.0f;
                scol[j] = a.scales_ready ? (c0 + j < a.cols ? v : 1.0f) : scale_from_amax(v, fmax, a.margin);
            }
            __syncthreads();
        }

#pragma unroll
        for (int i = 0; i < RB / 16; i++) {
            const int r = i * 16 + roff;
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            if constexpr (DELAYED) {
#pragma unroll
                for (int k = 0; k < 4; k++) amax_acc = absmax_bf16x2(amax_acc, w[k]);
            }
            uint32_t rowb0, rowb1, colb0, colb1;
            if constexpr (SMODE == 0) {
                const uint2 b = cvt8_scaled<FMT>(v[i], s_tensor);
                rowb0 = colb0 = b.x;
                rowb1 = colb1 = b.y;
            } else {
                if constexpr (DO_ROW) {
                    const uint2 b = cvt8_scaled<FMT>(v[i], srow[r]);
                    rowb0 = b.x;
                    rowb1 = b.y;
                }
                if constexpr (DO_COLT) {
                    const float *sc = scol + cg * 8;
                    const float cs[8] = {sc[0], sc[1], sc[2], sc[3], sc[4], sc[5], sc[6], sc[7]};
                    const uint2 b = cvt8_scaled<FMT>(v[i], cs);
                    colb0 = b.x;
                    colb1 = b.y;
                }
            }
            const bool ok = col_ok && r < rb.valid;
            if constexpr (DO_ROW) {
                if (ok) {
                    if constexpr (HINTS)
                        st_hint(a.q_row + (rb.in_row0 + r) * a.cols + col, make_uint2(rowb0, rowb1), pol);
                    else
                        *reinterpret_cast<uint2 *>(a.q_row + (rb.in_row0 + r) * a.cols + col) = make_uint2(rowb0, rowb1);
                }
            }
            if constexpr (DO_COLT) {
                uint32_t *dst = reinterpret_cast<uint32_t *>(tileT + r * QT_PITCH + cg * 8);
                dst[0] = ok ? colb0 : 0u;  // rows past the block's end become zero padding
                dst[1] = ok ? colb1 : 0u;
            }
        }

        if constexpr (DO_COLT) {
            __syncthreads();
            // transposed write-out: item = (column quad qa, 8-row chunk q)
            constexpr int NQ = RB / 8;
            for (int item = t; item < 32 * NQ; item += QT_THREADS) {
                const int q = item % NQ, qa = item / NQ;
                uint32_t wv[8];
#pragma unroll
                for (int i = 0; i < 8; i++) wv[i] = *reinterpret_cast<const uint32_t *>(tileT + (q * 8 + i) * QT_PITCH + qa * 4);
                // 8 rows x 4 columns of bytes -> 4 columns x 8 rows
                const uint32_t a01l = __byte_perm(wv[0], wv[1], 0x5140), a01h = __byte_perm(wv[0], wv[1], 0x7362);
                const uint32_t a23l = __byte_perm(wv[2], wv[3], 0x5140), a23h = __byte_perm(wv[2], wv[3], 0x7362);
                const uint32_t a45l = __byte_perm(wv[4], wv[5], 0x5140), a45h = __byte_perm(wv[4], wv[5], 0x7362);
                const uint32_t a67l = __byte_perm(wv[6], wv[7], 0x5140), a67h = __byte_perm(wv[6], wv[7], 0x7362);
                uint2 o[4];
                o[0] = make_uint2(__byte_perm(a01l, a23l, 0x5410), __byte_perm(a45l, a67l, 0x5410));
                o[1] = make_uint2(__byte_perm(a01l, a23l, 0x7632), __byte_perm(a45l, a67l, 0x7632));
                o[2] = make_uint2(__byte_perm(a01h, a23h, 0x5410), __byte_perm(a45h, a67h, 0x5410));
                o[3] = make_uint2(__byte_perm(a01h, a23h, 0x7632), __byte_perm(a45h, a67h, 0x7632));
                const int r0 = q * 8;
                // grouped blocks always write the full 32-byte padded extent
                const int lim = a.offsets ? RB : rb.valid;
                if (r0 >= lim) continue;
#pragma unroll
                for (int jj = 0; jj < 4; jj++) {
                    const int64_t c = c0 + qa * 4 + jj;
                    if (c >= a.cols) break;
                    uint8_t *dst = a.q_colT + c * a.ld_colT + rb.out_col0 + r0;
                    if (r0 + 8 <= lim) {
                        if constexpr (HINTS)
                            st_hint(dst, o[jj], pol);
                        else
                            *reinterpret_cast<uint2 *>(dst) = o[jj];
                    } else {
                        const uint64_t bits = ((uint64_t)o[jj].y << 32) | o[jj].x;
                        for (int k = 0; k < lim - r0; k++) dst[k] = (uint8_t)(bits >> (8 * k));
                    }
                }
            }
            __syncthreads();
        } else if constexpr (SMODE == 1) {
            __syncthreads();
        }
    }
    if constexpr (DELAYED) block_amax_atomic(fold_absmax(amax_acc), a.amax_out, red);
}

template <int FMT, int RB, int SMODE, bool DELAYED, bool DO_ROW, bool DO_COLT>
__global__ void __launch_bounds__(QT_THREADS) cast_kernel(QArgs a)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    cast_run<FMT, RB, SMODE, DELAYED, DO_ROW, DO_COLT>(a, dsm);
}

// ---------------------------------------------------------------------------
// Cast pass of a grouped tensor (expert token rows or stacked expert weights):
// tiles of four consecutive padded 32-row blocks (128 padded rows) x 64
// columns.  The four blocks may belong to different groups, but they are
// adjacent in the padded space, so each column of the tile is one contiguous
// 128-byte run of q_colT; each thread converts row r of every block (rows r,
// 32 + r, 64 + r, 96 + r of the tile) for 8 columns.  Scales as in the
// plain cast pass: one tensor scale (SMODE 0) or row scales plus the
// (group, column) scales of each block's group (SMODE 1).
// ---------------------------------------------------------------------------
constexpr int GT_BLOCKS = 4;   // padded 32-row blocks per tile
constexpr int GT_COLS = 64;    // columns per tile
constexpr int GT_ROWS = 32 * GT_BLOCKS;

// tileT word (row r, word w of the row's 16): the word index is XORed with
// the row's 8-row chunk, so the transposed read of a chunk spreads over banks
__device__ __forceinline__ int gt_word(int r, int w) { return r * (GT_COLS / 4) + (w ^ ((r >> 3) & 15)); }

template <int FMT, int SMODE, bool DELAYED, bool DO_ROW, bool DO_COLT, int PRO = QPRO_NONE>
__global__ void __launch_bounds__(QT_THREADS, 6) grouped_cast_kernel(QArgs a)
{
    __shared__ int64_t ssrc[PRO == QPRO_NONE ? 1 : GT_ROWS];  // input row of each row of the tile
    extern __shared__ __align__(16) unsigned char dsm[];
    int32_t *poff = reinterpret_cast<int32_t *>(dsm);
    __shared__ uint32_t tileT[GT_ROWS * GT_COLS / 4];
    __shared__ float srow[GT_ROWS];
    __shared__ float scol[GT_BLOCKS][GT_COLS];
    __shared__ RowBlock srb[GT_BLOCKS];
    __shared__ uint32_t red[QT_THREADS / 32];
    __shared__ int bad;
    const float fmax = fp8_max_of(FMT);
    compute_padded_offsets(a.offsets, a.G, a.rows, DO_COLT ? a.ld_colT : 0, poff, &bad, a.err);
    __syncthreads();
    if (bad) return;

    float s_tensor = 1.0f;
    if constexpr (SMODE == 0) {
        if constexpr (DELAYED)
            s_tensor = a.scale_in[0];
        else
            s_tensor = scale_from_amax(a.amax_out[0], fmax, a.margin);
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            const float sinv = recip_rn(s_tensor);
            if (DO_ROW) a.sinv_row[0] = sinv;
            if (DO_COLT) a.sinv_col[0] = sinv;
        }
    }

    const int t = threadIdx.x, cg = t & 7, roff = t >> 3;
    int hint = 0;  // threads 0 .. GT_BLOCKS - 1: the group of their previous block
    const int64_t n_cchunks = (a.cols + GT_COLS - 1) / GT_COLS;
    const int64_t n_tiles = (a.n_row_blocks + GT_BLOCKS - 1) / GT_BLOCKS * n_cchunks;
    uint32_t amax_acc = 0;
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int64_t b0 = tile / n_cchunks * GT_BLOCKS;
        const int64_t c0 = (tile % n_cchunks) * GT_COLS;
        if (t < GT_BLOCKS) {
            if (b0 + t < a.n_row_blocks) {
                srb[t] = row_block<32>(a, b0 + t, poff, &hint);
            } else {
                srb[t].skip = true;
                srb[t].valid = 0;
            }
        }
        __syncthreads();
        if (srb[0].skip) break;  // past the padded total: so is every later tile of this block
        const int64_t col = c0 + cg * 8;
        const bool col_ok = col < a.cols;
        if constexpr (PRO != QPRO_NONE) {
            if (t < GT_ROWS) {
                const RowBlock &rb = srb[t >> 5];
                const int r = t & 31;
                ssrc[t] = !rb.skip && r < rb.valid ? pro_src_row<PRO>(a, rb.in_row0 + r) : -1;
            }
            __syncthreads();
        }

        uint4 v[GT_BLOCKS];
#pragma unroll
        for (int i = 0; i < GT_BLOCKS; i++) {
            const RowBlock &rb = srb[i];
            if constexpr (PRO == QPRO_NONE) {
                if (!rb.skip && col_ok && roff < rb.valid)
                    v[i] = __ldg(reinterpret_cast<const uint4 *>(a.x + (rb.in_row0 + roff) * a.ld_x + col));
                else
                    v[i] = make_uint4(0, 0, 0, 0);
            } else {
                v[i] = pro_load8<PRO>(a, col_ok ? ssrc[i * 32 + roff] : -1, col);
                if constexpr (PRO == QPRO_SWIGLU) {
                    if (a.h_out && !rb.skip && col_ok && roff < rb.valid)
                        *reinterpret_cast<uint4 *>(a.h_out + (rb.in_row0 + roff) * a.ld_h + col) = v[i];
                }
            }
        }
        if constexpr (SMODE == 1) {
            if (DO_ROW && t < GT_ROWS) {
                const RowBlock &rb = srb[t >> 5];
                const int r = t & 31;
                const bool ok = !rb.skip && r < rb.valid;
                const float w = ok ? a.sinv_row[rb.in_row0 + r] : 0.0f;
                srow[t] = a.scales_ready ? (ok ? w : 1.0f) : scale_from_amax(w, fmax, a.margin);
            }
            if (DO_COLT) {
                const int i = t / GT_COLS, j = t % GT_COLS;
                const RowBlock &rb = srb[i];
                const bool ok = !rb.skip && c0 + j < a.cols;
                const float w = ok ? a.sinv_col[(int64_t)rb.group * a.cols + c0 + j] : 0.0f;
                scol[i][j] = a.scales_ready ? (ok ? w : 1.0f) : scale_from_amax(w, fmax, a.margin);
            }
            __syncthreads();
        }

#pragma unroll
        for (int i = 0; i < GT_BLOCKS; i++) {
            const RowBlock &rb = srb[i];
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            if constexpr (DELAYED) {
#pragma unroll
                for (int k = 0; k < 4; k++) amax_acc = absmax_bf16x2(amax_acc, w[k]);
            }
            uint32_t rowb0 = 0, rowb1 = 0, colb0 = 0, colb1 = 0;
            if constexpr (SMODE == 0) {
                const uint2 b = cvt8_scaled<FMT>(v[i], s_tensor);
                rowb0 = colb0 = b.x;
                rowb1 = colb1 = b.y;
            } else {
                if constexpr (DO_ROW) {
                    const uint2 b = cvt8_scaled<FMT>(v[i], srow[i * 32 + roff]);
                    rowb0 = b.x;
                    rowb1 = b.y;
                }
                if constexpr (DO_COLT) {
                    const float *sc = &scol[i][cg * 8];
                    const float cs[8] = {sc[0], sc[1], sc[2], sc[3], sc[4], sc[5], sc[6], sc[7]};
                    const uint2 b = cvt8_scaled<FMT>(v[i], cs);
                    colb0 = b.x;
                    colb1 = b.y;
                }
            }
            const bool ok = !rb.skip && col_ok && roff < rb.valid;
            if constexpr (DO_ROW) {
                if (ok)
                    *reinterpret_cast<uint2 *>(a.q_row + (rb.in_row0 + roff) * a.cols + col) = make_uint2(rowb0, rowb1);
            }
            if constexpr (DO_COLT) {
                const int r = i * 32 + roff;
                tileT[gt_word(r, 2 * cg)] = ok ? colb0 : 0u;  // rows past a block's end become zero padding
                tileT[gt_word(r, 2 * cg + 1)] = ok ? colb1 : 0u;
            }
        }

        if constexpr (DO_COLT) {
            __syncthreads();
            // item t = (column quad qa, 8-row chunk q); the 16 chunks of a
            // column quad are 16 adjacent lanes, so each column's 128 bytes
            // leave as one contiguous run
            const int q = t & 15, qa = t >> 4;
            const RowBlock &rb = srb[q >> 2];
            if (!rb.skip) {
                uint32_t wv[8];
#pragma unroll
                for (int i = 0; i < 8; i++) wv[i] = tileT[gt_word(q * 8 + i, qa)];
                // 8 rows x 4 columns of bytes -> 4 columns x 8 rows
                const uint32_t a01l = __byte_perm(wv[0], wv[1], 0x5140), a01h = __byte_perm(wv[0], wv[1], 0x7362);
                const uint32_t a23l = __byte_perm(wv[2], wv[3], 0x5140), a23h = __byte_perm(wv[2], wv[3], 0x7362);
                const uint32_t a45l = __byte_perm(wv[4], wv[5], 0x5140), a45h = __byte_perm(wv[4], wv[5], 0x7362);
                const uint32_t a67l = __byte_perm(wv[6], wv[7], 0x5140), a67h = __byte_perm(wv[6], wv[7], 0x7362);
                uint2 o[4];
                o[0] = make_uint2(__byte_perm(a01l, a23l, 0x5410), __byte_perm(a45l, a67l, 0x5410));
                o[1] = make_uint2(__byte_perm(a01l, a23l, 0x7632), __byte_perm(a45l, a67l, 0x7632));
                o[2] = make_uint2(__byte_perm(a01h, a23h, 0x5410), __byte_perm(a45h, a67h, 0x5410));
                o[3] = make_uint2(__byte_perm(a01h, a23h, 0x7632), __byte_perm(a45h, a67h, 0x7632));
                // grouped blocks always write their full 32-byte padded extent
#pragma unroll
                for (int jj = 0; jj < 4; jj++) {
                    const int64_t c = c0 + qa * 4 + jj;
                    if (c < a.cols)
                        *reinterpret_cast<uint2 *>(a.q_colT + c * a.ld_colT + rb.out_col0 + (q & 3) * 8) = o[jj];
                }
            }
        }
        __syncthreads();
    }
    if constexpr (DELAYED) block_amax_atomic(fold_absmax(amax_acc), a.amax_out, red);
}

// Zero the ROWWISE amax accumulators (row, column, and the optional tensor
// amax) before the amax pass.
__global__ void clear_amax_kernel(float *row, int64_t n_row, float *col, int64_t n_col, float *tensor)
{
    const int64_t total = n_row + n_col;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        if (i < n_row)
            row[i] = 0.0f;
        else
            col[i - n_row] = 0.0f;
    }
    if (tensor && blockIdx.x == 0 && threadIdx.x == 0) tensor[0] = 0.0f;
}

// ROWWISE scale buffers, in place: mode 0 turns the accumulated amax into
// the scale (before the cast pass), mode 1 turns the scale into scale_inv =
// 1 / scale (after it), mode 2 turns the amax into scale_inv directly.
__global__ void scales_kernel(float *sinv_row, int64_t n_row, float *sinv_col, int64_t n_col, float fmax, int margin,
                              int mode)
{
    const int64_t total = n_row + n_col;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        float *p = i < n_row ? sinv_row + i : sinv_col + (i - n_row);
        const float v = *p;
        *p = mode == 0 ? scale_from_amax(v, fmax, margin)
                       : (mode == 1 ? recip_rn(v) : recip_rn(scale_from_amax(v, fmax, margin)));
    }
}

// ---------------------------------------------------------------------------
// The ROWWISE recipe on a plain tensor in one cooperative launch: zero the
// amax accumulators, amax pass, cast pass, scale_inv; grid-wide barriers in
// between.  For a tensor that fits in L2 the cast pass re-reads x from L2,
// and the whole quantize is one launch instead of six (three clears, two
// passes, the scale conversion).
//
// The barrier counters are the kernel's only scratch memory, and they live
// in a file-scope device array instead of an allocation: RESIDENT_SLOTS
// counters, 128 bytes apart (8 KB in all, held by every device that loads
// the library until the process exits).  Each call takes the next slot in
// turn, clears that slot's counter on its stream before the launch (the
// array keeps whatever the previous user of the slot left), and barrier k
// completes when the counter reaches k * gridDim.x.  A call uses one counter
// whatever the tensor size.  Calls that overlap on the GPU use different
// counters while fewer than RESIDENT_SLOTS are in flight; past that, two
// in-flight calls share a counter and race.  Every block of a cooperative
// launch is resident, so every block reaches every barrier; the wait is
// still bounded and records ERR_GRID_WAIT if it gives up.
// ---------------------------------------------------------------------------
constexpr int RESIDENT_SLOTS = 64;
constexpr int RESIDENT_SLOT_WORDS = 32;  // 128 bytes per counter
static __device__ __align__(256) unsigned int g_resident_scratch[RESIDENT_SLOTS * RESIDENT_SLOT_WORDS];

constexpr uint64_t GRID_WAIT_LIMIT_NS = 2000000000ull;

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ bool grid_sync(unsigned int *count, unsigned int k, unsigned int *err)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(count, 1u);
        const unsigned int target = k * gridDim.x;
        const uint64_t t0 = global_timer_ns();
        int ok = 1;
        for (uint32_t it = 0; ld_acquire_gpu(count) < target; ++it) {
            if ((it & 255u) == 255u && global_timer_ns() - t0 > GRID_WAIT_LIMIT_NS) {
                record_error(err, ERR_GRID_WAIT);
                ok = 0;
                break;
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

template <int FMT, bool DO_ROW, bool DO_COLT>
__global__ void __launch_bounds__(QT_THREADS, 4)
    rowwise_resident_kernel(QArgs a, int64_t tiles_per_block, unsigned int *count)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    const int64_t n_row = DO_ROW ? a.rows : 0, n_col = DO_COLT ? a.cols : 0;
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = i0; i < n_row + n_col; i += stride) {
        if (i < n_row)
            a.sinv_row[i] = 0.0f;
        else
            a.sinv_col[i - n_row] = 0.0f;
    }
    if (i0 == 0 && a.amax_out) a.amax_out[0] = 0.0f;
    if (!grid_sync(count, 1, a.err)) return;

    const int64_t n_tiles = a.n_row_blocks * a.n_col_chunks;
    const int64_t first = (int64_t)blockIdx.x * tiles_per_block;
    const int64_t last = first + tiles_per_block < n_tiles ? first + tiles_per_block : n_tiles;
    dense_rowcol_amax_run<64, true>(a, first, last);
    if (!grid_sync(count, 2, a.err)) return;

    // the cast pass walks the block's own run backwards: the tiles the amax
    // pass read last are the likeliest to still be in L2
    cast_run<FMT, 64, 1, false, DO_ROW, DO_COLT, true>(a, dsm, first, last - 1);
    if (!grid_sync(count, 3, a.err)) return;

    const float fmax = fp8_max_of(FMT);
    for (int64_t i = i0; i < n_row + n_col; i += stride) {
        float *p = i < n_row ? a.sinv_row + i : a.sinv_col + (i - n_row);
        *p = recip_rn(scale_from_amax(*p, fmax, a.margin));
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Grid size.  Ungrouped tensors get one thread block per tile, so the
// hardware block scheduler balances the tail at tile granularity (measured
// faster on GB300 than a persistent grid of a few blocks per SM, which leaves
// a partial last round).  Grouped tensors keep a persistent grid because
// every block first builds the padded-offset table of all groups.
template <typename K>
static int blocks_for(K kernel, size_t dyn_smem, int64_t n_tiles, bool persistent)
{
    if (!persistent) return (int)(n_tiles < 1 ? 1 : (n_tiles < INT32_MAX ? n_tiles : INT32_MAX));
    int per_sm = 0;
    if (dyn_smem > 48 * 1024) cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_smem);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, QT_THREADS, dyn_smem);
    if (per_sm < 1) per_sm = 1;
    int64_t g = (int64_t)num_sms() * per_sm;
    if (n_tiles < g) g = n_tiles;
    if (g < 1) g = 1;
    return (int)g;
}

template <int FMT, int SMODE, bool DELAYED, int PRO = QPRO_NONE>
static fp8_status_t launch_grouped_cast(const QArgs &a, int layouts, size_t group_smem, cudaStream_t st)
{
    const int64_t n_tiles = (a.n_row_blocks + GT_BLOCKS - 1) / GT_BLOCKS * ((a.cols + GT_COLS - 1) / GT_COLS);
    if (layouts == (FP8_LAYOUT_ROW | FP8_LAYOUT_COLT)) {
        auto k = grouped_cast_kernel<FMT, SMODE, DELAYED, true, true, PRO>;
        k<<<blocks_for(k, group_smem, n_tiles, true), QT_THREADS, group_smem, st>>>(a);
    } else if (layouts == FP8_LAYOUT_ROW) {
        auto k = grouped_cast_kernel<FMT, SMODE, DELAYED, true, false, PRO>;
        k<<<blocks_for(k, group_smem, n_tiles, true), QT_THREADS, group_smem, st>>>(a);
    } else {
        auto k = grouped_cast_kernel<FMT, SMODE, DELAYED, false, true, PRO>;
        k<<<blocks_for(k, group_smem, n_tiles, true), QT_THREADS, group_smem, st>>>(a);
    }
    return check_launch();
}

template <int FMT, int RB, int SMODE, bool DELAYED, int PRO = QPRO_NONE>
static fp8_status_t launch_cast(const QArgs &a, int layouts, size_t group_smem, cudaStream_t st)
{
    if (a.offsets) return launch_grouped_cast<FMT, SMODE, DELAYED, PRO>(a, layouts, group_smem, st);
    if constexpr (RB == 32) {
        return FP8_ERR_INVALID_ARG;  // 32-row blocks are the grouped layout's; plain tensors use 64
    } else {
    const int64_t n_tiles = a.n_row_blocks * a.n_col_chunks;
    const size_t smem = (size_t)RB * QT_PITCH + group_smem;
    if (layouts == (FP8_LAYOUT_ROW | FP8_LAYOUT_COLT)) {
        auto k = cast_kernel<FMT, RB, SMODE, DELAYED, true, true>;
        k<<<blocks_for(k, smem, n_tiles, a.offsets != nullptr), QT_THREADS, smem, st>>>(a);
    } else if (layouts == FP8_LAYOUT_ROW) {
        auto k = cast_kernel<FMT, RB, SMODE, DELAYED, true, false>;
        k<<<blocks_for(k, smem, n_tiles, a.offsets != nullptr), QT_THREADS, smem, st>>>(a);
    } else {
        auto k = cast_kernel<FMT, RB, SMODE, DELAYED, false, true>;
        k<<<blocks_for(k, smem, n_tiles, a.offsets != nullptr), QT_THREADS, smem, st>>>(a);
    }
    return check_launch();
    }
}

template <int FMT, int RB, int PRO = QPRO_NONE>
static fp8_status_t run_quantize(QArgs a, int kind, int layouts, cudaStream_t st)
{
    const size_t group_smem = a.offsets ? 2 * sizeof(int32_t) * (size_t)(a.G + 1) : 0;  // poff + offsets
    const int64_t n_tiles = a.n_row_blocks * a.n_col_chunks;
    fp8_status_t s;
    if (kind == FP8_RECIPE_DELAYED) {
        return launch_cast<FMT, RB, 0, true>(a, layouts, group_smem, st);
    }
    if (kind == FP8_RECIPE_TENSORWISE) {
        if (cudaMemsetAsync(a.amax_out, 0, sizeof(float), st) != cudaSuccess) return cuda_fail();
        auto k = amax_kernel<RB, 0>;
        k<<<blocks_for(k, group_smem, n_tiles, a.offsets != nullptr), QT_THREADS, group_smem, st>>>(a);
        if ((s = check_launch()) != FP8_OK) return s;
        return launch_cast<FMT, RB, 0, false>(a, layouts, group_smem, st);
    }
    // ROWWISE
    const int64_t n_row = (layouts & FP8_LAYOUT_ROW) ? a.rows : 0;
    const int64_t n_col = (layouts & FP8_LAYOUT_COLT) ? a.cols * (a.offsets || a.group_rows ? a.G : 1) : 0;
    if (!(layouts & FP8_LAYOUT_ROW)) a.sinv_row = nullptr;
    if (!(layouts & FP8_LAYOUT_COLT)) a.sinv_col = nullptr;
    // the amax accumulators start at zero: one launch clears all three
    {
        const int64_t n = n_row + n_col + (a.amax_out ? 1 : 0);
        const int zgrid = (int)((n + 255) / 256 < 1024 ? ((n + 255) / 256 > 0 ? (n + 255) / 256 : 1) : 1024);
        clear_amax_kernel<<<zgrid, 256, 0, st>>>(a.sinv_row, n_row, a.sinv_col, n_col, a.amax_out);
        if ((s = check_launch()) != FP8_OK) return s;
    }
    if (!a.offsets) {
        auto k = dense_rowcol_amax_kernel<RB>;
        const int64_t grid = blocks_for(k, 0, n_tiles, true);
        k<<<(unsigned)grid, QT_THREADS, 0, st>>>(a, (n_tiles + grid - 1) / grid);
        if ((s = check_launch()) != FP8_OK) return s;
    } else {
        // pass 1 works on 32-row blocks for both layouts of the row space
        QArgs b = a;
        b.n_row_blocks = a.offsets ? a.n_row_blocks * RB / 32 : (a.rows + 31) / 32;
        // the largest super tile that still gives about 6 blocks per SM
        const int64_t target = 6LL * num_sms();
        b.sup_blocks = SUP_BLOCKS;
        b.sup_chunks = SUP_CHUNKS;
        auto n_super_of = [&](const QArgs &q) {
            return ((q.n_row_blocks + q.sup_blocks - 1) / q.sup_blocks) *
                   ((q.n_col_chunks + q.sup_chunks - 1) / q.sup_chunks);
        };
        while (n_super_of(b) < target && (b.sup_blocks > 1 || b.sup_chunks > 1)) {
            if (b.sup_chunks > 2 || b.sup_blocks == 1)
                b.sup_chunks /= 2;
            else
                b.sup_blocks /= 2;
        }
        const int64_t n_super = n_super_of(b);
        rowcol_amax_kernel<PRO><<<(unsigned)(n_super < 1 ? 1 : (n_super < INT32_MAX ? n_super : INT32_MAX)), QT_THREADS,
                             group_smem, st>>>(b);
        if ((s = check_launch()) != FP8_OK) return s;
    }
    const int64_t total = n_row + n_col;
    const int sgrid = (int)((total + 255) / 256 < 4096 ? ((total + 255) / 256 > 0 ? (total + 255) / 256 : 1) : 4096);
    // grouped tensors: turn the amaxes into scales once (a grouped tile is
    // small, so per-tile divisions would cost more than one extra launch);
    // plain tensors: the cast pass divides per tile and saves the launch
    a.scales_ready = a.offsets != nullptr;
    if (a.scales_ready && total > 0) {
        scales_kernel<<<sgrid, 256, 0, st>>>(a.sinv_row, n_row, a.sinv_col, n_col, fp8_max_of(FMT), a.margin, 0);
        if ((s = check_launch()) != FP8_OK) return s;
    }
    if ((s = launch_cast<FMT, RB, 1, false, PRO>(a, layouts, group_smem, st)) != FP8_OK) return s;
    if (total > 0) {
        scales_kernel<<<sgrid, 256, 0, st>>>(a.sinv_row, n_row, a.sinv_col, n_col, fp8_max_of(FMT), a.margin,
                                             a.scales_ready ? 1 : 2);
        return check_launch();
    }
    return FP8_OK;
}

}  // namespace fp8gb

using namespace fp8gb;

extern "C" fp8_status_t fp8_quantize(const void *x_bf16, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                                     const fp8_recipe_t *recipe, int layouts, const float *scale_in,
                                     float *amax_out, uint8_t *q_row, float *scale_inv_row, uint8_t *q_colT,
                                     int64_t ld_colT, float *scale_inv_col, const int32_t *group_offsets,
                                     int num_groups, void *stream)
{
    // ---- validation (host only; nothing is launched on failure) ----
    if (!recipe || (!x_bf16 && rows > 0)) return FP8_ERR_INVALID_ARG;
    if (rows < 0 || cols < 1 || ld_x < cols) return FP8_ERR_INVALID_ARG;
    if (fmt != FP8_E4M3FN && fmt != FP8_E5M2 && fmt != FP8_E4M3FNUZ && fmt != FP8_E5M2FNUZ)
        return FP8_ERR_INVALID_ARG;
    if (recipe->kind < FP8_RECIPE_DELAYED || recipe->kind > FP8_RECIPE_ROWWISE) return FP8_ERR_INVALID_ARG;
    if (recipe->margin < 0 || recipe->margin > 64) return FP8_ERR_INVALID_ARG;
    if (layouts < 1 || layouts > 3) return FP8_ERR_INVALID_ARG;
    // an empty tensor may come with empty (NULL) row-layout buffers
    if ((layouts & FP8_LAYOUT_ROW) && rows > 0 && (!q_row || !scale_inv_row)) return FP8_ERR_INVALID_ARG;
    if ((layouts & FP8_LAYOUT_ROW) && recipe->kind != FP8_RECIPE_ROWWISE && !scale_inv_row)
        return FP8_ERR_INVALID_ARG;
    if ((layouts & FP8_LAYOUT_COLT) && (!q_colT || !scale_inv_col)) return FP8_ERR_INVALID_ARG;
    if (recipe->kind == FP8_RECIPE_DELAYED && (!scale_in || !amax_out)) return FP8_ERR_INVALID_ARG;
    if (recipe->kind == FP8_RECIPE_TENSORWISE && !amax_out) return FP8_ERR_INVALID_ARG;
    if (group_offsets && (num_groups < 1 || num_groups > QT_MAX_GROUPS)) return FP8_ERR_INVALID_ARG;
    // equal groups without offsets: num_groups groups of rows / num_groups rows, a multiple of 64
    if (!group_offsets && (num_groups < 0 || num_groups > QT_MAX_GROUPS)) return FP8_ERR_INVALID_ARG;
    if (!group_offsets && num_groups > 0 && (rows % num_groups != 0 || (rows / num_groups) % 64 != 0))
        return FP8_ERR_INVALID_ARG;
    if (cols % 8 != 0 || ld_x % 8 != 0 || !aligned(x_bf16, 16)) return FP8_ERR_ALIGNMENT;
    if ((layouts & FP8_LAYOUT_ROW) && !aligned(q_row, 8)) return FP8_ERR_ALIGNMENT;
    if (layouts & FP8_LAYOUT_COLT) {
        if (!aligned(q_colT, 16) || ld_colT % 16 != 0) return FP8_ERR_ALIGNMENT;
        if (!group_offsets && ld_colT < rows) return FP8_ERR_INVALID_ARG;
        if (group_offsets && ld_colT < rows) return FP8_ERR_INVALID_ARG;  // padded width is >= rows
    }
    if (rows > ((int64_t)1 << 40) || cols > ((int64_t)1 << 31)) return FP8_ERR_INVALID_ARG;
    // grouped padded offsets are int32 on the device
    if (group_offsets && (rows + 32LL * num_groups > INT32_MAX || ld_colT > INT32_MAX)) return FP8_ERR_INVALID_ARG;

    QArgs a{};
    a.x = static_cast<const uint16_t *>(x_bf16);
    a.rows = rows;
    a.cols = cols;
    a.ld_x = ld_x;
    a.q_row = q_row;
    a.q_colT = q_colT;
    a.ld_colT = (layouts & FP8_LAYOUT_COLT) ? ld_colT : 0;
    a.sinv_row = scale_inv_row;
    a.sinv_col = scale_inv_col;
    a.scale_in = scale_in;
    a.amax_out = amax_out;
    a.offsets = group_offsets;
    a.err = device_error_word();
    a.G = num_groups;
    a.group_rows = !group_offsets && num_groups > 0 ? rows / num_groups : 0;
    a.margin = recipe->margin;
    a.n_col_chunks = (cols + QT_COLS - 1) / QT_COLS;
    a.scales_ready = 0;
    a.sup_blocks = SUP_BLOCKS;
    a.sup_chunks = SUP_CHUNKS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (group_offsets) {
        // padded space: rows + at most 31 padding rows per group
        const int64_t padded_max = ld_colT > 0 && (layouts & FP8_LAYOUT_COLT) ? ld_colT : rows + 32LL * num_groups;
        a.n_row_blocks = (padded_max + 31) / 32;
        if (fmt == FP8_E5M2) return run_quantize<FP8_E5M2, 32>(a, recipe->kind, layouts, st);
        if (fmt == FP8_E4M3FNUZ) return run_quantize<FP8_E4M3FNUZ, 32>(a, recipe->kind, layouts, st);
        if (fmt == FP8_E5M2FNUZ) return run_quantize<FP8_E5M2FNUZ, 32>(a, recipe->kind, layouts, st);
        return run_quantize<FP8_E4M3FN, 32>(a, recipe->kind, layouts, st);
    }
    a.n_row_blocks = (rows + 63) / 64;
    if (fmt == FP8_E5M2) return run_quantize<FP8_E5M2, 64>(a, recipe->kind, layouts, st);
    if (fmt == FP8_E4M3FNUZ) return run_quantize<FP8_E4M3FNUZ, 64>(a, recipe->kind, layouts, st);
    if (fmt == FP8_E5M2FNUZ) return run_quantize<FP8_E5M2FNUZ, 64>(a, recipe->kind, layouts, st);
    return run_quantize<FP8_E4M3FN, 64>(a, recipe->kind, layouts, st);
}

namespace fp8gb {

// Device address of g_resident_scratch on the current device.  In host code
// the array's name denotes a host-side stand-in, not device memory, so the
// address is looked up with cudaGetSymbolAddress: once per device, by the
// first call made while that device is current, and kept for later calls.
constexpr int RESIDENT_MAX_DEVICES = 64;
static std::mutex g_resident_mu;
static unsigned int *g_resident_ptr[RESIDENT_MAX_DEVICES];

static unsigned int *resident_scratch(cudaError_t *e)
{
    int dev = 0;
    if ((*e = cudaGetDevice(&dev)) != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= RESIDENT_MAX_DEVICES) {
        *e = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_resident_mu);
    if (!g_resident_ptr[dev]) {
        void *p = nullptr;
        if ((*e = cudaGetSymbolAddress(&p, g_resident_scratch)) != cudaSuccess) {
            cudaGetLastError();  // not sticky: clear it so later launch checks do not see it
            return nullptr;
        }
        g_resident_ptr[dev] = static_cast<unsigned int *>(p);
    }
    *e = cudaSuccess;
    return g_resident_ptr[dev];
}

template <int FMT, bool DO_ROW, bool DO_COLT>
static fp8_status_t launch_resident(QArgs a, cudaStream_t st)
{
    auto k = rowwise_resident_kernel<FMT, DO_ROW, DO_COLT>;
    const size_t smem = (size_t)64 * QT_PITCH;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, QT_THREADS, smem) != cudaSuccess || per_sm < 1)
        return cuda_fail();
    const int64_t n_tiles = a.n_row_blocks * a.n_col_chunks;
    int64_t grid = (int64_t)num_sms() * per_sm;
    if (grid > n_tiles) grid = n_tiles;
    if (grid < 1) grid = 1;
    int64_t tiles_per_block = (n_tiles + grid - 1) / grid;
    cudaError_t se = cudaSuccess;
    unsigned int *scratch = resident_scratch(&se);
    if (!scratch) return cuda_fail_with(se);
    static std::atomic<unsigned int> next_slot{0};
    unsigned int *count =
        scratch + (size_t)(next_slot.fetch_add(1, std::memory_order_relaxed) % RESIDENT_SLOTS) * RESIDENT_SLOT_WORDS;
    if (cudaMemsetAsync(count, 0, sizeof(unsigned int), st) != cudaSuccess) return cuda_fail();
    void *args[] = {&a, &tiles_per_block, &count};
    const cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(k), dim3((unsigned)grid),
                                                      dim3(QT_THREADS), args, smem, st);
    if (e != cudaSuccess) return cuda_fail_with(e);
    return FP8_OK;
}

template <int FMT>
static fp8_status_t run_resident(const QArgs &a, int layouts, cudaStream_t st)
{
    if (layouts == (FP8_LAYOUT_ROW | FP8_LAYOUT_COLT)) return launch_resident<FMT, true, true>(a, st);
    if (layouts == FP8_LAYOUT_ROW) return launch_resident<FMT, true, false>(a, st);
    return launch_resident<FMT, false, true>(a, st);
}

}  // namespace fp8gb

extern "C" fp8_status_t fp8_quantize_rowwise_resident(const void *x_bf16, int64_t rows, int64_t cols, int64_t ld_x,
                                                      int fmt, int margin, int layouts, float *amax_out,
                                                      uint8_t *q_row, float *scale_inv_row, uint8_t *q_colT,
                                                      int64_t ld_colT, float *scale_inv_col, void *stream)
{
    // ---- validation (host only; nothing is launched on failure) ----
    if (!x_bf16 && rows > 0) return FP8_ERR_INVALID_ARG;
    if (rows < 0 || cols < 1 || ld_x < cols) return FP8_ERR_INVALID_ARG;
    if (fmt != FP8_E4M3FN && fmt != FP8_E5M2 && fmt != FP8_E4M3FNUZ && fmt != FP8_E5M2FNUZ)
        return FP8_ERR_INVALID_ARG;
    if (margin < 0 || margin > 64) return FP8_ERR_INVALID_ARG;
    if (layouts < 1 || layouts > 3) return FP8_ERR_INVALID_ARG;
    if ((layouts & FP8_LAYOUT_ROW) && rows > 0 && (!q_row || !scale_inv_row)) return FP8_ERR_INVALID_ARG;
    if ((layouts & FP8_LAYOUT_COLT) && (!q_colT || !scale_inv_col)) return FP8_ERR_INVALID_ARG;
    if (cols % 8 != 0 || ld_x % 8 != 0 || !aligned(x_bf16, 16)) return FP8_ERR_ALIGNMENT;
    if ((layouts & FP8_LAYOUT_ROW) && !aligned(q_row, 8)) return FP8_ERR_ALIGNMENT;
    if (layouts & FP8_LAYOUT_COLT) {
        if (!aligned(q_colT, 16) || ld_colT % 16 != 0) return FP8_ERR_ALIGNMENT;
        if (ld_colT < rows) return FP8_ERR_INVALID_ARG;
    }
    if (rows > ((int64_t)1 << 40) || cols > ((int64_t)1 << 31)) return FP8_ERR_INVALID_ARG;
    // rows == 0 still launches (one block, no tiles): like fp8_quantize it
    // writes scale_inv_col = 1 and amax_out = 0 for an empty tensor

    QArgs a{};
    a.x = static_cast<const uint16_t *>(x_bf16);
    a.rows = rows;
    a.cols = cols;
    a.ld_x = ld_x;
    a.q_row = q_row;
    a.q_colT = q_colT;
    a.ld_colT = (layouts & FP8_LAYOUT_COLT) ? ld_colT : 0;
    a.sinv_row = (layouts & FP8_LAYOUT_ROW) ? scale_inv_row : nullptr;
    a.sinv_col = (layouts & FP8_LAYOUT_COLT) ? scale_inv_col : nullptr;
    a.scale_in = nullptr;
    a.amax_out = amax_out;
    a.offsets = nullptr;
    a.err = device_error_word();
    a.G = 0;
    a.margin = margin;
    a.n_col_chunks = (cols + QT_COLS - 1) / QT_COLS;
    a.n_row_blocks = (rows + 63) / 64;
    a.scales_ready = 0;
    a.sup_blocks = SUP_BLOCKS;
    a.sup_chunks = SUP_CHUNKS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (fmt == FP8_E5M2) return run_resident<FP8_E5M2>(a, layouts, st);
    if (fmt == FP8_E4M3FNUZ) return run_resident<FP8_E4M3FNUZ>(a, layouts, st);
    if (fmt == FP8_E5M2FNUZ) return run_resident<FP8_E5M2FNUZ>(a, layouts, st);
    return run_resident<FP8_E4M3FN>(a, layouts, st);
}

// ---------------------------------------------------------------------------
// Fused MoE prologues of the ROWWISE recipe (grouped tensors): the gather of
// routed token rows into expert order, and SwiGLU of the gate|up projection
// output, applied by both grouped passes to what they read.
// ---------------------------------------------------------------------------
static fp8_status_t prologue_args(QArgs &a, int fmt, int margin, int layouts, uint8_t *q_row, float *scale_inv_row,
                                  uint8_t *q_colT, int64_t ld_colT, float *scale_inv_col, const int32_t *group_offsets,
                                  int num_groups)
{
    const int64_t rows = a.rows, cols = a.cols;
    if (rows < 0 || cols < 1) return FP8_ERR_INVALID_ARG;
    if (fmt != FP8_E4M3FN && fmt != FP8_E5M2 && fmt != FP8_E4M3FNUZ && fmt != FP8_E5M2FNUZ)
        return FP8_ERR_INVALID_ARG;
    if (margin < 0 || margin > 64) return FP8_ERR_INVALID_ARG;
    if (layouts < 1 || layouts > 3) return FP8_ERR_INVALID_ARG;
    if (!group_offsets || num_groups < 1 || num_groups > QT_MAX_GROUPS) return FP8_ERR_INVALID_ARG;
    if ((layouts & FP8_LAYOUT_ROW) && rows > 0 && (!q_row || !scale_inv_row)) return FP8_ERR_INVALID_ARG;
    if ((layouts & FP8_LAYOUT_COLT) && (!q_colT || !scale_inv_col)) return FP8_ERR_INVALID_ARG;
    if (rows > 0 && !a.x) return FP8_ERR_INVALID_ARG;
    if (cols % 8 != 0 || a.ld_x % 8 != 0 || !aligned(a.x, 16)) return FP8_ERR_ALIGNMENT;
    if ((layouts & FP8_LAYOUT_ROW) && !aligned(q_row, 8)) return FP8_ERR_ALIGNMENT;
    if (layouts & FP8_LAYOUT_COLT) {
        if (!aligned(q_colT, 16) || ld_colT % 16 != 0) return FP8_ERR_ALIGNMENT;
        if (ld_colT < rows) return FP8_ERR_INVALID_ARG;
    }
    if (cols > ((int64_t)1 << 31) || rows + 32LL * num_groups > INT32_MAX || ld_colT > INT32_MAX)
        return FP8_ERR_INVALID_ARG;
    a.q_row = q_row;
    a.q_colT = q_colT;
    a.ld_colT = (layouts & FP8_LAYOUT_COLT) ? ld_colT : 0;
    a.sinv_row = scale_inv_row;
    a.sinv_col = scale_inv_col;
    a.offsets = group_offsets;
    a.G = num_groups;
    a.margin = margin;
    a.err = device_error_word();
    a.n_col_chunks = (cols + QT_COLS - 1) / QT_COLS;
    a.scales_ready = 0;
    a.sup_blocks = SUP_BLOCKS;
    a.sup_chunks = SUP_CHUNKS;
    // padded space: rows + at most 31 padding rows per group
    const int64_t padded_max = (layouts & FP8_LAYOUT_COLT) ? ld_colT : rows + 32LL * num_groups;
    a.n_row_blocks = (padded_max + 31) / 32;
    return FP8_OK;
}

template <int PRO>
static fp8_status_t run_prologue(const QArgs &a, int fmt, int layouts, cudaStream_t st)
{
    if (fmt == FP8_E5M2) return run_quantize<FP8_E5M2, 32, PRO>(a, FP8_RECIPE_ROWWISE, layouts, st);
    if (fmt == FP8_E4M3FNUZ) return run_quantize<FP8_E4M3FNUZ, 32, PRO>(a, FP8_RECIPE_ROWWISE, layouts, st);
    if (fmt == FP8_E5M2FNUZ) return run_quantize<FP8_E5M2FNUZ, 32, PRO>(a, FP8_RECIPE_ROWWISE, layouts, st);
    return run_quantize<FP8_E4M3FN, 32, PRO>(a, FP8_RECIPE_ROWWISE, layouts, st);
}

extern "C" fp8_status_t fp8_permute_quantize(const void *x_bf16, int64_t x_rows, int64_t cols, int64_t ld_x,
                                             const int32_t *src_rows, int64_t rows, int fmt, int margin, int layouts,
                                             float *amax_out, uint8_t *q_row, float *scale_inv_row, uint8_t *q_colT,
                                             int64_t ld_colT, float *scale_inv_col, const int32_t *group_offsets,
                                             int num_groups, void *stream)
{
    if (x_rows < 0 || ld_x < cols) return FP8_ERR_INVALID_ARG;
    if (rows > 0 && (!src_rows || x_rows < 1)) return FP8_ERR_INVALID_ARG;
    QArgs a{};
    a.x = static_cast<const uint16_t *>(x_bf16);
    a.rows = rows;
    a.cols = cols;
    a.ld_x = ld_x;
    a.amax_out = amax_out;
    a.src_rows = src_rows;
    a.x_rows = x_rows;
    const fp8_status_t s = prologue_args(a, fmt, margin, layouts, q_row, scale_inv_row, q_colT, ld_colT,
                                         scale_inv_col, group_offsets, num_groups);
    if (s != FP8_OK) return s;
    return run_prologue<QPRO_GATHER>(a, fmt, layouts, static_cast<cudaStream_t>(stream));
}

extern "C" fp8_status_t fp8_swiglu_quantize(const void *gate_up_bf16, int64_t rows, int64_t F, int64_t ld, int fmt,
                                            int margin, int layouts, void *h_bf16, int64_t ld_h, float *amax_out,
                                            uint8_t *q_row, float *scale_inv_row, uint8_t *q_colT, int64_t ld_colT,
                                            float *scale_inv_col, const int32_t *group_offsets, int num_groups,
                                            void *stream)
{
    if (F < 1 || ld < 2 * F) return FP8_ERR_INVALID_ARG;
    if (h_bf16 && ld_h < F) return FP8_ERR_INVALID_ARG;
    if (h_bf16 && (ld_h % 8 != 0 || !aligned(h_bf16, 16))) return FP8_ERR_ALIGNMENT;
    QArgs a{};
    a.x = static_cast<const uint16_t *>(gate_up_bf16);
    a.rows = rows;
    a.cols = F;
    a.ld_x = ld;
    a.amax_out = amax_out;
    a.up_off = F;
    a.h_out = static_cast<uint16_t *>(h_bf16);
    a.ld_h = ld_h;
    const fp8_status_t s = prologue_args(a, fmt, margin, layouts, q_row, scale_inv_row, q_colT, ld_colT,
                                         scale_inv_col, group_offsets, num_groups);
    if (s != FP8_OK) return s;
    return run_prologue<QPRO_SWIGLU>(a, fmt, layouts, static_cast<cudaStream_t>(stream));
}
