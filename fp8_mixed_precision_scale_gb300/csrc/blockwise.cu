// blockwise.cu -- blockwise FP8 quantize: 1 x 128 blocks along the
// contraction for activations and gradients, 128 x 128 blocks for weights,
// one power-of-two scale per block, row and transposed layouts from one read.
//
// Method: the "blockwise" recipe listed on "FP8 training for Flux models"
// (Configuration > Key FP8 Parameters), which the page names without a
// definition.  Each block takes the largest power-of-two scale s with
// amax * s <= fp8_max (amax 0 or non-finite: s = 1), q = sat_rne(v * s); the
// dequantisation factor 1/s is an exact E8M0 value, written into the MX
// scale layout (each 128-block's code in its four 32-element slots), so the
// block-scaled tensor-core GEMM (fp8_mx_gemm) applies it unchanged.
//
// Design (GB300): persistent 512-thread blocks (two per SM) looping over
// 128 x 128 tiles; each block issues the next tile's loads before working on
// the current one, so loads stay in flight while it converts.  Four threads
// own a row (32 columns each: 64 bytes, whole 32-byte sectors); the 1 x 128
// block maximum is shared by two shuffles, weights reduce the whole tile
// through shared memory; each thread writes its 32 row-layout codes with one
// 32-byte store (two 16-byte halves took 15 % longer on a [8192, 14336]
// gradient).  The tile is staged in shared memory as column-pair
// words, XOR-swizzled by the row's 16-row group; for the transposed layout
// eight threads own a column pair's eight 16-row slices, combine their maxima
// by three shuffles and write 16 contiguous bytes per column (128 per column
// and tile).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8gb.h"
#include "fp8gb_device.cuh"
#include "fp8gb_host.h"

namespace fp8gb {

constexpr int BW_THREADS = 512;
constexpr int BW_TILE = 128;
constexpr int BW_PITCH_W = BW_TILE / 2 + 8;  // 32-bit words per shared row: 64 column pairs + two 4-word pads

struct BwArgs {
    const uint16_t *x;
    int64_t rows, cols, ld_x;
    uint8_t *q_row, *s_row, *q_colT, *s_col;
    int64_t ld_colT;
    int64_t rs_row;  // scale rows of s_row (rows rounded up to 128)
    int64_t n_row_tiles, n_col_tiles;
    int do_row, do_col;
    int ld32;  // every row's 32-column slice starts on a 32-byte boundary
    int st32;  // q_row is 32-byte aligned (so is every thread's 32-byte slice of it)
};

// E8M0 code of 1/s for a block whose largest magnitude has fp32 bits
// amax_bits: s = 2^e with e the largest integer such that amax * 2^e <=
// fp8_max = 1.75 * 2^EF.  For a normal amax = m * 2^E (1 <= m < 2) that is
// e = EF - E, one less when m > 1.75; subnormal maxima clamp to e = 127.
template <int FMT>
__device__ __forceinline__ uint32_t bw_code(uint32_t amax_bits)
{
    constexpr int EF = FMT == FP8_E5M2 ? 15 : 8;
    if (amax_bits >= 0x7F800000u || amax_bits == 0u) return 127u;  // non-finite or zero block: s = 1
    if (amax_bits < 0x00800000u) return 0u;                        // subnormal maximum: e clamps to 127
    int e = EF - ((int)(amax_bits >> 23) - 127) - ((amax_bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
    return (uint32_t)(127 - e);
}

__device__ __forceinline__ float bw_scale(uint32_t code)  // s = 2^(127 - code), code <= 254
{
    return __uint_as_float((254u - code) << 23);
}

// Shared tile word of (row, column pair).  The pair index is XORed with 4 x
// the row's 16-row group, rows are 72 words apart (8 banks mod 32) and a
// 4-word gap follows the first 32 pairs of a row: each quarter warp of the
// row phase's 16-byte stores (two rows x four 32-column slices) reaches all
// 32 banks, and so does each warp of the transposed phase's word reads
// (eight 16-row slices x four column pairs).
__device__ __forceinline__ int bw_word(int row, int pair)
{
    const int pp = pair ^ (((row >> 4) & 7) << 2);
    return row * BW_PITCH_W + pp + 4 * (pp >> 5);
}

// 32 bytes (16 bf16) from a 32-byte-aligned address through the read-only
// path, as two 16-byte halves
__device__ __forceinline__ void bw_ld_32b(const uint16_t *p, uint4 &lo, uint4 &hi)
{
    asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
                 : "l"(p));
}

// 32 bytes to a 32-byte-aligned address
__device__ __forceinline__ void bw_st_32b(void *p, const uint32_t (&o)[8])
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(o[0]), "r"(o[1]),
                 "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                 : "memory");
}

// Thread (lr, q) = (tid / 4, tid % 4): row lr of tile (rt, ct), columns 32 q ..
// 32 q + 31 (zeros past the rows).
__device__ __forceinline__ void bw_load(const BwArgs &a, uint32_t rt, uint32_t ct, int lr, int q, uint4 (&v)[4])
{
    const int64_t r = (int64_t)rt * BW_TILE + lr;
    if (r < a.rows) {
        const uint16_t *src = a.x + r * a.ld_x + (int64_t)ct * BW_TILE + 32 * q;
        if (a.ld32) {
            bw_ld_32b(src, v[0], v[1]);
            bw_ld_32b(src + 16, v[2], v[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; j++) v[j] = __ldg(reinterpret_cast<const uint4 *>(src) + j);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; j++) v[j] = make_uint4(0, 0, 0, 0);
    }
}

template <int FMT, bool WEIGHT>
__global__ void __launch_bounds__(BW_THREADS, 2)
    bw_quantize_kernel(BwArgs a)
{
    __shared__ __align__(16) uint32_t tile[BW_TILE * BW_PITCH_W];
    __shared__ uint32_t warp_max[BW_THREADS / 32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lr = tid >> 2, q = tid & 3;  // row phase: row lr, columns 32 q .. 32 q + 31
    const int sl = tid & 7, p = tid >> 3;  // transposed phase: column pair p, rows 16 sl .. 16 sl + 15
    // tile indexes fit 32 bits (the host checks the tile count)
    const uint32_t total = (uint32_t)(a.n_row_tiles * a.n_col_tiles), nct = (uint32_t)a.n_col_tiles;
    const bool staged = a.do_col || WEIGHT;

    uint32_t t = blockIdx.x;
    uint32_t nrt = t / nct, nct_ = t - nrt * nct;  // coordinates of the tile being prefetched
    uint4 nv[4];
    if (t < total) bw_load(a, nrt, nct_, lr, q, nv);
    for (; t < total; t += gridDim.x) {
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; j++) v[j] = nv[j];
        const uint32_t rt = nrt, ct = nct_;
        if (t + gridDim.x < total) {
            nrt = (t + gridDim.x) / nct;
            nct_ = t + gridDim.x - nrt * nct;
            bw_load(a, nrt, nct_, lr, q, nv);
        }
        const int64_t r0 = (int64_t)rt * BW_TILE, c0 = (int64_t)ct * BW_TILE;
        const bool row_real = r0 + lr < a.rows;

        uint32_t am = 0;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            am = absmax_bf16x2(am, v[j].x);
            am = absmax_bf16x2(am, v[j].y);
            am = absmax_bf16x2(am, v[j].z);
            am = absmax_bf16x2(am, v[j].w);
        }
        uint32_t row_bits = fold_absmax(am);  // the row's 1 x 128 block: lanes 4i .. 4i + 3
        row_bits = max(row_bits, __shfl_xor_sync(0xffffffffu, row_bits, 1));
        row_bits = max(row_bits, __shfl_xor_sync(0xffffffffu, row_bits, 2));
        if constexpr (WEIGHT) {
            uint32_t m = row_bits;
#pragma unroll
            for (int d = 4; d < 32; d <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, d));
            if (lane == 0) warp_max[warp] = m;
        }
        if (staged) {
#pragma unroll
            for (int j = 0; j < 4; j++) *reinterpret_cast<uint4 *>(&tile[bw_word(lr, 16 * q + 4 * j)]) = v[j];
            __syncthreads();
        }
        uint32_t block_code = 0;
        if constexpr (WEIGHT) {
            uint32_t m = warp_max[0];
#pragma unroll
            for (int w = 1; w < BW_THREADS / 32; w++) m = max(m, warp_max[w]);
            block_code = bw_code<FMT>(m);
        }

        // ---- row layout ----
        if (a.do_row) {
            const uint32_t code = WEIGHT ? block_code : bw_code<FMT>(row_bits);
            if (row_real) {
                const float sc = bw_scale(code);
                uint32_t out[8];
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const uint2 b = cvt8_scaled<FMT>(v[j], sc);
                    out[2 * j] = b.x;
                    out[2 * j + 1] = b.y;
                }
                uint8_t *dst = a.q_row + (r0 + lr) * a.cols + c0 + 32 * q;
                if (a.st32) {
                    bw_st_32b(dst, out);
                } else {
                    reinterpret_cast<uint4 *>(dst)[0] = make_uint4(out[0], out[1], out[2], out[3]);
                    reinterpret_cast<uint4 *>(dst)[1] = make_uint4(out[4], out[5], out[6], out[7]);
                }
            }
            // one scale word per row and 128-column tile: the code in all four slots
            if (q == 0 && r0 + lr < a.rs_row)
                *reinterpret_cast<uint32_t *>(a.s_row + mx_scale_word(ct, r0 + lr, a.rs_row) * 4) =
                    row_real ? code * 0x01010101u : 0u;
        }

        // ---- transposed layout ----
        if (a.do_col) {
            uint32_t w[16];
            uint32_t cm = 0;
#pragma unroll
            for (int i = 0; i < 16; i++) {
                w[i] = tile[bw_word(16 * sl + i, p)];
                cm = absmax_bf16x2(cm, w[i]);
            }
            // the column pair's 128-row blocks: lanes 8k .. 8k + 7
            cm = __vmaxu2(cm, __shfl_xor_sync(0xffffffffu, cm, 1));
            cm = __vmaxu2(cm, __shfl_xor_sync(0xffffffffu, cm, 2));
            cm = __vmaxu2(cm, __shfl_xor_sync(0xffffffffu, cm, 4));
            const uint32_t code0 = WEIGHT ? block_code : bw_code<FMT>(cm << 16);
            const uint32_t code1 = WEIGHT ? block_code : bw_code<FMT>(cm & 0xFFFF0000u);
            const float s0 = bw_scale(code0), s1 = bw_scale(code1);
            uint32_t o0[4], o1[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const uint32_t x0 = w[4 * i], x1 = w[4 * i + 1], x2 = w[4 * i + 2], x3 = w[4 * i + 3];
                float a0 = bf16lo(x0), a1 = bf16lo(x1), a2 = bf16lo(x2), a3 = bf16lo(x3);
                float b0 = bf16hi(x0), b1 = bf16hi(x1), b2 = bf16hi(x2), b3 = bf16hi(x3);
                mul2_rn(a0, a1, s0, s0);
                mul2_rn(a2, a3, s0, s0);
                mul2_rn(b0, b1, s1, s1);
                mul2_rn(b2, b3, s1, s1);
                o0[i] = cvt4<FMT>(a0, a1, a2, a3);
                o1[i] = cvt4<FMT>(b0, b1, b2, b3);
            }
            const int64_t c = c0 + 2 * p;
            *reinterpret_cast<uint4 *>(a.q_colT + c * a.ld_colT + r0 + 16 * sl) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
            *reinterpret_cast<uint4 *>(a.q_colT + (c + 1) * a.ld_colT + r0 + 16 * sl) =
                make_uint4(o1[0], o1[1], o1[2], o1[3]);
            if (sl == 0) {  // scale rows c and c + 1 of s_col (cols is a multiple of 128)
                *reinterpret_cast<uint32_t *>(a.s_col + mx_scale_word(rt, c, a.cols) * 4) = code0 * 0x01010101u;
                *reinterpret_cast<uint32_t *>(a.s_col + mx_scale_word(rt, c + 1, a.cols) * 4) = code1 * 0x01010101u;
            }
        }
        if (staged) __syncthreads();  // the tile and the warp maxima are rewritten by the next tile
    }
}

template <int FMT, bool WEIGHT>
static fp8_status_t launch_bw(const BwArgs &a, int64_t n_tiles, cudaStream_t st)
{
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bw_quantize_kernel<FMT, WEIGHT>, BW_THREADS, 0);
    if (per_sm < 1) per_sm = 1;
    const int64_t grid = n_tiles < (int64_t)num_sms() * per_sm ? n_tiles : (int64_t)num_sms() * per_sm;
    bw_quantize_kernel<FMT, WEIGHT><<<(unsigned)grid, BW_THREADS, 0, st>>>(a);
    return check_launch();
}

}  // namespace fp8gb

using namespace fp8gb;

extern "C" fp8_status_t fp8_blockwise_quantize(const void *x_bf16, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                                               int block_rows, int layouts, uint8_t *q_row, uint8_t *s_row,
                                               uint8_t *q_colT, int64_t ld_colT, uint8_t *s_col, void *stream)
{
    if (rows < 0 || cols < 1 || ld_x < cols) return FP8_ERR_INVALID_ARG;
    if (fmt == FP8_E4M3FNUZ || fmt == FP8_E5M2FNUZ) return FP8_ERR_UNSUPPORTED;
    if (fmt != FP8_E4M3FN && fmt != FP8_E5M2) return FP8_ERR_INVALID_ARG;
    if (block_rows != 1 && block_rows != BW_TILE) return FP8_ERR_INVALID_ARG;
    if (layouts < 1 || layouts > 3) return FP8_ERR_INVALID_ARG;
    if (rows == 0) return FP8_OK;
    const bool do_row = layouts & FP8_LAYOUT_ROW, do_col = layouts & FP8_LAYOUT_COLT;
    if (!x_bf16 || (do_row && (!q_row || !s_row)) || (do_col && (!q_colT || !s_col))) return FP8_ERR_INVALID_ARG;
    if (rows > INT32_MAX || cols > INT32_MAX) return FP8_ERR_INVALID_ARG;
    if (cols % BW_TILE != 0 || ld_x % 8 != 0 || !aligned(x_bf16, 16)) return FP8_ERR_ALIGNMENT;
    if ((do_col || block_rows == BW_TILE) && rows % BW_TILE != 0) return FP8_ERR_ALIGNMENT;
    if (do_row && (!aligned(q_row, 16) || !aligned(s_row, 4))) return FP8_ERR_ALIGNMENT;
    if (do_col) {
        if (ld_colT % 16 != 0 || !aligned(q_colT, 16) || !aligned(s_col, 4)) return FP8_ERR_ALIGNMENT;
        if (ld_colT < rows) return FP8_ERR_INVALID_ARG;
    }
    BwArgs a{};
    a.x = static_cast<const uint16_t *>(x_bf16);
    a.rows = rows;
    a.cols = cols;
    a.ld_x = ld_x;
    a.q_row = q_row;
    a.s_row = s_row;
    a.q_colT = q_colT;
    a.s_col = s_col;
    a.ld_colT = ld_colT;
    a.rs_row = round_up_128(rows);
    a.n_row_tiles = a.rs_row / BW_TILE;
    a.n_col_tiles = cols / BW_TILE;
    a.do_row = do_row;
    a.do_col = do_col;
    a.ld32 = aligned(x_bf16, 32) && ld_x % 16 == 0;
    a.st32 = do_row && aligned(q_row, 32);
    const int64_t n_tiles = a.n_row_tiles * a.n_col_tiles;
    if (n_tiles > INT32_MAX) return FP8_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool w = block_rows == BW_TILE;
    if (fmt == FP8_E5M2) return w ? launch_bw<FP8_E5M2, true>(a, n_tiles, st) : launch_bw<FP8_E5M2, false>(a, n_tiles, st);
    return w ? launch_bw<FP8_E4M3FN, true>(a, n_tiles, st) : launch_bw<FP8_E4M3FN, false>(a, n_tiles, st);
}
