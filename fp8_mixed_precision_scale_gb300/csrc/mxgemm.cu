// mxgemm.cu -- MXFP8 GEMM and grouped GEMM on the block-scaled tcgen05
// tensor cores.
//
// C[m][n] = bf16( sum_k A[m][k] X_A(m, k/32) B[n][k] X_B(n, k/32) ): FP8
// E4M3 / E5M2 operands, one E8M0 scale per 32 elements along K for every row
// of A and of B, fp32 accumulation in tensor memory.  The scales are applied
// by the MMA itself (tcgen05.mma kind::mxf8f6f4 block_scale), which reads
// them from tensor memory, so the epilogue only converts to bf16.
//
// Method: the "mxfp8" recipe ("FP8 training for Flux models", Key FP8
// Parameters) and MXFP8 grouped GEMM for MoE ("FP8 Training on AMD GPUs with
// TorchTitan and TorchAO"), with the OCP Microscaling block rule.
//
// Design (GB300, sm_103a): the persistent warp-specialised structure of the
// tensor-scaled GEMM plus a scale-copy warp, 352 threads per CTA, one CTA
// per SM.
//   warp 0     producer: TMA tiles of A (128 x 128 bytes) and B (256 x 128
//              bytes), plus one bulk copy each of the tiles' scale blocks,
//              all counted on one mbarrier per stage of the ring (4 stages
//              dense, 3 grouped and with the TMA-store epilogue).  The MX
//              scale layout stores every 128 scale rows of a K tile as the
//              512-byte block tcgen05.cp 32x128b.warpx4 reads (word of row
//              32j + L at lane L, column j, replicated into every lane
//              quarter: the column and lane the block-scaled MMA reads for
//              that row), so the copies land ready to use.
//   warp 10    scale copies: one thread waits for each stage's loads, issues
//              the three copies of its scale blocks into the stage's own
//              TMEM scale columns and commits them to a per-stage barrier,
//              running ahead of the MMA thread by up to the ring.
//   warp 1     MMA: one thread waits for a stage's scales and issues its
//              four K=32 MMAs, each selecting its byte of the scale words by
//              the scale-factor ids of the instruction descriptor.
//   warps 2-9  epilogue: each warp drains its 32 x 128 block of the
//              accumulator into registers and releases it, then converts to
//              bf16 and stores (shared-memory transpose and whole-sector
//              stores, or 128-byte-swizzled boxes and TMA stores for the
//              K-grouped output).
// Tiles are 128 x 256 with one 256-column accumulator (TMEM columns 0 ..
// 255); each ring stage has its own scale columns (A from 256, B from 288),
// so a stage's scale copies never wait for the MMAs of the stage before.
// Every wait is bounded as in the tensor-scaled GEMM.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fp8gb.h"
#include "fp8gb_device.cuh"
#include "fp8gb_host.h"

namespace fp8gb {
namespace mx {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int UMMA_K = 32;
constexpr int STAGES = 4;         // dense; grouped kernels keep 3 (room for the group tables)
constexpr int STAGES_GROUPED = 3;
constexpr int THREADS = 352;  // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue, warp 10 scale copies
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int SFA_RAW = BM * 4;   // one scale word per A row
constexpr int SFB_RAW = 256 * 4;  // BN words used; room for two 128-row blocks
constexpr uint32_t TMEM_COLS = 512;
// one 256-column accumulator at column 0; scale columns, one set per ring
// stage so a stage's copies never overwrite scales that MMAs of an earlier
// stage may still be reading: A's 4 columns per stage from 256, B's 8 per
// stage from 288
constexpr uint32_t SFA_COL = 256;
constexpr uint32_t SFB_COL = 288;
static_assert(SFA_COL + 4 * STAGES <= SFB_COL && SFB_COL + 8 * STAGES <= TMEM_COLS, "scale columns");
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr int MAX_GROUPS = 1024;


enum { MODE_DENSE = 0, MODE_MGROUP = 1, MODE_KGROUP = 2 };

struct Params {
    int64_t M, N, K;
    const uint8_t *sA, *sB;
    int64_t rsA, rsB;  // scale rows of the A / B scale layouts (multiples of 128)
    uint16_t *C;
    int64_t ldc;
    int c_vec16;
    int num_m_blk, num_n_blk, num_k_blk;
    int m_fastest;
    int64_t total_tiles;  // dense
    const int32_t *offsets;
    int G;
    int64_t ld_T;
    int b_trans;   // M-grouped with B in the grouped transposed layout [N][ld_T]
    int64_t kpad;  // b_trans: column stride between experts, roundup(K, 128)
    unsigned int *err;
};

struct Tile {
    int32_t a_y, b_y;        // first TMA row of the A / B tile
    int32_t a_x0, b_x0;      // first K column (bytes) of the A / B tile
    int64_t sa_row, sb_row;  // first scale row of the A / B tile
    int64_t kt0a, kt0b;      // first K tile of A's / B's scale layout
    int nkb, last_steps;
    int64_t row0, row_end, col0, col_end, c_base;
};

template <int NS, bool TMA_OUT = false>
struct Smem {
    static constexpr int a_off = 0;
    static constexpr int b_off = NS * A_BYTES;
    static constexpr int sfa_raw_off = b_off + NS * B_BYTES;
    static constexpr int sfb_raw_off = sfa_raw_off + NS * SFA_RAW;
    static constexpr int bar_off = sfb_raw_off + NS * SFB_RAW;
    static constexpr int n_bars = 3 * NS + 2 + 2 + 2;
    static constexpr int slot_off = bar_off + n_bars * 8;
    // epilogue staging per warp: a 32 x 32 transpose block (direct stores) or
    // one 32-row x 32-column TMA box (64-byte rows, 64-byte swizzle), filled
    // four times per tile; 2 KB a warp leaves room for a four-stage ring
    static constexpr int stage_warp = TMA_OUT ? 32 * 64 : 32 * 80;
    static constexpr int stage_off = TMA_OUT ? (slot_off + 16 + 1023) / 1024 * 1024 : (slot_off + 16 + 127) / 128 * 128;
    static constexpr int misc_off = stage_off + 8 * stage_warp;  // group tables
};
constexpr int STAGE_PITCH = 80;  // epilogue staging: 32 rows x 32 bf16 per warp, rows padded to 80 bytes
__host__ __device__ constexpr int ring_stages(int mode, bool tma_out)
{
    return tma_out ? STAGES : (mode == 0 ? STAGES : STAGES_GROUPED);
}
// dynamic (ring, staging, group tables, 1024 alignment slack) plus the static
// block fit the 227 KB a block may use
static_assert(1024 + Smem<STAGES, true>::misc_off + 8 * (MAX_GROUPS + 1) + 1024 <= 227 * 1024, "smem");
static_assert(1024 + Smem<STAGES_GROUPED, false>::misc_off + 8 * (MAX_GROUPS + 1) + 1024 <= 227 * 1024, "smem");
static_assert(1024 + Smem<STAGES, false>::misc_off + 1024 <= 227 * 1024, "smem");

// Tile prefix [G+1] and offsets padded to FP8_MX_GROUP_ALIGN [G+1]; one warp.
__device__ bool build_group_tables(const Params &p, int MODE, int32_t *tile_prefix, int32_t *poff,
                                   int64_t *total_tiles)
{
    constexpr int AL = FP8_MX_GROUP_ALIGN;
    const int lane = threadIdx.x & 31;
    const int G = p.G;
    const int per = (G + 31) / 32;
    const int g0 = min(G, lane * per), g1 = min(G, g0 + per);
    int64_t lt = 0, lp = 0;
    int bad = 0;
    for (int e = g0; e < g1; e++) {
        const int m = p.offsets[e + 1] - p.offsets[e];
        if (m < 0) bad = 1;
        const int mm = max(m, 0);
        lt += MODE == MODE_MGROUP ? (int64_t)((mm + BM - 1) / BM) * p.num_n_blk : (int64_t)p.num_m_blk * p.num_n_blk;
        lp += (int64_t)((mm + AL - 1) / AL) * AL;
    }
    int64_t it = lt, ip = lp;
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t vt = __shfl_up_sync(0xffffffffu, it, d), vp = __shfl_up_sync(0xffffffffu, ip, d);
        if (lane >= d) {
            it += vt;
            ip += vp;
        }
    }
    int64_t rt = it - lt, rp = ip - lp;
    for (int e = g0; e < g1; e++) {
        tile_prefix[e] = (int32_t)rt;
        poff[e] = (int32_t)rp;
        const int mm = max(p.offsets[e + 1] - p.offsets[e], 0);
        rt += MODE == MODE_MGROUP ? (int64_t)((mm + BM - 1) / BM) * p.num_n_blk : (int64_t)p.num_m_blk * p.num_n_blk;
        rp += (int64_t)((mm + AL - 1) / AL) * AL;
    }
    const int64_t tt = __shfl_sync(0xffffffffu, it, 31), tp = __shfl_sync(0xffffffffu, ip, 31);
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        tile_prefix[G] = (int32_t)tt;
        poff[G] = (int32_t)tp;
    }
    *total_tiles = tt;
    const bool ok = !bad && p.offsets[0] == 0 && (int64_t)p.offsets[G] == p.M &&
                    (MODE != MODE_KGROUP || tp <= p.ld_T) && tp <= INT32_MAX && tt < (int64_t)1 << 31;
    return ok;
}

template <int MODE>
__device__ __forceinline__ Tile tile_info(const Params &p, int64_t t, const int32_t *tile_prefix, const int32_t *poff)
{
    Tile ti;
    if constexpr (MODE == MODE_DENSE) {
        int mb, nb;
        if (p.m_fastest) {
            mb = (int)(t % p.num_m_blk);
            nb = (int)(t / p.num_m_blk);
        } else {
            nb = (int)(t % p.num_n_blk);
            mb = (int)(t / p.num_n_blk);
        }
        ti.a_y = mb * BM;
        ti.b_y = nb * BN;
        ti.a_x0 = ti.b_x0 = 0;
        ti.sa_row = (int64_t)mb * BM;
        ti.sb_row = (int64_t)nb * BN;
        ti.kt0a = ti.kt0b = 0;
        ti.nkb = p.num_k_blk;
        ti.last_steps = (int)((p.K - (int64_t)(ti.nkb - 1) * BK) / UMMA_K);
        ti.row0 = (int64_t)mb * BM;
        ti.row_end = p.M;
        ti.col0 = (int64_t)nb * BN;
        ti.col_end = p.N;
        ti.c_base = 0;
    } else if constexpr (MODE == MODE_KGROUP) {
        // K-grouped: every group owns num_m_blk x num_n_blk tiles of its
        // [N][K] output block, so the group is a division (the tile count is
        // below 2^31).  The contraction runs over group e's columns, which
        // start at poff[e] (a multiple of 128).
        const int per = p.num_m_blk * p.num_n_blk;
        const int tt = (int)t;
        const int e = tt / per;
        const int local = tt - e * per;
        const int mb = local / p.num_n_blk, nb = local - mb * p.num_n_blk;
        const int m_e = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
        ti.a_y = mb * BM;
        ti.b_y = nb * BN;
        ti.a_x0 = ti.b_x0 = poff[e];
        ti.sa_row = (int64_t)mb * BM;
        ti.sb_row = (int64_t)nb * BN;
        ti.kt0a = ti.kt0b = poff[e] / BK;
        ti.nkb = (m_e + BK - 1) / BK;
        ti.last_steps = ti.nkb > 0 ? (m_e - (ti.nkb - 1) * BK + UMMA_K - 1) / UMMA_K : 0;
        ti.row0 = (int64_t)mb * BM;
        ti.row_end = p.N;
        ti.col0 = (int64_t)nb * BN;
        ti.col_end = p.K;
        ti.c_base = (int64_t)e * p.N * p.K;
    } else {
        int lo = 0, hi = p.G;  // group e: last with tile_prefix[e] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tile_prefix[mid] <= t)
                lo = mid;
            else
                hi = mid;
        }
        const int e = lo;
        const int64_t local = t - tile_prefix[e];
        const int64_t m_e = (int64_t)p.offsets[e + 1] - p.offsets[e];
        if constexpr (MODE == MODE_MGROUP) {
            const int64_t mt = (m_e + BM - 1) / BM;
            const int64_t mb = local % mt, nb = local / mt;  // rows fastest: the expert's weight tile stays in L2
            ti.a_y = (int32_t)(p.offsets[e] + mb * BM);
            ti.a_x0 = 0;
            ti.sa_row = poff[e] + mb * BM;
            ti.kt0a = 0;
            if (p.b_trans) {
                // expert e's [N][K] block starts at column e * kpad of B; its
                // scale words at K tile e * kpad / 128
                ti.b_y = (int32_t)(nb * BN);
                ti.b_x0 = (int32_t)(e * p.kpad);
                ti.sb_row = nb * BN;
                ti.kt0b = e * p.kpad / BK;
            } else {
                ti.b_y = (int32_t)((int64_t)e * p.N + nb * BN);
                ti.b_x0 = 0;
                ti.sb_row = (int64_t)e * p.N + nb * BN;
                ti.kt0b = 0;
            }
            ti.nkb = p.num_k_blk;
            ti.last_steps = (int)((p.K - (int64_t)(ti.nkb - 1) * BK) / UMMA_K);
            ti.row0 = p.offsets[e] + mb * BM;
            ti.row_end = p.offsets[e + 1];
            ti.col0 = nb * BN;
            ti.col_end = p.N;
            ti.c_base = 0;
        }
    }
    return ti;
}

// One finished tile for one epilogue warp: TMEM lane quarter q (rows q*32 ..
// q*32+31 of the tile), columns [cb, cb + 128).  The warp first copies its
// 32 x 128 accumulator block into registers and releases the accumulator
// (one arrive on `tempty`), so the next tile's MMAs start while this warp
// converts to bf16 and stores through its shared staging block.
__device__ __forceinline__ void epilogue_tile(const Params &p, const Tile &ti, uint32_t tmem_base, int q, int cb,
                                              int lane, uint8_t *stage, uint64_t *tempty)
{
    uint32_t r[4][32];
    const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)cb;
#pragma unroll
    for (int u = 0; u < 4; u++) tmem_ld_32x32b_x32(taddr + 32 * u, r[u]);
    tmem_ld_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tempty);
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const int64_t cu = ti.col0 + cb + u * 32;
        if (cu >= ti.col_end) break;  // warp-uniform
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; j++)
            packed[j] = pack_bf16x2(__uint_as_float(r[u][2 * j]), __uint_as_float(r[u][2 * j + 1]));
#pragma unroll
        for (int g = 0; g < 4; g++)
            *reinterpret_cast<uint4 *>(stage + lane * STAGE_PITCH + g * 16) =
                make_uint4(packed[4 * g], packed[4 * g + 1], packed[4 * g + 2], packed[4 * g + 3]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int rr = i * 8 + (lane >> 2), seg = lane & 3;
            const uint4 v = *reinterpret_cast<const uint4 *>(stage + rr * STAGE_PITCH + seg * 16);
            const int64_t row = ti.row0 + q * 32 + rr;
            const int64_t c = cu + seg * 8;
            if (row < ti.row_end && c < ti.col_end) {
                uint16_t *dst = p.C + ti.c_base + row * p.ldc + c;
                if (p.c_vec16 && c + 8 <= ti.col_end) {
                    *reinterpret_cast<uint4 *>(dst) = v;
                } else {
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                    for (int j = 0; j < 8 && c + j < ti.col_end; j++)
                        dst[j] = (uint16_t)(w[j / 2] >> (16 * (j & 1)));
                }
            }
        }
        __syncwarp();
    }
}

// The same drain for the K-grouped output through TMA stores: the warp's
// 32 x 128 block goes to two 128-byte-swizzled 32 x 64 boxes and the warp's
// lane 0 issues their stores; the warp first waits until its previous
// stores have read the boxes.  Rows of the tile past N are not stored (N %
// 32 == 0, so a quarter is all in or all out).
__device__ __forceinline__ void epilogue_tile_tma(const Params &p, const Tile &ti, uint32_t tmem_base, int q, int cb,
                                                  int lane, uint8_t *box, uint64_t *tempty, const CUtensorMap *tmC)
{
    uint32_t r[4][32];
    const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)cb;
#pragma unroll
    for (int u = 0; u < 4; u++) tmem_ld_32x32b_x32(taddr + 32 * u, r[u]);
    tmem_ld_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tempty);
    const int64_t qrow0 = ti.row0 + q * 32;
    const int32_t y = (int32_t)(ti.c_base / p.ldc + qrow0);  // row of the [G*N][K] view of C
    // four rounds of 32 columns through the warp's one box
#pragma unroll
    for (int b = 0; b < 4; b++) {
        // the box's previous store must have read it before it is refilled
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
        uint8_t *brow = box + lane * 64;
#pragma unroll
        for (int g = 0; g < 4; g++) {
            // 64-byte swizzle: 16-byte chunk g of row `lane` at chunk g ^ ((lane >> 1) & 3)
            const int chunk = g ^ ((lane >> 1) & 3);
            *reinterpret_cast<uint4 *>(brow + chunk * 16) =
                make_uint4(pack_bf16x2(__uint_as_float(r[b][8 * g]), __uint_as_float(r[b][8 * g + 1])),
                           pack_bf16x2(__uint_as_float(r[b][8 * g + 2]), __uint_as_float(r[b][8 * g + 3])),
                           pack_bf16x2(__uint_as_float(r[b][8 * g + 4]), __uint_as_float(r[b][8 * g + 5])),
                           pack_bf16x2(__uint_as_float(r[b][8 * g + 6]), __uint_as_float(r[b][8 * g + 7])));
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0 && qrow0 < ti.row_end) {
            const int64_t x = ti.col0 + cb + 32 * b;
            if (x < ti.col_end) tma_store_2d(tmC, (int32_t)x, y, box);
            bulk_commit_group();
        }
    }
}

// An empty K-group's block of C for one epilogue warp (rows q*32 .. q*32+31
// of the tile, columns [cb, cb + 128)): the warp's box filled with zeros and
// stored over its two 64-column chunks by TMA.  Out of line: it is off the
// hot path and would otherwise take registers from the epilogue.
__device__ __noinline__ void zero_block_tma(const Params &p, const Tile &ti, int q, int cb, int lane, uint8_t *box,
                                            const CUtensorMap *tmC)
{
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 32 * 64 / 16 / 32; k++) reinterpret_cast<uint4 *>(box)[k * 32 + lane] = make_uint4(0, 0, 0, 0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    const int64_t qrow0 = ti.row0 + q * 32;
    if (lane == 0 && qrow0 < ti.row_end) {
        const int32_t y = (int32_t)(ti.c_base / p.ldc + qrow0);
        for (int b = 0; b < 4; b++) {
            const int64_t x = ti.col0 + cb + 32 * b;
            if (x < ti.col_end) tma_store_2d(tmC, (int32_t)x, y, box);
        }
        bulk_commit_group();
    }
}

// NS_: ring stages (0: ring_stages(MODE, TMA_OUT)); the M-grouped modes run
// a four-stage ring when the group tables leave room for it
template <int MODE, bool TMA_OUT, int NS_ = 0>
__global__ void __launch_bounds__(THREADS, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, Params p, uint32_t idesc)
{
    constexpr int NS = NS_ ? NS_ : ring_stages(MODE, TMA_OUT);
    using L = Smem<NS, TMA_OUT>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem + L::a_off;
    uint8_t *sB = smem + L::b_off;
    uint8_t *sfa_raw = smem + L::sfa_raw_off;
    uint8_t *sfb_raw = smem + L::sfb_raw_off;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    uint64_t *full = bars;
    uint64_t *empty = bars + NS;
    uint64_t *tfull = bars + 2 * NS;
    uint64_t *tempty = tfull + 2;
    uint64_t *done = tempty + 2;
    uint64_t *sf_done = done + 1;
    uint64_t *sf_full = sf_done + 1;  // [NS]: the stage's scales are in TMEM
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::slot_off);
    int32_t *tile_prefix = reinterpret_cast<int32_t *>(smem + L::misc_off);
    int32_t *poff = tile_prefix + (p.G + 1);
    __shared__ int64_t s_total;
    __shared__ int s_ok;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_full[s], 1);
        }
        mbar_init(sf_done, 1);
        for (int b = 0; b < 2; b++) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 8);  // one arrive per epilogue warp
        }
        mbar_init(done, 1);
        fence_barrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if constexpr (MODE != MODE_DENSE) {
        if (warp == 2) {
            int64_t tt = 0;
            const bool ok = build_group_tables(p, MODE, tile_prefix, poff, &tt);
            if (lane == 0) {
                s_total = tt;
                s_ok = ok;
                if (!ok) record_error(p.err, ERR_BAD_OFFSETS);
            }
        }
    } else {
        if (threadIdx.x == 0) {
            s_total = p.total_tiles;
            s_ok = 1;
        }
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int64_t total = s_ok ? s_total : 0;

    if (warp == 0 && lane == 0) {
        // ---------------- producer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int issued_parity[NS];
        for (int s = 0; s < NS; s++) issued_parity[s] = -1;
        bool ok = true;
        // M-grouped: A's scale layout has one row per padded row (the padded total)
        const int64_t rsA = MODE == MODE_MGROUP ? (int64_t)poff[p.G] : p.rsA;
        for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const Tile ti = tile_info<MODE>(p, t, tile_prefix, poff);
            const int64_t na = rsA - ti.sa_row, nb = p.rsB - ti.sb_row;
            const uint32_t sfa_bytes = (uint32_t)((na < BM ? na : BM) * 4);
            const uint32_t sfb_bytes = (uint32_t)((nb < BN ? nb : BN) * 4);
            for (int kb = 0; kb < ti.nkb; kb++) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1, WAIT_LIMIT_NS, p.err, ERR_PRODUCER_WAIT)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES + sfa_bytes + sfb_bytes);
                tma_load_2d(sA + stage * A_BYTES, &tmA, ti.a_x0 + kb * BK, ti.a_y, &full[stage]);
                tma_load_2d(sB + stage * B_BYTES, &tmB, ti.b_x0 + kb * BK, ti.b_y, &full[stage]);
                bulk_load(sfa_raw + stage * SFA_RAW, p.sA + ((ti.kt0a + kb) * rsA + ti.sa_row) * 4, sfa_bytes,
                          &full[stage]);
                bulk_load(sfb_raw + stage * SFB_RAW, p.sB + ((ti.kt0b + kb) * p.rsB + ti.sb_row) * 4, sfb_bytes,
                          &full[stage]);
                issued_parity[stage] = (int)phase;
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        for (int s = 0; s < NS; s++)
            if (issued_parity[s] >= 0)
                mbar_wait_bounded(&full[s], (uint32_t)issued_parity[s], WAIT_LIMIT_NS, p.err, ERR_TEARDOWN_WAIT);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        int stage = 0;
        uint32_t phase = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const Tile ti = tile_info<MODE>(p, t, tile_prefix, poff);
            if (ti.nkb == 0) continue;  // empty K-grouped block: the epilogue writes zeros
            if (!mbar_wait_bounded(&tempty[0], acc_phase ^ 1, WAIT_LIMIT_NS, p.err, ERR_MMA_WAIT)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base;
            for (int kb = 0; kb < ti.nkb; kb++) {
                // the scale warp's copies of this stage completed (so did its TMA loads)
                if (!mbar_wait_bounded(&sf_full[stage], phase, WAIT_LIMIT_NS, p.err, ERR_MMA_WAIT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sfa = tmem_base + SFA_COL + 4 * stage, sfb = tmem_base + SFB_COL + 8 * stage;
                const uint32_t a_addr = smem_u32(sA + stage * A_BYTES);
                const uint32_t b_addr = smem_u32(sB + stage * B_BYTES);
                const int steps = kb == ti.nkb - 1 ? ti.last_steps : BK / UMMA_K;
                for (int k = 0; k < steps; k++) {
                    const uint64_t ad = smem_desc_k128_sw128(a_addr + k * UMMA_K);
                    const uint64_t bd = smem_desc_k128_sw128(b_addr + k * UMMA_K);
                    mma_mxf8f6f4(d_tmem, ad, bd, idesc_sf_ids(idesc, (uint32_t)k, (uint32_t)k), sfa, sfb,
                                 (kb | k) != 0);
                }
                mma_commit(&empty[stage]);
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            mma_commit(&tfull[0]);
            acc_phase ^= 1;
        }
        // all issued MMAs complete before TMEM is released
        mma_commit(done);
        mbar_wait_bounded(done, 0, WAIT_LIMIT_NS, p.err, ERR_TEARDOWN_WAIT);
    } else if (warp == 10 && lane == 0) {
        // ---------------- scale copies ----------------
        // the scale blocks arrive in copy order: each stage's three copies go
        // out as soon as its loads have landed
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const Tile ti = tile_info<MODE>(p, t, tile_prefix, poff);
            for (int kb = 0; kb < ti.nkb; kb++) {
                if (!mbar_wait_bounded(&full[stage], phase, WAIT_LIMIT_NS, p.err, ERR_MMA_WAIT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sfa = tmem_base + SFA_COL + 4 * stage, sfb = tmem_base + SFB_COL + 8 * stage;
                const uint32_t ra = smem_u32(sfa_raw + stage * SFA_RAW), rb = smem_u32(sfb_raw + stage * SFB_RAW);
                tmem_cp_32x128b_x4(sfa, smem_desc_sf(ra));
                tmem_cp_32x128b_x4(sfb, smem_desc_sf(rb));
                tmem_cp_32x128b_x4(sfb + 4, smem_desc_sf(rb + 512));
                mma_commit(&sf_full[stage]);
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // every issued copy lands before TMEM is released
        mma_commit(sf_done);
        mbar_wait_bounded(sf_done, 0, WAIT_LIMIT_NS, p.err, ERR_TEARDOWN_WAIT);
    } else if (warp >= 2 && warp < 10) {
        // ---------------- epilogue ----------------
        // warp w reads TMEM lane quarter w % 4 and one half (128 columns) of
        // the tile
        const int q = warp & 3;
        const int cb = ((warp - 2) >> 2) * 128;
        uint8_t *stage = smem + L::stage_off + (warp - 2) * L::stage_warp;
        uint32_t acc_phase = 0;
        for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
            const Tile ti = tile_info<MODE>(p, t, tile_prefix, poff);
            if (ti.nkb == 0) {  // empty K-group: its block of C is zero
                if constexpr (TMA_OUT) {
                    zero_block_tma(p, ti, q, cb, lane, stage, &tmC);
                } else {
                    const int64_t gr = ti.row0 + q * 32 + lane;
                    if (gr < ti.row_end) {
                        uint16_t *crow = p.C + ti.c_base + gr * p.ldc;
                        const int64_t c1 = ti.col0 + cb + 128 < ti.col_end ? ti.col0 + cb + 128 : ti.col_end;
                        for (int64_t c = ti.col0 + cb; c < c1; c++) crow[c] = 0;
                    }
                }
                continue;
            }
            if (!mbar_wait_bounded(&tfull[0], acc_phase, WAIT_LIMIT_NS, p.err, ERR_EPILOGUE_WAIT)) break;
            tc_fence_after();
            if constexpr (TMA_OUT)
                epilogue_tile_tma(p, ti, tmem_base, q, cb, lane, stage, &tempty[0], &tmC);
            else
                epilogue_tile(p, ti, tmem_base, q, cb, lane, stage, &tempty[0]);
            acc_phase ^= 1;
        }
        if constexpr (TMA_OUT) {
            if (lane == 0) bulk_wait_group0();  // every store completed before the block exits
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

// 2D map over a row-major u8 matrix [rows][ld] (inner extent `cols`), box
// {128 bytes, box_rows}, 128-byte swizzle, zero fill out of bounds.
static bool make_map(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int64_t ld, int box_rows)
{
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int MODE, bool TMA_OUT, int NS_ = 0>
static size_t smem_bytes(int G)
{
    constexpr int NS = NS_ ? NS_ : ring_stages(MODE, TMA_OUT);
    return 1024 + Smem<NS, TMA_OUT>::misc_off + (G > 0 ? 8 * (size_t)(G + 1) : 0);
}

// 2D map over the bf16 output viewed as [rows][cols] (row stride cols), box
// {32, 32}, 64-byte swizzle: the TMA-store epilogue.
static bool make_map_c(CUtensorMap *map, void *base, int64_t rows, int64_t cols)
{
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int MODE, bool TMA_OUT, int NS_>
static fp8_status_t launch_ns(const CUtensorMap &ma, const CUtensorMap &mb, const Params &p, int fa, int fb,
                              int64_t grid, cudaStream_t st, const CUtensorMap *mc)
{
    const size_t smem = smem_bytes<MODE, TMA_OUT, NS_>(MODE == MODE_DENSE ? 0 : p.G);
    cudaError_t e = cudaFuncSetAttribute(mx_gemm_kernel<MODE, TMA_OUT, NS_>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail_with(e);
    const uint32_t idesc = idesc_mxf8f6f4(fa, fb, BM, BN);
    mx_gemm_kernel<MODE, TMA_OUT, NS_><<<(unsigned)grid, THREADS, smem, st>>>(ma, mb, mc ? *mc : ma, p, idesc);
    return check_launch();
}

template <int MODE, bool TMA_OUT = false>
static fp8_status_t launch(const CUtensorMap &ma, const CUtensorMap &mb, const Params &p, int fa, int fb,
                           int64_t grid, cudaStream_t st, const CUtensorMap *mc = nullptr)
{
    // grouped modes with direct stores: four stages when the group tables fit
    // beside them (up to about 800 groups), else three
    if constexpr (MODE != MODE_DENSE && !TMA_OUT) {
        if (smem_bytes<MODE, false, STAGES>(p.G) <= 227 * 1024)
            return launch_ns<MODE, false, STAGES>(ma, mb, p, fa, fb, grid, st, mc);
    }
    return launch_ns<MODE, TMA_OUT, 0>(ma, mb, p, fa, fb, grid, st, mc);
}

static bool format_ok(int f) { return f == FP8_E4M3FN || f == FP8_E5M2; }

}  // namespace mx
}  // namespace fp8gb

using namespace fp8gb;

extern "C" fp8_status_t fp8_mx_gemm(const uint8_t *A, int fa, int64_t lda, const uint8_t *sA, const uint8_t *B,
                                    int fb, int64_t ldb, const uint8_t *sB, int64_t M, int64_t N, int64_t K,
                                    void *C_bf16, int64_t ldc, void *stream)
{
    if (!A || !B || !sA || !sB || !C_bf16) return FP8_ERR_INVALID_ARG;
    if (fa == FP8_E4M3FNUZ || fb == FP8_E4M3FNUZ || fa == FP8_E5M2FNUZ || fb == FP8_E5M2FNUZ)
        return FP8_ERR_UNSUPPORTED;
    if (!mx::format_ok(fa) || !mx::format_ok(fb)) return FP8_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1 || lda < K || ldb < K || ldc < N) return FP8_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FP8_ERR_INVALID_ARG;
    if (K % FP8_MX_BLOCK != 0 || lda % 16 != 0 || ldb % 16 != 0) return FP8_ERR_ALIGNMENT;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sA, 16) || !aligned(sB, 16) || !aligned(C_bf16, 2))
        return FP8_ERR_ALIGNMENT;

    mx::Params p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.sA = sA;
    p.sB = sB;
    p.rsA = round_up_128(M);
    p.rsB = round_up_128(N);
    p.C = static_cast<uint16_t *>(C_bf16);
    p.ldc = ldc;
    p.c_vec16 = ldc % 8 == 0 && aligned(C_bf16, 16);
    p.num_m_blk = (int)((M + mx::BM - 1) / mx::BM);
    p.num_n_blk = (int)((N + mx::BN - 1) / mx::BN);
    p.num_k_blk = (int)((K + mx::BK - 1) / mx::BK);
    p.m_fastest = M <= N;
    p.total_tiles = (int64_t)p.num_m_blk * p.num_n_blk;
    p.err = device_error_word();

    CUtensorMap ma, mb;
    if (!mx::make_map(&ma, A, M, K, lda, mx::BM) || !mx::make_map(&mb, B, N, K, ldb, mx::BN)) return FP8_ERR_CUDA;
    const int64_t grid = p.total_tiles < num_sms() ? p.total_tiles : num_sms();
    return mx::launch<mx::MODE_DENSE>(ma, mb, p, fa, fb, grid, static_cast<cudaStream_t>(stream));
}

extern "C" fp8_status_t fp8_mx_grouped_gemm(int mode, const uint8_t *A, int fa, const uint8_t *sA,
                                            const uint8_t *B, int fb, const uint8_t *sB,
                                            const int32_t *group_offsets, int G, int64_t M_total, int64_t N,
                                            int64_t K, void *C_bf16, int64_t ld_T, void *stream)
{
    if (!A || !B || !sA || !sB || !C_bf16 || !group_offsets) return FP8_ERR_INVALID_ARG;
    if (fa == FP8_E4M3FNUZ || fb == FP8_E4M3FNUZ || fa == FP8_E5M2FNUZ || fb == FP8_E5M2FNUZ)
        return FP8_ERR_UNSUPPORTED;
    if (!mx::format_ok(fa) || !mx::format_ok(fb)) return FP8_ERR_INVALID_ARG;
    if (mode != FP8_GROUPED_M && mode != FP8_GROUPED_K && mode != FP8_GROUPED_M_BT) return FP8_ERR_INVALID_ARG;
    if (G < 1 || G > mx::MAX_GROUPS || M_total < 0 || N < 1 || K < 1) return FP8_ERR_INVALID_ARG;
    if (M_total > INT32_MAX || N > INT32_MAX || K > INT32_MAX || (int64_t)G * N > INT32_MAX)
        return FP8_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sA, 16) || !aligned(sB, 16) || !aligned(C_bf16, 2))
        return FP8_ERR_ALIGNMENT;
    // M-grouped: expert e's weight rows start at scale row e * N, which must
    // start a 128-row block of the MX scale layout
    if (mode == FP8_GROUPED_M && N % 128 != 0) return FP8_ERR_ALIGNMENT;

    mx::Params p{};
    p.M = M_total;
    p.N = N;
    p.K = K;
    p.sA = sA;
    p.sB = sB;
    p.C = static_cast<uint16_t *>(C_bf16);
    p.offsets = group_offsets;
    p.G = G;
    p.err = device_error_word();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUtensorMap ma, mb;
    const int64_t grid = num_sms();

    if (mode == FP8_GROUPED_M || mode == FP8_GROUPED_M_BT) {
        if (K % FP8_MX_BLOCK != 0 || N % 4 != 0) return FP8_ERR_ALIGNMENT;
        p.rsA = 0;  // the padded total, known on the device from the offsets
        p.rsB = (int64_t)G * N;
        p.kpad = (K + mx::BK - 1) / mx::BK * mx::BK;
        if (mode == FP8_GROUPED_M_BT) {
            if (ld_T % 16 != 0) return FP8_ERR_ALIGNMENT;
            if (ld_T < (int64_t)G * p.kpad || ld_T > INT32_MAX) return FP8_ERR_INVALID_ARG;
            p.b_trans = 1;
            p.rsB = round_up_128(N);  // B's scale rows: the N rows of the transposed layout
        }
        p.ldc = N;
        p.c_vec16 = N % 8 == 0 && aligned(C_bf16, 16);
        p.num_m_blk = 0;
        p.num_n_blk = (int)((N + mx::BN - 1) / mx::BN);
        p.num_k_blk = (int)((K + mx::BK - 1) / mx::BK);
        if (M_total == 0) return FP8_OK;
        if (!mx::make_map(&ma, A, M_total, K, K, mx::BM)) return FP8_ERR_CUDA;
        if (p.b_trans ? !mx::make_map(&mb, B, N, (int64_t)G * p.kpad, ld_T, mx::BN)
                      : !mx::make_map(&mb, B, (int64_t)G * N, K, K, mx::BN))
            return FP8_ERR_CUDA;
        return mx::launch<mx::MODE_MGROUP>(ma, mb, p, fa, fb, grid, st);
    }
    // K-grouped (wgrad): C[e] = A_e [N][m_e] . B_e [K][m_e]^T
    if (ld_T < 128 || ld_T % 128 != 0 || N % 4 != 0 || K % 4 != 0) return FP8_ERR_ALIGNMENT;
    p.rsA = round_up_128(N);
    p.rsB = round_up_128(K);
    p.ldc = K;
    p.c_vec16 = K % 8 == 0 && aligned(C_bf16, 16);
    p.ld_T = ld_T;
    p.num_m_blk = (int)((N + mx::BM - 1) / mx::BM);
    p.num_n_blk = (int)((K + mx::BN - 1) / mx::BN);
    p.num_k_blk = 0;
    if (!mx::make_map(&ma, A, N, ld_T, ld_T, mx::BM) || !mx::make_map(&mb, B, K, ld_T, ld_T, mx::BN))
        return FP8_ERR_CUDA;
    if (N % 32 == 0 && K % 8 == 0 && aligned(C_bf16, 16) && (int64_t)G * N <= INT32_MAX) {
        // the output is the whole cost of this mode: TMA-store epilogue
        CUtensorMap mc;
        if (!mx::make_map_c(&mc, C_bf16, (int64_t)G * N, K)) return FP8_ERR_CUDA;
        return mx::launch<mx::MODE_KGROUP, true>(ma, mb, p, fa, fb, grid, st, &mc);
    }
    return mx::launch<mx::MODE_KGROUP>(ma, mb, p, fa, fb, grid, st);
}
