// gemm.cu -- FP8 scaled GEMM and grouped GEMM on the tcgen05 tensor cores.
//
// C[m][n] = bf16( sum_k A[m][k] B[n][k] * sa(m) * sb(n) ), FP8 E4M3 / E5M2
// operands, fp32 accumulation in tensor memory, per-tensor or per-row /
// per-column scales applied in the epilogue.  The grouped variants run the
// per-expert GEMMs of a Mixture-of-Experts layer over variable-size row
// groups in one launch.
//
// Method: FP8 for the linear layers' forward and backward GEMMs ("FP8
// Training on MI300X", Patched nanochat/fp8.py; "FP8 training for Flux
// models", fp8_wgrad); per-row / per-column scales ("How PyTorch FP8
// Optimizations on AMD GPUs ...", rowwise FP8); grouped GEMM for MoE (same
// page and "FP8 Training on AMD GPUs with TorchTitan and TorchAO").
//
// Design (GB300, sm_103a): persistent, warp-specialised kernel, one CTA per
// SM, 320 threads.
//   warp 0     TMA producer: 128x128-byte A and 256x128-byte B tiles into a
//              4-stage shared-memory ring (128-byte swizzle), completion by
//              mbarrier transaction counts.
//   warp 1     MMA issuer: one thread issues tcgen05.mma kind::f8f6f4
//              (M=128, N=256, K=32) into a TMEM accumulator; tcgen05.commit
//              frees ring stages and hands finished accumulators over.
//   warps 2-9  epilogue: tcgen05.ld 32 columns at a time (each warp one TMEM
//              lane quarter and half of the columns), scale, convert to
//              bf16, store.  Two 256-column accumulators (all 512 TMEM
//              columns) let the epilogue of one tile overlap the main loop of
//              the next.
// Two more kernels share this structure (each described where it is
// defined): fp8_gemm_pair_kernel, the dense GEMM for M > 128 on CTA pairs
// (256 x 256 tiles from 2-SM MMAs, each CTA staging half of A and of B), and
// fp8_gemm_kgroup_tma_kernel, the K-grouped wgrad (576 threads: two groups
// of eight epilogue warps on alternate tiles and accumulators, writing
// through 128-byte-swizzled boxes and TMA stores).
// Every mbarrier wait is bounded (about 2 s of wall time); a wait that gives
// up records the device error word, drains in-flight copies, releases TMEM
// and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fp8gb.h"
#include "fp8gb_device.cuh"
#include "fp8gb_host.h"

namespace fp8gb {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;  // bytes = FP8 elements per k-block (one 128B swizzle row)
constexpr int UMMA_K = 32;
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK;
constexpr int B_STAGE_BYTES = BN * BK;
constexpr int GEMM_THREADS = 320;   // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr int MAX_GROUPS = 1024;  // group tables share shared memory with the ring

enum { MODE_DENSE = 0, MODE_MGROUP = 1, MODE_KGROUP = 2 };

struct GemmParams {
    int64_t M, N, K;  // dense / M-grouped: A [M][K], B [N][K]; K-grouped: C[e] is [M=N][N=K]
    const float *sa;
    const float *sb;
    int sa_per_row, sb_per_row;
    uint16_t *C;
    int64_t ldc;
    int c_vec16;  // every row of C starts 16-byte aligned: 8-wide vector stores
    int num_m_blk, num_n_blk, num_k_blk;
    int m_fastest;
    int64_t total_tiles;  // dense
    const int32_t *offsets;
    int G;
    int64_t ld_T;  // K-grouped: padded width of A and B
    int b_trans;   // M-grouped with B in the grouped colwise layout [N][G * kpad]
    int64_t kpad;  // roundup(K, 32): column stride between experts when b_trans
    unsigned int *err;
};

struct TileInfo {
    int32_t a_y, b_y;
    int32_t a_x0, b_x0;  // first K column (bytes) of the A and B tiles
    int nkb, last_steps;
    int64_t row0, row_end, col0, col_end;
    int64_t c_base;
    int64_t sa_base, sb_base;
};

struct SmemLayout {
    static constexpr int a_off = 0;
    static constexpr int b_off = STAGES * A_STAGE_BYTES;
    static constexpr int bar_off = b_off + STAGES * B_STAGE_BYTES;
    static constexpr int n_bars = 2 * STAGES + 2 + 2 + 1;
    static constexpr int slot_off = bar_off + n_bars * 8;
    // epilogue staging: per epilogue warp a 32-row x 32-column bf16 block,
    // rows padded to 80 bytes (conflict-free 16-byte accesses both ways)
    static constexpr int stage_pitch = 80;
    static constexpr int stage_warp_bytes = 32 * stage_pitch;
    static constexpr int stage_off = (slot_off + 16 + 127) / 128 * 128;
    static constexpr int misc_off = stage_off + 8 * stage_warp_bytes;  // int32 group tables start here
    static constexpr int base_bytes = misc_off;
};

// Group tables in shared memory: tile prefix [G+1] then padded offsets [G+1].
__device__ bool build_group_tables(const GemmParams &p, int MODE, int32_t *tile_prefix, int32_t *poff,
                                   int64_t *total_tiles)
{
    // executed by one warp
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
        lp += (int64_t)((mm + 31) / 32) * 32;
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
        rp += (int64_t)((mm + 31) / 32) * 32;
    }
    const int64_t tt = __shfl_sync(0xffffffffu, it, 31), tp = __shfl_sync(0xffffffffu, ip, 31);
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        tile_prefix[G] = (int32_t)tt;
        poff[G] = (int32_t)tp;
    }
    *total_tiles = tt;
    const bool ok = !bad && p.offsets[0] == 0 && (int64_t)p.offsets[G] == p.M &&
                    (MODE != MODE_KGROUP || tp <= p.ld_T) && tt < (int64_t)1 << 31;
    return ok;
}

template <int MODE>
__device__ __forceinline__ TileInfo tile_info(const GemmParams &p, int64_t t, const int32_t *tile_prefix,
                                              const int32_t *poff)
{
    TileInfo ti;
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
        ti.nkb = p.num_k_blk;
        ti.last_steps = BK / UMMA_K;
        ti.row0 = (int64_t)mb * BM;
        ti.row_end = p.M;
        ti.col0 = (int64_t)nb * BN;
        ti.col_end = p.N;
        ti.c_base = 0;
        ti.sa_base = 0;
        ti.sb_base = 0;
    } else if constexpr (MODE == MODE_KGROUP) {
        // K-grouped: every group owns num_m_blk x num_n_blk tiles of its
        // [N][K] output block, so the group is a division (the tile count is
        // below 2^31); the group's padded column count is the difference of
        // its padded offsets.  Output block e is [N][K]; the contraction runs
        // over the group's padded columns.
        const int per = p.num_m_blk * p.num_n_blk;
        const int tt = (int)t;
        const int e = tt / per;
        const int local = tt - e * per;
        const int mb = local / p.num_n_blk, nb = local - mb * p.num_n_blk;
        const int pad = poff[e + 1] - poff[e];
        ti.a_y = mb * BM;
        ti.b_y = nb * BN;
        ti.a_x0 = ti.b_x0 = poff[e];
        ti.nkb = (pad + BK - 1) / BK;
        ti.last_steps = ti.nkb > 0 ? (pad - (ti.nkb - 1) * BK) / UMMA_K : 0;
        ti.row0 = (int64_t)mb * BM;
        ti.row_end = p.N;  // rows of C[e]
        ti.col0 = (int64_t)nb * BN;
        ti.col_end = p.K;
        ti.c_base = (int64_t)e * p.N * p.K;
        ti.sa_base = (int64_t)e * p.N;
        ti.sb_base = (int64_t)e * p.K;
    } else {
        // group e: last with tile_prefix[e] <= t
        int lo = 0, hi = p.G;
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
            ti.nkb = p.num_k_blk;
            if (p.b_trans) {
                // expert e's K columns start at e * kpad; only the MMA steps
                // up to kpad are issued so the next expert's columns are unused
                ti.b_y = (int32_t)(nb * BN);
                ti.a_x0 = 0;
                ti.b_x0 = (int32_t)(e * p.kpad);
                ti.last_steps = (int)((p.kpad - (int64_t)(ti.nkb - 1) * BK) / UMMA_K);
            } else {
                ti.b_y = (int32_t)((int64_t)e * p.N + nb * BN);
                ti.a_x0 = ti.b_x0 = 0;
                ti.last_steps = BK / UMMA_K;
            }
            ti.row0 = p.offsets[e] + mb * BM;
            ti.row_end = p.offsets[e + 1];
            ti.col0 = nb * BN;
            ti.col_end = p.N;
            ti.c_base = 0;
            ti.sa_base = 0;
            ti.sb_base = (int64_t)e * p.N;
        }
    }
    return ti;
}

// Epilogue of one finished tile for one warp: TMEM lane quarter q (rows
// q*32 .. q*32+31 of the tile), column half `half` (128 columns).  Reads the
// accumulator at TMEM column `acc_col`, applies the row / column scales,
// converts to bf16 and stores through the warp's shared staging block.
__device__ __forceinline__ void epilogue_tile(const GemmParams &p, const TileInfo &ti, uint32_t tmem_base,
                                              uint32_t acc_col, int q, int half, int lane, uint8_t *stage)
{
    const int64_t gr = ti.row0 + q * 32 + lane;
    const bool row_ok = gr < ti.row_end;
    const int64_t cbeg = ti.col0 + half * (BN / 2);
    const int64_t cend = min(cbeg + BN / 2, ti.col_end);
    const float sa_v = row_ok ? (p.sa_per_row ? __ldg(p.sa + ti.sa_base + gr) : __ldg(p.sa)) : 0.0f;
    const float sb0 = p.sb_per_row ? 0.0f : __ldg(p.sb);
    // two 32-column chunks per round: both TMEM loads are in flight
    // before the first wait
    for (int ch = 0; ch < BN / 64; ch += 2) {
        const int64_t c0 = cbeg + ch * 32;
        if (c0 >= cend) break;  // warp-uniform
        uint32_t r[2][32];
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) +
                               acc_col + (uint32_t)(half * (BN / 2) + ch * 32);
        tmem_ld_32x32b_x32(taddr, r[0]);
        tmem_ld_32x32b_x32(taddr + 32, r[1]);
        // column scales: lane j holds the scale of column c + j; the
        // other lanes read it by shuffle (one coalesced load per chunk)
        float sbl[2] = {sb0, sb0};
        if (p.sb_per_row) {
#pragma unroll
            for (int u = 0; u < 2; u++) {
                const int64_t cc = c0 + u * 32 + lane;
                sbl[u] = cc < cend ? __ldg(p.sb + ti.sb_base + cc) : 0.0f;
            }
        }
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 2; u++) {
            const int64_t cu = c0 + u * 32;
            if (cu >= cend) break;  // warp-uniform
            uint32_t packed[16];
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const float sb_lo = __shfl_sync(0xffffffffu, sbl[u], 2 * j);
                const float sb_hi = __shfl_sync(0xffffffffu, sbl[u], 2 * j + 1);
                const float lo = __uint_as_float(r[u][2 * j]) * sa_v * sb_lo;
                const float hi = __uint_as_float(r[u][2 * j + 1]) * sa_v * sb_hi;
                packed[j] = pack_bf16x2(lo, hi);
            }
            // transpose through shared memory so that each store
            // instruction writes 8 rows x 64 contiguous bytes (whole
            // sectors) instead of 32 rows x 16 bytes
#pragma unroll
            for (int g = 0; g < 4; g++)
                *reinterpret_cast<uint4 *>(stage + lane * SmemLayout::stage_pitch + g * 16) =
                    make_uint4(packed[4 * g], packed[4 * g + 1], packed[4 * g + 2], packed[4 * g + 3]);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int rr = i * 8 + (lane >> 2), seg = lane & 3;
                const uint4 v =
                    *reinterpret_cast<const uint4 *>(stage + rr * SmemLayout::stage_pitch + seg * 16);
                const int64_t row = ti.row0 + q * 32 + rr;
                const int64_t c = cu + seg * 8;
                if (row < ti.row_end && c < cend) {
                    uint16_t *dst = p.C + ti.c_base + row * p.ldc + c;
                    if (p.c_vec16 && c + 8 <= cend) {
                        *reinterpret_cast<uint4 *>(dst) = v;
                    } else {
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                        for (int j = 0; j < 8 && c + j < cend; j++)
                            dst[j] = (uint16_t)(w[j / 2] >> (16 * (j & 1)));
                    }
                }
            }
            __syncwarp();
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmParams p,
                    uint32_t idesc)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem + SmemLayout::a_off;
    uint8_t *sB = smem + SmemLayout::b_off;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SmemLayout::bar_off);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *tfull = bars + 2 * STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SmemLayout::slot_off);
    int32_t *tile_prefix = reinterpret_cast<int32_t *>(smem + SmemLayout::misc_off);
    int32_t *poff = tile_prefix + (p.G + 1);
    __shared__ int64_t s_total;
    __shared__ int s_ok;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
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
        // ---------------- TMA producer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int issued_parity[STAGES];
        for (int s = 0; s < STAGES; s++) issued_parity[s] = -1;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const TileInfo ti = tile_info<MODE>(p, t, tile_prefix, poff);
            for (int kb = 0; kb < ti.nkb; kb++) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1, WAIT_LIMIT_NS, p.err, ERR_PRODUCER_WAIT)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[stage], A_STAGE_BYTES + B_STAGE_BYTES);
                tma_load_2d(sA + stage * A_STAGE_BYTES, &tmA, ti.a_x0 + kb * BK, ti.a_y, &full[stage]);
                tma_load_2d(sB + stage * B_STAGE_BYTES, &tmB, ti.b_x0 + kb * BK, ti.b_y, &full[stage]);
                issued_parity[stage] = (int)phase;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // drain: every issued copy must have landed before the CTA exits
        for (int s = 0; s < STAGES; s++)
            if (issued_parity[s] >= 0)
                mbar_wait_bounded(&full[s], (uint32_t)issued_parity[s], WAIT_LIMIT_NS, p.err, ERR_TEARDOWN_WAIT);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const TileInfo ti = tile_info<MODE>(p, t, tile_prefix, poff);
            if (ti.nkb == 0) continue;  // empty K-grouped block: the epilogue writes zeros
            if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, WAIT_LIMIT_NS, p.err, ERR_MMA_WAIT)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < ti.nkb; kb++) {
                if (!mbar_wait_bounded(&full[stage], phase, WAIT_LIMIT_NS, p.err, ERR_MMA_WAIT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(sA + stage * A_STAGE_BYTES);
                const uint32_t b_addr = smem_u32(sB + stage * B_STAGE_BYTES);
                const int steps = kb == ti.nkb - 1 ? ti.last_steps : BK / UMMA_K;
                for (int k = 0; k < steps; k++) {
                    const uint64_t ad = smem_desc_k128_sw128(a_addr + k * UMMA_K);
                    const uint64_t bd = smem_desc_k128_sw128(b_addr + k * UMMA_K);
                    mma_f8f6f4(d_tmem, ad, bd, idesc, (kb | k) != 0);
                }
                mma_commit(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            mma_commit(&tfull[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        // all issued MMAs complete before TMEM is released
        mma_commit(done);
        mbar_wait_bounded(done, 0, WAIT_LIMIT_NS, p.err, ERR_TEARDOWN_WAIT);
    } else if (warp >= 2) {
        // ---------------- epilogue ----------------
        // 8 warps: warp w reads TMEM lane quarter (w % 4) -- the hardware rule
        // for tcgen05.ld -- and one half of the tile's 256 columns.
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        uint8_t *stage = smem + SmemLayout::stage_off + (warp - 2) * SmemLayout::stage_warp_bytes;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
            const TileInfo ti = tile_info<MODE>(p, t, tile_prefix, poff);
            const int64_t gr = ti.row0 + q * 32 + lane;
            const bool row_ok = gr < ti.row_end;
            uint16_t *crow = p.C + ti.c_base + gr * p.ldc;
            const int64_t cbeg = ti.col0 + half * (BN / 2);
            const int64_t cend = min(cbeg + BN / 2, ti.col_end);
            if (ti.nkb == 0) {
                if (row_ok)
                    for (int64_t c = cbeg; c < cend; c += 8) {
                        if (p.c_vec16 && c + 8 <= cend)
                            *reinterpret_cast<uint4 *>(crow + c) = make_uint4(0, 0, 0, 0);
                        else
                            for (int64_t j = c; j < cend; j++) crow[j] = 0;
                    }
                continue;
            }
            if (!mbar_wait_bounded(&tfull[acc], acc_phase, WAIT_LIMIT_NS, p.err, ERR_EPILOGUE_WAIT)) break;
            tc_fence_after();
            epilogue_tile(p, ti, tmem_base, (uint32_t)(acc * BN), q, half, lane, stage);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
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

// ---------------------------------------------------------------------------
// K-grouped GEMM (MoE wgrad) with a TMA-store epilogue.
//
// Each output tile of dW_e is written once and its contraction is short (one
// expert's tokens), so the kernel is bound by writing C.  Two groups of eight
// epilogue warps take the CTA's tiles alternately, each group draining its
// own TMEM accumulator, so a group has two tile periods for its drain,
// conversion and stores while the MMAs of the next tile fill the other
// accumulator.  Each epilogue warp converts its 32 x 128 block to bf16 in
// two rounds of 64 columns through one 32-row x 64-column box in shared
// memory (128-byte swizzle: conflict-free 16-byte writes) and issues the TMA
// stores itself; it waits only for the box's previous store to finish
// reading shared memory before refilling it.  An empty group's blocks are
// stored from a zeroed box.  A 3-stage operand ring leaves room for the 64
// KB of boxes.  Used when N is a multiple of 32 (a 32-row quarter never
// straddles two experts' blocks), K a multiple of 8 and C 16-byte aligned.
// ---------------------------------------------------------------------------
constexpr int KT_STAGES = 3;
constexpr int KT_BOX_BYTES = 32 * 128;  // 32 rows x 64 bf16
constexpr int KT_THREADS = 576;         // warp 0 TMA, warp 1 MMA, warps 2-9 and 10-17: two epilogue groups

struct SmemLayoutKT {
    static constexpr int a_off = 0;
    static constexpr int b_off = KT_STAGES * A_STAGE_BYTES;
    static constexpr int box_off = b_off + KT_STAGES * B_STAGE_BYTES;      // 1024-aligned
    static constexpr int bar_off = box_off + 16 * KT_BOX_BYTES;            // one box per epilogue warp
    static constexpr int n_bars = 2 * KT_STAGES + 2 + 2 + 1;
    static constexpr int slot_off = bar_off + n_bars * 8;
    static constexpr int misc_off = (slot_off + 16 + 127) / 128 * 128;    // group tables
};
static_assert(1024 + SmemLayoutKT::misc_off + 8 * (MAX_GROUPS + 1) + 1024 <= 227 * 1024,
              "K-grouped ring, boxes and group tables fit in shared memory");

__global__ void __launch_bounds__(KT_THREADS, 1)
    fp8_gemm_kgroup_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                               const __grid_constant__ CUtensorMap tmC, GemmParams p, uint32_t idesc)
{
    constexpr int MODE = MODE_KGROUP;
    using L = SmemLayoutKT;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem + L::a_off;
    uint8_t *sB = smem + L::b_off;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    uint64_t *full = bars;
    uint64_t *empty = bars + KT_STAGES;
    uint64_t *tfull = bars + 2 * KT_STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::slot_off);
    int32_t *tile_prefix = reinterpret_cast<int32_t *>(smem + L::misc_off);
    int32_t *poff = tile_prefix + (p.G + 1);
    __shared__ int64_t s_total;
    __shared__ int s_ok;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < KT_STAGES; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 8);
        }
        mbar_init(done, 1);
        fence_barrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmC);
    }
    if (warp == 2) {
        int64_t tt = 0;
        const bool ok = build_group_tables(p, MODE, tile_prefix, poff, &tt);
        if (lane == 0) {
            s_total = tt;
            s_ok = ok;
            if (!ok) record_error(p.err, ERR_BAD_OFFSETS);
        }
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int64_t total = s_ok ? s_total : 0;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int issued_parity[KT_STAGES];
        for (int s = 0; s < KT_STAGES; s++) issued_parity[s] = -1;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const TileInfo ti = tile_info<MODE>(p, t, tile_prefix, poff);
            for (int kb = 0; kb < ti.nkb; kb++) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1, WAIT_LIMIT_NS, p.err, ERR_PRODUCER_WAIT)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[stage], A_STAGE_BYTES + B_STAGE_BYTES);
                tma_load_2d(sA + stage * A_STAGE_BYTES, &tmA, ti.a_x0 + kb * BK, ti.a_y, &full[stage]);
                tma_load_2d(sB + stage * B_STAGE_BYTES, &tmB, ti.b_x0 + kb * BK, ti.b_y, &full[stage]);
                issued_parity[stage] = (int)phase;
                if (++stage == KT_STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        for (int s = 0; s < KT_STAGES; s++)
            if (issued_parity[s] >= 0)
                mbar_wait_bounded(&full[s], (uint32_t)issued_parity[s], WAIT_LIMIT_NS, p.err, ERR_TEARDOWN_WAIT);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        // the CTA's i-th tile goes to accumulator i % 2 (drained by epilogue
        // group i % 2); bit a of acc_phase is the phase of accumulator a
        int stage = 0;
        uint32_t phase = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        int64_t i = 0;
        for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x, ++i) {
            const TileInfo ti = tile_info<MODE>(p, t, tile_prefix, poff);
            if (ti.nkb == 0) continue;
            const int acc = (int)(i & 1);
            if (!mbar_wait_bounded(&tempty[acc], ((acc_phase >> acc) & 1u) ^ 1u, WAIT_LIMIT_NS, p.err, ERR_MMA_WAIT))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < ti.nkb; kb++) {
                if (!mbar_wait_bounded(&full[stage], phase, WAIT_LIMIT_NS, p.err, ERR_MMA_WAIT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(sA + stage * A_STAGE_BYTES);
                const uint32_t b_addr = smem_u32(sB + stage * B_STAGE_BYTES);
                const int steps = kb == ti.nkb - 1 ? ti.last_steps : BK / UMMA_K;
                for (int k = 0; k < steps; k++)
                    mma_f8f6f4(d_tmem, smem_desc_k128_sw128(a_addr + k * UMMA_K),
                               smem_desc_k128_sw128(b_addr + k * UMMA_K), idesc, (kb | k) != 0);
                mma_commit(&empty[stage]);
                if (++stage == KT_STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            mma_commit(&tfull[acc]);
            acc_phase ^= 1u << acc;
        }
        mma_commit(done);
        mbar_wait_bounded(done, 0, WAIT_LIMIT_NS, p.err, ERR_TEARDOWN_WAIT);
    } else if (warp >= 2) {
        // ---------------- epilogue: TMEM -> bf16 boxes -> TMA stores ----------------
        // Two groups of 8 warps take alternate tiles of the CTA: group g
        // drains accumulator g, so each group has two tile periods for its
        // drain, conversion and stores, and looks up only its own tiles.  In
        // a group, warp w reads TMEM lane quarter w % 4 (the quarter its id
        // may access) and one half (128 columns) of the tile, in two rounds
        // of 64 columns through one box.  An empty group's tiles are zeros.
        const int g = (warp - 2) >> 3;
        const int q = warp & 3;
        const int half = ((warp - 2) >> 2) & 1;
        uint8_t *box = smem + L::box_off + (warp - 2) * KT_BOX_BYTES;
        uint32_t acc_phase = 0;
        for (int64_t t = blockIdx.x + (int64_t)g * gridDim.x; t < total; t += 2 * (int64_t)gridDim.x) {
            const TileInfo ti = tile_info<MODE>(p, t, tile_prefix, poff);
            const int64_t qrow0 = ti.row0 + q * 32;  // this warp's first row of C[e]
            const bool live = qrow0 < ti.row_end;    // N % 32 == 0: the quarter is all in or all out
            const int64_t cbeg = ti.col0 + half * (BN / 2);
            if (ti.nkb == 0) {
                // empty group: the warp's box filled with zeros, stored over
                // its two 64-column chunks by TMA
                if (lane == 0) bulk_wait_group_read0();
                __syncwarp();
                for (int k = lane; k < KT_BOX_BYTES / 16; k += 32)
                    reinterpret_cast<uint4 *>(box)[k] = make_uint4(0, 0, 0, 0);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0 && live) {
                    const int32_t y = (int32_t)(ti.c_base / p.ldc + qrow0);
                    for (int rd = 0; rd < 2; rd++) {
                        const int64_t x = cbeg + 64 * rd;
                        if (x < ti.col_end) tma_store_2d(&tmC, (int32_t)x, y, box);
                    }
                    bulk_commit_group();
                }
                continue;
            }
            // this tile's scales, loaded before the accumulator wait so their
            // latency hides behind it: the lane's row scale and, for each of
            // the four 32-column chunks, the scale of column (chunk, lane)
            const float sa_v = live ? (p.sa_per_row ? __ldg(p.sa + ti.sa_base + qrow0 + lane) : __ldg(p.sa)) : 0.0f;
            float sbl4[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int64_t cc = cbeg + u * 32 + lane;
                sbl4[u] = p.sb_per_row ? (cc < ti.col_end ? __ldg(p.sb + ti.sb_base + cc) : 0.0f) : __ldg(p.sb);
            }
            if (!mbar_wait_bounded(&tfull[g], acc_phase, WAIT_LIMIT_NS, p.err, ERR_EPILOGUE_WAIT)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(g * BN) +
                                   (uint32_t)(half * (BN / 2));
            const int32_t y = (int32_t)(ti.c_base / p.ldc + qrow0);  // row of the [G*N][K] view
#pragma unroll
            for (int rd = 0; rd < 2; rd++) {  // round rd: columns 64 rd .. 64 rd + 63 of this warp's 128
                // the box's previous store must have read it before it is refilled
                if (lane == 0) bulk_wait_group_read0();
                __syncwarp();
#pragma unroll
                for (int cu = 0; cu < 2; cu++) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + 64 * rd + 32 * cu, r);
                    tmem_ld_wait();
                    if (rd == 1 && cu == 1) {
                        // the whole block is read: release the accumulator to the MMA warp
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&tempty[g]);
                    }
                    uint32_t packed[16];
                    const float sbv = sbl4[2 * rd + cu];
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        const float lo = __uint_as_float(r[2 * j]) * sa_v * __shfl_sync(0xffffffffu, sbv, 2 * j);
                        const float hi = __uint_as_float(r[2 * j + 1]) * sa_v * __shfl_sync(0xffffffffu, sbv, 2 * j + 1);
                        packed[j] = pack_bf16x2(lo, hi);
                    }
                    // 16-byte chunks 4 cu .. 4 cu + 3 of this lane's 128-byte row,
                    // 128-byte swizzle: chunk index XOR (row % 8)
                    uint8_t *brow = box + lane * 128;
#pragma unroll
                    for (int gg = 0; gg < 4; gg++) {
                        const int chunk = (cu * 4 + gg) ^ (lane & 7);
                        *reinterpret_cast<uint4 *>(brow + chunk * 16) =
                            make_uint4(packed[4 * gg], packed[4 * gg + 1], packed[4 * gg + 2], packed[4 * gg + 3]);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0 && live) {
                    const int64_t x = cbeg + 64 * rd;
                    if (x < ti.col_end) tma_store_2d(&tmC, (int32_t)x, y, box);
                    bulk_commit_group();
                }
            }
            acc_phase ^= 1;
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Dense GEMM on CTA pairs: 256 x 256 tiles computed by 2-SM tcgen05 MMAs.
//
// The two CTAs of a cluster each stage half of the A tile (128 rows) and
// half of the B tile (128 rows) at the same shared-memory offsets; the even
// CTA's single MMA thread issues tcgen05.mma.cta_group::2 (M = 256, N = 256),
// which reads both CTAs' halves and leaves each CTA's 128 rows of D in its
// own TMEM.  Per SM this halves the shared-memory footprint of B, so a stage
// is 32 KB and the ring holds 6 stages.  Both CTAs' TMA loads count on the
// even CTA's "full" barrier; the MMA thread's commits are multicast to both
// CTAs ("empty" frees a stage in both, "tmem full" starts both epilogues);
// both CTAs' epilogue warps arrive on the even CTA's "tmem empty".
// ---------------------------------------------------------------------------
constexpr int STAGES2 = 6;
constexpr int A2_STAGE_BYTES = 128 * BK;
constexpr int B2_STAGE_BYTES = 128 * BK;

struct SmemLayout2 {
    static constexpr int a_off = 0;
    static constexpr int b_off = STAGES2 * A2_STAGE_BYTES;
    static constexpr int bar_off = b_off + STAGES2 * B2_STAGE_BYTES;
    static constexpr int n_bars = 2 * STAGES2 + 2 + 2 + 1;
    static constexpr int slot_off = bar_off + n_bars * 8;
    static constexpr int stage_off = (slot_off + 16 + 127) / 128 * 128;
    static constexpr int total = stage_off + 8 * SmemLayout::stage_warp_bytes;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         GemmParams p, uint32_t idesc)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem + SmemLayout2::a_off;
    uint8_t *sB = smem + SmemLayout2::b_off;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SmemLayout2::bar_off);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES2;
    uint64_t *tfull = bars + 2 * STAGES2;
    uint64_t *tempty = tfull + 2;
    uint64_t *done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SmemLayout2::slot_off);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int64_t cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES2; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 16);  // 8 epilogue warps in each of the two CTAs
        }
        mbar_init(done, 1);
        fence_barrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers are initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int64_t total = p.total_tiles;
    const int num_m2 = (int)((p.M + 255) / 256);

    auto coords = [&](int64_t t, int &mb, int &nb) {
        if (p.m_fastest) {
            mb = (int)(t % num_m2);
            nb = (int)(t / num_m2);
        } else {
            nb = (int)(t % p.num_n_blk);
            mb = (int)(t / p.num_n_blk);
        }
    };

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        int stage = 0;
        uint32_t phase = 0;
        int issued_parity[STAGES2];
        for (int s = 0; s < STAGES2; s++) issued_parity[s] = -1;
        bool ok = true;
        for (int64_t t = cluster; t < total && ok; t += n_clusters) {
            int mb, nb;
            coords(t, mb, nb);
            for (int kb = 0; kb < p.num_k_blk; kb++) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1, WAIT_LIMIT_NS, p.err, ERR_PRODUCER_WAIT)) {
                    ok = false;
                    break;
                }
                if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (A2_STAGE_BYTES + B2_STAGE_BYTES));
                const uint32_t full_leader = mapa_shared(smem_u32(&full[stage]), 0);
                tma_load_2d_pair(sA + stage * A2_STAGE_BYTES, &tmA, kb * BK, mb * 256 + (int)rank * 128, full_leader);
                tma_load_2d_pair(sB + stage * B2_STAGE_BYTES, &tmB, kb * BK, nb * 256 + (int)rank * 128, full_leader);
                issued_parity[stage] = (int)phase;
                if (++stage == STAGES2) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // the even CTA's full barriers count both CTAs' copies: draining them
        // there covers the pair (the odd CTA waits at the final cluster barrier)
        if (leader)
            for (int s = 0; s < STAGES2; s++)
                if (issued_parity[s] >= 0)
                    mbar_wait_bounded(&full[s], (uint32_t)issued_parity[s], WAIT_LIMIT_NS, p.err, ERR_TEARDOWN_WAIT);
    } else if (warp == 1 && lane == 0 && leader) {
        // ---------------- MMA issuer (even CTA) ----------------
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int64_t t = cluster; t < total && ok; t += n_clusters) {
            if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, WAIT_LIMIT_NS, p.err, ERR_MMA_WAIT)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < p.num_k_blk; kb++) {
                if (!mbar_wait_bounded(&full[stage], phase, WAIT_LIMIT_NS, p.err, ERR_MMA_WAIT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(sA + stage * A2_STAGE_BYTES);
                const uint32_t b_addr = smem_u32(sB + stage * B2_STAGE_BYTES);
#pragma unroll
                for (int k = 0; k < BK / UMMA_K; k++)
                    mma_f8f6f4_pair(d_tmem, smem_desc_k128_sw128(a_addr + k * UMMA_K),
                                    smem_desc_k128_sw128(b_addr + k * UMMA_K), idesc, (kb | k) != 0);
                mma_commit_pair(&empty[stage], 0x3);
                if (++stage == STAGES2) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            mma_commit_pair(&tfull[acc], 0x3);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        mma_commit_pair_local(done);
        mbar_wait_bounded(done, 0, WAIT_LIMIT_NS, p.err, ERR_TEARDOWN_WAIT);
    } else if (warp >= 2) {
        // ---------------- epilogue (both CTAs) ----------------
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        uint8_t *stage = smem + SmemLayout2::stage_off + (warp - 2) * SmemLayout::stage_warp_bytes;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int64_t t = cluster; t < total; t += n_clusters) {
            int mb, nb;
            coords(t, mb, nb);
            TileInfo ti;
            ti.row0 = (int64_t)mb * 256 + rank * 128;
            ti.row_end = p.M;
            ti.col0 = (int64_t)nb * BN;
            ti.col_end = p.N;
            ti.c_base = 0;
            ti.sa_base = 0;
            ti.sb_base = 0;
            if (!mbar_wait_bounded(&tfull[acc], acc_phase, WAIT_LIMIT_NS, p.err, ERR_EPILOGUE_WAIT)) break;
            tc_fence_after();
            epilogue_tile(p, ti, tmem_base, (uint32_t)(acc * BN), q, half, lane, stage);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still touch its shared memory or TMEM
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps via the driver entry point (no link-time libcuda).
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
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

// 2D map over a row-major bf16 matrix [rows][cols] (row stride cols), box
// {64 elements, 32 rows}, 128-byte swizzle: the K-grouped epilogue's stores.
static bool make_map_c(CUtensorMap *map, void *base, int64_t rows, int64_t cols)
{
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static fp8_status_t launch_kgroup_tma(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mc,
                                      const GemmParams &p, int fa, int fb, int64_t grid, cudaStream_t st)
{
    const size_t smem = 1024 + SmemLayoutKT::misc_off + 8 * (size_t)(p.G + 1);
    cudaError_t e = cudaFuncSetAttribute(fp8_gemm_kgroup_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return cuda_fail_with(e);
    const uint32_t idesc = idesc_f8f6f4(fa, fb, BM, BN);
    fp8_gemm_kgroup_tma_kernel<<<(unsigned)grid, KT_THREADS, smem, st>>>(ma, mb, mc, p, idesc);
    return check_launch();
}

static size_t gemm_smem_bytes(int G) { return 1024 + SmemLayout::base_bytes + (G > 0 ? 8 * (size_t)(G + 1) : 0); }

template <int MODE>
static fp8_status_t launch_gemm(const CUtensorMap &ma, const CUtensorMap &mb, const GemmParams &p, int fa, int fb,
                                int64_t grid, cudaStream_t st)
{
    const size_t smem = gemm_smem_bytes(MODE == MODE_DENSE ? 0 : p.G);
    cudaError_t e = cudaFuncSetAttribute(fp8_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail_with(e);
    const uint32_t idesc = idesc_f8f6f4(fa, fb, BM, BN);
    fp8_gemm_kernel<MODE><<<(unsigned)grid, GEMM_THREADS, smem, st>>>(ma, mb, p, idesc);
    return check_launch();
}

static fp8_status_t launch_gemm_pair(const CUtensorMap &ma, const CUtensorMap &mb, const GemmParams &p, int fa,
                                     int fb, cudaStream_t st)
{
    const size_t smem = 1024 + SmemLayout2::total;
    cudaError_t e = cudaFuncSetAttribute(fp8_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail_with(e);
    // as many pairs as can be resident at once, never more than tiles
    static int max_pairs[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && max_pairs[dev] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (num_sms() / 2));
        cfg.blockDim = dim3(GEMM_THREADS);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_pair_kernel, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = num_sms() / 2;
        }
        max_pairs[dev] = n;
    }
    int64_t pairs = (dev >= 0 && dev < 64) ? max_pairs[dev] : num_sms() / 2;
    if (pairs > p.total_tiles) pairs = p.total_tiles;
    if (pairs < 1) pairs = 1;
    const uint32_t idesc = idesc_f8f6f4(fa, fb, 256, BN);
    fp8_gemm_pair_kernel<<<(unsigned)(2 * pairs), GEMM_THREADS, smem, st>>>(ma, mb, p, idesc);
    return check_launch();
}

static bool gemm_format_ok(int f) { return f == FP8_E4M3FN || f == FP8_E5M2; }

}  // namespace fp8gb

using namespace fp8gb;

extern "C" fp8_status_t fp8_scaled_gemm(const uint8_t *A, int fa, int64_t lda, const uint8_t *B, int fb, int64_t ldb,
                                        int64_t M, int64_t N, int64_t K, const float *sa, int sa_mode,
                                        const float *sb, int sb_mode, void *C_bf16, int64_t ldc, void *stream)
{
    if (!A || !B || !sa || !sb || !C_bf16) return FP8_ERR_INVALID_ARG;
    if (fa == FP8_E4M3FNUZ || fb == FP8_E4M3FNUZ || fa == FP8_E5M2FNUZ || fb == FP8_E5M2FNUZ)
        return FP8_ERR_UNSUPPORTED;
    if (!gemm_format_ok(fa) || !gemm_format_ok(fb)) return FP8_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1 || lda < K || ldb < K || ldc < N) return FP8_ERR_INVALID_ARG;
    if ((sa_mode != FP8_SCALE_TENSOR && sa_mode != FP8_SCALE_PER_ROW) ||
        (sb_mode != FP8_SCALE_TENSOR && sb_mode != FP8_SCALE_PER_ROW))
        return FP8_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FP8_ERR_INVALID_ARG;
    if (K % 16 != 0 || lda % 16 != 0 || ldb % 16 != 0) return FP8_ERR_ALIGNMENT;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C_bf16, 2) || !aligned(sa, 4) || !aligned(sb, 4))
        return FP8_ERR_ALIGNMENT;

    GemmParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.sa = sa;
    p.sb = sb;
    p.sa_per_row = sa_mode == FP8_SCALE_PER_ROW;
    p.sb_per_row = sb_mode == FP8_SCALE_PER_ROW;
    p.C = static_cast<uint16_t *>(C_bf16);
    p.ldc = ldc;
    p.c_vec16 = ldc % 8 == 0 && aligned(C_bf16, 16);
    p.num_m_blk = (int)((M + BM - 1) / BM);
    p.num_n_blk = (int)((N + BN - 1) / BN);
    p.num_k_blk = (int)((K + BK - 1) / BK);
    // sweep the dimension whose operand is smaller fastest, so that operand
    // stays resident in L2 while the other streams through once
    p.m_fastest = M <= N;
    p.total_tiles = (int64_t)p.num_m_blk * p.num_n_blk;
    p.err = device_error_word();
    p.offsets = nullptr;
    p.G = 0;

    CUtensorMap ma, mb;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (M > 128) {
        // CTA pairs with 256 x 256 tiles
        const int64_t num_m2 = (M + 255) / 256;
        p.total_tiles = num_m2 * p.num_n_blk;
        p.m_fastest = M <= N;
        if (!make_map(&ma, A, M, K, lda, 128) || !make_map(&mb, B, N, K, ldb, 128)) return FP8_ERR_CUDA;
        return launch_gemm_pair(ma, mb, p, fa, fb, st);
    }
    if (!make_map(&ma, A, M, K, lda, BM) || !make_map(&mb, B, N, K, ldb, BN)) return FP8_ERR_CUDA;
    const int64_t grid = p.total_tiles < num_sms() ? p.total_tiles : num_sms();
    return launch_gemm<MODE_DENSE>(ma, mb, p, fa, fb, grid, st);
}

extern "C" fp8_status_t fp8_grouped_gemm(int mode, const uint8_t *A, int fa, const uint8_t *B, int fb,
                                         const int32_t *group_offsets, int G, int64_t M_total, int64_t N, int64_t K,
                                         const float *sa, int sa_mode, const float *sb, int sb_mode, void *C_bf16,
                                         int64_t ld_T, void *stream)
{
    if (!A || !B || !sa || !sb || !C_bf16 || !group_offsets) return FP8_ERR_INVALID_ARG;
    if (fa == FP8_E4M3FNUZ || fb == FP8_E4M3FNUZ || fa == FP8_E5M2FNUZ || fb == FP8_E5M2FNUZ)
        return FP8_ERR_UNSUPPORTED;
    if (!gemm_format_ok(fa) || !gemm_format_ok(fb)) return FP8_ERR_INVALID_ARG;
    if (mode != FP8_GROUPED_M && mode != FP8_GROUPED_K && mode != FP8_GROUPED_M_BT) return FP8_ERR_INVALID_ARG;
    if (G < 1 || G > MAX_GROUPS || M_total < 0 || N < 1 || K < 1) return FP8_ERR_INVALID_ARG;
    if ((sa_mode != FP8_SCALE_TENSOR && sa_mode != FP8_SCALE_PER_ROW) ||
        (sb_mode != FP8_SCALE_TENSOR && sb_mode != FP8_SCALE_PER_ROW))
        return FP8_ERR_INVALID_ARG;
    if (M_total > INT32_MAX || N > INT32_MAX || K > INT32_MAX || (int64_t)G * N > INT32_MAX)
        return FP8_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C_bf16, 2) || !aligned(sa, 4) || !aligned(sb, 4))
        return FP8_ERR_ALIGNMENT;

    GemmParams p{};
    p.M = M_total;
    p.N = N;
    p.K = K;
    p.sa = sa;
    p.sb = sb;
    p.sa_per_row = sa_mode == FP8_SCALE_PER_ROW;
    p.sb_per_row = sb_mode == FP8_SCALE_PER_ROW;
    p.C = static_cast<uint16_t *>(C_bf16);
    p.offsets = group_offsets;
    p.G = G;
    p.err = device_error_word();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUtensorMap ma, mb;
    const int64_t grid = num_sms();

    if (mode == FP8_GROUPED_M || mode == FP8_GROUPED_M_BT) {
        if (K % 16 != 0) return FP8_ERR_ALIGNMENT;
        p.ldc = N;
        p.c_vec16 = N % 8 == 0 && aligned(C_bf16, 16);
        p.num_m_blk = 0;
        p.num_n_blk = (int)((N + BN - 1) / BN);
        p.num_k_blk = (int)((K + BK - 1) / BK);
        p.kpad = (K + 31) / 32 * 32;
        if (mode == FP8_GROUPED_M_BT) {
            if (ld_T % 16 != 0) return FP8_ERR_ALIGNMENT;
            if (ld_T < (int64_t)G * p.kpad || ld_T > INT32_MAX) return FP8_ERR_INVALID_ARG;
            p.b_trans = 1;
        }
        if (M_total == 0) return FP8_OK;
        if (!make_map(&ma, A, M_total, K, K, BM)) return FP8_ERR_CUDA;
        if (p.b_trans ? !make_map(&mb, B, N, (int64_t)G * p.kpad, ld_T, BN)
                      : !make_map(&mb, B, (int64_t)G * N, K, K, BN))
            return FP8_ERR_CUDA;
        return launch_gemm<MODE_MGROUP>(ma, mb, p, fa, fb, grid, st);
    }
    // K-grouped (wgrad): C[e] = A_e [N][m_e] . B_e [K][m_e]^T
    if (ld_T < 16 || ld_T % 16 != 0) return FP8_ERR_ALIGNMENT;
    p.ldc = K;
    p.c_vec16 = K % 8 == 0 && aligned(C_bf16, 16);  // then N*K % 8 == 0 too
    p.ld_T = ld_T;
    p.num_m_blk = (int)((N + BM - 1) / BM);
    p.num_n_blk = (int)((K + BN - 1) / BN);
    p.num_k_blk = 0;
    if (!make_map(&ma, A, N, ld_T, ld_T, BM) || !make_map(&mb, B, K, ld_T, ld_T, BN)) return FP8_ERR_CUDA;
    if (N % 32 == 0 && K % 8 == 0 && aligned(C_bf16, 16) && (int64_t)G * N <= INT32_MAX) {
        CUtensorMap mc;
        if (!make_map_c(&mc, C_bf16, (int64_t)G * N, K)) return FP8_ERR_CUDA;
        return launch_kgroup_tma(ma, mb, mc, p, fa, fb, grid, st);
    }
    return launch_gemm<MODE_KGROUP>(ma, mb, p, fa, fb, grid, st);
}
