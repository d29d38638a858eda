// fp8gb_device.cuh -- device helpers shared by the library's kernels:
// the scale formula, FP8 conversions, the device error word, bounded
// mbarrier waits, and thin inline-PTX wrappers for TMA and tcgen05.
//
// Target: sm_103a only (tcgen05 / TMEM / TMA).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8gb.h"

namespace fp8gb {

// ---------------------------------------------------------------------------
// Device error word (one per device, defined in api.cu; kernels receive its
// address): set by a bounded wait that gave up or by malformed device-side
// arguments; read and cleared by fp8_sync_status().
// ---------------------------------------------------------------------------
enum : unsigned int {
    ERR_PRODUCER_WAIT = 1u,
    ERR_MMA_WAIT = 2u,
    ERR_EPILOGUE_WAIT = 4u,
    ERR_TEARDOWN_WAIT = 8u,
    ERR_SELFTEST_WAIT = 16u,
    ERR_BAD_OFFSETS = 32u,
    ERR_BAD_INDEX = 64u,  // a gather index outside the source rows
    ERR_GRID_WAIT = 128u, // a grid-wide barrier of a cooperative launch gave up
};

__device__ __forceinline__ void record_error(unsigned int *err, unsigned int bits)
{
    if (err) atomicOr(err, bits);
}

// ---------------------------------------------------------------------------
// Scale arithmetic ("FP8 training for Flux models", Key FP8 Parameters:
// scale = fp8_max / amax / 2^margin).  IEEE fp32 operations, no contraction.
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ float fp8_max_of(int fmt)
{
    return (fmt == FP8_E5M2 || fmt == FP8_E5M2FNUZ) ? 57344.0f : (fmt == FP8_E4M3FNUZ ? 240.0f : 448.0f);
}

__device__ __forceinline__ float pow2_neg(int margin)  // 2^-margin, 0 <= margin <= 126
{
    return __int_as_float((127 - margin) << 23);
}

// Current scaling: amax == 0 or non-finite -> 1; overflow -> FLT_MAX.
__device__ __forceinline__ float scale_from_amax(float amax, float fmax, int margin)
{
    if (!(amax > 0.0f) || !isfinite(amax)) return 1.0f;
    float s = __fdiv_rn(fmax, amax);
    s = __fmul_rn(s, pow2_neg(margin));
    if (isinf(s)) s = 3.402823466e38f;
    return s;
}

__device__ __forceinline__ float recip_rn(float s) { return __fdiv_rn(1.0f, s); }

// ---------------------------------------------------------------------------
// FP8 conversion: saturating, round-to-nearest-even, two fp32 at a time.
// Result: low byte = lo, high byte = hi.
// ---------------------------------------------------------------------------
// e4m3fnuz (bias 8) from the e4m3fn conversion: fnuz code c is worth half
// of e4m3fn code c for every finite code, so fnuz(v) = e4m3fn(2 v) (doubling
// is exact and preserves the rounding decision) with the format's own rules
// on top: |v| above 232 (the tie between 224 and 240 rounds to the even code
// 0x7E) gives +-240 = 0x7F / 0xFF, which e4m3fn reserves for NaN; NaN gives
// the single fnuz NaN 0x80; and a negative zero becomes the unsigned zero.
__device__ __forceinline__ uint32_t fnuz_fix(uint32_t code, float v)
{
    if (v != v) return 0x80u;
    if (fabsf(v) > 232.0f) return v < 0.0f ? 0xFFu : 0x7Fu;
    return code == 0x80u ? 0x00u : code;
}

// e5m2fnuz (bias 16) likewise: fnuz code c is worth half of e5m2 code c, so
// fnuz(v) = e5m2(2 v) while 2 v stays inside e5m2's finite range.  The top
// fnuz binade [2^15, 57344] has no finite e5m2 counterpart at 2 v, so for
// |v| >= 2^14 the code comes from e5m2(v / 2) two binades up (+8: two steps
// of the 2-bit mantissa field); v / 2 is normal there, so the rounding is
// the same.  Above 57344 (and +-Inf) it saturates; NaN gives 0x80; a
// negative zero becomes the unsigned zero.
__device__ __forceinline__ uint32_t e5m2_code(float v)
{
    unsigned short r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xFFu;
}

__device__ __forceinline__ uint32_t e5m2fnuz_fix(uint32_t code, float v)
{
    if (v != v) return 0x80u;
    const float a = fabsf(v);
    if (a > 57344.0f) return v < 0.0f ? 0xFFu : 0x7Fu;
    if (a >= 16384.0f) return e5m2_code(v * 0.5f) + 8u;
    return code == 0x80u ? 0x00u : code;
}

template <int FMT>
__device__ __forceinline__ uint32_t cvt2(float lo, float hi)
{
    unsigned short r;
    if constexpr (FMT == FP8_E5M2) {
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    } else if constexpr (FMT == FP8_E4M3FNUZ) {
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi * 2.0f), "f"(lo * 2.0f));
        return fnuz_fix(r & 0xFFu, lo) | (fnuz_fix(r >> 8, hi) << 8);
    } else if constexpr (FMT == FP8_E5M2FNUZ) {
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi * 2.0f), "f"(lo * 2.0f));
        return e5m2fnuz_fix(r & 0xFFu, lo) | (e5m2fnuz_fix(r >> 8, hi) << 8);
    } else {
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    }
    return (uint32_t)r;
}

// bf16 pair (one 32-bit word: element 0 in the low half) -> two fp32.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// |x| bit patterns of a bf16 pair, max'ed per half: NaN patterns (0x7F81..)
// are above Inf (0x7F80) so NaN propagates through an unsigned max.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w)
{
    return __vmaxu2(acc, w & 0x7FFF7FFFu);
}

// Fold the two halves of a packed |bf16| max into the fp32 bit pattern of
// the larger one (bf16 -> fp32 is exact, so the order is preserved).
__device__ __forceinline__ uint32_t fold_absmax(uint32_t acc)
{
    uint32_t a = acc & 0xFFFFu, b = acc >> 16;
    return (a > b ? a : b) << 16;
}

// ---------------------------------------------------------------------------
// Shared-memory addresses and mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase of `parity` to complete.  Gives up after about
// limit_ns of wall time (checked every 256 polls), records `err_bits` and
// returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                                  unsigned int *err, unsigned int err_bits)
{
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && global_timer_ns() - t0 > limit_ns) {
            record_error(err, err_bits);
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) -- 2D tile load into shared memory, completing
// on an mbarrier by transaction bytes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int32_t x, int32_t y,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(smem_dst)), "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in TMEM)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *slot_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile stored as rows of
// 128 bytes with the 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B): 8-row groups are 1024 bytes apart (SBO),
// LBO unused for this layout, descriptor version 1, layout type 2 (128B).
__device__ __forceinline__ uint64_t smem_desc_k128_sw128(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);  // start address, bits 0-13
    d |= (uint64_t)1 << 16;                        // leading byte offset (unused), bits 16-29
    d |= (uint64_t)(1024 >> 4) << 32;              // stride byte offset, bits 32-45
    d |= (uint64_t)1 << 46;                        // version, bits 46-47
    d |= (uint64_t)2 << 61;                        // swizzle 128B, bits 61-63
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4, fp32 accumulate,
// both operands K-major, dense.  fa / fb: 0 = E4M3, 1 = E5M2.
__host__ __device__ constexpr uint32_t idesc_f8f6f4(int fa, int fb, int M, int N)
{
    return (1u << 4)                         // D format f32
           | ((uint32_t)fa << 7)             // A format
           | ((uint32_t)fb << 10)            // B format
           | ((uint32_t)(N >> 3) << 17)      // N / 8
           | ((uint32_t)(M >> 4) << 24);     // M / 16
}

__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp receives lane
// (quarter*32 + i), columns col .. col+31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// CTA pairs (thread-block clusters of 2) for the 2-SM tcgen05 MMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address, in the cluster's shared window, of this CTA's shared variable at
// `local` as seen in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t *slot_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// One 2-SM MMA (issued by the pair's even CTA): each CTA supplies its half
// of A (M/2 rows) and of B (N/2 rows) at the same shared-memory offsets and
// receives its M/2 rows of D in its own TMEM.
__device__ __forceinline__ void mma_f8f6f4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at `bar`'s offset in every CTA of `cta_mask` once
// the pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t *bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

__device__ __forceinline__ void mma_commit_pair_local(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// TMA 2D load into this CTA's shared memory whose completion is counted on
// an mbarrier that may live in the peer CTA (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void *smem_dst, const CUtensorMap *map, int32_t x, int32_t y,
                                                 uint32_t bar_cluster_addr)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(smem_dst)), "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar_cluster_addr)
        : "memory");
}

// ---------------------------------------------------------------------------
// Block-scaled MMA (tcgen05.mma kind::mxf8f6f4, E8M0 scales in TMEM)
// ---------------------------------------------------------------------------
// Plain bulk copy global -> shared (no tensor map), completing on an mbarrier
// by transaction bytes; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(smem_dst)), "l"((uint64_t)gsrc), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Shared-memory descriptor of a 32-row x 16-byte block without swizzle
// (8-row core matrices of 128 contiguous bytes, 128 bytes apart): the source
// of tcgen05.cp 32x128b.
__device__ __forceinline__ uint64_t smem_desc_sf(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)(128 >> 4) << 32;               // stride byte offset: next 8 rows
    d |= (uint64_t)1 << 46;                        // version; layout type 0 (no swizzle)
    return d;
}

// Copy 32 lanes x 128 bits from shared memory into TMEM columns
// taddr .. taddr+3, replicated into all four lane quarters (warpx4).
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with E8M0 block scales, fp32
// accumulate, K-major operands: formats at bits 7 / 10, N/8 at bit 17, the
// scale type (E8M0 = 1) at bit 23, M/16 at bit 24; the byte of the scale word
// used by an MMA (its 32-element block within a 128-element K tile) is
// selected by the scale-factor ids, B's at bit 4 and A's at bit 29.
__host__ __device__ constexpr uint32_t idesc_mxf8f6f4(int fa, int fb, int M, int N)
{
    return ((uint32_t)fa << 7) | ((uint32_t)fb << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(M >> 4) << 24);
}

__host__ __device__ constexpr uint32_t idesc_sf_ids(uint32_t idesc, uint32_t a_id, uint32_t b_id)
{
    return idesc | (b_id << 4) | (a_id << 29);
}

// Scale factors for A row m: TMEM lane m, column sfa + m / 32; for B row n:
// column sfb + n / 32 in every lane quarter (lane 32q + n % 32).
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// TMA tile store shared -> global (bulk async group of the issuing thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int32_t x, int32_t y, const void *smem_src)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(smem_src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until the issuing thread's committed stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_group_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// wait until they have completed
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Two fp32 -> packed bf16x2 (round to nearest even); lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---------------------------------------------------------------------------
// Scaled conversion of eight bf16 (one 16-byte word) to eight FP8 codes (two
// words, bytes in element order): each element times its scale in IEEE fp32
// (round to nearest), then the saturating round-to-nearest-even conversion.
// Two products per mul.rn.f32x2 and four codes per packed word keep the
// instruction count per element low (the cast passes run at HBM speed).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mul2_rn(float &a, float &b, float sa, float sb)
{
    asm("{.reg .b64 x, s, r;\n\t"
        "mov.b64 x, {%0, %1};\n\t"
        "mov.b64 s, {%2, %3};\n\t"
        "mul.rn.f32x2 r, x, s;\n\t"
        "mov.b64 {%0, %1}, r;}"
        : "+f"(a), "+f"(b)
        : "f"(sa), "f"(sb));
}

template <int FMT>
__device__ __forceinline__ uint32_t cvt4(float a, float b, float c, float d)
{
    uint32_t r;
    if constexpr (FMT == FP8_E4M3FN) {
        asm("{.reg .b16 l, h;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n\t"
            "mov.b32 %0, {l, h};}"
            : "=r"(r)
            : "f"(a), "f"(b), "f"(c), "f"(d));
    } else if constexpr (FMT == FP8_E5M2) {
        asm("{.reg .b16 l, h;\n\t"
            "cvt.rn.satfinite.e5m2x2.f32 l, %2, %1;\n\t"
            "cvt.rn.satfinite.e5m2x2.f32 h, %4, %3;\n\t"
            "mov.b32 %0, {l, h};}"
            : "=r"(r)
            : "f"(a), "f"(b), "f"(c), "f"(d));
    } else {
        r = cvt2<FMT>(a, b) | (cvt2<FMT>(c, d) << 16);
    }
    return r;
}

template <int FMT>
__device__ __forceinline__ uint2 cvt8_scaled(const uint4 &v, const float (&s)[8])
{
    float f[8] = {bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y),
                  bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w)};
#pragma unroll
    for (int j = 0; j < 8; j += 2) mul2_rn(f[j], f[j + 1], s[j], s[j + 1]);
    return make_uint2(cvt4<FMT>(f[0], f[1], f[2], f[3]), cvt4<FMT>(f[4], f[5], f[6], f[7]));
}

// the same with one scale for all eight
template <int FMT>
__device__ __forceinline__ uint2 cvt8_scaled(const uint4 &v, float s)
{
    const float ss[8] = {s, s, s, s, s, s, s, s};
    return cvt8_scaled<FMT>(v, ss);
}

// ---------------------------------------------------------------------------
// SwiGLU element function shared by the fused MoE prologues of the MX and
// the rowwise quantizers.
// ---------------------------------------------------------------------------

// silu(g) * u in fp32, with sigma(g) = 1 / (1 + e^-g) formed from t = e^-|g|
// (never overflows): sigma = 1 / (1 + t) for g >= 0, t / (1 + t) for g < 0.
// For g < 0 the product is carried scaled by 2^126 (t is computed as 2^126
// e^-|g|, a normal fp32 for |g| < 174) and unscaled by the last multiply,
// applied to u first when |u| >= 1, so no intermediate overflows or turns
// subnormal before the end.  __expf and __fdividef (1 + t lies in [1, 2])
// err by far less than 2^-9 relative, so the bf16 rounding of the result is
// within one bf16 ulp of the exact bf16_rne(silu(g) * u) for every g when
// |u| <= 2^110 (NaN, +-Inf and the sign of zero as IEEE arithmetic gives
// them; silu(-Inf) = -0).
__device__ __forceinline__ float swiglu1(float g, float u)
{
    constexpr float LN2_X126 = 87.3365479f;  // 126 ln 2: e^(x + 126 ln 2) = 2^126 e^x
    const float t = __expf(LN2_X126 - fabsf(g));
    const float r = __fdividef(1.0f, fmaf(t, 0x1p-126f, 1.0f));
    // both signs' forms are evaluated and one is selected: the signs of a
    // warp's elements differ, and a branch per element diverges
    const float pos = (g * r) * u;
    const float s = t == 0.0f ? -0.0f : g * (t * r);  // 2^126 silu(g); t == 0 also for g = -Inf
    const float neg = fabsf(u) >= 1.0f ? s * (u * 0x1p-126f) : (s * u) * 0x1p-126f;
    return g >= 0.0f ? pos : neg;
}

// h = bf16(silu(g) * u) for a packed pair: one round-to-nearest-even
// conversion of both products (a NaN product becomes the canonical NaN).
__device__ __forceinline__ uint32_t swiglu2(uint32_t g2, uint32_t u2)
{
    return pack_bf16x2(swiglu1(bf16lo(g2), bf16lo(u2)), swiglu1(bf16hi(g2), bf16hi(u2)));
}

// ---------------------------------------------------------------------------
// MX scale layout: word (four E8M0 codes, one per 32-element block of a
// 128-element K tile) of scale row r in K tile kt, for R128 scale rows per K
// tile (a multiple of 128).  Each 128-row block is 512 contiguous bytes in the
// order a tcgen05.cp 32x128b copy reads them: row 32 j + L at lane L, word j.
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int64_t mx_scale_word(int64_t kt, int64_t r, int64_t R128)
{
    return kt * R128 + (r & ~(int64_t)127) + ((r & 31) << 2) + ((r >> 5) & 3);
}

__host__ __device__ __forceinline__ int64_t round_up_128(int64_t v) { return (v + 127) / 128 * 128; }

}  // namespace fp8gb
