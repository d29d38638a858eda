// update.cu -- the delayed-scaling amax-history roll and scale update for
// many tensors in one launch.
//
// Method: "FP8 training for Flux models", Configuration > Key FP8 Parameters
// (fp8_amax_history_len: the window; fp8_amax_compute_algo: "most_recent" or
// "max"; fp8_margin) and its Numerical verification status list, which names
// a fused delayed-scale update.
//
// One thread block per tensor: the row is read once into shared memory while
// the window maximum is reduced, then written back shifted by one slot with
// slot 0 cleared.  The new scale is computed by thread 0 in fp32 (IEEE
// divide), so the next step's quantize reads it straight from device memory
// with no host round trip.
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8gb.h"
#include "fp8gb_device.cuh"
#include "fp8gb_host.h"

namespace fp8gb {

constexpr int UPD_THREADS = 256;
constexpr int UPD_MAX_L = 32768;

__global__ void __launch_bounds__(UPD_THREADS)
    update_history_kernel(float *hist, float *scale, float *scale_inv, const uint8_t *fmt, int L, int algo,
                          int margin, int32_t *nonfinite_count)
{
    extern __shared__ float row[];
    __shared__ float wmax[UPD_THREADS / 32];
    __shared__ int wnan[UPD_THREADS / 32];
    const int i = blockIdx.x;
    float *H = hist + (int64_t)i * L;

    float m = -INFINITY;
    int has_nan = 0;
    for (int j = threadIdx.x; j < L; j += UPD_THREADS) {
        const float v = H[j];
        row[j] = v;
        if (v != v)
            has_nan = 1;
        else
            m = fmaxf(m, v);
    }
    for (int d = 16; d > 0; d >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
        has_nan |= __shfl_xor_sync(0xffffffffu, has_nan, d);
    }
    if ((threadIdx.x & 31) == 0) {
        wmax[threadIdx.x >> 5] = m;
        wnan[threadIdx.x >> 5] = has_nan;
    }
    __syncthreads();

    if (threadIdx.x == 0) {
        float a;
        if (algo == FP8_AMAX_MOST_RECENT) {
            a = row[0];
        } else {
            // max over the window; NaN anywhere gives NaN
            float mm = -INFINITY;
            int nn = 0;
            for (int w = 0; w < UPD_THREADS / 32; w++) {
                mm = fmaxf(mm, wmax[w]);
                nn |= wnan[w];
            }
            a = nn ? __int_as_float(0x7fc00000) : mm;
        }
        if (isfinite(a) && a > 0.0f) {
            float s = __fdiv_rn(fp8_max_of(fmt[i]), a);
            s = __fmul_rn(s, pow2_neg(margin));
            if (isinf(s)) s = 3.402823466e38f;
            scale[i] = s;
            scale_inv[i] = recip_rn(s);
        } else if (!isfinite(a) && nonfinite_count) {
            nonfinite_count[i] += 1;
        }
    }
    // roll: H[j] = H[j-1] for j >= 1, H[0] = 0 (reads came from shared memory)
    for (int j = threadIdx.x; j < L; j += UPD_THREADS) H[j] = j == 0 ? 0.0f : row[j - 1];
}

}  // namespace fp8gb

using namespace fp8gb;

extern "C" fp8_status_t fp8_update_amax_history(float *hist, float *scale, float *scale_inv, const uint8_t *fmt,
                                                int n, int L, int algo, int margin, int32_t *nonfinite_count,
                                                void *stream)
{
    if (!hist || !scale || !scale_inv || !fmt) return FP8_ERR_INVALID_ARG;
    if (n < 1 || L < 1 || L > UPD_MAX_L) return FP8_ERR_INVALID_ARG;
    if (algo != FP8_AMAX_MOST_RECENT && algo != FP8_AMAX_MAX) return FP8_ERR_INVALID_ARG;
    if (margin < 0 || margin > 64) return FP8_ERR_INVALID_ARG;
    if (!aligned(hist, 4) || !aligned(scale, 4) || !aligned(scale_inv, 4)) return FP8_ERR_ALIGNMENT;
    const size_t smem = sizeof(float) * (size_t)L;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(update_history_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return cuda_fail_with(e);
    }
    update_history_kernel<<<n, UPD_THREADS, smem, static_cast<cudaStream_t>(stream)>>>(
        hist, scale, scale_inv, fmt, L, algo, margin, nonfinite_count);
    return check_launch();
}
