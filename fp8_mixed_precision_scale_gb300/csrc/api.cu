// api.cu -- library-wide entry points: status strings, the device error word,
// fp8_sync_status, the bounded-wait self test and the grouped-layout helper.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "fp8gb.h"
#include "fp8gb_device.cuh"
#include "fp8gb_host.h"

namespace fp8gb {

// The library's error word; one instance per device that loads the library.
__device__ unsigned int g_error_word = 0;

constexpr int MAX_DEVICES = 64;
static std::mutex g_mu;
static int g_sms[MAX_DEVICES];
static unsigned int *g_err_ptr[MAX_DEVICES];
static bool g_err_ready[MAX_DEVICES];
static thread_local char g_last_cuda_error[256] = "no error";

fp8_status_t cuda_fail_with(cudaError_t e)
{
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return FP8_ERR_CUDA;
}

int num_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

unsigned int *device_error_word()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ready[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_err_ptr[dev] = static_cast<unsigned int *>(p);
        g_err_ready[dev] = true;
    }
    return g_err_ptr[dev];
}

// A single thread block waits on a barrier that nothing completes.
__global__ void selftest_wait_kernel(uint64_t limit_ns, unsigned int *err)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, limit_ns, err, ERR_SELFTEST_WAIT);
}

}  // namespace fp8gb

using namespace fp8gb;

extern "C" const char *fp8_status_string(fp8_status_t s)
{
    switch (s) {
    case FP8_OK: return "FP8_OK";
    case FP8_ERR_INVALID_ARG: return "FP8_ERR_INVALID_ARG";
    case FP8_ERR_UNSUPPORTED: return "FP8_ERR_UNSUPPORTED";
    case FP8_ERR_ALIGNMENT: return "FP8_ERR_ALIGNMENT";
    case FP8_ERR_CUDA: return "FP8_ERR_CUDA";
    case FP8_ERR_TIMEOUT: return "FP8_ERR_TIMEOUT";
    }
    return "FP8_ERR_UNKNOWN";
}

extern "C" const char *fp8_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" const char *fp8_version(void) { return "fp8gb 0.1 sm_103a"; }

extern "C" int64_t fp8_group_padded_offsets(const int32_t *host_offsets, int G, int align, int64_t *host_padded_out)
{
    if (!host_offsets || G < 1 || align < 16 || align % 16 != 0) return -1;
    int64_t acc = 0;
    for (int e = 0; e < G; e++) {
        const int64_t m = (int64_t)host_offsets[e + 1] - host_offsets[e];
        if (m < 0) return -1;
        if (host_padded_out) host_padded_out[e] = acc;
        acc += (m + align - 1) / align * align;
    }
    if (host_padded_out) host_padded_out[G] = acc;
    return acc;
}

extern "C" fp8_status_t fp8_sync_status(void *stream)
{
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail_with(e);
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word));
    if (e != cudaSuccess) return cuda_fail_with(e);
    if (word != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail_with(e);
        // a wait that gave up outranks malformed device-side offsets
        return (word & ~(ERR_BAD_OFFSETS | ERR_BAD_INDEX)) ? FP8_ERR_TIMEOUT : FP8_ERR_INVALID_ARG;
    }
    return FP8_OK;
}

extern "C" fp8_status_t fp8_selftest_bounded_wait(int64_t wait_ns, void *stream)
{
    if (wait_ns < 1000 || wait_ns > 10000000000LL) return FP8_ERR_INVALID_ARG;
    unsigned int *err = device_error_word();
    if (!err) return cuda_fail();
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)wait_ns, err);
    return check_launch();
}
