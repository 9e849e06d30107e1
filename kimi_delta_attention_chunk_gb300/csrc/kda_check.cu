// Debug range check of an input tensor (the prefill's precondition: every log
// decay g in [-5, 0], the K3 gate_lower_bound): a grid-stride pass that sets a
// caller-owned device status word to KDA_ERR_RANGE when any element lies outside
// [lo, hi] or is NaN; the word is left at KDA_OK otherwise.
#include "kda_chunk.h"
#include "kda_common.cuh"

namespace kda {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) check_range_kernel(const T* __restrict__ x, int64_t n, float lo, float hi,
                                                          int32_t* status) {
    bool bad = false;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = to_f32<T>(x[i]);
        bad |= !(v >= lo && v <= hi);  // NaN fails both comparisons
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicExch(status, (int32_t)KDA_ERR_RANGE);
}

}  // namespace

cudaError_t check_range(kda_dtype dt, const void* x, int64_t n, float lo, float hi, int32_t* status,
                        cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
    if (e != cudaSuccess || n == 0) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t want = (n + 255) / 256, cap = (int64_t)sms * 8;
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    if (dt == KDA_BF16)
        check_range_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), n, lo, hi,
                                                                status);
    else
        check_range_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(x), n, lo, hi, status);
    return cudaGetLastError();
}

}  // namespace kda
