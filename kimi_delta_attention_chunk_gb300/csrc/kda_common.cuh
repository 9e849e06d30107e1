// Shared device helpers of the KDA kernels (element loads/stores, launch
// plumbing).  Nothing here is shared with the CPU oracle.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr float kGateLowerBound = -5.0f;

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

template <typename T> __device__ __forceinline__ float ld(const T* p, int64_t i) {
    return to_f32<T>(p[i]);
}

// Rank of sequence m among N sequences when ordered longest first (ties by
// index).  Used to hand the longest sequences to the lowest block indices so
// that the block scheduler starts them first.
__device__ __forceinline__ int seq_len_clamped(const int32_t* cu, int n, int T) {
    int b = min(max(cu[n], 0), T);
    int e = min(max(cu[n + 1], 0), T);
    return e > b ? e - b : 0;
}

}  // namespace kda

// Host-side helpers -------------------------------------------------------
namespace kda_host {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline kda_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda_host
