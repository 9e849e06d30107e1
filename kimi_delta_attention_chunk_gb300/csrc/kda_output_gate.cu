// Output gate of the KDA layer, applied to the prefill's (or decode's) fp32 o:
// per (token, head) row of V values
//
//     out = o / sqrt(mean(o^2) + eps) * w * sigmoid(gate)
//
// ("kimi-k3-mlx" review, section "Attention is 93 layers ...": KDA carries a
// full-rank output gate; "NeMo AutoModel draft_kimi_k3", module description:
// K3's norms are RMS norms with the variance in fp32, its output gates sigmoid
// gates.)  The op streams o, gate and out once through HBM: one warp per row,
// each lane holding V/32 consecutive values (one 16-byte load of o), the
// row's sum of squares reduced with warp shuffles.
#include "kda_chunk.h"
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kRowsPerBlock = 8;  // 256 threads

// E consecutive values of a row (E = 2 or 4) as floats.
template <int E> struct Vec;
template <> struct Vec<4> {
    __device__ static void load(const float* p, float* x) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
    __device__ static void load(const __nv_bfloat16* p, float* x) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xffff0000u);
        x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xffff0000u);
    }
    __device__ static void store(float* p, const float* x) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
    __device__ static void store(__nv_bfloat16* p, const float* x) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
        *reinterpret_cast<uint2*>(p) = make_uint2(*reinterpret_cast<const uint32_t*>(&a),
                                                  *reinterpret_cast<const uint32_t*>(&b));
    }
};
template <> struct Vec<2> {
    __device__ static void load(const float* p, float* x) {
        const float2 v = *reinterpret_cast<const float2*>(p);
        x[0] = v.x; x[1] = v.y;
    }
    __device__ static void load(const __nv_bfloat16* p, float* x) {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
        x[0] = __uint_as_float(v << 16); x[1] = __uint_as_float(v & 0xffff0000u);
    }
    __device__ static void store(float* p, const float* x) {
        *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
    }
    __device__ static void store(__nv_bfloat16* p, const float* x) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
        *reinterpret_cast<__nv_bfloat162*>(p) = a;
    }
};

template <typename TG, typename TOut, int V>
__global__ void __launch_bounds__(kRowsPerBlock * 32)
output_gate_kernel(const float* o, const TG* __restrict__ gate, const float* __restrict__ w, float eps,
                   int64_t rows, TOut* out) {
    constexpr int E = V / 32;
    const int lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * kRowsPerBlock;
    float wv[E];
    if (w != nullptr) {
        Vec<E>::load(w + lane * E, wv);
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) wv[e] = 1.f;
    }
    for (int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5); row < rows; row += stride) {
        const int64_t base = row * V + lane * E;
        float x[E], gv[E];
        Vec<E>::load(o + base, x);
        Vec<E>::load(gate + base, gv);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss += x[e] * x[e];
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
        const float inv = rsqrtf(ss * (1.f / V) + eps);
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] = x[e] * inv * wv[e] * __fdividef(1.f, 1.f + __expf(-gv[e]));
        Vec<E>::store(out + base, x);
    }
}

template <typename TG, typename TOut>
cudaError_t launch_v(int V, const float* o, const void* gate, const float* w, float eps, int64_t rows,
                     void* out, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // persistent-style grid: 8 blocks of 8 rows per SM, rows strided over it
    const int64_t want = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    const int64_t cap = (int64_t)sms * 8;
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    if (V == 128)
        output_gate_kernel<TG, TOut, 128><<<grid, kRowsPerBlock * 32, 0, st>>>(
            o, static_cast<const TG*>(gate), w, eps, rows, static_cast<TOut*>(out));
    else
        output_gate_kernel<TG, TOut, 64><<<grid, kRowsPerBlock * 32, 0, st>>>(
            o, static_cast<const TG*>(gate), w, eps, rows, static_cast<TOut*>(out));
    return cudaGetLastError();
}

}  // namespace

cudaError_t output_gate(kda_dtype gate_dt, kda_dtype out_dt, int V, const float* o, const void* gate,
                        const float* w, float eps, int64_t rows, void* out, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    const bool gb = gate_dt == KDA_BF16, ob = out_dt == KDA_BF16;
    if (gb && ob) return launch_v<__nv_bfloat16, __nv_bfloat16>(V, o, gate, w, eps, rows, out, st);
    if (gb) return launch_v<__nv_bfloat16, float>(V, o, gate, w, eps, rows, out, st);
    if (ob) return launch_v<float, __nv_bfloat16>(V, o, gate, w, eps, rows, out, st);
    return launch_v<float, float>(V, o, gate, w, eps, rows, out, st);
}

}  // namespace kda
