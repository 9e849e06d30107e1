// Single-token KDA decode: one HBM pass over the fp32 state per step.
//
// For each (sequence n, head h) one CTA reads the K x V state slice once with
// 128-bit loads, forms the two channel reductions
//     a = S_old^T (k * e^g),   b = S_old^T (q * e^g)
// (per-thread partial sums over its rows, then a cross-warp reduction through
// shared memory), then
//     delta = beta (v - a),    o = scale (b + (q . k) delta),
//     S_new = Diag(e^g) S_old + k delta^T
// and writes S_new back in place.  This is the recurrence's decay, delta
// update and read-out folded into one pass, so the state is read once and
// written once ("ISEEKYAN/k3" README: the KDA recurrence as the operator's
// recurrent path; per-channel decay from the "kimi-k3-mlx" review, section
// "The A_log shape mismatch ...").
#include "kda_chunk.h"
#include "kda_common.cuh"

namespace kda {

constexpr int kDecodeThreads = 256;

template <typename TIn, typename TOut, int K, int V>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_step_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                   const TIn* __restrict__ v, const TIn* __restrict__ g,
                   const TIn* __restrict__ beta, float scale, float* __restrict__ state,
                   TOut* __restrict__ o) {
    constexpr int NT = kDecodeThreads;
    constexpr int LPR = V / 4;   // threads per state row (one float4 each)
    constexpr int RG = NT / LPR; // row groups
    constexpr int RPT = K / RG;  // rows per thread
    static_assert(RG * LPR == NT && RPT * RG == K, "decode tiling");

    const int64_t nh = blockIdx.x;
    const int tid = threadIdx.x;
    const int c4 = tid % LPR;
    const int rg = tid / LPR;

    float4* S = reinterpret_cast<float4*>(state + nh * K * V);
    float4 s[RPT];
    // Issue every state load first so that the whole slice is in flight.
#pragma unroll
    for (int i = 0; i < RPT; ++i) s[i] = __ldcs(&S[(rg + i * RG) * LPR + c4]);

    __shared__ float eg[K], kk[K], qq[K];
    __shared__ __align__(16) float red_a[RG][V];
    __shared__ __align__(16) float red_b[RG][V];
    __shared__ float dl[V];
    __shared__ float qk_s;

    for (int c = tid; c < K; c += NT) {
        eg[c] = expf(ld(g, nh * K + c));
        kk[c] = ld(k, nh * K + c);
        qq[c] = ld(q, nh * K + c);
    }
    __syncthreads();
    if (tid < 32) {
        float acc = 0.f;
        for (int c = tid; c < K; c += 32) acc += qq[c] * kk[c];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (tid == 0) qk_s = acc;
    }

    float4 pa = make_float4(0.f, 0.f, 0.f, 0.f), pb = pa;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int r = rg + i * RG;
        const float wa = kk[r] * eg[r], wb = qq[r] * eg[r];
        pa.x += wa * s[i].x; pa.y += wa * s[i].y; pa.z += wa * s[i].z; pa.w += wa * s[i].w;
        pb.x += wb * s[i].x; pb.y += wb * s[i].y; pb.z += wb * s[i].z; pb.w += wb * s[i].w;
    }
    reinterpret_cast<float4*>(red_a[rg])[c4] = pa;
    reinterpret_cast<float4*>(red_b[rg])[c4] = pb;
    __syncthreads();

    if (tid < V) {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int j = 0; j < RG; ++j) { a += red_a[j][tid]; b += red_b[j][tid]; }
        const float bt = ld(beta, nh);
        const float d = bt * (ld(v, nh * V + tid) - a);
        dl[tid] = d;
        o[nh * V + tid] = from_f32<TOut>(scale * (b + qk_s * d));
    }
    __syncthreads();

    const float4 d4 = reinterpret_cast<const float4*>(dl)[c4];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int r = rg + i * RG;
        const float e = eg[r], kr = kk[r];
        float4 n;
        n.x = e * s[i].x + kr * d4.x;
        n.y = e * s[i].y + kr * d4.y;
        n.z = e * s[i].z + kr * d4.z;
        n.w = e * s[i].w + kr * d4.w;
        __stcs(&S[r * LPR + c4], n);
    }
}

template <typename TIn, typename TOut, int K, int V>
static cudaError_t launch_decode(const void* q, const void* k, const void* v, const void* g,
                                 const void* beta, float scale, float* state, int N, int H,
                                 void* o, cudaStream_t st) {
    const int64_t blocks = (int64_t)N * H;
    if (blocks == 0) return cudaSuccess;
    decode_step_kernel<TIn, TOut, K, V><<<(unsigned)blocks, kDecodeThreads, 0, st>>>(
        (const TIn*)q, (const TIn*)k, (const TIn*)v, (const TIn*)g, (const TIn*)beta, scale,
        state, (TOut*)o);
    return cudaGetLastError();
}

template <typename TIn, typename TOut>
static cudaError_t dispatch_kv(int K, int V, const void* q, const void* k, const void* v,
                               const void* g, const void* beta, float scale, float* state, int N,
                               int H, void* o, cudaStream_t st) {
    if (K == 128 && V == 128) return launch_decode<TIn, TOut, 128, 128>(q, k, v, g, beta, scale, state, N, H, o, st);
    if (K == 128 && V == 64) return launch_decode<TIn, TOut, 128, 64>(q, k, v, g, beta, scale, state, N, H, o, st);
    if (K == 64 && V == 128) return launch_decode<TIn, TOut, 64, 128>(q, k, v, g, beta, scale, state, N, H, o, st);
    return launch_decode<TIn, TOut, 64, 64>(q, k, v, g, beta, scale, state, N, H, o, st);
}

cudaError_t decode_step(kda_dtype in_dt, kda_dtype out_dt, int K, int V, const void* q,
                        const void* k, const void* v, const void* g, const void* beta,
                        float scale, float* state, int N, int H, void* o, cudaStream_t st) {
    if (in_dt == KDA_BF16) {
        if (out_dt == KDA_F32) return dispatch_kv<__nv_bfloat16, float>(K, V, q, k, v, g, beta, scale, state, N, H, o, st);
        return dispatch_kv<__nv_bfloat16, __nv_bfloat16>(K, V, q, k, v, g, beta, scale, state, N, H, o, st);
    }
    if (out_dt == KDA_F32) return dispatch_kv<float, float>(K, V, q, k, v, g, beta, scale, state, N, H, o, st);
    return dispatch_kv<float, __nv_bfloat16>(K, V, q, k, v, g, beta, scale, state, N, H, o, st);
}

}  // namespace kda
