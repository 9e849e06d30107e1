// Backward of the KDA recurrence, token by token (CUDA cores, fp32).
//
// Gradients of L = <dO, o> + <dS_T, S_T> with respect to q, k, v, g, beta and
// the initial state.  Per token, with S' = Diag(e^{g_t}) S_{t-1}, a = S'^T k_t,
// delta = beta_t (v_t - a) and S_t = S' + k_t delta^T, the reverse step from the
// gradient dS of S_t is
//
//     dq_t   = scale S_t dO_t              dS    += scale q_t dO_t^T
//     ddelta = dS^T k_t                    dk_t   = dS delta + S' da
//     dbeta_t = ddelta . (v_t - a)         dv_t   = beta_t ddelta
//     da     = -beta_t ddelta              dg_t[c] = sum_x (dS + k_t da^T)[c, x] S'[c, x]
//     dS_{t-1} = Diag(e^{g_t}) (dS + k_t da^T)
//
// One CTA per (sequence, head).  The state and its gradient live in shared
// memory (rows padded by one float so that row and column walks are both free
// of bank conflicts).  A first forward pass stores the state every 64 tokens in
// the workspace; walking the blocks backwards, each block's 64 states are
// recomputed into the workspace and then consumed in reverse.  This is the
// straightforward form of the backward (the reference for a chunked one).
#include "kda_chunk.h"
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kBwdThreads = 512;
constexpr int kBwdBlock = 64;

template <typename TIn>
__global__ void __launch_bounds__(kBwdThreads)
recurrent_bwd_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
                     const TIn* __restrict__ g, const TIn* __restrict__ beta, float scale,
                     const float* __restrict__ s0, const int32_t* __restrict__ cu, int B, int T, int H, int K,
                     int V, const float* __restrict__ dO, const float* __restrict__ dST, float* __restrict__ dq,
                     float* __restrict__ dk, float* __restrict__ dv, float* __restrict__ dg,
                     float* __restrict__ dbeta, float* __restrict__ dS0, float* __restrict__ ckpt,
                     float* __restrict__ states, int64_t max_blocks, int32_t* __restrict__ status) {
    extern __shared__ float sm[];
    const int LD = V + 1;
    float* S = sm;                      // running state, then S' of the current token [K][LD]
    float* dS = S + K * LD;             // state gradient [K][LD]
    float* qv = dS + K * LD;            // q_t [K]
    float* kv = qv + K;                 // k_t [K]
    float* ev = kv + K;                 // e^{g_t} [K]
    float* vv = ev + K;                 // v_t [V]
    float* ov = vv + V;                 // dO_t [V]
    float* av = ov + V;                 // a [V]
    float* dlt = av + V;                // delta [V]
    float* dda = dlt + V;               // ddelta [V]
    float* red = dda + V;               // [32] warp partials
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    int64_t bos, eos, ck0;
    if (cu == nullptr) {
        bos = (int64_t)n * T;
        eos = bos + T;
        ck0 = (int64_t)n * ((T + kBwdBlock - 1) / kBwdBlock);
    } else {
        bos = min(max(cu[n], 0), T);
        eos = max(bos, (int64_t)min(max(cu[n + 1], 0), T));
        // this sequence's first checkpoint: the blocks of the sequences before it
        ck0 = 0;
        for (int m = 0; m < n; ++m) ck0 += (seq_len_clamped(cu, m, T) + kBwdBlock - 1) / kBwdBlock;
    }
    const int64_t len = eos - bos;
    const int nblk = (int)((len + kBwdBlock - 1) / kBwdBlock);
    const int64_t KV = (int64_t)K * V;
    if (ck0 + nblk > max_blocks) {
        // offsets that overlap can need more checkpoints than the workspace holds:
        // such a chain is not computed, its gradients are marked NaN (rows that a
        // computed chain shares with it may be overwritten by that chain) and the
        // status word says KDA_ERR_RANGE
        if (tid == 0 && status != nullptr) *reinterpret_cast<volatile int32_t*>(status) = (int32_t)KDA_ERR_RANGE;
        const float nan = __int_as_float(0x7fc00000);
        for (int64_t i = tid; i < len * K; i += kBwdThreads) {
            const int64_t t = bos + i / K;
            const int64_t e = (t * H + h) * K + i % K;
            dq[e] = nan; dk[e] = nan; dg[e] = nan;
        }
        for (int64_t i = tid; i < len * V; i += kBwdThreads) dv[((bos + i / V) * H + h) * V + i % V] = nan;
        for (int64_t i = tid; i < len; i += kBwdThreads) dbeta[(bos + i) * H + h] = nan;
        if (dS0)
            for (int64_t e = tid; e < KV; e += kBwdThreads) dS0[((int64_t)n * H + h) * KV + e] = nan;
        return;
    }
    float* ck = ckpt + (ck0 * H + (int64_t)h * nblk) * KV;  // nblk checkpoints of this chain
    float* st = states + (int64_t)blockIdx.x * kBwdBlock * KV;
    const int64_t sbase = ((int64_t)n * H + h) * KV;

    auto tok = [&](int64_t t, int64_t i, int D) { return (t * H + h) * D + i; };
    // token t's q, k, e^g (and v, dO when asked) into shared memory
    auto load_token = [&](int64_t t, bool with_q) {
        for (int i = tid; i < K; i += kBwdThreads) {
            kv[i] = to_f32<TIn>(k[tok(t, i, K)]);
            ev[i] = expf(to_f32<TIn>(g[tok(t, i, K)]));
            if (with_q) qv[i] = to_f32<TIn>(q[tok(t, i, K)]);
        }
        for (int x = tid; x < V; x += kBwdThreads) {
            vv[x] = to_f32<TIn>(v[tok(t, x, V)]);
            if (with_q) ov[x] = dO[tok(t, x, V)];
        }
    };
    // S <- Diag(e^g) S; a = S^T k; delta = beta (v - a); S <- S + k delta^T
    auto step_forward = [&](float bt) {
        for (int e = tid; e < K * V; e += kBwdThreads) S[(e / V) * LD + e % V] *= ev[e / V];
        __syncthreads();
        for (int x = tid; x < V; x += kBwdThreads) {
            float acc = 0.f;
            for (int c = 0; c < K; ++c) acc += S[c * LD + x] * kv[c];
            av[x] = acc;
            dlt[x] = bt * (vv[x] - acc);
        }
        __syncthreads();
        for (int e = tid; e < K * V; e += kBwdThreads) S[(e / V) * LD + e % V] += kv[e / V] * dlt[e % V];
        __syncthreads();
    };
    auto store_state = [&](float* dst) {
        for (int e = tid; e < K * V; e += kBwdThreads) dst[e] = S[(e / V) * LD + e % V];
    };
    auto load_state = [&](const float* src, float* dstm) {
        for (int e = tid; e < K * V; e += kBwdThreads) dstm[(e / V) * LD + e % V] = src ? src[e] : 0.f;
    };

    // ---- forward: checkpoints at the start of every block
    load_state(s0 ? s0 + sbase : nullptr, S);
    __syncthreads();
    for (int b = 0; b < nblk; ++b) {
        store_state(ck + (int64_t)b * KV);
        const int64_t t1 = min(bos + (int64_t)(b + 1) * kBwdBlock, eos);
        for (int64_t t = bos + (int64_t)b * kBwdBlock; t < t1; ++t) {
            __syncthreads();
            load_token(t, false);
            __syncthreads();
            step_forward(to_f32<TIn>(beta[t * H + h]));
        }
    }

    // ---- backward
    load_state(dST ? dST + sbase : nullptr, dS);
    for (int b = nblk - 1; b >= 0; --b) {
        const int64_t ts = bos + (int64_t)b * kBwdBlock, te = min(ts + kBwdBlock, eos);
        // the block's states S_{t-1}, recomputed from its checkpoint
        __syncthreads();
        load_state(ck + (int64_t)b * KV, S);
        __syncthreads();
        for (int64_t t = ts; t < te; ++t) {
            store_state(st + (t - ts) * KV);
            __syncthreads();
            load_token(t, false);
            __syncthreads();
            step_forward(to_f32<TIn>(beta[t * H + h]));
        }
        __syncthreads();  // (the global stores of the states are read back below by the same CTA)
        for (int64_t t = te - 1; t >= ts; --t) {
            const float bt = to_f32<TIn>(beta[t * H + h]);
            load_token(t, true);
            __syncthreads();
            // S' = Diag(e^g) S_{t-1}
            const float* sp = st + (t - ts) * KV;
            for (int e = tid; e < K * V; e += kBwdThreads) S[(e / V) * LD + e % V] = ev[e / V] * sp[e];
            __syncthreads();
            // a, delta
            for (int x = tid; x < V; x += kBwdThreads) {
                float acc = 0.f;
                for (int c = 0; c < K; ++c) acc += S[c * LD + x] * kv[c];
                av[x] = acc;
                dlt[x] = bt * (vv[x] - acc);
            }
            __syncthreads();
            // dq = scale (S' + k delta^T) dO
            for (int c = tid; c < K; c += kBwdThreads) {
                float acc = 0.f;
                for (int x = 0; x < V; ++x) acc += (S[c * LD + x] + kv[c] * dlt[x]) * ov[x];
                dq[tok(t, c, K)] = scale * acc;
            }
            // dS += scale q dO^T
            for (int e = tid; e < K * V; e += kBwdThreads) dS[(e / V) * LD + e % V] += scale * qv[e / V] * ov[e % V];
            __syncthreads();
            // ddelta = dS^T k; dv = beta ddelta; dbeta = ddelta . (v - a)
            float db = 0.f;
            for (int x = tid; x < V; x += kBwdThreads) {
                float acc = 0.f;
                for (int c = 0; c < K; ++c) acc += dS[c * LD + x] * kv[c];
                dda[x] = acc;
                dv[tok(t, x, V)] = bt * acc;
                db += acc * (vv[x] - av[x]);
            }
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) db += __shfl_xor_sync(0xffffffffu, db, d);
            if (lane == 0) red[warp] = db;
            __syncthreads();
            if (tid == 0) {
                float s = 0.f;
                for (int w = 0; w < kBwdThreads / 32; ++w) s += red[w];
                dbeta[t * H + h] = s;
            }
            // dk = dS delta + S' da; dg = rowsum((dS + k da^T) * S'), da = -beta ddelta
            for (int c = tid; c < K; c += kBwdThreads) {
                float a1 = 0.f, a2 = 0.f, a3 = 0.f;
                for (int x = 0; x < V; ++x) {
                    const float da = -bt * dda[x];
                    const float sp_ = S[c * LD + x];
                    const float d = dS[c * LD + x] + kv[c] * da;
                    a1 += dS[c * LD + x] * dlt[x];
                    a2 += sp_ * da;
                    a3 += d * sp_;
                }
                dk[tok(t, c, K)] = a1 + a2;
                dg[tok(t, c, K)] = a3;
            }
            __syncthreads();
            // dS_{t-1} = Diag(e^g) (dS + k da^T)
            for (int e = tid; e < K * V; e += kBwdThreads) {
                const int c = e / V, x = e % V;
                dS[c * LD + x] = ev[c] * (dS[c * LD + x] + kv[c] * (-bt * dda[x]));
            }
            __syncthreads();
        }
    }
    if (dS0)
        for (int e = tid; e < K * V; e += kBwdThreads) dS0[sbase + e] = dS[(e / V) * LD + e % V];
}

}  // namespace

size_t recurrent_bwd_workspace(int B, int T, int H, int K, int V, int N, bool packed) {
    const int64_t blocks = packed ? ((int64_t)T + kBwdBlock - 1) / kBwdBlock + N
                                  : (int64_t)B * (((int64_t)T + kBwdBlock - 1) / kBwdBlock);
    const int64_t KV = (int64_t)K * V;
    return (size_t)((blocks * H + (int64_t)N * H * kBwdBlock) * KV) * sizeof(float);
}

cudaError_t recurrent_bwd(kda_dtype in_dt, const void* q, const void* k, const void* v, const void* g,
                          const void* beta, float scale, const float* s0, const int32_t* cu, int B, int T, int H,
                          int K, int V, int N, const float* dO, const float* dST, float* dq, float* dk, float* dv,
                          float* dg, float* dbeta, float* dS0, void* ws, int32_t* status, cudaStream_t st) {
    if (status != nullptr) {
        const cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
        if (e != cudaSuccess) return e;
    }
    const int64_t chains = (int64_t)N * H;
    if (chains == 0) return cudaSuccess;
    float* ckpt = static_cast<float*>(ws);
    const int64_t blocks = cu ? ((int64_t)T + kBwdBlock - 1) / kBwdBlock + N
                              : (int64_t)B * (((int64_t)T + kBwdBlock - 1) / kBwdBlock);
    float* states = ckpt + blocks * H * (int64_t)K * V;
    const size_t smem = ((size_t)2 * K * (V + 1) + 3 * (size_t)K + 5 * (size_t)V + 32) * sizeof(float);
    if (in_dt == KDA_BF16) {
        auto kern = recurrent_bwd_kernel<__nv_bfloat16>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)chains, kBwdThreads, smem, st>>>(
            static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
            static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(g),
            static_cast<const __nv_bfloat16*>(beta), scale, s0, cu, B, T, H, K, V, dO, dST, dq, dk, dv, dg, dbeta,
            dS0, ckpt, states, blocks, status);
    } else {
        auto kern = recurrent_bwd_kernel<float>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)chains, kBwdThreads, smem, st>>>(
            static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
            static_cast<const float*>(g), static_cast<const float*>(beta), scale, s0, cu, B, T, H, K, V, dO, dST,
            dq, dk, dv, dg, dbeta, dS0, ckpt, states, blocks, status);
    }
    return cudaGetLastError();
}

}  // namespace kda
