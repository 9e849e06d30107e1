// Chunked KDA prefill on the CUDA cores, fp32 throughout.
//
// This is the fp32-input path (fp32 arithmetic is needed for fp32 inputs: a
// tensor-core pass through tf32 or bf16 operands cannot hold a 1e-5 relative
// error) and the reference layout of the chunk algebra that the tensor-core
// kernel follows.  One CTA owns one (sequence, head, V-tile) and walks the
// sequence in chunks of C = 64 tokens, keeping the K x VT state slice in
// shared memory.  Per chunk, with G the in-chunk cumulative sum of g (per key
// channel), the algebra is:
//
//   A[r,j] = sum_c k[r,c] k[j,c] e^{G[r,c]-G[j,c]}   (j <  r)
//   P[r,j] = sum_c q[r,c] k[j,c] e^{G[r,c]-G[j,c]}   (j <= r)
//   T      = (I + Diag(beta) A)^{-1}                 (unit lower triangular)
//   W      = T Diag(beta) (k * e^G),   U~ = T Diag(beta) v
//   U      = U~ - W S
//   O      = scale ((q * e^G) S + P U)
//   S     <- Diag(e^{G_last}) S + (k * e^{G_last - G})^T U
//
// which reproduces the token-by-token recurrence exactly in real arithmetic.
// The gated products use 16-token row blocks with the reference point G at
// the row just before the block, so every exponent stays in [-80, 80] (the
// gate is bounded below by -5).  Partial chunks are padded with k = q = v = 0,
// beta = 0, g = 0 rows, which leave the state unchanged.
//
// With kPrologue the tile loads apply the K3 KDA input prologue ("kimi-k3-mlx"
// review, section "Attention is 93 layers ...": kernel-4 short convolution on
// q, k, v and the per-channel forget gate with lower bound -5; section "The
// A_log shape mismatch ...": A_log[K] shared by all heads, dt_bias[H*K]).
#include "kda_chunk.h"
#include "kda_common.cuh"

namespace kda {

constexpr int kC = 64;        // chunk length
constexpr int kSub = 16;      // row block of the gated products
constexpr int kSimtThreads = 256;

template <int K, int V> struct SimtCfg {
    static constexpr int VT = (V == 64) ? 64 : 32;  // V columns per CTA
    static constexpr int kFloats = 4 * kC * K + K * VT + kC * VT + 3 * kC * kC + kC + K;
    static constexpr size_t kSmem = sizeof(float) * kFloats;
};

// Every output (m, n) of an M x N block is owned by exactly one thread, which
// computes a TM x TN register tile.
template <int M, int N, int TM, int TN, typename F>
__device__ __forceinline__ void for_tiles(F&& f) {
    constexpr int NTN = N / TN;
    constexpr int TILES = (M / TM) * NTN;
    for (int t = threadIdx.x; t < TILES; t += kSimtThreads) f((t / NTN) * TM, (t % NTN) * TN);
}

__device__ __forceinline__ float softplus_f(float z) {
    return z > 0.f ? z + log1pf(expf(-z)) : log1pf(expf(z));
}

template <typename TIn, typename TOut, int K, int V, bool kPrologue>
__global__ void __launch_bounds__(kSimtThreads, 1) chunk_simt_kernel(ChunkParams p) {
    using Cfg = SimtCfg<K, V>;
    constexpr int VT = Cfg::VT;
    constexpr int NVT = V / VT;
    extern __shared__ __align__(16) float sm[];
    float* Qb = sm;                 // [C][K]  q, then q * e^G
    float* Kb = Qb + kC * K;        // [C][K]  k, then W
    float* Gb = Kb + kC * K;        // [C][K]  g, then beta k e^G
    float* Wb = Gb + kC * K;        // [C][K]  right factors of the gated products, then K-bar
    float* Sb = Wb + kC * K;        // [K][VT] state slice
    float* Vb = Sb + K * VT;        // [C][VT] v, then beta v
    float* Pb = Vb + kC * VT;       // [C][C]  P
    float* Ab = Pb + kC * kC;       // [C][C]  A, then U~ / U ([C][VT])
    float* Tb = Ab + kC * kC;       // [C][C]  left factors (2 x 16 x K), then T
    float* bb = Tb + kC * kC;       // [C]     beta
    float* eGC = bb + kC;           // [K]     e^{G_last}

    const int tid = threadIdx.x;
    const int H = p.H;
    const int item = blockIdx.x;
    const int vt = item % NVT;
    const int h = (item / NVT) % H;
    const int rank = item / (NVT * H);

    // ---- which sequence: longest first when packed --------------------------
    __shared__ int s_seq;
    int n = rank;
    if (p.cu_seqlens != nullptr && p.N <= 1024) {
        if (tid == 0) s_seq = rank;
        __syncthreads();
        for (int m = tid; m < p.N; m += kSimtThreads) {
            const int lm = seq_len_clamped(p.cu_seqlens, m, p.T);
            int r = 0;
            for (int x = 0; x < p.N; ++x) {
                const int lx = seq_len_clamped(p.cu_seqlens, x, p.T);
                r += (lx > lm) || (lx == lm && x < m);
            }
            if (r == rank) s_seq = m;
        }
        __syncthreads();
        n = s_seq;
    }
    int64_t bos, eos;
    if (p.cu_seqlens != nullptr) {
        bos = min(max((int)p.cu_seqlens[n], 0), p.T);
        eos = min(max((int)p.cu_seqlens[n + 1], 0), p.T);
        if (eos < bos) eos = bos;
    } else {
        bos = (int64_t)n * p.T;
        eos = bos + p.T;
    }
    const int v0 = vt * VT;
    const TIn* __restrict__ q = (const TIn*)p.q;
    const TIn* __restrict__ k = (const TIn*)p.k;
    const TIn* __restrict__ v = (const TIn*)p.v;
    const TIn* __restrict__ g = (const TIn*)p.g;
    const TIn* __restrict__ beta = (const TIn*)p.beta;
    TOut* __restrict__ o = (TOut*)p.o;

    // ---- initial state -------------------------------------------------------
    const int64_t sbase = (((int64_t)n * H + h) * K) * V + v0;
    for (int i = tid; i < K * VT; i += kSimtThreads) {
        const int c = i / VT, x = i % VT;
        Sb[i] = p.initial_state ? p.initial_state[sbase + (int64_t)c * V + x] : 0.f;
    }

    for (int64_t c0 = bos; c0 < eos; c0 += kC) {
        const int L = (eos - c0 < (int64_t)kC) ? (int)(eos - c0) : kC;
        __syncthreads();  // previous chunk fully consumed

        // ---- (0) tile loads (with the prologue when fused) -------------------
        for (int i = tid; i < kC * K; i += kSimtThreads) {
            const int r = i / K, c = i % K;
            float qv = 0.f, kv = 0.f, gv = 0.f;
            if (r < L) {
                const int64_t t = c0 + r;
                const int64_t e = (t * H + h) * K + c;
                if constexpr (kPrologue) {
                    const int ch = h * K + c;
                    float aq = 0.f, ak = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int64_t s = t - 3 + j;
                        if (s >= bos) {
                            const int64_t es = (s * H + h) * K + c;
                            aq += p.conv_q[ch * 4 + j] * ld(q, es);
                            ak += p.conv_k[ch * 4 + j] * ld(k, es);
                        }
                    }
                    if (p.conv_act == 1) {
                        aq = aq / (1.f + expf(-aq));
                        ak = ak / (1.f + expf(-ak));
                    }
                    qv = aq;
                    kv = ak;
                    const float z = ld(g, e) + p.dt_bias[ch];
                    gv = fmaxf(p.lower_bound, -expf(p.A_log[c]) * softplus_f(z));
                } else {
                    qv = ld(q, e);
                    kv = ld(k, e);
                    gv = ld(g, e);
                }
            }
            Qb[i] = qv;
            Kb[i] = kv;
            Gb[i] = gv;
        }
        for (int i = tid; i < kC * VT; i += kSimtThreads) {
            const int r = i / VT, x = i % VT;
            float vv = 0.f;
            if (r < L) {
                const int64_t t = c0 + r;
                if constexpr (kPrologue) {
                    const int ch = h * V + v0 + x;
                    float a = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int64_t s = t - 3 + j;
                        if (s >= bos) a += p.conv_v[ch * 4 + j] * ld(v, (s * H + h) * V + v0 + x);
                    }
                    if (p.conv_act == 1) a = a / (1.f + expf(-a));
                    vv = a;
                } else {
                    vv = ld(v, (t * H + h) * V + v0 + x);
                }
            }
            Vb[i] = vv;
        }
        if (tid < kC) bb[tid] = (tid < L) ? ld(beta, (c0 + tid) * H + h) : 0.f;
        __syncthreads();

        if constexpr (kPrologue) {
            // L2-normalise q and k rows over the K channels of the head.
            const int warp = tid / 32, lane = tid % 32;
            for (int rr = warp; rr < 2 * kC; rr += kSimtThreads / 32) {
                float* row = (rr < kC) ? (Qb + rr * K) : (Kb + (rr - kC) * K);
                float ss = 0.f;
                for (int c = lane; c < K; c += 32) ss += row[c] * row[c];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float inv = rsqrtf(ss + p.l2_eps);
                for (int c = lane; c < K; c += 32) row[c] *= inv;
            }
            __syncthreads();
        }

        // ---- (1)+(2) gated products A (strict) and P (with diagonal) ---------
        // Exponents are formed as direct sums of the (non-positive) gates over
        // exactly the tokens they span, never as differences of cumulative
        // sums: a difference of two large cumulative sums would lose the
        // small exponents that matter to cancellation.
        for (int R = 0; R < kC / kSub; ++R) {
            const int r0 = R * kSub;
            const int jmax = r0 + kSub;  // columns j < jmax can be non-zero
            if (tid < K) {
                const int c = tid;
                // rows of block R: left factor e^{sum g[r0..r]}, diagonal-block
                // right factor e^{-sum g[r0..j]}
                float acc = 0.f;
                for (int r = r0; r < jmax; ++r) {
                    acc += Gb[r * K + c];
                    const float el = expf(acc);
                    Tb[(r - r0) * K + c] = Kb[r * K + c] * el;
                    Tb[kSub * K + (r - r0) * K + c] = Qb[r * K + c] * el;
                    Wb[r * K + c] = Kb[r * K + c] * expf(-acc);
                }
                // earlier rows: right factor e^{sum g[j+1 .. r0-1]} <= 1
                float sfx = 0.f;
                for (int j = r0 - 1; j >= 0; --j) {
                    Wb[j * K + c] = Kb[j * K + c] * expf(sfx);
                    sfx += Gb[j * K + c];
                }
            }
            __syncthreads();
            for (int i = tid; i < kSub * jmax; i += kSimtThreads) {
                const int rl = i / jmax, j = i % jmax;
                const int r = r0 + rl;
                float a = 0.f, pq = 0.f;
                if (j <= r) {
                    const float* lk = Tb + rl * K;
                    const float* lq = Tb + kSub * K + rl * K;
                    const float* rk = Wb + j * K;
#pragma unroll 8
                    for (int c = 0; c < K; ++c) {
                        a += lk[c] * rk[c];
                        pq += lq[c] * rk[c];
                    }
                }
                Ab[r * kC + j] = (j < r) ? a : 0.f;
                Pb[r * kC + j] = (j <= r) ? pq : 0.f;
            }
            for (int i = tid; i < kSub * (kC - jmax); i += kSimtThreads) {
                const int rl = i / (kC - jmax), j = jmax + i % (kC - jmax);
                Ab[(r0 + rl) * kC + j] = 0.f;
                Pb[(r0 + rl) * kC + j] = 0.f;
            }
            __syncthreads();
        }

        // ---- (3) T = (I + Diag(beta) A)^{-1}, four lanes per column ----------
        {
            const int col = tid / 4, part = tid % 4;
            float* Tc = Tb;  // T[r][col] at Tc[r * C + col]
            for (int r = part; r < kC; r += 4) Tc[r * kC + col] = (r == col) ? 1.f : 0.f;
            __syncwarp();
            // Every lane of the warp runs the same r range so the shuffles
            // always see the full warp; columns with r <= col contribute 0.
            for (int r = 1; r < kC; ++r) {
                float acc = 0.f;
                if (r > col)
                    for (int j = col + part; j < r; j += 4) acc += Ab[r * kC + j] * Tc[j * kC + col];
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                if (part == 0 && r > col) Tc[r * kC + col] = -bb[r] * acc;
                __syncwarp();
            }
        }
        __syncthreads();

        // ---- (4) decayed operands --------------------------------------------
        // Per key channel: K-bar_j = k_j e^{sum g[j+1..C-1]} (into Wb), then
        // q e^{sum g[0..r]} (in place) and beta k e^{sum g[0..r]} (over g).
        if (tid < K) {
            const int c = tid;
            float sfx = 0.f;
            for (int j = kC - 1; j >= 0; --j) {
                Wb[j * K + c] = Kb[j * K + c] * expf(sfx);
                sfx += Gb[j * K + c];
            }
            float acc = 0.f;
            for (int r = 0; r < kC; ++r) {
                acc += Gb[r * K + c];
                const float e = expf(acc);
                Qb[r * K + c] *= e;
                Gb[r * K + c] = bb[r] * Kb[r * K + c] * e;
            }
            eGC[c] = expf(acc);
        }
        for (int i = tid; i < kC * VT; i += kSimtThreads) Vb[i] *= bb[i / VT];
        __syncthreads();

        // ---- (5) W = T (beta k e^G),  U~ = T (beta v) ------------------------
        for_tiles<kC, K, 4, K / 32>([&](int m0, int n0) {
            constexpr int TN = K / 32;
            float acc[4][TN] = {};
            for (int j = 0; j <= m0 + 3; ++j) {
                float b[TN];
#pragma unroll
                for (int y = 0; y < TN; ++y) b[y] = Gb[j * K + n0 + y];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float a = Tb[(m0 + x) * kC + j];
#pragma unroll
                    for (int y = 0; y < TN; ++y) acc[x][y] += a * b[y];
                }
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < TN; ++y) Kb[(m0 + x) * K + n0 + y] = acc[x][y];
        });
        for_tiles<kC, VT, 2, VT / 16>([&](int m0, int n0) {
            constexpr int TN = VT / 16;
            float acc[2][TN] = {};
            for (int j = 0; j <= m0 + 1; ++j) {
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const float a = Tb[(m0 + x) * kC + j];
#pragma unroll
                    for (int y = 0; y < TN; ++y) acc[x][y] += a * Vb[j * VT + n0 + y];
                }
            }
#pragma unroll
            for (int x = 0; x < 2; ++x)
#pragma unroll
                for (int y = 0; y < TN; ++y) Ab[(m0 + x) * VT + n0 + y] = acc[x][y];
        });
        __syncthreads();

        // ---- (6) U = U~ - W S ------------------------------------------------
        for_tiles<kC, VT, 2, VT / 16>([&](int m0, int n0) {
            constexpr int TN = VT / 16;
            float acc[2][TN] = {};
            for (int c = 0; c < K; ++c) {
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const float a = Kb[(m0 + x) * K + c];
#pragma unroll
                    for (int y = 0; y < TN; ++y) acc[x][y] += a * Sb[c * VT + n0 + y];
                }
            }
#pragma unroll
            for (int x = 0; x < 2; ++x)
#pragma unroll
                for (int y = 0; y < TN; ++y) Ab[(m0 + x) * VT + n0 + y] -= acc[x][y];
        });
        __syncthreads();

        // ---- (7) O = scale ((q e^G) S + P U) ---------------------------------
        for_tiles<kC, VT, 2, VT / 16>([&](int m0, int n0) {
            constexpr int TN = VT / 16;
            float acc[2][TN] = {};
            for (int c = 0; c < K; ++c) {
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const float a = Qb[(m0 + x) * K + c];
#pragma unroll
                    for (int y = 0; y < TN; ++y) acc[x][y] += a * Sb[c * VT + n0 + y];
                }
            }
            for (int j = 0; j <= m0 + 1; ++j) {
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const float a = Pb[(m0 + x) * kC + j];
#pragma unroll
                    for (int y = 0; y < TN; ++y) acc[x][y] += a * Ab[j * VT + n0 + y];
                }
            }
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const int r = m0 + x;
                if (r < L) {
                    const int64_t ob = ((c0 + r) * H + h) * (int64_t)V + v0 + n0;
#pragma unroll
                    for (int y = 0; y < TN; ++y) o[ob + y] = from_f32<TOut>(p.scale * acc[x][y]);
                }
            }
        });
        __syncthreads();

        // ---- (8) S <- Diag(e^{G_last}) S + Kbar^T U --------------------------
        for_tiles<K, VT, 4, VT / 8 < 4 ? VT / 8 : 4>([&](int m0, int n0) {
            constexpr int TN = VT / 8 < 4 ? VT / 8 : 4;
            float acc[4][TN];
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < TN; ++y) acc[x][y] = eGC[m0 + x] * Sb[(m0 + x) * VT + n0 + y];
            for (int j = 0; j < L; ++j) {
                float b[TN];
#pragma unroll
                for (int y = 0; y < TN; ++y) b[y] = Ab[j * VT + n0 + y];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const float a = Wb[j * K + m0 + x];
#pragma unroll
                    for (int y = 0; y < TN; ++y) acc[x][y] += a * b[y];
                }
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < TN; ++y) Sb[(m0 + x) * VT + n0 + y] = acc[x][y];
        });
    }
    __syncthreads();

    if (p.final_state) {
        for (int i = tid; i < K * VT; i += kSimtThreads) {
            const int c = i / VT, x = i % VT;
            p.final_state[sbase + (int64_t)c * V + x] = Sb[i];
        }
    }
}

}  // namespace kda

namespace kda {

template <typename TIn, typename TOut, int K, int V, bool kPro>
static cudaError_t launch_simt(const ChunkParams& p, cudaStream_t st) {
    using Cfg = SimtCfg<K, V>;
    constexpr int NVT = V / Cfg::VT;
    const int64_t blocks = (int64_t)p.N * p.H * NVT;
    if (blocks == 0) return cudaSuccess;
    auto kern = chunk_simt_kernel<TIn, TOut, K, V, kPro>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Cfg::kSmem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)blocks, kSimtThreads, Cfg::kSmem, st>>>(p);
    return cudaGetLastError();
}

template <typename TIn, typename TOut, bool kPro>
static cudaError_t simt_kv(int K, int V, const ChunkParams& p, cudaStream_t st) {
    if (K == 128 && V == 128) return launch_simt<TIn, TOut, 128, 128, kPro>(p, st);
    if (K == 128 && V == 64) return launch_simt<TIn, TOut, 128, 64, kPro>(p, st);
    if (K == 64 && V == 128) return launch_simt<TIn, TOut, 64, 128, kPro>(p, st);
    return launch_simt<TIn, TOut, 64, 64, kPro>(p, st);
}

template <typename TIn, typename TOut>
static cudaError_t simt_pro(int K, int V, bool pro, const ChunkParams& p, cudaStream_t st) {
    return pro ? simt_kv<TIn, TOut, true>(K, V, p, st) : simt_kv<TIn, TOut, false>(K, V, p, st);
}

cudaError_t chunk_simt(kda_dtype in_dt, kda_dtype out_dt, int K, int V, bool prologue,
                       const ChunkParams& p, cudaStream_t st) {
    if (in_dt == KDA_BF16) {
        if (out_dt == KDA_F32) return simt_pro<__nv_bfloat16, float>(K, V, prologue, p, st);
        return simt_pro<__nv_bfloat16, __nv_bfloat16>(K, V, prologue, p, st);
    }
    if (out_dt == KDA_F32) return simt_pro<float, float>(K, V, prologue, p, st);
    return simt_pro<float, __nv_bfloat16>(K, V, prologue, p, st);
}

}  // namespace kda
