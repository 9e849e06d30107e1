// Chunked backward of the KDA prefill (bf16 inputs, K = V = 128), built on the
// forward's per-chunk operands.  Gradients of L = <dO, o> + <dS_T, S_T> with
// respect to q, k, v, g, beta and the initial state.  Per chunk of C = 64
// tokens with entering state S (the forward's chunk algebra: G the in-chunk
// cumulative log-decay, X = k e^G, Xq = q e^G, Kb = k e^{G_C - G},
// A = tril(X (k e^-G)^T, -1), P = tril(Xq (k e^-G)^T), T = (I + Diag(beta) A)^{-1},
// W = T Diag(beta) X, U~ = T Diag(beta) v, U = U~ - W S,
// O = scale (Xq S + P U), S' = Diag(e^{G_C}) S + Kb^T U), the reverse step from
// the gradient dS' of S' is
//
//     dU = scale P^T dO + Kb dS'
//     dS = scale Xq^T dO + Diag(e^{G_C}) dS' - W^T dU
//
// and the chunk's input gradients follow from (S, dU, dS', dO) alone:
//
//     dXq = scale dO S^T + dP Y,  dP = scale tril(dO U^T),  dKb = U dS'^T,  dW = -dU S^T
//     dT = dW (Diag(beta) X)^T + dU (Diag(beta) v)^T,  dM = -T^T dT T^T,  dA = Diag(beta) tril(dM, -1)
//     dbeta = rowsum(dM A) + rowsum((T^T dW) X) + rowsum((T^T dU) v),  dv = Diag(beta) T^T dU
//     then the gated products back to k, q and G, and dg = the reverse cumulative sum of dG.
//
// Kernels, on the caller's stream:
//   the forward (chunk_tc_forward_states): the tensor-core prefill, also writing the
//       state entering every chunk; its workspace slots keep W, Qs = scale Xq, Kb,
//       scale P, U~ and e^{G_C} per (chunk, head);
//   bwd_chain_kernel: one CTA per (sequence, head) carries dS backwards through the
//       chunks (the first two lines above, fp32 on the CUDA cores, operands read
//       from the slots) and stores dS' and dU of every chunk;
//   bwd_chunk_kernel: one CTA per (chunk, head) task forms dq, dk, dv, dg, dbeta.
#include "kda_chunk.h"
#include "kda_chunk_plan.cuh"
#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace cplan;

constexpr int kChainThreads = 512;
constexpr int LDX = D + 4;   // fp32 rows of 128 values, padded
constexpr int LDR = C + 4;   // fp32 rows of 64 values, padded

// bf16 hi + lo at the same offset of two images -> 8 floats
__device__ __forceinline__ void hilo8(const uint8_t* hi, const uint8_t* lo, float* x) {
    float a[8], b[8];
    tc::unpack8(*reinterpret_cast<const uint4*>(hi), a);
    tc::unpack8(*reinterpret_cast<const uint4*>(lo), b);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = a[i] + b[i];
}

// ---- reverse chain --------------------------------------------------------------
// Shared memory (fp32): dSp [128][LDX] (the gradient of the state after the chunk),
// dO, dU, Wn = -W, Qs [64][LDX] each (Qs over KbT once dU is formed), P [64][LDR],
// KbT [128][LDR] (Kb transposed), e^{G_C} [128].
constexpr uint32_t BC_DSP = 0;
constexpr uint32_t BC_DO = BC_DSP + D * LDX * 4;
constexpr uint32_t BC_DU = BC_DO + C * LDX * 4;
constexpr uint32_t BC_WN = BC_DU + C * LDX * 4;
constexpr uint32_t BC_P = BC_WN + C * LDX * 4;
constexpr uint32_t BC_KB = BC_P + C * LDR * 4;   // KbT [128][LDR], later Qs [64][LDX]
constexpr uint32_t BC_EGC = BC_KB + D * LDR * 4;
constexpr uint32_t BC_TOTAL = BC_EGC + D * 4;
static_assert(C * LDX <= D * LDR, "Qs fits the KbT region");
static_assert(BC_TOTAL <= 232448, "shared memory of the chain kernel");

__global__ void __launch_bounds__(kChainThreads, 1)
bwd_chain_kernel(const Plan pl, const float* __restrict__ dO, const float* __restrict__ dST,
                 float* __restrict__ dS0, float* __restrict__ dsp_out, float* __restrict__ du_out) {
    extern __shared__ __align__(16) uint8_t smem[];
    float* dSp = reinterpret_cast<float*>(smem + BC_DSP);
    float* dOs = reinterpret_cast<float*>(smem + BC_DO);
    float* dUs = reinterpret_cast<float*>(smem + BC_DU);
    float* Wn = reinterpret_cast<float*>(smem + BC_WN);
    float* Ps = reinterpret_cast<float*>(smem + BC_P);
    float* KbT = reinterpret_cast<float*>(smem + BC_KB);
    float* Qs = KbT;
    float* egc = reinterpret_cast<float*>(smem + BC_EGC);
    const int tid = threadIdx.x;
    const Chain chn = chain_of(pl, blockIdx.x);
    const int H = pl.H, h = chn.h;
    const int64_t sbase = ((int64_t)chn.n * H + h) * D * D;

    for (int e = tid; e < D * D; e += kChainThreads)
        dSp[(e >> 7) * LDX + (e & 127)] = dST != nullptr ? dST[sbase + e] : 0.f;

    for (int64_t i = chn.nchunks - 1; i >= 0; --i) {
        const int64_t c0 = chn.bos + i * C;
        const int L = (chn.eos - c0 < (int64_t)C) ? (int)(chn.eos - c0) : C;
        const int64_t task = (chn.g0 + i) * H + h;
        const uint8_t* slot = pl.slots + task * (int64_t)SLOT_BYTES;
        __syncthreads();   // the previous chunk's readers are done
        // dO rows of the chunk (0 past the sequence end)
        for (int f = tid; f < C * (D / 4); f += kChainThreads) {
            const int r = f >> 5, x4 = (f & 31) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < L) v = *reinterpret_cast<const float4*>(dO + ((c0 + r) * H + h) * D + x4);
            *reinterpret_cast<float4*>(dOs + r * LDX + x4) = v;
        }
        // scale P [r][j] (K-major [64 r][64 j]): one 16-byte unit = 8 consecutive j of a row
        for (int u = tid; u < C * 8; u += kChainThreads) {
            const int r = ((u >> 6) << 3) | (u & 7), jg = (u >> 3) & 7;
            float x[8];
            hilo8(slot + SLOT_P + u * 16, slot + SLOT_P + 8192 + u * 16, x);
            *reinterpret_cast<float4*>(Ps + r * LDR + 8 * jg) = make_float4(x[0], x[1], x[2], x[3]);
            *reinterpret_cast<float4*>(Ps + r * LDR + 8 * jg + 4) = make_float4(x[4], x[5], x[6], x[7]);
        }
        // Kb (K-major [128 c][64 r]): a unit = 8 consecutive r of a channel c -> KbT[c][r]
        for (int u = tid; u < D * 8; u += kChainThreads) {
            const int c = ((u >> 6) << 3) | (u & 7), rg = (u >> 3) & 7;
            float x[8];
            hilo8(slot + SLOT_KH + u * 16, slot + SLOT_KL + u * 16, x);
            *reinterpret_cast<float4*>(KbT + c * LDR + 8 * rg) = make_float4(x[0], x[1], x[2], x[3]);
            *reinterpret_cast<float4*>(KbT + c * LDR + 8 * rg + 4) = make_float4(x[4], x[5], x[6], x[7]);
        }
        // -W (the first half of the merged image, n-group major: a unit = 8 consecutive
        // rows r of a channel c)
        for (int u = tid; u < 8 * D; u += kChainThreads) {
            const int c = u & 127, ng = u >> 7;
            float x[8];
            hilo8(slot + SLOT_WQH + u * 16, slot + SLOT_WQL + u * 16, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) Wn[(8 * ng + e) * LDX + c] = x[e];
        }
        if (tid < D) egc[tid] = reinterpret_cast<const float*>(slot + SLOT_EGC)[tid];
        __syncthreads();

        // the gradient of the state after this chunk, for the chunk's own gradients
        {
            float* dst = dsp_out + task * (int64_t)(D * D);
            for (int f = tid; f < D * (D / 4); f += kChainThreads) {
                const int c = f >> 5, x4 = (f & 31) * 4;
                *reinterpret_cast<float4*>(dst + c * D + x4) = *reinterpret_cast<const float4*>(dSp + c * LDX + x4);
            }
        }
        // dU = (scale P)^T dO + Kb dSp: rows 4 rg.., columns 4 cg..
        {
            const int rg = tid >> 5, cg = tid & 31;
            float acc[4][4] = {};
#pragma unroll 4
            for (int j = 0; j < C; ++j) {
                const float4 a = *reinterpret_cast<const float4*>(Ps + j * LDR + 4 * rg);
                const float4 b = *reinterpret_cast<const float4*>(dOs + j * LDX + 4 * cg);
                const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int p = 0; p < 4; ++p)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[p][q] += av[p] * bv[q];
            }
#pragma unroll 4
            for (int c = 0; c < D; ++c) {
                const float4 a = *reinterpret_cast<const float4*>(KbT + c * LDR + 4 * rg);
                const float4 b = *reinterpret_cast<const float4*>(dSp + c * LDX + 4 * cg);
                const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int p = 0; p < 4; ++p)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[p][q] += av[p] * bv[q];
            }
            float* gdu = du_out + task * (int64_t)(C * D);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float4 v = make_float4(acc[p][0], acc[p][1], acc[p][2], acc[p][3]);
                *reinterpret_cast<float4*>(dUs + (4 * rg + p) * LDX + 4 * cg) = v;
                *reinterpret_cast<float4*>(gdu + (4 * rg + p) * D + 4 * cg) = v;
            }
        }
        __syncthreads();   // KbT is read; dU is complete
        // Qs = scale Xq (the second half of the merged image) over KbT
        for (int u = tid; u < 8 * D; u += kChainThreads) {
            const int c = u & 127, ng = u >> 7;
            float x[8];
            hilo8(slot + SLOT_WQH + 16384 + u * 16, slot + SLOT_WQL + 16384 + u * 16, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) Qs[(8 * ng + e) * LDX + c] = x[e];
        }
        __syncthreads();
        // dSp <- Diag(e^{G_C}) dSp + Qs^T dO + (-W)^T dU: rows c = 4 rg.., columns x = 8 cg..
        {
            const int rg = tid >> 4, cg = tid & 15;
            float acc[4][8];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float e = egc[4 * rg + p];
                const float4 s0 = *reinterpret_cast<const float4*>(dSp + (4 * rg + p) * LDX + 8 * cg);
                const float4 s1 = *reinterpret_cast<const float4*>(dSp + (4 * rg + p) * LDX + 8 * cg + 4);
                acc[p][0] = e * s0.x; acc[p][1] = e * s0.y; acc[p][2] = e * s0.z; acc[p][3] = e * s0.w;
                acc[p][4] = e * s1.x; acc[p][5] = e * s1.y; acc[p][6] = e * s1.z; acc[p][7] = e * s1.w;
            }
#pragma unroll 2
            for (int r = 0; r < C; ++r) {
                const float4 a = *reinterpret_cast<const float4*>(Qs + r * LDX + 4 * rg);
                const float4 b0 = *reinterpret_cast<const float4*>(dOs + r * LDX + 8 * cg);
                const float4 b1 = *reinterpret_cast<const float4*>(dOs + r * LDX + 8 * cg + 4);
                const float4 w = *reinterpret_cast<const float4*>(Wn + r * LDX + 4 * rg);
                const float4 u0 = *reinterpret_cast<const float4*>(dUs + r * LDX + 8 * cg);
                const float4 u1 = *reinterpret_cast<const float4*>(dUs + r * LDX + 8 * cg + 4);
                const float av[4] = {a.x, a.y, a.z, a.w}, wv[4] = {w.x, w.y, w.z, w.w};
                const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                for (int p = 0; p < 4; ++p)
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[p][q] += av[p] * bv[q] + wv[p] * uv[q];
            }
            // (each thread reads and writes only its own elements of dSp here)
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                *reinterpret_cast<float4*>(dSp + (4 * rg + p) * LDX + 8 * cg) =
                    make_float4(acc[p][0], acc[p][1], acc[p][2], acc[p][3]);
                *reinterpret_cast<float4*>(dSp + (4 * rg + p) * LDX + 8 * cg + 4) =
                    make_float4(acc[p][4], acc[p][5], acc[p][6], acc[p][7]);
            }
        }
    }
    __syncthreads();
    if (dS0 != nullptr)
        for (int e = tid; e < D * D; e += kChainThreads) dS0[sbase + e] = dSp[(e >> 7) * LDX + (e & 127)];
}

// ---- chunk-parallel gradients ------------------------------------------------------
constexpr int kChunkThreads = 512;
constexpr int kBwdCtas = 152;   // persistent CTAs of the chunk kernel (the workspace holds a scratch area for each)
constexpr int MR = C * D;       // floats of a [64][128] matrix
constexpr int MQ = C * C;       // floats of a [64][64] matrix
// Per-CTA scratch (fp32, in the workspace; offsets in floats).  [dW | dU] and
// [dBk | dBv] are [64][256] (the two side by side).
enum : int {
    SC_K = 0, SC_Q = SC_K + MR, SC_V = SC_Q + MR, SC_DO = SC_V + MR, SC_WN = SC_DO + MR,
    SC_PRE = SC_WN + MR, SC_EA = SC_PRE + MR, SC_KL = SC_EA + MR, SC_QL = SC_KL + MR,
    SC_U = SC_QL + MR, SC_DXQ = SC_U + MR, SC_DWU = SC_DXQ + MR, SC_DKB = SC_DWU + 2 * MR,
    SC_DBKV = SC_DKB + MR, SC_XVB = SC_DBKV + 2 * MR, SC_GB = SC_XVB + 2 * MR, SC_GF = SC_GB + MR,
    SC_GC = SC_GF + MR,
    SC_DP = SC_GC + MR, SC_A = SC_DP + MQ, SC_T = SC_A + MQ, SC_DT = SC_T + MQ, SC_TMP = SC_DT + MQ,
    SC_DM = SC_TMP + MQ, SC_DA = SC_DM + MQ,
    SC_TOTAL = SC_DA + MQ
};
// shared memory of the chunk kernel: the GEMM staging area, then small tables
constexpr int GEMM_FLOATS = 128 * 68 + 4 * 128 * 68;   // the largest staging (the gated A product)
constexpr uint32_t BK_TOT = GEMM_FLOATS * 4;            // tot [4][128]: e^g products over each 16-token block
constexpr uint32_t BK_PT = BK_TOT + 4 * D * 4;          // ptot [4 B][4 b][128]: prod of tot over blocks [B, b)
constexpr uint32_t BK_BETA = BK_PT + 16 * D * 4;        // beta [64]
constexpr uint32_t BK_DEC = BK_BETA + C * 4;            // dEC [128]
constexpr uint32_t BK_EC = BK_DEC + D * 4;              // e^{G_C} [128]
constexpr uint32_t BK_TOTAL = BK_EC + D * 4;
static_assert(BK_TOTAL <= 232448, "shared memory of the chunk kernel");

// The float4 unit i of an [R][CO] matrix -> its row r and first column c.  For a
// transposed store (TR), each warp covers eight consecutive rows of four column
// groups, which keeps the scattered shared-memory stores free of most conflicts.
template <int R, int CO, bool TR>
__device__ __forceinline__ void unit_rc(int i, int& r, int& c) {
    if (TR) {
        const int rest = i >> 3;
        c = 4 * (rest % (CO / 4));
        r = (rest / (CO / 4)) * 8 + (i & 7);
    } else {
        r = i / (CO / 4);
        c = 4 * (i % (CO / 4));
    }
}

// An [R][CO] fp32 matrix in global memory (row stride ld, 16-byte aligned rows) into
// shared memory, each float4 passed through f(r, c, v) first: dst[r][c] (TR false) or
// dst[c][r] (TR true), row stride ldd.  Four float4 loads in flight per thread.
struct Ident {
    __device__ __forceinline__ void operator()(int, int, float4&) const {}
};
template <int R, int CO, bool TR, typename F = Ident>
__device__ __forceinline__ void stage(const float* src, int ld, float* dst, int ldd, F f = F()) {
    constexpr int NV = R * (CO / 4);
    for (int i0 = threadIdx.x; i0 < NV; i0 += 4 * kChunkThreads) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kChunkThreads;
            if (i < NV) {
                int r, c;
                unit_rc<R, CO, TR>(i, r, c);
                v[u] = *reinterpret_cast<const float4*>(src + (int64_t)r * ld + c);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kChunkThreads;
            if (i >= NV) break;
            int r, c;
            unit_rc<R, CO, TR>(i, r, c);
            f(r, c, v[u]);
            if (TR) {
                dst[(c + 0) * ldd + r] = v[u].x;
                dst[(c + 1) * ldd + r] = v[u].y;
                dst[(c + 2) * ldd + r] = v[u].z;
                dst[(c + 3) * ldd + r] = v[u].w;
            } else {
                *reinterpret_cast<float4*>(dst + r * ldd + c) = v[u];
            }
        }
    }
}

// C[M x N] (row-major, ldc) = alpha A B (+ C when acc), fp32, by the whole CTA, with
// the operands staged into shared memory by the caller's functions: sa(As, LA) writes
// As[k][m], sb(Bs, LB, b) writes Bs[k][n] for B variant b (nb of them: with nb = 4 the
// output rows [16 b, 16 b + 16) use variant b).  A thread computes 4 x 4 outputs.
template <int M, int N, int K, typename SA, typename SB>
__device__ __forceinline__ void cta_mm(float* Cm, int ldc, SA sa, SB sb, int nb, float alpha, bool acc, float* sm) {
    constexpr int LA = M + 4, LB = N + 4;
    float* As = sm;
    float* Bs = sm + K * LA;
    __syncthreads();   // the previous readers of the staging area and writers of the operands are done
    sa(As, LA);
    for (int b = 0; b < nb; ++b) sb(Bs + b * K * LB, LB, b);
    __syncthreads();
    constexpr int TN = N / 4;
    for (int t = threadIdx.x; t < (M / 4) * TN; t += kChunkThreads) {
        const int tm = t / TN, tn = t % TN;
        const float* Bsb = Bs + (nb > 1 ? ((4 * tm) >> 4) * K * LB : 0);
        float a4[4][4] = {};
#pragma unroll 4
        for (int k = 0; k < K; ++k) {
            const float4 a = *reinterpret_cast<const float4*>(As + k * LA + 4 * tm);
            const float4 b = *reinterpret_cast<const float4*>(Bsb + k * LB + 4 * tn);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int q = 0; q < 4; ++q) a4[p][q] += av[p] * bv[q];
        }
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            float* cr = Cm + (int64_t)(4 * tm + p) * ldc + 4 * tn;
            float4 v = make_float4(alpha * a4[p][0], alpha * a4[p][1], alpha * a4[p][2], alpha * a4[p][3]);
            if (acc) {
                const float4 o = *reinterpret_cast<const float4*>(cr);
                v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
            }
            *reinterpret_cast<float4*>(cr) = v;
        }
    }
    __syncthreads();   // C is complete
}

// The plain case: op(A)(m, k) = A[m lda + k] (ta false) or A[k lda + m]; op(B)(k, n) =
// B[k ldb + n] (tb false) or B[n ldb + k].
template <int M, int N, int K>
__device__ __noinline__ void cta_gemm(float* Cm, int ldc, const float* A, int lda, bool ta, const float* B, int ldb,
                                      bool tb, float alpha, bool acc, float* sm) {
    cta_mm<M, N, K>(
        Cm, ldc,
        [&](float* As, int LA) {
            if (ta) stage<K, M, false>(A, lda, As, LA);
            else stage<M, K, true>(A, lda, As, LA);
        },
        [&](float* Bs, int LB, int) {
            if (tb) stage<N, K, true>(B, ldb, Bs, LB);
            else stage<K, N, false>(B, ldb, Bs, LB);
        },
        1, alpha, acc, sm);
}

template <typename TIn>
__device__ __forceinline__ float ld_in(const TIn* p) { return to_f32<TIn>(*p); }

// Decay factors of the gated products, applied while staging (see bwd_chunk_kernel):
// Krf(b): k_j e^{G_m(b) - G_j}, 0 for j past block b (staging k, rows j)
struct Krf {
    const float* pre;
    const float* ptot;
    int b;
    __device__ __forceinline__ void operator()(int j, int c, float4& x) const {
        const int B = j >> 4;
        if (B > b) {
            x = make_float4(0.f, 0.f, 0.f, 0.f);
            return;
        }
        const float4 pr = *reinterpret_cast<const float4*>(pre + j * D + c);
        const float* pt = ptot + (B * 4 + b) * D + c;
        x.x *= pt[0] / pr.x; x.y *= pt[1] / pr.y; x.z *= pt[2] / pr.z; x.w *= pt[3] / pr.w;
    }
};
// Alp(Bo): a_r e^{G_r - G_m(b(r))} times the block totals over [Bo, b(r)), 0 for rows
// before block Bo (staging k e^{G - G_m} or q e^{G - G_m}, rows r)
struct Alp {
    const float* ptot;
    int Bo;
    __device__ __forceinline__ void operator()(int r, int c, float4& x) const {
        const int b = r >> 4;
        if (b < Bo) {
            x = make_float4(0.f, 0.f, 0.f, 0.f);
            return;
        }
        const float* pt = ptot + (Bo * 4 + b) * D + c;
        x.x *= pt[0]; x.y *= pt[1]; x.z *= pt[2]; x.w *= pt[3];
    }
};

// A[r][j] = sum_c kL[r][c] Krf(b(r))(k)[j][c]: the gated k k^T product (before masking)
__device__ __noinline__ void gated_kk(float* Am, const float* KL, const float* K_, const float* pre, const float* ptot,
                                      float* sm) {
    cta_mm<C, C, D>(
        Am, C, [&](float* As, int LA) { stage<C, D, true>(KL, D, As, LA); },
        [&](float* Bs, int LB, int b) { stage<C, D, true>(K_, D, Bs, LB, Krf{pre, ptot, b}); }, 4, 1.f, false, sm);
}
// out[r][c] = sum_j M[r][j] Krf(b(r))(k)[j][c]
__device__ __noinline__ void gated_rows(float* out, const float* M, const float* K_, const float* pre,
                                        const float* ptot, float* sm) {
    cta_mm<C, D, C>(
        out, D, [&](float* As, int LA) { stage<C, C, true>(M, C, As, LA); },
        [&](float* Bs, int LB, int b) { stage<C, D, false>(K_, D, Bs, LB, Krf{pre, ptot, b}); }, 4, 1.f, false, sm);
}
// out[j][c] (+)= sum_r M[r][j] Alp(b(j))(aL)[r][c]
__device__ __noinline__ void gated_cols(float* out, const float* M, const float* aL, const float* ptot, bool acc,
                                        float* sm) {
    cta_mm<C, D, C>(
        out, D, [&](float* As, int LA) { stage<C, C, false>(M, C, As, LA); },
        [&](float* Bs, int LB, int b) { stage<C, D, false>(aL, D, Bs, LB, Alp{ptot, b}); }, 4, 1.f, acc, sm);
}

// One (chunk, head) task per CTA at a time: the chunk's dq, dk, dv, dg, dbeta from the
// entering state S, the gradient dS' of the state after it, dU and dO, plus the
// forward's W and U~ (slot), all in fp32.  Decay factors are formed per 16-token row
// block from products over exactly the tokens they span (never e^{-G} alone):
// e^{G_r - G_m(b)} = pre_r for a row r of block b (m(b) the token before the block),
// e^{G_m(b) - G_j} = ptot[B(j)][b] / pre_j for j up to the end of block b.
__global__ void __launch_bounds__(kChunkThreads, 1)
bwd_chunk_kernel(const Plan pl, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                 const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ g,
                 const __nv_bfloat16* __restrict__ beta, float scale, const float* __restrict__ dO,
                 const float* __restrict__ states, const float* __restrict__ dsp, const float* __restrict__ du,
                 float* __restrict__ scratch, float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv,
                 float* __restrict__ dg, float* __restrict__ dbeta) {
    extern __shared__ __align__(16) uint8_t smem[];
    float* gsm = reinterpret_cast<float*>(smem);
    float* tot = reinterpret_cast<float*>(smem + BK_TOT);
    float* ptot = reinterpret_cast<float*>(smem + BK_PT);
    float* bs = reinterpret_cast<float*>(smem + BK_BETA);
    float* dec = reinterpret_cast<float*>(smem + BK_DEC);
    float* ec = reinterpret_cast<float*>(smem + BK_EC);
    const int tid = threadIdx.x;
    const int H = pl.H;
    float* sc = scratch + (int64_t)blockIdx.x * SC_TOTAL;
    float* K_ = sc + SC_K;
    float* Q_ = sc + SC_Q;
    float* V_ = sc + SC_V;
    float* DO_ = sc + SC_DO;
    float* WN = sc + SC_WN;
    float* PRE = sc + SC_PRE;
    float* EA = sc + SC_EA;
    float* KL = sc + SC_KL;
    float* QL = sc + SC_QL;
    float* U = sc + SC_U;
    float* DXQ = sc + SC_DXQ;
    float* DWU = sc + SC_DWU;    // [dW | dU] [64][256]
    float* DKB = sc + SC_DKB;
    float* DBKV = sc + SC_DBKV;  // [dBk | dBv] [64][256]
    float* XVB = sc + SC_XVB;    // [Diag(beta) X | Diag(beta) v] [64][256]
    float* GB = sc + SC_GB;
    float* GF = sc + SC_GF;
    float* GC = sc + SC_GC;
    float* DP = sc + SC_DP;
    float* Am = sc + SC_A;
    float* Tm = sc + SC_T;
    float* DT = sc + SC_DT;
    float* TMP = sc + SC_TMP;
    float* DM = sc + SC_DM;
    float* DA = sc + SC_DA;
    const int64_t ntasks = pl.max_chunks * H;

    for (int64_t task = blockIdx.x; task < ntasks; task += gridDim.x) {
        const Chunk ch = decode_task(pl, task);
        if (!ch.valid) continue;
        const int h = ch.h;
        const int64_t c0 = ch.c0;
        const int L = (ch.eos - c0 < (int64_t)C) ? (int)(ch.eos - c0) : C;
        const uint8_t* slot = pl.slots + task * (int64_t)SLOT_BYTES;
        const float* S = states + task * (int64_t)(D * D);
        const float* DSP = dsp + task * (int64_t)(D * D);
        const float* DU = du + task * (int64_t)(C * D);
        __syncthreads();   // the previous task is done with the scratch and the tables

        // ---- inputs (0 past the sequence end), U~ and dU, prefix products, -W ----------
        for (int u = tid; u < MR / 8; u += kChunkThreads) {
            const int r = u >> 4, c = 8 * (u & 15);
            const int64_t ti = ((c0 + r) * H + h) * D + c;
            float kx[8], qx[8], vx[8];
            if (r < L) {
                tc::unpack8(*reinterpret_cast<const uint4*>(k + ti), kx);
                tc::unpack8(*reinterpret_cast<const uint4*>(q + ti), qx);
                tc::unpack8(*reinterpret_cast<const uint4*>(v + ti), vx);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) kx[e] = qx[e] = vx[e] = 0.f;
            }
            const int o = r * D + c;
            *reinterpret_cast<float4*>(K_ + o) = make_float4(kx[0], kx[1], kx[2], kx[3]);
            *reinterpret_cast<float4*>(K_ + o + 4) = make_float4(kx[4], kx[5], kx[6], kx[7]);
            *reinterpret_cast<float4*>(Q_ + o) = make_float4(qx[0], qx[1], qx[2], qx[3]);
            *reinterpret_cast<float4*>(Q_ + o + 4) = make_float4(qx[4], qx[5], qx[6], qx[7]);
            *reinterpret_cast<float4*>(V_ + o) = make_float4(vx[0], vx[1], vx[2], vx[3]);
            *reinterpret_cast<float4*>(V_ + o + 4) = make_float4(vx[4], vx[5], vx[6], vx[7]);
        }
        for (int u = tid; u < MR / 4; u += kChunkThreads) {
            const int r = u >> 5, c = 4 * (u & 31);
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < L) x = *reinterpret_cast<const float4*>(dO + ((c0 + r) * H + h) * D + c);
            *reinterpret_cast<float4*>(DO_ + r * D + c) = x;
            *reinterpret_cast<float4*>(U + r * D + c) =
                *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(slot + SLOT_UT) + r * D + c);
            *reinterpret_cast<float4*>(DWU + r * 2 * D + D + c) = *reinterpret_cast<const float4*>(DU + r * D + c);
        }
        if (tid < C) bs[tid] = tid < L ? ld_in(beta + (c0 + tid) * H + h) : 0.f;
        {
            const int c = tid & 127, J = tid >> 7;
            float run = 1.f;
            for (int u = 0; u < 16; ++u) {
                const int r = 16 * J + u;
                const float eg = r < L ? __expf(ld_in(g + ((c0 + r) * H + h) * D + c)) : 1.f;
                run *= eg;
                PRE[r * D + c] = run;
            }
            tot[J * D + c] = run;
        }
        for (int u = tid; u < 8 * D; u += kChunkThreads) {
            const int c = u & 127, ng = u >> 7;
            float x[8];
            hilo8(slot + SLOT_WQH + u * 16, slot + SLOT_WQL + u * 16, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) WN[(8 * ng + e) * D + c] = x[e];
        }
        __syncthreads();
        if (tid < D) {
            const int c = tid;
            ec[c] = tot[c] * tot[D + c] * tot[2 * D + c] * tot[3 * D + c];
            for (int B = 0; B < 4; ++B) {
                float p = 1.f;
                for (int b = 0; b < 4; ++b) {
                    ptot[(B * 4 + b) * D + c] = b >= B ? p : 0.f;
                    if (b >= B) p *= tot[b * D + c];
                }
            }
        }
        // derived operands: e^{G_r}, a e^{G_r - G_m(b(r))}, Diag(beta) X, Diag(beta) v
        for (int u = tid; u < MR / 4; u += kChunkThreads) {
            const int r = u >> 5, c = 4 * (u & 31), B = r >> 4;
            const float4 pr = *reinterpret_cast<const float4*>(PRE + r * D + c);
            const float4 kx = *reinterpret_cast<const float4*>(K_ + r * D + c);
            const float4 qx = *reinterpret_cast<const float4*>(Q_ + r * D + c);
            const float4 vx = *reinterpret_cast<const float4*>(V_ + r * D + c);
            float4 bf = make_float4(1.f, 1.f, 1.f, 1.f);
            for (int b = 0; b < B; ++b) {
                bf.x *= tot[b * D + c]; bf.y *= tot[b * D + c + 1]; bf.z *= tot[b * D + c + 2]; bf.w *= tot[b * D + c + 3];
            }
            const float4 ea = make_float4(bf.x * pr.x, bf.y * pr.y, bf.z * pr.z, bf.w * pr.w);
            const float br = bs[r];
            *reinterpret_cast<float4*>(EA + r * D + c) = ea;
            *reinterpret_cast<float4*>(KL + r * D + c) = make_float4(kx.x * pr.x, kx.y * pr.y, kx.z * pr.z, kx.w * pr.w);
            *reinterpret_cast<float4*>(QL + r * D + c) = make_float4(qx.x * pr.x, qx.y * pr.y, qx.z * pr.z, qx.w * pr.w);
            *reinterpret_cast<float4*>(XVB + r * 2 * D + c) =
                make_float4(br * kx.x * ea.x, br * kx.y * ea.y, br * kx.z * ea.z, br * kx.w * ea.w);
            *reinterpret_cast<float4*>(XVB + r * 2 * D + D + c) = make_float4(br * vx.x, br * vx.y, br * vx.z, br * vx.w);
        }

        // ---- the products with S, dS', U ----------------------------------------------------
        cta_gemm<C, D, D>(U, D, WN, D, false, S, D, false, 1.f, true, gsm);              // U = U~ - W S
        cta_gemm<C, D, D>(DXQ, D, DO_, D, false, S, D, true, scale, false, gsm);         // scale dO S^T
        cta_gemm<C, D, D>(DWU, 2 * D, DU, D, false, S, D, true, -1.f, false, gsm);       // dW = -dU S^T
        cta_gemm<C, D, D>(DKB, D, U, D, false, DSP, D, true, 1.f, false, gsm);           // U dS'^T
        cta_gemm<C, C, D>(DP, C, DO_, D, false, U, D, true, scale, false, gsm);          // scale dO U^T
        {
            // dEC[c] = sum_x dS'[c][x] S[c][x]: four threads per channel, eight float4 each
            const int c = tid >> 2, part = tid & 3;
            float4 a4[8], b4[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                a4[i] = *reinterpret_cast<const float4*>(DSP + c * D + part * 32 + 4 * i);
                b4[i] = *reinterpret_cast<const float4*>(S + c * D + part * 32 + 4 * i);
            }
            float a = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) a += a4[i].x * b4[i].x + a4[i].y * b4[i].y + a4[i].z * b4[i].z + a4[i].w * b4[i].w;
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            if (part == 0) dec[c] = a;
        }
        // A: the gated k k^T product per row block (strictly lower)
        gated_kk(Am, KL, K_, PRE, ptot, gsm);
        for (int e = tid; e < MQ; e += kChunkThreads) {
            const int r = e >> 6, j = e & 63;
            if (j >= r) Am[e] = 0.f;
            if (j > r) DP[e] = 0.f;
        }
        __syncthreads();
        // T = (I + Diag(beta) A)^{-1} in shared memory: eight threads per column, rows in order
        {
            float* Ns = gsm;                // Diag(beta) A [64][65]
            float* Ts = gsm + C * (C + 1);  // T [64][65]
            for (int e = tid; e < MQ; e += kChunkThreads) Ns[(e >> 6) * (C + 1) + (e & 63)] = bs[e >> 6] * Am[e];
            __syncthreads();
            const int j = tid >> 3, part = tid & 7;
            for (int r = 0; r < C; ++r) {
                float a = 0.f;
                for (int i = j + part; i < r; i += 8) a += Ns[r * (C + 1) + i] * Ts[i * (C + 1) + j];
                a += __shfl_xor_sync(0xffffffffu, a, 1);
                a += __shfl_xor_sync(0xffffffffu, a, 2);
                a += __shfl_xor_sync(0xffffffffu, a, 4);
                if (part == 0) Ts[r * (C + 1) + j] = r == j ? 1.f : (r < j ? 0.f : -a);
                __syncwarp();
            }
            __syncthreads();
            for (int e = tid; e < MQ; e += kChunkThreads) Tm[e] = Ts[(e >> 6) * (C + 1) + (e & 63)];
        }
        // dT = [dW | dU] [Diag(beta) X | Diag(beta) v]^T;  [dBk | dBv] = T^T [dW | dU];
        // dM = -T^T dT T^T
        cta_gemm<C, C, 2 * D>(DT, C, DWU, 2 * D, false, XVB, 2 * D, true, 1.f, false, gsm);
        cta_gemm<C, 2 * D, C>(DBKV, 2 * D, Tm, C, true, DWU, 2 * D, false, 1.f, false, gsm);
        cta_gemm<C, C, C>(TMP, C, DT, C, false, Tm, C, true, 1.f, false, gsm);
        cta_gemm<C, C, C>(DM, C, Tm, C, true, TMP, C, false, -1.f, false, gsm);
        for (int e = tid; e < MQ; e += kChunkThreads) {
            const int r = e >> 6, j = e & 63;
            DA[e] = j < r ? bs[r] * DM[e] : 0.f;
        }
        // dbeta = rowsum(dM A) + rowsum(dBk X) + rowsum(dBv v);  dv = Diag(beta) dBv
        {
            const int r = tid >> 3, part = tid & 7;
            float a = 0.f;
            for (int j = part; j < C; j += 8) a += DM[r * C + j] * Am[r * C + j];
            for (int c = part; c < D; c += 8)
                a += DBKV[r * 2 * D + c] * K_[r * D + c] * EA[r * D + c] + DBKV[r * 2 * D + D + c] * V_[r * D + c];
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            if (part == 0 && r < L) dbeta[(c0 + r) * H + h] = a;
        }
        for (int u = tid; u < MR / 4; u += kChunkThreads) {
            const int r = u >> 5, c = 4 * (u & 31);
            if (r < L) {
                const float4 x = *reinterpret_cast<const float4*>(DBKV + r * 2 * D + D + c);
                const float br = bs[r];
                *reinterpret_cast<float4*>(dv + ((c0 + r) * H + h) * D + c) =
                    make_float4(br * x.x, br * x.y, br * x.z, br * x.w);
            }
        }
        // the gated back-products: GB = (dA k e^{G_m - G_j}) per row block, GF the same with
        // dP (both times e^{G_r - G_m} later); GC = the transposed ones with kL and qL (times
        // 1 / pre_j later)
        gated_rows(GB, DA, K_, PRE, ptot, gsm);
        gated_rows(GF, DP, K_, PRE, ptot, gsm);
        gated_cols(GC, DA, KL, ptot, false, gsm);
        gated_cols(GC, DP, QL, ptot, true, gsm);

        // ---- dq, dk, dG ----------------------------------------------------------------------
        for (int e = tid; e < MR; e += kChunkThreads) {
            const int r = e >> 7, c = e & 127, B = r >> 4;
            const float pr = PRE[e], ea = EA[e], kk = K_[e], qq = Q_[e];
            const float kbf = ptot[(B * 4 + 3) * D + c] * tot[3 * D + c] / pr;   // e^{G_C - G_r}
            const float dxe = bs[r] * DBKV[r * 2 * D + c] * ea + GB[e] * pr;  // dX e^G
            const float dye = GC[e] / pr;                                       // dY e^{-G}
            const float dqq = DXQ[e] * ea + GF[e] * pr;                         // dXq e^G
            const float dkb = DKB[e];
            gsm[e] = kk * dxe - kk * dye + qq * dqq - dkb * kk * kbf;   // dG
            gsm[MR + e] = dkb * kk * kbf;                              // dKb Kb
            if (r < L) {
                const int64_t o = ((c0 + r) * H + h) * D + c;
                dq[o] = dqq;
                dk[o] = dxe + dye + dkb * kbf;
            }
        }
        __syncthreads();
        // dg: reverse cumulative sum over the chunk's tokens; the last row also takes
        // dEC e^{G_C} + sum_r dKb Kb
        if (tid < D) {
            const int c = tid;
            float colsum = 0.f;
            for (int r = 0; r < C; ++r) colsum += gsm[MR + r * D + c];
            float acc = dec[c] * ec[c] + colsum;
            for (int r = C - 1; r >= 0; --r) {
                acc += gsm[r * D + c];
                if (r < L) dg[((c0 + r) * H + h) * D + c] = acc;
            }
        }
    }
}

// Workspace of the chunked backward: the forward's (bookkeeping and slots), o as
// bf16, then per (chunk slot, head) the entering state, dS' and dU.
struct BwdLayout {
    size_t fwd, o, states, dsp, du, scratch, total;
};
BwdLayout bwd_layout(int B, int T, int H, int N, bool packed) {
    BwdLayout l{};
    const int64_t cps = ((int64_t)T + C - 1) / C;
    const int64_t max_chunks = packed ? cps + N : (int64_t)B * cps;
    const size_t slots = (size_t)max_chunks * (size_t)H;
    l.fwd = (chunk_tc_workspace(B, T, H, N, packed) + 255) & ~size_t(255);
    l.o = (((size_t)B * (size_t)T * (size_t)H * D * 2) + 255) & ~size_t(255);
    l.states = slots * D * D * 4;
    l.dsp = l.states;
    l.du = slots * C * D * 4;
    l.scratch = (size_t)kBwdCtas * SC_TOTAL * 4;
    l.total = (int64_t)N * H == 0 ? 0 : l.fwd + l.o + l.states + l.dsp + l.du + l.scratch;
    return l;
}

}  // namespace

bool chunk_bwd_supported(kda_dtype in_dt, int K, int V) { return in_dt == KDA_BF16 && K == D && V == D; }

size_t chunk_bwd_workspace(int B, int T, int H, int N, bool packed) { return bwd_layout(B, T, H, N, packed).total; }

cudaError_t chunk_bwd(const ChunkParams& p, const float* dO, const float* dST, float* dq, float* dk, float* dv,
                      float* dg, float* dbeta, float* dS0, void* ws, size_t ws_bytes, int32_t* status,
                      cudaStream_t st) {
    const BwdLayout lo = bwd_layout(p.B, p.T, p.H, p.N, p.cu_seqlens != nullptr);
    if ((int64_t)p.N * p.H == 0) {
        if (status != nullptr) return cudaMemsetAsync(status, 0, sizeof(int32_t), st);
        return cudaSuccess;
    }
    if (ws == nullptr || ws_bytes < lo.total) return cudaErrorMemoryAllocation;
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint8_t* fwd = base;
    void* o = base + lo.fwd;
    float* states = reinterpret_cast<float*>(base + lo.fwd + lo.o);
    float* dsp = reinterpret_cast<float*>(base + lo.fwd + lo.o + lo.states);
    float* du = reinterpret_cast<float*>(base + lo.fwd + lo.o + lo.states + lo.dsp);
    float* scratch = reinterpret_cast<float*>(base + lo.fwd + lo.o + lo.states + lo.dsp + lo.du);
    ChunkParams fp = p;
    fp.o = o;
    fp.final_state = nullptr;
    Plan pl{};
    cudaError_t e = chunk_tc_forward_states(fp, fwd, lo.fwd, states, &pl, status, st);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BC_TOTAL);
    if (e != cudaSuccess) return e;
    bwd_chain_kernel<<<(unsigned)((int64_t)p.N * p.H), kChainThreads, BC_TOTAL, st>>>(pl, dO, dST, dS0, dsp, du);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t tasks = pl.max_chunks * p.H;
    if (tasks > 0) {
        e = cudaFuncSetAttribute(bwd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BK_TOTAL);
        if (e != cudaSuccess) return e;
        const unsigned grid = (unsigned)(tasks < kBwdCtas ? tasks : kBwdCtas);
        bwd_chunk_kernel<<<grid, kChunkThreads, BK_TOTAL, st>>>(
            pl, static_cast<const __nv_bfloat16*>(p.q), static_cast<const __nv_bfloat16*>(p.k),
            static_cast<const __nv_bfloat16*>(p.v), static_cast<const __nv_bfloat16*>(p.g),
            static_cast<const __nv_bfloat16*>(p.beta), p.scale, dO, states, dsp, du, scratch, dq, dk, dv, dg, dbeta);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace kda
