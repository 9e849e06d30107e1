// Chunked KDA prefill on the sm_103a tensor cores (bf16 inputs, K = V = 128).
//
// One CTA owns one (sequence, head) chain and walks it in chunks of C = 64
// tokens.  The fp32 state lives in tensor memory for the whole sequence as
// S^T (lane = value column x, column = key channel c).  Per chunk (G = in-chunk
// cumulative log-decay per key channel; all products below are the chunk
// algebra of the recurrence, see kda_chunk_simt.cu):
//
//   A, P   gated in-chunk products, per 32-token row block R with the decay
//          reference at the block centre (so every factor is within e^{+-80}):
//          D_R[i, j] = L_R[i] . Rt_R[j]   (tcgen05, M = 64: 32 rows of k and 32
//          rows of q, N = 32 (R+1))
//   T      = (I + Diag(beta) A)^{-1}, 16x16 block forward substitution (CUDA cores)
//   W^T    = (k e^G)^T (T Diag(beta))^T,   U~^T = v^T (T Diag(beta))^T     (tcgen05)
//   U^T    = U~^T - S^T W^T                                              (tcgen05, negated A)
//   O^T    = S^T (q e^G)^T + U^T P^T                                     (tcgen05)
//   S^T   <- S^T Diag(e^{G_C}) + U^T (k e^{G_C - G})                     (tcgen05, in TMEM)
//
// Operand precision: every operand that feeds o or the state directly is
// split x = hi + lo into two bf16 values and multiplied as hi*hi + hi*lo +
// lo*hi (about 16 significant bits); W and the correction W S use one bf16
// term; v is exact in bf16.  Decay factors are running products of e^{g}
// over exactly the tokens they span, built from per-16-token-block prefix
// products (each >= e^-80 since g >= -5, so ratios inside a block are safe)
// and block totals; nothing overflows and nothing cancels.
//
// Sources: "ISEEKYAN/k3" README (chunked KDA forward as the compute path);
// "kimi-k3-mlx" review, "The A_log shape mismatch ..." (per-channel decay) and
// "Attention is 93 layers ..." (gate lower bound -5, 96 heads of 128).
#include <cuda.h>

#include "kda_chunk.h"
#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int C = 64;
constexpr int D = 128;  // K = V
constexpr int NT = 512;  // 16 warps: four warpgroups, each covering all 128 TMEM lanes

// ---- shared memory map (bytes) ----------------------------------------------
constexpr uint32_t SM_STG = 0;            // 64 KB: q | k | v | g tiles, [64][128] bf16, 128B-swizzled halves
constexpr uint32_t SM_OPA = 65536;        // 64 KB, A/P phase: row block 1's L hi|lo (A op [64 i][128 c])
                                          //   and Rt hi|lo (B op [64 j][128 c]); then
                                          //   (q e^G) hi|lo (B op [64 r][128 c], K-major) and
                                          //   (k e^{G_C-G}) hi|lo (B op, MN-major: n = c, k = j)
constexpr uint32_t SM_QT = SM_OPA;
constexpr uint32_t SM_KB = SM_OPA + 32768;
constexpr uint32_t SM_OPB = 131072;       // 48 KB, A/P phase: row block 0's L hi|lo and Rt hi|lo (32 rows); then
constexpr uint32_t SM_TB = SM_OPB;        //   (T Diag beta) hi|lo, B op [64 r][64 j] K-major
constexpr uint32_t SM_PB = SM_OPB + 16384;//   P hi|lo, B op [64 r][64 j] K-major
constexpr uint32_t SM_WB = SM_OPB + 32768;//   W hi, B op MN-major (n = r, k = c)
constexpr uint32_t SM_PRE = 180224;       // fp32 [64][PRE_LD] in-block prefix products of e^g,
constexpr int PRE_LD = 132;               //   later Diag(beta) A and T as fp32 [64][MAT_LD] each
constexpr int MAT_LD = 68;
constexpr uint32_t SM_AF = SM_PRE;
constexpr uint32_t SM_TF = SM_PRE + 64 * MAT_LD * 4;
constexpr uint32_t SM_SMALL = SM_PRE + 64 * 2 * MAT_LD * 4;   // 215040
// A/P operands of row block R: L (A, [64 i][128 c]) and Rt (B, [32 (R+1) j][128 c]), hi then lo
__host__ __device__ constexpr uint32_t sm_l(int R) { return R == 0 ? SM_OPB : SM_OPA; }
__host__ __device__ constexpr uint32_t sm_rt(int R) { return R == 0 ? SM_OPB + 32768 : SM_OPA + 32768; }
__host__ __device__ constexpr uint32_t rt_lo(int R) { return R == 0 ? 8192 : 16384; }
constexpr uint32_t SM_TOT = SM_SMALL;     // fp32 [4][128] block totals of e^g
constexpr uint32_t SM_BETA = SM_SMALL + 2048;   // fp32 [64]
constexpr uint32_t SM_EGC = SM_BETA + 256;      // fp32 [128] e^{G_C}
constexpr uint32_t SM_BAR = SM_EGC + 512;       // barriers (tma, mma, w), tmem base, flag
constexpr uint32_t SM_TOTAL = SM_BAR + 64;
static_assert(64 * PRE_LD * 4 <= 2 * 64 * MAT_LD * 4, "prefix array fits the A/T region");
static_assert(SM_TOTAL + 1024 <= 232448, "shared memory");

// ---- tensor memory map (columns) ----------------------------------------------
constexpr uint32_t TM_S = 0;      // S^T fp32 [128 x][128 c]
constexpr uint32_t TM_SH = 128;   // S^T hi (bf16 pairs) [128 x][64]
constexpr uint32_t TM_SL = 192;   // S^T lo
constexpr uint32_t TM_VT = 256;   // v^T (bf16 pairs) [128 x][32]
constexpr uint32_t TM_UH = 288;   // U^T hi [128 x][32]   (alias: (k e^G)^T hi [128 c][32])
constexpr uint32_t TM_UL = 320;   // U^T lo               (alias: (k e^G)^T lo)
constexpr uint32_t TM_KTH = TM_UH;
constexpr uint32_t TM_KTL = TM_UL;
constexpr uint32_t TM_AU = 352;   // U^T accumulator fp32 [128 x][64 r]
constexpr uint32_t TM_AO = 416;   // O^T accumulator fp32 [128 x][64 r]   (alias: W^T [128 c][64 r])
constexpr uint32_t TM_AP = 352;   // A/P accumulators (M = 64 layout): R=0 32 cols, R=1 64 cols
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t kWaitIter = 1u << 26;

__device__ __forceinline__ uint32_t lane_base(int warp) { return (uint32_t)((warp & 3) * 32) << 16; }

template <typename TOut>
__global__ void __launch_bounds__(NT, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mg,
                const ChunkParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte-swizzled TMA tiles need a 1024-byte aligned base
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* beta_s = reinterpret_cast<float*>(smem + SM_BETA);   // [64]
    float* egc_s = reinterpret_cast<float*>(smem + SM_EGC);     // [128]
    float* tot_s = reinterpret_cast<float*>(smem + SM_TOT);     // [4][128]
    float* pre_s = reinterpret_cast<float*>(smem + SM_PRE);     // [64][PRE_LD]
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(smem + SM_BAR);
    uint64_t* bar_mma = bar_tma + 1;
    uint64_t* bar_w = bar_tma + 2;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(bar_tma + 3);
    int* flag_s = reinterpret_cast<int*>(bar_tma + 4);

    const int H = p.H;
    const int h = blockIdx.x % H;
    const int rank = blockIdx.x / H;

    // ---- sequence of this CTA: longest first when packed -------------------
    __shared__ int s_seq;
    int n = rank;
    if (p.cu_seqlens != nullptr && p.N <= 1024) {
        if (tid == 0) s_seq = rank;
        __syncthreads();
        for (int m = tid; m < p.N; m += NT) {
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

    if (warp == 0) tc::tmem_alloc(tmem_base_s, TM_COLS);
    if (tid == 0) {
        tc::bar_init(bar_tma, 1);
        tc::bar_init(bar_mma, 1);
        tc::bar_init(bar_w, 1);
        tc::bar_init_fence();
        *flag_s = 0;
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tmem_base_s;

    uint32_t tma_phase = 0, mma_phase = 0, w_phase = 0;
    bool failed = false;
    bool tma_pending = false;  // a tile load was issued and not yet waited for

    auto issue_tma = [&](int64_t t0) {
        tc::bar_expect_tx(bar_tma, 4u * 16384u);
        const CUtensorMap* maps[4] = {&mq, &mk, &mv, &mg};
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int half = 0; half < 2; ++half)
                tc::tma_load_3d(smem + SM_STG + t * 16384 + half * 8192, maps[t], half * 64, h, (int)t0, bar_tma);
    };
    // Wait for the MMAs committed so far; all threads.
    // One warp polls the barrier; the others park at the CTA barrier, so 16
    // spinning warps do not compete with the tensor core for shared memory.
    auto wait_one = [&](uint64_t* bar, uint32_t& phase) {
        bool ok = true;
        if (warp == 0) ok = tc::bar_wait(bar, phase, kWaitIter);
        phase ^= 1;
        failed = __syncthreads_or(failed || !ok);
        tc::fence_after();
    };
    auto mma_sync = [&]() { wait_one(bar_mma, mma_phase); };
    // Make generic-proxy smem writes and TMEM stores visible to the MMA issuer.
    auto publish = [&]() {
        tc::fence_async_smem();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    };

    if (eos > bos) {
        if (tid == 0) issue_tma(bos);
        tma_pending = true;
    }

    // ---- initial state: S^T in TMEM (lane x holds row x of S^T = column x of S)
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
    {
        const int x = (warp & 3) * 32 + lane;
        const int cbeg = (warp >> 2) * 32;  // warpgroup w covers c in [32 w, 32 w + 32)
        for (int cc = cbeg; cc < cbeg + 32; cc += 16) {
            uint32_t r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                r[i] = __float_as_uint(p.initial_state ? p.initial_state[sbase + (int64_t)(cc + i) * D + x] : 0.f);
            tc::tmem_st16(tm + lane_base(warp) + TM_S + cc, r);
        }
        tc::tmem_st_wait();
    }

    const uint32_t id_n64 = tc::idesc_bf16(128, 64);
    const uint32_t id_n64_neg_bmn = tc::idesc_bf16(128, 64, true, true);
    const uint32_t id_n128_bmn = tc::idesc_bf16(128, 128, false, true);
    const float scale = p.scale;
    TOut* __restrict__ o = reinterpret_cast<TOut*>(p.o);
    const __nv_bfloat16* __restrict__ beta_g = reinterpret_cast<const __nv_bfloat16*>(p.beta);

    // S hi/lo from the fp32 state in TMEM (lane x; warpgroup splits columns).
    auto s_epilogue = [&]() {
        const int cc = (warp >> 2) * 32;
        uint32_t a[32];
        tc::tmem_ld16(tm + lane_base(warp) + TM_S + cc, a);
        tc::tmem_ld16(tm + lane_base(warp) + TM_S + cc + 16, a + 16);
        tc::tmem_ld_wait();
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            __nv_bfloat16 h0, l0, h1, l1;
            tc::split_bf16(__uint_as_float(a[2 * i]), h0, l0);
            tc::split_bf16(__uint_as_float(a[2 * i + 1]), h1, l1);
            hi[i] = tc::pack_bf16(h0, h1);
            lo[i] = tc::pack_bf16(l0, l1);
        }
        tc::tmem_st16(tm + lane_base(warp) + TM_SH + cc / 2, hi);
        tc::tmem_st16(tm + lane_base(warp) + TM_SL + cc / 2, lo);
        tc::tmem_st_wait();
    };
    s_epilogue();

    for (int64_t c0 = bos; c0 < eos && !failed; c0 += C) {
        const int L = (eos - c0 < (int64_t)C) ? (int)(eos - c0) : C;
        // ---- wait for this chunk's tiles ------------------------------------
        wait_one(bar_tma, tma_phase);
        tma_pending = false;
        if (failed) break;

        const uint8_t* qs = smem + SM_STG;
        const uint8_t* ks = smem + SM_STG + 16384;
        const uint8_t* vs = smem + SM_STG + 32768;
        const uint8_t* gs = smem + SM_STG + 49152;
        auto ld_bf = [&](const uint8_t* t, int r, int c) {
            return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(t + tc::swz128(r, c)));
        };
        // 8 consecutive channels [c, c+8) of row r as floats (0 for rows >= L)
        auto ld8 = [&](const uint8_t* t, int r, int c, float* x) {
            if (r < L) {
                tc::unpack8(*reinterpret_cast<const uint4*>(t + tc::swz128(r, c)), x);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] = 0.f;
            }
        };
        auto ld_pre8 = [&](int r, int c, float* x) {
            const float4 a = *reinterpret_cast<const float4*>(pre_s + r * PRE_LD + c);
            const float4 b = *reinterpret_cast<const float4*>(pre_s + r * PRE_LD + c + 4);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        };
        auto ld_tot8 = [&](int J, int c, float* x) {
            const float4 a = *reinterpret_cast<const float4*>(tot_s + J * 128 + c);
            const float4 b = *reinterpret_cast<const float4*>(tot_s + J * 128 + c + 4);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        };

        // ---- (1) in-block prefix products of e^g, block totals --------------------
        {
            const int c = tid & 127, J = tid >> 7;  // block J of channel c
            float gv[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) gv[u] = 16 * J + u < L ? ld_bf(gs, 16 * J + u, c) : 0.f;
            float run = 1.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                run *= __expf(gv[u]);
                pre_s[(16 * J + u) * PRE_LD + c] = run;
            }
            tot_s[J * 128 + c] = run;
        }
        if (tid < C) beta_s[tid] = tid < L ? __bfloat162float(beta_g[(c0 + tid) * H + h]) : 0.f;
        __syncthreads();

        // Every build loop below gives a thread the same 8 channels [8 cg, 8 cg + 8).
        const int cg = (tid >> 3) & 15;

        // ---- (3) A and P: two 32-token row blocks, reference at the block centre --
        // Both blocks' operands are built first (block 0 in OPB, block 1 in OPA),
        // then all their MMAs go out in one round.
#pragma unroll
        for (int R = 0; R < 2; ++R) {
            const int nrows = 32 * (R + 1);  // columns j of this block's products
            // L_R (A operand [64 i][128 c]): i < 32 k-rows, i >= 32 q-rows of block R;
            // e^{G_r - G_mid} = pre_r / tot_{2R} before the centre, pre_r after it
            float itc[8];
            ld_tot8(2 * R, 8 * cg, itc);
#pragma unroll
            for (int u = 0; u < 8; ++u) itc[u] = __fdividef(1.f, itc[u]);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int item = tid + NT * kk;
                const int i = ((item >> 7) << 3) | (item & 7);
                const int r = 32 * R + (i & 31);
                float x[8], pr[8], f[8];
                ld8(i < 32 ? ks : qs, r, 8 * cg, x);
                ld_pre8(r, 8 * cg, pr);
                const bool first = (i & 16) == 0;  // r in the first 16-token block of R
#pragma unroll
                for (int u = 0; u < 8; ++u) f[u] = x[u] * (first ? pr[u] * itc[u] : pr[u]);
                uint4 hi, lo;
                tc::split8(f, hi, lo);
                *reinterpret_cast<uint4*>(smem + sm_l(R) + tc::kmaj(i, 8 * cg, D)) = hi;
                *reinterpret_cast<uint4*>(smem + sm_l(R) + 16384 + tc::kmaj(i, 8 * cg, D)) = lo;
            }
            // Rt_R (B operand [nrows j][128 c]): e^{G_mid - G_j} k_j =
            //   1 / pre_j after the centre, tot_J / pre_j * prod_{J < J2 <= 2R} tot_J2 before it
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int item = tid + NT * kk;
                if (item >= nrows * 16) break;
                const int j = ((item >> 7) << 3) | (item & 7);
                const int J = j >> 4;
                float x[8], pr[8], m[8], t[8];
                ld8(ks, j, 8 * cg, x);
                ld_pre8(j, 8 * cg, pr);
                // in-block ratio first (in (0, 1], or 1/pre_j <= e^80 after the centre),
                // then the totals of the later blocks: every intermediate lies between 1
                // and the true factor, so nothing underflows that the result needs
                if (J == 2 * R + 1) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) m[u] = __fdividef(1.f, pr[u]);
                } else {
                    ld_tot8(J, 8 * cg, t);
#pragma unroll
                    for (int u = 0; u < 8; ++u) m[u] = __fdividef(t[u], pr[u]);
                }
                for (int J2 = J + 1; J2 <= 2 * R; ++J2) {
                    ld_tot8(J2, 8 * cg, t);
#pragma unroll
                    for (int u = 0; u < 8; ++u) m[u] *= t[u];
                }
                float f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) f[u] = x[u] * m[u];
                uint4 hi, lo;
                tc::split8(f, hi, lo);
                *reinterpret_cast<uint4*>(smem + sm_rt(R) + tc::kmaj(j, 8 * cg, D)) = hi;
                *reinterpret_cast<uint4*>(smem + sm_rt(R) + rt_lo(R) + tc::kmaj(j, 8 * cg, D)) = lo;
            }
        }
        publish();
        if (warp == 0) {
            uint64_t ah[2], al[2], bh[2], bl[2];
#pragma unroll
            for (int R = 0; R < 2; ++R) {
                const uint32_t la = tc::smem_u32(smem + sm_l(R)), rb = tc::smem_u32(smem + sm_rt(R));
                ah[R] = tc::sdesc(la, 128, D * 16);
                al[R] = tc::sdesc(la + 16384, 128, D * 16);
                bh[R] = tc::sdesc(rb, 128, D * 16);
                bl[R] = tc::sdesc(rb + rt_lo(R), 128, D * 16);
            }
#pragma unroll
            for (int ks_ = 0; ks_ < D / 16; ++ks_) {
#pragma unroll
                for (int R = 0; R < 2; ++R) {  // two independent accumulators, interleaved
                    const uint32_t d = tm + TM_AP + 32 * R;
                    const uint32_t id = R == 0 ? tc::idesc_bf16(64, 32) : tc::idesc_bf16(64, 64);
                    const uint32_t o = ks_ * 256;
                    tc::mma_ss_w(d, tc::dadv(ah[R], o), tc::dadv(bh[R], o), id, ks_ > 0);
                    tc::mma_ss_w(d, tc::dadv(ah[R], o), tc::dadv(bl[R], o), id, 1);
                    tc::mma_ss_w(d, tc::dadv(al[R], o), tc::dadv(bh[R], o), id, 1);
                }
            }
            tc::commit_w(bar_mma);
        }
        // ---- (2) (k e^G)^T and v^T into TMEM (lane = channel / value column), while
        //      the A/P MMAs run (disjoint TMEM columns, no shared memory they read) --
        {
            const int c = (warp & 3) * 32 + lane;
            const int jb = (warp >> 2) * 16;  // warpgroup w covers tokens [16 w, 16 w + 16)
            const float t0v = tot_s[c], t1v = tot_s[128 + c], t2v = tot_s[256 + c];
            const float pfx[4] = {1.f, t0v, t0v * t1v, t0v * t1v * t2v};
            uint32_t kh[8], kl[8], vv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = jb + 2 * i;
                const float k0 = j < L ? ld_bf(ks, j, c) : 0.f;
                const float k1 = j + 1 < L ? ld_bf(ks, j + 1, c) : 0.f;
                __nv_bfloat16 h0, l0, h1, l1;
                tc::split_bf16(k0 * pfx[j >> 4] * pre_s[j * PRE_LD + c], h0, l0);
                tc::split_bf16(k1 * pfx[(j + 1) >> 4] * pre_s[(j + 1) * PRE_LD + c], h1, l1);
                kh[i] = tc::pack_bf16(h0, h1);
                kl[i] = tc::pack_bf16(l0, l1);
                const __nv_bfloat16 z = __float2bfloat16(0.f);
                const __nv_bfloat16 v0 = j < L ? *reinterpret_cast<const __nv_bfloat16*>(vs + tc::swz128(j, c)) : z;
                const __nv_bfloat16 v1 = j + 1 < L ? *reinterpret_cast<const __nv_bfloat16*>(vs + tc::swz128(j + 1, c)) : z;
                vv[i] = tc::pack_bf16(v0, v1);
            }
            tc::tmem_st8(tm + lane_base(warp) + TM_KTH + jb / 2, kh);
            tc::tmem_st8(tm + lane_base(warp) + TM_KTL + jb / 2, kl);
            tc::tmem_st8(tm + lane_base(warp) + TM_VT + jb / 2, vv);
            if (tid < 128) egc_s[c] = t0v * t1v * t2v * tot_s[384 + c];
        }
        tc::tmem_st_wait();

        mma_sync();
        if (failed) break;

        // ---- (4) (q e^G) (K-major) and (k e^{G_C - G})^T (MN-major) operands -------
        {
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int item = tid + NT * kk;
                const int r = ((item >> 7) << 3) | (item & 7);
                const int J = r >> 4;
                // products of the block totals before (pf) and after (sf) block J
                float pf[8], sf[8], tj[8], t[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) { pf[u] = 1.f; sf[u] = 1.f; }
                for (int J2 = 0; J2 < 4; ++J2) {
                    ld_tot8(J2, 8 * cg, t);
                    if (J2 == J) {
#pragma unroll
                        for (int u = 0; u < 8; ++u) tj[u] = t[u];
                    } else if (J2 < J) {
#pragma unroll
                        for (int u = 0; u < 8; ++u) pf[u] *= t[u];
                    } else {
#pragma unroll
                        for (int u = 0; u < 8; ++u) sf[u] *= t[u];
                    }
                }
                float q[8], k[8], pr[8], fq[8], fk[8];
                ld8(qs, r, 8 * cg, q);
                ld8(ks, r, 8 * cg, k);
                ld_pre8(r, 8 * cg, pr);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    fq[u] = q[u] * (pf[u] * pr[u]);
                    fk[u] = k[u] * (sf[u] * __fdividef(tj[u], pr[u]));
                }
                uint4 hi, lo;
                tc::split8(fq, hi, lo);
                *reinterpret_cast<uint4*>(smem + SM_QT + tc::kmaj(r, 8 * cg, D)) = hi;
                *reinterpret_cast<uint4*>(smem + SM_QT + 16384 + tc::kmaj(r, 8 * cg, D)) = lo;
                tc::split8(fk, hi, lo);
                *reinterpret_cast<uint4*>(smem + SM_KB + tc::mnmaj(8 * cg, r, D)) = hi;
                *reinterpret_cast<uint4*>(smem + SM_KB + 16384 + tc::mnmaj(8 * cg, r, D)) = lo;
            }
        }

        // staging is consumed: prefetch the next chunk into it
        tc::fence_async_smem();
        __syncthreads();
        if (c0 + C < eos) {
            if (tid == 0) issue_tma(c0 + C);
            tma_pending = true;
        }

        // ---- (5) A/P out of TMEM: Diag(beta) A -> fp32, P -> hi/lo operand ---------
        {
            float* Af = reinterpret_cast<float*>(smem + SM_AF);  // [64 r][MAT_LD]
            const int R = (warp >> 2) & 1;                    // warpgroup w: block w % 2,
            const int jb = 32 * (warp >> 3);                  //   columns [32 (w / 2), +32)
            const int ncol = 32 * (R + 1);
            const int i = (warp & 3) * 16 + (lane & 15);      // M = 64 row held by this lane
            const bool is_q = i >= 32;
            const int r = 32 * R + (i & 31);
            uint32_t a[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) a[u] = 0u;
            if (jb < ncol) {
                tc::tmem_ld16(tm + lane_base(warp) + TM_AP + 32 * R + jb, a);
                tc::tmem_ld16(tm + lane_base(warp) + TM_AP + 32 * R + jb + 16, a + 16);
                tc::tmem_ld_wait();
            }
            if (lane < 16) {
                const float br = beta_s[r];
#pragma unroll
                for (int j0 = 0; j0 < 32; j0 += 8) {
                    float v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int j = jb + j0 + u;
                        const float x = __uint_as_float(a[j0 + u]);
                        v[u] = is_q ? (j <= r ? x : 0.f) : (j < r ? br * x : 0.f);
                    }
                    if (is_q) {
                        uint4 hi, lo;
                        tc::split8(v, hi, lo);
                        *reinterpret_cast<uint4*>(smem + SM_PB + tc::kmaj(r, jb + j0, C)) = hi;
                        *reinterpret_cast<uint4*>(smem + SM_PB + 8192 + tc::kmaj(r, jb + j0, C)) = lo;
                    } else {
                        *reinterpret_cast<float4*>(Af + r * MAT_LD + jb + j0) = make_float4(v[0], v[1], v[2], v[3]);
                        *reinterpret_cast<float4*>(Af + r * MAT_LD + jb + j0 + 4) = make_float4(v[4], v[5], v[6], v[7]);
                    }
                }
            }
        }
        __syncthreads();

        // ---- (6) T = (I + Diag(beta) A)^{-1} ----------------------------------------
        {
            const float* N = reinterpret_cast<const float*>(smem + SM_AF);
            float* T = reinterpret_cast<float*>(smem + SM_TF);
            float* Y = reinterpret_cast<float*>(smem + SM_TB);  // scratch: [2][16][16] then [32][32]
            // (blocks above the diagonal are never written; the operand build masks them)
            // diagonal blocks: forward substitution with the column in registers;
            // warp w: block w/2, columns 8 (w%2) .. + 8; lane: column lane/4, rows = lane%4 (mod 4)
            if (warp < 8) {
                const int blk = warp >> 1, col = 8 * (warp & 1) + (lane >> 2), part = lane & 3;
                const int i = 16 * blk + col;
                float x[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) x[m] = (part + 4 * m == col) ? 1.f : 0.f;
                const float* nb = N + 16 * blk * MAT_LD + 16 * blk;
#pragma unroll
                for (int rr = 1; rr < 16; ++rr) {
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        if (part + 4 * m < rr) acc += nb[rr * MAT_LD + part + 4 * m] * x[m];
                    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                    if (part == (rr & 3) && rr > col) x[rr >> 2] = -acc;
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) T[(16 * blk + part + 4 * m) * MAT_LD + i] = x[m];
            }
            __syncthreads();
            // off-diagonal blocks, as two 32 x 32 halves T11 (tokens 0..31) and T22
            // (32..63): first the lower 16 x 16 block inside each half,
            //   T_{2p+1,2p} = -T_{2p+1,2p+1} (N_{2p+1,2p} T_{2p,2p}),   p = 0, 1,
            // then the lower half  T21 = -T22 (N21 T11).
            {
                // one thread per (p, row a, 4 columns): 128 items
                const int pp = tid >> 6, a = (tid >> 2) & 15, b4 = tid & 3;
                const int R = 2 * pp + 1, J = 2 * pp;
                if (tid < 128) {
                    const float* nrow = N + (16 * R + a) * MAT_LD + 16 * J;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int m4 = 0; m4 < 4; ++m4) {
                        const float4 nv = *reinterpret_cast<const float4*>(nrow + 4 * m4);
                        const float nn[4] = {nv.x, nv.y, nv.z, nv.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float4 t = *reinterpret_cast<const float4*>(T + (16 * J + 4 * m4 + u) * MAT_LD + 16 * J + 4 * b4);
                            acc.x += nn[u] * t.x; acc.y += nn[u] * t.y; acc.z += nn[u] * t.z; acc.w += nn[u] * t.w;
                        }
                    }
                    *reinterpret_cast<float4*>(Y + (pp << 8) + (a << 4) + 4 * b4) = acc;
                }
                __syncthreads();
                if (tid < 128) {
                    const float* trow = T + (16 * R + a) * MAT_LD + 16 * R;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const float tv = trow[m];
                        const float4 y = *reinterpret_cast<const float4*>(Y + (pp << 8) + (m << 4) + 4 * b4);
                        acc.x += tv * y.x; acc.y += tv * y.y; acc.z += tv * y.z; acc.w += tv * y.w;
                    }
                    *reinterpret_cast<float4*>(T + (16 * R + a) * MAT_LD + 16 * J + 4 * b4) =
                        make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
                }
                __syncthreads();
            }
            {
                // two lanes per (row a, 4 columns) of a 32 x 32 block, each summing half of
                // the inner range; 256 items over 512 threads
                float* X = Y + 512;
                const int item = tid >> 1, half = tid & 1;
                const int a = item >> 3, b4 = item & 7;
                {
                    const float* nrow = N + (32 + a) * MAT_LD;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    // T11 is zero above its diagonal blocks: columns >= 16 start at row 16
                    const int m0 = (b4 >= 4 ? 4 : 0) + half * (b4 >= 4 ? 2 : 4);
                    const int m1 = b4 >= 4 ? m0 + 2 : m0 + 4;
                    for (int m4 = m0; m4 < m1; ++m4) {
                        const float4 nv = *reinterpret_cast<const float4*>(nrow + 4 * m4);
                        const float nn[4] = {nv.x, nv.y, nv.z, nv.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float4 t = *reinterpret_cast<const float4*>(T + (4 * m4 + u) * MAT_LD + 4 * b4);
                            acc.x += nn[u] * t.x; acc.y += nn[u] * t.y; acc.z += nn[u] * t.z; acc.w += nn[u] * t.w;
                        }
                    }
                    acc.x += __shfl_xor_sync(0xffffffffu, acc.x, 1);
                    acc.y += __shfl_xor_sync(0xffffffffu, acc.y, 1);
                    acc.z += __shfl_xor_sync(0xffffffffu, acc.z, 1);
                    acc.w += __shfl_xor_sync(0xffffffffu, acc.w, 1);
                    if (half == 0) *reinterpret_cast<float4*>(X + a * 32 + 4 * b4) = acc;
                }
                __syncthreads();
                {
                    const float* trow = T + (32 + a) * MAT_LD + 32;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    // T22 is zero above its diagonal blocks: rows < 16 stop at 16
                    const int mlen = a < 16 ? 8 : 16;
                    const int mb = half * mlen;
#pragma unroll 4
                    for (int m = mb; m < mb + mlen; ++m) {
                        const float tv = trow[m];
                        const float4 y = *reinterpret_cast<const float4*>(X + m * 32 + 4 * b4);
                        acc.x += tv * y.x; acc.y += tv * y.y; acc.z += tv * y.z; acc.w += tv * y.w;
                    }
                    acc.x += __shfl_xor_sync(0xffffffffu, acc.x, 1);
                    acc.y += __shfl_xor_sync(0xffffffffu, acc.y, 1);
                    acc.z += __shfl_xor_sync(0xffffffffu, acc.z, 1);
                    acc.w += __shfl_xor_sync(0xffffffffu, acc.w, 1);
                    if (half == 0)
                        *reinterpret_cast<float4*>(T + (32 + a) * MAT_LD + 4 * b4) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
                }
                __syncthreads();
            }
            // T Diag(beta) -> hi/lo B operand [64 r][64 j], K-major
            for (int item = tid; item < 64 * 8; item += NT) {
                const int r = ((item >> 6) << 3) | (item & 7);
                const int jg = (item >> 3) & 7;
                float t[8];
                // (jg is the same for both items of a thread)
                const float4 a = *reinterpret_cast<const float4*>(T + r * MAT_LD + 8 * jg);
                const float4 b = *reinterpret_cast<const float4*>(T + r * MAT_LD + 8 * jg + 4);
                t[0] = a.x; t[1] = a.y; t[2] = a.z; t[3] = a.w; t[4] = b.x; t[5] = b.y; t[6] = b.z; t[7] = b.w;
#pragma unroll
                for (int u = 0; u < 8; ++u) t[u] = (8 * jg + u > r) ? 0.f : t[u] * beta_s[8 * jg + u];
                uint4 hi, lo;
                tc::split8(t, hi, lo);
                *reinterpret_cast<uint4*>(smem + SM_TB + tc::kmaj(r, 8 * jg, C)) = hi;
                *reinterpret_cast<uint4*>(smem + SM_TB + 8192 + tc::kmaj(r, 8 * jg, C)) = lo;
            }
        }
        publish();

        // ---- W^T = (k e^G)^T (T Diag beta)^T into the U accumulator's columns (then
        //      read out); O^T = S^T (q e^G)^T behind it on a second commit -------------
        if (warp == 0) {
            const uint32_t tb = tc::smem_u32(smem + SM_TB), qt = tc::smem_u32(smem + SM_QT);
            const uint64_t tbh = tc::sdesc(tb, 128, C * 16), tbl = tc::sdesc(tb + 8192, 128, C * 16);
            const uint64_t qth = tc::sdesc(qt, 128, D * 16), qtl = tc::sdesc(qt + 16384, 128, D * 16);
#pragma unroll
            for (int ks_ = 0; ks_ < C / 16; ++ks_) {
                const uint64_t bh = tc::dadv(tbh, ks_ * 256), bl = tc::dadv(tbl, ks_ * 256);
                tc::mma_ts_w(tm + TM_AU, tm + TM_KTH + ks_ * 8, bh, id_n64, ks_ > 0);
                tc::mma_ts_w(tm + TM_AU, tm + TM_KTH + ks_ * 8, bl, id_n64, 1);
                tc::mma_ts_w(tm + TM_AU, tm + TM_KTL + ks_ * 8, bh, id_n64, 1);
            }
            tc::commit_w(bar_w);
#pragma unroll
            for (int ks_ = 0; ks_ < D / 16; ++ks_) {
                const uint32_t sh = tm + TM_SH + ks_ * 8, sl = tm + TM_SL + ks_ * 8;
                const uint64_t qh = tc::dadv(qth, ks_ * 256), ql = tc::dadv(qtl, ks_ * 256);
                tc::mma_ts_w(tm + TM_AO, sh, qh, id_n64, ks_ > 0);
                tc::mma_ts_w(tm + TM_AO, sh, ql, id_n64, 1);
                tc::mma_ts_w(tm + TM_AO, sl, qh, id_n64, 1);
            }
            tc::commit_w(bar_mma);
        }
        // decay the fp32 state by e^{G_C} while those MMAs run (they read S hi/lo,
        // not the fp32 state; the K-bar^T U MMA accumulates into it later)
        {
            const int cc = (warp >> 2) * 32;
            uint32_t s0[16], s1[16];
            tc::tmem_ld16(tm + lane_base(warp) + TM_S + cc, s0);
            tc::tmem_ld16(tm + lane_base(warp) + TM_S + cc + 16, s1);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                s0[i] = __float_as_uint(__uint_as_float(s0[i]) * egc_s[cc + i]);
                s1[i] = __float_as_uint(__uint_as_float(s1[i]) * egc_s[cc + 16 + i]);
            }
            tc::tmem_st16(tm + lane_base(warp) + TM_S + cc, s0);
            tc::tmem_st16(tm + lane_base(warp) + TM_S + cc + 16, s1);
            tc::tmem_st_wait();
        }
        wait_one(bar_w, w_phase);

        // ---- W out of TMEM into the B operand (MN-major: n = r, k = c) ----------
        {
            const int c = (warp & 3) * 32 + lane;
            const int rb = (warp >> 2) * 16;
            uint32_t a[16];
            tc::tmem_ld16(tm + lane_base(warp) + TM_AU + rb, a);
            tc::tmem_ld_wait();
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {
                float w[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) w[u] = __uint_as_float(a[8 * g8 + u]);
                *reinterpret_cast<uint4*>(smem + SM_WB + tc::mnmaj(rb + 8 * g8, c, C)) = tc::pack8(w);
            }
        }
        publish();
        mma_sync();  // S^T (q e^G)^T done as well

        // ---- U^T = v^T (T Diag beta)^T - S^T W^T ---------------------------------
        if (warp == 0) {
            const uint32_t tb = tc::smem_u32(smem + SM_TB), wb = tc::smem_u32(smem + SM_WB);
            const uint64_t tbh = tc::sdesc(tb, 128, C * 16), tbl = tc::sdesc(tb + 8192, 128, C * 16);
            const uint64_t wbd = tc::sdesc(wb, C * 16, 128);
#pragma unroll
            for (int ks_ = 0; ks_ < C / 16; ++ks_) {
                tc::mma_ts_w(tm + TM_AU, tm + TM_VT + ks_ * 8, tc::dadv(tbh, ks_ * 256), id_n64, ks_ > 0);
                tc::mma_ts_w(tm + TM_AU, tm + TM_VT + ks_ * 8, tc::dadv(tbl, ks_ * 256), id_n64, 1);
            }
#pragma unroll
            for (int ks_ = 0; ks_ < D / 16; ++ks_)
                tc::mma_ts_w(tm + TM_AU, tm + TM_SH + ks_ * 8, tc::dadv(wbd, ks_ * 2 * C * 16), id_n64_neg_bmn, 1);
            tc::commit_w(bar_mma);
        }
        mma_sync();

        // ---- U hi/lo into TMEM -------------------------------------------------------
        {
            const int rb = (warp >> 2) * 16;
            uint32_t a[16];
            tc::tmem_ld16(tm + lane_base(warp) + TM_AU + rb, a);
            tc::tmem_ld_wait();
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                __nv_bfloat16 h0, l0, h1, l1;
                tc::split_bf16(__uint_as_float(a[2 * i]), h0, l0);
                tc::split_bf16(__uint_as_float(a[2 * i + 1]), h1, l1);
                hi[i] = tc::pack_bf16(h0, h1);
                lo[i] = tc::pack_bf16(l0, l1);
            }
            tc::tmem_st8(tm + lane_base(warp) + TM_UH + rb / 2, hi);
            tc::tmem_st8(tm + lane_base(warp) + TM_UL + rb / 2, lo);
            tc::tmem_st_wait();
        }
        publish();

        // ---- O^T += U^T P^T ;  S^T += U^T (k e^{G_C-G}) --------------------------
        if (warp == 0) {
            const uint32_t pb = tc::smem_u32(smem + SM_PB), kb = tc::smem_u32(smem + SM_KB);
            const uint64_t pbh = tc::sdesc(pb, 128, C * 16), pbl = tc::sdesc(pb + 8192, 128, C * 16);
            const uint64_t kbh = tc::sdesc(kb, D * 16, 128), kbl = tc::sdesc(kb + 16384, D * 16, 128);
#pragma unroll
            for (int ks_ = 0; ks_ < C / 16; ++ks_) {
                const uint32_t uh = tm + TM_UH + ks_ * 8, ul = tm + TM_UL + ks_ * 8;
                const uint64_t ph = tc::dadv(pbh, ks_ * 256), pl = tc::dadv(pbl, ks_ * 256);
                const uint64_t kh = tc::dadv(kbh, ks_ * 2 * D * 16), kl = tc::dadv(kbl, ks_ * 2 * D * 16);
                tc::mma_ts_w(tm + TM_S, uh, kh, id_n128_bmn, 1);
                tc::mma_ts_w(tm + TM_AO, uh, ph, id_n64, 1);
                tc::mma_ts_w(tm + TM_S, uh, kl, id_n128_bmn, 1);
                tc::mma_ts_w(tm + TM_AO, uh, pl, id_n64, 1);
                tc::mma_ts_w(tm + TM_S, ul, kh, id_n128_bmn, 1);
                tc::mma_ts_w(tm + TM_AO, ul, ph, id_n64, 1);
            }
            tc::commit_w(bar_mma);
        }
        mma_sync();

        // ---- o out; S hi/lo for the next chunk ------------------------------------
        {
            const int x = (warp & 3) * 32 + lane;
            const int rb = (warp >> 2) * 16;
            const int cc = (warp >> 2) * 32;
            uint32_t a[16], s0[16], s1[16];
            tc::tmem_ld16(tm + lane_base(warp) + TM_AO + rb, a);
            tc::tmem_ld16(tm + lane_base(warp) + TM_S + cc, s0);
            tc::tmem_ld16(tm + lane_base(warp) + TM_S + cc + 16, s1);
            tc::tmem_ld_wait();
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                __nv_bfloat16 h0, l0, h1, l1;
                tc::split_bf16(__uint_as_float(i < 8 ? s0[2 * i] : s1[2 * i - 16]), h0, l0);
                tc::split_bf16(__uint_as_float(i < 8 ? s0[2 * i + 1] : s1[2 * i - 15]), h1, l1);
                hi[i] = tc::pack_bf16(h0, h1);
                lo[i] = tc::pack_bf16(l0, l1);
            }
            tc::tmem_st16(tm + lane_base(warp) + TM_SH + cc / 2, hi);
            tc::tmem_st16(tm + lane_base(warp) + TM_SL + cc / 2, lo);
            const int64_t ob = ((c0 + rb) * H + h) * (int64_t)D + x;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (rb + i < L) o[ob + (int64_t)i * H * D] = from_f32<TOut>(scale * __uint_as_float(a[i]));
            tc::tmem_st_wait();
        }
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    }

    // ---- final state -----------------------------------------------------------
    if (failed && tma_pending) {
        // drain a tile load that may still be in flight before the CTA exits
        tc::bar_wait(bar_tma, tma_phase, kWaitIter);
    }
    if (p.final_state) {
        const int x = (warp & 3) * 32 + lane;
        const int cbeg = (warp >> 2) * 32;
        for (int cc = cbeg; cc < cbeg + 32; cc += 16) {
            uint32_t s[16];
            tc::tmem_ld16(tm + lane_base(warp) + TM_S + cc, s);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
                p.final_state[sbase + (int64_t)(cc + i) * D + x] = failed ? __int_as_float(0x7fc00000) : __uint_as_float(s[i]);
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, TM_COLS);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// [rows][H][128] bf16 tensor; box = 64 rows x 64 channels of one head, 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int H) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename TOut>
cudaError_t launch_tc(const ChunkParams& p, cudaStream_t st) {
    const int64_t blocks = (int64_t)p.N * p.H;
    if (blocks == 0) return cudaSuccess;
    const int64_t rows = (int64_t)p.B * p.T;
    CUtensorMap mq, mk, mv, mg;
    const int64_t map_rows = rows > 0 ? rows : 1;
    if (!make_map(&mq, p.q, map_rows, p.H) || !make_map(&mk, p.k, map_rows, p.H) ||
        !make_map(&mv, p.v, map_rows, p.H) || !make_map(&mg, p.g, map_rows, p.H))
        return cudaErrorInvalidValue;
    auto kern = chunk_tc_kernel<TOut>;
    const int smem_bytes = (int)SM_TOTAL + 1024;  // + alignment slack
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)blocks, NT, smem_bytes, st>>>(mq, mk, mv, mg, p);
    return cudaGetLastError();
}

}  // namespace

bool chunk_tc_supported(kda_dtype in_dt, int K, int V) { return in_dt == KDA_BF16 && K == D && V == D; }

cudaError_t chunk_tc(kda_dtype out_dt, const ChunkParams& p, cudaStream_t st) {
    if (out_dt == KDA_F32) return launch_tc<float>(p, st);
    return launch_tc<__nv_bfloat16>(p, st);
}

}  // namespace kda
