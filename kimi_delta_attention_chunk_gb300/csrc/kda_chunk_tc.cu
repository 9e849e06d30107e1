// Chunked KDA prefill on the sm_103a tensor cores (bf16 inputs, K = V = 128).
//
// One CTA owns one (sequence, head) chain and walks it in chunks of C = 64
// tokens.  The fp32 state lives in tensor memory for the whole sequence as
// S^T (lane = value column x, column = key channel c).  Per chunk (G = in-chunk
// cumulative log-decay per key channel; all products below are the chunk
// algebra of the recurrence, see kda_chunk_simt.cu):
//
//   A, P   gated in-chunk products, per 16-token row block R with the decay
//          reference at the block start:  D_R[j, r] = Rt_R[j] . L_R[r]
//          (tcgen05, M = 64, N = 32: 16 rows of k and 16 of q)
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
// over exactly the tokens they span (values <= 1, or reciprocals of such
// within one 16-token block, <= e^80 since g >= -5), so nothing overflows and
// nothing cancels.
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
constexpr int NT = 256;

// ---- shared memory map (bytes) ----------------------------------------------
constexpr uint32_t SM_STG = 0;            // 64 KB: q | k | v | g tiles, [64 rows][128] bf16
constexpr uint32_t SM_Q = SM_STG;
constexpr uint32_t SM_K = SM_STG + 16384;
constexpr uint32_t SM_V = SM_STG + 32768;
constexpr uint32_t SM_G = SM_STG + 49152;
constexpr uint32_t SM_QT = 65536;         // 32 KB: (q e^G) hi | lo, B operand [64 r][128 c]
constexpr uint32_t SM_KB = 98304;         // 32 KB: (k e^{G_C-G})^T hi | lo, B operand [128 c][64 j]
constexpr uint32_t SM_X = 131072;         // 48 KB union:
constexpr uint32_t SM_RT = SM_X;          //   A/P phase: Rt_R hi | lo, A operand [64 j][128 c]
constexpr uint32_t SM_LQ = SM_X + 32768;  //               L_R hi | lo, B operand [32][128 c]
constexpr uint32_t SM_TB = SM_X;          //   later: (T Diag(beta)) hi | lo, B operand [64 r][64 j]
constexpr uint32_t SM_PB = SM_X + 16384;  //          P hi | lo, B operand [64 r][64 j]
constexpr uint32_t SM_WB = SM_X + 32768;  //          W hi, B operand [64 r][128 c]
constexpr uint32_t SM_AF = 180224;        // 16 KB fp32 [64][64]: Diag(beta) A   (or e^g, first half)
constexpr uint32_t SM_TF = 196608;        // 16 KB fp32 [64][64]: T               (or e^g, second half)
constexpr uint32_t SM_E = SM_AF;          // 32 KB fp32 [64][128]: e^g during the build
constexpr uint32_t SM_SMALL = 212992;     // beta[64], eGC[128], barriers, tmem base
constexpr uint32_t SM_TOTAL = SM_SMALL + 1024;

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
constexpr uint32_t TM_AP = 352;   // A/P accumulators, 4 x 32 columns, M = 64 layout (alias AU, AO)
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t kWaitIter = 1u << 26;

__device__ __forceinline__ uint32_t lane_base(int warp) { return (uint32_t)((warp & 3) * 32) << 16; }

template <typename TOut>
__global__ void __launch_bounds__(NT, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mg,
                const ChunkParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* beta_s = reinterpret_cast<float*>(smem + SM_SMALL);        // [64]
    float* egc_s = beta_s + 64;                                       // [128]
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(smem + SM_SMALL + 1024 - 64);
    uint64_t* bar_mma = bar_tma + 1;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(bar_tma + 2);
    int* flag_s = reinterpret_cast<int*>(bar_tma + 3);

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
        tc::bar_init_fence();
        *flag_s = 0;
    }
    // zero the A/P right-factor operand once (rows beyond a block are never
    // refreshed; they only reach accumulator rows that are not read)
    for (int i = tid; i < 32768 / 16; i += NT) reinterpret_cast<uint4*>(smem + SM_RT)[i] = make_uint4(0, 0, 0, 0);
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tmem_base_s;

    uint32_t tma_phase = 0, mma_phase = 0;
    bool failed = false;
    bool tma_pending = false;  // a tile load was issued and not yet waited for

    auto issue_tma = [&](int64_t t0) {
        tc::bar_expect_tx(bar_tma, 4u * 16384u);
        tc::tma_load_3d(smem + SM_Q, &mq, 0, h, (int)t0, bar_tma);
        tc::tma_load_3d(smem + SM_K, &mk, 0, h, (int)t0, bar_tma);
        tc::tma_load_3d(smem + SM_V, &mv, 0, h, (int)t0, bar_tma);
        tc::tma_load_3d(smem + SM_G, &mg, 0, h, (int)t0, bar_tma);
    };
    // Wait for the MMAs committed so far; all threads.
    auto mma_sync = [&]() {
        const bool ok = tc::bar_wait(bar_mma, mma_phase, kWaitIter);
        mma_phase ^= 1;
        failed = __syncthreads_or(failed || !ok);
        tc::fence_after();
    };
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
        const int cbeg = (warp >> 2) * 64;  // warpgroup 0: c in [0,64), warpgroup 1: [64,128)
        for (int cc = cbeg; cc < cbeg + 64; cc += 16) {
            uint32_t r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                r[i] = __float_as_uint(p.initial_state ? p.initial_state[sbase + (int64_t)(cc + i) * D + x] : 0.f);
            tc::tmem_st16(tm + lane_base(warp) + TM_S + cc, r);
        }
        tc::tmem_st_wait();
    }

    const uint32_t id_ap = tc::idesc_bf16(64, 32);
    const uint32_t id_n64 = tc::idesc_bf16(128, 64);
    const uint32_t id_n64_neg = tc::idesc_bf16(128, 64, true);
    const uint32_t id_n128 = tc::idesc_bf16(128, 128);
    const float scale = p.scale;
    TOut* __restrict__ o = reinterpret_cast<TOut*>(p.o);
    const __nv_bfloat16* __restrict__ beta_g = reinterpret_cast<const __nv_bfloat16*>(p.beta);

    // S hi/lo from the fp32 state in TMEM (lane x; warpgroup splits columns).
    auto s_epilogue = [&]() {
        const int cbeg = (warp >> 2) * 64;
        for (int c0 = cbeg; c0 < cbeg + 64; c0 += 32) {
            uint32_t a[16], b[16];
            tc::tmem_ld16(tm + lane_base(warp) + TM_S + c0, a);
            tc::tmem_ld16(tm + lane_base(warp) + TM_S + c0 + 16, b);
            tc::tmem_ld_wait();
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float x0 = __uint_as_float(i < 8 ? a[2 * i] : b[2 * i - 16]);
                const float x1 = __uint_as_float(i < 8 ? a[2 * i + 1] : b[2 * i - 15]);
                __nv_bfloat16 h0, l0, h1, l1;
                tc::split_bf16(x0, h0, l0);
                tc::split_bf16(x1, h1, l1);
                hi[i] = tc::pack_bf16(h0, h1);
                lo[i] = tc::pack_bf16(l0, l1);
            }
            tc::tmem_st16(tm + lane_base(warp) + TM_SH + c0 / 2, hi);
            tc::tmem_st16(tm + lane_base(warp) + TM_SL + c0 / 2, lo);
        }
        tc::tmem_st_wait();
    };
    s_epilogue();

    for (int64_t c0 = bos; c0 < eos && !failed; c0 += C) {
        const int L = (eos - c0 < (int64_t)C) ? (int)(eos - c0) : C;
        // ---- wait for this chunk's tiles ------------------------------------
        const bool ok = tc::bar_wait(bar_tma, tma_phase, kWaitIter);
        tma_phase ^= 1;
        tma_pending = false;
        failed = __syncthreads_or(!ok);
        if (failed) break;

        const __nv_bfloat16* qs = reinterpret_cast<const __nv_bfloat16*>(smem + SM_Q);
        const __nv_bfloat16* ks = reinterpret_cast<const __nv_bfloat16*>(smem + SM_K);
        const __nv_bfloat16* vs = reinterpret_cast<const __nv_bfloat16*>(smem + SM_V);
        const __nv_bfloat16* gs = reinterpret_cast<const __nv_bfloat16*>(smem + SM_G);
        float* E = reinterpret_cast<float*>(smem + SM_E);  // [64][128]

        // ---- build: decay factors and the chunk operands ------------------------
        if (tid < 128) {
            const int c = tid;
            float gp = 1.f;
            uint32_t kth[16], ktl[16];
            for (int r = 0; r < C; ++r) {
                const bool in = r < L;
                const float e = in ? __expf(__bfloat162float(gs[r * D + c])) : 1.f;
                E[r * D + c] = e;
                gp *= e;
                const float qv = in ? __bfloat162float(qs[r * D + c]) : 0.f;
                const float kv = in ? __bfloat162float(ks[r * D + c]) : 0.f;
                __nv_bfloat16 hi, lo;
                tc::split_bf16(qv * gp, hi, lo);
                *reinterpret_cast<__nv_bfloat16*>(smem + SM_QT + tc::kmaj(r, c, D)) = hi;
                *reinterpret_cast<__nv_bfloat16*>(smem + SM_QT + 16384 + tc::kmaj(r, c, D)) = lo;
                // (k e^G)^T: lane c, column pair r/2 of TMEM (flushed every 32 rows)
                __nv_bfloat16 kh, kl;
                tc::split_bf16(kv * gp, kh, kl);
                const int slot = (r & 31) >> 1;
                if ((r & 1) == 0) {
                    kth[slot] = (uint32_t)__bfloat16_as_ushort(kh);
                    ktl[slot] = (uint32_t)__bfloat16_as_ushort(kl);
                } else {
                    kth[slot] |= (uint32_t)__bfloat16_as_ushort(kh) << 16;
                    ktl[slot] |= (uint32_t)__bfloat16_as_ushort(kl) << 16;
                }
                if ((r & 31) == 31) {
                    tc::tmem_st16(tm + lane_base(warp) + TM_KTH + (r >> 5) * 16, kth);
                    tc::tmem_st16(tm + lane_base(warp) + TM_KTL + (r >> 5) * 16, ktl);
                }
            }
            egc_s[c] = gp;
            // (k e^{G_C - G})^T: suffix products, row c of a [128 c][64 j] operand
            float sfx = 1.f;
            for (int j = C - 1; j >= 0; --j) {
                const float kv = j < L ? __bfloat162float(ks[j * D + c]) : 0.f;
                __nv_bfloat16 hi, lo;
                tc::split_bf16(kv * sfx, hi, lo);
                *reinterpret_cast<__nv_bfloat16*>(smem + SM_KB + tc::kmaj(c, j, C)) = hi;
                *reinterpret_cast<__nv_bfloat16*>(smem + SM_KB + 16384 + tc::kmaj(c, j, C)) = lo;
                sfx *= E[j * D + c];
            }
        } else {
            // v^T into TMEM: lane x, bf16 pairs of consecutive tokens
            const int x = tid - 128;
            for (int j0 = 0; j0 < C; j0 += 32) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int j = j0 + 2 * i;
                    const __nv_bfloat16 a = j < L ? vs[j * D + x] : __float2bfloat16(0.f);
                    const __nv_bfloat16 b = j + 1 < L ? vs[(j + 1) * D + x] : __float2bfloat16(0.f);
                    w[i] = tc::pack_bf16(a, b);
                }
                tc::tmem_st16(tm + lane_base(warp) + TM_VT + j0 / 2, w);
            }
            if (x < C) beta_s[x] = x < L ? __bfloat162float(beta_g[(c0 + x) * H + h]) : 0.f;
        }
        tc::tmem_st_wait();
        __syncthreads();

        // ---- A and P: four row blocks, reference at each block start -------------
        for (int R = 0; R < 4; ++R) {
            const int r0 = R * 16;
            if (tid < 128) {
                const int c = tid;
                // block rows: left factors e^{sum g[r0..r]} and right factors e^{-sum g[r0..j]}
                float pre = 1.f;
                for (int j = r0; j < r0 + 16; ++j) {
                    pre *= E[j * D + c];
                    const bool in = j < L;
                    const float kv = in ? __bfloat162float(ks[j * D + c]) : 0.f;
                    const float qv = in ? __bfloat162float(qs[j * D + c]) : 0.f;
                    __nv_bfloat16 hi, lo;
                    tc::split_bf16(kv * pre, hi, lo);
                    *reinterpret_cast<__nv_bfloat16*>(smem + SM_LQ + tc::kmaj(j - r0, c, D)) = hi;
                    *reinterpret_cast<__nv_bfloat16*>(smem + SM_LQ + 8192 + tc::kmaj(j - r0, c, D)) = lo;
                    tc::split_bf16(qv * pre, hi, lo);
                    *reinterpret_cast<__nv_bfloat16*>(smem + SM_LQ + tc::kmaj(16 + j - r0, c, D)) = hi;
                    *reinterpret_cast<__nv_bfloat16*>(smem + SM_LQ + 8192 + tc::kmaj(16 + j - r0, c, D)) = lo;
                    tc::split_bf16(kv / pre, hi, lo);
                    *reinterpret_cast<__nv_bfloat16*>(smem + SM_RT + tc::kmaj(j, c, D)) = hi;
                    *reinterpret_cast<__nv_bfloat16*>(smem + SM_RT + 16384 + tc::kmaj(j, c, D)) = lo;
                }
                // earlier rows: right factor e^{sum g[j+1 .. r0-1]} <= 1
                float sfx = 1.f;
                for (int j = r0 - 1; j >= 0; --j) {
                    const float kv = j < L ? __bfloat162float(ks[j * D + c]) : 0.f;
                    __nv_bfloat16 hi, lo;
                    tc::split_bf16(kv * sfx, hi, lo);
                    *reinterpret_cast<__nv_bfloat16*>(smem + SM_RT + tc::kmaj(j, c, D)) = hi;
                    *reinterpret_cast<__nv_bfloat16*>(smem + SM_RT + 16384 + tc::kmaj(j, c, D)) = lo;
                    sfx *= E[j * D + c];
                }
            }
            publish();
            if (tid == 0) {
                const uint32_t rt = tc::smem_u32(smem + SM_RT), lq = tc::smem_u32(smem + SM_LQ);
                const uint32_t d = tm + TM_AP + 32 * R;
                int acc = 0;
                for (int ks_ = 0; ks_ < D / 16; ++ks_) {
                    const uint64_t ah = tc::sdesc(rt + ks_ * 256, 128, D * 16);
                    const uint64_t al = tc::sdesc(rt + 16384 + ks_ * 256, 128, D * 16);
                    const uint64_t bh = tc::sdesc(lq + ks_ * 256, 128, D * 16);
                    const uint64_t bl = tc::sdesc(lq + 8192 + ks_ * 256, 128, D * 16);
                    tc::mma_ss(d, ah, bh, id_ap, acc);
                    acc = 1;
                    tc::mma_ss(d, ah, bl, id_ap, 1);
                    tc::mma_ss(d, al, bh, id_ap, 1);
                }
                tc::commit(bar_mma);
            }
            mma_sync();
        }
        if (failed) break;

        // staging is consumed: prefetch the next chunk into it
        tc::fence_async_smem();
        __syncthreads();
        if (c0 + C < eos) {
            if (tid == 0) issue_tma(c0 + C);
            tma_pending = true;
        }

        // ---- A/P out of TMEM: Diag(beta) A -> fp32, P -> hi/lo operand ----------
        {
            float* Af = reinterpret_cast<float*>(smem + SM_AF);  // [64 r][64 j]
            const int quad = warp & 3;
            const int j = quad * 16 + (lane & 15);
            for (int R = (warp >> 2) * 2; R < (warp >> 2) * 2 + 2; ++R) {
                uint32_t a[16], b[16];
                tc::tmem_ld16(tm + lane_base(warp) + TM_AP + 32 * R, a);
                tc::tmem_ld16(tm + lane_base(warp) + TM_AP + 32 * R + 16, b);
                tc::tmem_ld_wait();
                if (lane < 16) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int r = 16 * R + i;
                        const float av = __uint_as_float(a[i]);
                        const float pv = __uint_as_float(b[i]);
                        Af[r * C + j] = (j < r) ? beta_s[r] * av : 0.f;
                        __nv_bfloat16 hi, lo;
                        tc::split_bf16(j <= r ? pv : 0.f, hi, lo);
                        *reinterpret_cast<__nv_bfloat16*>(smem + SM_PB + tc::kmaj(r, j, C)) = hi;
                        *reinterpret_cast<__nv_bfloat16*>(smem + SM_PB + 8192 + tc::kmaj(r, j, C)) = lo;
                    }
                }
            }
        }
        __syncthreads();

        // ---- T = (I + Diag(beta) A)^{-1} ----------------------------------------
        {
            const float* N = reinterpret_cast<const float*>(smem + SM_AF);
            float* T = reinterpret_cast<float*>(smem + SM_TF);
            float* Y = reinterpret_cast<float*>(smem + SM_TB);  // scratch [4][16][16]
            for (int i = tid; i < C * C; i += NT) T[i] = (i / C == i % C) ? 1.f : 0.f;
            __syncthreads();
            // diagonal blocks: forward substitution, four lanes per column
            {
                const int blk = tid >> 6, col = (tid & 63) >> 2, part = tid & 3;
                const int i = 16 * blk + col;
                for (int rr = 1; rr < 16; ++rr) {
                    const int r = 16 * blk + rr;
                    float acc = 0.f;
                    if (rr > col)
                        for (int jj = col + part; jj < rr; jj += 4) acc += N[r * C + 16 * blk + jj] * T[(16 * blk + jj) * C + i];
                    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                    if (part == 0 && rr > col) T[r * C + i] = -acc;
                    __syncwarp();
                }
            }
            __syncthreads();
            // off-diagonal blocks by distance d = R - J:
            //   Y = sum_{M=J}^{R-1} N_{R,M} T_{M,J};   T_{R,J} = -T_{R,R} Y
            for (int d = 1; d < 4; ++d) {
                const int nb = 4 - d;
                for (int e = tid; e < nb * 256; e += NT) {
                    const int J = e >> 8, a = (e >> 4) & 15, b = e & 15;
                    const int R = J + d;
                    float acc = 0.f;
                    for (int m = 16 * J + b; m < 16 * R; ++m) acc += N[(16 * R + a) * C + m] * T[m * C + 16 * J + b];
                    Y[e] = acc;
                }
                __syncthreads();
                for (int e = tid; e < nb * 256; e += NT) {
                    const int J = e >> 8, a = (e >> 4) & 15, b = e & 15;
                    const int R = J + d;
                    float acc = 0.f;
                    for (int m = 0; m <= a; ++m) acc += T[(16 * R + a) * C + 16 * R + m] * Y[(J << 8) + (m << 4) + b];
                    T[(16 * R + a) * C + 16 * J + b] = -acc;
                }
                __syncthreads();
            }
            // T Diag(beta) -> hi/lo B operand [64 r][64 j]
            for (int e = tid; e < C * C; e += NT) {
                const int r = e >> 6, j = e & 63;
                __nv_bfloat16 hi, lo;
                tc::split_bf16(T[e] * beta_s[j], hi, lo);
                *reinterpret_cast<__nv_bfloat16*>(smem + SM_TB + tc::kmaj(r, j, C)) = hi;
                *reinterpret_cast<__nv_bfloat16*>(smem + SM_TB + 8192 + tc::kmaj(r, j, C)) = lo;
            }
        }
        publish();

        // ---- W^T = (k e^G)^T (T Diag beta)^T ;  U~^T = v^T (T Diag beta)^T ------
        if (tid == 0) {
            const uint32_t tb = tc::smem_u32(smem + SM_TB);
            for (int ks_ = 0; ks_ < C / 16; ++ks_) {
                const uint64_t bh = tc::sdesc(tb + ks_ * 256, 128, C * 16);
                const uint64_t bl = tc::sdesc(tb + 8192 + ks_ * 256, 128, C * 16);
                tc::mma_ts(tm + TM_AO, tm + TM_KTH + ks_ * 8, bh, id_n64, ks_ > 0);
                tc::mma_ts(tm + TM_AO, tm + TM_KTH + ks_ * 8, bl, id_n64, 1);
                tc::mma_ts(tm + TM_AO, tm + TM_KTL + ks_ * 8, bh, id_n64, 1);
                tc::mma_ts(tm + TM_AU, tm + TM_VT + ks_ * 8, bh, id_n64, ks_ > 0);
                tc::mma_ts(tm + TM_AU, tm + TM_VT + ks_ * 8, bl, id_n64, 1);
            }
            tc::commit(bar_mma);
        }
        mma_sync();

        // ---- W out of TMEM into the B operand [64 r][128 c] --------------------
        {
            const int c = (warp & 3) * 32 + lane;
            const int rb = (warp >> 2) * 32;
            uint32_t a[16], b[16];
            tc::tmem_ld16(tm + lane_base(warp) + TM_AO + rb, a);
            tc::tmem_ld16(tm + lane_base(warp) + TM_AO + rb + 16, b);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float w = __uint_as_float(i < 16 ? a[i] : b[i - 16]);
                *reinterpret_cast<__nv_bfloat16*>(smem + SM_WB + tc::kmaj(rb + i, c, D)) = __float2bfloat16_rn(w);
            }
        }
        publish();

        // ---- U^T = U~^T - S^T W^T ;  O^T = S^T (q e^G)^T -------------------------
        if (tid == 0) {
            const uint32_t wb = tc::smem_u32(smem + SM_WB), qt = tc::smem_u32(smem + SM_QT);
            for (int ks_ = 0; ks_ < D / 16; ++ks_) {
                const uint32_t sh = tm + TM_SH + ks_ * 8, sl = tm + TM_SL + ks_ * 8;
                tc::mma_ts(tm + TM_AU, sh, tc::sdesc(wb + ks_ * 256, 128, D * 16), id_n64_neg, 1);
                const uint64_t qh = tc::sdesc(qt + ks_ * 256, 128, D * 16);
                const uint64_t ql = tc::sdesc(qt + 16384 + ks_ * 256, 128, D * 16);
                tc::mma_ts(tm + TM_AO, sh, qh, id_n64, ks_ > 0);
                tc::mma_ts(tm + TM_AO, sh, ql, id_n64, 1);
                tc::mma_ts(tm + TM_AO, sl, qh, id_n64, 1);
            }
            tc::commit(bar_mma);
        }
        mma_sync();

        // ---- U hi/lo into TMEM; decay the fp32 state by e^{G_C} -----------------
        {
            const int rb = (warp >> 2) * 32;
            uint32_t a[16], b[16];
            tc::tmem_ld16(tm + lane_base(warp) + TM_AU + rb, a);
            tc::tmem_ld16(tm + lane_base(warp) + TM_AU + rb + 16, b);
            tc::tmem_ld_wait();
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float x0 = __uint_as_float(i < 8 ? a[2 * i] : b[2 * i - 16]);
                const float x1 = __uint_as_float(i < 8 ? a[2 * i + 1] : b[2 * i - 15]);
                __nv_bfloat16 h0, l0, h1, l1;
                tc::split_bf16(x0, h0, l0);
                tc::split_bf16(x1, h1, l1);
                hi[i] = tc::pack_bf16(h0, h1);
                lo[i] = tc::pack_bf16(l0, l1);
            }
            tc::tmem_st16(tm + lane_base(warp) + TM_UH + rb / 2, hi);
            tc::tmem_st16(tm + lane_base(warp) + TM_UL + rb / 2, lo);
            const int cbeg = (warp >> 2) * 64;
            for (int cc = cbeg; cc < cbeg + 64; cc += 16) {
                uint32_t s[16];
                tc::tmem_ld16(tm + lane_base(warp) + TM_S + cc, s);
                tc::tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) s[i] = __float_as_uint(__uint_as_float(s[i]) * egc_s[cc + i]);
                tc::tmem_st16(tm + lane_base(warp) + TM_S + cc, s);
            }
            tc::tmem_st_wait();
        }
        publish();

        // ---- O^T += U^T P^T ;  S^T += U^T (k e^{G_C-G}) --------------------------
        if (tid == 0) {
            const uint32_t pb = tc::smem_u32(smem + SM_PB), kb = tc::smem_u32(smem + SM_KB);
            for (int ks_ = 0; ks_ < C / 16; ++ks_) {
                const uint32_t uh = tm + TM_UH + ks_ * 8, ul = tm + TM_UL + ks_ * 8;
                const uint64_t ph = tc::sdesc(pb + ks_ * 256, 128, C * 16);
                const uint64_t pl = tc::sdesc(pb + 8192 + ks_ * 256, 128, C * 16);
                tc::mma_ts(tm + TM_AO, uh, ph, id_n64, 1);
                tc::mma_ts(tm + TM_AO, uh, pl, id_n64, 1);
                tc::mma_ts(tm + TM_AO, ul, ph, id_n64, 1);
                const uint64_t kh = tc::sdesc(kb + ks_ * 256, 128, C * 16);
                const uint64_t kl = tc::sdesc(kb + 16384 + ks_ * 256, 128, C * 16);
                tc::mma_ts(tm + TM_S, uh, kh, id_n128, 1);
                tc::mma_ts(tm + TM_S, uh, kl, id_n128, 1);
                tc::mma_ts(tm + TM_S, ul, kh, id_n128, 1);
            }
            tc::commit(bar_mma);
        }
        mma_sync();

        // ---- o out; S hi/lo for the next chunk ------------------------------------
        {
            const int x = (warp & 3) * 32 + lane;
            const int rb = (warp >> 2) * 32;
            uint32_t a[16], b[16];
            tc::tmem_ld16(tm + lane_base(warp) + TM_AO + rb, a);
            tc::tmem_ld16(tm + lane_base(warp) + TM_AO + rb + 16, b);
            tc::tmem_ld_wait();
            const int64_t ob = ((c0 + rb) * H + h) * (int64_t)D + x;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (rb + i < L) {
                    const float v = scale * __uint_as_float(i < 16 ? a[i] : b[i - 16]);
                    o[ob + (int64_t)i * H * D] = from_f32<TOut>(v);
                }
            }
        }
        s_epilogue();
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
        const int cbeg = (warp >> 2) * 64;
        for (int cc = cbeg; cc < cbeg + 64; cc += 16) {
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

// [rows][H][128] bf16 tensor, box = 64 rows of one head.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int H) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM_TOTAL);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)blocks, NT, SM_TOTAL, st>>>(mq, mk, mv, mg, p);
    return cudaGetLastError();
}

}  // namespace

bool chunk_tc_supported(kda_dtype in_dt, int K, int V) { return in_dt == KDA_BF16 && K == D && V == D; }

cudaError_t chunk_tc(kda_dtype out_dt, const ChunkParams& p, cudaStream_t st) {
    if (out_dt == KDA_F32) return launch_tc<float>(p, st);
    return launch_tc<__nv_bfloat16>(p, st);
}

}  // namespace kda
