// Chunked KDA prefill on the sm_103a tensor cores (bf16 inputs, K = V = 128).
//
// Per chunk of C = 64 tokens (G = in-chunk cumulative log-decay per key
// channel; the chunk algebra of the recurrence, see kda_chunk_simt.cu):
//
//   A, P   gated in-chunk products (A strictly lower, P lower incl. diagonal)
//   T      = (I + Diag(beta) A)^{-1}
//   W      = T Diag(beta) (k e^G),      U~ = T Diag(beta) v
//   U      = U~ - W S
//   O      = scale (q e^G) S + scale P U
//   S     <- Diag(e^{G_C}) S + (k e^{G_C - G})^T U
//
// Only the last three lines touch the state; everything else is independent of
// S and is computed for all chunks at once.  The prefill is therefore two
// kernels:
//
//   chunk_local_kernel   persistent, one (chunk, head) task at a time per CTA:
//                        A, P, T, W, U~, Kbar = k e^{G_C - G}, scale (q e^G) and
//                        e^{G_C}, written to a per-(chunk, head) workspace slot
//                        straight from registers (the MMA operands already in
//                        their shared-memory layout, so the next kernel fetches
//                        them with bulk copies)
//   chunk_state_kernel   one CTA per (sequence, head): the fp32 state lives in
//                        tensor memory as S^T for the whole sequence; per chunk
//                        [U^T | O^T] = [U~^T | 0] + S^T [-W | scale q e^G]^T,
//                        then S^T <- S^T Diag(e^{G_C}) + U^T Kbar and
//                        O^T += U^T (scale P)^T.
//
// Operand precision: every operand that feeds o or the state directly is
// split x = hi + lo into two bf16 values and multiplied as hi*hi + hi*lo +
// lo*hi (about 16 significant bits); that includes W and S in the correction
// W S (long, weakly gated sequences need both split); v is exact in bf16 for
// direct inputs and split after the fused prologue.  Decay factors are running
// products of e^{g} over exactly the tokens they span, built from
// per-16-token-block prefix products (each >= e^-80 since g >= -5, so ratios
// inside a block are safe) and block totals; nothing overflows and nothing
// cancels.
//
// Sources: "ISEEKYAN/k3" README (chunked KDA forward as the compute path);
// "kimi-k3-mlx" review, "The A_log shape mismatch ..." (per-channel decay) and
// "Attention is 93 layers ..." (gate lower bound -5, 96 heads of 128).
// Every wait is bounded (a launch parameter, about a second by default).  A
// wait that gives up records KDA_ERR_TIMEOUT in the caller's status word (when
// one is given), the kernel leaves its loop, drains the copies and MMAs it has
// in flight and exits; the affected outputs are unspecified.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "kda_chunk.h"
#include "kda_chunk_plan.cuh"
#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {

std::atomic<uint32_t> g_wait_limit{0};
uint32_t wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }

namespace {

using namespace cplan;

constexpr int NT = 512;  // 16 warps: four warpgroups, each covering all 128 TMEM lanes
constexpr uint32_t kWaitIter = 1u << 26;   // default poll count of a bounded wait, and of the exit drains

__device__ __forceinline__ uint32_t lane_base(int warp) { return (uint32_t)((warp & 3) * 32) << 16; }

// ============================================================================
// Chunk-local kernel
// ============================================================================

// ---- shared memory map (bytes) ----------------------------------------------
constexpr uint32_t SM_STG = 0;             // 64 KB: q | k | v | g tiles, [64][128] bf16, 128B-swizzled halves
constexpr uint32_t SM_OPB = 65536;         // 48 KB, A/P phase: Rt hi|lo (B op [96 j][128 c]); then
constexpr uint32_t SM_TB = SM_OPB;         //   (T Diag beta) hi|lo, B op [64 r][64 j] K-major
constexpr uint32_t SM_PRE = 114688;        // fp32 [64][PRE_LD] in-block prefix products of e^g
constexpr int PRE_LD = 132;
constexpr int MAT_LD = 68;
constexpr uint32_t SM_AF = SM_PRE + 64 * PRE_LD * 4;   // Diag(beta) A, fp32 [64][MAT_LD]
constexpr uint32_t SM_TF = SM_AF + 64 * MAT_LD * 4;    // T, fp32 [64][MAT_LD]
constexpr uint32_t SM_SMALL = SM_TF + 64 * MAT_LD * 4;  // 183296
// A/P operands of both row blocks R: L rows 64 R + i (i < 32: k rows, else q rows of
// block R) in TMEM, Rt rows j (block 0, j < 32) and 32 + j (block 1, j < 64) in SM_OPB
constexpr uint32_t RT_LO = 96 * D * 2;
constexpr uint32_t SM_TOT = SM_SMALL;            // fp32 [4][128] block totals of e^g
constexpr uint32_t SM_ITOT = SM_SMALL + 2048;    // fp32 [2][128] inverses of the totals of blocks 0, 2
constexpr uint32_t SM_BETA = SM_SMALL + 3072;    // fp32 [64]
constexpr uint32_t SM_BAR = SM_BETA + 256;       // barriers (tiles, mma), tmem base, exit drain, testing, g tile
constexpr uint32_t SM_LOCAL_TOTAL = SM_BAR + 64;
// with the input prologue (raw q, k, v and gate input in the staging tiles):
constexpr uint32_t SM_RED = SM_SMALL + 3456;     // fp32 [2][64][4] partial sums of squares of q, k rows
constexpr uint32_t SM_HALO = SM_RED + 2048;      // bf16 [3][2][3][64] the 3 raw rows before the chunk (q, k, v)
constexpr uint32_t SM_CONV = SM_HALO + 2304;     // fp32 [3][128][4] this head's conv weights (q, k, v)
constexpr uint32_t SM_DTB = SM_CONV + 6144;      // fp32 [128] this head's dt_bias
constexpr uint32_t SM_ALOG = SM_DTB + 512;       // fp32 [128] A_log
constexpr uint32_t SM_LOCAL_TOTAL_FUSED = SM_ALOG + 512;
constexpr uint32_t PRO_TX = 6 * 384 + 6144 + 512 + 512;   // prologue bytes per task load
static_assert(SM_LOCAL_TOTAL + 1024 <= 232448, "shared memory");
static_assert(SM_RED >= SM_LOCAL_TOTAL && SM_HALO % 128 == 0, "prologue regions");
static_assert(SM_LOCAL_TOTAL_FUSED + 1024 <= 232448, "shared memory with the prologue");

// ---- tensor memory map (columns) ----------------------------------------------
constexpr uint32_t TL_AP = 0;      // [L_0; L_1] [Rt_0 | Rt_1]^T accumulator, M = 128, N = 96
constexpr uint32_t TL_KTH = 96;    // (k e^G)^T hi (bf16 pairs) [128 c][32]
constexpr uint32_t TL_KTL = 128;   // (k e^G)^T lo
constexpr uint32_t TL_VT = 160;    // v^T (bf16 pairs) [128 v][32]
constexpr uint32_t TL_AW = 192;    // W^T accumulator fp32 [128 c][64 r]
constexpr uint32_t TL_AU = 256;    // U~^T accumulator fp32 [128 v][64 r]
constexpr uint32_t TL_VTL = 320;   // v^T lo (bf16 pairs), with the prologue (v is then not bf16-exact)
constexpr uint32_t TL_LH = 352;    // A/P A operand [L_0; L_1] hi (bf16 pairs) [128 i][64]
constexpr uint32_t TL_LL = 416;    // its lo
constexpr uint32_t TL_COLS = 512;
// Thread that issues the first task's tile loads and posts each next task's byte
// count; it and the next 63 fetch beta.  (The next task's tile loads are spread over
// lane 0 of the warps of scheduler partitions 2 and 3.)
constexpr int kIssueTid = 320;

// Input prologue ("kimi-k3-mlx" review: short convolution of kernel size 4 on
// q, k, v; per-channel forget gate with gate_lower_bound; A_log of K entries
// shared by all heads): q, k = l2norm(act(conv4(raw))), v = act(conv4(raw)),
// g = max(lower_bound, -exp(A_log) softplus(gate_x + dt_bias)).
struct Prologue {
    const float* conv_q;   // [H * 128][4]
    const float* conv_k;
    const float* conv_v;
    const float* A_log;    // [128]
    const float* dt_bias;  // [H * 128]
    float lower_bound;
    float l2_eps;
};

// Base-2 exponential and logarithm on the special-function unit (PTX ex2.approx,
// lg2.approx).  The gate uses them: only its absolute error matters (it enters
// as e^g), and log2(1 + t), t in (0, 1], is within ~1e-7 absolute.
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// FUSED: the staging tiles hold the raw inputs (q_raw, k_raw, v_raw, gate_x);
// the prologue runs on them first and leaves q, k as bf16 hi (in the q, k tiles)
// plus lo (in the v, g tiles), v as hi/lo in TMEM and g folded into pass 1.
// SILU: the convolution is followed by SiLU (a separate instance, so that the
// other never evaluates it).  AT: also write each chunk's A and T to pl.at_out
// (for the backward; an instance of its own so that the prefill carries no trace
// of it).
template <bool FUSED, bool SILU = false, bool AT = false>
__global__ void __launch_bounds__(NT, 1)
chunk_local_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mg,
                   const __grid_constant__ CUtensorMap hq, const __grid_constant__ CUtensorMap hk,
                   const __grid_constant__ CUtensorMap hv, const void* __restrict__ beta_ptr, const float scale,
                   const Plan pl, const Prologue pro) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte-swizzled TMA tiles need a 1024-byte aligned base
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* beta_s = reinterpret_cast<float*>(smem + SM_BETA);   // [64]
    float* tot_s = reinterpret_cast<float*>(smem + SM_TOT);     // [4][128]
    float* itot_s = reinterpret_cast<float*>(smem + SM_ITOT);   // [2][128]
    float* pre_s = reinterpret_cast<float*>(smem + SM_PRE);     // [64][PRE_LD]
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(smem + SM_BAR);
    uint64_t* bar_mma = bar_tma + 1;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(bar_tma + 2);
    uint64_t* bar_fin = bar_tma + 3;   // every MMA issued has completed (exit drain)
    uint64_t* bar_never = bar_tma + 4; // testing: nothing arrives on it
    uint64_t* bar_g = bar_tma + 5;     // the g tile, loaded one task ahead of q, k, v (without the prologue)
    const int H = pl.H;
    const __nv_bfloat16* __restrict__ beta_g = reinterpret_cast<const __nv_bfloat16*>(beta_ptr);

    if (warp == 0) tc::tmem_alloc(tmem_base_s, TL_COLS);
    if (tid == 0) {
        tc::bar_init(bar_tma, 1);
        tc::bar_init(bar_mma, 1);
        tc::bar_init(bar_fin, 1);
        tc::bar_init(bar_never, 1);
        tc::bar_init(bar_g, 1);
        tc::bar_init_fence();
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tmem_base_s;

    uint32_t tma_phase = 0, mma_phase = 0, g_phase = 0;
    bool failed = false;
    bool tma_pending = false, g_pending = false;

    // Without the prologue the g tile has a barrier of its own: its only reader is
    // the prefix pass, which for task n + 1 runs during task n's T inverse, so the
    // tile of task n + 1 is requested when task n starts and has landed by the
    // time that pass needs it.  (With the prologue the g tile later holds the lo
    // half of k, so all four tiles travel together.)
    constexpr uint32_t kTileTx = FUSED ? 4u * 16384u + PRO_TX : 3u * 16384u;
    auto issue_g = [&](const Chunk& ch) {
        tc::bar_expect_tx(bar_g, 16384u);
#pragma unroll
        for (int half = 0; half < 2; ++half)
            tc::tma_load_3d(smem + SM_STG + 3 * 16384 + half * 8192, &mg, half * 64, ch.h, (int)ch.c0, bar_g);
    };
    auto issue_tma = [&](const Chunk& ch) {
        tc::bar_expect_tx(bar_tma, kTileTx);
        const CUtensorMap* maps[4] = {&mq, &mk, &mv, &mg};
#pragma unroll
        for (int t = 0; t < (FUSED ? 4 : 3); ++t)
#pragma unroll
            for (int half = 0; half < 2; ++half)
                tc::tma_load_3d(smem + SM_STG + t * 16384 + half * 8192, maps[t], half * 64, ch.h, (int)ch.c0, bar_tma);
        if constexpr (!FUSED) issue_g(ch);
        if constexpr (FUSED) {
            // the 3 raw rows before the chunk (row -3 and up; rows before the tensor
            // arrive as zeros, rows of another sequence are masked when used)
            const CUtensorMap* hmaps[3] = {&hq, &hk, &hv};
#pragma unroll
            for (int t = 0; t < 3; ++t)
#pragma unroll
                for (int half = 0; half < 2; ++half)
                    tc::tma_load_3d(smem + SM_HALO + t * 768 + half * 384, hmaps[t], half * 64, ch.h, (int)ch.c0 - 3,
                                    bar_tma);
            tc::bulk_load(smem + SM_CONV, pro.conv_q + (int64_t)ch.h * D * 4, 2048, bar_tma);
            tc::bulk_load(smem + SM_CONV + 2048, pro.conv_k + (int64_t)ch.h * D * 4, 2048, bar_tma);
            tc::bulk_load(smem + SM_CONV + 4096, pro.conv_v + (int64_t)ch.h * D * 4, 2048, bar_tma);
            tc::bulk_load(smem + SM_DTB, pro.dt_bias + (int64_t)ch.h * D, 512, bar_tma);
            tc::bulk_load(smem + SM_ALOG, pro.A_log, 512, bar_tma);
        }
    };
    // The same, spread over lane 0 of the warps of scheduler partitions 2 and 3 (one
    // tile each, the prologue's extra loads round-robin), for a task whose byte count
    // bar_tma already expects (the g tile only with the prologue).
    auto issue_tma_spread = [&](const Chunk& ch) {
        if ((warp & 2) == 0 || lane != 0) return;
        const int i = ((warp >> 2) << 1) | (warp & 1);
        if (!FUSED && i >= 6) return;
        const CUtensorMap* mp = i < 2 ? &mq : (i < 4 ? &mk : (i < 6 ? &mv : &mg));
        tc::tma_load_3d(smem + SM_STG + (i >> 1) * 16384 + (i & 1) * 8192, mp, (i & 1) * 64, ch.h, (int)ch.c0,
                        bar_tma);
        if constexpr (FUSED) {
            if (i < 6) {
                const int t = i >> 1, half = i & 1;
                tc::tma_load_3d(smem + SM_HALO + t * 768 + half * 384, t == 0 ? &hq : (t == 1 ? &hk : &hv),
                                half * 64, ch.h, (int)ch.c0 - 3, bar_tma);
            }
            if (i < 3) {
                const float* w = i == 0 ? pro.conv_q : (i == 1 ? pro.conv_k : pro.conv_v);
                tc::bulk_load(smem + SM_CONV + i * 2048, w + (int64_t)ch.h * D * 4, 2048, bar_tma);
            } else if (i == 3) {
                tc::bulk_load(smem + SM_DTB, pro.dt_bias + (int64_t)ch.h * D, 512, bar_tma);
            } else if (i == 4) {
                tc::bulk_load(smem + SM_ALOG, pro.A_log, 512, bar_tma);
            }
        }
    };
    // One warp polls the barrier; the others park at the CTA barrier.  A wait
    // that gives up leaves its phase pending (the exit drains it) and sets failed
    // in every thread.
    bool inject = pl.inject == 1;
    auto wait_one = [&](uint64_t* bar, uint32_t& phase) {
        bool ok = true;
        if (warp == 0) ok = inject ? tc::bar_wait(bar_never, 0, pl.wait_iter) : tc::bar_wait(bar, phase, pl.wait_iter);
        inject = false;
        const bool gave_up = __syncthreads_or(!ok) != 0;
        if (!gave_up) phase ^= 1;
        failed = failed || gave_up;
        tc::fence_after();
        return !gave_up;
    };
    auto mma_sync = [&]() { wait_one(bar_mma, mma_phase); };
    // Make generic-proxy smem writes and TMEM stores visible to the MMA issuer.
    auto publish = [&]() {
        tc::fence_async_smem();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    };

    const uint32_t id_n64 = tc::idesc_bf16(128, 64);

    // beta of a task, fetched as raw bf16 bits into registers of threads
    // kIssueTid .. + 63 when its tiles are requested (a predicated load into the
    // zeroed register: nothing waits for it until the next task stores it)
    const int bt = tid - kIssueTid;
    auto fetch_beta = [&](const Chunk& ch) {
        unsigned short b = 0;
        const bool have = bt >= 0 && bt < C && ch.c0 + bt < ch.eos;
        const __nv_bfloat16* src = beta_g + (have ? (ch.c0 + bt) * H + ch.h : 0);
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p ld.global.nc.u16 %0, [%1];\n\t}"
                     : "+h"(b) : "l"(src), "r"((uint32_t)have));
        return b;
    };

    // (1) for one (channel c, 16-token block J) of a task with Ln tokens: the in-block
    // prefix products of e^g (1 past the sequence end) and the block total
    auto prefix_item = [&](int c, int J, int Ln) {
        const uint8_t* gs = smem + SM_STG + 49152;
        auto g_at = [&](int r) {
            return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(gs + tc::swz128(r, c)));
        };
        float eg[16];
        if constexpr (FUSED) {
            // g = max(lower_bound, -exp(A_log) softplus(gate_x + dt_bias)), in base 2:
            //   g log2(e) = max(lower_bound log2(e), -exp(A_log) sp2(y)),  y = (gate_x + dt_bias) log2(e),
            //   sp2(y) = log2(1 + 2^y) = max(y, 0) + log2(1 + 2^-|y|)
            // (three special-function operations per element, no branch)
            const float ea = __expf(reinterpret_cast<const float*>(smem + SM_ALOG)[c]);
            const float db = reinterpret_cast<const float*>(smem + SM_DTB)[c];
            const float lb2 = pro.lower_bound * kLog2e;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float y = (g_at(16 * J + u) + db) * kLog2e;
                const float sp2 = fmaxf(y, 0.f) + lg2_approx(1.f + ex2_approx(-fabsf(y)));
                eg[u] = 16 * J + u < Ln ? ex2_approx(fmaxf(lb2, -ea * sp2)) : 1.f;
            }
        } else {
#pragma unroll
            for (int u = 0; u < 16; ++u) eg[u] = 16 * J + u < Ln ? __expf(g_at(16 * J + u)) : 1.f;
        }
        float run = 1.f;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            run *= eg[u];
            pre_s[(16 * J + u) * PRE_LD + c] = run;
        }
        tot_s[J * 128 + c] = run;
        if ((J & 1) == 0) itot_s[(J >> 1) * 128 + c] = __fdividef(1.f, run);
    };
    // (2a) the A/P A operand L in TMEM for one item (16 channels: [16 item, 16 item
    // + 16) of every stack row of this warp's lane quadrant) of a task with Lr
    // tokens: lane quadrant q4 holds the k rows (even q4) or q rows (odd q4) of row
    // block R = q4 / 2; e^{G_r - G_mid} = pre_r / tot_{2R} before the block centre,
    // pre_r after it
    auto build_L = [&](int item, int Lr) {
        const int q4 = warp & 3, R = q4 >> 1;
        const int r = 32 * R + lane;
        const bool first = (lane & 16) == 0;  // r in the first 16-token block of R
        const uint8_t* src = smem + SM_STG + ((q4 & 1) != 0 ? 0 : 16384);
        uint32_t lh[8], ll[8];
#pragma unroll
        for (int g8 = 0; g8 < 2; ++g8) {
            const int c = 16 * item + 8 * g8;
            float x[8], pr[8], it[8];
            if (r < Lr) {
                tc::unpack8(*reinterpret_cast<const uint4*>(src + tc::swz128(r, c)), x);
                if constexpr (FUSED) {
                    float y[8];
                    tc::unpack8(*reinterpret_cast<const uint4*>(src + 32768 + tc::swz128(r, c)), y);
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[i] += y[i];
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] = 0.f;
            }
            const float4 p0 = *reinterpret_cast<const float4*>(pre_s + r * PRE_LD + c);
            const float4 p1 = *reinterpret_cast<const float4*>(pre_s + r * PRE_LD + c + 4);
            pr[0] = p0.x; pr[1] = p0.y; pr[2] = p0.z; pr[3] = p0.w; pr[4] = p1.x; pr[5] = p1.y; pr[6] = p1.z; pr[7] = p1.w;
            const float4 a = *reinterpret_cast<const float4*>(itot_s + R * 128 + c);
            const float4 b = *reinterpret_cast<const float4*>(itot_s + R * 128 + c + 4);
            it[0] = a.x; it[1] = a.y; it[2] = a.z; it[3] = a.w; it[4] = b.x; it[5] = b.y; it[6] = b.z; it[7] = b.w;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                tc::split2(x[2 * u] * (first ? pr[2 * u] * it[2 * u] : pr[2 * u]),
                           x[2 * u + 1] * (first ? pr[2 * u + 1] * it[2 * u + 1] : pr[2 * u + 1]),
                           lh[4 * g8 + u], ll[4 * g8 + u]);
        }
        tc::tmem_st8(tm + lane_base(warp) + TL_LH + 8 * item, lh);
        tc::tmem_st8(tm + lane_base(warp) + TL_LL + 8 * item, ll);
    };
    bool pre_done = false;  // the current task's prefix pass (and, without the prologue, its L operand) has run

    int64_t task = blockIdx.x;
    Chunk cur = decode_task(pl, task);
    unsigned short beta_r = 0;
    if (cur.valid) {
        if (tid == kIssueTid) issue_tma(cur);
        tma_pending = true;
        g_pending = !FUSED;
        beta_r = fetch_beta(cur);
    }

    while (cur.valid) {
        const int h = cur.h;
        const int64_t c0 = cur.c0;
        const int L = (cur.eos - c0 < (int64_t)C) ? (int)(cur.eos - c0) : C;
        uint8_t* slot = pl.slots + ((int64_t)cur.gc * H + h) * (int64_t)SLOT_BYTES;
        const int64_t next_task = task + gridDim.x;
        const Chunk nxt = decode_task(pl, next_task);

        if (!pre_done) {
            if (wait_one(bar_tma, tma_phase)) tma_pending = false;
            if (failed) break;
            if constexpr (!FUSED) {
                if (wait_one(bar_g, g_phase)) g_pending = false;
                if (failed) break;
            }
        } else if (!FUSED && nxt.valid) {
            // (the last task's T-inverse window has read this task's g tile)
            if (tid == kIssueTid) issue_g(nxt);
            g_pending = true;
        }
        // the next task's byte count, posted long before its loads are issued (by
        // several threads, so none of them may complete the phase early)
        if (tid == kIssueTid && nxt.valid) tc::bar_expect_tx(bar_tma, kTileTx);

        uint8_t* qs = smem + SM_STG;
        uint8_t* ks = smem + SM_STG + 16384;
        uint8_t* vs = smem + SM_STG + 32768;
        uint8_t* gs = smem + SM_STG + 49152;
        auto ld_bf = [&](const uint8_t* t, int r, int c) {
            return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(t + tc::swz128(r, c)));
        };
        // q (is_q) or k: 8 consecutive channels [c, c+8) of row r as floats (0 for
        // rows >= L); after the prologue the value is its hi + lo
        auto ld8 = [&](bool is_q, int r, int c, float* x) {
            if (r < L) {
                tc::unpack8(*reinterpret_cast<const uint4*>((is_q ? qs : ks) + tc::swz128(r, c)), x);
                if constexpr (FUSED) {
                    float y[8];
                    tc::unpack8(*reinterpret_cast<const uint4*>((is_q ? vs : gs) + tc::swz128(r, c)), y);
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[i] += y[i];
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] = 0.f;
            }
        };
        // one channel of k, of q
        auto ld_k = [&](int r, int c) {
            float x = ld_bf(ks, r, c);
            if constexpr (FUSED) x += ld_bf(gs, r, c);
            return x;
        };
        auto ld_q = [&](int r, int c) {
            float x = ld_bf(qs, r, c);
            if constexpr (FUSED) x += ld_bf(vs, r, c);
            return x;
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

        // raw input of tensor t (0 q, 1 k, 2 v) at chunk row sr >= -3, channel c;
        // zero before the start of the sequence
        // (branch-free: the address is selected, rows of another sequence read as zero)
        auto raw_addr = [&](int t, int sr, int c) -> const uint8_t* {
            const uint8_t* halo = smem + SM_HALO + t * 768 + (c >> 6) * 384 + (sr + 3) * 128 + (c & 63) * 2;
            const uint8_t* stg = smem + SM_STG + t * 16384 + tc::swz128(sr, c);
            return sr < 0 ? halo : stg;
        };
        auto raw1 = [&](int t, int sr, int c) -> float {
            const float x = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(raw_addr(t, sr, c)));
            return c0 + sr < cur.bos ? 0.f : x;
        };
        auto raw8 = [&](int t, int sr, int c, float* x) {
            uint4 v = *reinterpret_cast<const uint4*>(raw_addr(t, sr, c));
            if (c0 + sr < cur.bos) v = make_uint4(0u, 0u, 0u, 0u);
            tc::unpack8(v, x);
        };
        auto act = [&](float y) {
            if constexpr (SILU) return __fdividef(y, 1.f + __expf(-y));
            else return y;
        };

        // ---- (1) in-block prefix products of e^g, block totals (for the first task;
        //      every later task's ran while the previous task inverted T) ----------
        if (!pre_done) prefix_item(tid & 127, tid >> 7, L);
        if constexpr (FUSED) {
            // v = act(conv4(v_raw)): this thread's value column, 16 tokens, as hi|lo
            // pairs into TMEM (lane = value column)
            const int c = (warp & 3) * 32 + lane;
            const int jb = (warp >> 2) * 16;
            const float4 w = *reinterpret_cast<const float4*>(smem + SM_CONV + 4096 + c * 16);
            float xr[19];
#pragma unroll
            for (int m = 0; m < 19; ++m) xr[m] = raw1(2, jb - 3 + m, c);
            uint32_t vh[8], vl[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float y[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int m = 2 * i + e;
                    const float acc = act(w.x * xr[m] + w.y * xr[m + 1] + w.z * xr[m + 2] + w.w * xr[m + 3]);
                    y[e] = jb + m < L ? acc : 0.f;
                }
                tc::split2(y[0], y[1], vh[i], vl[i]);
            }
            tc::tmem_st8(tm + lane_base(warp) + TL_VT + jb / 2, vh);
            tc::tmem_st8(tm + lane_base(warp) + TL_VTL + jb / 2, vl);
            tc::tmem_st_wait();
        }
        if (bt >= 0 && bt < C) beta_s[bt] = __uint_as_float((uint32_t)beta_r << 16);
        if (!FUSED && !pre_done) tc::fence_async_smem();   // (the g tile is read: the next one may land)
        __syncthreads();
        if (!FUSED && !pre_done && nxt.valid) {
            if (tid == kIssueTid) issue_g(nxt);
            g_pending = true;
        }

        if constexpr (FUSED) {
            // q, k = l2norm(act(conv4(raw))) over the 128 channels of each row, written
            // back as bf16 hi (q, k tiles) + lo (v, g tiles, consumed above)
            const int cgp = (tid >> 3) & 15;
            float* red = reinterpret_cast<float*>(smem + SM_RED);  // [2][64][4]
            float y[2][2][8];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const float* wt = reinterpret_cast<const float*>(smem + SM_CONV + t * 2048) + 8 * cgp * 4;
                float4 w[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) w[u] = *reinterpret_cast<const float4*>(wt + 4 * u);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int item = tid + NT * kk;
                    const int r = ((item >> 7) << 3) | (item & 7);
                    float acc[8], xv[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
                    raw8(t, r - 3, 8 * cgp, xv);
#pragma unroll
                    for (int u = 0; u < 8; ++u) acc[u] += w[u].x * xv[u];
                    raw8(t, r - 2, 8 * cgp, xv);
#pragma unroll
                    for (int u = 0; u < 8; ++u) acc[u] += w[u].y * xv[u];
                    raw8(t, r - 1, 8 * cgp, xv);
#pragma unroll
                    for (int u = 0; u < 8; ++u) acc[u] += w[u].z * xv[u];
                    raw8(t, r, 8 * cgp, xv);
#pragma unroll
                    for (int u = 0; u < 8; ++u) acc[u] += w[u].w * xv[u];
                    float ss = 0.f;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        acc[u] = r < L ? act(acc[u]) : 0.f;
                        ss += acc[u] * acc[u];
                        y[t][kk][u] = acc[u];
                    }
                    ss += __shfl_xor_sync(0xffffffffu, ss, 8);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 16);
                    if (lane < 8) red[(t * 64 + r) * 4 + (warp & 3)] = ss;
                }
            }
            __syncthreads();
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int item = tid + NT * kk;
                    const int r = ((item >> 7) << 3) | (item & 7);
                    const float4 pss = *reinterpret_cast<const float4*>(red + (t * 64 + r) * 4);
                    const float inv = rsqrtf(pss.x + pss.y + pss.z + pss.w + pro.l2_eps);
#pragma unroll
                    for (int u = 0; u < 8; ++u) y[t][kk][u] *= inv;
                    uint4 hi, lo;
                    tc::split8(y[t][kk], hi, lo);
                    *reinterpret_cast<uint4*>((t == 0 ? qs : ks) + tc::swz128(r, 8 * cgp)) = hi;
                    *reinterpret_cast<uint4*>((t == 0 ? vs : gs) + tc::swz128(r, 8 * cgp)) = lo;
                }
            __syncthreads();
        }

        // Every build loop below gives a thread the same 8 channels [8 cg, 8 cg + 8).
        const int cg = (tid >> 3) & 15;

        // ---- (2) A and P: two 32-token row blocks, reference at the block centre --
        // Both blocks' operands are stacked (L rows 64 R + i, Rt rows of block 1 after
        // those of block 0) and multiplied in one M = 128, N = 96 round; the two
        // off-diagonal products of the stack are not used.
        // (Without the prologue, L was built while the last task's W/U MMAs ran.)
        if (FUSED || !pre_done) {
#pragma unroll 1
            for (int it = 0; it < 2; ++it) build_L(2 * (warp >> 2) + it, L);
        }
        // the last task's -W bulk stores have read the operand region before Rt overwrites it
        if (tid == kIssueTid) tc::bulk_wait_read();
        __syncthreads();
#pragma unroll
        for (int R = 0; R < 2; ++R) {
            const int nrows = 32 * (R + 1);  // columns j of this block's products
            // Rt_R (B operand rows 32 R + j): e^{G_mid - G_j} k_j =
            //   1 / pre_j after the centre, tot_J / pre_j * prod_{J < J2 <= 2R} tot_J2 before it
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int item = tid + NT * kk;
                if (item >= nrows * 16) break;
                const int j = ((item >> 7) << 3) | (item & 7);
                const int J = j >> 4;
                float x[8], pr[8], m[8], t[8];
                ld8(false, j, 8 * cg, x);
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
                *reinterpret_cast<uint4*>(smem + SM_OPB + tc::kmaj(32 * R + j, 8 * cg, D)) = hi;
                *reinterpret_cast<uint4*>(smem + SM_OPB + RT_LO + tc::kmaj(32 * R + j, 8 * cg, D)) = lo;
            }
        }
        tc::tmem_st_wait();
        publish();
        if (warp == 0) {
            const uint32_t rb = tc::smem_u32(smem + SM_OPB);
            const uint64_t bh = tc::sdesc(rb, 128, D * 16), bl = tc::sdesc(rb + RT_LO, 128, D * 16);
            const uint32_t id = tc::idesc_bf16(128, 96);
#pragma unroll
            for (int ks_ = 0; ks_ < D / 16; ++ks_) {
                const uint32_t o = ks_ * 256;
                tc::mma_ts_w(tm + TL_AP, tm + TL_LH + ks_ * 8, tc::dadv(bh, o), id, ks_ > 0);
                tc::mma_ts_w(tm + TL_AP, tm + TL_LH + ks_ * 8, tc::dadv(bl, o), id, 1);
                tc::mma_ts_w(tm + TL_AP, tm + TL_LL + ks_ * 8, tc::dadv(bh, o), id, 1);
            }
            tc::commit_w(bar_mma);
        }
        // ---- (3) per channel and 16-token block, while the A/P MMAs run: (k e^G)^T
        //      and v^T into TMEM (lane = channel / value column); the slot's
        //      Qs = scale q e^G (the second half of the merged image) and
        //      Kbar = k e^{G_C - G} (K-major), hi|lo, and e^{G_C}, stored straight
        //      from registers: a thread's 8 consecutive tokens of one channel are one
        //      16-byte unit of both layouts, and a warp's 32 channels 512 (Qs) or four
        //      runs of 128 (Kbar) contiguous bytes
        {
            const int c = (warp & 3) * 32 + lane;
            const int jblk = warp >> 2, jb = 16 * jblk;  // warpgroup w covers tokens [16 w, 16 w + 16)
            const float t0v = tot_s[c], t1v = tot_s[128 + c], t2v = tot_s[256 + c], t3v = tot_s[384 + c];
            // products of the block totals before this block (pf) and from it on (sf)
            const float pf = jblk == 0 ? 1.f : (jblk == 1 ? t0v : (jblk == 2 ? t0v * t1v : t0v * t1v * t2v));
            const float sf = jblk == 0 ? t0v * t1v * t2v * t3v
                                       : (jblk == 1 ? t1v * t2v * t3v : (jblk == 2 ? t2v * t3v : t3v));
            // two halves of 8 tokens, each stored as soon as it is done
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
                uint32_t kh[4], kl[4], vv[4];
                float fq[8], fk[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int j = jb + 8 * h8 + 2 * i;
                    const float p0 = pre_s[j * PRE_LD + c], p1 = pre_s[(j + 1) * PRE_LD + c];
                    const float k0 = j < L ? ld_k(j, c) : 0.f;
                    const float k1 = j + 1 < L ? ld_k(j + 1, c) : 0.f;
                    const float q0 = j < L ? ld_q(j, c) : 0.f;
                    const float q1 = j + 1 < L ? ld_q(j + 1, c) : 0.f;
                    const float e0 = pf * p0, e1 = pf * p1;   // e^{G_j}, e^{G_{j+1}}
                    tc::split2(k0 * e0, k1 * e1, kh[i], kl[i]);
                    fq[2 * i] = q0 * (scale * e0);
                    fq[2 * i + 1] = q1 * (scale * e1);
                    fk[2 * i] = k0 * __fdividef(sf, p0);
                    fk[2 * i + 1] = k1 * __fdividef(sf, p1);
                    if constexpr (!FUSED) {
                        const __nv_bfloat16 z = __float2bfloat16(0.f);
                        const __nv_bfloat16 v0 = j < L ? *reinterpret_cast<const __nv_bfloat16*>(vs + tc::swz128(j, c)) : z;
                        const __nv_bfloat16 v1 = j + 1 < L ? *reinterpret_cast<const __nv_bfloat16*>(vs + tc::swz128(j + 1, c)) : z;
                        vv[i] = tc::pack_bf16(v0, v1);
                    }
                }
                uint4 hi, lo;
                tc::split8(fq, hi, lo);
                *reinterpret_cast<uint4*>(slot + SLOT_WQH + tc::mnmaj_ng(C + jb + 8 * h8, c, D)) = hi;
                *reinterpret_cast<uint4*>(slot + SLOT_WQL + tc::mnmaj_ng(C + jb + 8 * h8, c, D)) = lo;
                tc::split8(fk, hi, lo);
                *reinterpret_cast<uint4*>(slot + SLOT_KH + tc::kmaj(c, jb + 8 * h8, C)) = hi;
                *reinterpret_cast<uint4*>(slot + SLOT_KL + tc::kmaj(c, jb + 8 * h8, C)) = lo;
                tc::tmem_st4(tm + lane_base(warp) + TL_KTH + jb / 2 + 4 * h8, kh);
                tc::tmem_st4(tm + lane_base(warp) + TL_KTL + jb / 2 + 4 * h8, kl);
                if constexpr (!FUSED) tc::tmem_st4(tm + lane_base(warp) + TL_VT + jb / 2 + 4 * h8, vv);
            }
            if (tid < 128) reinterpret_cast<float*>(slot + SLOT_EGC)[c] = t0v * t1v * t2v * t3v;
        }
        tc::tmem_st_wait();
        // (the staging tiles are consumed: the next task's loads may overwrite them)
        tc::fence_async_smem();

        mma_sync();
        if (failed) break;
        if (nxt.valid) {
            issue_tma_spread(nxt);
            beta_r = fetch_beta(nxt);
            tma_pending = true;
        }

        // ---- (5) A/P out of TMEM: Diag(beta) A -> fp32, P -> hi/lo operand ---------
        // lane quadrant q4 holds stack rows 32 q4 + lane: block R = q4 / 2, k rows for
        // even q4, q rows for odd; block 0 uses columns 0..31, block 1 columns 32..95
        {
            float* Af = reinterpret_cast<float*>(smem + SM_AF);  // [64 r][MAT_LD]
            const int q4 = warp & 3, wg = warp >> 2;
            const int R = q4 >> 1;
            const bool is_q = (q4 & 1) != 0;
            const int r = 32 * R + lane;
            const int j0 = R == 0 ? 8 * wg : 16 * wg;
            uint32_t a[16];
            if (R == 0) {
                tc::tmem_ld8(tm + lane_base(warp) + TL_AP + j0, a);
            } else {
                tc::tmem_ld16(tm + lane_base(warp) + TL_AP + 32 + j0, a);
            }
            tc::tmem_ld_wait();
            const float br = beta_s[r];
            // (for the backward: A itself, without beta)
            float* ao = AT ? pl.at_out + ((int64_t)cur.gc * H + h) * (2 * C * C) + r * C : nullptr;
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {
                if (R == 0 && g8 == 1) break;
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = j0 + 8 * g8 + u;
                    const float xv = __uint_as_float(a[8 * g8 + u]);
                    v[u] = is_q ? (j <= r ? scale * xv : 0.f) : (j < r ? br * xv : 0.f);
                }
                if (AT && !is_q) {
                    float w[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) w[u] = j0 + 8 * g8 + u < r ? __uint_as_float(a[8 * g8 + u]) : 0.f;
                    *reinterpret_cast<float4*>(ao + j0 + 8 * g8) = make_float4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<float4*>(ao + j0 + 8 * g8 + 4) = make_float4(w[4], w[5], w[6], w[7]);
                    if (R == 0) {
                        *reinterpret_cast<float4*>(ao + 32 + j0) = make_float4(0.f, 0.f, 0.f, 0.f);
                        *reinterpret_cast<float4*>(ao + 32 + j0 + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                if (is_q) {
                    uint4 hi, lo;
                    tc::split8(v, hi, lo);
                    *reinterpret_cast<uint4*>(slot + SLOT_P + tc::kmaj(r, j0 + 8 * g8, C)) = hi;
                    *reinterpret_cast<uint4*>(slot + SLOT_P + 8192 + tc::kmaj(r, j0 + 8 * g8, C)) = lo;
                } else {
                    *reinterpret_cast<float4*>(Af + r * MAT_LD + j0 + 8 * g8) = make_float4(v[0], v[1], v[2], v[3]);
                    *reinterpret_cast<float4*>(Af + r * MAT_LD + j0 + 8 * g8 + 4) = make_float4(v[4], v[5], v[6], v[7]);
                }
            }
            // P rows of block 0 are zero in columns 32..63 (the P operand spans all 64)
            if (R == 0 && is_q) {
                *reinterpret_cast<uint4*>(slot + SLOT_P + tc::kmaj(r, 32 + j0, C)) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(slot + SLOT_P + 8192 + tc::kmaj(r, 32 + j0, C)) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        __syncthreads();

        // ---- (6) T = (I + Diag(beta) A)^{-1} on warps 0..3 (named barrier 1), while
        //      warps 4..15 wait for the next task's tiles and run its prefix pass ------
        bool nxt_ok = true;
        const float* N = reinterpret_cast<const float*>(smem + SM_AF);
        float* T = reinterpret_cast<float*>(smem + SM_TF);
        if (warp < 4) {
            float* Y = reinterpret_cast<float*>(smem + SM_TB);  // scratch: [2][16][16] then [32][32]
            // (blocks above the diagonal are never written; the operand build masks them)
            // diagonal blocks: one thread per column of each 16 x 16 block (warps 0, 1),
            // right-looking: once x[m] is known every later row's sum takes its term,
            // so each step waits for one FMA
            if (warp < 2) {
                const int blk = tid >> 4, col = tid & 15;
                const float* nb = N + 16 * blk * MAT_LD + 16 * blk;
                float x[16], acc[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) acc[r] = 0.f;
                // four columns m of N at a time, each row's four as one float4
#pragma unroll
                for (int w4 = 0; w4 < 4; ++w4) {
                    float4 nv[16];
#pragma unroll
                    for (int r = 4 * w4 + 1; r < 16; ++r) nv[r] = *reinterpret_cast<const float4*>(nb + r * MAT_LD + 4 * w4);
#pragma unroll
                    for (int mm = 0; mm < 4; ++mm) {
                        const int m = 4 * w4 + mm;
                        x[m] = m == col ? 1.f : (m > col ? -acc[m] : 0.f);
#pragma unroll
                        for (int r = m + 1; r < 16; ++r) {
                            const float nrm = mm == 0 ? nv[r].x : (mm == 1 ? nv[r].y : (mm == 2 ? nv[r].z : nv[r].w));
                            acc[r] += nrm * x[m];
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) T[(16 * blk + r) * MAT_LD + 16 * blk + col] = x[r];
            }
            tc::named_sync(1, 128);
            // off-diagonal blocks, as two 32 x 32 halves T11 (tokens 0..31) and T22
            // (32..63): first the lower 16 x 16 block inside each half,
            //   T_{2p+1,2p} = -T_{2p+1,2p+1} (N_{2p+1,2p} T_{2p,2p}),   p = 0, 1,
            // then the lower half  T21 = -T22 (N21 T11).
            {
                // one thread per (p, row a, 4 columns): 128 items
                const int pp = tid >> 6, a = (tid >> 2) & 15, b4 = tid & 3;
                const int R = 2 * pp + 1, J = 2 * pp;
                {
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
                tc::named_sync(1, 128);
                {
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
                tc::named_sync(1, 128);
            }
            {
                // one thread per (rows a and a + 16, 4 columns) of a 32 x 32 block:
                // 128 items, each loaded row serving two outputs
                float* X = Y + 512;
                const int a = tid >> 3, b4 = tid & 7;
                {
                    const float* n0 = N + (32 + a) * MAT_LD;
                    const float* n1 = N + (48 + a) * MAT_LD;
                    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
                    // T11 is zero above its diagonal blocks: columns >= 16 start at row 16
                    for (int m4 = (b4 >= 4 ? 4 : 0); m4 < 8; ++m4) {
                        const float4 v0 = *reinterpret_cast<const float4*>(n0 + 4 * m4);
                        const float4 v1 = *reinterpret_cast<const float4*>(n1 + 4 * m4);
                        const float nn0[4] = {v0.x, v0.y, v0.z, v0.w}, nn1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float4 t = *reinterpret_cast<const float4*>(T + (4 * m4 + u) * MAT_LD + 4 * b4);
                            acc0.x += nn0[u] * t.x; acc0.y += nn0[u] * t.y; acc0.z += nn0[u] * t.z; acc0.w += nn0[u] * t.w;
                            acc1.x += nn1[u] * t.x; acc1.y += nn1[u] * t.y; acc1.z += nn1[u] * t.z; acc1.w += nn1[u] * t.w;
                        }
                    }
                    *reinterpret_cast<float4*>(X + a * 32 + 4 * b4) = acc0;
                    *reinterpret_cast<float4*>(X + (a + 16) * 32 + 4 * b4) = acc1;
                }
                tc::named_sync(1, 128);
                {
                    // T22 is zero above its diagonal blocks: row a < 16 stops at column 16
                    const float* t0 = T + (32 + a) * MAT_LD + 32;
                    const float* t1 = T + (48 + a) * MAT_LD + 32;
                    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
#pragma unroll 4
                    for (int m = 0; m < 16; ++m) {
                        const float tv0 = t0[m], tv1 = t1[m];
                        const float4 y = *reinterpret_cast<const float4*>(X + m * 32 + 4 * b4);
                        acc0.x += tv0 * y.x; acc0.y += tv0 * y.y; acc0.z += tv0 * y.z; acc0.w += tv0 * y.w;
                        acc1.x += tv1 * y.x; acc1.y += tv1 * y.y; acc1.z += tv1 * y.z; acc1.w += tv1 * y.w;
                    }
#pragma unroll 4
                    for (int m = 16; m < 32; ++m) {
                        const float tv1 = t1[m];
                        const float4 y = *reinterpret_cast<const float4*>(X + m * 32 + 4 * b4);
                        acc1.x += tv1 * y.x; acc1.y += tv1 * y.y; acc1.z += tv1 * y.z; acc1.w += tv1 * y.w;
                    }
                    *reinterpret_cast<float4*>(T + (32 + a) * MAT_LD + 4 * b4) = make_float4(-acc0.x, -acc0.y, -acc0.z, -acc0.w);
                    *reinterpret_cast<float4*>(T + (48 + a) * MAT_LD + 4 * b4) = make_float4(-acc1.x, -acc1.y, -acc1.z, -acc1.w);
                }
            }
        } else if (nxt.valid) {
            bool ok = true;
            if (warp == 4) ok = FUSED ? tc::bar_wait(bar_tma, tma_phase, pl.wait_iter)
                                      : tc::bar_wait(bar_g, g_phase, pl.wait_iter);
            nxt_ok = !tc::named_any(2, NT - 128, !ok);
            const int Ln = (nxt.eos - nxt.c0 < (int64_t)C) ? (int)(nxt.eos - nxt.c0) : C;
            if (nxt_ok) {
                tc::fence_after();
                for (int item = tid - 128; item < 4 * 128; item += NT - 128) prefix_item(item & 127, item >> 7, Ln);
                if constexpr (!FUSED) tc::fence_async_smem();   // (the g tile is read: the next one may land)
            }
            if constexpr (!FUSED) {
                // the q, k, v tiles (their L operand is built while the W/U MMAs run)
                if (nxt_ok) {
                    if (warp == 4) ok = tc::bar_wait(bar_tma, tma_phase, pl.wait_iter);
                    nxt_ok = !tc::named_any(2, NT - 128, !ok);
                }
            }
        }
        {
            // join: T is complete, and the next task's tiles have landed (or a wait gave up)
            const bool gave_up = __syncthreads_or(!nxt_ok) != 0;
            if (nxt.valid && !gave_up) {
                tma_phase ^= 1;
                tma_pending = false;
                if constexpr (!FUSED) {
                    g_phase ^= 1;
                    g_pending = false;
                }
            }
            failed = failed || gave_up;
            pre_done = nxt.valid && !gave_up;
            if (failed) break;
        }
        {
            // T Diag(beta) -> hi/lo B operand [64 r][64 j], K-major
            for (int item = tid; item < 64 * 8; item += NT) {
                const int r = ((item >> 6) << 3) | (item & 7);
                const int jg = (item >> 3) & 7;
                float t[8];
                const float4 a = *reinterpret_cast<const float4*>(T + r * MAT_LD + 8 * jg);
                const float4 b = *reinterpret_cast<const float4*>(T + r * MAT_LD + 8 * jg + 4);
                t[0] = a.x; t[1] = a.y; t[2] = a.z; t[3] = a.w; t[4] = b.x; t[5] = b.y; t[6] = b.z; t[7] = b.w;
#pragma unroll
                for (int u = 0; u < 8; ++u) t[u] = (8 * jg + u > r) ? 0.f : t[u];
                if constexpr (AT) {
                    // (for the backward: T itself)
                    float* to = pl.at_out + ((int64_t)cur.gc * H + h) * (2 * C * C) + C * C + r * C + 8 * jg;
                    *reinterpret_cast<float4*>(to) = make_float4(t[0], t[1], t[2], t[3]);
                    *reinterpret_cast<float4*>(to + 4) = make_float4(t[4], t[5], t[6], t[7]);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) t[u] *= beta_s[8 * jg + u];
                uint4 hi, lo;
                tc::split8(t, hi, lo);
                *reinterpret_cast<uint4*>(smem + SM_TB + tc::kmaj(r, 8 * jg, C)) = hi;
                *reinterpret_cast<uint4*>(smem + SM_TB + 8192 + tc::kmaj(r, 8 * jg, C)) = lo;
            }
        }
        publish();

        // ---- (7) W^T = (k e^G)^T (T Diag beta)^T,  U~^T = v^T (T Diag beta)^T -------
        if (warp == 0) {
            const uint32_t tb = tc::smem_u32(smem + SM_TB);
            const uint64_t tbh = tc::sdesc(tb, 128, C * 16), tbl = tc::sdesc(tb + 8192, 128, C * 16);
#pragma unroll
            for (int ks_ = 0; ks_ < C / 16; ++ks_) {
                const uint64_t bh = tc::dadv(tbh, ks_ * 256), bl = tc::dadv(tbl, ks_ * 256);
                tc::mma_ts_w(tm + TL_AW, tm + TL_KTH + ks_ * 8, bh, id_n64, ks_ > 0);
                tc::mma_ts_w(tm + TL_AU, tm + TL_VT + ks_ * 8, bh, id_n64, ks_ > 0);
                tc::mma_ts_w(tm + TL_AW, tm + TL_KTH + ks_ * 8, bl, id_n64, 1);
                tc::mma_ts_w(tm + TL_AU, tm + TL_VT + ks_ * 8, bl, id_n64, 1);
                tc::mma_ts_w(tm + TL_AW, tm + TL_KTL + ks_ * 8, bh, id_n64, 1);
                if constexpr (FUSED) tc::mma_ts_w(tm + TL_AU, tm + TL_VTL + ks_ * 8, bh, id_n64, 1);
            }
            tc::commit_w(bar_mma);
        }
        if (!FUSED && pre_done) {
            // meanwhile the next task's L operand (its A/P MMAs' TMEM is free)
            tc::fence_after();
            const int Ln = (nxt.eos - nxt.c0 < (int64_t)C) ? (int)(nxt.eos - nxt.c0) : C;
#pragma unroll 1
            for (int it = 0; it < 2; ++it) build_L(2 * (warp >> 2) + it, Ln);
            tc::tmem_st_wait();
        }
        mma_sync();
        if (failed) break;

        // ---- (8) -W hi|lo (the first half of the merged image) staged in the dead
        //      operand region for two bulk stores; U~ fp32 [64 r][128 v] straight from
        //      TMEM to the slot (a warp's 32 value columns are 128 contiguous bytes) --
        {
            const int x = (warp & 3) * 32 + lane;  // channel c of W^T, value column v of U~^T
            const int rb = (warp >> 2) * 16;
            uint32_t a[16], b[16];
            tc::tmem_ld16(tm + lane_base(warp) + TL_AW + rb, a);
            tc::tmem_ld16(tm + lane_base(warp) + TL_AU + rb, b);
            tc::tmem_ld_wait();
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {
                float w[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) w[u] = -__uint_as_float(a[8 * g8 + u]);
                uint4 hi, lo;
                tc::split8(w, hi, lo);
                *reinterpret_cast<uint4*>(smem + SM_OPB + tc::mnmaj_ng(rb + 8 * g8, x, D)) = hi;
                *reinterpret_cast<uint4*>(smem + SM_OPB + 16384 + tc::mnmaj_ng(rb + 8 * g8, x, D)) = lo;
            }
            float* ut = reinterpret_cast<float*>(slot + SLOT_UT);
#pragma unroll
            for (int i = 0; i < 16; ++i) ut[(rb + i) * D + x] = __uint_as_float(b[i]);
        }
        tc::fence_async_smem();
        __syncthreads();
        if (tid == kIssueTid) {
            tc::bulk_store(slot + SLOT_WQH, smem + SM_OPB, 16384);
            tc::bulk_store(slot + SLOT_WQL, smem + SM_OPB + 16384, 16384);
            tc::bulk_commit();
        }

        task = next_task;
        cur = nxt;
    }

    if (failed) {
        if (tid == 0) report_timeout(pl);
        // mark the slot of the task that could not finish (its e^{G_C} becomes NaN,
        // which poisons the state of that sequence), then drain a tile load in flight
        if (cur.valid && tid < 128)
            reinterpret_cast<float*>(pl.slots + ((int64_t)cur.gc * H + cur.h) * (int64_t)SLOT_BYTES + SLOT_EGC)[tid] =
                __int_as_float(0x7fc00000);
        if (tma_pending && tid == 0) tc::bar_wait(bar_tma, tma_phase, kWaitIter);
        if (g_pending && tid == 0) tc::bar_wait(bar_g, g_phase, kWaitIter);
    }
    if (tid == kIssueTid) tc::bulk_wait();
    // MMAs that a wait gave up on may still run: they complete before TMEM is released
    if (warp == 0) {
        tc::commit_w(bar_fin);
        if (lane == 0) tc::bar_wait(bar_fin, 0, kWaitIter);
        __syncwarp();
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, TL_COLS);
}

// ============================================================================
// Chunk bookkeeping for packed sequences
// ============================================================================

// chunk_off[n] = first global chunk of sequence n (exclusive prefix of
// ceil(len / C)); order = sequences longest first (ties by index) when given;
// chunk_seq[gc] = sequence of global chunk gc, -1 past the last chunk.
// One block of 1024 threads.
__global__ void __launch_bounds__(1024)
chunk_plan_kernel(const int32_t* __restrict__ cu, int N, int T, int64_t max_chunks,
                  int32_t* __restrict__ chunk_off, int32_t* __restrict__ order, int32_t* __restrict__ chunk_seq) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int n = base + tid;
        const int cnt = n < N ? (seq_len_clamped(cu, n, T) + C - 1) / C : 0;
        int v = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, d);
            if (lane >= d) v += y;
        }
        if (lane == 31) warp_sums[warp] = v;
        __syncthreads();
        if (warp == 0) {
            int w = warp_sums[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, d);
                if (lane >= d) w += y;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int incl = v + (warp > 0 ? warp_sums[warp - 1] : 0);
        const int carry = carry_s;
        if (n < N) chunk_off[n] = carry + incl - cnt;
        __syncthreads();
        if (tid == 1023) carry_s = carry + incl;
        __syncthreads();
    }
    if (tid == 0) chunk_off[N] = carry_s;
    if (order != nullptr) {
        for (int m = tid; m < N; m += 1024) {
            const int lm = seq_len_clamped(cu, m, T);
            int r = 0;
            for (int x = 0; x < N; ++x) {
                const int lx = seq_len_clamped(cu, x, T);
                r += (lx > lm) || (lx == lm && x < m);
            }
            order[r] = m;
        }
    }
    __syncthreads();
    const int total = chunk_off[N];
    for (int64_t gc = tid; gc < max_chunks; gc += 1024) {
        int s = -1;
        if (gc < total) {
            // the last sequence starting at or before gc holds it (empty ones are skipped)
            int lo = 0, hi = N - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (chunk_off[mid] <= gc) lo = mid; else hi = mid - 1;
            }
            s = lo;
        }
        chunk_seq[gc] = s;
    }
}

// ============================================================================
// State kernel
// ============================================================================

// Warps 0..15 do the TMEM epilogues (warp w: TMEM lanes 32 (w % 4).., column
// group w / 4); warp 16 only issues MMAs and bulk copies.  The two sides meet
// at mbarriers: MMA commits (u: the first round, s: the state update, o: the
// P U term) and the epilogue warps' arrivals (uready: U hi/lo written; sready:
// S hi/lo written, O read out and the chunk's o staged), once per chunk.
constexpr int NT2 = 544;
constexpr int ISSUER = 16;

// ---- shared memory map (bytes) -------------------------------------------------
constexpr uint32_t SS_KB = 2 * SLOT_IMG;    // [-W | Qs] images + e^{G_C} of two chunks, then Kbar
constexpr uint32_t SS_UT = SS_KB + SLOT_KBP;//   and P, and U~, of one chunk
constexpr uint32_t SS_BAR = SS_UT + 32768;  // img 0, img 1, u, o, s, ut, kb, uready, sready;
constexpr uint32_t SS_TOTAL = SS_BAR + 128; //   tmem base; abort flag; exit drain; testing
static_assert(SS_TOTAL + 128 <= 232448, "shared memory");

// ---- tensor memory map (columns) ----------------------------------------------
constexpr uint32_t TS_S = 0;      // S^T fp32 [128 v][128 c]
constexpr uint32_t TS_SH = 128;   // S^T hi (bf16 pairs) [128 v][64]
constexpr uint32_t TS_SL = 192;   // S^T lo
constexpr uint32_t TS_AU = 256;   // U^T accumulator fp32 [128 v][64 r]   } one N = 128
constexpr uint32_t TS_AO = 320;   // O^T accumulator fp32 [128 v][64 r]   } accumulator
constexpr uint32_t TS_UH = 384;   // U^T hi (bf16 pairs) [128 v][32]
constexpr uint32_t TS_UL = 416;   // U^T lo
constexpr uint32_t TS_COLS = 512;

// STATES: also write the state entering every chunk to pl.states_out and every chunk's
// U = U~ - W S to pl.u_out (for the backward).
template <typename TOut, bool STATES = false>
__global__ void __launch_bounds__(NT2, 1)
chunk_state_kernel(const __grid_constant__ CUtensorMap mo, const float* __restrict__ initial_state,
                   float* __restrict__ final_state, TOut* __restrict__ o, const Plan pl) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bar_img = reinterpret_cast<uint64_t*>(smem + SS_BAR);  // [2]
    uint64_t* bar_u = bar_img + 2;
    uint64_t* bar_o = bar_img + 3;
    uint64_t* bar_s = bar_img + 4;
    uint64_t* bar_ut = bar_img + 5;
    uint64_t* bar_kb = bar_img + 6;
    uint64_t* bar_uready = bar_img + 7;
    uint64_t* bar_sready = bar_img + 8;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(bar_img + 9);
    volatile int* abort_s = reinterpret_cast<volatile int*>(bar_img + 10);
    uint64_t* bar_fin = bar_img + 11;   // every MMA issued has completed (exit drain)
    uint64_t* bar_never = bar_img + 12; // testing: nothing arrives on it
    const float* ut_s = reinterpret_cast<const float*>(smem + SS_UT);   // U~ [64 r][128 v]

    const int H = pl.H;
    const Chain chn = chain_of(pl, blockIdx.x);
    const int h = chn.h, n = chn.n;
    const int64_t bos = chn.bos, eos = chn.eos, g0 = chn.g0, nchunks = chn.nchunks;

    if (warp == 0) tc::tmem_alloc(tmem_base_s, TS_COLS);
    if (tid == 0) {
#pragma unroll
        for (int b = 0; b < 7; ++b) tc::bar_init(bar_img + b, 1);
        tc::bar_init(bar_fin, 1);
        tc::bar_init(bar_never, 1);
        tc::bar_init(bar_uready, 16);
        tc::bar_init(bar_sready, 16);
        *abort_s = 0;
        tc::bar_init_fence();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tmem_base_s;

    auto slot_of = [&](int64_t i) { return pl.slots + ((g0 + i) * H + h) * (int64_t)SLOT_BYTES; };
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        return tc::bar_wait_or_abort(bar, parity, pl.wait_iter, abort_s);
    };
    auto chunk_rows = [&](int64_t i) {
        const int64_t c0 = bos + i * C;
        return (eos - c0 < (int64_t)C) ? (int)(eos - c0) : C;
    };
    const int64_t sbase = ((int64_t)n * H + h) * D * D;

    if (warp == ISSUER) {
        // ================= MMA and copy issue =================
        auto issue_img = [&](int64_t i) {
            if (lane == 0) {
                uint64_t* b = bar_img + (i & 1);
                tc::bar_expect_tx(b, SLOT_IMG);
                uint8_t* dst = smem + (i & 1) * SLOT_IMG;
                const uint8_t* src = slot_of(i);
                tc::bulk_load(dst, src, 32768, b);
                tc::bulk_load(dst + 32768, src + 32768, 32768, b);
                tc::bulk_load(dst + SLOT_EGC, src + SLOT_EGC, SLOT_IMG - SLOT_EGC, b);
            }
            __syncwarp();
        };
        // Kbar + P and U~ of one chunk (single buffers, refilled once consumed)
        auto issue_vec = [&](int64_t i, uint64_t* bar, uint32_t sm_off, uint32_t slot_off, uint32_t bytes) {
            if (lane == 0) {
                tc::bar_expect_tx(bar, bytes);
                tc::bulk_load(smem + sm_off, slot_of(i) + slot_off, bytes, bar);
            }
            __syncwarp();
        };
        // o of a full chunk, staged in its image buffer by the epilogue warps
        // (a sequence's ragged last chunk is stored by the epilogue warps)
        auto store_o = [&](int64_t i) {
            if (chunk_rows(i) == C && lane == 0) {
                tc::tma_store_3d(&mo, smem + (i & 1) * SLOT_IMG + SLOT_WQH, 0, h, (int)(bos + i * C));
                tc::bulk_commit();
            }
        };
        int64_t issued = 0, done = 0;  // image loads issued / known complete
        int64_t ut_issued = 0, kb_issued = 0;
        if (nchunks > 0) {
            issue_img(0);
            issue_vec(0, bar_kb, SS_KB, SLOT_KH, SLOT_KBP);
            issue_vec(0, bar_ut, SS_UT, SLOT_UT, 32768);
            issued = 1;
            ut_issued = kb_issued = 1;
        }
        if (nchunks > 1) { issue_img(1); issued = 2; }
        const uint32_t id_n128_bmn = tc::idesc_bf16(128, 128, false, true);
        const uint32_t id_n128 = tc::idesc_bf16(128, 128);
        const uint32_t id_n64 = tc::idesc_bf16(128, 64);
        bool ok = true;
        if (pl.inject == 2) ok = wait(bar_never, 0);
        for (int64_t i = 0; i < nchunks && ok; ++i) {
            const uint32_t par = (uint32_t)(i & 1);
            if (!wait(bar_img + (i & 1), (uint32_t)((i >> 1) & 1))) { ok = false; break; }
            done = i + 1;
            // S_i hi/lo are written, and chunk i-1's o is staged
            if (!wait(bar_sready, par)) { ok = false; break; }
            tc::fence_after();
            if (i >= 1) store_o(i - 1);
            const uint32_t img = tc::smem_u32(smem + (i & 1) * SLOT_IMG);
            // [U^T | O^T] = S^T [-W | Qs]^T with both operands split hi|lo:
            //   S_hi [-W hi | Qs hi] + S_lo [-W hi | Qs hi] + S_hi [-W lo | Qs lo]
            const uint64_t bh = tc::sdesc(img + SLOT_WQH, 128, D * 16);
            const uint64_t bl = tc::sdesc(img + SLOT_WQL, 128, D * 16);
#pragma unroll
            for (int ks_ = 0; ks_ < D / 16; ++ks_) {
                const uint32_t off = ks_ * 256;
                tc::mma_ts_w(tm + TS_AU, tm + TS_SH + ks_ * 8, tc::dadv(bh, off), id_n128_bmn, ks_ > 0);
                tc::mma_ts_w(tm + TS_AU, tm + TS_SL + ks_ * 8, tc::dadv(bh, off), id_n128_bmn, 1);
                tc::mma_ts_w(tm + TS_AU, tm + TS_SH + ks_ * 8, tc::dadv(bl, off), id_n128_bmn, 1);
            }
            tc::commit_w(bar_u);
            // chunk i+1's images go where chunk i-1's were, once its o has left
            if (i >= 1 && i + 1 < nchunks) {
                tc::bulk_wait_read();
                __syncwarp();
                issue_img(i + 1);
                issued = i + 2;
            }
            // once U hi/lo are in TMEM (the decay came before them):
            // S^T += U^T Kbar, then O^T += U^T (scale P)^T
            if (!wait(bar_uready, par) || !wait(bar_kb, par)) { ok = false; break; }
            tc::fence_after();
            const uint32_t kb = tc::smem_u32(smem + SS_KB);
            const uint64_t khd = tc::sdesc(kb, 128, C * 16), kld = tc::sdesc(kb + 16384, 128, C * 16);
            const uint64_t phd = tc::sdesc(kb + (SLOT_P - SLOT_KH), 128, C * 16);
            const uint64_t pld = tc::sdesc(kb + (SLOT_P - SLOT_KH) + 8192, 128, C * 16);
#pragma unroll
            for (int ks_ = 0; ks_ < C / 16; ++ks_) {
                const uint32_t uh = tm + TS_UH + ks_ * 8, ul = tm + TS_UL + ks_ * 8;
                const uint64_t bh2 = tc::dadv(khd, ks_ * 256), bl2 = tc::dadv(kld, ks_ * 256);
                tc::mma_ts_w(tm + TS_S, uh, bh2, id_n128, 1);
                tc::mma_ts_w(tm + TS_S, uh, bl2, id_n128, 1);
                tc::mma_ts_w(tm + TS_S, ul, bh2, id_n128, 1);
            }
            tc::commit_w(bar_s);
#pragma unroll
            for (int ks_ = 0; ks_ < C / 16; ++ks_) {
                const uint32_t uh = tm + TS_UH + ks_ * 8, ul = tm + TS_UL + ks_ * 8;
                const uint64_t ph = tc::dadv(phd, ks_ * 256), pl_ = tc::dadv(pld, ks_ * 256);
                tc::mma_ts_w(tm + TS_AO, uh, ph, id_n64, 1);
                tc::mma_ts_w(tm + TS_AO, uh, pl_, id_n64, 1);
                tc::mma_ts_w(tm + TS_AO, ul, ph, id_n64, 1);
            }
            tc::commit_w(bar_o);
            // U~ of this chunk is consumed (U hi/lo are written): fetch the next one
            if (i + 1 < nchunks) {
                issue_vec(i + 1, bar_ut, SS_UT, SLOT_UT, 32768);
                ut_issued = i + 2;
                // Kbar and P are free once this chunk's last MMAs have completed
                if (!wait(bar_o, par)) { ok = false; break; }
                issue_vec(i + 1, bar_kb, SS_KB, SLOT_KH, SLOT_KBP);
                kb_issued = i + 2;
            }
        }
        // the last chunk's o
        if (ok && nchunks > 0 && wait(bar_sready, (uint32_t)(nchunks & 1))) store_o(nchunks - 1);
        // drain loads that may still be in flight before the CTA exits
        if (*abort_s && lane == 0) {
            report_timeout(pl);
            for (int64_t j = done; j < issued; ++j) tc::bar_wait(bar_img + (j & 1), (uint32_t)((j >> 1) & 1), kWaitIter);
            if (ut_issued > 0) tc::bar_wait(bar_ut, (uint32_t)((ut_issued - 1) & 1), kWaitIter);
            if (kb_issued > 0) tc::bar_wait(bar_kb, (uint32_t)((kb_issued - 1) & 1), kWaitIter);
        }
        // MMAs that a wait gave up on may still run: they complete before TMEM is released
        tc::commit_w(bar_fin);
        if (lane == 0) tc::bar_wait(bar_fin, 0, kWaitIter);
        __syncwarp();
        tc::bulk_wait();
    } else {
        // ================= TMEM epilogues =================
        const int x = (warp & 3) * 32 + lane;   // TMEM lane: value column v
        const int rb = (warp >> 2) * 16;        // accumulator columns (tokens) of this warp
        const int cc = (warp >> 2) * 32;        // state columns (key channels) of this warp
        auto arrive = [&](uint64_t* bar) {
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::bar_arrive(bar);
        };
        // S hi/lo from the fp32 state in TMEM
        auto s_epilogue = [&]() {
            uint32_t a[32];
            tc::tmem_ld16(tm + lane_base(warp) + TS_S + cc, a);
            tc::tmem_ld16(tm + lane_base(warp) + TS_S + cc + 16, a + 16);
            tc::tmem_ld_wait();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    tc::split2(__uint_as_float(a[16 * half + 2 * j]), __uint_as_float(a[16 * half + 2 * j + 1]), hi[j], lo[j]);
                tc::tmem_st8(tm + lane_base(warp) + TS_SH + cc / 2 + 8 * half, hi);
                tc::tmem_st8(tm + lane_base(warp) + TS_SL + cc / 2 + 8 * half, lo);
            }
            tc::tmem_st_wait();
        };
        // initial state: S^T in TMEM (lane x holds row x of S^T = column x of S)
        for (int c = cc; c < cc + 32; c += 16) {
            uint32_t r[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                r[j] = __float_as_uint(initial_state ? initial_state[sbase + (int64_t)(c + j) * D + x] : 0.f);
            tc::tmem_st16(tm + lane_base(warp) + TS_S + c, r);
        }
        tc::tmem_st_wait();
        s_epilogue();
        arrive(bar_sready);

        for (int64_t i = 0; i < nchunks; ++i) {
            const uint32_t par = (uint32_t)(i & 1);
            const int64_t c0 = bos + i * C;
            const int L = chunk_rows(i);

            // decay the fp32 state by e^{G_C} (the MMAs under way read S hi/lo)
            if (!wait(bar_img + (i & 1), (uint32_t)((i >> 1) & 1))) break;
            {
                const float* eg = reinterpret_cast<const float*>(smem + (i & 1) * SLOT_IMG + SLOT_EGC) + cc;
                uint32_t s0[16], s1[16];
                tc::tmem_ld16(tm + lane_base(warp) + TS_S + cc, s0);
                tc::tmem_ld16(tm + lane_base(warp) + TS_S + cc + 16, s1);
                tc::tmem_ld_wait();
                if constexpr (STATES) {
                    // the state entering this chunk, S[c][x] (a warp's 32 lanes are 32 consecutive x)
                    float* so = pl.states_out + ((g0 + i) * H + h) * (int64_t)(D * D) + x;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        so[(int64_t)(cc + j) * D] = __uint_as_float(s0[j]);
                        so[(int64_t)(cc + 16 + j) * D] = __uint_as_float(s1[j]);
                    }
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    s0[j] = __float_as_uint(__uint_as_float(s0[j]) * eg[j]);
                    s1[j] = __float_as_uint(__uint_as_float(s1[j]) * eg[16 + j]);
                }
                tc::tmem_st16(tm + lane_base(warp) + TS_S + cc, s0);
                tc::tmem_st16(tm + lane_base(warp) + TS_S + cc + 16, s1);
                tc::tmem_st_wait();
            }

            // U = U~ - W S, hi/lo into TMEM
            if (!wait(bar_ut, par) || !wait(bar_u, par)) break;
            tc::fence_after();
            {
                uint32_t a[16];
                tc::tmem_ld16(tm + lane_base(warp) + TS_AU + rb, a);
                tc::tmem_ld_wait();
                uint32_t hi[8], lo[8];
                float u[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) u[j] = ut_s[(rb + j) * D + x] + __uint_as_float(a[j]);
                if constexpr (STATES) {
                    // U of this chunk, U[r][x] (a warp's 32 lanes are 32 consecutive x)
                    float* uo = pl.u_out + ((g0 + i) * H + h) * (int64_t)(C * D) + x;
#pragma unroll
                    for (int j = 0; j < 16; ++j) uo[(int64_t)(rb + j) * D] = u[j];
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) tc::split2(u[2 * j], u[2 * j + 1], hi[j], lo[j]);
                tc::tmem_st8(tm + lane_base(warp) + TS_UH + rb / 2, hi);
                tc::tmem_st8(tm + lane_base(warp) + TS_UL + rb / 2, lo);
                tc::tmem_st_wait();
            }
            arrive(bar_uready);

            // S hi/lo for the next chunk
            if (!wait(bar_s, par)) break;
            tc::fence_after();
            s_epilogue();

            // o = O: a full chunk is staged as [64 r][128 v] in the [-W | Qs] image
            // region, which this chunk's MMAs are done with, for one tiled store by
            // the issuer
            if (!wait(bar_o, par)) break;
            tc::fence_after();
            {
                uint32_t a[16];
                tc::tmem_ld16(tm + lane_base(warp) + TS_AO + rb, a);
                tc::tmem_ld_wait();
                if (L == C) {
                    TOut* ost = reinterpret_cast<TOut*>(smem + (i & 1) * SLOT_IMG + SLOT_WQH);
#pragma unroll
                    for (int j = 0; j < 16; ++j) ost[(rb + j) * D + x] = from_f32<TOut>(__uint_as_float(a[j]));
                } else {
                    const int64_t ob = ((c0 + rb) * H + h) * (int64_t)D + x;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (rb + j < L) o[ob + (int64_t)j * H * D] = from_f32<TOut>(__uint_as_float(a[j]));
                }
            }
            tc::fence_async_smem();
            arrive(bar_sready);
        }
        // ---- final state ---------------------------------------------------------
        if (final_state) {
            const bool failed = *abort_s != 0;
            for (int c = cc; c < cc + 32; c += 16) {
                uint32_t sv[16];
                tc::tmem_ld16(tm + lane_base(warp) + TS_S + c, sv);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    final_state[sbase + (int64_t)(c + j) * D + x] = failed ? __int_as_float(0x7fc00000) : __uint_as_float(sv[j]);
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, TS_COLS);
}

// ============================================================================
// Host side
// ============================================================================

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

// [rows][H][128] output tensor; box = 64 rows x 128 values of one head, no swizzle.
template <typename TOut>
bool make_out_map(CUtensorMap* m, void* base, int64_t rows, int H) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * sizeof(TOut), (cuuint64_t)H * D * sizeof(TOut)};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        sizeof(TOut) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return fn(m, dt, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][H][128] bf16 tensor; box = 64 rows x 64 channels of one head, 128B
// swizzle (halo = false), or 3 rows x 64 channels without swizzle (halo = true).
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int H, bool halo = false) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, halo ? 3u : (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, halo ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// SM count of the current device, looked up once per device.
constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
int g_sm_count[kMaxDevices];

cudaError_t device_sms(int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_sm_count[dev] == 0) {
        e = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    *sms = g_sm_count[dev];
    return cudaSuccess;
}

// Events that the next prefill call on this host thread records (timing hook).
thread_local cudaEvent_t g_trace[3] = {nullptr, nullptr, nullptr};
// Wait-timeout injection of the next prefill call on this host thread (testing hook).
thread_local int g_inject = 0;

void trace_record(cudaEvent_t ev, cudaStream_t st) {
    if (ev != nullptr) cudaEventRecord(ev, st);
}

// Workspace of one call: packed-sequence bookkeeping (chunk offsets, longest-
// first order, chunk -> sequence map) rounded up to 1 KiB, then one slot per
// (chunk, head).  max_chunks is exact without cu_seqlens and an upper bound
// (ceil(T / 64) + N) with it.
struct Layout {
    int64_t max_chunks;
    size_t hdr_bytes;
    size_t bytes;
};
Layout layout(int B, int T, int H, int N, bool packed) {
    Layout l{};
    const int64_t cps = ((int64_t)T + C - 1) / C;
    l.max_chunks = packed ? cps + N : (int64_t)B * cps;
    const size_t hdr_ints = packed ? (size_t)(2 * (int64_t)N + 1) + (size_t)l.max_chunks : 0;
    l.hdr_bytes = (hdr_ints * 4 + 1023) & ~size_t(1023);
    l.bytes = l.hdr_bytes + (size_t)l.max_chunks * (size_t)H * SLOT_BYTES;
    if ((int64_t)N * H == 0) l.bytes = 0;
    return l;
}

// The prefill's kernels on a caller-owned workspace of ws_bytes.  With states_out the
// state kernel also writes the state entering every chunk there, with at_out the
// local kernel each chunk's A and T; plan_out receives the work plan (all for the
// backward).
template <typename TOut>
cudaError_t launch_tc(const ChunkParams& p, cudaStream_t st, void* ws, size_t ws_bytes, int32_t* status,
                      bool fused, float* states_out = nullptr, Plan* plan_out = nullptr, float* at_out = nullptr,
                      float* u_out = nullptr) {
    cudaEvent_t trace[3] = {g_trace[0], g_trace[1], g_trace[2]};
    g_trace[0] = g_trace[1] = g_trace[2] = nullptr;
    cudaError_t e = cudaSuccess;
    if (status != nullptr) {
        e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
        if (e != cudaSuccess) return e;
    }
    const int64_t NH = (int64_t)p.N * p.H;
    if (NH == 0) return cudaSuccess;
    const bool packed = p.cu_seqlens != nullptr;
    const Layout lo = layout(p.B, p.T, p.H, p.N, packed);
    if (lo.bytes > ws_bytes || (lo.bytes > 0 && ws == nullptr)) return cudaErrorMemoryAllocation;
    int sms = 0;
    e = device_sms(&sms);
    if (e != cudaSuccess) return e;
    Plan pl{};
    pl.cu_seqlens = p.cu_seqlens;
    pl.T = p.T;
    pl.H = p.H;
    pl.N = p.N;
    pl.cps = packed ? 0 : (p.T + C - 1) / C;
    pl.max_chunks = lo.max_chunks;
    pl.status = status;
    const uint32_t lim = g_wait_limit.load(std::memory_order_relaxed);
    pl.wait_iter = lim != 0 ? lim : kWaitIter;
    pl.inject = g_inject;
    g_inject = 0;
    pl.states_out = states_out;
    pl.at_out = at_out;
    pl.u_out = u_out;
    int32_t* hdr = reinterpret_cast<int32_t*>(ws);
    pl.slots = reinterpret_cast<uint8_t*>(ws) + lo.hdr_bytes;
    trace_record(trace[0], st);
    if (packed) {
        pl.chunk_off = hdr;
        pl.order = p.N <= 1024 ? hdr + (p.N + 1) : nullptr;
        pl.chunk_seq = hdr + (2 * (int64_t)p.N + 1);
        chunk_plan_kernel<<<1, 1024, 0, st>>>(p.cu_seqlens, p.N, p.T, pl.max_chunks,
                                              const_cast<int32_t*>(pl.chunk_off), const_cast<int32_t*>(pl.order),
                                              const_cast<int32_t*>(pl.chunk_seq));
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int64_t tasks = pl.max_chunks * p.H;
    if (tasks >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
    if (tasks > 0) {
        const int64_t rows = (int64_t)p.B * p.T;
        CUtensorMap mq, mk, mv, mg, hq, hk, hv;
        bool ok = make_map(&mq, p.q, rows, p.H) && make_map(&mk, p.k, rows, p.H) && make_map(&mv, p.v, rows, p.H) &&
                  make_map(&mg, p.g, rows, p.H);
        if (fused) {
            ok = ok && make_map(&hq, p.q, rows, p.H, true) && make_map(&hk, p.k, rows, p.H, true) &&
                 make_map(&hv, p.v, rows, p.H, true);
        } else {
            hq = mq; hk = mk; hv = mv;  // unused
        }
        if (!ok) return cudaErrorInvalidValue;
        Prologue pro{};
        pro.conv_q = p.conv_q; pro.conv_k = p.conv_k; pro.conv_v = p.conv_v;
        pro.A_log = p.A_log; pro.dt_bias = p.dt_bias;
        pro.lower_bound = p.lower_bound; pro.l2_eps = p.l2_eps;
        auto kern = !fused ? (at_out != nullptr ? chunk_local_kernel<false, false, true> : chunk_local_kernel<false>)
                           : (p.conv_act == 1 ? chunk_local_kernel<true, true> : chunk_local_kernel<true, false>);
        const int smem_bytes = (int)(fused ? SM_LOCAL_TOTAL_FUSED : SM_LOCAL_TOTAL) + 1024;  // + alignment slack
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess) return e;
        const int64_t grid = tasks < sms ? tasks : sms;
        kern<<<(unsigned)grid, NT, smem_bytes, st>>>(mq, mk, mv, mg, hq, hk, hv, p.beta, p.scale, pl, pro);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        trace_record(trace[1], st);
    }
    if (plan_out != nullptr) *plan_out = pl;
    auto kern = states_out != nullptr ? chunk_state_kernel<TOut, true> : chunk_state_kernel<TOut, false>;
    const int smem_bytes = (int)SS_TOTAL + 128;
    CUtensorMap mo;
    const int64_t rows = (int64_t)p.B * p.T;
    if (!make_out_map<TOut>(&mo, p.o, rows > 0 ? rows : 1, p.H)) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)NH, NT2, smem_bytes, st>>>(mo, p.initial_state, p.final_state, reinterpret_cast<TOut*>(p.o), pl);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    trace_record(trace[2], st);
    return cudaSuccess;
}

// ---- prefill without any allocation ---------------------------------------------
// Workspace in a fixed device array that every GPU loading the library holds
// until exit.  Its device address is looked up once per device, on the first
// call made with that device current.
static __device__ __align__(256) uint8_t g_fixed_scratch[kFixedScratchBytes];
std::mutex g_fixed_mutex;
void* g_fixed_ptr[kMaxDevices];

cudaError_t fixed_scratch(void** ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_fixed_mutex);
    if (g_fixed_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fixed_scratch);
        if (e != cudaSuccess) return e;
        g_fixed_ptr[dev] = p;
    }
    *ptr = g_fixed_ptr[dev];
    return cudaSuccess;
}

}  // namespace

bool chunk_tc_supported(kda_dtype in_dt, int K, int V) { return in_dt == KDA_BF16 && K == D && V == D; }

size_t chunk_tc_workspace(int B, int T, int H, int N, bool packed) { return layout(B, T, H, N, packed).bytes; }

void trace_set(void* begin, void* split, void* end) {
    g_trace[0] = static_cast<cudaEvent_t>(begin);
    g_trace[1] = static_cast<cudaEvent_t>(split);
    g_trace[2] = static_cast<cudaEvent_t>(end);
}

void set_wait_limit(uint32_t iterations) { g_wait_limit.store(iterations, std::memory_order_relaxed); }

void inject_wait_timeout(int kernel) { g_inject = (kernel >= 1 && kernel <= 4) ? kernel : 0; }

cudaError_t chunk_tc(kda_dtype out_dt, const ChunkParams& p, void* ws, size_t ws_bytes, int32_t* status,
                     cudaStream_t st) {
    if (out_dt == KDA_F32) return launch_tc<float>(p, st, ws, ws_bytes, status, false);
    return launch_tc<__nv_bfloat16>(p, st, ws, ws_bytes, status, false);
}

cudaError_t chunk_tc_fused(kda_dtype out_dt, const ChunkParams& p, void* ws, size_t ws_bytes, int32_t* status,
                           cudaStream_t st) {
    if (out_dt == KDA_F32) return launch_tc<float>(p, st, ws, ws_bytes, status, true);
    return launch_tc<__nv_bfloat16>(p, st, ws, ws_bytes, status, true);
}

cudaError_t chunk_tc_forward_states(const ChunkParams& p, void* ws, size_t ws_bytes, float* states_out,
                                    float* at_out, float* u_out, cplan::Plan* plan_out, int32_t* status,
                                    cudaStream_t st) {
    return launch_tc<__nv_bfloat16>(p, st, ws, ws_bytes, status, false, states_out, plan_out, at_out, u_out);
}

cudaError_t chunk_tc_fixed_scratch(kda_dtype out_dt, const ChunkParams& p, cudaStream_t st) {
    void* ws = nullptr;
    const cudaError_t e = fixed_scratch(&ws);
    if (e != cudaSuccess) return e;
    if (out_dt == KDA_F32) return launch_tc<float>(p, st, ws, kFixedScratchBytes, nullptr, false);
    return launch_tc<__nv_bfloat16>(p, st, ws, kFixedScratchBytes, nullptr, false);
}

}  // namespace kda
