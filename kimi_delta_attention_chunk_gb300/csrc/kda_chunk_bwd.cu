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
//       state S entering every chunk, each chunk's U = U~ - W S (its state kernel
//       forms it anyway) and each chunk's A and T; its workspace slots keep W,
//       Qs = scale Xq, Kb, scale P, U~ and e^{G_C} per (chunk, head);
//   bwd_chain_kernel: one CTA per (sequence, head) carries dS backwards through the
//       chunks (the first two lines above) with dS'^T in tensor memory, tcgen05
//       rounds on the slots' operand images, and stores dS' and dU of every chunk;
//   bwd_chunk_kernel: one CTA per (chunk, head) task forms dq, dk, dv, dg, dbeta; its
//       products are tensor-core rounds (tcgen05, operands split hi | lo into bf16,
//       fp32 accumulators in tensor memory) on operands staged from a per-CTA scratch.
#include "kda_chunk.h"
#include "kda_chunk_plan.cuh"
#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace cplan;

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
    SC_DXQ = SC_QL + MR, SC_DWU = SC_DXQ + MR, SC_DKB = SC_DWU + 2 * MR,
    SC_DBKV = SC_DKB + MR, SC_GB = SC_DBKV + 2 * MR, SC_GF = SC_GB + MR,
    SC_GC = SC_GF + MR,
    SC_DP = SC_GC + MR, SC_DM = SC_DP + MQ, SC_DA = SC_DM + MQ,
    SC_TOTAL = SC_DA + MQ
};
static_assert(SC_TOTAL * 4 == 638976, "the per-CTA scratch size stated in kda.h");
// Shared memory of the chunk kernel: the operand images of one tensor-core round
// (bf16 hi | lo), then small tables and the MMA barriers.
constexpr uint32_t OP_BYTES = 160 * 1024;               // the largest round: A 128 x 64 + 4 B variants 128 x 64
constexpr uint32_t BK_TOT = OP_BYTES;                   // tot [4][128]: e^g products over each 16-token block
constexpr uint32_t BK_PT = BK_TOT + 4 * D * 4;          // ptot [4 B][4 b][128]: prod of tot over blocks [B, b)
constexpr uint32_t BK_BETA = BK_PT + 16 * D * 4;        // beta [64]
constexpr uint32_t BK_DEC = BK_BETA + C * 4;            // dEC [128]
constexpr uint32_t BK_EC = BK_DEC + D * 4;              // e^{G_C} [128]
constexpr uint32_t BK_BAR = BK_EC + D * 4;              // MMA barrier, exit barrier, TMEM base
constexpr uint32_t BK_TOTAL = BK_BAR + 64;
static_assert(BK_TOTAL <= 232448, "shared memory of the chunk kernel");
static_assert(2 * C * (C + 1) * 4 <= OP_BYTES && 2 * MR * 4 <= OP_BYTES, "scratch uses of the operand area");

// The float4 unit i of an [R][CO] matrix -> its row r and first column c: each warp
// covers eight consecutive rows of four consecutive column groups, so that the
// operand stores below fill whole 128-byte runs.
template <int R, int CO>
__device__ __forceinline__ void unit_rc(int i, int& r, int& c) {
    const int rest = i >> 3;
    c = 4 * (rest % (CO / 4));
    r = (rest / (CO / 4)) * 8 + (i & 7);
}

struct Ident {
    __device__ __forceinline__ void operator()(int, int, float4&) const {}
};
constexpr int kStageInFlight = 8;   // float4 loads in flight per thread while staging an operand
struct Neg {
    __device__ __forceinline__ void operator()(int, int, float4& x) const {
        x.x = -x.x; x.y = -x.y; x.z = -x.z; x.w = -x.w;
    }
};
struct OneVariant {
    __device__ __forceinline__ int operator()(int) const { return 0; }
};

// ---- tensor-core rounds ------------------------------------------------------------
// An operand image is [rows][Kd] bf16 without swizzle: 8-row groups Kd * 16 bytes
// apart, groups of 8 k 128 bytes apart; inside a 16-byte core-matrix row either 8
// consecutive k of one operand row (K-major) or 8 consecutive operand rows of one k
// (MN-major).  Both take the descriptor strides (128, Kd * 16), and 16 k further on
// is 256 bytes further.  Each product is formed as hi hi + hi lo + lo hi of the
// operands split x = hi + lo into bf16 (about 16 significant bits), accumulated in
// fp32 in tensor memory.
__device__ __forceinline__ uint32_t op_off(int row, int k, int Kd, bool mn) {
    return (uint32_t)((row >> 3) * (Kd * 16) + (k >> 3) * 128 +
                      (mn ? (k & 7) * 16 + (row & 7) * 2 : (row & 7) * 16 + (k & 7) * 2));
}

// An [R][CO] fp32 matrix in global memory (row stride ld) into an operand image, each
// float4 passed through f(r + r_off, c + c_off, v) first (its coordinates in the
// whole matrix).  KROW: the matrix rows are operand rows row0 + r and its columns
// are k (K-major image); else its rows are k and its columns operand rows row0 + c
// (MN-major image).  kStageInFlight float4 loads in flight per thread.  ONCE: the
// source's last read in the task, loaded with the streaming hint (first out of L2),
// so that the per-CTA scratch, read again round after round, keeps its place.
template <int R, int CO, bool KROW, bool ONCE = false, typename F = Ident>
__device__ __forceinline__ void stage_op(const float* src, int ld, uint8_t* hi, uint8_t* lo, int Kd, int row0,
                                         int r_off = 0, int c_off = 0, F f = F()) {
    static_assert(R % 8 == 0 && CO % 4 == 0, "operand tile");
    constexpr int NV = R * (CO / 4);
    constexpr int IF = kStageInFlight;
    for (int i0 = threadIdx.x; i0 < NV; i0 += IF * kChunkThreads) {
        float4 v[IF];
#pragma unroll
        for (int u = 0; u < IF; ++u) {
            const int i = i0 + u * kChunkThreads;
            if (i < NV) {
                int r, c;
                unit_rc<R, CO>(i, r, c);
                const float4* a = reinterpret_cast<const float4*>(src + (int64_t)r * ld + c);
                v[u] = ONCE ? __ldcs(a) : *a;
            }
        }
#pragma unroll
        for (int u = 0; u < IF; ++u) {
            const int i = i0 + u * kChunkThreads;
            if (i >= NV) break;
            int r, c;
            unit_rc<R, CO>(i, r, c);
            f(r + r_off, c + c_off, v[u]);
            uint2 h, l;
            tc::split2(v[u].x, v[u].y, h.x, l.x);
            tc::split2(v[u].z, v[u].w, h.y, l.y);
            const uint32_t o = KROW ? op_off(row0 + r, c, Kd, false) : op_off(row0 + c, r, Kd, true);
            *reinterpret_cast<uint2*>(hi + o) = h;
            *reinterpret_cast<uint2*>(lo + o) = l;
        }
    }
}
// Operand rows [row0, 128) of an image set to zero (one contiguous range per half).
__device__ __forceinline__ void zero_rows(uint8_t* hi, uint8_t* lo, int Kd, int row0) {
    const int b0 = (row0 >> 3) * Kd * 16, n = (16 - (row0 >> 3)) * Kd * 16;
    for (int i = threadIdx.x * 16; i < n; i += kChunkThreads * 16) {
        *reinterpret_cast<uint4*>(hi + b0 + i) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(lo + b0 + i) = make_uint4(0u, 0u, 0u, 0u);
    }
}

// The tensor-memory accumulators and the barrier of the rounds.
struct Tc {
    uint8_t* op;        // operand area
    uint32_t tm;        // TMEM base (512 columns)
    uint64_t* bar;      // MMA completion
    uint32_t phase;
    uint32_t wait_iter;
    bool failed;
    uint64_t* never;    // testing: an mbarrier that nothing arrives on
    bool inject;        // testing: the next wait is on it
};

// One round: D_b (+)= A B_b^T for the NB variants b (TMEM columns [b N, b N + N)),
// M = 128 rows, K = Kd; sa(a_hi, a_lo) writes A [128][Kd], sb(b_hi, b_lo, b) B_b
// [N][Kd].  acc: add to what the accumulators hold.  False if the wait gave up.
template <int N, int NB, bool A_MN, bool B_MN, typename SA, typename SB>
__device__ __forceinline__ bool tc_round(Tc& t, int Kd, bool acc, SA sa, SB sb) {
    static_assert(N % 16 == 0 && N >= 16 && N <= 256 && N * NB <= 512, "accumulator shape");
    const int warp = threadIdx.x >> 5;
    uint8_t* a_hi = t.op;
    uint8_t* a_lo = a_hi + 128 * Kd * 2;
    uint8_t* b_base = a_hi + 128 * Kd * 4;
    const int bstride = N * Kd * 4;
    tc::fence_before();
    __syncthreads();   // the last round's MMAs and epilogue are done with the operand area and TMEM
    sa(a_hi, a_lo);
    for (int b = 0; b < NB; ++b) sb(b_base + b * bstride, b_base + b * bstride + N * Kd * 2, b);
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) {
        constexpr uint32_t id = tc::idesc_bf16(128, N, false, B_MN, A_MN);
        const uint32_t ah = tc::smem_u32(a_hi), al = tc::smem_u32(a_lo);
        for (int b = 0; b < NB; ++b) {
            const uint32_t bh = tc::smem_u32(b_base + b * bstride), bl = bh + N * Kd * 2;
            const uint32_t d = t.tm + (uint32_t)(b * N);
            for (int ks = 0; ks < Kd / 16; ++ks) {
                const uint32_t o = ks * 256;
                const uint64_t dah = tc::sdesc(ah + o, 128, Kd * 16), dal = tc::sdesc(al + o, 128, Kd * 16);
                const uint64_t dbh = tc::sdesc(bh + o, 128, Kd * 16), dbl = tc::sdesc(bl + o, 128, Kd * 16);
                tc::mma_ss_w(d, dah, dbh, id, (acc || ks > 0) ? 1u : 0u);
                tc::mma_ss_w(d, dah, dbl, id, 1u);
                tc::mma_ss_w(d, dal, dbh, id, 1u);
            }
        }
        tc::commit_w(t.bar);
    }
    bool ok = true;
    if (warp == 0) ok = t.inject ? tc::bar_wait(t.never, 0, t.wait_iter) : tc::bar_wait(t.bar, t.phase, t.wait_iter);
    t.inject = false;
    const bool gave_up = __syncthreads_or(!ok) != 0;
    if (!gave_up) t.phase ^= 1;
    t.failed = t.failed || gave_up;
    tc::fence_after();
    return !gave_up;
}

// Epilogue of a round: row r < rows of D_{vsel(r)} (vsel constant over 16 rows), the
// N columns split over the four warpgroups, 16 at a time: epi(r, c0, v[16]); called
// by every thread, it returns once all the outputs are written.
template <int N, int NB, typename VS, typename EPI>
__device__ __forceinline__ void tc_epi(const Tc& t, int rows, VS vsel, EPI epi) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3, wg = warp >> 2;
    constexpr int CW = N / 4;
    static_assert(CW % 16 == 0, "columns per warpgroup");
    if (32 * q < rows) {
        const int r = 32 * q + lane;
        const uint32_t base = t.tm + ((uint32_t)(32 * q) << 16);
        const int b0 = NB > 1 ? vsel(32 * q) : 0, b1 = NB > 1 ? vsel(32 * q + 16) : 0;
#pragma unroll 1
        for (int c0 = wg * CW; c0 < (wg + 1) * CW; c0 += 16) {
            uint32_t u[16];
            tc::tmem_ld16(base + (uint32_t)(b0 * N + c0), u);
            if (NB > 1 && b1 != b0) {
                uint32_t w[16];
                tc::tmem_ld16(base + (uint32_t)(b1 * N + c0), w);
                tc::tmem_ld_wait();
                if (lane >= 16)
#pragma unroll
                    for (int e = 0; e < 16; ++e) u[e] = w[e];
            } else {
                tc::tmem_ld_wait();
            }
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(u[e]);
            epi(r, c0, v);
        }
    }
    tc::fence_before();
    __syncthreads();   // the outputs are complete
}

// C[c0 .. c0 + 16) of a row = alpha v (+ what it holds when acc)
__device__ __forceinline__ void put16(float* cr, const float* v, float alpha, bool acc) {
#pragma unroll
    for (int e = 0; e < 16; e += 4) {
        float4 x = make_float4(alpha * v[e], alpha * v[e + 1], alpha * v[e + 2], alpha * v[e + 3]);
        if (acc) {
            const float4 o = *reinterpret_cast<const float4*>(cr + e);
            x.x += o.x; x.y += o.y; x.z += o.z; x.w += o.w;
        }
        *reinterpret_cast<float4*>(cr + e) = x;
    }
}

template <typename TIn>
__device__ __forceinline__ float ld_in(const TIn* p) { return to_f32<TIn>(*p); }
__device__ __forceinline__ void ld4(const float* p, float* x) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
// (a source's last read in the task: streaming hint)
__device__ __forceinline__ void ld4_once(const float* p, float* x) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(p));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}

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

// ---- reverse chain (tensor cores) ----------------------------------------------------
// One CTA per (sequence, head).  The gradient of the state after the chunk, dS', lives
// in tensor memory as dS'^T (lane = value column x, column = key channel c, fp32) for
// the whole sequence; per chunk, last to first:
//   store dS' (for the chunk kernel), split it hi | lo into TMEM, scale it by e^{G_C}
//   (columns c), then
//   dU^T  = dO^T (scale P)^T + dS'^T Kb^T              (M = 128 x, N = 64 r)
//   store dU, split it hi | lo into TMEM, and
//   dS^T += dO^T (Qs)^T + dU^T (-W)^T                   (M = 128 x, N = 128 c)
// The forward's slot images serve as the B operands in place: P and Kb (K-major
// images of P and Kb^T) are read MN-major as P^T and Kb^T... with their core-matrix
// groups along k 1024 bytes apart; -W and Qs (the n-group-major image of [-W | Qs]
// over c) are read K-major with k (= r) groups 2048 bytes apart.  dO^T is staged from
// global memory as an MN-major image.  Operands split hi | lo, three MMA terms each.
constexpr int kChainThreads = 256;
constexpr uint32_t CS_IMG = 0;                        // [-W | Qs] hi, lo, e^{G_C} (the slot's first SLOT_IMG bytes)
constexpr uint32_t CS_KBP = SLOT_IMG;                 // Kb hi, lo, P hi, lo (SLOT_KBP bytes from SLOT_KH)
constexpr uint32_t CS_DO = CS_KBP + SLOT_KBP;         // dO^T hi | lo, MN-major [128 x][64 r]
constexpr uint32_t CS_BAR = CS_DO + 2 * D * C * 2;    // barriers, TMEM base
constexpr uint32_t CS_TOTAL = CS_BAR + 64;
static_assert(CS_KBP % 16 == 0 && CS_DO % 16 == 0 && CS_TOTAL <= 232448, "chain kernel shared memory");
static_assert(SLOT_KL == SLOT_KH + 16384 && SLOT_P == SLOT_KH + 32768, "Kb and P contiguous in the slot");
// tensor memory (columns)
constexpr uint32_t CT_S = 0;      // dS'^T fp32 [128 x][128 c]
constexpr uint32_t CT_SH = 128;   // dS'^T hi (bf16 pairs over c) [128 x][64]
constexpr uint32_t CT_SL = 192;   // its lo
constexpr uint32_t CT_U = 256;    // dU^T accumulator fp32 [128 x][64 r]
constexpr uint32_t CT_UH = 320;   // dU^T hi (bf16 pairs over r) [128 x][32]
constexpr uint32_t CT_UL = 352;   // its lo

__global__ void __launch_bounds__(kChainThreads, 1)
bwd_chain_kernel(const Plan pl, const float* __restrict__ dO, const float* __restrict__ dST,
                 float* __restrict__ dS0, float* __restrict__ dsp_out, float* __restrict__ du_out) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bar_ld = reinterpret_cast<uint64_t*>(smem + CS_BAR);
    uint64_t* bar_u = bar_ld + 1;
    uint64_t* bar_s = bar_ld + 2;
    uint64_t* bar_fin = bar_ld + 3;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(bar_ld + 4);
    uint64_t* bar_never = bar_ld + 5;   // testing: nothing arrives on it
    const Chain chn = chain_of(pl, blockIdx.x);
    const int H = pl.H, h = chn.h;
    const int64_t sbase = ((int64_t)chn.n * H + h) * D * D;
    if (warp == 0) tc::tmem_alloc(tmem_base_s, 512);
    if (tid == 0) {
        tc::bar_init(bar_ld, 1);
        tc::bar_init(bar_u, 1);
        tc::bar_init(bar_s, 1);
        tc::bar_init(bar_fin, 1);
        tc::bar_init(bar_never, 1);
        tc::bar_init_fence();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tmem_base_s;
    // thread -> TMEM lane x (value column) and a half of the columns
    const int x = (warp & 3) * 32 + lane, half = warp >> 2;
    const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;

    uint32_t ph_ld = 0, ph_u = 0, ph_s = 0;
    bool failed = false;
    bool inject = pl.inject == 3;
    auto wait = [&](uint64_t* bar, uint32_t& phase) {
        bool ok = true;
        if (tid == 0) ok = tc::bar_wait(inject ? bar_never : bar, inject ? 0u : phase, pl.wait_iter);
        inject = false;
        const bool gave_up = __syncthreads_or(!ok) != 0;
        if (!gave_up) phase ^= 1;
        failed = failed || gave_up;
        tc::fence_after();
        return !gave_up;
    };
    auto issue_loads = [&](int64_t i) {
        if (tid == 0) {
            const uint8_t* slot = pl.slots + ((chn.g0 + i) * H + h) * (int64_t)SLOT_BYTES;
            tc::bar_expect_tx(bar_ld, SLOT_IMG + SLOT_KBP);
            tc::bulk_load(smem + CS_IMG, slot, 32768, bar_ld);
            tc::bulk_load(smem + CS_IMG + 32768, slot + 32768, 32768, bar_ld);
            tc::bulk_load(smem + CS_IMG + 65536, slot + 65536, SLOT_IMG - 65536, bar_ld);
            tc::bulk_load(smem + CS_KBP, slot + SLOT_KH, 32768, bar_ld);
            tc::bulk_load(smem + CS_KBP + 32768, slot + SLOT_KH + 32768, SLOT_KBP - 32768, bar_ld);
        }
    };
    bool ld_pending = false;

    // dS'^T of the last chunk: the caller's dS_T (or zero), column x of dS_T [c][x]
    for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 16) {
        uint32_t v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(dST != nullptr ? dST[sbase + (int64_t)(c0 + e) * D + x] : 0.f);
        tc::tmem_st16(tm + lanes + CT_S + c0, v);
    }
    tc::tmem_st_wait();
    if (chn.nchunks > 0) {
        issue_loads(chn.nchunks - 1);
        ld_pending = true;
    }

    const uint32_t id_u1 = tc::idesc_bf16(128, C, false, true, true);     // A dO^T (MN), B P^T (MN)
    const uint32_t id_u2 = tc::idesc_bf16(128, C, false, true, false);    // A dS'^T (TMEM), B Kb^T (MN)
    const uint32_t id_s1 = tc::idesc_bf16(128, D, false, false, true);    // A dO^T (MN), B Qs^T (K-major)
    const uint32_t id_s2 = tc::idesc_bf16(128, D, false, false, false);   // A dU^T (TMEM), B (-W)^T (K-major)
    for (int64_t i = chn.nchunks - 1; i >= 0 && !failed; --i) {
        const int64_t c0t = chn.bos + i * C;
        const int L = (chn.eos - c0t < (int64_t)C) ? (int)(chn.eos - c0t) : C;
        const int64_t task = (chn.g0 + i) * H + h;
        // dO^T of the chunk as an MN-major image (rows past the sequence end are zero):
        // thread -> 8 rows r of 4 consecutive columns x, eight float4 in flight
        {
            uint8_t* hi = smem + CS_DO;
            uint8_t* lo = hi + D * C * 2;
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int idx = tid + u * kChainThreads;   // 2048 units of [64 r][32 x4]
                const int r = ((idx >> 8) << 3) | (idx & 7), xg = (idx >> 3) & 31;
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < L) v[u] = *reinterpret_cast<const float4*>(dO + ((c0t + r) * H + h) * D + 4 * xg);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int idx = tid + u * kChainThreads;
                const int r = ((idx >> 8) << 3) | (idx & 7), xg = (idx >> 3) & 31;
                uint2 hv, lv;
                tc::split2(v[u].x, v[u].y, hv.x, lv.x);
                tc::split2(v[u].z, v[u].w, hv.y, lv.y);
                const uint32_t o = op_off(4 * xg, r, C, true);
                *reinterpret_cast<uint2*>(hi + o) = hv;
                *reinterpret_cast<uint2*>(lo + o) = lv;
            }
        }
        if (!wait(bar_ld, ph_ld)) break;
        ld_pending = false;
        // dS': store it, split it, scale it by e^{G_C}
        {
            const float* egc = reinterpret_cast<const float*>(smem + CS_IMG + SLOT_EGC);
            float* dst = dsp_out + task * (int64_t)(D * D) + x;
            for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 16) {
                uint32_t v[16];
                tc::tmem_ld16(tm + lanes + CT_S + c0, v);
                tc::tmem_ld_wait();
                float f[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    f[e] = __uint_as_float(v[e]);
                    dst[(int64_t)(c0 + e) * D] = f[e];
                }
                uint32_t hv[8], lv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) tc::split2(f[2 * e], f[2 * e + 1], hv[e], lv[e]);
                tc::tmem_st8(tm + lanes + CT_SH + c0 / 2, hv);
                tc::tmem_st8(tm + lanes + CT_SL + c0 / 2, lv);
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(f[e] * egc[c0 + e]);
                tc::tmem_st16(tm + lanes + CT_S + c0, v);
            }
            tc::tmem_st_wait();
        }
        tc::fence_async_smem();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        // dU^T = dO^T (scale P)^T + dS'^T Kb^T
        if (warp == 0) {
            const uint32_t doh = tc::smem_u32(smem + CS_DO), dol = doh + D * C * 2;
            const uint32_t kbh = tc::smem_u32(smem + CS_KBP), kbl = kbh + 16384;
            const uint32_t phh = kbh + 32768, phl = kbh + 40960;
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks) {
                const uint64_t ah = tc::sdesc(doh + ks * 256, 128, C * 16), al = tc::sdesc(dol + ks * 256, 128, C * 16);
                const uint64_t bh = tc::sdesc(phh + ks * 2048, 1024, 128), bl = tc::sdesc(phl + ks * 2048, 1024, 128);
                tc::mma_ss_w(tm + CT_U, ah, bh, id_u1, ks > 0 ? 1u : 0u);
                tc::mma_ss_w(tm + CT_U, ah, bl, id_u1, 1u);
                tc::mma_ss_w(tm + CT_U, al, bh, id_u1, 1u);
            }
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t bh = tc::sdesc(kbh + ks * 2048, 1024, 128), bl = tc::sdesc(kbl + ks * 2048, 1024, 128);
                tc::mma_ts_w(tm + CT_U, tm + CT_SH + ks * 8, bh, id_u2, 1u);
                tc::mma_ts_w(tm + CT_U, tm + CT_SH + ks * 8, bl, id_u2, 1u);
                tc::mma_ts_w(tm + CT_U, tm + CT_SL + ks * 8, bh, id_u2, 1u);
            }
            tc::commit_w(bar_u);
        }
        if (!wait(bar_u, ph_u)) break;
        // dU: store it, split it
        {
            float* dst = du_out + task * (int64_t)(C * D) + x;
            for (int r0 = 32 * half; r0 < 32 * half + 32; r0 += 16) {
                uint32_t v[16];
                tc::tmem_ld16(tm + lanes + CT_U + r0, v);
                tc::tmem_ld_wait();
                float f[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    f[e] = __uint_as_float(v[e]);
                    dst[(int64_t)(r0 + e) * D] = f[e];
                }
                uint32_t hv[8], lv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) tc::split2(f[2 * e], f[2 * e + 1], hv[e], lv[e]);
                tc::tmem_st8(tm + lanes + CT_UH + r0 / 2, hv);
                tc::tmem_st8(tm + lanes + CT_UL + r0 / 2, lv);
            }
            tc::tmem_st_wait();
        }
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        // dS^T += dO^T Qs^T + dU^T (-W)^T
        if (warp == 0) {
            const uint32_t doh = tc::smem_u32(smem + CS_DO), dol = doh + D * C * 2;
            const uint32_t wh = tc::smem_u32(smem + CS_IMG + SLOT_WQH), wl = tc::smem_u32(smem + CS_IMG + SLOT_WQL);
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks) {
                const uint64_t ah = tc::sdesc(doh + ks * 256, 128, C * 16), al = tc::sdesc(dol + ks * 256, 128, C * 16);
                const uint64_t bh = tc::sdesc(wh + 16384 + ks * 4096, 2048, 128);
                const uint64_t bl = tc::sdesc(wl + 16384 + ks * 4096, 2048, 128);
                tc::mma_ss_w(tm + CT_S, ah, bh, id_s1, 1u);
                tc::mma_ss_w(tm + CT_S, ah, bl, id_s1, 1u);
                tc::mma_ss_w(tm + CT_S, al, bh, id_s1, 1u);
            }
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks) {
                const uint64_t bh = tc::sdesc(wh + ks * 4096, 2048, 128), bl = tc::sdesc(wl + ks * 4096, 2048, 128);
                tc::mma_ts_w(tm + CT_S, tm + CT_UH + ks * 8, bh, id_s2, 1u);
                tc::mma_ts_w(tm + CT_S, tm + CT_UH + ks * 8, bl, id_s2, 1u);
                tc::mma_ts_w(tm + CT_S, tm + CT_UL + ks * 8, bh, id_s2, 1u);
            }
            tc::commit_w(bar_s);
        }
        if (!wait(bar_s, ph_s)) break;
        // the slot buffers and dO^T are free: the previous chunk's loads
        if (i > 0) {
            issue_loads(i - 1);
            ld_pending = true;
        }
    }
    if (failed) {
        if (tid == 0) {
            report_timeout(pl);
            if (ld_pending) tc::bar_wait(bar_ld, ph_ld, 1u << 26);
        }
    } else if (dS0 != nullptr) {
        for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 16) {
            uint32_t v[16];
            tc::tmem_ld16(tm + lanes + CT_S + c0, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) dS0[sbase + (int64_t)(c0 + e) * D + x] = __uint_as_float(v[e]);
        }
    }
    // MMAs that a wait gave up on may still run: they complete before TMEM is released
    if (warp == 0) {
        tc::commit_w(bar_fin);
        if (lane == 0) tc::bar_wait(bar_fin, 0, 1u << 26);
        __syncwarp();
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, 512);
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
                 const float* __restrict__ states, const float* __restrict__ at, const float* __restrict__ uu,
                 const float* __restrict__ dsp, const float* __restrict__ du,
                 float* __restrict__ scratch, float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv,
                 float* __restrict__ dg, float* __restrict__ dbeta) {
    extern __shared__ __align__(16) uint8_t smem[];
    float* gsm = reinterpret_cast<float*>(smem);
    float* tot = reinterpret_cast<float*>(smem + BK_TOT);
    float* ptot = reinterpret_cast<float*>(smem + BK_PT);
    float* bs = reinterpret_cast<float*>(smem + BK_BETA);
    float* dec = reinterpret_cast<float*>(smem + BK_DEC);
    float* ec = reinterpret_cast<float*>(smem + BK_EC);
    uint64_t* bar_mma = reinterpret_cast<uint64_t*>(smem + BK_BAR);
    uint64_t* bar_fin = bar_mma + 1;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(bar_mma + 2);
    uint64_t* bar_never = bar_mma + 3;   // testing: nothing arrives on it
    const int tid = threadIdx.x;
    const int H = pl.H;
    if ((tid >> 5) == 0) tc::tmem_alloc(tmem_base_s, 512);
    if (tid == 0) {
        tc::bar_init(bar_mma, 1);
        tc::bar_init(bar_fin, 1);
        tc::bar_init(bar_never, 1);
        tc::bar_init_fence();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    Tc t{smem, *tmem_base_s, bar_mma, 0u, pl.wait_iter, false, bar_never, pl.inject == 4};
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
    float* DXQ = sc + SC_DXQ;
    float* DWU = sc + SC_DWU;    // [dW | dU] [64][256]
    float* DKB = sc + SC_DKB;
    float* DBKV = sc + SC_DBKV;  // [dBk | dBv] [64][256]
    float* GB = sc + SC_GB;
    float* GF = sc + SC_GF;
    float* GC = sc + SC_GC;
    float* DP = sc + SC_DP;
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
        const float* Am = at + task * (int64_t)(2 * MQ);   // A (strictly lower), from the forward
        const float* Tm = Am + MQ;                          // T, from the forward
        const float* U = uu + task * (int64_t)(C * D);     // U = U~ - W S, from the forward
        __syncthreads();   // the previous task is done with the scratch and the tables

        // ---- inputs (0 past the sequence end), dU, prefix products, -W ---------------
        // (every loop below has a fixed count per thread and is unrolled, so that its
        // loads are in flight together)
        constexpr int NKV = MR / 8 / kChunkThreads;
        uint4 kr[NKV], qr[NKV], vr[NKV];
#pragma unroll
        for (int it = 0; it < NKV; ++it) {
            const int u = tid + it * kChunkThreads;
            const int r = u >> 4, c = 8 * (u & 15);
            const int64_t ti = ((c0 + r) * H + h) * D + c;
            kr[it] = qr[it] = vr[it] = make_uint4(0u, 0u, 0u, 0u);
            if (r < L) {
                kr[it] = __ldcs(reinterpret_cast<const uint4*>(k + ti));
                qr[it] = __ldcs(reinterpret_cast<const uint4*>(q + ti));
                vr[it] = __ldcs(reinterpret_cast<const uint4*>(v + ti));
            }
        }
#pragma unroll
        for (int it = 0; it < NKV; ++it) {
            const int u = tid + it * kChunkThreads;
            const int r = u >> 4, c = 8 * (u & 15);
            float kx[8], qx[8], vx[8];
            tc::unpack8(kr[it], kx);
            tc::unpack8(qr[it], qx);
            tc::unpack8(vr[it], vx);
            const int o = r * D + c;
            *reinterpret_cast<float4*>(K_ + o) = make_float4(kx[0], kx[1], kx[2], kx[3]);
            *reinterpret_cast<float4*>(K_ + o + 4) = make_float4(kx[4], kx[5], kx[6], kx[7]);
            *reinterpret_cast<float4*>(Q_ + o) = make_float4(qx[0], qx[1], qx[2], qx[3]);
            *reinterpret_cast<float4*>(Q_ + o + 4) = make_float4(qx[4], qx[5], qx[6], qx[7]);
            *reinterpret_cast<float4*>(V_ + o) = make_float4(vx[0], vx[1], vx[2], vx[3]);
            *reinterpret_cast<float4*>(V_ + o + 4) = make_float4(vx[4], vx[5], vx[6], vx[7]);
        }
        {
            // (all loads first)
            constexpr int NI = MR / 4 / kChunkThreads;
            float4 xo[NI], xd[NI];
#pragma unroll
            for (int it = 0; it < NI; ++it) {
                const int u = tid + it * kChunkThreads;
                const int r = u >> 5, c = 4 * (u & 31);
                xo[it] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < L) xo[it] = __ldcs(reinterpret_cast<const float4*>(dO + ((c0 + r) * H + h) * D + c));
                xd[it] = *reinterpret_cast<const float4*>(DU + r * D + c);
            }
#pragma unroll
            for (int it = 0; it < NI; ++it) {
                const int u = tid + it * kChunkThreads;
                const int r = u >> 5, c = 4 * (u & 31);
                *reinterpret_cast<float4*>(DO_ + r * D + c) = xo[it];
                *reinterpret_cast<float4*>(DWU + r * 2 * D + D + c) = xd[it];
            }
        }
        if (tid < C) bs[tid] = tid < L ? ld_in(beta + (c0 + tid) * H + h) : 0.f;
        {
            // (the block's 16 gate values are loaded first, all in flight together)
            const int c = tid & 127, J = tid >> 7;
            float gv[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int r = 16 * J + u;
                gv[u] = r < L ? ld_in(g + ((c0 + r) * H + h) * D + c) : 0.f;
            }
            float run = 1.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                run *= 16 * J + u < L ? __expf(gv[u]) : 1.f;
                PRE[(16 * J + u) * D + c] = run;
            }
            tot[J * D + c] = run;
        }
        {
            constexpr int NI = 8 * D / kChunkThreads;
            uint4 wh[NI], wl[NI];
#pragma unroll
            for (int it = 0; it < NI; ++it) {
                const int u = tid + it * kChunkThreads;
                wh[it] = __ldcs(reinterpret_cast<const uint4*>(slot + SLOT_WQH + u * 16));
                wl[it] = __ldcs(reinterpret_cast<const uint4*>(slot + SLOT_WQL + u * 16));
            }
#pragma unroll
            for (int it = 0; it < NI; ++it) {
                const int u = tid + it * kChunkThreads;
                const int c = u & 127, ng = u >> 7;
                float a[8], b[8];
                tc::unpack8(wh[it], a);
                tc::unpack8(wl[it], b);
#pragma unroll
                for (int e = 0; e < 8; ++e) WN[(8 * ng + e) * D + c] = a[e] + b[e];
            }
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
        // derived operands: e^{G_r}, a e^{G_r - G_m(b(r))}
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
            *reinterpret_cast<float4*>(EA + r * D + c) = ea;
            *reinterpret_cast<float4*>(KL + r * D + c) = make_float4(kx.x * pr.x, kx.y * pr.y, kx.z * pr.z, kx.w * pr.w);
            *reinterpret_cast<float4*>(QL + r * D + c) = make_float4(qx.x * pr.x, qx.y * pr.y, qx.z * pr.z, qx.w * pr.w);
        }

        // ---- the products with S, dS', U (tensor-core rounds) ----------------------------
        // [dO; dU] [S; U]^T: scale dO S^T, dW = -dU S^T, scale dO U^T (dU U^T unused)
        tc_round<D + C, 1, false, false>(
            t, D, false,
            [&](uint8_t* hi, uint8_t* lo) {
                stage_op<C, D, true>(DO_, D, hi, lo, D, 0);
                stage_op<C, D, true, true>(DU, D, hi, lo, D, C);
            },
            [&](uint8_t* hi, uint8_t* lo, int) {
                stage_op<D, D, true>(S, D, hi, lo, D, 0);
                stage_op<C, D, true>(U, D, hi, lo, D, D);
            });
        if (t.failed) break;
        tc_epi<D + C, 1>(t, 2 * C, OneVariant{}, [&](int r, int c0, const float* x) {
            if (r < C) {
                if (c0 < D) put16(DXQ + r * D + c0, x, scale, false);
                else put16(DP + r * C + (c0 - D), x, scale, false);
            } else if (c0 < D) {
                put16(DWU + (r - C) * 2 * D + c0, x, -1.f, false);
            }
        });
        // U dS'^T
        tc_round<D, 1, false, false>(
            t, D, false,
            [&](uint8_t* hi, uint8_t* lo) { stage_op<C, D, true, true>(U, D, hi, lo, D, 0); zero_rows(hi, lo, D, C); },
            [&](uint8_t* hi, uint8_t* lo, int) { stage_op<D, D, true>(DSP, D, hi, lo, D, 0); });
        if (t.failed) break;
        tc_epi<D, 1>(t, C, OneVariant{}, [&](int r, int c0, const float* x) { put16(DKB + r * D + c0, x, 1.f, false); });
        {
            // dEC[c] = sum_x dS'[c][x] S[c][x]: four threads per channel, eight float4 each
            const int c = tid >> 2, part = tid & 3;
            float4 a4[8], b4[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                a4[i] = __ldcs(reinterpret_cast<const float4*>(DSP + c * D + part * 32 + 4 * i));
                b4[i] = __ldcs(reinterpret_cast<const float4*>(S + c * D + part * 32 + 4 * i));
            }
            float a = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) a += a4[i].x * b4[i].x + a4[i].y * b4[i].y + a4[i].z * b4[i].z + a4[i].w * b4[i].w;
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            if (part == 0) dec[c] = a;
        }
        for (int e = tid; e < MQ; e += kChunkThreads) {
            const int r = e >> 6, j = e & 63;
            if (j > r) DP[e] = 0.f;
        }
        // [dBk | dBv] = T^T [dW | dU];  dM = -T^T dT T^T with dT = [dW | dU] (Diag(beta)
        // [X | v])^T, and since T Diag(beta) [X | v] = [W | U~] (the forward's own
        // products):  dM = -[dBk | dBv] [W | U~]^T = dBk (-W)^T + dBv (-U~)^T
        tc_round<2 * D, 1, true, true>(
            t, C, false,
            [&](uint8_t* hi, uint8_t* lo) { stage_op<C, C, false, true>(Tm, C, hi, lo, C, 0); zero_rows(hi, lo, C, C); },
            [&](uint8_t* hi, uint8_t* lo, int) { stage_op<C, 2 * D, false>(DWU, 2 * D, hi, lo, C, 0); });
        if (t.failed) break;
        tc_epi<2 * D, 1>(t, C, OneVariant{},
                         [&](int r, int c0, const float* x) { put16(DBKV + r * 2 * D + c0, x, 1.f, false); });
        for (int hk = 0; hk < 2 && !t.failed; ++hk)
            tc_round<C, 1, false, false>(
                t, D, hk > 0,
                [&](uint8_t* hi, uint8_t* lo) {
                    stage_op<C, D, true>(DBKV + hk * D, 2 * D, hi, lo, D, 0);
                    zero_rows(hi, lo, D, C);
                },
                [&](uint8_t* hi, uint8_t* lo, int) {
                    if (hk == 0) stage_op<C, D, true>(WN, D, hi, lo, D, 0);
                    else stage_op<C, D, true, true>(reinterpret_cast<const float*>(slot + SLOT_UT), D, hi, lo, D, 0, 0, 0,
                                              Neg{});
                });
        if (t.failed) break;
        tc_epi<C, 1>(t, C, OneVariant{}, [&](int r, int c0, const float* x) { put16(DM + r * C + c0, x, 1.f, false); });
        for (int e = tid; e < MQ; e += kChunkThreads) {
            const int r = e >> 6, j = e & 63;
            DA[e] = j < r ? bs[r] * DM[e] : 0.f;
        }
        // dbeta = rowsum(dM A) + rowsum(dBk X) + rowsum(dBv v);  dv = Diag(beta) dBv
        // (eight threads per row, each over 8 contiguous j and 16 contiguous c)
        {
            const int r = tid >> 3, part = tid & 7;
            float m4[8], a4[8], xb[16], kx[16], ea[16], vb[16], vx[16];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                ld4(DM + r * C + 8 * part + 4 * i, m4 + 4 * i);
                ld4_once(Am + r * C + 8 * part + 4 * i, a4 + 4 * i);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = 16 * part + 4 * i;
                ld4(DBKV + r * 2 * D + c, xb + 4 * i);
                ld4(K_ + r * D + c, kx + 4 * i);
                ld4(EA + r * D + c, ea + 4 * i);
                ld4(DBKV + r * 2 * D + D + c, vb + 4 * i);
                ld4(V_ + r * D + c, vx + 4 * i);
            }
            float a = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) a += m4[i] * a4[i];
#pragma unroll
            for (int i = 0; i < 16; ++i) a += xb[i] * kx[i] * ea[i] + vb[i] * vx[i];
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            if (part == 0 && r < L) __stcs(dbeta + (c0 + r) * H + h, a);
        }
#pragma unroll
        for (int it = 0; it < MR / 4 / kChunkThreads; ++it) {
            const int u = tid + it * kChunkThreads;
            const int r = u >> 5, c = 4 * (u & 31);
            if (r < L) {
                const float4 x = *reinterpret_cast<const float4*>(DBKV + r * 2 * D + D + c);
                const float br = bs[r];
                __stcs(reinterpret_cast<float4*>(dv + ((c0 + r) * H + h) * D + c),
                       make_float4(br * x.x, br * x.y, br * x.z, br * x.w));
            }
        }
        // the gated back-products: GB = (dA k e^{G_m - G_j}) per row block, GF the same with
        // dP (both times e^{G_r - G_m} later); GC = the transposed ones with kL and qL (times
        // 1 / pre_j later)
        tc_round<D, 4, false, true>(
            t, C, false,
            [&](uint8_t* hi, uint8_t* lo) {
                stage_op<C, C, true>(DA, C, hi, lo, C, 0);
                stage_op<C, C, true>(DP, C, hi, lo, C, C);
            },
            [&](uint8_t* hi, uint8_t* lo, int b) {
                stage_op<C, D, false>(K_, D, hi, lo, C, 0, 0, 0, Krf{PRE, ptot, b});
            });
        if (t.failed) break;
        tc_epi<D, 4>(t, 2 * C, [](int r) { return (r & 63) >> 4; }, [&](int r, int c0, const float* x) {
            put16((r < C ? GB + r * D : GF + (r - C) * D) + c0, x, 1.f, false);
        });
        for (int part = 0; part < 2 && !t.failed; ++part)
            tc_round<D, 4, true, true>(
                t, C, part > 0,
                [&](uint8_t* hi, uint8_t* lo) {
                    stage_op<C, C, false>(part == 0 ? DA : DP, C, hi, lo, C, 0);
                    zero_rows(hi, lo, C, C);
                },
                [&](uint8_t* hi, uint8_t* lo, int b) {
                    stage_op<C, D, false>(part == 0 ? KL : QL, D, hi, lo, C, 0, 0, 0, Alp{ptot, b});
                });
        if (t.failed) break;
        tc_epi<D, 4>(t, C, [](int r) { return r >> 4; },
                     [&](int r, int c0, const float* x) { put16(GC + r * D + c0, x, 1.f, false); });

        // ---- dq, dk, dG ----------------------------------------------------------------------
        // (four consecutive channels per item, the items' loads unrolled together)
#pragma unroll 2
        for (int u = tid; u < MR / 4; u += kChunkThreads) {
            const int e = 4 * u, r = e >> 7, c = e & 127, B = r >> 4;
            float pr[4], ea[4], kk[4], qq[4], xb[4], gb[4], gc[4], dx[4], gf[4], kb[4], pt[4], t3[4];
            ld4(PRE + e, pr); ld4(EA + e, ea); ld4(K_ + e, kk); ld4(Q_ + e, qq);
            ld4(DBKV + r * 2 * D + c, xb); ld4(GB + e, gb); ld4(GC + e, gc); ld4(DXQ + e, dx);
            ld4(GF + e, gf); ld4(DKB + e, kb); ld4(ptot + (B * 4 + 3) * D + c, pt); ld4(tot + 3 * D + c, t3);
            const float br = bs[r];
            float dG[4], dKbKb[4], dqv[4], dkv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float kbf = pt[i] * t3[i] / pr[i];          // e^{G_C - G_r}
                const float dxe = br * xb[i] * ea[i] + gb[i] * pr[i];  // dX e^G
                const float dye = gc[i] / pr[i];                   // dY e^{-G}
                const float dqq = dx[i] * ea[i] + gf[i] * pr[i];      // dXq e^G
                dG[i] = kk[i] * dxe - kk[i] * dye + qq[i] * dqq - kb[i] * kk[i] * kbf;
                dKbKb[i] = kb[i] * kk[i] * kbf;
                dqv[i] = dqq;
                dkv[i] = dxe + dye + kb[i] * kbf;
            }
            *reinterpret_cast<float4*>(gsm + e) = make_float4(dG[0], dG[1], dG[2], dG[3]);
            *reinterpret_cast<float4*>(gsm + MR + e) = make_float4(dKbKb[0], dKbKb[1], dKbKb[2], dKbKb[3]);
            if (r < L) {
                const int64_t o = ((c0 + r) * H + h) * D + c;
                __stcs(reinterpret_cast<float4*>(dq + o), make_float4(dqv[0], dqv[1], dqv[2], dqv[3]));
                __stcs(reinterpret_cast<float4*>(dk + o), make_float4(dkv[0], dkv[1], dkv[2], dkv[3]));
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
                if (r < L) __stcs(dg + ((c0 + r) * H + h) * D + c, acc);
            }
        }
    }
    // a wait that gave up: report it; MMAs it left running complete before TMEM is released
    if (t.failed && tid == 0) report_timeout(pl);
    if ((tid >> 5) == 0) {
        tc::commit_w(bar_fin);
        if ((tid & 31) == 0) tc::bar_wait(bar_fin, 0, 1u << 26);
        __syncwarp();
    }
    tc::fence_before();
    __syncthreads();
    if ((tid >> 5) == 0) tc::tmem_dealloc(t.tm, 512);
}

// Workspace of the chunked backward: the forward's (bookkeeping and slots), o as
// bf16, then per (chunk slot, head) the entering state, A and T, U, dS' and dU,
// then the chunk kernel's per-CTA scratch.
struct BwdLayout {
    size_t fwd, o, states, at, u, dsp, du, scratch, total;
};
BwdLayout bwd_layout(int B, int T, int H, int N, bool packed) {
    BwdLayout l{};
    const int64_t cps = ((int64_t)T + C - 1) / C;
    const int64_t max_chunks = packed ? cps + N : (int64_t)B * cps;
    const size_t slots = (size_t)max_chunks * (size_t)H;
    l.fwd = (chunk_tc_workspace(B, T, H, N, packed) + 255) & ~size_t(255);
    l.o = (((size_t)B * (size_t)T * (size_t)H * D * 2) + 255) & ~size_t(255);
    l.states = slots * D * D * 4;
    l.at = slots * 2 * C * C * 4;
    l.u = slots * C * D * 4;
    l.dsp = l.states;
    l.du = slots * C * D * 4;
    l.scratch = (size_t)kBwdCtas * SC_TOTAL * 4;
    l.total = (int64_t)N * H == 0 ? 0 : l.fwd + l.o + l.states + l.at + l.u + l.dsp + l.du + l.scratch;
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
    float* at = reinterpret_cast<float*>(base + lo.fwd + lo.o + lo.states);
    float* uu = reinterpret_cast<float*>(base + lo.fwd + lo.o + lo.states + lo.at);
    float* dsp = reinterpret_cast<float*>(base + lo.fwd + lo.o + lo.states + lo.at + lo.u);
    float* du = reinterpret_cast<float*>(base + lo.fwd + lo.o + lo.states + lo.at + lo.u + lo.dsp);
    float* scratch = reinterpret_cast<float*>(base + lo.fwd + lo.o + lo.states + lo.at + lo.u + lo.dsp + lo.du);
    ChunkParams fp = p;
    fp.o = o;
    fp.final_state = nullptr;
    Plan pl{};
    cudaError_t e = chunk_tc_forward_states(fp, fwd, lo.fwd, states, at, uu, &pl, status, st);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CS_TOTAL);
    if (e != cudaSuccess) return e;
    bwd_chain_kernel<<<(unsigned)((int64_t)p.N * p.H), kChainThreads, CS_TOTAL, st>>>(pl, dO, dST, dS0, dsp, du);
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
            static_cast<const __nv_bfloat16*>(p.beta), p.scale, dO, states, at, uu, dsp, du, scratch,
            dq, dk, dv, dg, dbeta);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace kda
