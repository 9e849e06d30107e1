// Projections ahead of the gate on the sm_103a tensor cores ("kimi-k3-mlx"
// review, "Attention is 93 layers ...": a low-rank forget gate through f_a and
// f_b; "The A_log shape mismatch ...": b_proj is [96, H], H = 7168).  Per
// token x_t (a row of D bf16 values):
//
//     y_t      = f_a x_t                       f_a    [R, D]   (fp32, kept as bf16 hi + lo)
//     gate_x_t = f_b y_t                       f_b    [HK, R]
//     beta_t   = sigmoid(b_proj x_t)           b_proj [NH, D]
//
// gate_x and beta are the bf16 inputs of the fused prefill's gate and of its
// delta rule.  Three kernels:
//
//   gate_proj_xa_kernel      [y | z] = x [f_a; b_proj]^T for one 128-token tile and
//                            one of S ranges of D (split K, so that a few thousand
//                            tokens still fill the GPU): a 4-stage TMA -> tcgen05
//                            pipeline of 128-byte swizzled tiles, fp32 accumulator in
//                            TMEM, the partial sums stored column by column.
//   gate_proj_finish_kernel  sums the S partials in a fixed order (the result does not
//                            depend on scheduling), writes y as bf16 hi|lo rows and
//                            beta = sigmoid(z) (R and NH are multiples of 16).
//   gate_proj_fb_kernel      gate_x = y_hi f_b^T + y_lo f_b^T: one CTA per 128-token
//                            tile and run of 128-channel tiles, y resident in shared
//                            memory, f_b tiles double-buffered, two TMEM accumulators
//                            and two output stagings so that the loads, MMAs, epilogue
//                            and TMA stores of consecutive tiles overlap.
//
// Every wait is bounded; a wait that gives up records KDA_ERR_TIMEOUT in the
// status word (when one is given), and the kernel drains what it has in flight.
#include <cuda.h>

#include "kda_chunk.h"
#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int GM = 128;            // tokens per tile (TMEM lanes)
constexpr int GK = 64;             // K elements per 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kThreads = 192;      // warp 0: TMA, warp 1: MMA, warps 2..5: epilogue
constexpr int kThreadsFB = 320;    // the second product: warps 2..9 share the epilogue
constexpr uint32_t kWaitDefault = 1u << 26;
constexpr uint32_t kTileA = GM * GK * 2;   // 16 KB: [128 rows][64] bf16
constexpr int kMaxSplit = 8;
constexpr int GN2 = 128;           // channels per tile of the second product
constexpr int kRingB = 3;          // f_b tiles in flight in the second product
constexpr int kFinRows = 32;       // tokens per CTA of the finishing kernel
constexpr int kFinCols = 16;       // columns of [y | z] per CTA of the finishing kernel
constexpr int kThreadsFin = 256;

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}
__device__ __forceinline__ uint32_t lane_base(int warp) { return (uint32_t)((warp & 3) * 32) << 16; }
__device__ __forceinline__ void report(int32_t* status) {
    if (status != nullptr) *reinterpret_cast<volatile int32_t*>(status) = (int32_t)KDA_ERR_TIMEOUT;
}
__host__ __device__ __forceinline__ uint32_t stage_bytes_xa(int n1) {
    return kTileA + (((uint32_t)n1 * 128u + 1023u) & ~1023u);
}

// ---- partial [y | z] = x [f_a; b_proj]^T over the K blocks of range blockIdx.y -------
// part[s][j][row] fp32 (for each column j the 32 lanes of a warp store 32 consecutive rows).
__global__ void __launch_bounds__(kThreads, 1)
gate_proj_xa_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mfa,
                    const __grid_constant__ CUtensorMap mbp, int rows, int nk, int nk_per, int R, int NH,
                    float* __restrict__ part, int32_t* status, uint32_t wait_iter) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = align1k(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int N1 = R + NH;
    const uint32_t sbytes = stage_bytes_xa(N1);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * sbytes);
    uint64_t* empty = full + kStages;
    uint64_t* done = empty + kStages;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_s = reinterpret_cast<volatile int*>(done + 2);
    const int m0 = blockIdx.x * GM;
    const int s = blockIdx.y;
    const int kb0 = s * nk_per;
    const int nkb = min(nk, kb0 + nk_per) - kb0;   // >= 1: the host leaves no range empty
    tc::grid_dep_launch();   // (the finishing kernel waits for this grid before it reads)

    if (warp == 0) tc::tmem_alloc(tmem_base_s, 256);
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::bar_init(full + i, 1);
            tc::bar_init(empty + i, 1);
        }
        tc::bar_init(done, 1);
        *abort_s = 0;
        tc::bar_init_fence();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tmem_base_s;
    const uint32_t tx = kTileA + (uint32_t)N1 * 128u;

    if (warp == 0) {
        // ---- TMA producer --------------------------------------------------------
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < nkb; ++i) {
                const int st = i % kStages;
                if (i >= kStages) {
                    // the MMAs that read this stage kStages blocks ago have completed
                    ok = tc::bar_wait_or_abort(empty + st, (uint32_t)(((i / kStages) - 1) & 1), wait_iter, abort_s);
                    if (!ok) break;
                }
                uint8_t* a = smem + st * sbytes;
                uint8_t* b = a + kTileA;
                const int k = (kb0 + i) * GK;
                tc::bar_expect_tx(full + st, tx);
                tc::tma_load_2d(a, &mx, k, m0, full + st);
                tc::tma_load_2d(b, &mfa, k, 0, full + st);
                tc::tma_load_2d(b + R * 128, &mbp, k, 0, full + st);
                issued = i + 1;
            }
            if (!ok) report(status);
            // every load issued lands before the CTA exits (the last kStages, one per
            // stage; on the normal path they have long since landed)
            for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
                tc::bar_wait(full + i % kStages, (uint32_t)((i / kStages) & 1), kWaitDefault);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issue -----------------------------------------------------------
        const uint32_t id = tc::idesc_bf16(GM, N1);
        bool ok = true;
        for (int i = 0; i < nkb; ++i) {
            const int st = i % kStages;
            ok = tc::bar_wait_or_abort(full + st, (uint32_t)((i / kStages) & 1), wait_iter, abort_s);
            if (!ok) break;
            tc::fence_after();
            const uint32_t a = tc::smem_u32(smem + st * sbytes);
            const uint32_t b = a + kTileA;
#pragma unroll
            for (int kk = 0; kk < GK / 16; ++kk)
                tc::mma_ss_w(tm, tc::sdesc_sw128(a + 32 * kk), tc::sdesc_sw128(b + 32 * kk), id, (i | kk) != 0);
            tc::commit_w(empty + st);
        }
        if (!ok && lane == 0) report(status);
        tc::commit_w(done);   // completes once every MMA issued has
    } else {
        // ---- epilogue: the partial sums, column by column -------------------------
        const bool ok = tc::bar_wait_or_abort(done, 0, wait_iter, abort_s);
        tc::fence_after();
        if (!ok && lane == 0) report(status);
        const int row = m0 + (warp & 3) * 32 + lane;
        const bool have = ok && row < rows;
        float* ps = part + (int64_t)s * N1 * rows + row;
        for (int c = 0; c < N1; c += 16) {
            uint32_t a[16];
            tc::tmem_ld16(tm + lane_base(warp) + c, a);
            tc::tmem_ld_wait();
            if (have) {
#pragma unroll
                for (int j = 0; j < 16; ++j) ps[(int64_t)(c + j) * rows] = __uint_as_float(a[j]);
            }
        }
    }
    if (warp == 1 && lane == 0) tc::bar_wait(done, 0, kWaitDefault);   // every MMA has completed
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, 256);
}

// ---- y = sum_s part[s] (in order s = 0, 1, ...) as bf16 hi|lo rows; beta = sigmoid(z) ----
// One CTA per 32 tokens x 16 columns: every warp requests the S partials of its two
// columns at once (the ranges past S add zeros, which leaves the sums unchanged), the
// sums meet in shared memory, and the rows leave as 16-byte pieces.
__global__ void __launch_bounds__(kThreadsFin)
gate_proj_finish_kernel(const float* __restrict__ part, int S, int rows, int R, int NH,
                        __nv_bfloat16* __restrict__ y_hi, __nv_bfloat16* __restrict__ y_lo,
                        __nv_bfloat16* __restrict__ beta) {
    __shared__ float tile[kFinCols][kFinRows + 1];
    const int N1 = R + NH;
    const int r0 = blockIdx.x * kFinRows, j0 = blockIdx.y * kFinCols;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int row = r0 + lane;
    constexpr int kCols = kFinCols / (kThreadsFin / 32);   // columns per warp
    tc::grid_dep_launch();   // (the second product waits for this grid before it reads y)
    tc::grid_dep_wait();     // the partial sums are complete
    float v[kCols][kMaxSplit];
#pragma unroll
    for (int q = 0; q < kCols; ++q) {
        const float* p = part + (int64_t)(j0 + w * kCols + q) * rows + row;
#pragma unroll
        for (int s = 0; s < kMaxSplit; ++s) v[q][s] = (row < rows && s < S) ? p[(int64_t)s * N1 * rows] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kCols; ++q) {
        float acc = v[q][0];
#pragma unroll
        for (int s = 1; s < kMaxSplit; ++s) acc += v[q][s];
        tile[w * kCols + q][lane] = acc;
    }
    __syncthreads();
    // (8 consecutive columns, one row) per thread: 32 rows x 2 groups
    if (threadIdx.x < kFinRows * (kFinCols / 8)) {
        const int r = threadIdx.x % kFinRows, jg = threadIdx.x / kFinRows;
        if (r0 + r >= rows) return;
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = tile[8 * jg + u][r];
        const int64_t gr = r0 + r;
        const int j = j0 + 8 * jg;
        if (j < R) {
            uint4 hi, lo;
            tc::split8(x, hi, lo);
            *reinterpret_cast<uint4*>(y_hi + gr * R + j) = hi;
            *reinterpret_cast<uint4*>(y_lo + gr * R + j) = lo;
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = 1.f / (1.f + __expf(-x[u]));
            *reinterpret_cast<uint4*>(beta + gr * NH + (j - R)) = tc::pack8(x);
        }
    }
}

// ---- gate_x = (y_hi + y_lo) f_b^T ----------------------------------------------------
// One CTA: the 128-token tile blockIdx.x and the channel tiles [t0, t0 + nt) of GN2 each.
// Shared memory: A hi | A lo ([128][R] each: R/64 swizzle atoms of 16 KB), a ring of
// kRingB f_b tiles ([128][R]), two output stagings ([128][128] bf16 as two 16 KB atoms).
__host__ __device__ __forceinline__ uint32_t fb_smem_bytes(int R) {
    return (uint32_t)(R / GK) * kTileA * 2 + (uint32_t)kRingB * (uint32_t)(R / GK) * kTileA + 2u * 2u * kTileA;
}

__global__ void __launch_bounds__(kThreadsFB, 1)
gate_proj_fb_kernel(const __grid_constant__ CUtensorMap myh, const __grid_constant__ CUtensorMap myl,
                    const __grid_constant__ CUtensorMap mfb, const __grid_constant__ CUtensorMap mout, int R,
                    int ntiles, int per_cta, int32_t* status, uint32_t wait_iter) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = align1k(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int na = R / GK;
    uint8_t* ah = smem;
    uint8_t* al = ah + na * kTileA;
    uint8_t* bring = al + na * kTileA;              // [kRingB stages][na][16 KB]
    uint8_t* ostg = bring + kRingB * na * kTileA;   // [2][2 atoms][16 KB]
    uint64_t* a_full = reinterpret_cast<uint64_t*>(ostg + 4 * kTileA);
    uint64_t* b_full = a_full + 1;              // [kRingB]
    uint64_t* b_empty = b_full + kRingB;        // [kRingB]
    uint64_t* t_full = b_empty + kRingB;        // [2]
    uint64_t* t_empty = t_full + 2;             // [2]
    uint64_t* fin = t_empty + 2;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort_s = reinterpret_cast<volatile int*>(fin + 2);
    const int m0 = blockIdx.x * GM;
    const int t0 = blockIdx.y * per_cta;
    const int nt = min(per_cta, ntiles - t0);   // >= 1: the host leaves no CTA empty

    if (warp == 0) tc::tmem_alloc(tmem_base_s, 2 * GN2);
    if (tid == 0) {
        tc::bar_init(a_full, 1);
        for (int i = 0; i < kRingB; ++i) {
            tc::bar_init(b_full + i, 1);
            tc::bar_init(b_empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::bar_init(t_full + i, 1);
            tc::bar_init(t_empty + i, 8);   // one arrival per epilogue warp
        }
        tc::bar_init(fin, 1);
        *abort_s = 0;
        tc::bar_init_fence();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tmem_base_s;
    auto wait = [&](uint64_t* bar, uint32_t parity) { return tc::bar_wait_or_abort(bar, parity, wait_iter, abort_s); };

    if (warp == 0) {
        // ---- TMA producer: the first f_b tiles, then y hi|lo once the kernel that
        //      writes it has completed, then the rest of the f_b tiles through the ring
        if (lane == 0) {
            bool y_issued = false;
            auto issue_y = [&]() {
                tc::grid_dep_wait();
                tc::bar_expect_tx(a_full, 2u * na * kTileA);
                for (int a = 0; a < na; ++a) {
                    tc::tma_load_2d(ah + a * kTileA, &myh, a * GK, m0, a_full);
                    tc::tma_load_2d(al + a * kTileA, &myl, a * GK, m0, a_full);
                }
                y_issued = true;
            };
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < nt; ++i) {
                const int st = i % kRingB;
                if (i >= kRingB) {
                    if (!y_issued) issue_y();
                    ok = wait(b_empty + st, (uint32_t)(((i / kRingB) - 1) & 1));
                    if (!ok) break;
                }
                tc::bar_expect_tx(b_full + st, (uint32_t)na * kTileA);
                for (int a = 0; a < na; ++a)
                    tc::tma_load_2d(bring + (st * na + a) * kTileA, &mfb, a * GK, (t0 + i) * GN2, b_full + st);
                issued = i + 1;
            }
            if (!y_issued) issue_y();
            if (!ok) report(status);
            // every load issued lands before the CTA exits
            tc::bar_wait(a_full, 0, kWaitDefault);
            for (int i = issued > kRingB ? issued - kRingB : 0; i < issued; ++i)
                tc::bar_wait(b_full + i % kRingB, (uint32_t)((i / kRingB) & 1), kWaitDefault);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issue: tile i into TMEM columns (i % 2) * GN2 ---------------------
        const uint32_t id = tc::idesc_bf16(GM, GN2);
        bool ok = wait(a_full, 0);
        for (int i = 0; ok && i < nt; ++i) {
            const int b = i & 1, st = i % kRingB;
            ok = wait(b_full + st, (uint32_t)((i / kRingB) & 1));
            if (!ok) break;
            if (i >= 2) {
                // the epilogue has read this accumulator's previous tile
                ok = wait(t_empty + b, (uint32_t)(((i >> 1) - 1) & 1));
                if (!ok) break;
            }
            tc::fence_after();
            const uint32_t d = tm + (uint32_t)(b * GN2);
            const uint32_t hb = tc::smem_u32(ah), lb = tc::smem_u32(al);
            const uint32_t bb = tc::smem_u32(bring + st * na * kTileA);
            for (int a = 0; a < na; ++a) {
#pragma unroll
                for (int kk = 0; kk < GK / 16; ++kk) {
                    const uint32_t off = a * kTileA + 32 * kk;
                    const uint64_t bd = tc::sdesc_sw128(bb + off);
                    tc::mma_ss_w(d, tc::sdesc_sw128(hb + off), bd, id, (a | kk) != 0);
                    tc::mma_ss_w(d, tc::sdesc_sw128(lb + off), bd, id, 1);
                }
            }
            tc::commit_w(b_empty + st);  // the f_b stage is free once these MMAs are done
            tc::commit_w(t_full + b);    // and the accumulator is ready
        }
        if (!ok && lane == 0) report(status);
        tc::commit_w(fin);
        if (lane == 0) tc::bar_wait(fin, 0, kWaitDefault);   // every MMA issued has completed
        __syncwarp();
    } else {
        // ---- epilogue: TMEM -> bf16 staging (128-byte swizzle) -> two TMA stores;
        //      warp w reads TMEM lanes 32 (w % 4).. and the 64 columns of staging atom
        //      (w - 2) / 4 ---------------------------------------------------------
        const int et = tid - 64;                 // 0..255
        const int r = (warp & 3) * 32 + lane;    // the row this thread's TMEM lane holds
        const int c0 = ((warp - 2) >> 2) * GK;
        for (int i = 0; i < nt; ++i) {
            const int b = i & 1;
            // staging b is free once the stores of tile i - 2 have read it
            if (et == 0) tc::bulk_wait_read_1();
            const bool ok = wait(t_full + b, (uint32_t)((i >> 1) & 1));
            if (tc::named_any(1, kThreadsFB - 64, !ok)) {
                if (et == 0) report(status);
                break;
            }
            tc::fence_after();
            uint8_t* stg = ostg + b * 2 * kTileA;
            for (int c = c0; c < c0 + GK; c += 16) {
                uint32_t a[16];
                tc::tmem_ld16(tm + lane_base(warp) + (uint32_t)(b * GN2 + c), a);
                tc::tmem_ld_wait();
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(a[j]);
                uint8_t* box = stg + (c >> 6) * kTileA;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int ch = ((c & 63) >> 3) + h;   // 16-byte chunk within the 128-byte row
                    *reinterpret_cast<uint4*>(box + r * 128 + ((ch ^ (r & 7)) << 4)) = tc::pack8(v + 8 * h);
                }
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::bar_arrive(t_empty + b);
            tc::fence_async_smem();
            tc::named_sync(1, kThreadsFB - 64);
            if (et == 0) {
                tc::tma_store_2d(&mout, stg, (t0 + i) * GN2, m0);
                tc::tma_store_2d(&mout, stg + kTileA, (t0 + i) * GN2 + GK, m0);
                tc::bulk_commit();
            }
        }
        if (et == 0) tc::bulk_wait();
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, 2 * GN2);
}

// ---- host side -----------------------------------------------------------------------
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

// [rows][cols] bf16, box = box_rows x 64 columns, 128-byte swizzle
bool map2d(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)GK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

// Number of K ranges of the first product: enough 128-token tiles x ranges to
// cover about 128 SMs, at most 8 and at most one per 64-wide K block (a fixed
// function of the sizes, so that the workspace query needs no device), then
// made exact so that no range is empty.
int split_for(int64_t rows, int D) {
    const int64_t mt = (rows + GM - 1) / GM;
    const int nk = D / GK;
    int64_t s = mt > 0 ? 128 / mt : 1;
    if (s < 1) s = 1;
    if (s > kMaxSplit) s = kMaxSplit;
    if (s > nk) s = nk;
    const int nk_per = (nk + (int)s - 1) / (int)s;
    return (nk + nk_per - 1) / nk_per;
}

}  // namespace

bool gate_proj_supported(int D, int R, int HK, int NH) {
    return D > 0 && D % GK == 0 && (R == 64 || R == 128) && NH > 0 && NH % 16 == 0 && R + NH <= 256 &&
           HK > 0 && HK % GN2 == 0;
}

size_t gate_proj_workspace(int64_t rows, int D, int R, int NH) {
    if (rows <= 0 || D <= 0 || D % GK != 0) return 0;
    const size_t y = (size_t)rows * (size_t)R * 2 * sizeof(__nv_bfloat16);
    const size_t parts = (size_t)split_for(rows, D) * (size_t)(R + NH) * (size_t)rows * sizeof(float);
    return y + parts;
}

cudaError_t gate_proj(const void* x, const void* f_a, const void* f_b, const void* b_proj, int64_t rows, int D,
                      int R, int HK, int NH, void* gate_x, void* beta, void* ws, int32_t* status,
                      cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    if (status != nullptr) {
        e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
        if (e != cudaSuccess) return e;
    }
    if (rows == 0) return cudaSuccess;
    const uint32_t lim = wait_limit();
    const uint32_t wait_iter = lim != 0 ? lim : kWaitDefault;
    const int N1 = R + NH;
    const int S = split_for(rows, D);
    const int nk = D / GK;
    const int nk_per = (nk + S - 1) / S;
    __nv_bfloat16* yh = reinterpret_cast<__nv_bfloat16*>(ws);
    __nv_bfloat16* yl = yh + rows * R;
    float* part = reinterpret_cast<float*>(yl + rows * R);
    CUtensorMap mx, mfa, mbp, myh, myl, mfb, mout;
    if (!map2d(&mx, x, rows, D, GM) || !map2d(&mfa, f_a, R, D, R) || !map2d(&mbp, b_proj, NH, D, NH) ||
        !map2d(&myh, yh, rows, R, GM) || !map2d(&myl, yl, rows, R, GM) || !map2d(&mfb, f_b, HK, R, GN2) ||
        !map2d(&mout, gate_x, rows, HK, GM))
        return cudaErrorInvalidValue;
    const unsigned mt = (unsigned)((rows + GM - 1) / GM);
    {
        const int smem = (int)(kStages * stage_bytes_xa(N1) + 256 + 1024);
        e = cudaFuncSetAttribute(gate_proj_xa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        gate_proj_xa_kernel<<<dim3(mt, (unsigned)S), kThreads, smem, st>>>(mx, mfa, mbp, (int)rows, nk, nk_per, R,
                                                                           NH, part, status, wait_iter);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        const dim3 grid((unsigned)((rows + kFinRows - 1) / kFinRows), (unsigned)(N1 / kFinCols));
        e = tc::launch_dependent(gate_proj_finish_kernel, grid, dim3(kThreadsFin), 0, st, (const float*)part, S,
                             (int)rows, R, NH, yh, yl, reinterpret_cast<__nv_bfloat16*>(beta));
        if (e != cudaSuccess) return e;
    }
    {
        const int ntiles = HK / GN2;
        int ng = device_sms() / (int)mt;       // CTAs per token tile: about one wave in all
        if (ng < 1) ng = 1;
        if (ng > ntiles) ng = ntiles;
        const int per_cta = (ntiles + ng - 1) / ng;
        ng = (ntiles + per_cta - 1) / per_cta;  // no CTA without a tile
        const int smem = (int)(fb_smem_bytes(R) + 128 + 1024);
        static_assert(2 * 2 * kTileA + kRingB * 2 * kTileA + 2 * 2 * kTileA + 128 + 1024 <= 232448,
                      "shared memory of the second product");
        e = cudaFuncSetAttribute(gate_proj_fb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        e = tc::launch_dependent(gate_proj_fb_kernel, dim3(mt, (unsigned)ng), dim3(kThreadsFB), (size_t)smem, st, myh, myl,
                             mfb, mout, R, ntiles, per_cta, status, wait_iter);
    }
    return e;
}

}  // namespace kda
