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
// delta rule.  Two kernels:
//
//   gate_proj_xa_kernel   one 128-token tile per CTA: [y | z] = x [f_a; b_proj]^T,
//                         K = D streamed through a 4-stage TMA -> tcgen05 pipeline
//                         (128-byte swizzled tiles), fp32 accumulator in TMEM; the
//                         epilogue writes y as bf16 hi|lo and beta = sigmoid(z).
//   gate_proj_fb_kernel   one 128-token x 256-channel tile per CTA:
//                         gate_x = y_hi f_b^T + y_lo f_b^T, stored by TMA.
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
constexpr int GK = 64;             // K elements per stage: one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kThreadsXA = 192;    // warp 0: TMA, warp 1: MMA, warps 2..5: epilogue
constexpr uint32_t kWaitDefault = 1u << 26;
constexpr uint32_t kTileA = GM * GK * 2;   // 16 KB

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}
__device__ __forceinline__ uint32_t lane_base(int warp) { return (uint32_t)((warp & 3) * 32) << 16; }
__device__ __forceinline__ void report(int32_t* status) {
    if (status != nullptr) *reinterpret_cast<volatile int32_t*>(status) = (int32_t)KDA_ERR_TIMEOUT;
}
__device__ __forceinline__ uint32_t stage_bytes_xa(int n1) {
    return kTileA + (((uint32_t)n1 * 128u + 1023u) & ~1023u);
}

// ---- [y | z] = x [f_a; b_proj]^T -------------------------------------------------
__global__ void __launch_bounds__(kThreadsXA, 1)
gate_proj_xa_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mfa,
                    const __grid_constant__ CUtensorMap mbp, int rows, int D, int R, int NH,
                    __nv_bfloat16* __restrict__ y_hi, __nv_bfloat16* __restrict__ y_lo,
                    __nv_bfloat16* __restrict__ beta, int32_t* status, uint32_t wait_iter) {
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
    const int nk = D / GK;

    if (warp == 0) tc::tmem_alloc(tmem_base_s, 256);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::bar_init(full + s, 1);
            tc::bar_init(empty + s, 1);
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
        int issued = 0;
        bool ok = true;
        if (lane == 0) {
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % kStages;
                if (kb >= kStages) {
                    // the MMAs that read this stage kStages blocks ago have completed
                    ok = tc::bar_wait_or_abort(empty + s, (uint32_t)(((kb / kStages) - 1) & 1), wait_iter, abort_s);
                    if (!ok) break;
                }
                uint8_t* a = smem + s * sbytes;
                uint8_t* b = a + kTileA;
                tc::bar_expect_tx(full + s, tx);
                tc::tma_load_2d(a, &mx, kb * GK, m0, full + s);
                tc::tma_load_2d(b, &mfa, kb * GK, 0, full + s);
                tc::tma_load_2d(b + R * 128, &mbp, kb * GK, 0, full + s);
                issued = kb + 1;
            }
            if (!ok) report(status);
            // every load issued has landed before the CTA exits (the last kStages
            // loads, one per stage; on the normal path they have long since landed)
            const int first = issued > kStages ? issued - kStages : 0;
            for (int kb = first; kb < issued; ++kb)
                tc::bar_wait(full + kb % kStages, (uint32_t)((kb / kStages) & 1), kWaitDefault);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issue -----------------------------------------------------------
        const uint32_t id = tc::idesc_bf16(GM, N1);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % kStages;
            ok = tc::bar_wait_or_abort(full + s, (uint32_t)((kb / kStages) & 1), wait_iter, abort_s);
            if (!ok) break;
            tc::fence_after();
            const uint32_t a = tc::smem_u32(smem + s * sbytes);
            const uint32_t b = a + kTileA;
#pragma unroll
            for (int kk = 0; kk < GK / 16; ++kk)
                tc::mma_ss_w(tm, tc::sdesc_sw128(a + 32 * kk), tc::sdesc_sw128(b + 32 * kk), id, (kb | kk) != 0);
            tc::commit_w(empty + s);
        }
        if (!ok && lane == 0) report(status);
        tc::commit_w(done);   // every MMA issued has completed
    } else {
        // ---- epilogue: y as bf16 hi|lo, beta = sigmoid(z) --------------------------
        const bool ok = tc::bar_wait_or_abort(done, 0, wait_iter, abort_s);
        tc::fence_after();
        if (!ok && lane == 0) report(status);
        const int r = (warp & 3) * 32 + lane;
        const int row = m0 + r;
        const bool have = ok && row < rows;
        for (int c = 0; c < N1; c += 16) {
            uint32_t a[16];
            tc::tmem_ld16(tm + lane_base(warp) + c, a);
            tc::tmem_ld_wait();
            if (!have) continue;
            if (c < R) {
                uint4 hi[2], lo[2];
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(a[j]);
                tc::split8(v, hi[0], lo[0]);
                tc::split8(v + 8, hi[1], lo[1]);
                uint4* ph = reinterpret_cast<uint4*>(y_hi + (int64_t)row * R + c);
                uint4* pl = reinterpret_cast<uint4*>(y_lo + (int64_t)row * R + c);
                ph[0] = hi[0]; ph[1] = hi[1];
                pl[0] = lo[0]; pl[1] = lo[1];
            } else {
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = 1.f / (1.f + __expf(-__uint_as_float(a[j])));
                uint4* pb = reinterpret_cast<uint4*>(beta + (int64_t)row * NH + (c - R));
                pb[0] = tc::pack8(v);
                pb[1] = tc::pack8(v + 8);
            }
        }
    }
    // (warp 1's final commit completes once every MMA it issued has)
    if (warp == 1 && lane == 0) tc::bar_wait(done, 0, kWaitDefault);
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, 256);
}

// ---- gate_x = (y_hi + y_lo) f_b^T ----------------------------------------------------
constexpr int GN2 = 256;                       // channels per tile
constexpr int kThreadsFB = 160;                // warp 0: TMA + MMA, warps 1..4: epilogue
// shared memory: A hi | A lo ([128][R] each, R/64 swizzle rows of 16 KB), B [256][R]
// (R/64 boxes of 32 KB); the output tile [128][256] bf16 (4 swizzled boxes of 16 KB)
// is staged over A once the MMAs are done.

__global__ void __launch_bounds__(kThreadsFB, 1)
gate_proj_fb_kernel(const __grid_constant__ CUtensorMap myh, const __grid_constant__ CUtensorMap myl,
                    const __grid_constant__ CUtensorMap mfb, const __grid_constant__ CUtensorMap mout, int rows,
                    int R, int32_t* status, uint32_t wait_iter) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = align1k(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int na = R / GK;                              // swizzle rows along K
    uint8_t* ah = smem;                                 // [na][128 x 64]
    uint8_t* al = ah + na * kTileA;
    uint8_t* bb = al + na * kTileA;                     // [na][256 x 64]
    uint64_t* loaded = reinterpret_cast<uint64_t*>(bb + na * (GN2 * GK * 2));
    uint64_t* done = loaded + 1;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_s = reinterpret_cast<volatile int*>(done + 2);
    const int m0 = blockIdx.x * GM, n0 = blockIdx.y * GN2;

    if (warp == 0) tc::tmem_alloc(tmem_base_s, 256);
    if (tid == 0) {
        tc::bar_init(loaded, 1);
        tc::bar_init(done, 1);
        *abort_s = 0;
        tc::bar_init_fence();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tmem_base_s;

    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            tc::bar_expect_tx(loaded, (uint32_t)na * (2 * kTileA + GN2 * GK * 2));
            for (int a = 0; a < na; ++a) {
                tc::tma_load_2d(ah + a * kTileA, &myh, a * GK, m0, loaded);
                tc::tma_load_2d(al + a * kTileA, &myl, a * GK, m0, loaded);
                tc::tma_load_2d(bb + a * (GN2 * GK * 2), &mfb, a * GK, n0, loaded);
            }
        }
        __syncwarp();
        ok = tc::bar_wait_or_abort(loaded, 0, wait_iter, abort_s);
        if (!ok) {
            // the copies still land before the CTA exits
            if (lane == 0) tc::bar_wait(loaded, 0, kWaitDefault);
            __syncwarp();
        }
        tc::fence_after();
        const uint32_t id = tc::idesc_bf16(GM, GN2);
        for (int a = 0; a < (ok ? na : 0); ++a) {
            const uint32_t h = tc::smem_u32(ah + a * kTileA), l = tc::smem_u32(al + a * kTileA);
            const uint32_t b = tc::smem_u32(bb + a * (GN2 * GK * 2));
#pragma unroll
            for (int kk = 0; kk < GK / 16; ++kk) {
                tc::mma_ss_w(tm, tc::sdesc_sw128(h + 32 * kk), tc::sdesc_sw128(b + 32 * kk), id, (a | kk) != 0);
                tc::mma_ss_w(tm, tc::sdesc_sw128(l + 32 * kk), tc::sdesc_sw128(b + 32 * kk), id, 1);
            }
        }
        tc::commit_w(done);
        if (!ok && lane == 0) report(status);
    } else {
        // epilogue: TMEM -> bf16 staged over A (4 boxes of [128][64], 128-byte swizzle)
        ok = tc::bar_wait_or_abort(done, 0, wait_iter, abort_s);
        tc::fence_after();
        if (!ok && lane == 0) report(status);
        const int r = (warp & 3) * 32 + lane;
        for (int c = 0; c < GN2; c += 16) {
            uint32_t a[16];
            tc::tmem_ld16(tm + lane_base(warp) + c, a);
            tc::tmem_ld_wait();
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(a[j]);
            uint8_t* box = smem + (c >> 6) * kTileA;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int ch = ((c & 63) >> 3) + h;   // 16-byte chunk within the 128-byte row
                *reinterpret_cast<uint4*>(box + r * 128 + ((ch ^ (r & 7)) << 4)) = tc::pack8(v + 8 * h);
            }
        }
        tc::fence_async_smem();
    }
    if (warp == 0 && lane == 0) tc::bar_wait(done, 0, kWaitDefault);   // MMAs done before the staging is read
    tc::fence_before();
    __syncthreads();
    if (tid == 0 && *abort_s == 0) {
        for (int b4 = 0; b4 < GN2 / GK; ++b4) tc::tma_store_2d(&mout, smem + b4 * kTileA, n0 + b4 * GK, m0);
        tc::bulk_commit();
        tc::bulk_wait();
    }
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, 256);
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

}  // namespace

bool gate_proj_supported(int D, int R, int HK, int NH) {
    return D > 0 && D % GK == 0 && (R == 64 || R == 128) && NH > 0 && NH % 16 == 0 && R + NH <= 256 &&
           HK > 0 && HK % GN2 == 0;
}

size_t gate_proj_workspace(int64_t rows, int R) { return (size_t)rows * (size_t)R * 2 * sizeof(__nv_bfloat16); }

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
    __nv_bfloat16* yh = reinterpret_cast<__nv_bfloat16*>(ws);
    __nv_bfloat16* yl = yh + rows * R;
    CUtensorMap mx, mfa, mbp, myh, myl, mfb, mout;
    if (!map2d(&mx, x, rows, D, GM) || !map2d(&mfa, f_a, R, D, R) || !map2d(&mbp, b_proj, NH, D, NH) ||
        !map2d(&myh, yh, rows, R, GM) || !map2d(&myl, yl, rows, R, GM) || !map2d(&mfb, f_b, HK, R, GN2) ||
        !map2d(&mout, gate_x, rows, HK, GM))
        return cudaErrorInvalidValue;
    const unsigned mt = (unsigned)((rows + GM - 1) / GM);
    {
        const int n1 = R + NH;
        const uint32_t sbytes = kTileA + (((uint32_t)n1 * 128u + 1023u) & ~1023u);
        const int smem = (int)(kStages * sbytes + 256 + 1024);
        e = cudaFuncSetAttribute(gate_proj_xa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        gate_proj_xa_kernel<<<mt, kThreadsXA, smem, st>>>(mx, mfa, mbp, (int)rows, D, R, NH, yh, yl,
                                                          reinterpret_cast<__nv_bfloat16*>(beta), status, wait_iter);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        const int na = R / GK;
        const int smem = (int)(na * (2 * kTileA + GN2 * GK * 2) + 256 + 1024);
        e = cudaFuncSetAttribute(gate_proj_fb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        dim3 grid(mt, (unsigned)(HK / GN2));
        gate_proj_fb_kernel<<<grid, kThreadsFB, smem, st>>>(myh, myl, mfb, mout, (int)rows, R, status, wait_iter);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace kda
