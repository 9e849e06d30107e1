// Composition of segment transitions for context-parallel KDA.
//
// The recurrence is affine in the state: over a segment of tokens,
//     S_end = M S_start + S_zero,
// M = prod_t (I - beta_t k_t k_t^T) Diag(e^{g_t}) (later tokens on the left) and
// S_zero the segment's final state from a zero start.  Given every segment's
// (M_r, S_zero_r), the initial state of segment r + 1 is
//     S_in(r + 1) = M_r S_in(r) + S_zero_r,
// which this kernel evaluates for all heads at once: out[h] = M[h] S[h] + A[h]
// (K x K times K x V, fp32).  One CTA computes a 64 x 64 tile of one head with
// the two operands staged through shared memory in 32-deep slices; each thread
// holds a 4 x 4 block of the tile.
#include "kda_chunk.h"
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int TILE = 64, DEPTH = 32;

__global__ void __launch_bounds__(256)
state_compose_kernel(const float* __restrict__ M, const float* __restrict__ S, const float* A, float* out, int K,
                     int V) {
    __shared__ float Ms[DEPTH][TILE + 4];  // M tile, transposed: [j][row]
    __shared__ float Ss[DEPTH][TILE + 4];  // S tile: [j][col]
    const int tilesV = V / TILE;
    const int h = blockIdx.y;
    const int r0 = (blockIdx.x / tilesV) * TILE, c0 = (blockIdx.x % tilesV) * TILE;
    const int tid = threadIdx.x, tr = tid >> 4, tc = tid & 15;  // 16 x 16 threads, 4 x 4 each
    const float* Mh = M + (int64_t)h * K * K;
    const float* Sh = S + (int64_t)h * K * V;
    float acc[4][4] = {};
    for (int j0 = 0; j0 < K; j0 += DEPTH) {
        // 64 x 32 slice of M (rows r0.., columns j0..) and 32 x 64 slice of S
        for (int i = tid; i < TILE * DEPTH; i += 256) {
            const int r = i / DEPTH, j = i % DEPTH;
            Ms[j][r] = Mh[(int64_t)(r0 + r) * K + j0 + j];
            const int jj = i / TILE, c = i % TILE;
            Ss[jj][c] = Sh[(int64_t)(j0 + jj) * V + c0 + c];
        }
        __syncthreads();
#pragma unroll 8
        for (int j = 0; j < DEPTH; ++j) {
            float a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a[u] = Ms[j][tr * 4 + u];
                b[u] = Ss[j][tc * 4 + u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int w = 0; w < 4; ++w) acc[u][w] += a[u] * b[w];
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t row = (int64_t)h * K * V + (int64_t)(r0 + tr * 4 + u) * V + c0 + tc * 4;
#pragma unroll
        for (int w = 0; w < 4; ++w) out[row + w] = acc[u][w] + (A ? A[row + w] : 0.f);
    }
}

}  // namespace

cudaError_t state_compose(const float* M, const float* S, const float* A, float* out, int H, int K, int V,
                          cudaStream_t st) {
    if (H == 0) return cudaSuccess;
    const dim3 grid((unsigned)((K / TILE) * (V / TILE)), (unsigned)H);
    state_compose_kernel<<<grid, 256, 0, st>>>(M, S, A, out, K, V);
    return cudaGetLastError();
}

}  // namespace kda
