// Parameters and launchers of the KDA prefill and decode kernels (internal to
// libkda.so; the public surface is include/kda.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

struct ChunkParams {
    // Direct inputs, or the raw prologue inputs (q_raw, k_raw, v_raw, gate_x).
    const void* q;
    const void* k;
    const void* v;
    const void* g;
    const void* beta;
    float scale;
    const float* initial_state;
    const int32_t* cu_seqlens;
    int B, T, H, N;
    void* o;
    float* final_state;
    // Prologue (only read by the fused variants).
    const float* conv_q;
    const float* conv_k;
    const float* conv_v;
    int conv_act;
    const float* A_log;
    const float* dt_bias;
    float lower_bound;
    float l2_eps;
};

// CUDA-core fp32 chunk kernel (any supported K/V, fp32 or bf16 inputs).
cudaError_t chunk_simt(kda_dtype in_dt, kda_dtype out_dt, int K, int V, bool prologue,
                       const ChunkParams& p, cudaStream_t st);

// Tensor-core chunk kernels (bf16 inputs, K = V = 128): the workspace bytes a
// call needs, and the launch with a caller-owned workspace (cudaErrorMemoryAllocation
// before anything is enqueued if ws_bytes is too small).  status (device, may be
// null) is set to KDA_OK on the stream and to KDA_ERR_TIMEOUT by a kernel whose
// bounded wait gave up.
bool chunk_tc_supported(kda_dtype in_dt, int K, int V);
size_t chunk_tc_workspace(int B, int T, int H, int N, bool packed);
cudaError_t chunk_tc(kda_dtype out_dt, const ChunkParams& p, void* ws, size_t ws_bytes, int32_t* status,
                     cudaStream_t st);
// With the input prologue (p.q, p.k, p.v, p.g are the raw inputs).
cudaError_t chunk_tc_fused(kda_dtype out_dt, const ChunkParams& p, void* ws, size_t ws_bytes, int32_t* status,
                           cudaStream_t st);

// The same with the workspace in a fixed device array of kFixedScratchBytes
// (no allocation); cudaErrorMemoryAllocation, before anything is enqueued,
// when the call needs more.
constexpr size_t kFixedScratchBytes = (size_t)64 << 20;
cudaError_t chunk_tc_fixed_scratch(kda_dtype out_dt, const ChunkParams& p, cudaStream_t st);

// Polls before a bounded device-side wait of the tensor-core prefill gives up
// (0 = the default, about a second); read at each launch.
void set_wait_limit(uint32_t iterations);
// The current setting (0 = the default).
uint32_t wait_limit();
// Testing: the next tensor-core prefill call on this host thread makes the
// first wait of its chunk-local (1) or state (2) kernel one on an mbarrier that
// nothing arrives on, so that it gives up; the call consumes the setting.
void inject_wait_timeout(int kernel);

// Events that the next tensor-core prefill call made on this host thread
// records: before its first kernel, after the chunk-local kernel, after its
// last kernel (any may be null); the call consumes them.
void trace_set(void* begin, void* split, void* end);

// Single-token decode.
cudaError_t decode_step(kda_dtype in_dt, kda_dtype out_dt, int K, int V, const void* q,
                        const void* k, const void* v, const void* g, const void* beta,
                        float scale, float* state, int N, int H, void* o, cudaStream_t st);

// Output gate: out = o / sqrt(mean_V(o^2) + eps) * w * sigmoid(gate), rows of V.
cudaError_t output_gate(kda_dtype gate_dt, kda_dtype out_dt, int V, const float* o, const void* gate,
                        const float* w, float eps, int64_t rows, void* out, cudaStream_t st);

// Projections ahead of the gate: gate_x = f_b (f_a x), beta = sigmoid(b_proj x),
// bf16 in and out; ws (gate_proj_workspace bytes) holds the split-K partial sums of
// f_a x and b_proj x and y = f_a x as a bf16 hi/lo pair.  status as for chunk_tc.
bool gate_proj_supported(int D, int R, int HK, int NH);
size_t gate_proj_workspace(int64_t rows, int D, int R, int NH);
cudaError_t gate_proj(const void* x, const void* f_a, const void* f_b, const void* b_proj, int64_t rows, int D,
                      int R, int HK, int NH, void* gate_x, void* beta, void* ws, int32_t* status,
                      cudaStream_t st);

// out[h] = M[h] S[h] + A[h] (A may be null or out), K x K times K x V, fp32.
cudaError_t state_compose(const float* M, const float* S, const float* A, float* out, int H, int K, int V,
                          cudaStream_t st);

// Sets *status (device) to KDA_OK, then to KDA_ERR_RANGE if any x is outside [lo, hi] or NaN.
cudaError_t check_range(kda_dtype dt, const void* x, int64_t n, float lo, float hi, int32_t* status,
                        cudaStream_t st);

// Backward of the recurrence (CUDA cores, fp32): workspace bytes, and the launch.
// status (device, may be null): KDA_ERR_RANGE when a chain was skipped because
// malformed offsets would need more workspace than the call has.
size_t recurrent_bwd_workspace(int B, int T, int H, int K, int V, int N, bool packed);
cudaError_t recurrent_bwd(kda_dtype in_dt, const void* q, const void* k, const void* v, const void* g,
                          const void* beta, float scale, const float* s0, const int32_t* cu, int B, int T, int H,
                          int K, int V, int N, const float* dO, const float* dST, float* dq, float* dk, float* dv,
                          float* dg, float* dbeta, float* dS0, void* ws, int32_t* status, cudaStream_t st);

// Chunked backward (bf16 inputs, K = V = 128) on the forward's per-chunk operands:
// workspace bytes, and the launch (cudaErrorMemoryAllocation, before anything is
// enqueued, if ws_bytes is too small); status as for chunk_tc.
bool chunk_bwd_supported(kda_dtype in_dt, int K, int V);
size_t chunk_bwd_workspace(int B, int T, int H, int N, bool packed);
cudaError_t chunk_bwd(const ChunkParams& p, const float* dO, const float* dST, float* dq, float* dk, float* dv,
                      float* dg, float* dbeta, float* dS0, void* ws, size_t ws_bytes, int32_t* status,
                      cudaStream_t st);

}  // namespace kda
