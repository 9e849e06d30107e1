// C-ABI entry points of libkda.so (declared in include/kda.h): argument
// validation on the host, then one kernel launch on the caller's stream.
#include <math.h>

#include "kda_chunk.h"
#include "kda_common.cuh"

namespace {

constexpr int kAbiVersion = 2;

bool head_size_ok(int d) { return d == 64 || d == 128; }
bool dtype_ok(kda_dtype d) { return d == KDA_F32 || d == KDA_BF16; }

// Sizes: all non-negative, element counts representable in int64 and
// per-sequence token offsets in int32 (the kernels index tokens with int64).
kda_status check_sizes(int B, int T, int H, int K, int V, int N) {
    if (B < 0 || T < 0 || H <= 0 || N < 0) return KDA_ERR_INVALID_ARG;
    if (!head_size_ok(K) || !head_size_ok(V)) return KDA_ERR_UNSUPPORTED;
    const double elems = (double)B * (double)T * (double)H * (double)(K > V ? K : V);
    if (elems > 9.0e18) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

float resolve_scale(float scale, int K) { return scale > 0.f ? scale : 1.0f / sqrtf((float)K); }

kda_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return KDA_OK;
    return e == cudaErrorMemoryAllocation ? KDA_ERR_WORKSPACE : KDA_ERR_CUDA;
}

kda_status check_common(const void* q, const void* k, const void* v, const void* g,
                        const void* beta, kda_dtype in_dtype, const float* initial_state,
                        const int32_t* cu_seqlens, int B, int T, int H, int K, int V, int N,
                        const void* o, kda_dtype o_dtype, const float* final_state) {
    kda_status s = check_sizes(B, T, H, K, V, N);
    if (s != KDA_OK) return s;
    if (!dtype_ok(in_dtype) || !dtype_ok(o_dtype)) return KDA_ERR_UNSUPPORTED;
    if (cu_seqlens != nullptr) {
        if (B != 1) return KDA_ERR_INVALID_ARG;
    } else if (N != B) {
        return KDA_ERR_INVALID_ARG;
    }
    const bool have_tokens = (int64_t)B * T > 0;
    if (have_tokens && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, o, initial_state, final_state};
    for (const void* p : ptrs)
        if (p && !kda_host::aligned16(p)) return KDA_ERR_INVALID_ARG;
    const size_t esz = in_dtype == KDA_BF16 ? 2 : 4;
    if (beta && ((uintptr_t)beta % esz)) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && ((uintptr_t)cu_seqlens % 4)) return KDA_ERR_INVALID_ARG;
    if (final_state && initial_state && final_state != initial_state) {
        // Partial overlap of the two state tensors is not allowed.
        const char* a = (const char*)initial_state;
        const char* b = (const char*)final_state;
        const size_t bytes = (size_t)N * H * K * V * sizeof(float);
        if (a < b + bytes && b < a + bytes) return KDA_ERR_INVALID_ARG;
    }
    return KDA_OK;
}

// A caller-owned workspace of at least the queried size (16-byte aligned) and an
// optional 4-byte aligned device status word.
kda_status check_workspace(kda_dtype in_dtype, int B, int T, int H, int K, int V, int N, bool packed,
                           const void* ws, size_t ws_bytes, const int32_t* status) {
    if (status != nullptr && ((uintptr_t)status % 4)) return KDA_ERR_INVALID_ARG;
    if (ws != nullptr && !kda_host::aligned16(ws)) return KDA_ERR_INVALID_ARG;
    if (!kda::chunk_tc_supported(in_dtype, K, V)) return KDA_OK;
    const size_t need = kda::chunk_tc_workspace(B, T, H, N, packed);
    if (ws_bytes < need || (need > 0 && ws == nullptr)) return KDA_ERR_WORKSPACE;
    return KDA_OK;
}

}  // namespace

extern "C" {

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: head size or dtype not supported";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: the workspace is smaller than the call needs (see the *_workspace_size queries), or the call needs more than kda_chunk_fwd_noalloc's fixed scratch holds";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime error";
        case KDA_ERR_RANGE: return "KDA_ERR_RANGE: input out of range";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: device-side wait gave up";
    }
    return "unknown kda_status";
}

int kda_abi_version(void) { return kAbiVersion; }

size_t kda_chunk_fwd_workspace_size(kda_dtype in_dtype, int B, int T, int H, int K, int V, int N, int packed) {
    if (B < 0 || T < 0 || H <= 0 || N < 0) return 0;
    if (!kda::chunk_tc_supported(in_dtype, K, V)) return 0;
    return kda::chunk_tc_workspace(B, T, H, N, packed != 0);
}

void kda_set_wait_limit(uint32_t iterations) { kda::set_wait_limit(iterations); }

void kda_inject_wait_timeout(int kernel) { kda::inject_wait_timeout(kernel); }

kda_status kda_chunk_fwd(const void* q, const void* k, const void* v, const void* g,
                         const void* beta, kda_dtype in_dtype, float scale,
                         const float* initial_state, const int32_t* cu_seqlens, int B, int T,
                         int H, int K, int V, int N, void* o, kda_dtype o_dtype,
                         float* final_state, void* workspace, size_t workspace_bytes, int32_t* status,
                         void* stream) {
    kda_status s = check_common(q, k, v, g, beta, in_dtype, initial_state, cu_seqlens, B, T, H,
                                K, V, N, o, o_dtype, final_state);
    if (s != KDA_OK) return s;
    s = check_workspace(in_dtype, B, T, H, K, V, N, cu_seqlens != nullptr, workspace, workspace_bytes, status);
    if (s != KDA_OK) return s;
    kda::ChunkParams p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
    p.scale = resolve_scale(scale, K);
    p.initial_state = initial_state;
    p.cu_seqlens = cu_seqlens;
    p.B = B; p.T = T; p.H = H; p.N = N;
    p.o = o;
    p.final_state = final_state;
    cudaStream_t st = (cudaStream_t)stream;
    if (kda::chunk_tc_supported(in_dtype, K, V))
        return from_cuda(kda::chunk_tc(o_dtype, p, workspace, workspace_bytes, status, st));
    kda::trace_set(nullptr, nullptr, nullptr);
    if (status != nullptr && cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return KDA_ERR_CUDA;
    return from_cuda(kda::chunk_simt(in_dtype, o_dtype, K, V, false, p, st));
}

kda_status kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                                 const void* beta, kda_dtype in_dtype, float scale,
                                 const float* initial_state, const int32_t* cu_seqlens, int B,
                                 int T, int H, int K, int V, int N, void* o, kda_dtype o_dtype,
                                 float* final_state, void* stream) {
    kda_status s = check_common(q, k, v, g, beta, in_dtype, initial_state, cu_seqlens, B, T, H,
                                K, V, N, o, o_dtype, final_state);
    if (s != KDA_OK) return s;
    if (!kda::chunk_tc_supported(in_dtype, K, V)) return KDA_ERR_UNSUPPORTED;
    kda::ChunkParams p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
    p.scale = resolve_scale(scale, K);
    p.initial_state = initial_state;
    p.cu_seqlens = cu_seqlens;
    p.B = B; p.T = T; p.H = H; p.N = N;
    p.o = o;
    p.final_state = final_state;
    return from_cuda(kda::chunk_tc_fixed_scratch(o_dtype, p, (cudaStream_t)stream));
}

kda_status kda_chunk_fwd_fused(const void* q_raw, const void* k_raw, const void* v_raw,
                               const void* gate_x, const void* beta, kda_dtype in_dtype,
                               const float* conv_q, const float* conv_k, const float* conv_v,
                               int conv_act, const float* A_log, const float* dt_bias,
                               float lower_bound, float l2_eps, float scale,
                               const float* initial_state, const int32_t* cu_seqlens, int B,
                               int T, int H, int K, int V, int N, void* o, kda_dtype o_dtype,
                               float* final_state, void* workspace, size_t workspace_bytes,
                               int32_t* status, void* stream) {
    kda_status s = check_common(q_raw, k_raw, v_raw, gate_x, beta, in_dtype, initial_state,
                                cu_seqlens, B, T, H, K, V, N, o, o_dtype, final_state);
    if (s != KDA_OK) return s;
    s = check_workspace(in_dtype, B, T, H, K, V, N, cu_seqlens != nullptr, workspace, workspace_bytes, status);
    if (s != KDA_OK) return s;
    if (conv_act != 0 && conv_act != 1) return KDA_ERR_INVALID_ARG;
    if (!(l2_eps >= 0.f) || !(lower_bound <= 0.f) || isnan(lower_bound)) return KDA_ERR_INVALID_ARG;
    const bool have_tokens = (int64_t)B * T > 0;
    if (have_tokens && (!conv_q || !conv_k || !conv_v || !A_log || !dt_bias)) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {conv_q, conv_k, conv_v, A_log, dt_bias};
    for (const void* p : ptrs)
        if (p && !kda_host::aligned16(p)) return KDA_ERR_INVALID_ARG;
    kda::ChunkParams p{};
    p.q = q_raw; p.k = k_raw; p.v = v_raw; p.g = gate_x; p.beta = beta;
    p.scale = resolve_scale(scale, K);
    p.initial_state = initial_state;
    p.cu_seqlens = cu_seqlens;
    p.B = B; p.T = T; p.H = H; p.N = N;
    p.o = o;
    p.final_state = final_state;
    p.conv_q = conv_q; p.conv_k = conv_k; p.conv_v = conv_v;
    p.conv_act = conv_act;
    p.A_log = A_log; p.dt_bias = dt_bias;
    p.lower_bound = lower_bound;
    p.l2_eps = l2_eps;
    cudaStream_t st = (cudaStream_t)stream;
    if (kda::chunk_tc_supported(in_dtype, K, V))
        return from_cuda(kda::chunk_tc_fused(o_dtype, p, workspace, workspace_bytes, status, st));
    kda::trace_set(nullptr, nullptr, nullptr);
    if (status != nullptr && cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return KDA_ERR_CUDA;
    return from_cuda(kda::chunk_simt(in_dtype, o_dtype, K, V, true, p, st));
}

void kda_trace_events(void* begin, void* split, void* end) { kda::trace_set(begin, split, end); }

kda_status kda_recurrent_step(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, kda_dtype in_dtype, float scale, float* state,
                              int N, int H, int K, int V, void* o, kda_dtype o_dtype,
                              void* stream) {
    if (N < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
    if (!head_size_ok(K) || !head_size_ok(V)) return KDA_ERR_UNSUPPORTED;
    if (!dtype_ok(in_dtype) || !dtype_ok(o_dtype)) return KDA_ERR_UNSUPPORTED;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !state || !o) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, state, o};
    for (const void* p : ptrs)
        if (!kda_host::aligned16(p)) return KDA_ERR_INVALID_ARG;
    if ((uintptr_t)beta % (in_dtype == KDA_BF16 ? 2 : 4)) return KDA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    return from_cuda(kda::decode_step(in_dtype, o_dtype, K, V, q, k, v, g, beta,
                                      resolve_scale(scale, K), state, N, H, o, st));
}

kda_status kda_output_gate(const float* o, const void* gate, kda_dtype gate_dtype, const float* weight,
                           float eps, int B, int T, int H, int V, void* out, kda_dtype out_dtype,
                           void* stream) {
    if (B < 0 || T < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || isinf(eps)) return KDA_ERR_INVALID_ARG;
    if (!head_size_ok(V)) return KDA_ERR_UNSUPPORTED;
    if (!dtype_ok(gate_dtype) || !dtype_ok(out_dtype)) return KDA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * T * H;
    if ((double)rows * V > 9.0e18) return KDA_ERR_INVALID_ARG;
    if (rows == 0) return KDA_OK;
    if (!o || !gate || !out) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {o, gate, weight, out};
    for (const void* p : ptrs)
        if (p && !kda_host::aligned16(p)) return KDA_ERR_INVALID_ARG;
    // in place only for an fp32 out; no other overlap with the inputs
    const char* ob = reinterpret_cast<const char*>(o);
    const char* gb = reinterpret_cast<const char*>(gate);
    const char* xb = reinterpret_cast<const char*>(out);
    const size_t o_bytes = (size_t)rows * V * 4;
    const size_t g_bytes = (size_t)rows * V * (gate_dtype == KDA_BF16 ? 2 : 4);
    const size_t x_bytes = (size_t)rows * V * (out_dtype == KDA_BF16 ? 2 : 4);
    const bool same = xb == ob && out_dtype == KDA_F32;
    if (!same && xb < ob + o_bytes && ob < xb + x_bytes) return KDA_ERR_INVALID_ARG;
    if (xb < gb + g_bytes && gb < xb + x_bytes) return KDA_ERR_INVALID_ARG;
    return from_cuda(kda::output_gate(gate_dtype, out_dtype, V, o, gate, weight, eps, rows, out,
                                      (cudaStream_t)stream));
}

size_t kda_gate_proj_workspace_size(int B, int T, int D, int R, int NH) {
    if (B < 0 || T < 0 || (R != 64 && R != 128) || NH <= 0 || R + NH > 256) return 0;
    return kda::gate_proj_workspace((int64_t)B * T, D, R, NH);
}

kda_status kda_gate_proj(const void* x, const void* f_a, const void* f_b, const void* b_proj, kda_dtype dtype,
                         int B, int T, int D, int R, int HK, int NH, void* gate_x, void* beta, void* workspace,
                         size_t workspace_bytes, int32_t* status, void* stream) {
    if (B < 0 || T < 0 || D <= 0 || R <= 0 || HK <= 0 || NH <= 0) return KDA_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)B * T;
    if (rows > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_BF16 || !kda::gate_proj_supported(D, R, HK, NH)) return KDA_ERR_UNSUPPORTED;
    if (status != nullptr && ((uintptr_t)status % 4)) return KDA_ERR_INVALID_ARG;
    if (rows > 0) {
        const void* ptrs[] = {x, f_a, f_b, b_proj, gate_x, beta};
        for (const void* p : ptrs)
            if (!p || !kda_host::aligned16(p)) return KDA_ERR_INVALID_ARG;
        const size_t need = kda::gate_proj_workspace(rows, D, R, NH);
        if (workspace_bytes < need || workspace == nullptr) return KDA_ERR_WORKSPACE;
        if (!kda_host::aligned16(workspace)) return KDA_ERR_INVALID_ARG;
        // the outputs and the workspace overlap nothing else
        struct Span { const char* p; size_t n; };
        const Span in[] = {{(const char*)x, (size_t)rows * D * 2}, {(const char*)f_a, (size_t)R * D * 2},
                           {(const char*)f_b, (size_t)HK * R * 2}, {(const char*)b_proj, (size_t)NH * D * 2}};
        const Span out[] = {{(const char*)gate_x, (size_t)rows * HK * 2}, {(const char*)beta, (size_t)rows * NH * 2},
                            {(const char*)workspace, need}};
        for (int i = 0; i < 3; ++i) {
            for (const Span& a : in)
                if (out[i].p < a.p + a.n && a.p < out[i].p + out[i].n) return KDA_ERR_INVALID_ARG;
            for (int j = i + 1; j < 3; ++j)
                if (out[i].p < out[j].p + out[j].n && out[j].p < out[i].p + out[i].n) return KDA_ERR_INVALID_ARG;
        }
    }
    return from_cuda(kda::gate_proj(x, f_a, f_b, b_proj, rows, D, R, HK, NH, gate_x, beta, workspace, status,
                                    (cudaStream_t)stream));
}

kda_status kda_state_compose(const float* M, const float* S, const float* A, float* out, int H, int K, int V,
                             void* stream) {
    if (H < 0) return KDA_ERR_INVALID_ARG;
    if (!head_size_ok(K) || !head_size_ok(V)) return KDA_ERR_UNSUPPORTED;
    if (H == 0) return KDA_OK;
    if (!M || !S || !out) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {M, S, A, out};
    for (const void* p : ptrs)
        if (p && !kda_host::aligned16(p)) return KDA_ERR_INVALID_ARG;
    const char* xb = reinterpret_cast<const char*>(out);
    const size_t x_bytes = (size_t)H * K * V * 4;
    const struct { const void* p; size_t n; } ins[] = {{M, (size_t)H * K * K * 4}, {S, x_bytes}};
    for (const auto& in : ins) {
        const char* b = reinterpret_cast<const char*>(in.p);
        if (xb < b + in.n && b < xb + x_bytes) return KDA_ERR_INVALID_ARG;
    }
    if (A && A != out) {
        const char* ab = reinterpret_cast<const char*>(A);
        if (xb < ab + x_bytes && ab < xb + x_bytes) return KDA_ERR_INVALID_ARG;
    }
    return from_cuda(kda::state_compose(M, S, A, out, H, K, V, (cudaStream_t)stream));
}

kda_status kda_check_range(const void* x, kda_dtype dtype, int64_t count, float lo, float hi, int32_t* status,
                           void* stream) {
    if (!dtype_ok(dtype)) return KDA_ERR_UNSUPPORTED;
    if (count < 0 || !(lo <= hi)) return KDA_ERR_INVALID_ARG;
    if (!status || ((uintptr_t)status % 4)) return KDA_ERR_INVALID_ARG;
    if (count > 0 && !x) return KDA_ERR_INVALID_ARG;
    if (x && ((uintptr_t)x % (dtype == KDA_BF16 ? 2 : 4))) return KDA_ERR_INVALID_ARG;
    return from_cuda(kda::check_range(dtype, x, count, lo, hi, status, (cudaStream_t)stream));
}

size_t kda_recurrent_bwd_workspace_size(kda_dtype in_dtype, int B, int T, int H, int K, int V, int N, int packed) {
    if (B < 0 || T < 0 || H <= 0 || N < 0 || !dtype_ok(in_dtype)) return 0;
    if (!head_size_ok(K) || !head_size_ok(V)) return 0;
    return kda::recurrent_bwd_workspace(B, T, H, K, V, N, packed != 0);
}

kda_status kda_recurrent_bwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
                             kda_dtype in_dtype, float scale, const float* initial_state,
                             const int32_t* cu_seqlens, int B, int T, int H, int K, int V, int N,
                             const float* dO, const float* dS_T, float* dq, float* dk, float* dv, float* dg,
                             float* dbeta, float* dS0, void* workspace, size_t workspace_bytes,
                             int32_t* status, void* stream) {
    kda_status s = check_common(q, k, v, g, beta, in_dtype, initial_state, cu_seqlens, B, T, H, K, V, N,
                                dO, KDA_F32, nullptr);
    if (s != KDA_OK) return s;
    const bool have_tokens = (int64_t)B * T > 0;
    if (have_tokens && (!dq || !dk || !dv || !dg || !dbeta)) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {dS_T, dq, dk, dv, dg, dS0};
    for (const void* p : ptrs)
        if (p && !kda_host::aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (dbeta && ((uintptr_t)dbeta % 4)) return KDA_ERR_INVALID_ARG;
    if (status != nullptr && ((uintptr_t)status % 4)) return KDA_ERR_INVALID_ARG;
    const size_t bytes = (int64_t)N * H == 0 ? 0 : kda::recurrent_bwd_workspace(B, T, H, K, V, N, cu_seqlens != nullptr);
    if (workspace_bytes < bytes || (bytes > 0 && workspace == nullptr)) return KDA_ERR_WORKSPACE;
    if (workspace != nullptr && !kda_host::aligned16(workspace)) return KDA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    return from_cuda(kda::recurrent_bwd(in_dtype, q, k, v, g, beta, resolve_scale(scale, K), initial_state,
                                        cu_seqlens, B, T, H, K, V, N, dO, dS_T, dq, dk, dv, dg, dbeta, dS0,
                                        workspace, status, st));
}

size_t kda_chunk_bwd_workspace_size(kda_dtype in_dtype, int B, int T, int H, int K, int V, int N, int packed) {
    if (B < 0 || T < 0 || H <= 0 || N < 0 || !dtype_ok(in_dtype)) return 0;
    if (!head_size_ok(K) || !head_size_ok(V)) return 0;
    if (kda::chunk_bwd_supported(in_dtype, K, V)) return kda::chunk_bwd_workspace(B, T, H, N, packed != 0);
    return kda::recurrent_bwd_workspace(B, T, H, K, V, N, packed != 0);
}

kda_status kda_chunk_bwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
                         kda_dtype in_dtype, float scale, const float* initial_state, const int32_t* cu_seqlens,
                         int B, int T, int H, int K, int V, int N, const float* dO, const float* dS_T, float* dq,
                         float* dk, float* dv, float* dg, float* dbeta, float* dS0, void* workspace,
                         size_t workspace_bytes, int32_t* status, void* stream) {
    if (!kda::chunk_bwd_supported(in_dtype, K, V))
        return kda_recurrent_bwd(q, k, v, g, beta, in_dtype, scale, initial_state, cu_seqlens, B, T, H, K, V, N, dO,
                                 dS_T, dq, dk, dv, dg, dbeta, dS0, workspace, workspace_bytes, status, stream);
    kda_status s = check_common(q, k, v, g, beta, in_dtype, initial_state, cu_seqlens, B, T, H, K, V, N,
                                dO, KDA_F32, nullptr);
    if (s != KDA_OK) return s;
    const bool have_tokens = (int64_t)B * T > 0;
    if (have_tokens && (!dq || !dk || !dv || !dg || !dbeta)) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {dS_T, dq, dk, dv, dg, dS0};
    for (const void* p : ptrs)
        if (p && !kda_host::aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (dbeta && ((uintptr_t)dbeta % 4)) return KDA_ERR_INVALID_ARG;
    if (status != nullptr && ((uintptr_t)status % 4)) return KDA_ERR_INVALID_ARG;
    const size_t bytes = kda::chunk_bwd_workspace(B, T, H, N, cu_seqlens != nullptr);
    if (workspace_bytes < bytes || (bytes > 0 && workspace == nullptr)) return KDA_ERR_WORKSPACE;
    if (workspace != nullptr && !kda_host::aligned16(workspace)) return KDA_ERR_INVALID_ARG;
    kda::ChunkParams p{};
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
    p.scale = resolve_scale(scale, K);
    p.initial_state = initial_state;
    p.cu_seqlens = cu_seqlens;
    p.B = B; p.T = T; p.H = H; p.N = N;
    return from_cuda(kda::chunk_bwd(p, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, workspace, workspace_bytes, status,
                                    (cudaStream_t)stream));
}

}  // extern "C"
