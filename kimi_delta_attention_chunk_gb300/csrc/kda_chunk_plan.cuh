// The work plan and the per-(chunk, head) workspace slot of the tensor-core
// prefill, shared by its kernels and by the chunked backward that reuses the
// forward's slots (internal to libkda.so).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {
namespace cplan {

constexpr int C = 64;
constexpr int D = 128;   // K = V

// ---- workspace slot of one (chunk, head), written by the local kernel --------
constexpr uint32_t SLOT_WQH = 0;        // [-W hi | Qs hi] (bf16) as one B operand, MN-major stored
                                        //   n-group by n-group (n = r for -W, n = 64 + r for
                                        //   Qs = scale q e^G; k = c): -W the first 16 KB, Qs the rest
constexpr uint32_t SLOT_WQL = 32768;    // [-W lo | Qs lo], same layout
constexpr uint32_t SLOT_EGC = 65536;    // e^{G_C} fp32 [128]
constexpr uint32_t SLOT_IMG = 66048;    // bytes of the images above (one shared-memory copy)
constexpr uint32_t SLOT_KH = 66048;     // Kbar hi as B operand [128 c][64 r], K-major
constexpr uint32_t SLOT_KL = 82432;     // Kbar lo
constexpr uint32_t SLOT_P = 98816;      // scale P hi | lo, B operand [64 r][64 j] K-major
constexpr uint32_t SLOT_KBP = 49152;    // bytes of Kbar and P (one shared-memory copy)
constexpr uint32_t SLOT_UT = 115200;    // U~ fp32 [64 r][128 v]
constexpr uint32_t SLOT_BYTES = 147968;


// Work description shared by the kernels.  Sequences are either B dense rows
// of T tokens (cu_seqlens == nullptr) or packed by cu_seqlens; chunks are
// numbered sequence by sequence (global chunk index gc), slots by gc * H + h.
struct Plan {
    const int32_t* cu_seqlens;
    const int32_t* chunk_off;  // [N + 1] first global chunk of each sequence (packed only)
    const int32_t* order;      // [N] sequences longest first (packed only; nullptr = identity)
    const int32_t* chunk_seq;  // [max_chunks] sequence of each global chunk, -1 past the end
    int T, H, N;
    int cps;                   // chunks per sequence (dense only)
    int64_t max_chunks;        // number of workspace chunk slots (an upper bound when packed)
    uint8_t* slots;
    int32_t* status;           // device status word (KDA_ERR_TIMEOUT on a wait that gave up), or null
    uint32_t wait_iter;        // polls before a wait gives up
    int inject;                // testing: 1 = the chunk-local kernel's, 2 = the state kernel's, 3 = the
                               //   backward chain kernel's, 4 = the backward chunk kernel's first wait
                               //   is on an mbarrier that nothing arrives on (0 = none)
    float* states_out;         // or null: the state entering every chunk, fp32 [slot][K][V] (for the backward)
    float* at_out;             // or null: per slot A (strictly lower, without beta) and T = (I + Diag(beta) A)^{-1},
                               //   fp32 [slot][2][C][C] (for the backward)
    float* u_out;              // with states_out: per slot U = U~ - W S, fp32 [slot][C][V] (for the backward)
};

__device__ __forceinline__ void report_timeout(const Plan& pl) {
    if (pl.status != nullptr) *reinterpret_cast<volatile int32_t*>(pl.status) = (int32_t)KDA_ERR_TIMEOUT;
}

struct Chunk {
    int64_t c0, eos;  // first token of the chunk, end of its sequence
    int64_t bos;      // first token of its sequence
    int64_t gc;       // global chunk index
    int h;
    bool valid;
};

// (the host keeps the number of tasks below 2^31, so the divisions are 32-bit)
__device__ __forceinline__ Chunk decode_task(const Plan& pl, int64_t task) {
    Chunk ch{};
    ch.valid = false;
    if (task >= pl.max_chunks * pl.H) return ch;
    const uint32_t t = (uint32_t)task, H = (uint32_t)pl.H;
    const uint32_t gc = t / H;
    ch.gc = gc;
    ch.h = (int)(t - gc * H);
    if (pl.cu_seqlens == nullptr) {
        const uint32_t cps = (uint32_t)pl.cps;
        const uint32_t n = gc / cps, j = gc - n * cps;
        ch.bos = (int64_t)n * pl.T;
        ch.c0 = ch.bos + (int64_t)j * C;
        ch.eos = ch.bos + pl.T;
    } else {
        const int n = pl.chunk_seq[gc];
        if (n < 0) return ch;
        ch.bos = min(max((int)pl.cu_seqlens[n], 0), pl.T);
        ch.c0 = ch.bos + (int64_t)(gc - (uint32_t)pl.chunk_off[n]) * C;
        ch.eos = min(max((int)pl.cu_seqlens[n + 1], 0), pl.T);
    }
    ch.valid = true;
    return ch;
}

// The sequence and chunk range of a (sequence, head) chain: CTA `blk` of a grid of
// N * H chains (packed: sequences longest first when the plan has an order).
struct Chain {
    int n, h;
    int64_t bos, eos;   // token range of the sequence
    int64_t g0;         // its first global chunk
    int64_t nchunks;    // its chunks (0 for an empty sequence)
};
__device__ __forceinline__ Chain chain_of(const Plan& pl, int blk) {
    Chain c{};
    c.h = blk % pl.H;
    const int rank = blk / pl.H;
    if (pl.cu_seqlens == nullptr) {
        c.n = rank;
        c.bos = (int64_t)c.n * pl.T;
        c.eos = c.bos + pl.T;
        c.g0 = (int64_t)c.n * pl.cps;
        c.nchunks = pl.cps;
    } else {
        c.n = pl.order != nullptr ? pl.order[rank] : rank;
        c.bos = min(max((int)pl.cu_seqlens[c.n], 0), pl.T);
        c.eos = min(max((int)pl.cu_seqlens[c.n + 1], 0), pl.T);
        if (c.eos < c.bos) c.eos = c.bos;
        // (offsets that overlap can need more chunks than the workspace holds:
        //  those are left out, never read past the end)
        c.g0 = min((int64_t)pl.chunk_off[c.n], pl.max_chunks);
        c.nchunks = min((int64_t)pl.chunk_off[c.n + 1], pl.max_chunks) - c.g0;
        if (c.nchunks < 0) c.nchunks = 0;
    }
    return c;
}

}  // namespace cplan

struct ChunkParams;
// The tensor-core prefill (bf16 inputs, K = V = 128, no prologue) for the backward:
// o goes to p.o as bf16 (scratch), the state entering every chunk to states_out
// (fp32 [max_chunks * H][K][V]), each chunk's A and T to at_out (fp32 [max_chunks *
// H][2][C][C]) and its U = U~ - W S to u_out (fp32 [max_chunks * H][C][V]), and
// *plan_out receives the work plan, whose slots (in ws) hold the forward's per-chunk
// operands.  Workspace as for chunk_tc.
cudaError_t chunk_tc_forward_states(const ChunkParams& p, void* ws, size_t ws_bytes, float* states_out,
                                    float* at_out, float* u_out, cplan::Plan* plan_out, int32_t* status,
                                    cudaStream_t st);
}  // namespace kda
