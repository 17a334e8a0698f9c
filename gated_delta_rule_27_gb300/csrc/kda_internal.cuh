// kda_internal.cuh -- shared definitions of libkda's CUDA sources (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kda.h"
#include "kda_check.cuh"

namespace kda {

// ---------------------------------------------------------------------------
// Element access.  Inputs q, k, v and the output o are bf16 or fp32; all
// arithmetic is fp32.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// ---------------------------------------------------------------------------
// Prefill workspace.  Everything of a chunk that does not depend on the
// incoming state is written by the chunk-parallel pass and read by the
// sequential state pass.
//
//   [0, 256)            int32 status word (0 = cu_seqlens valid), the failing line of a
//                       bounds check after it, the preparation's work counter at word
//                       kPrepCounterWord (zeroed by the chunk index kernel), then padding
//   doc_slot0           int32 [num_seqs + 1]: first chunk slot of each document
//                       (exclusive prefix sum of ceil(len / L)), 256-byte padded
//   records             one per (chunk slot, head), `record_bytes` each
//   flags               (tensor-core path) progress flags of the chain plan
//
// The number of chunk slots is bounded by total_tokens / L + num_seqs, so the
// size depends only on the call's scalar arguments.
// ---------------------------------------------------------------------------
enum Path { PATH_SIMT = 0, PATH_TC = 1 };

// int32 word of the workspace header that the persistent tensor-core preparation claims its units from
constexpr int kPrepCounterWord = 32;
// 64-bit word (int32 words 40-41) of the workspace header where a self-indexed pipe launch publishes its call
// token once its first CTA has written the slot table and the status word and cleared the flags
constexpr int kGoWord = 40;

struct WsLayout {
    size_t doc_slot0_off;
    size_t doc_order_off;  // int32 [num_seqs]: documents by descending chunk count (long chains start first)
    size_t records_off;
    size_t record_bytes;
    int64_t max_slots;
    size_t flags_off;    // tensor-core path: int32 [max_slots * H] record-published flags, int32 [max_slots * H]
                         // state-image counters, then two int32 work counters (chain and pipe plans)
    size_t flags_bytes;  // 0 on the CUDA-core path
    size_t total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// SIMT record (fp32): W [L,dk] | Ut [L,dv] | Qp [L,dk] | Oloc [L,dv] | Kend [L,dk] | gamma [dk]
struct SimtRecord {
    size_t W, Ut, Qp, Oloc, Kend, gamma, bytes;
};
__host__ __device__ inline SimtRecord simt_record(int L, int dk, int dv) {
    SimtRecord r;
    size_t off = 0;
    r.W = off;     off += (size_t)L * dk * 4;
    r.Ut = off;    off += (size_t)L * dv * 4;
    r.Qp = off;    off += (size_t)L * dk * 4;
    r.Oloc = off;  off += (size_t)L * dv * 4;
    r.Kend = off;  off += (size_t)L * dk * 4;
    r.gamma = off; off += (size_t)dk * 4;
    r.bytes = align256(off);
    return r;
}

// Tensor-core record (d = 128, L = 64).  Every operand is stored as the exact
// shared-memory image its consumer loads (bf16, swizzled), so each
// consumer moves its part of a record with one or two bulk copies.  The state
// pass reads [Mc, Qp) plus its column tile of Ut and writes S; the output
// pass reads [Qp, bytes) in one piece.
//   Mc     M' = -Kend^T W, K-major [128 d_k rows][128 d_k], 2 panels          32 KB
//   gamma  fp32 [128], padded to 1 KB
//   Kend   the chunk's keys decayed to its end, MN-major [64 tokens][128 d_k],
//          2 panels of 8 KB (the state pass forms Kend^T Ut from it)          16 KB
//   Qp     MN-major [128 d_k][64 tokens]                                       16 KB
//   P      intra-chunk scores, K-major [64 tokens][64 tokens]                   8 KB
//   Ut     Ut^T, K-major [128 d_v][64 tokens]                                  16 KB
//   S      the chunk's incoming state as the state pass multiplied it: bf16
//          MN-major [128 d_k rows][128 d_v], four 32-column chunks of 8 KB with
//          the 64-byte swizzle (written by the state pass, each chain its own
//          chunks in one piece)                                                32 KB
struct TcRecord {
    size_t Mc, gamma, Kend, Qp, P, Ut, S, state_part, out_part, bytes;
};
__host__ __device__ constexpr TcRecord tc_record() {
    return TcRecord{0, 32768, 33792, 50176, 66560, 74752, 91136, 50176, 123904 - 50176, 123904};
}

inline WsLayout ws_layout(int64_t total_tokens, int64_t num_seqs, int64_t H, int dk, int dv, int L, Path path) {
    WsLayout w;
    w.doc_slot0_off = 256;
    w.doc_order_off = w.doc_slot0_off + align256((size_t)(num_seqs + 1) * 4);
    w.records_off = w.doc_order_off + align256((size_t)(num_seqs > 0 ? num_seqs : 1) * 4);
    w.record_bytes = path == PATH_TC ? tc_record().bytes : simt_record(L, dk, dv).bytes;
    w.max_slots = total_tokens / L + num_seqs;
    w.flags_off = w.records_off + (size_t)w.max_slots * (size_t)H * w.record_bytes;
    w.flags_bytes = path == PATH_TC ? align256(((size_t)2 * w.max_slots * H + 2) * 4) : 0;
    w.total = w.flags_off + w.flags_bytes;
    return w;
}

// The workspace status word as a status: 0 valid, 1 invalid cu_seqlens (written by the chunk index kernel),
// KDA_ERR_TIMEOUT a bounded device-side wait that gave up (written by the kernel that waited).
inline kda_status status_from_word(int32_t word) {
    if (word == 0) return KDA_OK;
    if (word == (int32_t)KDA_ERR_TIMEOUT) return KDA_ERR_TIMEOUT;
    if (word == (int32_t)KDA_ERR_BOUNDS) return KDA_ERR_BOUNDS;
    return KDA_ERR_INVALID_ARG;
}

// Chunk slots of a call, bounded by its arguments: the record of (slot, head) exists iff slot < max_slots.
__device__ __forceinline__ int max_chunk_slots(const int32_t *cu, int num_seqs, int L) {
    return cu[num_seqs] / L + num_seqs;
}

// Locates the document and chunk of a chunk slot by binary search over the
// per-document first-slot table.  Returns false for slots past the last chunk.
__device__ __forceinline__ bool locate_slot(const int32_t *__restrict__ doc_slot0, const int32_t *__restrict__ cu,
                                            int num_seqs, int L, int slot, int *doc, int *t0, int *len) {
    if (slot >= doc_slot0[num_seqs]) return false;
    int lo = 0, hi = num_seqs - 1;  // find the last doc with doc_slot0[doc] <= slot
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (doc_slot0[mid] <= slot) lo = mid; else hi = mid - 1;
    }
    const int start = cu[lo] + (slot - doc_slot0[lo]) * L;
    *doc = lo;
    *t0 = start;
    *len = min(L, cu[lo + 1] - start);
    return true;
}

// ---------------------------------------------------------------------------
// The fused prologue and epilogue of kda_fusion_opts, as the kernels take them
// (all zero / null: neither).
// ---------------------------------------------------------------------------
struct Fusion {
    int qk_norm = 0;
    float qk_eps = 0.f;
    const void *gate = nullptr;
    const float *weight = nullptr;
    float out_eps = 0.f;
};

// The logistic function in fp32 (the gate of the output normalisation).
__device__ __forceinline__ float sigmoidf(float z) { return 1.f / (1.f + expf(-z)); }

// ---------------------------------------------------------------------------
// Optional profiling marks: an event recorded before every kernel of a call
// and one after the last, with the kernels' names (all may be null).
// ---------------------------------------------------------------------------
struct Marks {
    void *const *ev = nullptr;
    const char **names = nullptr;
    int n = 0;
    void before(cudaStream_t s, const char *kernel) {
        if (ev && n <= KDA_PREFILL_MAX_KERNELS && ev[n]) cudaEventRecord(static_cast<cudaEvent_t>(ev[n]), s);
        if (names && n < KDA_PREFILL_MAX_KERNELS) names[n] = kernel;
        ++n;
    }
    void end(cudaStream_t s) {
        if (ev && n <= KDA_PREFILL_MAX_KERNELS && ev[n]) cudaEventRecord(static_cast<cudaEvent_t>(ev[n]), s);
    }
};

// Launches `kernel` so that it may start while the previous kernel in the stream finishes (programmatic
// stream serialisation); the kernel must call griddepcontrol.wait before it reads that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// Launchers (each returns cudaSuccess or the launch error).
// ---------------------------------------------------------------------------
cudaError_t launch_chunk_index(const int32_t *cu, int num_seqs, int total_tokens, int L, void *ws, void *clear,
                               size_t clear_bytes, cudaStream_t st, Marks &marks);

// Launch plans of the tensor-core prefill: three kernels (preparation, state, output); the preparation
// followed by one cooperative launch running the state chains with the output units alongside (chain); or one
// cooperative launch of chains beside groups that prepare the records and then form the outputs (pipe).  The
// last two need the workspace's progress flags zeroed before they start.  The automatic choice takes the pipe
// plan or the state pass plan; the chain plan runs when the test hook forces it.
enum TcPlan { TC_THREE = 0, TC_CHAIN = 2, TC_PIPE = 3 };
TcPlan tc_plan(int num_seqs, int H, int total_tokens);
// Whether a call of this plan does without the chunk index kernel: the pipe plan on one document sets up its
// own slot table, status word and flags (never in the bounds-checking build, whose tests inject faults there).
bool pipe_self_indexed(TcPlan plan, int num_seqs);

// Test hooks behind include/kda_testing.h: force a plan (-1 automatic), inject a fault with a wait bound.
void testing_set_plan(int plan);
void testing_set_fault(int fault, long long wait_ns);
int testing_fault();
constexpr int kFaultChunkTable = 2;  // test hook of the bounds-checking build (KDA_TESTING_FAULT_CHUNK_TABLE)

cudaError_t launch_prefill_simt(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                const int32_t *cu, int num_seqs, int total_tokens, int H, int d, kda_dtype dt,
                                int L, const float *S0, void *o, float *S_final, void *ws, const Fusion &fu,
                                cudaStream_t st, Marks &marks);

cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const float *g, const float *beta,
                              const int32_t *cu, int num_seqs, int total_tokens, int H, const float *S0, void *o,
                              float *S_final, void *ws, TcPlan plan, const Fusion &fu, cudaStream_t st,
                              Marks &marks);

// Decode step of num_seqs sequences; with `idx` (device, [num_seqs]) their states are the pool slots idx[i] of
// S [num_slots, H, d, d], otherwise S[i].
cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g, const float *beta,
                          int num_seqs, int H, int d, kda_dtype dt, float *S, void *o, const int32_t *idx,
                          int num_slots, int32_t *status, const Fusion &fu, cudaStream_t st);

// Short causal convolution (kda_conv.cu): prefill over packed documents with carried states, and one decode
// step with a rolling state.
cudaError_t launch_conv_prefill(const void *x, const float *w, const int32_t *cu, int num_seqs, int total_tokens, int C,
                                int W, kda_dtype dt, const float *state_in, void *y, float *state_out,
                                cudaStream_t st);
cudaError_t launch_conv_decode(const void *x, const float *w, int N, int C, int W, kda_dtype dt, float *state, void *y,
                               cudaStream_t st);

// Snapshot (gather: dst[i] = src[idx[i]]) or restore (scatter: dst[idx[i]] = src[i]) of n whole slots of
// H heads' d x d fp32 states.
cudaError_t launch_state_copy(const float *src, float *dst, const int32_t *idx, int n, int num_slots, int H, int d,
                              bool scatter, int32_t *status, cudaStream_t st);

}  // namespace kda
