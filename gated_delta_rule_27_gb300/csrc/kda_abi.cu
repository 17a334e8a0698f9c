// kda_abi.cu -- the extern "C" entry points of libkda: argument checks,
// path selection and launches.  Every check here runs on the host before
// anything is enqueued; the kernels themselves live in the other files.
#include <limits.h>

#include "kda_internal.cuh"
#include "kda_testing.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool supported_d(int32_t d) { return d == 16 || d == 64 || d == 128; }
bool supported_chunk(int32_t L) { return L == 16 || L == 32 || L == 64; }
bool valid_dtype(kda_dtype dt) { return dt == KDA_F32 || dt == KDA_BF16; }

kda::Path prefill_path(int32_t d, kda_dtype dt, int32_t L) {
    return (dt == KDA_BF16 && d == 128 && L == 64) ? kda::PATH_TC : kda::PATH_SIMT;
}

kda_status shape_check(int32_t total_tokens, int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v,
                       kda_dtype dt, int32_t chunk) {
    if (total_tokens < 0 || num_seqs < 0 || H <= 0 || H > 65535) return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(dt)) return KDA_ERR_INVALID_ARG;
    if (d_k != d_v || !supported_d(d_k) || !supported_chunk(chunk)) return KDA_ERR_UNSUPPORTED;
    // every row index (token * H + head) * d must fit the kernels' 32-bit token arithmetic
    if ((int64_t)total_tokens * H > INT_MAX || (int64_t)num_seqs * H * 8 > INT_MAX) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

// The fused prologue / epilogue options, checked (pointers only when the call has rows to process).
kda_status fusion_from(const kda_fusion_opts *opts, bool any_rows, const void *o, kda::Fusion *fu) {
    *fu = kda::Fusion{};
    if (!opts) return KDA_OK;
    if (opts->qk_l2norm) {
        if (!(opts->qk_eps >= 0.f)) return KDA_ERR_INVALID_ARG;
        fu->qk_norm = 1;
        fu->qk_eps = opts->qk_eps;
    }
    if (opts->out_gate) {
        if (!(opts->out_eps > 0.f)) return KDA_ERR_INVALID_ARG;
        if (any_rows && (!aligned16(opts->out_gate) || opts->out_gate == o)) return KDA_ERR_INVALID_ARG;
        if (!aligned16(opts->out_weight)) return KDA_ERR_INVALID_ARG;  // (null passes)
        fu->gate = opts->out_gate;
        fu->weight = opts->out_weight;
        fu->out_eps = opts->out_eps;
    }
    return KDA_OK;
}

}  // namespace

extern "C" {

const char *kda_status_string(kda_status status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        case KDA_ERR_BOUNDS: return "KDA_ERR_BOUNDS";
        default: return "KDA_ERR_UNKNOWN";
    }
}

size_t kda_prefill_workspace_size(int32_t total_tokens, int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v,
                                  kda_dtype in_dtype, int32_t chunk_size) {
    const int32_t L = chunk_size == 0 ? 64 : chunk_size;
    if (shape_check(total_tokens, num_seqs, H, d_k, d_v, in_dtype, L) != KDA_OK) return 0;
    return kda::ws_layout(total_tokens, num_seqs, H, d_k, d_v, L, prefill_path(d_k, in_dtype, L)).total;
}

}  // extern "C"

namespace {

kda_status prefill_impl(const void *q, const void *k, const void *v, const float *g, const float *beta,
                        const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens, int32_t H, int32_t d_k,
                        int32_t d_v, kda_dtype in_dtype, int32_t chunk_size, const float *S0, void *o,
                        float *S_final, void *workspace, size_t workspace_bytes, void *stream, kda::Marks &marks,
                        const kda_fusion_opts *opts = nullptr) {
    const int32_t L = chunk_size == 0 ? 64 : chunk_size;
    kda_status st = shape_check(total_tokens, num_seqs, H, d_k, d_v, in_dtype, L);
    if (st != KDA_OK) return st;
    kda::Fusion fu;
    if ((st = fusion_from(opts, total_tokens > 0, o, &fu)) != KDA_OK) return st;
    if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0) {
        if (!q || !k || !v || !g || !beta || !o) return KDA_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(o)) return KDA_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(beta) & 3u) return KDA_ERR_INVALID_ARG;
        if (o == q || o == k || o == v || o == (const void *)g) return KDA_ERR_INVALID_ARG;
    }
    if (!aligned16(S0) || !aligned16(S_final)) return KDA_ERR_INVALID_ARG;
    const kda::Path path = prefill_path(d_k, in_dtype, L);
    const kda::WsLayout lay = kda::ws_layout(total_tokens, num_seqs, H, d_k, d_v, L, path);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < lay.total)
        return KDA_ERR_INVALID_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const kda::TcPlan plan =
        path == kda::PATH_TC ? kda::tc_plan(num_seqs, H, total_tokens) : kda::TC_THREE;
    const bool flags = plan != kda::TC_THREE;
    cudaError_t e = cudaSuccess;
    if (!(path == kda::PATH_TC && kda::pipe_self_indexed(plan, num_seqs)))
        e = kda::launch_chunk_index(cu_seqlens, num_seqs, total_tokens, L, workspace,
                                    flags ? static_cast<char *>(workspace) + lay.flags_off : nullptr,
                                    flags ? lay.flags_bytes : 0, s, marks);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    if (path == kda::PATH_TC)
        e = kda::launch_prefill_tc(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, H, S0, o, S_final, workspace,
                                   plan, fu, s, marks);
    else
        e = kda::launch_prefill_simt(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, H, d_k, in_dtype, L, S0,
                                     o, S_final, workspace, fu, s, marks);
    marks.end(s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

extern "C" {

kda_status kda_prefill_chunked(const void *q, const void *k, const void *v, const float *g, const float *beta,
                               const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens, int32_t H,
                               int32_t d_k, int32_t d_v, kda_dtype in_dtype, int32_t chunk_size, const float *S0,
                               void *o, float *S_final, void *workspace, size_t workspace_bytes, void *stream) {
    kda::Marks marks;
    return prefill_impl(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, in_dtype, chunk_size, S0,
                        o, S_final, workspace, workspace_bytes, stream, marks);
}

kda_status kda_prefill_chunked_ex(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                  const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens, int32_t H,
                                  int32_t d_k, int32_t d_v, kda_dtype in_dtype, int32_t chunk_size, const float *S0,
                                  void *o, float *S_final, void *workspace, size_t workspace_bytes, void *stream,
                                  const kda_fusion_opts *opts) {
    kda::Marks marks;
    return prefill_impl(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, in_dtype, chunk_size, S0,
                        o, S_final, workspace, workspace_bytes, stream, marks, opts);
}

kda_status kda_prefill_chunked_profiled(const void *q, const void *k, const void *v, const float *g,
                                        const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                        int32_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                        kda_dtype in_dtype, int32_t chunk_size, const float *S0, void *o,
                                        float *S_final, void *workspace, size_t workspace_bytes, void *stream,
                                        void *const *events, int32_t *num_kernels, const char **kernel_names) {
    kda::Marks marks;
    marks.ev = events;
    marks.names = kernel_names;
    const kda_status st = prefill_impl(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, in_dtype,
                                       chunk_size, S0, o, S_final, workspace, workspace_bytes, stream, marks);
    if (num_kernels) *num_kernels = marks.n;
    return st;
}

kda_status kda_prefill_check(const void *workspace, void *stream) {
    if (!workspace) return KDA_ERR_INVALID_ARG;
    int32_t flag = -1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&flag, workspace, sizeof(flag), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    return kda::status_from_word(flag);
}

kda_status kda_testing_set_plan(int32_t plan) {
    if (plan != -1 && plan != KDA_TESTING_PLAN_THREE && plan != KDA_TESTING_PLAN_CHAIN && plan != KDA_TESTING_PLAN_PIPE)
        return KDA_ERR_INVALID_ARG;
    kda::testing_set_plan(plan == KDA_TESTING_PLAN_THREE   ? kda::TC_THREE
                          : plan == KDA_TESTING_PLAN_CHAIN ? kda::TC_CHAIN
                          : plan == KDA_TESTING_PLAN_PIPE  ? kda::TC_PIPE
                                                           : -1);
    return KDA_OK;
}

kda_status kda_testing_set_fault(int32_t fault, int64_t wait_limit_ns) {
    if ((fault != KDA_TESTING_FAULT_NONE && fault != KDA_TESTING_FAULT_NO_PUBLISH &&
         fault != KDA_TESTING_FAULT_CHUNK_TABLE) ||
        wait_limit_ns < 0)
        return KDA_ERR_INVALID_ARG;
    kda::testing_set_fault(fault, (long long)wait_limit_ns);
    return KDA_OK;
}

kda_status kda_decode_step(const void *q, const void *k, const void *v, const float *g, const float *beta,
                           int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v, kda_dtype in_dtype,
                           float *S_inout, void *o, void *stream) {
    return kda_decode_step_ex(q, k, v, g, beta, num_seqs, H, d_k, d_v, in_dtype, S_inout, o, stream, nullptr);
}

kda_status kda_decode_step_ex(const void *q, const void *k, const void *v, const float *g, const float *beta,
                              int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v, kda_dtype in_dtype,
                              float *S_inout, void *o, void *stream, const kda_fusion_opts *opts) {
    if (num_seqs < 0 || H <= 0 || !valid_dtype(in_dtype)) return KDA_ERR_INVALID_ARG;
    kda::Fusion fu;
    if (kda_status st = fusion_from(opts, num_seqs > 0, o, &fu)) return st;
    if (d_k != d_v || !supported_d(d_k)) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)num_seqs * H > INT_MAX) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !S_inout || !o) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(S_inout) || !aligned16(o))
        return KDA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(beta) & 3u) return KDA_ERR_INVALID_ARG;
    if (o == q || o == k || o == v || o == (const void *)S_inout) return KDA_ERR_INVALID_ARG;
    cudaError_t e = kda::launch_decode(q, k, v, g, beta, num_seqs, H, d_k, in_dtype, S_inout, o, nullptr, num_seqs,
                                       nullptr, fu, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_decode_step_indexed(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                   const int32_t *seq_idx, int32_t num_active, int32_t num_slots, int32_t H,
                                   int32_t d_k, int32_t d_v, kda_dtype in_dtype, float *S_pool, void *o,
                                   int32_t *status, void *stream) {
    if (num_active < 0 || num_slots < 0 || H <= 0 || !valid_dtype(in_dtype)) return KDA_ERR_INVALID_ARG;
    if (d_k != d_v || !supported_d(d_k)) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)num_active * H > INT_MAX || (int64_t)num_slots * H > INT_MAX) return KDA_ERR_UNSUPPORTED;
    if (num_active == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !seq_idx || !S_pool || !o) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(S_pool) || !aligned16(o))
        return KDA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(beta) & 3u) || (reinterpret_cast<uintptr_t>(seq_idx) & 3u) ||
        (reinterpret_cast<uintptr_t>(status) & 3u))
        return KDA_ERR_INVALID_ARG;
    if (o == q || o == k || o == v || o == (const void *)S_pool) return KDA_ERR_INVALID_ARG;
    cudaError_t e = kda::launch_decode(q, k, v, g, beta, num_active, H, d_k, in_dtype, S_pool, o, seq_idx, num_slots,
                                       status, kda::Fusion{}, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

static kda_status state_copy(const float *src, float *dst, const int32_t *seq_idx, int32_t n, int32_t num_slots,
                             int32_t H, int32_t d_k, int32_t d_v, bool scatter, int32_t *status, void *stream) {
    if (n < 0 || num_slots < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
    if (d_k != d_v || !supported_d(d_k)) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)H * d_k * d_v > INT_MAX || (int64_t)n * H > INT_MAX) return KDA_ERR_UNSUPPORTED;
    if (n == 0) return KDA_OK;
    if (!src || !dst || !seq_idx || !aligned16(src) || !aligned16(dst) || (reinterpret_cast<uintptr_t>(seq_idx) & 3u) ||
        (reinterpret_cast<uintptr_t>(status) & 3u) || src == dst)
        return KDA_ERR_INVALID_ARG;
    cudaError_t e = kda::launch_state_copy(src, dst, seq_idx, n, num_slots, H, d_k, scatter, status,
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_short_conv_prefill(const void *x, const float *w, const int32_t *cu_seqlens, int32_t num_seqs,
                                  int32_t total_tokens, int32_t C, int32_t W, kda_dtype in_dtype,
                                  const float *conv_state, void *y, float *conv_state_out, void *stream) {
    if (total_tokens < 0 || num_seqs < 0 || C <= 0 || !valid_dtype(in_dtype)) return KDA_ERR_INVALID_ARG;
    if (W < 1 || W > KDA_SHORT_CONV_MAX_W) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)total_tokens * C > INT_MAX || (int64_t)num_seqs * W * C > INT_MAX) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    const uintptr_t el = in_dtype == KDA_BF16 ? 1u : 3u;
    if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!x || !w || !y || (reinterpret_cast<uintptr_t>(x) & el) ||
                             (reinterpret_cast<uintptr_t>(y) & el) || x == y))
        return KDA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(w) & 3u) || (reinterpret_cast<uintptr_t>(conv_state) & 3u) ||
        (reinterpret_cast<uintptr_t>(conv_state_out) & 3u))
        return KDA_ERR_INVALID_ARG;
    if (W > 1 && conv_state && conv_state == conv_state_out) return KDA_ERR_INVALID_ARG;
    cudaError_t e = kda::launch_conv_prefill(x, w, cu_seqlens, num_seqs, total_tokens, C, W, in_dtype,
                                             W > 1 ? conv_state : nullptr, y, W > 1 ? conv_state_out : nullptr,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_short_conv_decode(const void *x, const float *w, int32_t N, int32_t C, int32_t W, kda_dtype in_dtype,
                                 float *conv_state, void *y, void *stream) {
    if (N < 0 || C <= 0 || !valid_dtype(in_dtype)) return KDA_ERR_INVALID_ARG;
    if (W < 1 || W > KDA_SHORT_CONV_MAX_W) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)N * W * C > INT_MAX) return KDA_ERR_UNSUPPORTED;
    if (N == 0) return KDA_OK;
    const uintptr_t el = in_dtype == KDA_BF16 ? 1u : 3u;
    if (!x || !w || !y || (W > 1 && !conv_state) || (reinterpret_cast<uintptr_t>(x) & el) ||
        (reinterpret_cast<uintptr_t>(y) & el) || (reinterpret_cast<uintptr_t>(w) & 3u) ||
        (reinterpret_cast<uintptr_t>(conv_state) & 3u) || x == y)
        return KDA_ERR_INVALID_ARG;
    cudaError_t e = kda::launch_conv_decode(x, w, N, C, W, in_dtype, conv_state, y, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_state_snapshot(const float *S_pool, const int32_t *seq_idx, int32_t n, int32_t num_slots, int32_t H,
                              int32_t d_k, int32_t d_v, float *S_saved, int32_t *status, void *stream) {
    return state_copy(S_pool, S_saved, seq_idx, n, num_slots, H, d_k, d_v, false, status, stream);
}

kda_status kda_state_restore(const float *S_saved, const int32_t *seq_idx, int32_t n, int32_t num_slots, int32_t H,
                             int32_t d_k, int32_t d_v, float *S_pool, int32_t *status, void *stream) {
    return state_copy(S_saved, S_pool, seq_idx, n, num_slots, H, d_k, d_v, true, status, stream);
}

}  // extern "C"
