// kda_conv.cu -- short causal convolution on the inputs of the recurrence.
//
// Lecture 04, section 3: before Q/K normalisation, the sublayer mixes Q, K
// and/or V over a few neighbouring tokens with a short causal convolution; in
// decode that step needs a rolling convolution state, just as the recurrence
// needs S (Lecture 11, section 2, "Serving state" row: rollback must reconcile
// the convolution state too).  The pages give no formula; the kernels compute
// the plain depthwise causal convolution per channel c,
//
//     y_t[c] = sum_{j < W} w[c][j] x_{t-j}[c],
//
// inside each document of cu_seqlens, with the positions before a document's
// first token read from that document's carried state (its previous W - 1
// inputs, oldest first; zeros when none is given).
//
// Both kernels are bound by HBM: every input is read once (plus a halo of
// W - 1 rows per tile, served by L1/L2) and every output written once.  One
// thread owns one channel over a tile of tokens, so a warp's loads and stores
// are 32 consecutive channels of one token row (coalesced).  The tile's
// inputs are all loaded before any arithmetic (into the thread's own column
// of a shared-memory tile), so that every thread has its whole tile of loads
// in flight at once; the arithmetic then walks a register window.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kConvThreads = 256;
constexpr int kConvTile = 32;  // tokens per thread
constexpr int kMaxW = 8;

// The document of token t: the last n with cu[n] <= t (documents may be empty).
__device__ __forceinline__ int doc_of(const int32_t *__restrict__ cu, int num_seqs, int t) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <typename T>
__global__ void __launch_bounds__(kConvThreads)
conv_prefill_kernel(const T *__restrict__ x, const float *__restrict__ w, const int32_t *__restrict__ cu,
                    int num_seqs, int total_tokens, int C, int W, const float *__restrict__ state_in, T *__restrict__ y,
                    float *__restrict__ state_out) {
    __shared__ float xs[kConvTile][kConvThreads];  // column threadIdx.x: this thread's inputs
    const int c = blockIdx.x * kConvThreads + threadIdx.x;
    const int t_begin = blockIdx.y * kConvTile;
    if (c >= C || t_begin >= total_tokens) return;
    const int t_end = min(t_begin + kConvTile, total_tokens);
#pragma unroll
    for (int j = 0; j < kConvTile; ++j)
        if (t_begin + j < t_end) xs[j][threadIdx.x] = to_f32(x[(size_t)(t_begin + j) * C + c]);
    float wc[kMaxW];
#pragma unroll
    for (int j = 0; j < kMaxW; ++j) wc[j] = j < W ? w[(size_t)c * W + j] : 0.f;
    int n = doc_of(cu, num_seqs, t_begin);
    while (n + 1 < num_seqs && cu[n + 1] <= t_begin) ++n;  // skip empty documents ending at t_begin
    int doc_start = cu[n], doc_end = cu[n + 1];
    // window[i] = input at position t - i (i = 0 the current token), for the token about to be processed
    float win[kMaxW];
    // (every index below stays in bounds whatever cu_seqlens holds; its validity is the caller's contract)
    auto input_at = [&](int p) -> float {  // position p < current token, inside document n or its carried state
        if (p >= doc_start && p >= 0) return to_f32(x[(size_t)p * C + c]);
        const int back = doc_start - p;  // 1 .. W - 1 positions before the document
        if (!state_in || back < 1 || back > W - 1) return 0.f;
        return state_in[((size_t)n * (W - 1) + (W - 1 - back)) * C + c];
    };
#pragma unroll
    for (int i = 1; i < kMaxW; ++i) win[i] = (i < W) ? input_at(t_begin - i) : 0.f;
    for (int t = t_begin; t < t_end; ++t) {
        if (t >= doc_end && n + 1 < num_seqs) {  // the next document starts at t: its window comes from its state
            do {
                ++n;
            } while (n + 1 < num_seqs && cu[n + 1] <= t);
            doc_start = cu[n];
            doc_end = cu[n + 1];
#pragma unroll
            for (int i = 1; i < kMaxW; ++i) win[i] = (i < W) ? input_at(t - i) : 0.f;
        }
        win[0] = xs[t - t_begin][threadIdx.x];
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxW; ++j) acc = fmaf(wc[j], win[j], acc);
        y[(size_t)t * C + c] = from_f32<T>(acc);
        if (state_out && t >= doc_end - (W - 1) && t < doc_end) {
            // one of the document's last W - 1 inputs: slot W - 1 - (doc_end - t) of its new state
            state_out[((size_t)n * (W - 1) + (W - 1 - (doc_end - t))) * C + c] = win[0];
        }
#pragma unroll
        for (int i = kMaxW - 1; i > 0; --i) win[i] = win[i - 1];
    }
}

// The new state of documents shorter than W - 1 tokens keeps some carried entries (and an empty document keeps
// all of them): written here, one thread per (document, channel), for the slots no token of the document wrote.
__global__ void __launch_bounds__(kConvThreads)
conv_short_docs_kernel(const int32_t *__restrict__ cu, int num_seqs, int C, int W, const float *__restrict__ state_in,
                       float *__restrict__ state_out) {
    const int c = blockIdx.x * kConvThreads + threadIdx.x;
    const int n = blockIdx.y;
    if (c >= C) return;
    const int len = max(cu[n + 1] - cu[n], 0);
    for (int s = 0; s < W - 1 - len; ++s) {  // slot s of the new state is old slot s + len
        const float v = state_in ? state_in[((size_t)n * (W - 1) + s + len) * C + c] : 0.f;
        state_out[((size_t)n * (W - 1) + s) * C + c] = v;
    }
}

template <typename T>
__global__ void __launch_bounds__(kConvThreads)
conv_decode_kernel(const T *__restrict__ x, const float *__restrict__ w, int N, int C, int W, float *__restrict__ state,
                   T *__restrict__ y) {
    const size_t i = (size_t)blockIdx.x * kConvThreads + threadIdx.x;
    if (i >= (size_t)N * C) return;
    const int n = (int)(i / C), c = (int)(i % C);
    float *st = state + (size_t)n * (W - 1) * C + c;
    const float xin = to_f32(x[i]);
    // win[s]: state slot s (oldest first), the input W - 1 - s tokens back, weighted by w[c][W - 1 - s];
    // every load is issued before any arithmetic
    float win[kMaxW], wr[kMaxW];
#pragma unroll
    for (int s = 0; s < kMaxW; ++s) {
        win[s] = s < W - 1 ? st[(size_t)s * C] : 0.f;
        wr[s] = s < W - 1 ? w[(size_t)c * W + (W - 1 - s)] : 0.f;
    }
    float acc = w[(size_t)c * W] * xin;
#pragma unroll
    for (int s = kMaxW - 1; s >= 0; --s)  // the newest state slot first: the same order as the prefill kernel
        if (s < W - 1) acc = fmaf(wr[s], win[s], acc);
    y[i] = from_f32<T>(acc);
    // roll: drop the oldest input, append this one
#pragma unroll
    for (int s = 0; s < kMaxW - 1; ++s)
        if (s < W - 1) st[(size_t)s * C] = s + 1 < W - 1 ? win[s + 1] : xin;
}

template <typename T>
cudaError_t conv_prefill_t(const void *x, const float *w, const int32_t *cu, int num_seqs, int total_tokens, int C,
                           int W, const float *state_in, void *y, float *state_out, cudaStream_t st) {
    if (total_tokens > 0) {
        dim3 grid((unsigned)((C + kConvThreads - 1) / kConvThreads),
                  (unsigned)((total_tokens + kConvTile - 1) / kConvTile));
        conv_prefill_kernel<T><<<grid, kConvThreads, 0, st>>>((const T *)x, w, cu, num_seqs, total_tokens, C, W,
                                                              state_in, (T *)y, state_out);
        if (cudaError_t e = cudaGetLastError()) return e;
    }
    if (state_out && W > 1 && num_seqs > 0) {
        dim3 grid((unsigned)((C + kConvThreads - 1) / kConvThreads), (unsigned)num_seqs);
        conv_short_docs_kernel<<<grid, kConvThreads, 0, st>>>(cu, num_seqs, C, W, state_in, state_out);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_conv_prefill(const void *x, const float *w, const int32_t *cu, int num_seqs, int total_tokens, int C,
                                int W, kda_dtype dt, const float *state_in, void *y, float *state_out,
                                cudaStream_t st) {
    if (dt == KDA_BF16)
        return conv_prefill_t<__nv_bfloat16>(x, w, cu, num_seqs, total_tokens, C, W, state_in, y, state_out, st);
    return conv_prefill_t<float>(x, w, cu, num_seqs, total_tokens, C, W, state_in, y, state_out, st);
}

cudaError_t launch_conv_decode(const void *x, const float *w, int N, int C, int W, kda_dtype dt, float *state, void *y,
                               cudaStream_t st) {
    const size_t n = (size_t)N * C;
    if (n == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((n + kConvThreads - 1) / kConvThreads);
    if (dt == KDA_BF16)
        conv_decode_kernel<__nv_bfloat16><<<blocks, kConvThreads, 0, st>>>((const __nv_bfloat16 *)x, w, N, C, W, state,
                                                                           (__nv_bfloat16 *)y);
    else
        conv_decode_kernel<float><<<blocks, kConvThreads, 0, st>>>((const float *)x, w, N, C, W, state, (float *)y);
    return cudaGetLastError();
}

}  // namespace kda
