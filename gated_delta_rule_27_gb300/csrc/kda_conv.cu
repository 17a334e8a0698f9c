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

// ---------------------------------------------------------------------------
// Four-channel kernels (C a multiple of 4, x and y aligned to four elements): one thread owns four adjacent
// channels, so a warp moves 128 channels of a token row per access (256 B in bf16, 512 B in fp32), and the
// filter width is a template parameter, so the window lives in registers with static indices.  The sums are
// the scalar kernels' sums term for term (w[c][0] x_t first, then one fmaf per older input), so the two
// kernels and the decode step agree bit for bit.
// ---------------------------------------------------------------------------
constexpr int kVecTile = 16;    // tokens per thread: one batch of loads in flight
constexpr int kShortDocs = 64;  // documents per CTA row of the short-document state pass

template <typename T> struct Vec4;
template <> struct Vec4<float> {
    using raw = float4;
    __device__ __forceinline__ static void to(const raw &r, float (&f)[4]) { f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w; }
    __device__ __forceinline__ static raw from(const float (&f)[4]) { return make_float4(f[0], f[1], f[2], f[3]); }
};
template <> struct Vec4<__nv_bfloat16> {
    using raw = uint2;
    __device__ __forceinline__ static void to(const raw &r, float (&f)[4]) {
        f[0] = __uint_as_float(r.x << 16); f[1] = __uint_as_float(r.x & 0xffff0000u);
        f[2] = __uint_as_float(r.y << 16); f[3] = __uint_as_float(r.y & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
        const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
        return a | (b << 16);
    }
    __device__ __forceinline__ static raw from(const float (&f)[4]) { return make_uint2(pack(f[0], f[1]), pack(f[2], f[3])); }
};

template <typename T>
__device__ __forceinline__ typename Vec4<T>::raw load_vec4(const T *p) {
    return __ldg(reinterpret_cast<const typename Vec4<T>::raw *>(p));
}

// The window of the token at position t of document m, four channels: win[j] = the input j tokens back
// (j = 1 .. W - 1), from the document or, before its first token, from its carried state (zeros without one).
// Every index stays in bounds whatever cu_seqlens holds (its validity is the caller's contract).
template <typename T, int W>
__device__ __forceinline__ void load_window(float (&win)[W][4], const T *__restrict__ x,
                                            const float *__restrict__ state_in, int C, int c0, int m, int ds, int t) {
#pragma unroll
    for (int j = 1; j < W; ++j) {
        const int p = t - j;
        if (p >= ds && p >= 0) {
            Vec4<T>::to(load_vec4(x + (size_t)p * C + c0), win[j]);
        } else {
            const int back = ds - p;  // 1 .. j for a valid cu_seqlens
            if (state_in && back >= 1 && back <= W - 1) {
                const float4 s = __ldg(reinterpret_cast<const float4 *>(
                    state_in + ((size_t)m * (W - 1) + (W - 1 - back)) * C + c0));
                win[j][0] = s.x; win[j][1] = s.y; win[j][2] = s.z; win[j][3] = s.w;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) win[j][i] = 0.f;
            }
        }
    }
}

// A tile of kVecTile tokens x 4 channels per thread, the token loop unrolled: the tile's loads are issued
// first, then each token takes its input from registers.  A document that starts inside the tile reloads the
// window (a warp-uniform branch, rare); the document's last W - 1 inputs are written to its new state.
// Three CTAs per SM where the tile's registers fit in the 80 that allows (bf16 inputs, W <= 5); two
// (up to 128 registers) for fp32 inputs, whose tile is twice as many registers, and for wider filters.
template <typename T, int W>
constexpr int conv_vec_min_blocks() { return (sizeof(T) == 2 && W <= 5) ? 3 : 2; }

template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads, conv_vec_min_blocks<T, W>())
conv_prefill_vec_kernel(const T *__restrict__ x, const float *__restrict__ w, const int32_t *__restrict__ cu,
                        int num_seqs, int total_tokens, int C, const float *__restrict__ state_in, T *__restrict__ y,
                        float *__restrict__ state_out) {
    const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * 4;
    const int tiles = (total_tokens + kVecTile - 1) / kVecTile;
    if ((int)blockIdx.y >= tiles) {
        // the rows past the token tiles: documents shorter than W - 1, whose new state keeps some of the
        // carried one (slot s of the new state is old slot s + len), kShortDocs documents per row
        if (c0 >= C || W < 2 || !state_out) return;
        const int n0 = ((int)blockIdx.y - tiles) * kShortDocs;
        for (int n = n0; n < min(n0 + kShortDocs, num_seqs); ++n) {
            const int len = max(cu[n + 1] - cu[n], 0);
            for (int s = 0; s < W - 1 - len; ++s) {
                const float4 v = state_in ? __ldg(reinterpret_cast<const float4 *>(
                                                state_in + ((size_t)n * (W - 1) + s + len) * C + c0))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4 *>(state_out + ((size_t)n * (W - 1) + s) * C + c0) = v;
            }
        }
        return;
    }
    const int t_begin = blockIdx.y * kVecTile;
    if (c0 >= C) return;
    const int t_end = min(t_begin + kVecTile, total_tokens);
    typename Vec4<T>::raw xv[kVecTile];
#pragma unroll
    for (int u = 0; u < kVecTile; ++u)
        if (t_begin + u < t_end) xv[u] = load_vec4(x + (size_t)(t_begin + u) * C + c0);
    float wc[4][W];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < W; ++j) wc[i][j] = w[(size_t)(c0 + i) * W + j];
    // the inputs before the tile, loaded with it (kept where they belong to the tile's first document)
    typename Vec4<T>::raw pre[W > 1 ? W - 1 : 1];
#pragma unroll
    for (int j = 1; j < W; ++j)
        if (t_begin - j >= 0) pre[j - 1] = load_vec4(x + (size_t)(t_begin - j) * C + c0);
    int m = doc_of(cu, num_seqs, t_begin);
    while (m + 1 < num_seqs && cu[m + 1] <= t_begin) ++m;  // skip empty documents ending at t_begin
    int ds = cu[m], de = cu[m + 1];
    float win[W][4];  // win[j][i]: channel c0 + i, j tokens back (j = 0 the current token)
#pragma unroll
    for (int j = 1; j < W; ++j) {
        const int p = t_begin - j;
        if (p >= ds && p >= 0) {
            Vec4<T>::to(pre[j - 1], win[j]);
        } else {
            const int back = ds - p;  // 1 .. j for a valid cu_seqlens
            if (state_in && back >= 1 && back <= W - 1) {
                const float4 s = __ldg(reinterpret_cast<const float4 *>(
                    state_in + ((size_t)m * (W - 1) + (W - 1 - back)) * C + c0));
                win[j][0] = s.x; win[j][1] = s.y; win[j][2] = s.z; win[j][3] = s.w;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) win[j][i] = 0.f;
            }
        }
    }
#pragma unroll
    for (int u = 0; u < kVecTile; ++u) {
        const int t = t_begin + u;
        if (t < t_end) {
            if (t >= de && m + 1 < num_seqs) {  // the next document starts at t
                do {
                    ++m;
                } while (m + 1 < num_seqs && cu[m + 1] <= t);
                ds = cu[m];
                de = cu[m + 1];
                load_window<T, W>(win, x, state_in, C, c0, m, ds, t);
            }
            Vec4<T>::to(xv[u], win[0]);
            float out[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < W; ++j) acc = fmaf(wc[i][j], win[j][i], acc);
                out[i] = acc;
            }
            *reinterpret_cast<typename Vec4<T>::raw *>(y + (size_t)t * C + c0) = Vec4<T>::from(out);
            if (state_out && t >= de - (W - 1) && t < de)  // slot W - 1 - (de - t) of the document's new state
                *reinterpret_cast<float4 *>(state_out + ((size_t)m * (W - 1) + (W - 1 - (de - t))) * C + c0) =
                    make_float4(win[0][0], win[0][1], win[0][2], win[0][3]);
#pragma unroll
            for (int j = W - 1; j > 0; --j)
#pragma unroll
                for (int i = 0; i < 4; ++i) win[j][i] = win[j - 1][i];
        }
    }
}

// One decode step on four channels of one sequence per thread.
template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads)
conv_decode_vec_kernel(const T *__restrict__ x, const float *__restrict__ w, int N, int C, float *__restrict__ state,
                       T *__restrict__ y) {
    const size_t i4 = ((size_t)blockIdx.x * kConvThreads + threadIdx.x) * 4;
    if (i4 >= (size_t)N * C) return;
    const int n = (int)(i4 / C), c0 = (int)(i4 % C);
    float *st = state + (size_t)n * (W - 1) * C + c0;
    float xin[4];
    Vec4<T>::to(load_vec4(x + i4), xin);
    float4 win[W > 1 ? W - 1 : 1];  // state slot s (oldest first)
#pragma unroll
    for (int s = 0; s < W - 1; ++s) win[s] = __ldg(reinterpret_cast<const float4 *>(st + (size_t)s * C));
    float wc[4][W];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < W; ++j) wc[i][j] = w[(size_t)(c0 + i) * W + j];
    float out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float acc = fmaf(wc[i][0], xin[i], 0.f);
#pragma unroll
        for (int j = 1; j < W; ++j) {  // j tokens back is state slot W - 1 - j
            const float4 v = win[W - 1 - j];
            acc = fmaf(wc[i][j], i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w, acc);
        }
        out[i] = acc;
    }
    *reinterpret_cast<typename Vec4<T>::raw *>(y + i4) = Vec4<T>::from(out);
#pragma unroll
    for (int s = 0; s < W - 1; ++s)
        *reinterpret_cast<float4 *>(st + (size_t)s * C) =
            s + 1 < W - 1 ? win[s + 1] : make_float4(xin[0], xin[1], xin[2], xin[3]);
}

template <typename T, int W>
cudaError_t conv_prefill_vec(const T *x, const float *w, const int32_t *cu, int num_seqs, int total_tokens, int C,
                             const float *state_in, T *y, float *state_out, cudaStream_t st) {
    // token tiles, then (with a new state to write) rows for the documents shorter than W - 1
    const int short_rows = state_out && W > 1 ? (num_seqs + kShortDocs - 1) / kShortDocs : 0;
    dim3 grid((unsigned)((C / 4 + kConvThreads - 1) / kConvThreads),
              (unsigned)((total_tokens + kVecTile - 1) / kVecTile + short_rows));
    conv_prefill_vec_kernel<T, W><<<grid, kConvThreads, 0, st>>>(x, w, cu, num_seqs, total_tokens, C, state_in, y,
                                                                  state_out);
    return cudaGetLastError();
}

template <typename T, int W>
cudaError_t conv_decode_vec(const T *x, const float *w, int N, int C, float *state, T *y, cudaStream_t st) {
    const size_t n4 = (size_t)N * C / 4;
    conv_decode_vec_kernel<T, W><<<(unsigned)((n4 + kConvThreads - 1) / kConvThreads), kConvThreads, 0, st>>>(
        x, w, N, C, state, y);
    return cudaGetLastError();
}

// The four-channel kernels need C % 4 == 0 and 4-element alignment of x and y (and of the fp32 states).
template <typename T>
bool vec4_ok(int C, const void *x, const void *y, const float *s0, const float *s1) {
    const uintptr_t a = 4 * sizeof(T) - 1;
    return C % 4 == 0 && !(reinterpret_cast<uintptr_t>(x) & a) && !(reinterpret_cast<uintptr_t>(y) & a) &&
           !(reinterpret_cast<uintptr_t>(s0) & 15u) && !(reinterpret_cast<uintptr_t>(s1) & 15u);
}

template <typename T>
cudaError_t conv_prefill_t(const void *x, const float *w, const int32_t *cu, int num_seqs, int total_tokens, int C,
                           int W, const float *state_in, void *y, float *state_out, cudaStream_t st) {
    const bool vec = total_tokens > 0 && vec4_ok<T>(C, x, y, state_in, state_out);
    if (vec) {  // (its launch also writes the states of the documents shorter than W - 1)
        const T *xt = static_cast<const T *>(x);
        T *yt = static_cast<T *>(y);
        cudaError_t e;
        switch (W) {
            case 1: e = conv_prefill_vec<T, 1>(xt, w, cu, num_seqs, total_tokens, C, state_in, yt, state_out, st); break;
            case 2: e = conv_prefill_vec<T, 2>(xt, w, cu, num_seqs, total_tokens, C, state_in, yt, state_out, st); break;
            case 3: e = conv_prefill_vec<T, 3>(xt, w, cu, num_seqs, total_tokens, C, state_in, yt, state_out, st); break;
            case 4: e = conv_prefill_vec<T, 4>(xt, w, cu, num_seqs, total_tokens, C, state_in, yt, state_out, st); break;
            case 5: e = conv_prefill_vec<T, 5>(xt, w, cu, num_seqs, total_tokens, C, state_in, yt, state_out, st); break;
            case 6: e = conv_prefill_vec<T, 6>(xt, w, cu, num_seqs, total_tokens, C, state_in, yt, state_out, st); break;
            case 7: e = conv_prefill_vec<T, 7>(xt, w, cu, num_seqs, total_tokens, C, state_in, yt, state_out, st); break;
            default: e = conv_prefill_vec<T, 8>(xt, w, cu, num_seqs, total_tokens, C, state_in, yt, state_out, st); break;
        }
        if (e) return e;
    } else if (total_tokens > 0) {
        dim3 grid((unsigned)((C + kConvThreads - 1) / kConvThreads),
                  (unsigned)((total_tokens + kConvTile - 1) / kConvTile));
        conv_prefill_kernel<T><<<grid, kConvThreads, 0, st>>>((const T *)x, w, cu, num_seqs, total_tokens, C, W,
                                                              state_in, (T *)y, state_out);
        if (cudaError_t e = cudaGetLastError()) return e;
    }
    if (!vec && state_out && W > 1 && num_seqs > 0) {
        dim3 grid((unsigned)((C + kConvThreads - 1) / kConvThreads), (unsigned)num_seqs);
        conv_short_docs_kernel<<<grid, kConvThreads, 0, st>>>(cu, num_seqs, C, W, state_in, state_out);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

template <typename T>
cudaError_t conv_decode_dispatch(const void *x, const float *w, int N, int C, int W, float *state, void *y,
                                 cudaStream_t st) {
    const T *xt = static_cast<const T *>(x);
    T *yt = static_cast<T *>(y);
    switch (W) {
        case 1: return conv_decode_vec<T, 1>(xt, w, N, C, state, yt, st);
        case 2: return conv_decode_vec<T, 2>(xt, w, N, C, state, yt, st);
        case 3: return conv_decode_vec<T, 3>(xt, w, N, C, state, yt, st);
        case 4: return conv_decode_vec<T, 4>(xt, w, N, C, state, yt, st);
        case 5: return conv_decode_vec<T, 5>(xt, w, N, C, state, yt, st);
        case 6: return conv_decode_vec<T, 6>(xt, w, N, C, state, yt, st);
        case 7: return conv_decode_vec<T, 7>(xt, w, N, C, state, yt, st);
        default: return conv_decode_vec<T, 8>(xt, w, N, C, state, yt, st);
    }
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
    if (dt == KDA_BF16 ? vec4_ok<__nv_bfloat16>(C, x, y, state, nullptr) : vec4_ok<float>(C, x, y, state, nullptr))
        return dt == KDA_BF16 ? conv_decode_dispatch<__nv_bfloat16>(x, w, N, C, W, state, y, st)
                              : conv_decode_dispatch<float>(x, w, N, C, W, state, y, st);
    const unsigned blocks = (unsigned)((n + kConvThreads - 1) / kConvThreads);
    if (dt == KDA_BF16)
        conv_decode_kernel<__nv_bfloat16><<<blocks, kConvThreads, 0, st>>>((const __nv_bfloat16 *)x, w, N, C, W, state,
                                                                           (__nv_bfloat16 *)y);
    else
        conv_decode_kernel<float><<<blocks, kConvThreads, 0, st>>>((const float *)x, w, N, C, W, state, (float *)y);
    return cudaGetLastError();
}

}  // namespace kda
