// kda_decode.cu -- fused recurrent decode step (one new token per sequence).
//
// Lecture 04, section 2: in decode the state is already in memory and one
// fused step is the natural operation.  Per (sequence, head):
//
//     S' = D S                 (D = diag(exp(g)), scales the d_k rows)
//     x  = S'^T k,  y = S'^T q
//     u  = beta (v - x)
//     S  = S' + k u^T          (= (I - beta k k^T) D S + beta k v^T)
//     o  = S^T q = y + (q . k) u
//
// The step is bound by HBM: the fp32 state is read once and written once and
// every other operand is tiny.  One CTA owns one (sequence, head) state; each
// warp owns a band of 16 rows and each lane four adjacent d_v columns, so a
// warp's row load is one contiguous 512-byte transaction (d = 128).  The
// band's 16 float4 loads are all issued before any arithmetic, the decayed
// band stays in registers, and the two d_k reductions (x, y) are finished
// through shared memory in a fixed order, so the result is deterministic.
// State traffic uses streaming (evict-first) loads and stores: the state is
// touched once per step and is far larger than L2.
//
// The indexed variant serves a batch that mixes request phases (Lecture 04,
// section 2: the decode family takes the sequences that are generating,
// while others are still in prefill): its states live in a pool of slots and
// an index list names the slot each active sequence's token updates.  Slots
// not named are not touched.  Two copy kernels take a snapshot of listed
// slots and put it back, which is what a speculative rollback needs
// (Lecture 11, section 2, "Serving state" row: rollback must reconcile the
// KDA state).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kRows = 16;  // rows of S per thread

// Sum of squares of x[0, n) by the 32 lanes of a warp (every lane gets it), or by one thread, in a fixed order.
__device__ __forceinline__ float warp_sum_squares(const float *x, int n, int lane) {
    float ss = 0.f;
    for (int i = lane; i < n; i += 32) ss = fmaf(x[i], x[i], ss);
#pragma unroll
    for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    return ss;
}
__device__ __forceinline__ float serial_sum_squares(const float *x, int n) {
    float ss = 0.f;
    for (int i = 0; i < n; ++i) ss = fmaf(x[i], x[i], ss);
    return ss;
}

// One CTA per (active sequence, head).  With `idx` null, sequence i's state is S[i]; otherwise it is the
// pool slot idx[i] (a slot outside [0, num_slots) is skipped and recorded in *status, when given).
template <typename Tin, int D>
__global__ void __launch_bounds__((D / 4) * (D / kRows))
decode_step_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                   const float *__restrict__ g, const float *__restrict__ beta, float *__restrict__ S,
                   Tin *__restrict__ o, const int32_t *__restrict__ idx, int H, int num_slots,
                   int32_t *__restrict__ status, int qk_norm, float qk_eps, const Tin *__restrict__ gate,
                   const float *__restrict__ weight, float out_eps) {
    constexpr int CG = D / 4;        // column groups (float4)
    constexpr int RG = D / kRows;    // row bands
    constexpr int NT = CG * RG;
    __shared__ float s_q[D], s_k[D], s_dec[D], s_u[D], s_o[D];
    __shared__ float s_x[RG][D], s_y[RG][D];
    __shared__ float s_qk, s_scale[2];

    const int head = blockIdx.x;  // flattened (active sequence, head): the token's inputs and output
    size_t state = (size_t)head;  // flattened (slot, head) of its state
    if (idx) {
        const int slot = idx[head / H];
        if (slot < 0 || slot >= num_slots) {
            if (status && threadIdx.x == 0) atomicCAS(status, 0, (int32_t)KDA_ERR_INVALID_ARG);
            return;
        }
        state = (size_t)slot * H + head % H;
    }
    const int tid = threadIdx.x;
    const int cg = tid % CG, rg = tid / CG;
    const size_t vec = (size_t)head * D;
    float4 *Sv = reinterpret_cast<float4 *>(S + state * D * D);

    // Issue the state loads first: they are the long pole.
    float4 s[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) s[j] = __ldcs(&Sv[(size_t)(rg * kRows + j) * CG + cg]);

    for (int i = tid; i < D; i += NT) {
        s_q[i] = to_f32(q[vec + i]);
        s_k[i] = to_f32(k[vec + i]);
        s_dec[i] = expf(g[vec + i]);
    }
    __syncthreads();
    if (qk_norm) {  // fused prologue: q, k L2-normalised in fp32 (warps 0 / 1, or threads 0 / 1 of a small block)
        if (NT >= 64 && tid < 64) {
            const float ss = warp_sum_squares(tid < 32 ? s_q : s_k, D, tid & 31);
            if ((tid & 31) == 0) s_scale[tid >> 5] = rsqrtf(ss + qk_eps);
        } else if (NT < 64 && tid < 2) {
            s_scale[tid] = rsqrtf(serial_sum_squares(tid ? s_k : s_q, D) + qk_eps);
        }
        __syncthreads();
        for (int i = tid; i < D; i += NT) {
            s_q[i] *= s_scale[0];
            s_k[i] *= s_scale[1];
        }
        __syncthreads();
    }
    if (NT >= 32 && tid < 32) {  // q . k by one warp (a fixed shuffle tree: deterministic)
        float acc = 0.f;
        for (int i = tid; i < D; i += 32) acc = fmaf(s_q[i], s_k[i], acc);
#pragma unroll
        for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (tid == 0) s_qk = acc;
    } else if (NT < 32 && tid == 0) {
        float acc = 0.f;
        for (int i = 0; i < D; ++i) acc = fmaf(s_q[i], s_k[i], acc);
        s_qk = acc;
    }

    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
        const int r = rg * kRows + j;
        const float d = s_dec[r], kr = s_k[r], qr = s_q[r];
        s[j].x *= d; s[j].y *= d; s[j].z *= d; s[j].w *= d;
        x.x = fmaf(kr, s[j].x, x.x); x.y = fmaf(kr, s[j].y, x.y);
        x.z = fmaf(kr, s[j].z, x.z); x.w = fmaf(kr, s[j].w, x.w);
        y.x = fmaf(qr, s[j].x, y.x); y.y = fmaf(qr, s[j].y, y.y);
        y.z = fmaf(qr, s[j].z, y.z); y.w = fmaf(qr, s[j].w, y.w);
    }
    *reinterpret_cast<float4 *>(&s_x[rg][cg * 4]) = x;
    *reinterpret_cast<float4 *>(&s_y[rg][cg * 4]) = y;
    __syncthreads();

    const float b = beta[head];
    for (int c = tid; c < D; c += NT) {
        float xs = 0.f, ys = 0.f;
#pragma unroll
        for (int r = 0; r < RG; ++r) { xs += s_x[r][c]; ys += s_y[r][c]; }
        const float u = b * (to_f32(v[vec + c]) - xs);
        s_u[c] = u;
        const float out = fmaf(s_qk, u, ys);
        if (gate) s_o[c] = out;
        else o[vec + c] = from_f32<Tin>(out);
    }
    __syncthreads();
    if (gate) {  // fused epilogue: o / rms(o) * w * sigmoid(z)
        if (NT >= 32 && tid < 32) {
            const float ss = warp_sum_squares(s_o, D, tid);
            if (tid == 0) s_scale[0] = rsqrtf(ss / (float)D + out_eps);
        } else if (NT < 32 && tid == 0) {
            s_scale[0] = rsqrtf(serial_sum_squares(s_o, D) / (float)D + out_eps);
        }
        __syncthreads();
        for (int c = tid; c < D; c += NT)
            o[vec + c] = from_f32<Tin>(s_o[c] * s_scale[0] * (weight ? weight[c] : 1.f) * sigmoidf(to_f32(gate[vec + c])));
    }

    const float4 u = *reinterpret_cast<const float4 *>(&s_u[cg * 4]);
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
        const float kr = s_k[rg * kRows + j];
        float4 n;
        n.x = fmaf(kr, u.x, s[j].x); n.y = fmaf(kr, u.y, s[j].y);
        n.z = fmaf(kr, u.z, s[j].z); n.w = fmaf(kr, u.w, s[j].w);
        __stcs(&Sv[(size_t)(rg * kRows + j) * CG + cg], n);
    }
}

// Copies whole (slot, head) states between a pool and a compact buffer: gather (snapshot) writes
// dst[i] = pool[idx[i]], scatter (restore) writes pool[idx[i]] = src[i].  One CTA per listed state, 16-byte
// streaming loads and stores; a slot outside [0, num_slots) is skipped and recorded in *status.
__global__ void __launch_bounds__(256)
state_copy_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst, const int32_t *__restrict__ idx,
                  int num_slots, int state_vec4, int scatter, int32_t *__restrict__ status) {
    const int i = blockIdx.x;
    const int slot = idx[i];
    if (slot < 0 || slot >= num_slots) {
        if (status && threadIdx.x == 0) atomicCAS(status, 0, (int32_t)KDA_ERR_INVALID_ARG);
        return;
    }
    const size_t from = (size_t)(scatter ? i : slot) * state_vec4, to = (size_t)(scatter ? slot : i) * state_vec4;
    for (int j = threadIdx.x; j < state_vec4; j += blockDim.x) __stcs(&dst[to + j], __ldcs(&src[from + j]));
}

template <typename Tin, int D>
cudaError_t launch_d(const void *q, const void *k, const void *v, const float *g, const float *beta, int heads,
                     float *S, void *o, const int32_t *idx, int H, int num_slots, int32_t *status, const Fusion &fu,
                     cudaStream_t st) {
    constexpr int NT = (D / 4) * (D / kRows);
    decode_step_kernel<Tin, D><<<heads, NT, 0, st>>>((const Tin *)q, (const Tin *)k, (const Tin *)v, g, beta, S,
                                                     (Tin *)o, idx, H, num_slots, status, fu.qk_norm, fu.qk_eps,
                                                     (const Tin *)fu.gate, fu.weight, fu.out_eps);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_t(const void *q, const void *k, const void *v, const float *g, const float *beta, int heads,
                     int d, float *S, void *o, const int32_t *idx, int H, int num_slots, int32_t *status,
                     const Fusion &fu, cudaStream_t st) {
    switch (d) {
        case 16: return launch_d<Tin, 16>(q, k, v, g, beta, heads, S, o, idx, H, num_slots, status, fu, st);
        case 64: return launch_d<Tin, 64>(q, k, v, g, beta, heads, S, o, idx, H, num_slots, status, fu, st);
        case 128: return launch_d<Tin, 128>(q, k, v, g, beta, heads, S, o, idx, H, num_slots, status, fu, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g, const float *beta,
                          int num_seqs, int H, int d, kda_dtype dt, float *S, void *o, const int32_t *idx,
                          int num_slots, int32_t *status, const Fusion &fu, cudaStream_t st) {
    const int heads = num_seqs * H;
    if (heads == 0) return cudaSuccess;
    if (dt == KDA_BF16)
        return launch_t<__nv_bfloat16>(q, k, v, g, beta, heads, d, S, o, idx, H, num_slots, status, fu, st);
    return launch_t<float>(q, k, v, g, beta, heads, d, S, o, idx, H, num_slots, status, fu, st);
}

cudaError_t launch_state_copy(const float *src, float *dst, const int32_t *idx, int n, int num_slots, int H, int d,
                              bool scatter, int32_t *status, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int state_vec4 = H * d * d / 4;  // one slot: all its heads
    state_copy_kernel<<<n, 256, 0, st>>>(reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst), idx,
                                         num_slots, state_vec4, scatter ? 1 : 0, status);
    return cudaGetLastError();
}

}  // namespace kda
