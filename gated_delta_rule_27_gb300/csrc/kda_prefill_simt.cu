// kda_prefill_simt.cu -- chunked prefill on the fp32 CUDA cores.
//
// This is the general path (fp32 inputs, d in {16, 64, 128}, chunk in
// {16, 32, 64}); bf16 inputs at d = 128 with 64-token chunks take the
// tensor-core path instead.  Both compute the same chunk algebra (Lecture 04,
// section 1: a chunk's effect on the incoming state is one affine update that
// can be formed without that state; the structured diagonal-plus-rank-one
// form is kept, no d_k x d_k matrix is formed):
//
// For the chunk's tokens r = 0..Lc-1 and the channel-wise cumulative
// log-decay b_r = sum_{s<=r} g_s,
//     A[r,s] = beta_r sum_c k_rc k_sc exp(b_rc - b_sc)   (s < r)
//     P[r,s] = sum_c q_rc k_sc exp(b_rc - b_sc)          (s <= r)
//     (I + A) [W | Ut] = diag(beta) [exp(b) * K | V]       (forward substitution)
//     Qp   = exp(b) * Q - P W,     Oloc = P Ut
//     Kend = exp(b_last - b) * K,  gamma = exp(b_last)
// and then, in order over the chunks of a document, with S the incoming state:
//     U = Ut - W S;   O = Qp S + Oloc;   S <- gamma * S + Kend^T U.
//
// Three kernels: (1) the chunk index (one CTA scans cu_seqlens), (2) the
// chunk-parallel pass, one CTA per (chunk, head), writing the state-free
// terms to the workspace, and (3) the state pass, one CTA per (document,
// head, 32-column tile of S), sequential over the document's chunks.  On this
// path every exp(b_r - b_s) is taken pairwise, so no factor can overflow
// whatever the gates.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------------------
// (1) chunk index: doc_slot0[i] = sum_{j<i} ceil(len_j / L), and validation of
// cu_seqlens.  On invalid input every document gets zero chunks and the
// status word is set, so the later kernels write nothing.  Zeroes the
// preparation's work counter in the workspace header, and `clear_vec` 16-byte
// words at `clear` (the progress flags of the chain and pipe plans) when asked
// to.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
chunk_index_kernel(const int32_t *__restrict__ cu, int num_seqs, int total_tokens, int L, int32_t *status,
                   int32_t *doc_slot0, int32_t *doc_order, uint4 *clear, int clear_vec, int fault) {
    constexpr int kOrderMax = 512;  // documents ranked by chunk count up to this many (else the given order)
    __shared__ int s_bad;
    __shared__ int s_warp[32];
    __shared__ int s_carry;
    __shared__ int s_cnt[kOrderMax];
    const int tid = threadIdx.x, nt = blockDim.x;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the next kernel may get ready meanwhile
    for (int i = tid; i < clear_vec; i += nt) clear[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        status[kPrepCounterWord] = 0;
        s_bad = (cu[0] != 0) || (cu[num_seqs] != total_tokens);
        s_carry = 0;
    }
    __syncthreads();
    for (int i = tid; i < num_seqs; i += nt)
        if (cu[i + 1] < cu[i]) s_bad = 1;
    __syncthreads();
    if (s_bad) {
        for (int i = tid; i <= num_seqs; i += nt) doc_slot0[i] = 0;
        if (tid == 0) *status = 1;
        return;
    }
    const int lane = tid & 31, warp = tid >> 5, nwarps = (nt + 31) >> 5;
    for (int base = 0; base < num_seqs; base += nt) {
        const int i = base + tid;
        const int c = i < num_seqs ? (cu[i + 1] - cu[i] + L - 1) / L : 0;
        int incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += n;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += n;
            }
            if (lane < nwarps) s_warp[lane] = w;  // inclusive warp totals
        }
        __syncthreads();
        const int before = s_carry + (warp ? s_warp[warp - 1] : 0);
        if (i < num_seqs) doc_slot0[i] = before + incl - c;
        __syncthreads();
        if (tid == 0) s_carry += s_warp[nwarps - 1];
        __syncthreads();
    }
    // Documents by descending chunk count (ties in document order): a pass whose chains run in several waves
    // then starts the longest ones first.
    if (num_seqs <= kOrderMax) {
        for (int i = tid; i < num_seqs; i += nt) s_cnt[i] = (cu[i + 1] - cu[i] + L - 1) / L;
        __syncthreads();
        for (int i = tid; i < num_seqs; i += nt) {
            const int ci = s_cnt[i];
            int rank = 0;
            for (int j = 0; j < num_seqs; ++j) {
                const int cj = s_cnt[j];
                rank += (cj > ci) || (cj == ci && j < i);
            }
            doc_order[rank] = i;
        }
    } else {
        for (int i = tid; i < num_seqs; i += nt) doc_order[i] = i;
    }
    if (tid == 0) {
        doc_slot0[num_seqs] = s_carry;
        *status = 0;
        status[1] = 0;
#ifdef KDA_DEBUG_BOUNDS
        // test hook of the bounds-checking build only: a chunk table that claims more chunks than exist, which
        // the later kernels' checks must catch (the release build ignores it)
        if (fault == kFaultChunkTable) doc_slot0[num_seqs] = s_carry + 1000;
#else
        (void)fault;
#endif
    }
}

// ---------------------------------------------------------------------------
// (2) chunk-parallel pass, one CTA per (chunk slot, head).
// ---------------------------------------------------------------------------
template <int D, int L>
struct PrepSmem {
    static constexpr int DP = D + 1;  // padded row stride (bank-conflict free column walks)
    static constexpr size_t q = 0;                             // [L][DP]  q, then exp(b) q, then Qp
    static constexpr size_t k = q + (size_t)L * DP;            // [L][DP]  k, then beta exp(b) k, then W
    static constexpr size_t b = k + (size_t)L * DP;            // [L][DP]  cumulative log-decay
    static constexpr size_t v = b + (size_t)L * DP;            // [L][D]   v, then beta v, then Ut
    static constexpr size_t A = v + (size_t)L * D;             // [L][L]
    static constexpr size_t P = A + (size_t)L * L;             // [L][L]
    static constexpr size_t beta = P + (size_t)L * L;          // [L]
    static constexpr size_t floats = beta + L;
    static constexpr size_t bytes = floats * 4;
};

template <typename Tin, int D, int L>
__global__ void __launch_bounds__(kThreads)
prefill_prepare_simt(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                     const float *__restrict__ g, const float *__restrict__ beta, const int32_t *__restrict__ cu,
                     int num_seqs, int H, char *__restrict__ ws, size_t doc_slot0_off, size_t records_off,
                     size_t record_bytes, int qk_norm, float qk_eps) {
    using SM = PrepSmem<D, L>;
    constexpr int DP = SM::DP;
    extern __shared__ float smem[];
    float *sq = smem + SM::q, *sk = smem + SM::k, *sb = smem + SM::b, *sv = smem + SM::v;
    float *sA = smem + SM::A, *sP = smem + SM::P, *sbeta = smem + SM::beta;

    const int slot = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int32_t *doc_slot0 = reinterpret_cast<const int32_t *>(ws + doc_slot0_off);
    int doc, t0, Lc;
    if (!locate_slot(doc_slot0, cu, num_seqs, L, slot, &doc, &t0, &Lc)) return;
    if (!KDA_IN_BOUNDS(slot < max_chunk_slots(cu, num_seqs, L) && t0 >= 0 && Lc >= 1 && Lc <= L &&
                           t0 + Lc <= cu[num_seqs],
                       reinterpret_cast<int32_t *>(ws)))
        return;
    const SimtRecord R = simt_record(L, D, D);
    char *rec = ws + records_off + ((size_t)slot * H + h) * record_bytes;
    float *gW = reinterpret_cast<float *>(rec + R.W), *gUt = reinterpret_cast<float *>(rec + R.Ut);
    float *gQp = reinterpret_cast<float *>(rec + R.Qp), *gOl = reinterpret_cast<float *>(rec + R.Oloc);
    float *gKe = reinterpret_cast<float *>(rec + R.Kend), *gGam = reinterpret_cast<float *>(rec + R.gamma);

    for (int i = tid; i < Lc * D; i += kThreads) {
        const int r = i / D, c = i % D;
        const size_t src = ((size_t)(t0 + r) * H + h) * D + c;
        sq[r * DP + c] = to_f32(q[src]);
        sk[r * DP + c] = to_f32(k[src]);
        sv[r * D + c] = to_f32(v[src]);
        sb[r * DP + c] = g[src];
    }
    for (int r = tid; r < Lc; r += kThreads) sbeta[r] = beta[(size_t)(t0 + r) * H + h];
    __syncthreads();
    if (qk_norm) {  // fused prologue: every q and k row L2-normalised in fp32, one warp per row
        const int lane = tid & 31;
        for (int rr = tid >> 5; rr < 2 * Lc; rr += kThreads / 32) {
            float *x = (rr < Lc ? sq : sk) + (rr % Lc) * DP;
            float ss = 0.f;
            for (int c = lane; c < D; c += 32) ss = fmaf(x[c], x[c], ss);
#pragma unroll
            for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = rsqrtf(ss + qk_eps);
            for (int c = lane; c < D; c += 32) x[c] *= inv;
        }
        __syncthreads();
    }
    for (int c = tid; c < D; c += kThreads) {  // in-chunk cumulative log-decay
        float acc = 0.f;
        for (int r = 0; r < Lc; ++r) { acc += sb[r * DP + c]; sb[r * DP + c] = acc; }
    }
    __syncthreads();

    // A (strictly lower) and P (lower, with diagonal), pairwise exp(b_r - b_s) <= 1.
    for (int p = tid; p < Lc * Lc; p += kThreads) {
        const int r = p / Lc, s = p % Lc;
        float a = 0.f, pq = 0.f;
        if (s <= r) {
            for (int c = 0; c < D; ++c) {
                const float e = expf(sb[r * DP + c] - sb[s * DP + c]);
                const float ks = sk[s * DP + c] * e;
                a = fmaf(sk[r * DP + c], ks, a);
                pq = fmaf(sq[r * DP + c], ks, pq);
            }
        }
        sA[r * L + s] = s < r ? sbeta[r] * a : 0.f;
        sP[r * L + s] = pq;
    }
    __syncthreads();

    // Kend, gamma straight to the record; then the right-hand sides in place.
    for (int i = tid; i < Lc * D; i += kThreads) {
        const int r = i / D, c = i % D;
        const float bl = sb[(Lc - 1) * DP + c], br = sb[r * DP + c];
        gKe[r * D + c] = expf(bl - br) * sk[r * DP + c];
    }
    for (int c = tid; c < D; c += kThreads) gGam[c] = expf(sb[(Lc - 1) * DP + c]);
    __syncthreads();
    for (int i = tid; i < Lc * D; i += kThreads) {
        const int r = i / D, c = i % D;
        const float e = expf(sb[r * DP + c]);
        sq[r * DP + c] *= e;
        sk[r * DP + c] *= e * sbeta[r];
        sv[r * D + c] *= sbeta[r];
    }
    __syncthreads();

    // Forward substitution (I + A) X = RHS, one column per thread, in place.
    for (int col = tid; col < 2 * D; col += kThreads) {
        float *X = col < D ? sk + col : sv + (col - D);
        const int stride = col < D ? DP : D;
        for (int r = 1; r < Lc; ++r) {
            float acc = X[r * stride];
            for (int s = 0; s < r; ++s) acc = fmaf(-sA[r * L + s], X[s * stride], acc);
            X[r * stride] = acc;
        }
    }
    __syncthreads();

    // Qp = exp(b) Q - P W (in place), Oloc = P Ut; store W, Ut, Qp, Oloc.
    for (int col = tid; col < 2 * D; col += kThreads) {
        if (col < D) {
            for (int r = 0; r < Lc; ++r) {
                float acc = sq[r * DP + col];
                for (int s = 0; s <= r; ++s) acc = fmaf(-sP[r * L + s], sk[s * DP + col], acc);
                gQp[r * D + col] = acc;
            }
        } else {
            const int c = col - D;
            for (int r = 0; r < Lc; ++r) {
                float acc = 0.f;
                for (int s = 0; s <= r; ++s) acc = fmaf(sP[r * L + s], sv[s * D + c], acc);
                gOl[r * D + c] = acc;
            }
        }
    }
    for (int i = tid; i < Lc * D; i += kThreads) {
        const int r = i / D, c = i % D;
        gW[r * D + c] = sk[r * DP + c];
        gUt[r * D + c] = sv[r * D + c];
    }
}

// ---------------------------------------------------------------------------
// (3) state pass, one CTA per (document, head, column tile).
// ---------------------------------------------------------------------------
template <int D, int L, int TILE>
struct StateSmem {
    static constexpr int DP = D + 1;
    static constexpr size_t S = 0;                        // [D][TILE]
    static constexpr size_t W = S + (size_t)D * TILE;     // [L][DP]
    static constexpr size_t Q = W + (size_t)L * DP;       // [L][DP]
    static constexpr size_t Ke = Q + (size_t)L * DP;      // [L][DP]
    static constexpr size_t Ut = Ke + (size_t)L * DP;     // [L][TILE]
    static constexpr size_t Ol = Ut + (size_t)L * TILE;   // [L][TILE]
    static constexpr size_t U = Ol + (size_t)L * TILE;    // [L][TILE]
    static constexpr size_t gam = U + (size_t)L * TILE;   // [D]
    static constexpr size_t bytes = (gam + D) * 4;
};

template <typename Tout, int D, int L, int TILE>
__global__ void __launch_bounds__(kThreads)
prefill_state_simt(const int32_t *__restrict__ cu, int num_seqs, int H, const float *__restrict__ S0,
                   Tout *__restrict__ o, float *__restrict__ S_final, const char *__restrict__ ws,
                   size_t doc_slot0_off, size_t records_off, size_t record_bytes) {
    using SM = StateSmem<D, L, TILE>;
    constexpr int DP = SM::DP, NTILE = D / TILE;
    extern __shared__ float smem[];
    float *sS = smem + SM::S, *sW = smem + SM::W, *sQ = smem + SM::Q, *sKe = smem + SM::Ke;
    float *sUt = smem + SM::Ut, *sOl = smem + SM::Ol, *sU = smem + SM::U, *sG = smem + SM::gam;

    if (*reinterpret_cast<const int32_t *>(ws) != 0) return;  // invalid cu_seqlens: write nothing
    const int tile = blockIdx.x % NTILE;
    const int h = (blockIdx.x / NTILE) % H;
    const int n = blockIdx.x / (NTILE * H);
    const int tid = threadIdx.x;
    const int col0 = tile * TILE;
    const int32_t *doc_slot0 = reinterpret_cast<const int32_t *>(ws + doc_slot0_off);
    const SimtRecord R = simt_record(L, D, D);
    const size_t state_off = ((size_t)n * H + h) * D * D;

    for (int i = tid; i < D * TILE; i += kThreads) {
        const int c = i / TILE, j = i % TILE;
        sS[i] = S0 ? S0[state_off + (size_t)c * D + col0 + j] : 0.f;
    }
    const int first = doc_slot0[n], last = doc_slot0[n + 1];
    if (!KDA_IN_BOUNDS(first >= 0 && last >= first && last <= max_chunk_slots(cu, num_seqs, L),
                       reinterpret_cast<int32_t *>(const_cast<char *>(ws))))
        return;
    for (int slot = first; slot < last; ++slot) {
        const int t0 = cu[n] + (slot - first) * L;
        const int Lc = min(L, cu[n + 1] - t0);
        const char *rec = ws + records_off + ((size_t)slot * H + h) * record_bytes;
        const float *gW = reinterpret_cast<const float *>(rec + R.W);
        const float *gUt = reinterpret_cast<const float *>(rec + R.Ut);
        const float *gQp = reinterpret_cast<const float *>(rec + R.Qp);
        const float *gOl = reinterpret_cast<const float *>(rec + R.Oloc);
        const float *gKe = reinterpret_cast<const float *>(rec + R.Kend);
        const float *gGam = reinterpret_cast<const float *>(rec + R.gamma);
        __syncthreads();  // previous chunk's readers are done with the staging buffers
        for (int i = tid; i < Lc * D; i += kThreads) {
            const int r = i / D, c = i % D;
            sW[r * DP + c] = gW[i];
            sQ[r * DP + c] = gQp[i];
            sKe[r * DP + c] = gKe[i];
        }
        for (int i = tid; i < Lc * TILE; i += kThreads) {
            const int r = i / TILE, j = i % TILE;
            sUt[i] = gUt[r * D + col0 + j];
            sOl[i] = gOl[r * D + col0 + j];
        }
        for (int c = tid; c < D; c += kThreads) sG[c] = gGam[c];
        __syncthreads();
        for (int i = tid; i < Lc * TILE; i += kThreads) {
            const int r = i / TILE, j = i % TILE;
            float x = 0.f, y = 0.f;
            for (int c = 0; c < D; ++c) {
                const float s = sS[c * TILE + j];
                x = fmaf(sW[r * DP + c], s, x);
                y = fmaf(sQ[r * DP + c], s, y);
            }
            sU[i] = sUt[i] - x;
            if (KDA_IN_BOUNDS(t0 + r < cu[num_seqs], reinterpret_cast<int32_t *>(const_cast<char *>(ws))))
                o[((size_t)(t0 + r) * H + h) * D + col0 + j] = from_f32<Tout>(y + sOl[i]);
        }
        __syncthreads();
        for (int i = tid; i < D * TILE; i += kThreads) {
            const int c = i / TILE, j = i % TILE;
            float acc = sG[c] * sS[i];
            for (int r = 0; r < Lc; ++r) acc = fmaf(sKe[r * DP + c], sU[r * TILE + j], acc);
            sS[i] = acc;
        }
    }
    __syncthreads();
    if (S_final) {
        for (int i = tid; i < D * TILE; i += kThreads) {
            const int c = i / TILE, j = i % TILE;
            S_final[state_off + (size_t)c * D + col0 + j] = sS[i];
        }
    }
}

// ---------------------------------------------------------------------------
// (4) the fused epilogue's gated output normalisation, on this path a pass of its own (the state pass writes
// each row of o in column tiles from several CTAs): o <- o / rms(o) * w * sigmoid(z), one warp per row.
// ---------------------------------------------------------------------------
template <typename Tout, int D>
__global__ void __launch_bounds__(kThreads)
out_gated_norm_kernel(Tout *__restrict__ o, const Tout *__restrict__ gate, const float *__restrict__ weight,
                      float eps, int rows) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    constexpr int PER = (D + 31) / 32;
    float x[PER];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int c = lane + 32 * j;
        x[j] = c < D ? to_f32(o[(size_t)row * D + c]) : 0.f;
        ss = fmaf(x[j], x[j], ss);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float scale = rsqrtf(ss / (float)D + eps);
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int c = lane + 32 * j;
        if (c < D)
            o[(size_t)row * D + c] =
                from_f32<Tout>(x[j] * scale * (weight ? weight[c] : 1.f) * sigmoidf(to_f32(gate[(size_t)row * D + c])));
    }
}

template <typename Tin, int D, int L>
cudaError_t launch_dl(const void *q, const void *k, const void *v, const float *g, const float *beta,
                      const int32_t *cu, int num_seqs, int total_tokens, int H, const float *S0, void *o,
                      float *S_final, void *ws, const Fusion &fu, cudaStream_t st, Marks &marks) {
    constexpr int TILE = D < 32 ? D : 32;
    const WsLayout lay = ws_layout(total_tokens, num_seqs, H, D, D, L, PATH_SIMT);
    char *w = static_cast<char *>(ws);
    cudaError_t e;
    if (lay.max_slots > 0 && total_tokens > 0) {
        auto prep = prefill_prepare_simt<Tin, D, L>;
        const size_t sm_prep = PrepSmem<D, L>::bytes;
        if ((e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_prep)))
            return e;
        dim3 grid((unsigned)lay.max_slots, (unsigned)H);
        marks.before(st, "prefill_prepare_simt");
        prep<<<grid, kThreads, sm_prep, st>>>((const Tin *)q, (const Tin *)k, (const Tin *)v, g, beta, cu,
                                              num_seqs, H, w, lay.doc_slot0_off, lay.records_off,
                                              lay.record_bytes, fu.qk_norm, fu.qk_eps);
        if ((e = cudaGetLastError())) return e;
    }
    if (num_seqs == 0) return cudaSuccess;
    auto state = prefill_state_simt<Tin, D, L, TILE>;
    const size_t sm_state = StateSmem<D, L, TILE>::bytes;
    if ((e = cudaFuncSetAttribute(state, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_state))) return e;
    const unsigned blocks = (unsigned)((size_t)num_seqs * H * (D / TILE));
    marks.before(st, "prefill_state_simt");
    state<<<blocks, kThreads, sm_state, st>>>(cu, num_seqs, H, S0, (Tin *)o, S_final, w, lay.doc_slot0_off,
                                              lay.records_off, lay.record_bytes);
    if ((e = cudaGetLastError())) return e;
    if (fu.gate && total_tokens > 0) {
        const int rows = total_tokens * H;
        marks.before(st, "out_gated_norm");
        out_gated_norm_kernel<Tin, D><<<(rows + kThreads / 32 - 1) / (kThreads / 32), kThreads, 0, st>>>(
            (Tin *)o, (const Tin *)fu.gate, fu.weight, fu.out_eps, rows);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

template <typename Tin, int D>
cudaError_t launch_d(const void *q, const void *k, const void *v, const float *g, const float *beta,
                     const int32_t *cu, int num_seqs, int total_tokens, int H, int L, const float *S0, void *o,
                     float *S_final, void *ws, const Fusion &fu, cudaStream_t st, Marks &marks) {
    switch (L) {
        case 16: return launch_dl<Tin, D, 16>(q, k, v, g, beta, cu, num_seqs, total_tokens, H, S0, o, S_final, ws, fu, st, marks);
        case 32: return launch_dl<Tin, D, 32>(q, k, v, g, beta, cu, num_seqs, total_tokens, H, S0, o, S_final, ws, fu, st, marks);
        case 64: return launch_dl<Tin, D, 64>(q, k, v, g, beta, cu, num_seqs, total_tokens, H, S0, o, S_final, ws, fu, st, marks);
        default: return cudaErrorInvalidValue;
    }
}

template <typename Tin>
cudaError_t launch_t(const void *q, const void *k, const void *v, const float *g, const float *beta,
                     const int32_t *cu, int num_seqs, int total_tokens, int H, int d, int L, const float *S0,
                     void *o, float *S_final, void *ws, const Fusion &fu, cudaStream_t st, Marks &marks) {
    switch (d) {
        case 16: return launch_d<Tin, 16>(q, k, v, g, beta, cu, num_seqs, total_tokens, H, L, S0, o, S_final, ws, fu, st, marks);
        case 64: return launch_d<Tin, 64>(q, k, v, g, beta, cu, num_seqs, total_tokens, H, L, S0, o, S_final, ws, fu, st, marks);
        case 128: return launch_d<Tin, 128>(q, k, v, g, beta, cu, num_seqs, total_tokens, H, L, S0, o, S_final, ws, fu, st, marks);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_chunk_index(const int32_t *cu, int num_seqs, int total_tokens, int L, void *ws, void *clear,
                               size_t clear_bytes, cudaStream_t st, Marks &marks) {
    const int fault = testing_fault();
    char *w = static_cast<char *>(ws);
    const size_t doc_off = 256;  // (as ws_layout places the chunk table and the document order)
    const size_t order_off = doc_off + align256((size_t)(num_seqs + 1) * 4);
    const int clear_vec = (int)(clear_bytes / 16);
    const int busy = num_seqs > clear_vec ? num_seqs : clear_vec;
    const int threads = busy >= 512 ? 1024 : (busy >= 128 ? 256 : 64);
    marks.before(st, "chunk_index");
    chunk_index_kernel<<<1, threads, 0, st>>>(cu, num_seqs, total_tokens, L, reinterpret_cast<int32_t *>(w),
                                              reinterpret_cast<int32_t *>(w + doc_off),
                                              reinterpret_cast<int32_t *>(w + order_off), static_cast<uint4 *>(clear),
                                              clear_vec, fault);
    return cudaGetLastError();
}

cudaError_t launch_prefill_simt(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                const int32_t *cu, int num_seqs, int total_tokens, int H, int d, kda_dtype dt,
                                int L, const float *S0, void *o, float *S_final, void *ws, const Fusion &fu,
                                cudaStream_t st, Marks &marks) {
    if (dt == KDA_BF16)
        return launch_t<__nv_bfloat16>(q, k, v, g, beta, cu, num_seqs, total_tokens, H, d, L, S0, o, S_final, ws, fu,
                                       st, marks);
    return launch_t<float>(q, k, v, g, beta, cu, num_seqs, total_tokens, H, d, L, S0, o, S_final, ws, fu, st, marks);
}

}  // namespace kda
