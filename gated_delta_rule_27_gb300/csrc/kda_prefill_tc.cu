// kda_prefill_tc.cu -- chunked prefill on the Blackwell tensor cores (tcgen05),
// bf16 inputs, d_k = d_v = 128, 64-token chunks.
//
// Chunk algebra (Lecture 04, section 1: a chunk's effect on the incoming state
// is one affine update formed without that state).  With b_r = sum_{s<=r} g_s
// per channel, a reference point b_m and X_k = beta k exp(b - b_m),
// X_q = q exp(b - b_m), Kend = k exp(b_last - b):
//     A[r,s] = beta_r sum_c k_rc k_sc exp(b_rc - b_sc)  (s < r)
//     P[r,s] = sum_c q_rc k_sc exp(b_rc - b_sc)         (s <= r)
//     T = (I + A)^{-1},  W' = T X_k,  Ut = T (beta V)
//     Qp = (X_q - P W') exp(b_m),  M' = -Kend^T W' exp(b_m),  gamma = exp(b_last)
// and per document, chunk after chunk, with S_c the state entering chunk c:
//     S_{c+1} = gamma S_c + M' S_c + Kend^T Ut,      O_c = Qp S_c + P Ut.
//
// Preparation, prefill_prepare_tc: one unit per (chunk, head), 256 threads
// (two units per SM).  q, k, v, g tiles arrive by TMA.  The dense contractions
// run as three rounds of tcgen05.mma with fp32 accumulators in TMEM (A and P;
// W' and Ut; Qp and M'); the gates, their cumulative sums and the triangular
// solve stay fp32 on the CUDA cores, and nothing d_k x d_k is formed from a
// single token.  b_m is the chunk's middle token, so every factor is bounded
// by exp(+-80) while the chunk's log-decay range on each side of m stays
// within 80; a chunk outside that range takes exact pairwise exponentials for
// A and P and reference 0 instead.  Every result is written to the chunk's
// workspace record as a ready shared-memory image.
//
// State pass: one CTA per (document, head, 32- or 64-column tile of S),
// sequential over the document's chunks: per chunk one MMA group M' S on top
// of Kend^T Ut (issued one chunk ahead, off the chain's critical path), S kept
// fp32 in registers, its bf16 image in shared memory feeding the next MMA and
// copied to the chunk's record.
//
// Output: per (chunk, head), O = Qp S_c + P Ut from the record, written as
// bf16 (optionally through the fused gated RMS normalisation).
//
// Launch plans (host side, below): three kernels; the preparation then one
// cooperative launch of chains beside output groups (chain); or one
// cooperative launch of chains beside groups that prepare and then form
// outputs (pipe).  Every mbarrier and flag wait is bounded: on expiry the
// kernel records KDA_ERR_TIMEOUT in the workspace status word and stops.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <mutex>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int kD = 128, kL = 64, kTile = 32, kNTile = kD / kTile;
constexpr float kMaxHalfRange = 80.f;  // |b_r - b_m| bound of the tensor-core A/P path
constexpr uint64_t kFlagWaitNs = 2000000000ull;  // default bound of a wait on another CTA's publication flag
constexpr int kFaultNoPublish = 1;  // test-only: the chain plan publishes no state image

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ float bf16_at(const uint8_t *p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}
__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    const uint32_t a = tc::smem_u32(p);
    return p + (((a + 1023u) & ~1023u) - a);
}
// tcgen05.ld is warp-collective (.sync.aligned): every TMEM load below runs
// under a warp-uniform condition, and per-lane conditions only guard stores.
__device__ __forceinline__ bool warp_all(bool b) { return __all_sync(0xffffffffu, b); }
// 2^x by the hardware's approximate base-2 exponential (a few ulp; subnormal results flushed to zero)
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;
// Records a timed-out wait in the workspace status word (first writer wins), once the chunk index kernel,
// which writes that word, is complete (a thread that started before it waits for it here).
__device__ __forceinline__ void flag_timeout(char *ws) {
    tc::grid_dep_wait();
    atomicCAS(reinterpret_cast<int32_t *>(ws), 0, (int32_t)KDA_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Kernel 1: chunk-parallel preparation
// ---------------------------------------------------------------------------
// Compact block-major lower triangle of a 64 x 64 fp32 matrix: the ten
// 16 x 16 blocks (i, j), j <= i, each contiguous.
__device__ __forceinline__ int tri_blk(int i, int j) { return ((i * (i + 1)) / 2 + j) << 8; }
__device__ __forceinline__ int tri_idx(int r, int s) { return tri_blk(r >> 4, s >> 4) + ((r & 15) << 4) + (s & 15); }
// Cumulative log-decay b[r][c] lives in a [64][128] fp32 array.  Within row r,
// channel c sits in half h = (c / 4) mod 2 at position (c / 8) * 4 + c mod 4,
// rotated by 16 h inside the half: a warp writing 32 consecutive channels of
// one row, and eight threads reading one float4 each of eight consecutive
// channel octets, both touch 32 distinct banks.
__device__ __forceinline__ int bswz(int r, int c) {
    const int hf = (c >> 2) & 1;
    return r * kD + hf * 64 + ((((c >> 3) << 2) + (c & 3) + 16 * hf) & 63);
}

constexpr int kPrepThreads = 256;

struct PrepSmem {
    // X: two 16 KB panels (channels 0-63, 64-127); in each, rows 0-63 hold the k
    // tile and rows 64-127 the q tile (128-byte swizzled), so that after the
    // in-place scaling X is round 1's A operand, its k rows (panel stride
    // 16 KB) are round 2's MN-major A operand and its q rows round 3's.
    static constexpr uint32_t X = 0;
    static constexpr uint32_t V = 32768;   // v tile (MN-major) as loaded; then Ut^T, K-major [j][s]
    static constexpr uint32_t G = 49152;   // g fp32 [64][128] -> b (swizzled); then A, T, T(bf16); then Kend, W'^T
    static constexpr uint32_t Y = 81920;   // round-1 B operand (k / e1); then P (8 KB)
    static constexpr uint32_t Afp = G;             // compact fp32 A (10 KB)
    static constexpr uint32_t Tfp = G + 10240;     // compact fp32 T (10 KB)
    static constexpr uint32_t Scr = G + 20480;     // the solve's scratch (6 KB)
    static constexpr uint32_t Tb = Y + 8192;       // bf16 T diag(beta), K-major [r][s] (8 KB), written by the solve
    static constexpr uint32_t KendS = G;           // Kend, MN-major [s][c] (16 KB)
    static constexpr uint32_t WT = G + 16384;      // W'^T, K-major [c][s] (16 KB)
    static constexpr uint32_t P = Y;               // P, K-major [r][s] (8 KB)
    static constexpr uint32_t bytes = 98304;
};

// The 256 threads that run one preparation unit: the whole CTA (bar 0, __syncthreads), or one of two groups
// of a 512-thread CTA synchronised by named barrier `bar`; `tid` is the thread's index within the group.
// A group's warps are numbered from its first warp, whose index is a multiple of 4, so a warp's TMEM lane
// quarter (physical warp index mod 4) is its group-relative index mod 4.
struct PrepGroup {
    int tid;
    uint32_t bar;
    __device__ __forceinline__ void sync() const {
        if (bar == 0) __syncthreads();
        else tc::named_barrier(bar, kPrepThreads);
    }
    // barrier that also returns whether `pred` held for any thread of the group
    __device__ __forceinline__ bool sync_or(bool pred) const {
        if (bar == 0) return __syncthreads_or(pred) != 0;
        uint32_t r;
        asm volatile(
            "{\n"
            ".reg .pred p, q;\n"
            "setp.ne.u32 p, %1, 0;\n"
            "bar.red.or.pred q, %2, %3, p;\n"
            "selp.u32 %0, 1, 0, q;\n"
            "}\n"
            : "=r"(r)
            : "r"((uint32_t)pred), "r"(bar), "r"((uint32_t)kPrepThreads)
            : "memory");
        return r != 0;
    }
};

// Per-unit scratch of a preparation group (small per-channel and per-row vectors, outside the big tiles).
struct PrepShared {
    __align__(16) float beta[kL];
    __align__(16) float bm[kD];  // per-channel reference, exp factors (16-byte aligned for float4 reads)
    __align__(16) float F[kD];
    __align__(16) float Em[kD];
    __align__(16) float blast[kD];
    float half[kD], gabs[2][kD];
    float invk[kL], invq[kL];
    int abort;
};

// The 64 x 64 bf16 identity, K-major [r][r'] with the 128-byte swizzle (8 KB): round 3's operand that adds X_q.
// Written once per CTA (by its `n` threads) into a region no unit overwrites.
constexpr uint32_t kIdentBytes = 8192;
__device__ __forceinline__ void write_identity(uint8_t *id, int tid, int n) {
    for (int e = tid; e < 64 * 8; e += n) {  // 16-byte chunk e: row e / 8, columns 8 (e % 8) ..
        const int r = e >> 3, s0 = (e & 7) * 8;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if ((r >> 3) == (e & 7)) {  // the chunk holding (r, r)
            const uint32_t one = 0x3f80u << (16 * (r & 1));
            const int word = (r & 7) >> 1;
            w.x = word == 0 ? one : 0u;
            w.y = word == 1 ? one : 0u;
            w.z = word == 2 ? one : 0u;
            w.w = word == 3 ? one : 0u;
        }
        *reinterpret_cast<uint4 *>(id + tc::sw128_offset(r, s0)) = w;
    }
}

// T = (I + A)^{-1} for A strictly lower triangular (compact block-major, four
// 16-row blocks), 256 threads.  The diagonal blocks are inverted by forward
// substitution; then, with L = I + A split into 32-row halves
// [[L_lo, 0], [A_hl, L_hi]], each half's lower block is -T_ii A_ij T_jj and
// the lower-left quarter is -T_hi (A_hl T_lo): four phases of 256 equal items.
// Each block of T diag(beta) also goes, in bf16, to the K-major [r][s] image Tb
// (round 2's B operand) in the first phase after it is final; the blocks above
// the diagonal are zeroed there while the diagonal blocks are being solved.
__device__ void unit_lower_inverse(const float *A, float *T, float *scr, uint8_t *Tb, const float *s_beta,
                                   const PrepGroup &grp) {
    const int tid = grp.tid;
    // bf16 (T[r][s] beta_s, T[r][s+1] beta_{s+1}) as one 32-bit word of the image
    auto tb2 = [&](int r, int s, float a, float b) {
        *reinterpret_cast<uint32_t *>(Tb + tc::sw128_offset(r, s)) = pack_bf16x2(a * s_beta[s], b * s_beta[s + 1]);
    };
    if (tid >= 64) {  // the image's blocks above the diagonal: 16-byte units 2.. of rows 0-15, 4.. of rows
                      // 16-31, 6, 7 of rows 32-47: one per thread
        const int t = tid - 64;
        const int r = t < 96 ? t / 6 : (t < 160 ? 16 + (t - 96) / 4 : 32 + (t - 160) / 2);
        const int u = t < 96 ? 2 + t % 6 : (t < 160 ? 4 + (t - 96) % 4 : 6 + (t - 160) % 2);
        *reinterpret_cast<uint4 *>(Tb + (uint32_t)r * 128u + ((uint32_t)(u ^ (r & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (tid < 64) {  // diagonal block blk, column j: (I + A_bb) x = e_j
        const int blk = tid >> 4, j = tid & 15;
        const float *Ab = A + tri_blk(blk, blk);
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int s4 = 0; 4 * s4 < r; ++s4) {  // the row's entries left of the diagonal, four per load
                const float4 av = *reinterpret_cast<const float4 *>(Ab + (r << 4) + 4 * s4);
                a0 = fmaf(av.x, x[4 * s4], a0);
                if (4 * s4 + 1 < r) a1 = fmaf(av.y, x[4 * s4 + 1], a1);
                if (4 * s4 + 2 < r) a0 = fmaf(av.z, x[4 * s4 + 2], a0);
                if (4 * s4 + 3 < r) a1 = fmaf(av.w, x[4 * s4 + 3], a1);
            }
            x[r] = r < j ? 0.f : (r == j ? 1.f : -(a0 + a1));
        }
        float *Td = T + tri_blk(blk, blk);
#pragma unroll
        for (int r = 0; r < 16; ++r) Td[(r << 4) + j] = x[r];
    }
    grp.sync();
    {  // the diagonal blocks' image: item (block, row, four columns)
        const int blk = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
        const float4 t = *reinterpret_cast<const float4 *>(T + tri_blk(blk, blk) + (r << 4) + c4);
        tb2(16 * blk + r, 16 * blk + c4, t.x, t.y);
        tb2(16 * blk + r, 16 * blk + c4 + 2, t.z, t.w);
    }
    {  // F = T_ii A_{i,i-1} for i = 1, 3 (scratch blocks 0, 1): item (b, row, column pair)
        const int b = tid >> 7, r = (tid >> 3) & 15, c2 = (tid & 7) * 2, i = 1 + 2 * b;
        const float *Ti = T + tri_blk(i, i) + (r << 4);
        const float *Ai = A + tri_blk(i, i - 1) + c2;
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(Ti + k4);
            const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 a = *reinterpret_cast<const float2 *>(Ai + ((k4 + u) << 4));
                acc.x = fmaf(tv[u], a.x, acc.x);
                acc.y = fmaf(tv[u], a.y, acc.y);
            }
        }
        *reinterpret_cast<float2 *>(scr + (b << 8) + (r << 4) + c2) = acc;
    }
    grp.sync();
    {  // T_{i,i-1} = -F T_{i-1,i-1}
        const int b = tid >> 7, r = (tid >> 3) & 15, c2 = (tid & 7) * 2, i = 1 + 2 * b;
        const float *F = scr + (b << 8) + (r << 4);
        const float *Tj = T + tri_blk(i - 1, i - 1) + c2;
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
            const float4 f = *reinterpret_cast<const float4 *>(F + k4);
            const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 t = *reinterpret_cast<const float2 *>(Tj + ((k4 + u) << 4));
                acc.x = fmaf(fv[u], t.x, acc.x);
                acc.y = fmaf(fv[u], t.y, acc.y);
            }
        }
        *reinterpret_cast<float2 *>(T + tri_blk(i, i - 1) + (r << 4) + c2) = make_float2(-acc.x, -acc.y);
        tb2(16 * i + r, 16 * (i - 1) + c2, -acc.x, -acc.y);
    }
    grp.sync();
    {  // X_ij = sum_{k=j}^{1} A_ik T_kj, (i, j) in {2, 3} x {0, 1} (scratch blocks 2..5): item (i, row, column
       // pair) forms X_i0 (two block products) and X_i1 (one), the same work for every thread
        const int i = 2 + (tid >> 7), r = (tid >> 3) & 15, c2 = (tid & 7) * 2;
        const float *A0 = A + tri_blk(i, 0) + (r << 4), *A1 = A + tri_blk(i, 1) + (r << 4);
        const float *T00 = T + tri_blk(0, 0) + c2, *T10 = T + tri_blk(1, 0) + c2, *T11 = T + tri_blk(1, 1) + c2;
        float2 x0 = make_float2(0.f, 0.f), x1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {  // k = 0 for X_i0, k = 1 for X_i1
            const float4 a0 = *reinterpret_cast<const float4 *>(A0 + k4);
            const float4 a1 = *reinterpret_cast<const float4 *>(A1 + k4);
            const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 t0 = *reinterpret_cast<const float2 *>(T00 + ((k4 + u) << 4));
                const float2 t1 = *reinterpret_cast<const float2 *>(T11 + ((k4 + u) << 4));
                x0.x = fmaf(av0[u], t0.x, x0.x); x0.y = fmaf(av0[u], t0.y, x0.y);
                x1.x = fmaf(av1[u], t1.x, x1.x); x1.y = fmaf(av1[u], t1.y, x1.y);
            }
        }
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {  // k = 1 for X_i0
            const float4 a1 = *reinterpret_cast<const float4 *>(A1 + k4);
            const float av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 t = *reinterpret_cast<const float2 *>(T10 + ((k4 + u) << 4));
                x0.x = fmaf(av1[u], t.x, x0.x); x0.y = fmaf(av1[u], t.y, x0.y);
            }
        }
        float *Xi = scr + 512 + (((i - 2) << 1) << 8) + (r << 4) + c2;
        *reinterpret_cast<float2 *>(Xi) = x0;
        *reinterpret_cast<float2 *>(Xi + 256) = x1;
    }
    grp.sync();
    {  // T_ij = -sum_{k=2}^{i} T_ik X_kj: item (j, row, column pair) forms T_2j (one block product) and T_3j
       // (two), the same work for every thread; only their image is needed
        const int j = tid >> 7, r = (tid >> 3) & 15, c2 = (tid & 7) * 2;
        const float *T22 = T + tri_blk(2, 2) + (r << 4), *T32 = T + tri_blk(3, 2) + (r << 4);
        const float *T33 = T + tri_blk(3, 3) + (r << 4);
        const float *X2 = scr + 512 + (j << 8) + c2, *X3 = scr + 512 + ((2 + j) << 8) + c2;
        float2 y2 = make_float2(0.f, 0.f), y3 = make_float2(0.f, 0.f);
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {  // k = 2
            const float4 ta = *reinterpret_cast<const float4 *>(T22 + k4);
            const float4 tb = *reinterpret_cast<const float4 *>(T32 + k4);
            const float tv2[4] = {ta.x, ta.y, ta.z, ta.w}, tv3[4] = {tb.x, tb.y, tb.z, tb.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 x = *reinterpret_cast<const float2 *>(X2 + ((k4 + u) << 4));
                y2.x = fmaf(tv2[u], x.x, y2.x); y2.y = fmaf(tv2[u], x.y, y2.y);
                y3.x = fmaf(tv3[u], x.x, y3.x); y3.y = fmaf(tv3[u], x.y, y3.y);
            }
        }
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {  // k = 3
            const float4 tc4 = *reinterpret_cast<const float4 *>(T33 + k4);
            const float tv[4] = {tc4.x, tc4.y, tc4.z, tc4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 x = *reinterpret_cast<const float2 *>(X3 + ((k4 + u) << 4));
                y3.x = fmaf(tv[u], x.x, y3.x); y3.y = fmaf(tv[u], x.y, y3.y);
            }
        }
        tb2(32 + r, 16 * j + c2, -y2.x, -y2.y);
        tb2(48 + r, 16 * j + c2, -y3.x, -y3.y);
    }
    tc::fence_async_smem();  // the image is an MMA operand
    tc::tc_fence_before();
    grp.sync();
}

// Exact A and P on the CUDA cores for a chunk whose log-decay range is too
// wide for the factorised tensor-core form: pairwise exp(b_r - b_s) <= 1
// (s <= r).  Thread t owns row r = t / 4 and the 16 columns s of quarter t % 4.
__device__ void exact_ap(const uint8_t *X, const float *B, const float *s_beta, int Lc, int tid, float (&accA)[16],
                         float (&accP)[16], const float *invk, const float *invq) {
    const int r = tid >> 2, s0 = (tid & 3) * 16;
#pragma unroll
    for (int j = 0; j < 16; ++j) { accA[j] = 0.f; accP[j] = 0.f; }
    if (r >= Lc) return;
    // with the fused q / k normalisation, row norms enter as factors: k_r . k_s -> (k_r . k_s) ik_r ik_s
    const float ikr = invk ? invk[r] : 1.f, iqr = invq ? invq[r] : 1.f;
    for (int c = 0; c < kD; ++c) {
        const uint8_t *panel = X + (uint32_t)(c >> 6) * 16384u;
        const float brc = B[bswz(r, c)];
        const float krc = bf16_at(panel + tc::sw128_offset(r, c & 63));
        const float qrc = bf16_at(panel + tc::sw128_offset(64 + r, c & 63));
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int s = s0 + j;
            if (s <= r) {
                const float ks = bf16_at(panel + tc::sw128_offset(s, c & 63)) * expf(brc - B[bswz(s, c)]);
                accA[j] = fmaf(krc, ks, accA[j]);
                accP[j] = fmaf(qrc, ks, accP[j]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float iks = invk ? invk[s0 + j] : 1.f;
        accA[j] *= s_beta[r] * ikr * iks;
        accP[j] *= iqr * iks;
    }
}

__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8]) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(h[i]);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
    }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}
__device__ __forceinline__ uint4 pack8_at(const float *f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// Roles (256 threads).  Channel-wise steps: thread t <-> channel t % 128 and
// half t / 128 of the chunk's rows.  Row-wise steps: thread t <-> token row
// t / 4 and channel quarter t % 4.  TMEM epilogues: warp w reads lanes
// 32 (w % 4) .. + 31 (channel or token rows), warps w and w + 4 splitting the
// accumulator's columns.  MMAs are issued by lane 0 of warps 0 and 1.
struct PrepParams {
    const CUtensorMap *tm_q, *tm_k, *tm_v, *tm_g;  // tensor maps in kernel-parameter space
    const float *beta;
    const int32_t *cu;
    int num_seqs, H;
    char *ws;
    size_t doc_slot0_off, records_off, record_bytes;
    int qk_norm;     // fused prologue: q and k rows L2-normalised (x / sqrt(sum x^2 + qk_eps)) as they are read
    float qk_eps;
};
// mbarriers of one preparation, each completing exactly once per unit: the gate tile, the k, q, v
// tiles, and the three MMA rounds
struct PrepBars {
    uint64_t g, load, r1, r2, r3;
};
__device__ __forceinline__ void prep_bars_init(PrepBars *b) {
    tc::mbar_init(&b->g, 1);
    tc::mbar_init(&b->load, 1);
    tc::mbar_init(&b->r1, 2);  // rounds 1-3 are issued by two warps, one commit each
    tc::mbar_init(&b->r2, 2);
    tc::mbar_init(&b->r3, 2);
}

// One (chunk slot, head) of the preparation by a group of 256 threads whose 256
// TMEM columns start at `tmem`; `ph` is the parity of this unit's barrier phases
// (units the group has prepared before, mod 2).  With `claim_counter`, the group
// claims its next unit from that counter (claim_base + the counter's value)
// halfway through this one (into the shared word `next_claim`; `units` and
// beyond: none left) and pulls that unit's tiles into L2.  `mid_signal`, if
// set, is raised (a shared word) at the same point, once the unit's operands
// are built.  If `publish` is set, the group's previous record is published
// there (release, once its bulk stores are complete) as soon as this unit's
// gate tile has arrived.  Returns false after recording a timeout in the
// status word.
__device__ bool prepare_unit(const PrepParams &p, int slot, int h, int t0, int Lc, uint8_t *sm, PrepBars *bars,
                             uint32_t ph, uint32_t tmem, const uint8_t *ident, int32_t *publish,
                             const PrepGroup &grp,
                             PrepShared &sh, int32_t *claim_counter = nullptr, int claim_base = 0,
                             int *next_claim = nullptr, int units = 0, int *mid_signal = nullptr) {
    float *s_beta = sh.beta, *s_bm = sh.bm, *s_F = sh.F, *s_Em = sh.Em, *s_blast = sh.blast;
    float *s_half = sh.half, *s_invk = sh.invk, *s_invq = sh.invq;
    float(*s_gabs)[kD] = sh.gabs;
    int &s_abort = sh.abort;
    const int tid = grp.tid, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const int32_t *doc_slot0 = reinterpret_cast<const int32_t *>(p.ws + p.doc_slot0_off);
    char *ws = p.ws;
    constexpr TcRecord R = tc_record();
    char *rec = ws + p.records_off + ((size_t)slot * H + h) * p.record_bytes;
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    (void)status;  // (read by the bounds checks of the bounds-checking build only)
    if (!KDA_IN_BOUNDS(slot >= 0 && slot < max_chunk_slots(p.cu, p.num_seqs, kL) && h >= 0 && h < H && t0 >= 0 &&
                           Lc >= 1 && Lc <= kL && t0 + Lc <= p.cu[p.num_seqs],
                       status))
        return false;  // (uniform: every thread of the group evaluates the same condition)

    if (tid == 0) {
        s_abort = 0;
        // the gates first: the cumulative sums run while k, q, v are still arriving
        tc::mbar_arrive_expect_tx(&bars->g, 32768);
        tc::tma_load_3d(sm + PrepSmem::G, p.tm_g, 0, h, t0, &bars->g);
        tc::bulk_wait_read();  // the group's previous unit's M' copy has read X (the one copy it left pending)
        tc::mbar_arrive_expect_tx(&bars->load, 6 * 8192);
        tc::tma_load_3d(sm + PrepSmem::X, p.tm_k, 0, h, t0, &bars->load);
        tc::tma_load_3d(sm + PrepSmem::X + 8192, p.tm_q, 0, h, t0, &bars->load);
        tc::tma_load_3d(sm + PrepSmem::X + 16384, p.tm_k, 64, h, t0, &bars->load);
        tc::tma_load_3d(sm + PrepSmem::X + 24576, p.tm_q, 64, h, t0, &bars->load);
        tc::tma_load_3d(sm + PrepSmem::V, p.tm_v, 0, h, t0, &bars->load);
        tc::tma_load_3d(sm + PrepSmem::V + 8192, p.tm_v, 64, h, t0, &bars->load);
    }
    if (tid < kL) s_beta[tid] = tid < Lc ? p.beta[(size_t)(t0 + tid) * H + h] : 0.f;
    tc::tc_fence_before();
    grp.sync();
    tc::tc_fence_after();
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int trow = (warp & 3) * 32 + lane;  // this thread's TMEM lane
    const int hs = warp >> 2;                 // this warp's half of an accumulator's columns
    if (!tc::mbar_wait(&bars->g, ph)) s_abort = 1;
    if (publish && tid == 0) {
        // the previous record, once its bulk stores are complete: they were issued when that unit ended and
        // this unit's loads and gate tile have come in since, so the wait is short
        tc::bulk_wait_all();
        tc::fence_proxy_async_global();
        tc::st_release_gpu(publish, 1);
    }
    grp.sync();
    if (s_abort) {  // a lost TMA completion: report and leave without touching the record
        if (tid == 0) flag_timeout(ws);
        return false;
    }

    // cumulative log-decay of channel c over this thread's 32 rows; reference token m in the middle
    float *Gf = reinterpret_cast<float *>(sm + PrepSmem::G);
    bool unsafe;
    {
        const int c = tid & (kD - 1), hh = tid >> 7, r0 = hh * 32;
        if (Lc < kL) {  // a document's last, partial chunk: the rows past its end add nothing to the sums
            for (int e = Lc * kD + tid; e < kL * kD; e += kPrepThreads) Gf[e] = 0.f;
            grp.sync();
        }
        // (so every row's b is a valid row's: b_r = b_{Lc-1} past the end, inside the valid rows' range)
        float bcol[32];
        float acc = 0.f, aabs = 0.f;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const float gv = Gf[(r0 + u) * kD + c];
            acc += gv;
            aabs += fabsf(gv);
            bcol[u] = acc;
        }
        if (hh == 0) s_half[c] = acc;
        s_gabs[hh][c] = aabs;
        grp.sync();  // all of g has been read (b may now go to its swizzled places); s_half is final
        const float off = hh ? s_half[c] : 0.f;
#pragma unroll
        for (int u = 0; u < 32; ++u) Gf[bswz(r0 + u, c)] = bcol[u] + off;
        if (hh) s_blast[c] = bcol[31] + off;  // row 63's b is the last valid row's
        grp.sync();
        bool bad = false;
        float bm = 0.f;
        if (tid < kD) {
            bm = Gf[bswz((Lc - 1) >> 1, c)];  // the middle token's
            // |b_r - b_m| is at most the sum of |g| between r and m: within each half's sum for a full chunk
            // (m = 31), within the whole chunk's otherwise (NaN or infinite gates fail the test as well)
            const float a0 = s_gabs[0][c], a1 = s_gabs[1][c];
            bad = Lc == kL ? !(a0 <= kMaxHalfRange && a1 <= kMaxHalfRange) : !(a0 + a1 <= kMaxHalfRange);
        }
        // Reference point of the factorised exponentials: the middle token; a chunk whose range is too
        // wide for that takes exact A and P and the chunk start as reference (exp(b_r) <= 1 for
        // non-positive gates), so no operand can overflow.
        unsafe = grp.sync_or(bad);
        if (tid < kD) {
            const float blast = s_blast[c];
            const float bref = unsafe ? 0.f : bm;
            s_bm[c] = bref;
            s_F[c] = expf(blast - bref);
            s_Em[c] = expf(bref);
            reinterpret_cast<float *>(rec + R.gamma)[c] = expf(blast);
        }
        if (!tc::mbar_wait(&bars->load, ph)) s_abort = 1;
        grp.sync();
    }
    if (s_abort) {
        if (tid == 0) flag_timeout(ws);
        return false;
    }
    if (p.qk_norm) {
        // fused prologue: inverse L2 norms of the 64 k rows and 64 q rows; thread t sums row t / 4, channels
        // 32 (t % 4) .. + 31, and the four threads of a row combine by shuffles
        const int r = tid >> 2, qd = tid & 3;
        const uint8_t *panel = sm + PrepSmem::X + (uint32_t)(qd >> 1) * 16384u;
        const int c0 = (qd & 1) * 32;
        float sk2 = 0.f, sq2 = 0.f;
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
            float f[8], e[8];
            unpack8(*reinterpret_cast<const uint4 *>(panel + tc::sw128_offset(r, c0 + j)), f);
            unpack8(*reinterpret_cast<const uint4 *>(panel + tc::sw128_offset(64 + r, c0 + j)), e);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                sk2 = fmaf(f[u], f[u], sk2);
                sq2 = fmaf(e[u], e[u], sq2);
            }
        }
        sk2 += __shfl_xor_sync(0xffffffffu, sk2, 1);
        sq2 += __shfl_xor_sync(0xffffffffu, sq2, 1);
        sk2 += __shfl_xor_sync(0xffffffffu, sk2, 2);
        sq2 += __shfl_xor_sync(0xffffffffu, sq2, 2);
        if (qd == 0) {
            s_invk[r] = rsqrtf(sk2 + p.qk_eps);
            s_invq[r] = rsqrtf(sq2 + p.qk_eps);
        }
        grp.sync();
    }
    float accA[16], accP[16];
    if (unsafe) {
        exact_ap(sm + PrepSmem::X, Gf, s_beta, Lc, tid, accA, accP, p.qk_norm ? s_invk : nullptr,
                 p.qk_norm ? s_invq : nullptr);
        grp.sync();  // the raw k, q tiles are about to be scaled in place
    }

    // Operand build: thread t owns channel octet o = t % 16 (channels 8 o .. 8 o + 7) of token rows
    // t / 16 + 16 i, i = 0..3; the octet's per-channel factors are read once.
    uint4 kend[4];
    const int oct = tid & 15, opanel = oct >> 3, ocol = (oct & 7) * 8, orow = tid >> 4;
    {
        const int c0 = oct * 8;
        float bmv[8], fv[8], blv[8];
        *reinterpret_cast<float4 *>(bmv) = *reinterpret_cast<const float4 *>(s_bm + c0);
        *reinterpret_cast<float4 *>(bmv + 4) = *reinterpret_cast<const float4 *>(s_bm + c0 + 4);
        *reinterpret_cast<float4 *>(fv) = *reinterpret_cast<const float4 *>(s_F + c0);
        *reinterpret_cast<float4 *>(fv + 4) = *reinterpret_cast<const float4 *>(s_F + c0 + 4);
        *reinterpret_cast<float4 *>(blv) = *reinterpret_cast<const float4 *>(s_blast + c0);
        *reinterpret_cast<float4 *>(blv + 4) = *reinterpret_cast<const float4 *>(s_blast + c0 + 4);
        uint8_t *Xp = sm + PrepSmem::X + (uint32_t)opanel * 16384u;
        uint8_t *Yp = sm + PrepSmem::Y + (uint32_t)opanel * 8192u;
        // the reference in log2 units: exp(b - b_m) = 2^(b log2(e) - b_m log2(e)), one fused multiply-add
        float bml[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) bml[u] = bmv[u] * kLog2e;
        // beta is not applied here: it scales A's rows as they leave TMEM and T's columns in T's bf16
        // image, so that W' = T diag(beta) (k e1) and Ut = T diag(beta) v take k e1 and v as they are
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {  // a loop, not unrolled: one copy of the body stays in the instruction cache
            const int r = orow + 16 * i;
            const bool valid = r < Lc;
            const uint32_t off_k = tc::sw128_offset(r, ocol), off_q = tc::sw128_offset(64 + r, ocol);
            if (!KDA_IN_BOUNDS(r < kL && off_q + 16 <= 16384u, status)) continue;
            float k8[8], q8[8], xk[8], xq[8], ke[8];
            uint4 kraw = *reinterpret_cast<const uint4 *>(Xp + off_k), qraw = *reinterpret_cast<const uint4 *>(Xp + off_q);
            if (!valid) kraw = qraw = make_uint4(0u, 0u, 0u, 0u);  // rows past the chunk's end contribute nothing
            unpack8(kraw, k8);
            unpack8(qraw, q8);
            if (p.qk_norm) {
                const float ik = s_invk[r], iq = s_invq[r];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    k8[u] *= ik;
                    q8[u] *= iq;
                }
            }
            const float4 b0 = *reinterpret_cast<const float4 *>(Gf + bswz(r, c0));
            const float4 b1 = *reinterpret_cast<const float4 *>(Gf + bswz(r, c0 + 4));
            const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
            if (!unsafe) {
                float y8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float d = fmaf(bb[u], kLog2e, -bml[u]);
                    const float e1 = exp2_approx(d), inv = exp2_approx(-d);
                    xk[u] = k8[u] * e1;
                    xq[u] = q8[u] * e1;
                    y8[u] = k8[u] * inv;
                    ke[u] = y8[u] * fv[u];  // Kend = k exp(b_last - b_r) <= |k| via the bounded factors
                }
                *reinterpret_cast<uint4 *>(Yp + off_k) = pack8(y8);
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) {  // reference 0: exp(b_r) <= 1
                    const float e1 = valid ? __expf(bb[u] - bmv[u]) : 0.f;
                    xk[u] = k8[u] * e1;
                    xq[u] = q8[u] * e1;
                    ke[u] = valid ? k8[u] * __expf(blv[u] - bb[u]) : 0.f;
                }
            }
            *reinterpret_cast<uint4 *>(Xp + off_k) = pack8(xk);
            *reinterpret_cast<uint4 *>(Xp + off_q) = pack8(xq);
            kend[i] = pack8(ke);
        }
    }
    tc::fence_async_smem();
    tc::tc_fence_before();
    grp.sync();
    tc::tc_fence_after();
    if (mid_signal && tid == 0) *reinterpret_cast<volatile int *>(mid_signal) = 1;
    constexpr int kClaimer = 64;  // a thread of warp 2: neither issuer waits for the atomic
    if (claim_counter && tid == kClaimer) {
        *next_claim = claim_base + atomicAdd(claim_counter, 1);
    }

    constexpr uint64_t kKmaj = tc::smem_desc_base(16, 1024, tc::SW_128B);
    bool ok = true;
    float *Af = reinterpret_cast<float *>(sm + PrepSmem::Afp);
    uint8_t *Pb = sm + PrepSmem::P;
    if (unsafe) {
        if (lane == 0 && warp < 2) tc::mma_commit(&bars->r1);  // no MMAs: completes round 1's phase at once
        const int r = tid >> 2, s0 = (tid & 3) * 16;
#pragma unroll
        for (int j8 = 0; j8 < 16; j8 += 8) {
            float w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int s = s0 + j8 + u;
                if ((s >> 4) <= (r >> 4)) Af[tri_idx(r, s)] = s < r ? accA[j8 + u] : 0.f;
                w[u] = s <= r ? accP[j8 + u] : 0.f;
            }
            *reinterpret_cast<uint4 *>(Pb + tc::sw128_offset(r, s0 + j8)) = pack8(w);
        }
    } else {
        // round 1: [beta k e1 ; q e1] x (k / e1)^T (rows 0-63 A, 64-127 P) into TMEM cols 0..63, both K panels
        // accumulated by one issuer (lane 0 of warp 0; warp 1 only commits, the barrier counting two commits)
        if (lane == 0 && warp < 2) {
            if (warp == 0) {
                constexpr uint32_t id = tc::idesc_bf16_f32(128, 64, false, false);
                for (int s = 0; s < 8; ++s) {
                    const uint32_t ka = (uint32_t)(s >> 2) * 16384u + (uint32_t)(s & 3) * 32u;
                    const uint32_t kb = (uint32_t)(s >> 2) * 8192u + (uint32_t)(s & 3) * 32u;
                    tc::mma_bf16(tmem, tc::smem_desc(kKmaj, tc::smem_u32(sm + PrepSmem::X + ka)),
                                 tc::smem_desc(kKmaj, tc::smem_u32(sm + PrepSmem::Y + kb)), id, s > 0);
                }
            }
            tc::mma_commit(&bars->r1);
        }
        __syncwarp();
        ok = tc::mbar_wait(&bars->r1, ph);
        tc::tc_fence_after();
        if (warp_all(ok)) {  // the MMAs are complete: their operand Y may be overwritten by P
            float v[32];
            tc::tmem_ld32(tmem + lane_base + 32u * (uint32_t)hs, v);
            if (trow < 64) {
                const int r = trow;
                // A = diag(beta) (k e1)(k / e1)^T, strictly lower.  The blocks on and below the diagonal are
                // stored whole: the solve reads only the entries below the diagonal, so the others (which
                // may even overflow) need no mask.
                const float br = s_beta[r];
#pragma unroll
                for (int qb = 0; qb < 2; ++qb) {
                    const int q4 = 2 * hs + qb;
                    if (q4 <= (r >> 4) && KDA_IN_BOUNDS(tri_blk(r >> 4, q4) + 256 <= 2560, status)) {
                        float *dst = Af + tri_blk(r >> 4, q4) + ((r & 15) << 4);
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4 *>(dst + i) =
                                make_float4(br * v[qb * 16 + i], br * v[qb * 16 + i + 1], br * v[qb * 16 + i + 2],
                                            br * v[qb * 16 + i + 3]);
                    }
                }
            } else {
                const int r = trow - 64;
#pragma unroll
                for (int s8 = 0; s8 < 32; s8 += 8) {
                    const int s = 32 * hs + s8;
                    float w[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) w[u] = s + u <= r ? v[s8 + u] : 0.f;
                    *reinterpret_cast<uint4 *>(Pb + tc::sw128_offset(r, s)) = pack8(w);
                }
            }
        }
    }
    tc::tc_fence_before();
    if (!ok) s_abort = 1;
    grp.sync();
    if (s_abort) {
        if (tid == 0) flag_timeout(ws);
        return false;
    }
    if (claim_counter && tid == 0) {  // the unit claimed at the operand barrier: its tiles into L2
        const int un = *next_claim;
        int ndoc, nt0, nLc;
        if (un < units && locate_slot(doc_slot0, p.cu, p.num_seqs, kL, un / H, &ndoc, &nt0, &nLc)) {
            const int nhh = un % H;
            tc::tma_prefetch_3d(p.tm_g, 0, nhh, nt0);
            tc::tma_prefetch_3d(p.tm_k, 0, nhh, nt0);
            tc::tma_prefetch_3d(p.tm_k, 64, nhh, nt0);
            tc::tma_prefetch_3d(p.tm_q, 0, nhh, nt0);
            tc::tma_prefetch_3d(p.tm_q, 64, nhh, nt0);
            tc::tma_prefetch_3d(p.tm_v, 0, nhh, nt0);
            tc::tma_prefetch_3d(p.tm_v, 64, nhh, nt0);
        }
    }

    // triangular solve in fp32, writing T diag(beta) as the bf16 round-2 B operand (K-major [r][s])
    float *Tf = reinterpret_cast<float *>(sm + PrepSmem::Tfp);
    unit_lower_inverse(Af, Tf, reinterpret_cast<float *>(sm + PrepSmem::Scr), sm + PrepSmem::Tb, s_beta, grp);
    tc::tc_fence_after();
    if (tid == 0) {  // P is final: its image goes to the record for the output pass
        tc::bulk_s2g(rec + R.P, sm + PrepSmem::P, 8192);
        tc::bulk_commit();
    }

    // round 2: W'^T = (T diag(beta) X_k)^T -> cols 64..127;  Ut^T = (T diag(beta) V)^T -> cols 128..191
    if (lane == 0 && warp < 2) {  // warp 0: W', warp 1: Ut
        constexpr uint32_t id = tc::idesc_bf16_f32(128, 64, true, false);
        const uint64_t amn = warp == 0 ? tc::smem_desc_base(16384, 1024, tc::SW_128B)
                                       : tc::smem_desc_base(8192, 1024, tc::SW_128B);
        uint8_t *abase = sm + (warp == 0 ? PrepSmem::X : PrepSmem::V);
        for (int s = 0; s < 4; ++s)
            tc::mma_bf16(tmem + 64u * (uint32_t)(warp + 1), tc::smem_desc(amn, tc::smem_u32(abase + s * 2048)),
                         tc::smem_desc(kKmaj, tc::smem_u32(sm + PrepSmem::Tb + s * 32)), id, s > 0);
        tc::mma_commit(&bars->r2);
    }
    __syncwarp();
    ok = tc::mbar_wait(&bars->r2, ph);
    tc::tc_fence_after();
    if (warp_all(ok)) {
        // warps 0-3: W'^T row c -> WT;  warps 4-7: Ut^T row c -> V (round 2 has consumed V)
        float w[64];
        tc::tmem_ld64(tmem + lane_base + 64u + 64u * (uint32_t)hs, w);
        uint8_t *dst = sm + (hs ? PrepSmem::V : PrepSmem::WT);
#pragma unroll
        for (int s8 = 0; s8 < 64; s8 += 8)
            *reinterpret_cast<uint4 *>(dst + tc::sw128_offset(trow, s8)) = pack8_at(w + s8);
        // Kend (kept in registers since the operand build) -> MN-major [s][c] operand
        uint8_t *Ks = sm + PrepSmem::KendS + (uint32_t)opanel * 8192u;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4 *>(Ks + tc::sw128_offset(orow + 16 * i, ocol)) = kend[i];
    }
    tc::fence_async_smem();
    tc::tc_fence_before();
    if (!ok) s_abort = 1;
    grp.sync();
    tc::tc_fence_after();
    if (s_abort) {
        if (tid == 0) {
            flag_timeout(ws);
            tc::bulk_wait_read();  // record images already on their way still read shared memory
        }
        return false;
    }
    if (tid == 0) {  // so is Ut^T
        tc::bulk_s2g(rec + R.Ut, sm + PrepSmem::V, 16384);
        tc::bulk_commit();
    }

    // round 3:  (X_q - P W')^T -> cols 0..63 (warp 0);  Kend^T W' -> cols 128..255 (warp 1)
    if (lane == 0 && warp < 2) {
        if (warp == 0) {
            constexpr uint32_t id_neg = tc::idesc_bf16_f32(128, 64, false, false) | (1u << 14);  // negate B
            constexpr uint32_t id_xq = tc::idesc_bf16_f32(128, 64, true, false);
            constexpr uint64_t kXmn = tc::smem_desc_base(16384, 1024, tc::SW_128B);
            for (int s = 0; s < 4; ++s)
                tc::mma_bf16(tmem, tc::smem_desc(kKmaj, tc::smem_u32(sm + PrepSmem::WT + s * 32)),
                             tc::smem_desc(kKmaj, tc::smem_u32(sm + PrepSmem::P + s * 32)), id_neg, s > 0);
            for (int s = 0; s < 4; ++s)
                tc::mma_bf16(tmem, tc::smem_desc(kXmn, tc::smem_u32(sm + PrepSmem::X + 8192 + s * 2048)),
                             tc::smem_desc(kKmaj, tc::smem_u32(ident + s * 32)), id_xq, true);
        } else {
            constexpr uint32_t id128 = tc::idesc_bf16_f32(128, 128, true, false);
            constexpr uint64_t kKmn = tc::smem_desc_base(8192, 1024, tc::SW_128B);
            for (int s = 0; s < 4; ++s)
                tc::mma_bf16(tmem + 128, tc::smem_desc(kKmn, tc::smem_u32(sm + PrepSmem::KendS + s * 2048)),
                             tc::smem_desc(kKmaj, tc::smem_u32(sm + PrepSmem::WT + s * 32)), id128, s > 0);
        }
        tc::mma_commit(&bars->r3);
    }
    __syncwarp();
    ok = tc::mbar_wait(&bars->r3, ph);
    tc::tc_fence_after();
    if (warp_all(ok)) {
        // Qp = (X_q - P W') exp(b_m), MN-major [c][r]; M' = -Kend^T W' exp(b_m), K-major [c][c'].
        // Both are staged in shared memory (round 3 has consumed X and W'^T) and leave by bulk copy.
        // Warps 0-3: Qp and M' columns 0-31; warps 4-7: M' columns 32-127.
        const int c = trow;
        uint8_t *QpS = sm + PrepSmem::WT;
        uint8_t *McS = sm + PrepSmem::X;
        if (hs == 0) {
            const float em = s_Em[c];
            float qv[64];
            tc::tmem_ld64(tmem + lane_base, qv);
#pragma unroll
            for (int i = 0; i < 64; ++i) qv[i] *= em;
#pragma unroll
            for (int s8 = 0; s8 < 64; s8 += 8)
                *reinterpret_cast<uint4 *>(QpS + tc::sw128_offset(c, s8)) = pack8_at(qv + s8);
        }
        for (int q32 = hs ? 1 : 0; q32 < (hs ? 4 : 1); ++q32) {
            float mv[32];
            tc::tmem_ld32(tmem + lane_base + 128u + (uint32_t)(q32 * 32), mv);
#pragma unroll
            for (int i4 = 0; i4 < 32; i4 += 4) {
                const float4 e4 = *reinterpret_cast<const float4 *>(s_Em + q32 * 32 + i4);
                mv[i4] *= -e4.x; mv[i4 + 1] *= -e4.y; mv[i4 + 2] *= -e4.z; mv[i4 + 3] *= -e4.w;
            }
#pragma unroll
            for (int h8 = 0; h8 < 32; h8 += 8) {
                const int cp = q32 * 32 + h8;
                *reinterpret_cast<uint4 *>(McS + (uint32_t)(cp >> 6) * 16384u + tc::sw128_offset(c, cp & 63)) =
                    pack8_at(mv + h8);
            }
        }
    }
    tc::fence_async_smem();
    tc::tc_fence_before();
    if (!ok) s_abort = 1;
    grp.sync();
    tc::tc_fence_after();
    if (s_abort) {
        if (tid == 0) {
            flag_timeout(ws);
            tc::bulk_wait_read();  // record images already on their way still read shared memory
        }
        return false;
    }
    if (tid == 0) {
        tc::bulk_s2g(rec + R.Kend, sm + PrepSmem::KendS, 16384);  // round 3 has consumed it
        tc::bulk_s2g(rec + R.Qp, sm + PrepSmem::WT, 16384);
        tc::bulk_commit();
        tc::bulk_s2g(rec + R.Mc, sm + PrepSmem::X, 32768);
        tc::bulk_commit();
        // G and V are free for the next unit's tiles once all but the M' copy have read them; that copy may
        // still be reading X when this returns: the next unit waits for it before loading X, and the caller
        // before it reuses the shared memory otherwise or leaves
        tc::bulk_wait_read_all_but_one();
    }
    return true;
}

__global__ void __launch_bounds__(kPrepThreads, 2)
prefill_prepare_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                   const float *__restrict__ beta, const int32_t *__restrict__ cu, int num_seqs, int H,
                   char *__restrict__ ws, size_t doc_slot0_off, size_t records_off, size_t record_bytes,
                   int qk_norm, float qk_eps) {
    // Persistent: as many CTAs as are co-resident, each running units until none is left (its TMEM and
    // barriers set up once).  Unit u is (chunk slot u / H, head u % H); a CTA's first unit is its own index,
    // and each later one is claimed from the work counter halfway through the one before.
    extern __shared__ uint8_t smem_raw[];
    __shared__ PrepBars bars;
    __shared__ PrepShared psh;
    __shared__ uint32_t tmem_base;
    __shared__ int s_unit;
    uint8_t *sm = align1024(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0 && num_seqs == 1) {
        // A single document: chunk slot s starts at token 64 s, so the first unit's tiles (inputs of the call,
        // complete before it) can be pulled into L2 while the chunk index kernel still runs
        const int hh = (int)blockIdx.x % H;
        const int64_t tok = (int64_t)((int)blockIdx.x / H) * kL;
        if (tok < (int64_t)__ldg(cu + 1)) {
            tc::tma_prefetch_3d(&tm_g, 0, hh, (int)tok);
            tc::tma_prefetch_3d(&tm_k, 0, hh, (int)tok);
            tc::tma_prefetch_3d(&tm_k, 64, hh, (int)tok);
            tc::tma_prefetch_3d(&tm_q, 0, hh, (int)tok);
            tc::tma_prefetch_3d(&tm_q, 64, hh, (int)tok);
            tc::tma_prefetch_3d(&tm_v, 0, hh, (int)tok);
            tc::tma_prefetch_3d(&tm_v, 64, hh, (int)tok);
        }
    }
    tc::grid_dep_wait();    // the chunk index kernel's slot table and zeroed work counter
    tc::grid_dep_launch();  // the state pass may get ready once every CTA of this grid has started
    const int32_t *doc_slot0 = reinterpret_cast<const int32_t *>(ws + doc_slot0_off);
    const int units = doc_slot0[num_seqs] * H;
    if (tid == 0) {
        prep_bars_init(&bars);
        tc::fence_mbar_init();
        s_unit = (int)blockIdx.x;
    }
    uint8_t *ident = sm + PrepSmem::bytes;
    write_identity(ident, tid, kPrepThreads);
    tc::fence_async_smem();
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 256);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const PrepParams prm{&tm_q,         &tm_k,       &tm_v,          &tm_g,   beta,  cu, num_seqs, H, ws, doc_slot0_off,
                         records_off, record_bytes, qk_norm, qk_eps};
    int32_t *counter = reinterpret_cast<int32_t *>(ws) + kPrepCounterWord;
    const PrepGroup grp{tid, 0u};
    // s_unit is read at the top of each iteration; the unit overwrites it with its claim between two of its
    // own barriers, after every thread's read and before the unit's last barrier
    for (uint32_t n = 0;; ++n) {
        const int u = s_unit;
        if (u >= units) break;
        const int slot = u / H, h = u % H;
        int doc = 0, t0 = -1, Lc = 0;  // (stay out of range where the slot is not found)
        locate_slot(doc_slot0, cu, num_seqs, kL, slot, &doc, &t0, &Lc);
        if (!prepare_unit(prm, slot, h, t0, Lc, sm, &bars, n & 1u, tmem_base, ident, nullptr, grp, psh, counter,
                          (int)gridDim.x, &s_unit, units))
            break;
    }
    if (tid == 0) tc::bulk_wait_read();  // the last unit's M' copy has read shared memory
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem_base, 256);
}

// ---------------------------------------------------------------------------
// Kernel 2: sequential state pass
// ---------------------------------------------------------------------------
// A chain is one (document, head, TN-column tile of S), TN = 32 or 64, run by one CTA sequentially over the
// document's chunks.  Its shared memory: NB record buffers (M', gamma and Kend, then the chain's rows of Ut^T),
// with FOLD (the chain also forms its columns of each chunk's output) a ring of two (Qp, P) images, and a ring
// of NS bf16 images of S (the MN-major B operand of M' S, in the record's layout).
template <int TN, int NB = 3, int NS = (TN == 32 ? 5 : 3), bool FOLD = false>
struct ChainCfg {
    static_assert(TN == 32 || TN == 64, "column tile of a chain");
    static_assert(NB >= 2 && NS >= 3, "a record ahead of the one in use; images multiplied, written, copied");
    static constexpr bool kFold = FOLD;
    static constexpr int kNBuf = NB;                           // records in flight
    static constexpr int kNSb = NS;                            // images: multiplied, being written, awaiting copy
    static constexpr uint32_t Mc = 0, gam = 32768, Kend = 33792, Ut = 50176;
    static constexpr uint32_t kUt = (uint32_t)TN * 128;        // the chain's rows of Ut^T: 4 / 8 KB
    static constexpr uint32_t kBuf = Ut + kUt;                 // a multiple of 1 KB (operand alignment)
    static constexpr uint32_t kImg = (uint32_t)TN * 256;       // the image: TN / 32 column chunks of 8 KB
    static constexpr uint32_t kQP = 24576;                     // Qp (16 KB) then P (8 KB), as in the record
    static constexpr uint32_t QB = kNBuf * kBuf;               // the (Qp, P) ring (FOLD), placed before the images
    static constexpr uint32_t SB = QB + (FOLD ? 2 * kQP : 0);  // (the 128-row operands' unused upper rows of
    static constexpr uint32_t bytes = SB + kNSb * kImg;        //  the second Qp, P image fall on the images)
    static constexpr int kCols = TN / 2;                       // columns of S per epilogue thread
    static_assert(kBuf % 1024 == 0 && kImg % 1024 == 0, "1 KB aligned operands");
};

// A chunk's record into a chain's buffer: M', gamma and Kend in one copy, the chain's rows of Ut^T in another.
template <int TN>
__device__ __forceinline__ void issue_record(uint8_t *buf, const char *rec, int tile, uint64_t *bar) {
    constexpr TcRecord R = tc_record();
    constexpr uint32_t kUt = ChainCfg<TN>::kUt;
    tc::mbar_arrive_expect_tx(bar, (uint32_t)R.state_part + kUt);
    tc::bulk_g2s(buf, rec, (uint32_t)R.state_part, bar);
    tc::bulk_g2s(buf + ChainCfg<TN>::Ut, rec + R.Ut + (size_t)tile * kUt, kUt, bar);
}
// The same parts of a later chunk's record pulled into L2 only (no shared memory, nothing to wait for), so that
// its copy into a buffer, a few chunks later, is served from L2.
template <int TN, bool FOLD = false>
__device__ __forceinline__ void prefetch_record(const char *rec, int tile) {
    constexpr TcRecord R = tc_record();
    constexpr uint32_t kUt = ChainCfg<TN>::kUt;
    tc::bulk_prefetch_l2(rec, (uint32_t)R.state_part);
    tc::bulk_prefetch_l2(rec + R.Ut + (size_t)tile * kUt, kUt);
    if (FOLD) tc::bulk_prefetch_l2(rec + R.Qp, ChainCfg<TN>::kQP);  // (Qp, P): one copy
}
constexpr int kChainL2Ahead = 3;  // records pulled into L2 this many chunks beyond the buffered ones

// Writes S[i][jbase + j] (j < NC, this thread's columns) into an image of S as the MN-major B operand of the
// state MMA: 32-column chunks of 128 rows x 64 bytes (8 KB apart), each row i holding its 32 columns in bf16,
// rows 64 bytes apart, with the 64-byte swizzle (16-byte unit u of row i at u ^ ((i / 2) % 4)).  NC / 8
// 16-byte stores; the 32 rows of a warp cover every bank once per 8 rows.
template <int NC>
__device__ __forceinline__ void store_state_rows(uint8_t *SB, int i, int jbase, const float (&S)[NC]) {
    uint8_t *row = SB + (uint32_t)(i >> 3) * 512u + (uint32_t)(i & 7) * 64u;
    const uint32_t sw = ((uint32_t)i >> 1) & 3u;
#pragma unroll
    for (int q = 0; q < NC / 8; ++q) {
        const uint32_t j = (uint32_t)(jbase + 8 * q);
        *reinterpret_cast<uint4 *>(row + (j >> 5) * 8192u + ((((j >> 3) & 3u) ^ sw) << 4)) = pack8_at(S + 8 * q);
    }
}

// One CTA per chain, kStateThreads threads:
//   warps 0-7   epilogue: thread <-> state row i = 32 (w % 4) + lane (its TMEM lane) and column half
//               h = w / 4; S[i][TN/2 h ..] stays fp32 in registers
//   warps 8, 9  lane 0 issues M' S over K panel w - 8 of S
//   warp 10     publisher: copies each chunk's S image to its record and, when asked, publishes it
//   warp 11     loader: streams the records in, up to kNBuf - 1 chunks ahead, each once its buffer is free
//               and, when asked, once the record is published
// Per chunk c:  issuers (after the epilogue warps' arrival on the operand barrier) -> MMAs -> a_bar ->
// epilogue S <- gamma S + Bc + M' S, image of S_{c+1} -> arrivals on the operand barrier, img_full and the
// buffer's empty barrier.  The publisher hands each image slot back through img_free.
constexpr int kStateEpiWarps = 8;
constexpr int kStatePubWarp = kStateEpiWarps + 2;
constexpr int kStateLoadWarp = kStatePubWarp + 1;
constexpr int kStateThreads = (kStateLoadWarp + 1) * 32;
constexpr uint32_t kBarOperand = 1;  // named barrier: the next S image is complete
constexpr int kBarOperandThreads = (kStateEpiWarps + 2) * 32;  // epilogue and issuer warps
constexpr int kStatePubLag = 2;    // images are published once the copy two chunks later is issued ...
constexpr int kStatePubBatch = 4;  // ... four at a time, behind one release fence
constexpr int kChainOutGroups = 2;  // output groups of 128 threads in each non-chain CTA of the chain plan

// Hand-offs of a chain with the rest of a launch (all null / true when it runs alone).
struct ChainLinks {
    int32_t *sdone = nullptr;        // publish each chunk's state image there (count in 32-column units)
    bool publish = true;             // false only in tests of the timeout path
    const int32_t *ready = nullptr;  // wait for each record's publication flag there before loading it
    uint64_t flag_wait_ns = kFlagWaitNs;
    // Records are streamed in by the loader warp (required with `ready`), else by the second MMA issuer right
    // behind its MMAs; which is faster depends on what else the launch runs (measured per plan).
    bool loader = true;
    __nv_bfloat16 *o = nullptr;  // FOLD: where the chain writes its columns of each chunk's output
    // The r-th document's chains are those of document doc_order[r] (null: r): with more chains than SMs, the
    // documents with the most chunks then start first.
    const int32_t *doc_order = nullptr;
};

// Chain j by the first kStateThreads threads of a CTA over `smem_raw` (Cfg, a ChainCfg<TN, ...>); the CTA's
// other threads (if any) take part in its CTA barriers only.
template <int TN, typename Cfg = ChainCfg<TN>>
__device__ void state_chain(const int32_t *__restrict__ cu, int num_seqs, int H, const float *__restrict__ S0,
                            float *__restrict__ S_final, char *__restrict__ ws, size_t doc_slot0_off,
                            size_t records_off, size_t record_bytes, int j, uint8_t *smem_raw,
                            const ChainLinks &links) {
    constexpr int NB = Cfg::kNBuf, NS = Cfg::kNSb, NC = Cfg::kCols, NT = kD / TN;
    constexpr bool FOLD = Cfg::kFold;
    // TMEM columns: two regions of two K panels for the state update; with FOLD two output regions after them
    constexpr uint32_t kTmemCols = FOLD ? (TN == 64 ? 512u : 256u) : 4u * TN;
    __shared__ uint64_t full_bar[NB], empty_bar[NB], a_bar, img_full[NS], img_free[NS];
    __shared__ uint64_t q_full[2], q_empty[2], o_full[2], o_free[2];  // FOLD: the (Qp, P) ring, output regions
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;
    // (the slot table and the status word are complete: the kernel before this one waited for the chunk index
    // kernel before letting this one start, or, in the pipe plan, this CTA has waited for them)
    if (*reinterpret_cast<const volatile int32_t *>(ws) != 0) return;  // invalid cu_seqlens: write nothing
    uint8_t *sm = align1024(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool epi = warp < kStateEpiWarps;
    const bool issuer = warp == kStateEpiWarps || warp == kStateEpiWarps + 1;
    const int i = (warp & 3) * 32 + lane, hcol = (warp >> 2) & 1;
    const int tile = j % NT;
    const int h = (j / NT) % H;
    const int rdoc = j / (NT * H);
    const int n = links.doc_order && rdoc < num_seqs ? links.doc_order[rdoc] : rdoc;
    const int32_t *doc_slot0 = reinterpret_cast<const int32_t *>(ws + doc_slot0_off);
    const int first = doc_slot0[n], nchunks = doc_slot0[n + 1] - first;
    if (!KDA_IN_BOUNDS(n < num_seqs && first >= 0 && nchunks >= 0 &&
                           first + nchunks <= max_chunk_slots(cu, num_seqs, kL),
                       reinterpret_cast<int32_t *>(ws)))
        return;  // (uniform over the CTA)
    const int col0 = tile * TN + NC * hcol;
    const size_t state_off = ((size_t)n * H + h) * kD * kD + (size_t)i * kD + col0;
    constexpr TcRecord R = tc_record();

    float S[NC];
#pragma unroll
    for (int c4 = 0; c4 < NC; c4 += 4) {
        const float4 v = (S0 && epi) ? *reinterpret_cast<const float4 *>(S0 + state_off + c4)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        S[c4] = v.x; S[c4 + 1] = v.y; S[c4 + 2] = v.z; S[c4 + 3] = v.w;
    }
    bool ok = true;
    if (nchunks > 0) {
        if (epi) store_state_rows<NC>(sm + Cfg::SB, i, NC * hcol, S);
        tc::fence_async_smem();
        char *rec_h = ws + records_off + (size_t)h * record_bytes;  // record of (slot 0, head h)
        const size_t rec_stride = (size_t)H * record_bytes;          // one chunk slot further
        if (tid == 0) {
            for (int b = 0; b < NB; ++b) {
                tc::mbar_init(&full_bar[b], 1);
                // one arrival per epilogue warp (and, with FOLD, the output warps' once the chunk's output MMAs,
                // which read the chain's rows of Ut^T, have completed)
                tc::mbar_init(&empty_bar[b], kStateEpiWarps + (FOLD ? 1 : 0));
            }
            tc::mbar_init(&a_bar, 2);  // one commit from each issuer
            for (int b = 0; b < NS; ++b) {
                tc::mbar_init(&img_full[b], kStateEpiWarps);  // one arrival per epilogue warp
                tc::mbar_init(&img_free[b], 1);               // the publisher's (FOLD: the output warps')
            }
            for (int b = 0; b < 2; ++b) {
                tc::mbar_init(&q_full[b], 1);
                tc::mbar_init(&q_empty[b], 1);
                tc::mbar_init(&o_full[b], 1);
                tc::mbar_init(&o_free[b], 2);  // both output warps
            }
            tc::fence_mbar_init();
            s_abort = 0;
            tc::grid_dep_wait();  // the preparation has completed, or (pipe plan) its records are awaited by flag
            if (!links.loader) {  // records already complete: the first kNBuf - 1 stream in at once
                char *rec0 = ws + records_off + (size_t)h * record_bytes;
                for (int c = 0; c < NB - 1 && c < nchunks; ++c)
                    issue_record<TN>(sm + c * Cfg::kBuf, rec0 + (size_t)(first + c) * H * record_bytes, tile,
                                     &full_bar[c]);
                for (int c = NB - 1; c < NB - 1 + kChainL2Ahead && c < nchunks; ++c)
                    prefetch_record<TN>(rec0 + (size_t)(first + c) * H * record_bytes, tile);
            }
        }
        if (warp == 0) {
            tc::tmem_alloc(&tmem_base, kTmemCols);
            tc::tmem_relinquish();
        }
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
        // Only now (after this CTA's wait for the preparation) may the output pass start: it reads the
        // preparation's part of each record before it waits for this kernel.
        tc::grid_dep_launch();
        // TMEM: chunk c's products in region c % 2 (cols 2 TN (c % 2) ..): Kend^T Ut plus M' S over the first
        // K panel, then M' S over the second
        const uint32_t tmem = tmem_base;

        if (warp == kStateLoadWarp) {
            // (with records that are complete before the launch, the second issuer streams them in instead,
            // right behind its MMAs, which costs less per chunk than a hand-off to this warp)
            if (lane == 0 && links.loader) {
                int issued = 0;
                for (int c = 0; c < nchunks; ++c) {
                    const int b = c % NB;
                    if (c >= NB) ok = ok && tc::mbar_wait(&empty_bar[b], (uint32_t)((c / NB - 1) & 1));
                    if (ok && links.ready) {
                        ok = tc::wait_flag_geq(links.ready + (size_t)(first + c) * H + h, 1, links.flag_wait_ns);
                        tc::fence_proxy_async_global();
                    }
                    if (!ok) break;
                    issue_record<TN>(sm + b * Cfg::kBuf, rec_h + (size_t)(first + c) * rec_stride, tile, &full_bar[b]);
                    issued = c + 1;
                    if constexpr (FOLD) {  // the chunk's (Qp, P) into its ring slot, free once output c - 2 is done
                        if (c >= 2) ok = tc::mbar_wait(&q_empty[c & 1], (uint32_t)(((c - 2) >> 1) & 1));
                        if (!ok) break;
                        tc::mbar_arrive_expect_tx(&q_full[c & 1], Cfg::kQP);
                        tc::bulk_g2s(sm + Cfg::QB + (uint32_t)(c & 1) * Cfg::kQP,
                                     rec_h + (size_t)(first + c) * rec_stride + R.Qp, Cfg::kQP, &q_full[c & 1]);
                    }
                    // a later record that is already published goes to L2 ahead of its copy
                    const int cp = c + kChainL2Ahead;
                    if (!links.ready && cp < nchunks)
                        prefetch_record<TN, FOLD>(rec_h + (size_t)(first + cp) * rec_stride, tile);
                }
                if (!ok) {  // copies already on their way land before the CTA's shared memory can go away
                    for (int c = max(0, issued - NB); c < issued; ++c)
                        tc::mbar_wait(&full_bar[c % NB], (uint32_t)((c / NB) & 1), 10000000ull);
                    if constexpr (FOLD) {
                        for (int c = max(0, issued - 2); c < issued; ++c)
                            tc::mbar_wait(&q_full[c & 1], (uint32_t)((c >> 1) & 1), 10000000ull);
                    }
                }
            }
            __syncwarp();
        } else if (issuer) {
            const uint32_t panel = (uint32_t)(warp - kStateEpiWarps);
            constexpr uint64_t kKmaj = tc::smem_desc_base(16, 1024, tc::SW_128B);
            constexpr uint64_t kKendMn = tc::smem_desc_base(8192, 1024, tc::SW_128B);
            // the image: MN-major, 32-column chunks 8 KB apart, 8-row groups of 512 bytes
            constexpr uint64_t kImgMn = tc::smem_desc_base(8192, 512, tc::SW_64B);
            constexpr uint32_t idN = tc::idesc_bf16_f32(128, TN, false, true);
            constexpr uint32_t idKU = tc::idesc_bf16_f32(128, TN, true, false);
            // Kend^T Ut of chunk c (the state-free part of its update) into panel 0 of TMEM region c % 2, ahead
            // of the chunk's M' S MMAs, which accumulate onto it
            auto kend_ut = [&](int c) {
                const uint8_t *b = sm + (c % NB) * Cfg::kBuf;
                const uint32_t d = tmem + (uint32_t)(2 * TN * (c & 1));
                for (int s = 0; s < 4; ++s)  // K steps of 16 tokens: +2 KB of the MN-major Kend, +32 B of Ut
                    tc::mma_bf16(d, tc::smem_desc(kKendMn, tc::smem_u32(b + Cfg::Kend + s * 2048)),
                                 tc::smem_desc(kKmaj, tc::smem_u32(b + Cfg::Ut + s * 32)), idKU, s > 0);
            };
            for (int c = 0; c < nchunks; ++c) {
                const int bsel = c % NB;
                uint8_t *buf = sm + bsel * Cfg::kBuf;
                uint8_t *sbc = sm + Cfg::SB + (uint32_t)(c % NS) * Cfg::kImg;
                if (c > 0) tc::named_barrier(kBarOperand, kBarOperandThreads);  // S_c's image is complete
                tc::tc_fence_after();
                if (lane == 0) {
                    ok = ok && tc::mbar_wait(&full_bar[bsel], (uint32_t)((c / NB) & 1));
                    if (ok) {
                        if (panel == 0 && c == 0) kend_ut(0);
                        const uint64_t da = tc::smem_desc(kKmaj, tc::smem_u32(buf + Cfg::Mc + panel * 16384u));
                        const uint64_t db = tc::smem_desc(kImgMn, tc::smem_u32(sbc + panel * 4096u));  // rows 64 panel ..
                        const uint32_t d = tmem + (uint32_t)(2 * TN * (c & 1)) + (uint32_t)TN * panel;
                        for (int s = 0; s < 4; ++s)  // K steps of 16: M' +32 bytes, the image +1 KB (+2, +64 in the fields)
                            tc::mma_bf16(d, da + 2u * (uint32_t)s, db + 64u * (uint32_t)s, idN, panel == 0 || s > 0);
                    }
                    tc::mma_commit(&a_bar);  // always: the epilogue counts on one completion per chunk
                    if (panel == 0 && ok && c + 1 < nchunks) {
                        // the next chunk's Kend^T Ut, while this chunk's epilogue runs: region (c + 1) % 2 was
                        // read by chunk c - 1's epilogue before this chunk's operand barrier
                        ok = tc::mbar_wait(&full_bar[(c + 1) % NB], (uint32_t)(((c + 1) / NB) & 1));
                        if (ok) kend_ut(c + 1);
                    }
                    if (!links.loader && panel == 1 && ok) {
                        // the buffer chunk c - 1 used was released by the operand barrier of this chunk
                        const int cn = c + NB - 1;
                        if (cn < nchunks)
                            issue_record<TN>(sm + (cn % NB) * Cfg::kBuf, rec_h + (size_t)(first + cn) * rec_stride,
                                             tile, &full_bar[cn % NB]);
                        if (cn + kChainL2Ahead < nchunks)
                            prefetch_record<TN>(rec_h + (size_t)(first + cn + kChainL2Ahead) * rec_stride, tile);
                    }
                }
                __syncwarp();
            }
        } else if (FOLD && warp == kStatePubWarp) {
            // The chunk's output columns of this chain, O[:, tile] = P Ut[:, tile] + Qp S_c[:, tile], from the
            // image S_c the chain multiplies and its own rows of Ut^T: one 128-lane accumulator whose lanes 0-63
            // are the chunk's tokens (the operands' upper 64 rows fall on neighbouring images, unread).
            if (lane == 0) {
                constexpr uint64_t kKmaj = tc::smem_desc_base(16, 1024, tc::SW_128B);
                constexpr uint64_t kQpMn = tc::smem_desc_base(16384, 1024, tc::SW_128B);
                constexpr uint32_t idK = tc::idesc_bf16_f32(128, TN, false, false);
                constexpr uint64_t kImgMn = tc::smem_desc_base(8192, 512, tc::SW_64B);
                constexpr uint32_t idMN = tc::idesc_bf16_f32(128, TN, true, true);
                for (int c = 0; c < nchunks; ++c) {
                    const int sl = c % NS, qs = c & 1, bsel = c % NB;
                    if (c > 0) ok = ok && tc::mbar_wait(&img_full[sl], (uint32_t)(((c - 1) / NS) & 1));
                    ok = ok && tc::mbar_wait(&full_bar[bsel], (uint32_t)((c / NB) & 1));
                    ok = ok && tc::mbar_wait(&q_full[qs], (uint32_t)((c >> 1) & 1));
                    if (c >= 2) ok = ok && tc::mbar_wait(&o_free[qs], (uint32_t)(((c - 2) >> 1) & 1));
                    if (ok) {
                        tc::tc_fence_after();
                        const uint8_t *qb = sm + Cfg::QB + (uint32_t)qs * Cfg::kQP;
                        const uint8_t *buf = sm + bsel * Cfg::kBuf;
                        const uint8_t *sbc = sm + Cfg::SB + (uint32_t)sl * Cfg::kImg;
                        const uint32_t d = tmem + 4u * TN + (uint32_t)(TN * qs);
                        for (int s4 = 0; s4 < 4; ++s4)  // P Ut over the chunk's tokens
                            tc::mma_bf16(d, tc::smem_desc(kKmaj, tc::smem_u32(qb + 16384 + s4 * 32)),
                                         tc::smem_desc(kKmaj, tc::smem_u32(buf + Cfg::Ut + s4 * 32)), idK, s4 > 0);
                        for (int s8 = 0; s8 < 8; ++s8)  // + Qp S_c over d_k
                            tc::mma_bf16(d, tc::smem_desc(kQpMn, tc::smem_u32(qb + s8 * 2048)),
                                         tc::smem_desc(kImgMn, tc::smem_u32(sbc + s8 * 1024)),
                                         idMN, true);
                    }
                    tc::mma_commit(&o_full[qs]);  // always: the output warps count on one completion per chunk
                }
            }
            __syncwarp();
        } else if (FOLD && warp >= kStateThreads / 32) {
            // Output warps (TMEM lane quarters 0 and 1: the chunk's 64 tokens): each chunk's output columns of
            // this chain, read once its MMAs complete, which also frees the image, the (Qp, P) slot and the
            // record buffer they read.
            const int ow = warp - kStateThreads / 32, r = ow * 32 + lane;
            const uint32_t lane_base = (uint32_t)(ow * 32) << 16;
            const int doc_t0 = cu[n], doc_t1 = cu[n + 1];
            for (int c = 0; c < nchunks; ++c) {
                const int qs = c & 1;
                ok = ok && tc::mbar_wait(&o_full[qs], (uint32_t)((c >> 1) & 1));
                tc::tc_fence_after();
                if (ow == 0 && lane == 0) {
                    tc::mbar_arrive(&img_free[c % NS]);
                    tc::mbar_arrive(&q_empty[qs]);
                    tc::mbar_arrive(&empty_bar[c % NB]);
                }
                float v[TN];
                if (warp_all(ok)) {
                    const uint32_t ta = tmem + lane_base + 4u * TN + (uint32_t)(TN * qs);
                    if constexpr (TN == 32) {
                        tc::tmem_ld32(ta, v);
                    } else {
                        float v1[32];
                        tc::tmem_ld32(ta, *reinterpret_cast<float(*)[32]>(v));
                        tc::tmem_ld32(ta + 32u, v1);
#pragma unroll
                        for (int q = 0; q < 32; ++q) v[32 + q] = v1[q];
                    }
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&o_free[qs]);  // always: the issuer counts on both warps
                if (!warp_all(ok)) break;
                const int t0 = doc_t0 + c * kL, Lc = min(kL, doc_t1 - t0);
                if (r < Lc && KDA_IN_BOUNDS(t0 + r < cu[num_seqs], reinterpret_cast<int32_t *>(ws))) {
                    uint4 *dst = reinterpret_cast<uint4 *>(links.o + ((size_t)(t0 + r) * H + h) * kD + tile * TN);
#pragma unroll
                    for (int u = 0; u < TN / 8; ++u) dst[u] = pack8_at(v + 8 * u);
                }
            }
        } else if (warp == kStatePubWarp) {
            if (lane == 0) {
                int pub = 0;  // images published so far
                for (int c = 0; c < nchunks; ++c) {
                    const int sl = c % NS;
                    // image 0 was written before the CTA barrier; image c >= 1 by chunk c - 1's epilogue
                    if (c > 0) ok = ok && tc::mbar_wait(&img_full[sl], (uint32_t)(((c - 1) / NS) & 1));
                    if (ok) {
                        // S_c's image, this chain's column chunks, into chunk c's record
                        const uint8_t *sbc = sm + Cfg::SB + (uint32_t)sl * Cfg::kImg;
                        char *rec = rec_h + (size_t)(first + c) * rec_stride;
                        tc::bulk_s2g(rec + R.S + (size_t)tile * Cfg::kImg, sbc, Cfg::kImg);
                        tc::bulk_commit();
                        tc::bulk_wait_read();  // the slot may be rewritten
                    }
                    tc::mbar_arrive(&img_free[sl]);  // always: the epilogue counts on one per image
                    if (ok && links.sdone && links.publish && c + 1 - kStatePubLag - pub >= kStatePubBatch) {
                        // the copies of S_pub .. S_{c-2} have completed: publish them
                        static_assert(kStatePubLag == 2, "wait_group below");
                        tc::bulk_wait_all_but_two();
                        tc::fence_proxy_async_global();
                        tc::fence_acq_rel_gpu();
                        for (; pub <= c - kStatePubLag; ++pub)
                            tc::red_relaxed_gpu_add(links.sdone + (size_t)(first + pub) * H + h, TN / 32);
                    }
                }
                tc::bulk_wait_all();  // shared memory must outlive the image copies
                if (links.sdone && links.publish && ok) {
                    tc::fence_proxy_async_global();
                    tc::fence_acq_rel_gpu();
                    for (; pub < nchunks; ++pub)
                        tc::red_relaxed_gpu_add(links.sdone + (size_t)(first + pub) * H + h, TN / 32);
                }
            }
            __syncwarp();
        } else if (epi) {
            const uint32_t tacc0 = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(NC * hcol);
            for (int c = 0; c < nchunks; ++c) {
                const int bsel = c % NB;
                const uint8_t *buf = sm + bsel * Cfg::kBuf;
                ok = ok && tc::mbar_wait(&full_bar[bsel], (uint32_t)((c / NB) & 1));
                const float gam = reinterpret_cast<const float *>(buf + Cfg::gam)[i];  // read while the MMAs run
                const int nb = c + 1;                // the image this chunk writes: S_{c+1}, needed by chunk c + 1
                const bool img = nb < nchunks;
                uint8_t *sbn = sm + Cfg::SB + (uint32_t)(nb % NS) * Cfg::kImg;
                // the slot's previous image, S_{c+1-NS}, has been copied out
                if (img && nb >= NS) ok = ok && tc::mbar_wait(&img_free[nb % NS], (uint32_t)((nb / NS - 1) & 1));
                ok = ok && tc::mbar_wait(&a_bar, (uint32_t)(c & 1));
                tc::tc_fence_after();
                if (warp_all(ok)) {
                    // S <- gamma S + (P0 + P1): P0 = Kend^T Ut + the first K panel of M' S, P1 the second
                    const uint32_t tacc = tacc0 + (uint32_t)(2 * TN * (c & 1));
                    float t0[NC];
                    if constexpr (NC == 16) {
                        float t1[16];
                        tc::tmem_ld16x2(tacc, tacc + TN, t0, t1);
#pragma unroll
                        for (int q = 0; q < 16; ++q) S[q] = fmaf(gam, S[q], t0[q] + t1[q]);
                    } else {
                        // 32 columns: the second panel in halves, to stay within the register budget
                        tc::tmem_ld32(tacc, t0);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            float t1[16];
                            tc::tmem_ld16(tacc + TN + 16u * (uint32_t)hh, t1);
#pragma unroll
                            for (int q = 0; q < 16; ++q)
                                S[16 * hh + q] = fmaf(gam, S[16 * hh + q], t0[16 * hh + q] + t1[q]);
                        }
                    }
                    if (img) store_state_rows<NC>(sbn, i, NC * hcol, S);
                }
                tc::fence_async_smem();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0 && links.loader) tc::mbar_arrive(&empty_bar[bsel]);  // the MMAs and this warp are done
                if (img) {
                    tc::named_barrier_arrive(kBarOperand, kBarOperandThreads);
                    if (lane == 0) tc::mbar_arrive(&img_full[nb % NS]);
                }
            }
        }
        if (!ok) s_abort = 1;
        __syncthreads();
        if (s_abort && tid == 0) {
            flag_timeout(ws);
            if (!links.loader) {
                // record copies the issuer may still have on their way land before shared memory goes away
                // (best effort, 10 ms per buffer: the last chunk that could use each one)
                for (int b = 0; b < NB && b < nchunks; ++b) {
                    const int last = b + ((nchunks - 1 - b) / NB) * NB;
                    tc::mbar_wait(&full_bar[b], (uint32_t)((last / NB) & 1), 10000000ull);
                }
            }
        }
        if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
        if (s_abort) return;
    }
    if (S_final && epi) {
#pragma unroll
        for (int q = 0; q < NC; q += 4)
            *reinterpret_cast<float4 *>(S_final + state_off + q) = make_float4(S[q], S[q + 1], S[q + 2], S[q + 3]);
    }
}

template <int TN>
__global__ void __launch_bounds__(kStateThreads, 1)
prefill_state_tc(const int32_t *__restrict__ cu, int num_seqs, int H, const float *__restrict__ S0,
                 float *__restrict__ S_final, char *__restrict__ ws, size_t doc_slot0_off, size_t records_off,
                 size_t record_bytes, size_t doc_order_off) {
    extern __shared__ uint8_t smem_raw[];
    ChainLinks links;
    links.doc_order = reinterpret_cast<const int32_t *>(ws + doc_order_off);
    state_chain<TN>(cu, num_seqs, H, S0, S_final, ws, doc_slot0_off, records_off, record_bytes, (int)blockIdx.x,
                    smem_raw, links);
}

// The state pass with each chain also forming its columns of every chunk's output (no output pass, no state
// images in the records): the three-kernel plan's second kernel when the gated output normalisation (which
// needs whole rows) is not fused.  Two record buffers, the (Qp, P) ring and two more warps, the output warps.
constexpr int kFoldThreads = kStateThreads + 64;
template <int TN>
using FoldCfg = ChainCfg<TN, 2, (TN == 32 ? 5 : 3), true>;

template <int TN>
__global__ void __launch_bounds__(kFoldThreads, 1)
prefill_state_fold_tc(const int32_t *__restrict__ cu, int num_seqs, int H, const float *__restrict__ S0,
                      float *__restrict__ S_final, __nv_bfloat16 *__restrict__ o, char *__restrict__ ws,
                      size_t doc_slot0_off, size_t records_off, size_t record_bytes, size_t doc_order_off) {
    extern __shared__ uint8_t smem_raw[];
    ChainLinks links;
    links.o = o;
    links.doc_order = reinterpret_cast<const int32_t *>(ws + doc_order_off);
    state_chain<TN, FoldCfg<TN>>(cu, num_seqs, H, S0, S_final, ws, doc_slot0_off, records_off, record_bytes,
                                 (int)blockIdx.x, smem_raw, links);
}

// ---------------------------------------------------------------------------
// Kernel 3: chunk-parallel output
// ---------------------------------------------------------------------------
// One CTA (128 threads) per (chunk, head):  O = Qp S_c + P Ut, with S_c the
// state entering the chunk (its bf16 image, written by the state pass).  Both
// products accumulate into one 128-lane TMEM tile that holds the chunk's 64
// token rows twice: A = [Qp ; Qp] (MN-major, the stride between its two 64-row
// halves zero) and [P ; P] (K-major, P loaded twice, one copy after the other).
// The record's Qp and P as stored, P a second time (so that the 128-row operand [P ; P] repeats the chunk's
// rows), Ut, the state image, and a 512-byte exchange area of the gated epilogue.
struct OutSmem {
    static constexpr uint32_t Qp = 0, P = 16384, P2 = 24576, Ut = 32768, S = 49152, X = 81920;
    static constexpr uint32_t kRec = S;  // bytes of the record part (Qp, P, P, Ut)
    static constexpr uint32_t bytes = 82944;
};

struct OutBars {
    uint64_t load, sload, mma;  // the record's Qp, P, Ut; its state image; the MMAs
};

// The fused epilogue's gated output normalisation (gate null: o is written as it is).
struct OutNorm {
    const __nv_bfloat16 *gate;  // z [T, H, 128]
    const float *weight;        // w [128] or null (ones)
    float eps;
};

// A group of 128 threads of a CTA: thread `gtid` of it, synchronised by named
// barrier `gbar` (0: the whole CTA is the group, __syncthreads).
struct OutGroup {
    int gtid;
    uint32_t gbar;
    int *ok;  // shared word of the group
    __device__ __forceinline__ void sync() const {
        if (gbar == 0) __syncthreads();
        else tc::named_barrier(gbar, 128);
    }
};

// An output group's next unit (pipe plan): thread `thread` of the group loads its record, and its state image
// once published, into the group's shared memory as soon as the current unit's MMAs have completed, and
// stores what it issued in *pre (0 nothing, 1 the record, 2 both) for that unit's call.
struct OutNext {
    const int *unit;  // the claimed unit (slot * H + head), read by `thread` only
    int units, thread;
    const int32_t *ready, *sdone;  // per unit: record published; state image count
    int *pre;
};

// One (chunk slot, head) of the output pass, t0 / Lc the chunk's first token and
// length, by a group of 128 threads (its four warps each write 32 token rows by
// 64 columns) whose TMEM holds 128 columns at `tmem`; `ph` is the parity of this unit's
// barrier phases.  P Ut is formed first; the state image is then awaited
// through the launch dependency with `dep_wait` (the state pass is the
// previous kernel), or through its publication count at `sflag` (all column
// tiles), else it must already be complete.  `pre`: what the group's previous
// unit already loaded for this one (OutNext).  Returns false after recording a
// timeout in the status word.
__device__ bool output_unit(const int32_t *__restrict__ cu, int num_seqs, int H, __nv_bfloat16 *__restrict__ o, char *ws,
                            size_t records_off, size_t record_bytes, int slot, int h, int t0, int Lc, uint8_t *sm,
                            OutBars *bars, uint32_t ph, uint32_t tmem, const OutGroup &grp, const OutNorm &onorm,
                            bool dep_wait = false, const int32_t *sflag = nullptr,
                            uint64_t flag_wait_ns = kFlagWaitNs, const int32_t *rflag = nullptr, int pre = 0,
                            const OutNext *nx = nullptr) {
    const int tid = grp.gtid, warp = tid >> 5;
    constexpr TcRecord R = tc_record();
    static_assert(R.P - R.Qp == OutSmem::P && R.Ut - R.P == OutSmem::P2 - OutSmem::P &&
                      R.S - R.Ut == OutSmem::S - OutSmem::Ut && R.bytes - R.S == OutSmem::X - OutSmem::S,
                  "the record's Qp, P, Ut and image in the output unit's layout");
    // the record part: Qp and P in one copy, P again, Ut; the image in one copy
    auto load_rec = [&](const char *rc) {
        tc::mbar_arrive_expect_tx(&bars->load, OutSmem::kRec);
        tc::bulk_g2s(sm, rc + R.Qp, (uint32_t)(R.Ut - R.Qp), &bars->load);
        tc::bulk_g2s(sm + OutSmem::P2, rc + R.P, (uint32_t)(R.Ut - R.P), &bars->load);
        tc::bulk_g2s(sm + OutSmem::Ut, rc + R.Ut, (uint32_t)(R.S - R.Ut), &bars->load);
    };
    auto load_img = [&](const char *rc) {
        tc::mbar_arrive_expect_tx(&bars->sload, (uint32_t)(R.bytes - R.S));
        tc::bulk_g2s(sm + OutSmem::S, rc + R.S, (uint32_t)(R.bytes - R.S), &bars->sload);
    };
    const char *rec = ws + records_off + ((size_t)slot * H + h) * record_bytes;
#ifdef KDA_DEBUG_BOUNDS
    const int total_tokens = cu[num_seqs];
#endif
    if (!KDA_IN_BOUNDS(slot >= 0 && slot < max_chunk_slots(cu, num_seqs, kL) && h >= 0 && h < H && t0 >= 0 &&
                           Lc >= 1 && Lc <= kL && t0 + Lc <= total_tokens,
                       reinterpret_cast<int32_t *>(ws)))
        return false;  // (uniform over the group)
    if (tid == 0) {
        // Qp, P, Ut (written by the preparation; in the pipe plan, once published) ...
        bool rok = true;
        bool img_now = pre == 2;  // (pre >= 1: the record's copy is on its way; 2: the image's too)
        if (pre == 0) {
            if (rflag) {
                rok = tc::wait_flag_geq(rflag, 1, flag_wait_ns);
                tc::fence_proxy_async_global();
            }
            // a unit taken behind the chains finds its state image published already: both loads go at once
            img_now = sflag && !dep_wait && tc::ld_acquire_gpu(sflag) >= kNTile;
            if (img_now) tc::fence_proxy_async_global();
            load_rec(rec);
            if (img_now) load_img(rec);
        }
        bool ok = tc::mbar_wait(&bars->load, ph) && rok;
        constexpr uint64_t kKmaj = tc::smem_desc_base(16, 1024, tc::SW_128B);
        constexpr uint64_t kQpMn = tc::smem_desc_base(0, 1024, tc::SW_128B);  // rows 64-127 repeat rows 0-63
        constexpr uint64_t kSMn = tc::smem_desc_base(8192, 512, tc::SW_64B);     // the image, as the chains write it
        constexpr uint32_t id_mn = tc::idesc_bf16_f32(128, 128, true, true);
        constexpr uint32_t id_k = tc::idesc_bf16_f32(128, 128, false, false);
        if (ok) {
            tc::tc_fence_after();
            for (int s = 0; s < 4; ++s)  // P Ut over the chunk's tokens
                tc::mma_bf16(tmem, tc::smem_desc(kKmaj, tc::smem_u32(sm + OutSmem::P + s * 32)),
                             tc::smem_desc(kKmaj, tc::smem_u32(sm + OutSmem::Ut + s * 32)), id_k, s > 0);
        }
        // ... then the image of S_c (written by the state pass)
        if (dep_wait) tc::grid_dep_wait();
        if (!img_now) {
            if (sflag) {
                ok = tc::wait_flag_geq(sflag, kNTile, flag_wait_ns) && ok;
                tc::fence_proxy_async_global();
            }
            load_img(rec);
        }
        ok = tc::mbar_wait(&bars->sload, ph) && ok;
        *grp.ok = ok;
        if (ok) {
            tc::tc_fence_after();
            for (int s = 0; s < 8; ++s)  // + Qp S_c over d_k
                tc::mma_bf16(tmem, tc::smem_desc(kQpMn, tc::smem_u32(sm + OutSmem::Qp + s * 2048)),
                             tc::smem_desc(kSMn, tc::smem_u32(sm + OutSmem::S + s * 1024)),
                             id_mn, true);
        }
        tc::mma_commit(&bars->mma);  // arrives at once when nothing was issued
    }
    __syncwarp();
    if (nx && tid == nx->thread) {
        // the next unit's copies into this shared memory, free once this unit's MMAs have completed
        int p = 0;
        const int un = *nx->unit;
        if (un < nx->units && tc::mbar_wait(&bars->mma, ph) && tc::ld_acquire_gpu(nx->ready + un) >= 1) {
            const char *nrec = ws + records_off + (size_t)un * record_bytes;
            tc::fence_proxy_async_global();
            load_rec(nrec);
            p = 1;
            if (tc::ld_acquire_gpu(nx->sdone + un) >= kNTile) {
                tc::fence_proxy_async_global();
                load_img(nrec);
                p = 2;
            }
        }
        *nx->pre = p;
    }
    __syncwarp();  // (the lane of warp 2 that loaded the next unit rejoins its warp)
    {
        // O sits twice in the accumulator (A = [Qp ; Qp] and [P ; P]): warp w writes token row 32 (w % 2) +
        // lane, columns 64 (w / 2) .. + 63, from TMEM lane 32 w + lane.
        const bool done = tc::mbar_wait(&bars->mma, ph);
        tc::tc_fence_after();
        const bool wok = warp_all(done);
        const int lane = tid & 31, r = (warp & 1) * 32 + lane, ch = warp >> 1;
        const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(64 * ch);
        const size_t row = ((size_t)(t0 + r) * H + h) * kD + (size_t)(64 * ch);
        uint4 *dst = reinterpret_cast<uint4 *>(o + row);
        const bool row_ok = KDA_IN_BOUNDS(r >= Lc || t0 + r < total_tokens, reinterpret_cast<int32_t *>(ws));
        const bool write = wok && r < Lc && row_ok;
        if (!onorm.gate) {
            if (wok) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float v[32];
                    tc::tmem_ld32(ta + (uint32_t)(q * 32), v);
                    if (write) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) dst[q * 4 + u] = pack8_at(v + 8 * u);
                    }
                }
            }
        } else {
            // fused epilogue: o / rms(o) * w * sigmoid(z).  The mean square adds the two column halves' sums,
            // exchanged through shared memory; the gate inputs of the second 32 columns are fetched while the
            // first are written, the weights are uniform across the warp (broadcast loads), the logistic
            // function takes the fast exponential and division (bf16 output).
            const uint4 *z4 = reinterpret_cast<const uint4 *>(onorm.gate + row);
            uint4 zc[4], zn[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) zc[u] = write ? __ldg(z4 + u) : make_uint4(0u, 0u, 0u, 0u);
            float ss = 0.f;
            if (wok) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float v[32];
                    tc::tmem_ld32(ta + (uint32_t)(q * 32), v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ss = fmaf(v[i], v[i], ss);
                }
            }
            float *xs = reinterpret_cast<float *>(sm + OutSmem::X);
            xs[warp * 32 + lane] = ss;
            grp.sync();
            const float tot = xs[(warp & 1) * 32 + lane] + xs[(2 + (warp & 1)) * 32 + lane];  // (the same order in both)
            const float scale = rsqrtf(tot * (1.f / kD) + onorm.eps);
            if (wok) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if (q == 0) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) zn[u] = write ? __ldg(z4 + 4 + u) : make_uint4(0u, 0u, 0u, 0u);
                    }
                    float v[32];
                    tc::tmem_ld32(ta + (uint32_t)(q * 32), v);
                    if (write) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            float z[8], wv[8];
                            unpack8(zc[u], z);
                            if (onorm.weight) {
                                const float4 *w4 =
                                    reinterpret_cast<const float4 *>(onorm.weight + 64 * ch + q * 32 + u * 8);
                                *reinterpret_cast<float4 *>(wv) = __ldg(w4);
                                *reinterpret_cast<float4 *>(wv + 4) = __ldg(w4 + 1);
                            } else {
#pragma unroll
                                for (int i = 0; i < 8; ++i) wv[i] = 1.f;
                            }
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                v[u * 8 + i] *= scale * wv[i] * __fdividef(1.f, 1.f + __expf(-z[i]));
                            dst[q * 4 + u] = pack8_at(v + 8 * u);
                        }
                    }
                    if (q == 0) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) zc[u] = zn[u];
                    }
                }
            }
        }
        if (!wok && lane == 0) flag_timeout(ws);
    }
    tc::tc_fence_before();
    grp.sync();
    const bool ok = *grp.ok != 0;
    if (tid == 0 && !ok) flag_timeout(ws);
    return ok;
}

__global__ void __launch_bounds__(128)
prefill_output_tc(const int32_t *__restrict__ cu, int num_seqs, int H, __nv_bfloat16 *__restrict__ o,
                  char *__restrict__ ws, size_t doc_slot0_off, size_t records_off, size_t record_bytes,
                  int resident, OutNorm onorm) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ OutBars bars;
    __shared__ uint32_t tmem_base;
    // (the chunk index kernel's table and status word are complete: the state pass waited for them)
    if (*reinterpret_cast<const volatile int32_t *>(ws) != 0) return;  // invalid input or an earlier timeout
    uint8_t *sm = align1024(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int slot = blockIdx.x, h = blockIdx.y;
    const int32_t *doc_slot0 = reinterpret_cast<const int32_t *>(ws + doc_slot0_off);
    int doc = 0, t0 = -1, Lc = 0;  // (stay out of range where the slot is not found)
    if (!locate_slot(doc_slot0, cu, num_seqs, kL, slot, &doc, &t0, &Lc)) return;
    if (tid == 0) {
        tc::mbar_init(&bars.load, 1);
        tc::mbar_init(&bars.sload, 1);
        tc::mbar_init(&bars.mma, 1);
        tc::fence_mbar_init();
        // the CTA that takes this one's place next (CTAs start in launch order): its record into L2
        const int nxt = blockIdx.y * gridDim.x + blockIdx.x + resident;
        if (resident > 0 && nxt < (int)(gridDim.x * gridDim.y) && (nxt % gridDim.x) < doc_slot0[num_seqs])
            tc::bulk_prefetch_l2(ws + records_off + ((size_t)(nxt % gridDim.x) * H + nxt / gridDim.x) * record_bytes +
                                     tc_record().Qp,
                                 (uint32_t)(tc_record().bytes - tc_record().Qp));
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 128);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    __shared__ int s_ok;
    output_unit(cu, num_seqs, H, o, ws, records_off, record_bytes, slot, h, t0, Lc, sm, &bars, 0u, tmem_base,
                OutGroup{tid, 0u, &s_ok}, onorm, true);
    if (warp == 0) tc::tmem_dealloc(tmem_base, 128);
}

// ---------------------------------------------------------------------------
// State pass with the output pass alongside (one launch after the preparation)
// ---------------------------------------------------------------------------
// One CTA per SM.  CTAs [0, n_state) run one chain each (state_chain, which
// publishes each chunk's state image); in each of the others, two groups of
// 128 threads take output units in chunk order from a counter, form P Ut at
// once and Qp S_c as soon as all of S_c's column tiles are published, so that
// one group's loads overlap the other's products and stores.  Output groups wait only for
// chain CTAs, which have the lowest indices and are placed first; every wait is
// bounded.
__global__ void __launch_bounds__(kStateThreads, 1)
prefill_chain_tc(const int32_t *__restrict__ cu, int num_seqs, int H, const float *__restrict__ S0,
                 float *__restrict__ S_final, __nv_bfloat16 *__restrict__ o, char *__restrict__ ws,
                 size_t doc_slot0_off, size_t records_off, size_t record_bytes, int n_state, int32_t *sdone,
                 int32_t *counter, unsigned long long flag_wait_ns, int fault, OutNorm onorm) {
    extern __shared__ uint8_t smem_raw[];
    if ((int)blockIdx.x < n_state) {
        // (fault == kFaultNoPublish only in tests of the timeout path: no state image is published, so the
        // output groups' bounded waits run out)
        ChainLinks links;
        links.sdone = sdone;
        links.publish = fault != kFaultNoPublish;
        links.loader = false;
        state_chain<kTile>(cu, num_seqs, H, S0, S_final, ws, doc_slot0_off, records_off, record_bytes,
                           (int)blockIdx.x, smem_raw, links);
        return;
    }
    constexpr int kGroups = kChainOutGroups;
    static_assert(kGroups * 128 <= kStateThreads && kGroups * OutSmem::bytes <= ChainCfg<kTile>::bytes &&
                      OutSmem::bytes % 1024 == 0,
                  "output groups fit the chain CTA");
    __shared__ OutBars bars[kGroups];
    __shared__ uint32_t tmem_base;
    __shared__ int s_unit[kGroups], s_uok[kGroups];
    // (the chunk index kernel's table and status word are complete: the preparation waited for them)
    if (*reinterpret_cast<const volatile int32_t *>(ws) != 0) return;  // invalid cu_seqlens: write nothing
    uint8_t *sm = align1024(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int g = tid >> 7;  // output group; threads of groups >= kGroups only take part in setup and teardown
    const int32_t *doc_slot0 = reinterpret_cast<const int32_t *>(ws + doc_slot0_off);
    const int units = doc_slot0[num_seqs] * H;
    // records the workspace holds (from cu_seqlens, as the host sized it): a prefetch never leaves them, even
    // where a corrupted chunk table (bounds-checking build) claims more units
    const int rec_units = max_chunk_slots(cu, num_seqs, kL) * H;
    const int workers = ((int)gridDim.x - n_state) * kGroups;
    if (tid == 0) {
        for (int b = 0; b < kGroups; ++b) {
            tc::mbar_init(&bars[b].load, 1);
            tc::mbar_init(&bars[b].sload, 1);
            tc::mbar_init(&bars[b].mma, 1);
        }
        tc::fence_mbar_init();
        tc::grid_dep_wait();  // the preparation has completed: Qp, P, Ut of every record are visible
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 128 * kGroups);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (g < kGroups) {
        const OutGroup grp{tid & 127, 2u + (uint32_t)g, &s_uok[g]};
        const uint32_t tmem = tmem_base + 128u * (uint32_t)g;
        uint8_t *gsm = sm + (uint32_t)g * OutSmem::bytes;
        for (uint32_t k = 0;; ++k) {
            if (grp.gtid == 0) {
                const int u = atomicAdd(counter, 1);
                s_unit[g] = u;
                // the unit some group will take one round later: its Qp, P, Ut into L2 meanwhile
                const int un = u + workers;
                if (un < units && un < rec_units)
                    tc::bulk_prefetch_l2(ws + records_off + (size_t)un * record_bytes + tc_record().Qp,
                                         (uint32_t)(tc_record().S - tc_record().Qp));
            }
            grp.sync();
            const int u = s_unit[g];
            if (u >= units) break;
            const int slot = u / H, h = u % H;
            int doc = 0, t0 = -1, Lc = 0;  // (stay out of range where the slot is not found)
            locate_slot(doc_slot0, cu, num_seqs, kL, slot, &doc, &t0, &Lc);
            if (!output_unit(cu, num_seqs, H, o, ws, records_off, record_bytes, slot, h, t0, Lc, gsm, &bars[g], k & 1u, tmem,
                             grp, onorm, false, sdone + u, flag_wait_ns))
                break;
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem_base, 128 * kGroups);
}

constexpr int kChainMinWorkers = 48;  // output CTAs alongside the chains, at least

// ---------------------------------------------------------------------------
// Pipe plan: preparation, state chains and outputs in one cooperative launch
// ---------------------------------------------------------------------------
// One CTA of kPipeThreads per SM.
//   CTAs [0, n_chain): one chain each (state_chain, 32 or 64 columns), which loads each chunk's record as
//     soon as its publication flag is raised and publishes each chunk's state image.
//   Every other CTA: two groups of 256 threads that take the preparation units in (chunk slot, head) order
//     (each publishes its record with a GPU-scope release once its bulk stores are complete) and, when none
//     is left, output units from the output counter.  Group 1 starts half a unit after group 0, so that the
//     two groups' heavy phases and waits alternate instead of coinciding.
// So the preparation has all but the chains' SMs to itself, the chains start with the first chunk's records
// and follow the preparation, and the outputs are formed behind the chains.  Chains of 64 columns take half
// the SMs that chains of 32 would, at a longer step (a wider epilogue); they are used once the narrow ones
// would take more than kPipeChain32Max SMs.
//
// Progress: every CTA is resident (cooperative launch).  A preparation waits for nothing but its own copies
// and MMAs, and a worker group publishes its last record before it takes any output unit; a chain waits only
// for records; an output unit waits for a record and for the chains.  Every wait is bounded.
constexpr int kPipeThreads = 512;
constexpr int kPipeChainMax = 48;    // automatic choice: at most this many chains of 64 columns ...
constexpr int kPipeChain32Max = 32;  // ... and chains of 32 columns (a shorter step) up to this many of them
constexpr uint32_t kPipePrepShared = 2 * PrepSmem::bytes;  // the worker groups' PrepShared, after their tiles
// the workers' identity image, after both groups' PrepShared (1024-byte aligned)
constexpr uint32_t kPipeIdent = (kPipePrepShared + 2 * (uint32_t)sizeof(PrepShared) + 1023u) & ~1023u;
template <int TN>
constexpr size_t pipe_smem_bytes() {
    using PipeChainCfg = ChainCfg<TN>;
    return (PipeChainCfg::bytes > kPipeIdent + kIdentBytes ? PipeChainCfg::bytes : kPipeIdent + kIdentBytes) + 1024;
}
static_assert(PrepSmem::bytes % 1024 == 0 && OutSmem::bytes <= PrepSmem::bytes, "a group's region holds a unit");

struct PipeArgs {
    const float *S0;
    float *S_final;
    __nv_bfloat16 *o;
    int32_t *ready;         // [slot * H + h]: the record is published
    int32_t *sdone;         // [slot * H + h]: columns (in 32s) whose state image is published
    int32_t *prep_counter;  // next preparation unit
    int32_t *out_counter;   // next output unit
    int n_chain;
    int total_tokens;
    unsigned long long flag_wait_ns;
    int fault;  // kFaultNoPublish only in tests of the timeout path
    OutNorm onorm;
    // Self-indexed launch (one document, no chunk index kernel before it): the go word, this call's token, the
    // flags and counters to clear (16-byte words) and the document order; go null otherwise.
    unsigned long long *go = nullptr;
    unsigned long long token = 0;
    uint4 *clear = nullptr;
    int clear_vec = 0;
    int32_t *doc_order = nullptr;
};

// Output units taken in (chunk slot, head) order from the output counter by one group of 128 threads, until
// none is left or a wait gives up (false).  `s_unit` is a shared word of the group.
__device__ bool pipe_outputs(const PrepParams &pp, const PipeArgs &a, uint8_t *gsm, OutBars *bars, uint32_t tmem,
                             const OutGroup &og, int *s_unit, int *s_pre) {
    const int H = pp.H;
    const int32_t *doc_slot0 = reinterpret_cast<const int32_t *>(pp.ws + pp.doc_slot0_off);
    const int units = doc_slot0[pp.num_seqs] * H;
    // claimed one ahead by a thread of warp 2, which does not issue the unit's copies and MMAs nor write o
    constexpr int kClaimer = 64;
    constexpr TcRecord R = tc_record();
    // (the claimer pulls the claimed unit's record, the preparation's part, into L2 while the current one runs)
    auto claim = [&]() {
        const int un = atomicAdd(a.out_counter, 1);
        *s_unit = un;
        if (un < units)
            tc::bulk_prefetch_l2(pp.ws + pp.records_off + (size_t)un * pp.record_bytes + R.Qp, (uint32_t)(R.S - R.Qp));
    };
    if (og.gtid == kClaimer) {
        claim();
        *s_pre = 0;
    }
    const OutNext nx{s_unit, units, kClaimer, a.ready, a.sdone, s_pre};
    for (uint32_t nout = 0;; ++nout) {
        og.sync();
        const int u = *s_unit, pre = *s_pre;
        og.sync();  // every thread has read s_unit before the next claim overwrites it
        if (u >= units) return true;
        if (og.gtid == kClaimer) claim();
        const int slot = u / H, h = u % H;
        int doc = 0, t0 = -1, Lc = 0;  // (stay out of range where the slot is not found)
        locate_slot(doc_slot0, pp.cu, pp.num_seqs, kL, slot, &doc, &t0, &Lc);
        if (!output_unit(pp.cu, pp.num_seqs, H, a.o, pp.ws, pp.records_off, pp.record_bytes, slot, h, t0, Lc, gsm,
                         bars, nout & 1u, tmem, og, a.onorm, false, a.sdone + (size_t)slot * H + h, a.flag_wait_ns,
                         a.ready + (size_t)slot * H + h, pre, &nx)) {
            // copies still on their way (this unit's, if it left before waiting for them; the next one's) land
            // before the CTA's shared memory can go away (best effort, 10 ms each)
            if (og.gtid == kClaimer) {
                const int pn = *s_pre;
                if (pre >= 1) tc::mbar_wait(&bars->load, nout & 1u, 10000000ull);
                if (pre == 2) tc::mbar_wait(&bars->sload, nout & 1u, 10000000ull);
                if (pn >= 1) tc::mbar_wait(&bars->load, (nout + 1) & 1u, 10000000ull);
                if (pn == 2) tc::mbar_wait(&bars->sload, (nout + 1) & 1u, 10000000ull);
            }
            return false;
        }
    }
}

// A worker CTA of the pipe plan: two groups of 256 threads, each preparing units in chunk order, then forming
// output units, once the slot table, the status word and the cleared flags are in place.
__device__ void pipe_worker(const PrepParams &pp, const PipeArgs &a, uint8_t *sm) {
    __shared__ PrepBars pbars[2];
    __shared__ OutBars obars[2];
    __shared__ uint32_t tmem_base;
    PrepShared *psh = reinterpret_cast<PrepShared *>(sm + kPipePrepShared);
    __shared__ int s_unit[2], s_ok[2], s_go, s_pre[2];
    const int tid = threadIdx.x, g = tid >> 8, gtid = tid & 255;
    const int H = pp.H;
    const int32_t *doc_slot0 = reinterpret_cast<const int32_t *>(pp.ws + pp.doc_slot0_off);
    // preparation units, and as many output units
    const int units = doc_slot0[pp.num_seqs] * H;
    if (tid == 0) s_go = 0;
    if (gtid == 0) {
        prep_bars_init(&pbars[g]);
        tc::mbar_init(&obars[g].load, 1);
        tc::mbar_init(&obars[g].sload, 1);
        tc::mbar_init(&obars[g].mma, 1);
        tc::fence_mbar_init();
    }
    if (tid < 32) {  // one allocation for both groups (the permit is given up once, for the whole CTA)
        tc::tmem_alloc(&tmem_base, 512);
        tc::tmem_relinquish();
    }
    write_identity(sm + kPipeIdent, tid, kPipeThreads);  // one identity for both groups
    tc::fence_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const PrepGroup grp{gtid, 1u + (uint32_t)g};
    uint8_t *gsm = sm + (uint32_t)g * PrepSmem::bytes;
    const uint32_t tmem = tmem_base + 256u * (uint32_t)g;
    uint32_t nprep = 0;
    bool ok = true;
    int32_t *pending = nullptr;  // the last record this group prepared, not yet published
    // preparations, claimed one ahead, so that a preparation can pull the next one's input tiles into L2; the
    // claim is made by a thread of warp 2, whose wait for the atomic overlaps the unit's first loads (the
    // group's first thread issues them)
    if (g == 1) {
        // The two groups run equal units; started together they would stay in phase, and their heavy phases
        // (operand build, solve, epilogues) and their waits would coincide.  Group 1 starts once group 0's
        // first unit has built its operands (about half a unit), so that one group's waits overlap the other's
        // arithmetic (bounded: group 0 raises the flag on any way out of its loop as well).
        if (gtid == 0) {
            const uint64_t t0 = tc::globaltimer_ns();
            while (*reinterpret_cast<volatile int *>(&s_go) == 0 && tc::globaltimer_ns() - t0 < 10000000ull)
                __nanosleep(64);
        }
        grp.sync();
    }
    // Units are taken in the order the groups start them: the first 2 W (W worker CTAs) by position, group 0s
    // before group 1s; each later one is claimed from the counter halfway through the group's current unit
    // (which also pulls its tiles into L2).
    const int nw = (int)gridDim.x - a.n_chain, wid = (int)blockIdx.x - a.n_chain;
    if (gtid == 0) s_unit[g] = g * nw + wid;
    grp.sync();
    // s_unit is read at the top of each iteration; the unit overwrites it with its claim between two of its
    // own barriers, after every thread's read and before the unit's last barrier
    for (;;) {
        const int u = s_unit[g];
        if (u >= units) break;
        const int slot = u / H, h = u % H;
        int doc = 0, t0 = -1, Lc = 0;  // (stay out of range where the slot is not found)
        locate_slot(doc_slot0, pp.cu, pp.num_seqs, kL, slot, &doc, &t0, &Lc);
        // the previous record is published once this unit's gate tile has arrived; this one's stays pending
        ok = prepare_unit(pp, slot, h, t0, Lc, gsm, &pbars[g], nprep & 1u, tmem, sm + kPipeIdent, pending, grp, psh[g],
                          a.prep_counter, 2 * nw, &s_unit[g], units, g == 0 && nprep == 0 ? &s_go : nullptr);
        ++nprep;
        if (!ok) break;
        pending = a.ready + (size_t)slot * H + h;
        if (nprep == 1) {  // the group's first record: chains may be waiting for it, so it is published at once
            if (gtid == 0) {
                tc::bulk_wait_all();
                tc::fence_proxy_async_global();
                tc::st_release_gpu(pending, 1);
            }
            pending = nullptr;
        }
    }
    grp.sync();  // every thread has read s_unit before the output phase claims into it
    if (g == 0 && gtid == 0) *reinterpret_cast<volatile int *>(&s_go) = 1;
    if (gtid == 0) tc::bulk_wait_read();  // the last unit's M' copy has read the group's shared memory
    if (gtid == 0 && pending) {  // before any output unit: a chain may be waiting for this record
        tc::bulk_wait_all();
        tc::fence_proxy_async_global();
        tc::st_release_gpu(pending, 1);
    }
    if (ok && gtid < 128)
        pipe_outputs(pp, a, gsm, &obars[g], tmem, OutGroup{gtid, 3u + (uint32_t)g, &s_ok[g]}, &s_unit[g], &s_pre[g]);
    tc::tc_fence_before();
    __syncthreads();
    if (tid < 32) tc::tmem_dealloc(tmem_base, 512);
}

template <int TN>
__global__ void __launch_bounds__(kPipeThreads, 1)
prefill_pipe_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                const float *__restrict__ beta, const int32_t *__restrict__ cu, int num_seqs, int H,
                char *__restrict__ ws, size_t doc_slot0_off, size_t records_off, size_t record_bytes, int qk_norm,
                float qk_eps, PipeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    if (a.go) {
        // Self-indexed (one document, no chunk index kernel before this launch): CTA 0 checks cu_seqlens (the
        // condition above), writes the slot table, the document order and the status word and clears the flags
        // and counters, then publishes the call's token; the other CTAs go on once they see it, as if the chunk
        // index kernel had completed.  Invalid cu_seqlens: every CTA leaves at once and nothing is written but
        // the status.
        const bool valid = num_seqs == 1 && __ldg(cu) == 0 && __ldg(cu + 1) == a.total_tokens && a.total_tokens > 0;
        tc::grid_dep_wait();  // the previous kernel in the stream, which may use this workspace, has completed
        int32_t *status = reinterpret_cast<int32_t *>(ws);
        if (blockIdx.x == 0) {
            if (valid)
                for (int i = (int)threadIdx.x; i < a.clear_vec; i += (int)blockDim.x) a.clear[i] = make_uint4(0u, 0u, 0u, 0u);
            if (threadIdx.x == 0) {
                int32_t *slot0 = reinterpret_cast<int32_t *>(ws + doc_slot0_off);
                slot0[0] = 0;
                slot0[1] = valid ? (a.total_tokens + kL - 1) / kL : 0;
                a.doc_order[0] = 0;
                status[1] = 0;
                status[kPrepCounterWord] = 0;
                status[0] = valid ? 0 : 1;
            }
            __syncthreads();
            if (threadIdx.x == 0 && valid) {
                __threadfence();
                tc::st_release_gpu_u64(a.go, a.token);
            }
        } else if (valid) {
            __shared__ int s_go_ok;
            if (threadIdx.x == 0) {
                s_go_ok = tc::wait_u64_eq(a.go, a.token, a.flag_wait_ns);
                if (!s_go_ok) flag_timeout(ws);
            }
            __syncthreads();
            if (!s_go_ok) return;
        }
        if (!valid) return;
    }
    const bool worker = (int)blockIdx.x >= a.n_chain;
    tc::grid_dep_wait();  // the chunk index kernel (if any): slot table, status word, cleared flags
    if (*reinterpret_cast<const volatile int32_t *>(ws) != 0) return;  // invalid cu_seqlens: write nothing
    uint8_t *sm = align1024(smem_raw);
    const PrepParams pp{&tm_q,       &tm_k,        &tm_v,   &tm_g,  beta, cu, num_seqs, H, ws, doc_slot0_off,
                        records_off, record_bytes, qk_norm, qk_eps};
    if (worker) {
        pipe_worker(pp, a, sm);
        return;
    }
    ChainLinks links;
    links.sdone = a.sdone;
    links.publish = a.fault != kFaultNoPublish;
    links.ready = a.ready;
    links.flag_wait_ns = a.flag_wait_ns;
    state_chain<TN>(cu, num_seqs, H, a.S0, a.S_final, ws, doc_slot0_off, records_off, record_bytes,
                                  (int)blockIdx.x, sm, links);
}


// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [T, H, 128] bf16 tensor, boxes of 64 channels x 1 head x 64 tokens, 128-byte swizzle.
bool make_input_map(CUtensorMap *map, const void *base, int total_tokens, int H) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)total_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kL};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [T, H, 128] fp32 gates, boxes of 128 channels x 1 head x 64 tokens, unswizzled rows.
bool make_gate_map(CUtensorMap *map, const float *base, int total_tokens, int H) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)total_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 4, (cuuint64_t)H * kD * 4};
    cuuint32_t box[3] = {(cuuint32_t)kD, 1, (cuuint32_t)kL};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The four tensor maps of a call, remembered for the (q, k, v, g, T, H) they were encoded for: a serving
// loop that reuses its buffers pays for the encoding once.  A tensor map holds only the base address, sizes
// and strides, so an entry stays valid for as long as the same addresses describe the same shapes.
struct InputMaps {
    CUtensorMap q, k, v, g;
};
bool input_maps(const void *q, const void *k, const void *v, const float *g, int T, int H, InputMaps *out) {
    struct Entry {
        const void *q, *k, *v, *g;
        int T, H;
        InputMaps maps;
    };
    constexpr int kEntries = 16;
    static std::mutex lock;
    static Entry cache[kEntries];
    static int used = 0, next = 0;
    {
        std::lock_guard<std::mutex> guard(lock);
        for (int i = 0; i < used; ++i) {
            const Entry &e = cache[i];
            if (e.q == q && e.k == k && e.v == v && e.g == g && e.T == T && e.H == H) {
                *out = e.maps;
                return true;
            }
        }
    }
    InputMaps m;
    if (!make_input_map(&m.q, q, T, H) || !make_input_map(&m.k, k, T, H) || !make_input_map(&m.v, v, T, H) ||
        !make_gate_map(&m.g, g, T, H))
        return false;
    std::lock_guard<std::mutex> guard(lock);
    cache[next] = Entry{q, k, v, g, T, H, m};
    next = (next + 1) % kEntries;
    used = used < kEntries ? used + 1 : kEntries;
    *out = m;
    return true;
}

// CTAs of `kernel` that fit on the whole device at once (0 if unknown), cached per device: the smallest of
// what the SM's registers, shared memory (dynamic + static + the per-CTA reserve), threads and tensor
// memory (512 columns, `tmem_cols` per CTA) allow, times the SM count.  Worked out here from the
// kernel's attributes because the runtime's occupancy query does not know about tensor memory.
template <typename K>
int resident_ctas(K kernel, int threads, int smem, int tmem_cols) {
    static std::mutex lock;
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> g(lock);
    if (!cached[dev]) {
        cudaFuncAttributes fa;
        int sms = 0, smem_sm = 0, regs_sm = 0, thr_sm = 0, reserve = 0;
        if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&reserve, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
            return 0;
        const int regs_cta = ((fa.numRegs + 7) / 8 * 8) * 32 * ((threads + 31) / 32);
        int per_sm = smem_sm / (smem + (int)fa.sharedSizeBytes + reserve);
        per_sm = std::min(per_sm, regs_sm / std::max(regs_cta, 1));
        per_sm = std::min(per_sm, thr_sm / threads);
        per_sm = std::min(per_sm, 512 / tmem_cols);
        cached[dev] = std::max(per_sm, 0) * sms;
    }
    return cached[dev];
}

constexpr int kPrepSmem = PrepSmem::bytes + kIdentBytes + 1024;  // a unit's tiles, then the identity
constexpr int kStateSmem = ChainCfg<32>::bytes + 1024;
constexpr int kStateSmem64 = ChainCfg<64>::bytes + 1024;
constexpr int kFoldSmem32 = FoldCfg<32>::bytes + 1024;
constexpr int kFoldSmem64 = FoldCfg<64>::bytes + 1024;
constexpr int kOutSmem = OutSmem::bytes + 1024;

// Per-device facts the launches need, worked out (and the kernels' shared-memory limits raised) once per
// device rather than on every call.
struct DeviceSetup {
    cudaError_t err = cudaErrorNotReady;
    int sms = 0;
    int prep_resident = 0, out_resident = 0;
};
const DeviceSetup &device_setup() {
    static std::mutex lock;
    static DeviceSetup setups[64];
    int dev = 0;
    static DeviceSetup none;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        none.err = cudaErrorInvalidDevice;
        return none;
    }
    std::lock_guard<std::mutex> g(lock);
    DeviceSetup &d = setups[dev];
    if (d.err == cudaErrorNotReady) {
        cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (!e) e = cudaFuncSetAttribute(prefill_prepare_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
        if (!e) e = cudaFuncSetAttribute(prefill_state_tc<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kStateSmem);
        if (!e)
            e = cudaFuncSetAttribute(prefill_state_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kStateSmem64);
        if (!e) e = cudaFuncSetAttribute(prefill_chain_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kStateSmem);
        if (!e)
            e = cudaFuncSetAttribute(prefill_state_fold_tc<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kFoldSmem32);
        if (!e)
            e = cudaFuncSetAttribute(prefill_state_fold_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kFoldSmem64);
        if (!e) e = cudaFuncSetAttribute(prefill_output_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kOutSmem);
        if (!e)
            e = cudaFuncSetAttribute(prefill_pipe_tc<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)pipe_smem_bytes<32>());
        if (!e)
            e = cudaFuncSetAttribute(prefill_pipe_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)pipe_smem_bytes<64>());

        if (!e) {
            cudaFuncSetAttribute(prefill_prepare_tc, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
            cudaFuncSetAttribute(prefill_output_tc, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
            d.prep_resident = resident_ctas(prefill_prepare_tc, kPrepThreads, kPrepSmem, 256);
            d.out_resident = resident_ctas(prefill_output_tc, 128, kOutSmem, 128);
        }
        d.err = e;
    }
    return d;
}

// A token per self-indexed pipe launch, unique within the process (a counter from a clock-derived start), so
// that the go word a launch waits for was written by this launch.
unsigned long long next_call_token() {
    static std::atomic<unsigned long long> counter{
        (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() * 0x9E3779B97F4A7C15ull};
    unsigned long long z = counter.fetch_add(0x9E3779B97F4A7C15ull) + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;  // (the SplitMix64 finaliser)
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return (z ^ (z >> 31)) | 1ull;
}

// Test hooks (include/kda_testing.h): a forced launch plan and an injected fault with a short wait bound.
std::atomic<int> g_test_plan{-1};
std::atomic<int> g_test_fault{0};
std::atomic<long long> g_test_wait_ns{0};

// Launches `kernel` as a cooperative grid (every CTA co-resident, or the launch fails), allowed to start while
// the previous kernel in the stream finishes where the runtime accepts both attributes together.
template <typename... KArgs, typename... Args>
cudaError_t launch_cooperative(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                               Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e == cudaSuccess || e == cudaErrorCooperativeLaunchTooLarge) return e;
    cudaGetLastError();  // the pair of attributes was refused: a plain cooperative launch instead
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace

// Testing hooks (not part of the product path; see include/kda_testing.h).
void testing_set_plan(int plan) { g_test_plan.store(plan); }
void testing_set_fault(int fault, long long wait_ns) {
    g_test_fault.store(fault);
    g_test_wait_ns.store(wait_ns);
}
int testing_fault() { return g_test_fault.load(); }

bool pipe_self_indexed(TcPlan plan, int num_seqs) {
#ifdef KDA_DEBUG_BOUNDS
    (void)plan;
    (void)num_seqs;
    return false;
#else
    return plan == TC_PIPE && num_seqs == 1;
#endif
}

TcPlan tc_plan(int num_seqs, int H, int total_tokens) {
    // The pipe plan for at most kPipeChainMax chains of 64 columns, else the preparation and the state pass
    // (which, without the gated output normalisation, forms the outputs itself; with it, an output pass
    // follows, since that normalisation needs whole rows).  Measured on one document of 4096 tokens (pass
    // times, calls queued back to back): 8 heads pipe 75 us, chain 97, three 100; 24 heads pipe 132, three
    // 141, chain 154; 32 heads three 161, chain 162, pipe 194.  The chain plan is taken only when the test
    // hook forces it.
    const WsLayout lay = ws_layout(total_tokens, num_seqs, H, kD, kD, kL, PATH_TC);
    if (lay.max_slots <= 0 || total_tokens <= 0) return TC_THREE;
    const int forced = g_test_plan.load();
    if (forced == TC_THREE) return TC_THREE;
    const DeviceSetup &d = device_setup();
    if (d.err) return TC_THREE;
    const long long chains32 = (long long)num_seqs * H * kNTile, chains64 = chains32 / 2;
    const bool pipe_fits = chains64 + kChainMinWorkers <= d.sms;
    const bool chain_fits = chains32 + kChainMinWorkers <= d.sms;
    if (forced == TC_PIPE) return pipe_fits ? TC_PIPE : TC_THREE;
    if (forced == TC_CHAIN) return chain_fits ? TC_CHAIN : TC_THREE;
    return pipe_fits && chains64 <= kPipeChainMax ? TC_PIPE : TC_THREE;
}

cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const float *g, const float *beta,
                              const int32_t *cu, int num_seqs, int total_tokens, int H, const float *S0, void *o,
                              float *S_final, void *ws, TcPlan plan, const Fusion &fu, cudaStream_t st,
                              Marks &marks) {
    const OutNorm onorm{static_cast<const __nv_bfloat16 *>(fu.gate), fu.weight, fu.out_eps};
    const WsLayout lay = ws_layout(total_tokens, num_seqs, H, kD, kD, kL, PATH_TC);
    char *w = static_cast<char *>(ws);
    const DeviceSetup &dset = device_setup();
    if (dset.err) return dset.err;
    cudaError_t e;
    int32_t *flags = reinterpret_cast<int32_t *>(w + lay.flags_off);
    const size_t nflag = (size_t)lay.max_slots * H;
    const long long wait = g_test_wait_ns.load();
    const unsigned long long flag_wait = wait > 0 ? (unsigned long long)wait : kFlagWaitNs;
    if (plan == TC_PIPE) {
        InputMaps m;
        if (!input_maps(q, k, v, g, total_tokens, H, &m)) return cudaErrorInvalidValue;
        PipeArgs a;
        a.S0 = S0;
        a.S_final = S_final;
        a.o = static_cast<__nv_bfloat16 *>(o);
        a.ready = flags;
        a.sdone = flags + nflag;
        a.prep_counter = flags + 2 * nflag;
        a.out_counter = flags + 2 * nflag + 1;
        a.n_chain = num_seqs * H * (kD / 64);
        a.total_tokens = total_tokens;
        a.flag_wait_ns = flag_wait;
        a.fault = g_test_fault.load();
        a.onorm = onorm;
        const bool self = pipe_self_indexed(plan, num_seqs);
        if (self) {
            a.go = reinterpret_cast<unsigned long long *>(w) + kGoWord / 2;
            a.token = next_call_token();
            a.clear = reinterpret_cast<uint4 *>(flags);
            a.clear_vec = (int)(lay.flags_bytes / 16);
            a.doc_order = reinterpret_cast<int32_t *>(w + lay.doc_order_off);
        }
        marks.before(st, "prefill_pipe_tc");
        // chains of 32 columns while they are few (a shorter step), else of 64 (half the SMs)
        const long long chains32 = (long long)num_seqs * H * kNTile;
        if (chains32 <= kPipeChain32Max) {
            a.n_chain = (int)chains32;
            e = launch_cooperative(prefill_pipe_tc<32>, dim3((unsigned)dset.sms), dim3(kPipeThreads),
                                   pipe_smem_bytes<32>(), st, m.q, m.k, m.v, m.g, beta, cu, num_seqs, H, w,
                                   lay.doc_slot0_off, lay.records_off, lay.record_bytes, fu.qk_norm, fu.qk_eps, a);
        } else {
            e = launch_cooperative(prefill_pipe_tc<64>, dim3((unsigned)dset.sms), dim3(kPipeThreads),
                                   pipe_smem_bytes<64>(), st, m.q, m.k, m.v, m.g, beta, cu, num_seqs, H, w,
                                   lay.doc_slot0_off, lay.records_off, lay.record_bytes, fu.qk_norm, fu.qk_eps, a);
        }
        if (e != cudaErrorCooperativeLaunchTooLarge) return e;
        // Fewer SMs are available to this context than the device has: nothing was launched; run the three
        // kernels instead (after the chunk index kernel, which a self-indexed launch left out).
        cudaGetLastError();
        marks.n--;
        plan = TC_THREE;
        if (self && (e = launch_chunk_index(cu, num_seqs, total_tokens, kL, ws, nullptr, 0, st, marks)))
            return e;
    }
    if (lay.max_slots > 0 && total_tokens > 0) {
        InputMaps m;
        if (!input_maps(q, k, v, g, total_tokens, H, &m)) return cudaErrorInvalidValue;
        marks.before(st, "prefill_prepare_tc");
        // persistent: the co-resident CTAs (or one per unit, if fewer) claim the units in turn
        const long long units = (long long)lay.max_slots * H;
        const unsigned grid = (unsigned)std::max(1LL, std::min<long long>(dset.prep_resident, units));
        if ((e = launch_dependent(prefill_prepare_tc, dim3(grid), dim3(kPrepThreads), (size_t)kPrepSmem, st, m.q,
                                  m.k, m.v, m.g, beta, cu, num_seqs, H, w, lay.doc_slot0_off, lay.records_off,
                                  lay.record_bytes, fu.qk_norm, fu.qk_eps)))
            return e;
    }
    if (num_seqs == 0) return cudaSuccess;
    if (plan == TC_CHAIN) {
        const int n_state = num_seqs * H * kNTile;
        // Cooperative: the output groups wait for the chain CTAs' publications, so every CTA must be resident.
        marks.before(st, "prefill_chain_tc");
        e = launch_cooperative(prefill_chain_tc, dim3((unsigned)dset.sms), dim3(kStateThreads), (size_t)kStateSmem,
                               st, cu, num_seqs, H, S0, S_final, static_cast<__nv_bfloat16 *>(o), w,
                               lay.doc_slot0_off, lay.records_off, lay.record_bytes, n_state, flags + nflag,
                               flags + 2 * nflag, flag_wait, g_test_fault.load(), onorm);
        if (e != cudaErrorCooperativeLaunchTooLarge) return e;
        // Fewer SMs are available to this context than the device has: nothing was launched; run the state
        // pass and the output pass as separate kernels instead.
        cudaGetLastError();
        marks.n--;
    }
    // Chains of 32 columns while they fit on the SMs at once, else of 64 (half as many: fewer waves of chains)
    const size_t chains32 = (size_t)num_seqs * H * kNTile;
    if (!onorm.gate) {  // the chains form the outputs themselves: no output pass
        marks.before(st, "prefill_state_fold_tc");
        if (chains32 <= (size_t)dset.sms)
            return launch_dependent(prefill_state_fold_tc<32>, dim3((unsigned)chains32), dim3(kFoldThreads),
                                    (size_t)kFoldSmem32, st, cu, num_seqs, H, S0, S_final,
                                    static_cast<__nv_bfloat16 *>(o), w, lay.doc_slot0_off, lay.records_off,
                                    lay.record_bytes, lay.doc_order_off);
        return launch_dependent(prefill_state_fold_tc<64>, dim3((unsigned)(chains32 / 2)), dim3(kFoldThreads),
                                (size_t)kFoldSmem64, st, cu, num_seqs, H, S0, S_final, static_cast<__nv_bfloat16 *>(o),
                                w, lay.doc_slot0_off, lay.records_off, lay.record_bytes, lay.doc_order_off);
    }
    marks.before(st, "prefill_state_tc");
    if (chains32 <= (size_t)dset.sms)
        e = launch_dependent(prefill_state_tc<32>, dim3((unsigned)chains32), dim3(kStateThreads), (size_t)kStateSmem,
                             st, cu, num_seqs, H, S0, S_final, w, lay.doc_slot0_off, lay.records_off,
                             lay.record_bytes, lay.doc_order_off);
    else
        e = launch_dependent(prefill_state_tc<64>, dim3((unsigned)(chains32 / 2)), dim3(kStateThreads),
                             (size_t)kStateSmem64, st, cu, num_seqs, H, S0, S_final, w, lay.doc_slot0_off,
                             lay.records_off, lay.record_bytes, lay.doc_order_off);
    if (e) return e;
    if (lay.max_slots > 0 && total_tokens > 0) {
        marks.before(st, "prefill_output_tc");
        if ((e = launch_dependent(prefill_output_tc, dim3((unsigned)lay.max_slots, (unsigned)H), dim3(128),
                                  (size_t)kOutSmem, st, cu, num_seqs, H, static_cast<__nv_bfloat16 *>(o), w,
                                  lay.doc_slot0_off, lay.records_off, lay.record_bytes, dset.out_resident, onorm)))
            return e;
    }
    return cudaSuccess;
}

}  // namespace kda
