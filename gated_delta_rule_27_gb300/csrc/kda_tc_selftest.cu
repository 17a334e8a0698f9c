// kda_tc_selftest.cu -- a one-CTA tcgen05 GEMM over caller-built shared-memory
// images, used by the GPU tests to check the descriptor encodings in
// kda_tc.cuh against torch on the same bf16 operands.  Not part of the ABI.
//
// The caller passes the bytes of the A and B operand images exactly as they
// must sit in shared memory, the descriptor templates, and per-MMA start
// offsets inside each image; the kernel copies the images to 1024-byte
// aligned shared memory, issues the MMAs from one thread, waits (bounded),
// and writes the 128 x N fp32 accumulator to d_out.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int kRegion = 64 * 1024;  // per operand; images are at most 32 KB, so any
                                    // descriptor reach the tests use stays inside
constexpr int kMaxSteps = 16;

struct SelftestArgs {
    uint64_t a_desc_base, b_desc_base;
    uint32_t idesc;
    int steps, N, a_bytes, b_bytes;
    int a_off[kMaxSteps], b_off[kMaxSteps];
};

__global__ void __launch_bounds__(128) tc_selftest_kernel(const uint4 *__restrict__ a_img,
                                                          const uint4 *__restrict__ b_img, SelftestArgs args,
                                                          float *__restrict__ d_out, int *__restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t raw = tc::smem_u32(smem_raw);
    uint8_t *base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t *sa = base, *sb = base + kRegion;
    for (int i = tid; i < args.a_bytes / 16; i += 128) reinterpret_cast<uint4 *>(sa)[i] = a_img[i];
    for (int i = tid; i < args.b_bytes / 16; i += 128) reinterpret_cast<uint4 *>(sb)[i] = b_img[i];
    tc::fence_async_smem();
    uint32_t ncols = 32;
    while ((int)ncols < args.N) ncols <<= 1;
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, ncols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t d_tmem = tmem_base;
    if (tid == 0) {
        for (int s = 0; s < args.steps; ++s) {
            const uint64_t a = tc::smem_desc(args.a_desc_base, tc::smem_u32(sa + args.a_off[s]));
            const uint64_t b = tc::smem_desc(args.b_desc_base, tc::smem_u32(sb + args.b_off[s]));
            tc::mma_bf16(d_tmem, a, b, args.idesc, s > 0);
        }
        tc::mma_commit(&bar);
    }
    __syncwarp();
    const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&bar, 0));  // warp-uniform: tcgen05.ld is collective
    if (!ok && lane == 0) atomicExch(status, 1);
    tc::tc_fence_after();
    if (ok) {
        const int row = warp * 32 + lane;
        for (int c = 0; c < args.N; c += 16) {
            float r[16];
            tc::tmem_ld16(d_tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, r);
#pragma unroll
            for (int i = 0; i < 16; ++i) d_out[row * args.N + c + i] = r[i];
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0 && ok) tc::tmem_dealloc(d_tmem, ncols);
}

}  // namespace
}  // namespace kda

extern "C" __attribute__((visibility("default"))) int kda_internal_tc_gemm_selftest(
    const void *a_img, int a_bytes, const void *b_img, int b_bytes, unsigned long long a_desc_base,
    unsigned long long b_desc_base, unsigned idesc, int steps, const int *a_off, const int *b_off, int N,
    float *d_out, int *status, void *stream) {
    using namespace kda;
    if (steps < 1 || steps > kMaxSteps || N < 16 || N > 256 || N % 16) return 1;
    if (a_bytes <= 0 || b_bytes <= 0 || a_bytes > 32768 || b_bytes > 32768 || a_bytes % 16 || b_bytes % 16) return 1;
    SelftestArgs args;
    args.a_desc_base = a_desc_base;
    args.b_desc_base = b_desc_base;
    args.idesc = idesc;
    args.steps = steps;
    args.N = N;
    args.a_bytes = a_bytes;
    args.b_bytes = b_bytes;
    for (int s = 0; s < kMaxSteps; ++s) {
        args.a_off[s] = s < steps ? a_off[s] : 0;
        args.b_off[s] = s < steps ? b_off[s] : 0;
        if (args.a_off[s] < 0 || args.a_off[s] >= 32768 || args.b_off[s] < 0 || args.b_off[s] >= 32768) return 1;
    }
    const int smem = 2 * kRegion + 1024;
    if (cudaFuncSetAttribute(tc_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 2;
    tc_selftest_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(a_img), static_cast<const uint4 *>(b_img), args, d_out, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
