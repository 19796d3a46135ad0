// Throughput of back-to-back 5th-generation tensor-core MMAs on this GPU:
// one CTA per SM, one thread issuing `iters` tcgen05.mma of one kind
// (M = 128, N = 128 or 256, one K step of 32 bytes per row: K = 16 for
// kind::f16, K = 32 for kind::f8f6f4 with E4M3 operands) from shared-memory
// operands into a TMEM accumulator, then a commit and a bounded wait.  Prints,
// per kind and N, the dense rate in TFLOP/s over the whole grid, timed with
// CUDA events.  The operands' values do not matter to the rate.  (kind::i8
// has no form for this target: ptxas rejects it for sm_103a.)
//
//   mma_rate [iters]      -> lines "<kind> <M> <N> <K> <iters> <ms> <TFLOP/s>"
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "ulp_tc.cuh"

using namespace ulp::tc;

enum { KIND_F16 = 0, KIND_F8 = 1 };

// instruction descriptor: f32 accumulator (bits 4-5 = 1), A and B of type 0
// (f16 for kind::f16, E4M3 for kind::f8f6f4; bits 7-9, 10-12), both K-major,
// N >> 3 in bits 17-22, M >> 4 in bits 24-28
__host__ __device__ constexpr uint32_t idesc(int M, int N)
{
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <int KIND>
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc)
{
    if (KIND == KIND_F16)
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                     "l"(a), "l"(b), "r"(id), "r"(acc) : "memory");
    else
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                     "l"(a), "l"(b), "r"(id), "r"(acc) : "memory");
}

template <int KIND, int N>
__global__ void __launch_bounds__(128) mma_rate_kernel(int iters, int *status)
{
    constexpr int M = 128;
    // one tile of 256 rows x 128 B (one swizzle atom wide); A reads its first
    // 128 rows, B its first N
    __shared__ __align__(1024) uint8_t b_tile[256 * 128];
    uint8_t *a_tile = b_tile;
    __shared__ uint64_t done;
    __shared__ uint32_t tmem_slot;
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < N * 128 / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(b_tile)[i] = 0x3c003c00u;
    if (warp == 0) tmem_alloc(&tmem_slot, 256);
    if (threadIdx.x == 0) {
        mbar_init(&done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    fence_smem_to_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;
    if (threadIdx.x == 0) {
        const uint64_t a = sw128_desc(smem_u32(a_tile)), b = sw128_desc(smem_u32(b_tile));
        const uint32_t id = idesc(M, N);
        for (int i = 0; i < iters; ++i) mma<KIND>(tmem, a, b, id, i > 0);
        mma_commit(&done);
        if (!mbar_wait(&done, 0, 2000000000ull)) atomicExch(status, 1);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// dynamic shared memory requested (and not used) so that one CTA fits an SM
constexpr int kPadSmem = 120 * 1024;

template <int KIND, int N>
static int run(const char *name, int k, int iters, int sms, int *status)
{
    cudaFuncSetAttribute(mma_rate_kernel<KIND, N>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPadSmem);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    mma_rate_kernel<KIND, N><<<sms, 128, kPadSmem>>>(iters / 10, status);   // warm-up
    cudaEventRecord(e0);
    mma_rate_kernel<KIND, N><<<sms, 128, kPadSmem>>>(iters, status);
    cudaEventRecord(e1);
    if (cudaEventSynchronize(e1) != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", name, cudaGetErrorString(cudaGetLastError()));
        return 1;
    }
    float ms = 0.0f;
    cudaEventElapsedTime(&ms, e0, e1);
    const double ops = 2.0 * 128 * N * k * (double)iters * sms;
    printf("%s 128 %d %d %d %.4f %.1f\n", name, N, k, iters, ms, ops / (ms * 1e-3) / 1e12);
    return 0;
}

int main(int argc, char **argv)
{
    const int iters = argc > 1 ? atoi(argv[1]) : 20000;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int *status = nullptr;
    if (cudaMalloc(&status, sizeof(int)) != cudaSuccess) return 1;
    cudaMemset(status, 0, sizeof(int));
    int bad = run<KIND_F16, 128>("f16", 16, iters, sms, status);
    bad |= run<KIND_F16, 256>("f16", 16, iters, sms, status);
    bad |= run<KIND_F8, 128>("f8f6f4_e4m3", 32, iters, sms, status);
    bad |= run<KIND_F8, 256>("f8f6f4_e4m3", 32, iters, sms, status);
    int h = 0;
    cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost);
    if (h) {
        fprintf(stderr, "a wait timed out\n");
        return 2;
    }
    return bad;
}
