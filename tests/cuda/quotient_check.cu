// Exhaustive check of the corrected quotient used by the pack kernel's codecs:
// for binary32 significands x, s in [1, 2),
//     r = rn(1/s), y = rn(x r), z = fma(fma(-y, s, x), r, y)
// must equal the IEEE quotient __fdiv_rn(x, s).  Rounding to nearest commutes
// with power-of-two scaling, so this covers every quotient whose r, y and
// residual stay normal.  Test program: prints the mismatch count.
//   quotient_check <x_bits>   checks x significands on a 2^-x_bits grid
//                             (7: bf16, 10: fp16, 23: every binary32)
#include <cstdint>
#include <cstdio>
#include <cstdlib>

__device__ unsigned long long g_bad;
__device__ unsigned int g_first[3];   // count of recorded mismatches, then s, x of the first

__global__ void check(int x_count, uint32_t x_base, uint32_t x_step)
{
    const uint32_t sm = blockIdx.x * blockDim.x + threadIdx.x;   // s significand
    if (sm >= (1u << 23)) return;
    const float s = __uint_as_float(0x3F800000u | sm);
    const float r = __frcp_rn(s);
    unsigned long long bad = 0;
    for (int i = 0; i < x_count; ++i) {
        const uint32_t xm = x_base + (uint32_t)i * x_step;
        const float x = __uint_as_float(0x3F800000u | xm);
        const float y = __fmul_rn(x, r);
        const float z = __fmaf_rn(__fmaf_rn(-y, s, x), r, y);
        if (__float_as_uint(z) != __float_as_uint(__fdiv_rn(x, s))) {
            ++bad;
            if (atomicAdd(&g_first[0], 1u) == 0) {
                g_first[1] = sm;
                g_first[2] = xm;
            }
        }
    }
    if (bad) atomicAdd(&g_bad, bad);
}

int main(int argc, char **argv)
{
    const int x_bits = argc > 1 ? atoi(argv[1]) : 23;
    if (x_bits < 0 || x_bits > 23) return 2;
    const uint32_t step = 1u << (23 - x_bits), nx = 1u << x_bits;
    const uint32_t per_launch = 4096;                 // x values per thread per launch
    for (uint32_t done = 0; done < nx; done += per_launch) {
        const uint32_t cnt = nx - done < per_launch ? nx - done : per_launch;
        check<<<(1u << 23) / 256, 256>>>((int)cnt, done * step, step);
        const cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            printf("cuda error: %s\n", cudaGetErrorString(e));
            return 3;
        }
    }
    unsigned long long bad = 0;
    unsigned int first[3] = {0, 0, 0};
    cudaMemcpyFromSymbol(&bad, g_bad, sizeof bad);
    cudaMemcpyFromSymbol(first, g_first, sizeof first);
    printf("pairs %llu mismatches %llu first_s %u first_x %u\n",
           (unsigned long long)nx << 23, bad, first[1], first[2]);
    return 0;
}
