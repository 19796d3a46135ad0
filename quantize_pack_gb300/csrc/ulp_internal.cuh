// Internal helpers of the ulp library: geometry, argument checks, device
// conversions and reductions.  Not part of the ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <cstdarg>
#include <cstdio>

#include "ulp.h"

namespace ulp {

constexpr int kGK = 64;    // K group rows
constexpr int kGQ = 128;   // Q group rows
constexpr float kEps = 1e-7f;

// ------------------------------------------------------------------ errors

int fail(int status, const char *fmt, ...);
int check_launch(const char *what);

// ---------------------------------------------------------------- geometry

__host__ __device__ __forceinline__ int slots(int L, int G) { return (L + G - 1) / G + (L % G != 0); }
__host__ __device__ __forceinline__ int first_group(int r, int L, int G)
{
    return (int)(((long long)r * L) / G);
}
__host__ __device__ __forceinline__ int last_group(int r, int L, int G)
{
    return (int)(((long long)(r + 1) * L - 1) / G);
}
__host__ __device__ __forceinline__ size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

struct ChunkLayout {
    size_t q, k, v, qs, ks, bytes;
};

__host__ __device__ __forceinline__ ChunkLayout chunk_layout(int B, int L, int h, int D)
{
    ChunkLayout c;
    size_t n = (size_t)B * L * h * D;
    c.q = 0;
    c.k = align16(n);
    c.v = c.k + align16(n);
    c.qs = c.v + align16(n);
    c.ks = c.qs + align16(sizeof(float) * (size_t)B * h * slots(L, kGQ));
    c.bytes = c.ks + align16(sizeof(float) * (size_t)B * h * slots(L, kGK));
    return c;
}

// ---------------------------------------------------------- argument checks

bool aligned16(const void *p);
bool aligned4(const void *p);
int check_common(int dtype, int B, int L, int H, int D, int rank, int world_size,
                 int used_sequence, int enable_pdl);
int check_world(int world_size);

// ------------------------------------------------------------ device side

// 8 consecutive bf16/fp16 values (one 16-byte vector) -> fp32, exactly.
template <int DT>
__device__ __forceinline__ void to_f32x8(const uint4 &v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (DT == ULP_BF16) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        } else {
            __half2 hv = *reinterpret_cast<const __half2 *>(&w[i]);
            float2 p = __half22float2(hv);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    }
}

// Streaming 16-byte load (read once: do not keep in L1).
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_min(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float floor_eps(float x) { return x < kEps ? kEps : x; }

// int8 code: round half to even, saturate to [-128, 127].
__device__ __forceinline__ int int8_code(float y)
{
    int i = __float2int_rn(y);
    return max(-128, min(127, i));
}

// Pack four int codes (low byte of each) into one word, first in the lowest byte.
__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d)
{
    uint32_t lo = __byte_perm((uint32_t)a, (uint32_t)b, 0x0040);
    uint32_t hi = __byte_perm((uint32_t)c, (uint32_t)d, 0x0040);
    return __byte_perm(lo, hi, 0x5410);
}

// Two fp32 -> two E4M3 bytes (x in the low byte), round to nearest even, satfinite.
__device__ __forceinline__ uint32_t e4m3x2(float x, float y)
{
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x, y), __NV_SATFINITE, __NV_E4M3);
}

}  // namespace ulp
