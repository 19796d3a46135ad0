// Internal helpers of the ulp library: geometry, argument checks, device
// conversions and reductions.  Not part of the ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
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

// ------------------------------------------ programmatic dependent launch
//
// enable_pdl: -1 = on when the device supports it (compute capability >= 9),
// 0 = off, 1 = on, 2 = on and the pack kernel may read its inputs (q, k, v,
// k_mean, v_scale) before the preceding kernel on the stream completes (the
// caller guarantees that kernel does not write them).  Every kernel here lets
// its dependents launch as soon as all its CTAs have started
// (griddepcontrol.launch_dependents) and waits for its predecessor's
// completion (griddepcontrol.wait) before any read of a buffer the
// predecessor may write and before its first global write; without a
// programmatic launch both instructions are no-ops.
bool pdl_enabled(int enable_pdl);

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch a kernel taking one argument struct, optionally as a programmatic
// dependent launch.
template <typename Args>
cudaError_t launch_kernel(void (*kernel)(Args), dim3 grid, dim3 block, cudaStream_t stream, bool pdl,
                          const Args &args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

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

// 16-byte asynchronous global -> shared copy (completes at cp_async_wait_all).
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

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
__device__ __forceinline__ uint32_t pack4(uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    uint32_t lo = __byte_perm(a, b, 0x0040);
    uint32_t hi = __byte_perm(c, d, 0x0040);
    return __byte_perm(lo, hi, 0x5410);
}


// ---------------------------------------------------------------------------
// Exact quantisation of x / s by bracketing.
//
// The codes are those of the IEEE quotient z = rn(x / s).  Let r = rn(1/s)
// (__frcp_rn) and r_lo = rn(r (1 - 2^-22)), r_hi = rn(r (1 + 2^-22)).  Each of
// the three roundings in x * r_lo (and x * r_hi) is within 2^-24 relative, as
// is z's own, so for x != 0 the exact products x * r_lo and x * r_hi lie
// strictly on either side of z (for x < 0 the sides swap), with a bracket
// narrower than 2^-20 |x / s|.  Both the int8 code (round half to even, then
// saturate) and the E4M3 code (RNE, satfinite) are monotone in their input, so
// when the two bracket ends give the same code, z gives it too.  Otherwise --
// z near a rounding boundary, about 2^-14 of the values -- the code is taken
// from the IEEE quotient __fdiv_rn(x, s).
//
// int8: fma(x, r, 1.5 * 2^23) rounds the exact product to an integer (ties to
// even) in one step while |x r| < 2^22: the sum lies in the binade of unit
// spacing.  With |x| <= rn(127.25 s) the quotient is below 127.5 in magnitude,
// so no saturation applies and the code is the sum's low byte.
// E4M3: both ends are rounded products (one more rounding each), so the V
// brackets use the wider margin 2^-21.
constexpr float kRoundMagic = 12582912.0f;   // 1.5 * 2^23
constexpr float kBracketLo = 0.999999761581420898f;   // 1 - 2^-22
constexpr float kBracketHi = 1.000000238418579102f;   // 1 + 2^-22
constexpr float kBracketLoV = 0.999999523162841797f;  // 1 - 2^-21
constexpr float kBracketHiV = 1.000000476837158203f;  // 1 + 2^-21

struct Int8Scale {
    float s, lo, hi, xlim;   // scale, bracketing reciprocals, largest |x| without saturation
};

__device__ __forceinline__ Int8Scale int8_scale(float s)
{
    const float r = __frcp_rn(s);
    return Int8Scale{s, __fmul_rn(r, kBracketLo), __fmul_rn(r, kBracketHi), __fmul_rn(127.25f, s)};
}

// ---- packed fp32 pairs (Blackwell f32x2 arithmetic: two lanes per instruction)

__device__ __forceinline__ unsigned long long f2pack(float a, float b)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long r, float &a, float &b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2fma(unsigned long long a, unsigned long long b,
                                                    unsigned long long c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ unsigned long long f2mul(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long f2sub(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Eight int8 codes of x[e] / s, packed little-endian into two words.  The two
// bracket ends agree iff their bit patterns do; the range test folds |x| by
// max.  (NaN inputs are outside the domain: fmaxf drops them.)
__device__ __forceinline__ uint2 int8_codes8(const float (&x)[8], const Int8Scale &q)
{
    uint32_t t[8], diff = 0;
    float xm = 0.0f;
    const unsigned long long lo2 = f2pack(q.lo, q.lo), hi2 = f2pack(q.hi, q.hi);
    const unsigned long long mg2 = f2pack(kRoundMagic, kRoundMagic);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const unsigned long long x2 = f2pack(x[e], x[e + 1]);
        float a0, a1, b0, b1;
        f2unpack(f2fma(x2, lo2, mg2), a0, a1);
        f2unpack(f2fma(x2, hi2, mg2), b0, b1);
        t[e] = __float_as_uint(a0);
        t[e + 1] = __float_as_uint(a1);
        diff |= (t[e] ^ __float_as_uint(b0)) | (t[e + 1] ^ __float_as_uint(b1));
        xm = fmaxf(xm, fmaxf(fabsf(x[e]), fabsf(x[e + 1])));
    }
    if (diff != 0 || !(xm <= q.xlim)) {
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = (uint32_t)int8_code(__fdiv_rn(x[e], q.s));
    }
    return make_uint2(pack4(t[0], t[1], t[2], t[3]), pack4(t[4], t[5], t[6], t[7]));
}

// Four fp32 -> four E4M3 bytes (a in the lowest byte), RNE, satfinite.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d)
{
    uint32_t w;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(w)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return w;
}

// Eight E4M3 codes of x[e] / s[e] given the bracketing reciprocals of s[e]
// (e4m3_brackets), packed little-endian into two words.
__device__ __forceinline__ uint2 e4m3_codes8(const float (&x)[8], const float (&s)[8],
                                             const float (&rl)[8], const float (&rh)[8])
{
    uint32_t w[2], diff = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int o = 4 * e;
        float l[4], h[4];
#pragma unroll
        for (int k = 0; k < 4; k += 2) {
            const unsigned long long x2 = f2pack(x[o + k], x[o + k + 1]);
            f2unpack(f2mul(x2, f2pack(rl[o + k], rl[o + k + 1])), l[k], l[k + 1]);
            f2unpack(f2mul(x2, f2pack(rh[o + k], rh[o + k + 1])), h[k], h[k + 1]);
        }
        const uint32_t lo = e4m3x4(l[0], l[1], l[2], l[3]);
        const uint32_t hi = e4m3x4(h[0], h[1], h[2], h[3]);
        diff |= lo ^ hi;
        w[e] = lo;
    }
    if (diff != 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int o = 4 * e;
            w[e] = e4m3x4(__fdiv_rn(x[o], s[o]), __fdiv_rn(x[o + 1], s[o + 1]),
                          __fdiv_rn(x[o + 2], s[o + 2]), __fdiv_rn(x[o + 3], s[o + 3]));
        }
    }
    return make_uint2(w[0], w[1]);
}

// Bracketing reciprocals of a V scale for e4m3_codes8.
__device__ __forceinline__ void e4m3_brackets(float s, float &rl, float &rh)
{
    const float r = __frcp_rn(s);
    rl = __fmul_rn(r, kBracketLoV);
    rh = __fmul_rn(r, kBracketHiV);
}

// ------------------------------------------------- packed 16-bit min / max

// Per-lane running max and min of 16-bit floating-point pairs (exact).
template <int DT>
struct Pair16 {
    uint32_t mx, mn;
    __device__ __forceinline__ void init()
    {
        mx = DT == ULP_BF16 ? 0xFF80FF80u : 0xFC00FC00u;   // -inf, -inf
        mn = DT == ULP_BF16 ? 0x7F807F80u : 0x7C007C00u;   // +inf, +inf
    }
    __device__ __forceinline__ void add(uint32_t w)
    {
        if (DT == ULP_BF16) {
            const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&w);
            __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&mx), b = *reinterpret_cast<__nv_bfloat162 *>(&mn);
            a = __hmax2(a, v);
            b = __hmin2(b, v);
            mx = *reinterpret_cast<uint32_t *>(&a);
            mn = *reinterpret_cast<uint32_t *>(&b);
        } else {
            const __half2 v = *reinterpret_cast<const __half2 *>(&w);
            __half2 a = *reinterpret_cast<__half2 *>(&mx), b = *reinterpret_cast<__half2 *>(&mn);
            a = __hmax2(a, v);
            b = __hmin2(b, v);
            mx = *reinterpret_cast<uint32_t *>(&a);
            mn = *reinterpret_cast<uint32_t *>(&b);
        }
    }
};

// fp32 values of the two halves of a 16-bit pair word (low half first).
template <int DT>
__device__ __forceinline__ float2 pair_f32(uint32_t w)
{
    if (DT == ULP_BF16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}

}  // namespace ulp
