// Internal helpers of the ulp library: geometry, argument checks, device
// conversions and reductions.  Not part of the ABI.
#pragma once

#include <cuda.h>
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
constexpr int kGQ = 128;   // default Q group rows (q_group = 64 is the other width)
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

__host__ __device__ __forceinline__ ChunkLayout chunk_layout(int B, int L, int h, int D, int gq)
{
    ChunkLayout c;
    size_t n = (size_t)B * L * h * D;
    c.q = 0;
    c.k = align16(n);
    c.v = c.k + align16(n);
    c.qs = c.v + align16(n);
    c.ks = c.qs + align16(sizeof(float) * (size_t)B * h * slots(L, gq));
    c.bytes = c.ks + align16(sizeof(float) * (size_t)B * h * slots(L, kGK));
    return c;
}

// ------------------------------------------------------ device properties

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point
// (the library does not link libcuda); null when the driver lacks it.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled();

// ---------------------------------------------------------- argument checks

bool aligned16(const void *p);
int check_q_group(int q_group, const char *what);
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
// Exact quantisation of x / s without a divide per element.
//
// The codes are those of the IEEE quotient z = rn(x / s).  With r = rn(1/s)
// (__frcp_rn) and y = rn(x * r), Markstein's correction
//     e = fma(-y, s, x),   z = fma(e, r, y)
// gives z = rn(x / s).  Rounding to nearest commutes with scaling by powers
// of two, so the identity depends only on the significands of x and s; it
// was checked against __fdiv_rn for all 2^46 pairs of binary32 significands
// (x, s in [1, 2)) with zero mismatches.  It therefore holds whenever r, y and
// e stay normal.  e underflows only for |x| < 2^-102; then every int8 code is 0,
// and so is every E4M3 code when s >= 2^-92, whose sign is restored from y
// (the correction turns -0 into +0).  The only other failure is y overflowing
// to infinity (z becomes NaN): callers that can meet it test for it (int8
// saturating path, E4M3 path).
//
// int8 code = saturate(rne(z)): rne(z) is read off z + 1.5 * 2^23 (the sum's
// binade has unit spacing) and saturating first gives the same code.  Where
// the scale comes from the group's own amax, |x| <= amax bounds |z| by
// 127 (1 + 2^-23), so no saturation is needed (int8_codes8<false>).
constexpr float kRoundMagic = 12582912.0f;   // 1.5 * 2^23

struct Int8Scale {
    float s, r;   // scale and rn(1/scale)
};

__device__ __forceinline__ Int8Scale int8_scale(float s) { return Int8Scale{s, __frcp_rn(s)}; }

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
__device__ __forceinline__ unsigned long long f2add(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long f2sub(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// rn(x / s) for a pair sharing nothing: y = x * r, e = fma(-y, s, x), z = fma(e, r, y).
__device__ __forceinline__ unsigned long long f2quot(unsigned long long x2, unsigned long long r2,
                                                     unsigned long long ns2, unsigned long long &y2)
{
    y2 = f2mul(x2, r2);
    return f2fma(f2fma(y2, ns2, x2), r2, y2);
}

// Eight int8 codes of rn(x[e] / s), packed little-endian into two words.
// SAT = false: the caller guarantees |x| <= 127 s (1 + 2^-24), so no code
// saturates; SAT = true: any finite x.
template <bool SAT>
__device__ __forceinline__ uint2 int8_codes8(const float (&x)[8], const Int8Scale &q)
{
    const unsigned long long r2 = f2pack(q.r, q.r), ns2 = f2pack(-q.s, -q.s);
    const unsigned long long mg2 = f2pack(kRoundMagic, kRoundMagic);
    uint32_t t[8];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        unsigned long long y2;
        const unsigned long long z2 = f2quot(f2pack(x[e], x[e + 1]), r2, ns2, y2);
        float a0, a1;
        if (SAT) {
            float y0, y1;
            f2unpack(z2, a0, a1);
            f2unpack(y2, y0, y1);
            a0 = fabsf(y0) <= 3.4028235e38f ? a0 : y0;            // y overflowed: z is NaN
            a1 = fabsf(y1) <= 3.4028235e38f ? a1 : y1;
            a0 = __fadd_rn(fminf(fmaxf(a0, -128.0f), 127.0f), kRoundMagic);
            a1 = __fadd_rn(fminf(fmaxf(a1, -128.0f), 127.0f), kRoundMagic);
        } else {
            f2unpack(f2add(z2, mg2), a0, a1);
        }
        t[e] = __float_as_uint(a0);
        t[e + 1] = __float_as_uint(a1);
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

// fp32 values of the two halves of a 16-bit pair word (low half first).
template <int DT>
__device__ __forceinline__ float2 pair_f32(uint32_t w)
{
    if (DT == ULP_BF16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}

// Eight E4M3 codes of rn(x[e] / s[e]) given r[e] = rn(1/s[e]), x[e] element
// e of the 16-bit vector v (bf16 or fp16), packed little-endian into two
// words; rn, satfinite.  z = rn(x / s) by Markstein's correction, then:
//  - the sign: the correction turns the zero quotient of a negative x into +0
//    (the -0 + +0 of its last step) and never changes the sign of a nonzero
//    quotient, so OR-ing x's sign bits (bit 7 of each value's high byte,
//    gathered by one byte permute per four values) into the code bytes gives
//    the codes of z with x's sign restored;
//  - the overflow: the first product y overflows (possible only with extreme
//    caller scales) exactly when some z is NaN (z = fma(e, r, y) with
//    e = -inf), i.e. when some code byte reads 0x7F or 0xFF; such a group
//    goes to __fdiv_rn (as does x = NaN, which gives that code either way).
template <int DT>
__device__ __forceinline__ uint2 e4m3_codes8(const uint4 &v, const float (&s)[8], const float (&r)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[2];
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {
        float z[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int wi = 2 * hw + e;                  // elements 2 wi, 2 wi + 1
            const float2 x = pair_f32<DT>(w[wi]);
            unsigned long long y2;
            const unsigned long long z2 = f2quot(f2pack(x.x, x.y), f2pack(r[2 * wi], r[2 * wi + 1]),
                                                 f2pack(-s[2 * wi], -s[2 * wi + 1]), y2);
            f2unpack(z2, z[2 * e], z[2 * e + 1]);
        }
        const uint32_t sign = __byte_perm(w[2 * hw], w[2 * hw + 1], 0x7531) & 0x80808080u;
        c[hw] = e4m3x4(z[0], z[1], z[2], z[3]) | sign;
    }
    const uint32_t nan = (((c[0] & 0x7F7F7F7Fu) + 0x01010101u) | ((c[1] & 0x7F7F7F7Fu) + 0x01010101u)) & 0x80808080u;
    if (nan) {
        float f[8], z[8];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            const float2 x = pair_f32<DT>(w[wi]);
            f[2 * wi] = x.x;
            f[2 * wi + 1] = x.y;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) z[e] = __fdiv_rn(f[e], s[e]);
        c[0] = e4m3x4(z[0], z[1], z[2], z[3]);
        c[1] = e4m3x4(z[4], z[5], z[6], z[7]);
    }
    return make_uint2(c[0], c[1]);
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


}  // namespace ulp
