// Attention over the unpacked tensors (page "unpack_for_sage": INT8 Q/K
// [B, S, h, D] with FP32 per-group scales whose width the kernel derives from
// the rows it is given, FP8 E4M3 V [B, D, h, Spad], V scale from the caller):
//   O[b,t,j,:] = sum_u softmax_u(sm_scale * Q[t] . K[u]) V[u]   over t, u < n,
//   Q[t] = q8[t] * q_scale[t / G_Q], K[u] = k8[u] * k_scale[u / 64],
//   V[u, d] = e4m3(v8[d, u]) * v_scale[d].
//
// Tensor cores: tcgen05.mma kind::f16 (fp16 operands, fp32 accumulators in
// tensor memory).  INT8 codes widen to fp16 exactly, and since |q8 . k8| <=
// 128^3 = 2^21 the integer dot products accumulate exactly in fp32; E4M3 is a
// subset of fp16, so V widens exactly too.  The per-group scales multiply the
// integer logits in fp32.  P = exp2(x - m) is rounded to fp16 for the PV
// product, and the softmax denominator sums the rounded values, so the
// output is an exact weighted mean with weights perturbed by at most 2^-11
// relative.
//
// One CTA of 128 threads per (b, head, 128-query tile); thread i owns query
// row i (TMEM lane i).  Per 128-key tile:
//   1. K (int8 -> fp16) and V (E4M3 -> fp16) tiles go to shared memory in
//      the 128-byte swizzled K-major layout;
//   2. one thread issues S = Q K^T (D/16 MMAs, M = N = 128) into TMEM;
//   3. each thread reads its S row, applies the scales, updates its running
//      max m and sum l (online softmax), writes its P row (fp16) to shared
//      memory and rescales its O row in TMEM when m grew;
//   4. one thread issues O += P V (8 MMAs, M = 128, N = D).
// Every wait on an MMA completion is bounded; on timeout the kernel records
// a status, frees its tensor memory and returns.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "ulp_internal.cuh"
#include "ulp_tc.cuh"

namespace ulp {

namespace {

constexpr int kAttnThreads = 128;
constexpr int kTile = 128;                 // queries per CTA, keys per step
constexpr uint32_t kTmemCols = 256;        // S: 128 columns, O: D columns
constexpr uint64_t kWaitNs = 1000000000ull;

struct AttnArgs {
    const int8_t *q8, *k8;
    const uint8_t *v8;
    const float *qs, *ks, *vs;
    void *out;
    int *status;
    int out_dtype;
    int S, h, n, Spad, gq, wq, wk;
    float scale_log2;                      // sm_scale * log2(e)
};

template <int D>
struct AttnLayout {
    static constexpr uint32_t q = 0;
    static constexpr uint32_t k = q + kTile * D * 2;
    static constexpr uint32_t v = k + kTile * D * 2;
    static constexpr uint32_t p = v + D * kTile * 2;
    static constexpr uint32_t bars = p + kTile * kTile * 2;   // bar_s, bar_o, tmem address, abort
    static constexpr uint32_t bytes = bars + 64;
};

// 4 int8 -> 4 fp16, exact: byte u = x + 128 becomes fp16 1024 + u (bits
// 0x6400 | u), minus 1152.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = w ^ 0x80808080u;
    lo = __byte_perm(u, 0x64646464u, 0x5140);
    hi = __byte_perm(u, 0x64646464u, 0x7362);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    __half2 a = __hsub2(*reinterpret_cast<__half2 *>(&lo), bias);
    __half2 b = __hsub2(*reinterpret_cast<__half2 *>(&hi), bias);
    lo = *reinterpret_cast<uint32_t *>(&a);
    hi = *reinterpret_cast<uint32_t *>(&b);
}

// 2 E4M3 bytes (low 16 bits) -> fp16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16(uint32_t w)
{
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
    return (uint32_t)r.x | ((uint32_t)r.y << 16);
}

// 16 int8 codes -> two 16-byte fp16 chunks c0, c1 of row r in an R-row tile.
__device__ __forceinline__ void store_i8_row16(uint8_t *tile, int r, int c0, int R, uint4 w)
{
    uint4 a, b;
    i8x4_to_f16(w.x, a.x, a.y);
    i8x4_to_f16(w.y, a.z, a.w);
    i8x4_to_f16(w.z, b.x, b.y);
    i8x4_to_f16(w.w, b.z, b.w);
    *reinterpret_cast<uint4 *>(tile + tc::sw128_offset(r, c0, R)) = a;
    *reinterpret_cast<uint4 *>(tile + tc::sw128_offset(r, c0 + 1, R)) = b;
}

__device__ __forceinline__ void store_e4m3_row16(uint8_t *tile, int r, int c0, int R, uint4 w)
{
    uint4 a, b;
    a.x = e4m3x2_to_f16(w.x);
    a.y = e4m3x2_to_f16(w.x >> 16);
    a.z = e4m3x2_to_f16(w.y);
    a.w = e4m3x2_to_f16(w.y >> 16);
    b.x = e4m3x2_to_f16(w.z);
    b.y = e4m3x2_to_f16(w.z >> 16);
    b.z = e4m3x2_to_f16(w.w);
    b.w = e4m3x2_to_f16(w.w >> 16);
    *reinterpret_cast<uint4 *>(tile + tc::sw128_offset(r, c0, R)) = a;
    *reinterpret_cast<uint4 *>(tile + tc::sw128_offset(r, c0 + 1, R)) = b;
}

// Rows [row0, row0 + 128) of an int8 [.., S, h, D] tensor (head j of batch
// b) -> fp16 tile; rows >= n are zero.
template <int D>
__device__ __forceinline__ void load_i8_tile(uint8_t *tile, const int8_t *src, int row0, int n, int hD)
{
    constexpr int NV = D / 16;                 // 16-byte vectors per row
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int idx = i * kAttnThreads + threadIdx.x;
        const int r = idx / NV, cv = idx % NV;
        uint4 w = make_uint4(0, 0, 0, 0);
        if (row0 + r < n) w = *reinterpret_cast<const uint4 *>(src + (size_t)(row0 + r) * hD + cv * 16);
        store_i8_row16(tile, r, 2 * cv, kTile, w);
    }
}

// Keys [u0, u0 + 128) of every channel of V (E4M3 rows of Spad bytes, one per
// channel d at src + d * ch_stride) -> fp16 tile of D rows; keys >= n are zero.
template <int D>
__device__ __forceinline__ void load_v_tile(uint8_t *tile, const uint8_t *src, size_t ch_stride, int u0, int n)
{
    constexpr int NV = kTile / 16;             // 16-byte vectors per channel row
#pragma unroll
    for (int i = 0; i < D * NV / kAttnThreads; ++i) {
        const int idx = i * kAttnThreads + threadIdx.x;
        const int d = idx / NV, cv = idx % NV;
        const int key = u0 + cv * 16;
        uint4 w = make_uint4(0, 0, 0, 0);
        if (key < n) {
            w = *reinterpret_cast<const uint4 *>(src + (size_t)d * ch_stride + key);
            const int valid = n - key;         // bytes past it are zeroed
            if (valid < 16) {
                uint32_t *ww = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int keep = min(max(valid - 4 * x, 0), 4);
                    ww[x] = keep == 4 ? ww[x] : (keep == 0 ? 0u : (ww[x] & ((1u << (8 * keep)) - 1u)));
                }
            }
        }
        store_e4m3_row16(tile, d, 2 * cv, D, w);
    }
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) sage_attention_kernel(AttnArgs a)
{
    using Lay = AttnLayout<D>;
    extern __shared__ uint8_t dyn_smem[];
    // 1024-byte aligned base in the shared window (the swizzle is a function
    // of the address)
    const uint32_t raw = tc::smem_u32(dyn_smem);
    uint8_t *sm = dyn_smem + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sq = sm + Lay::q, *sk = sm + Lay::k, *sv = sm + Lay::v, *sp = sm + Lay::p;
    uint64_t *bar_s = reinterpret_cast<uint64_t *>(sm + Lay::bars);
    uint64_t *bar_o = bar_s + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_s + 2);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int t0 = blockIdx.x * kTile, j = blockIdx.y, b = blockIdx.z;
    const int hD = a.h * D;
    const int n = a.n;

    if (warp == 0) tc::tmem_alloc(tmem_slot, kTmemCols);
    if (tid == 0) {
        tc::mbar_init(bar_s, 1);
        tc::mbar_init(bar_o, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // Q tile and this thread's Q scale
    const int8_t *qsrc = a.q8 + (size_t)b * a.S * hD + (size_t)j * D;
    const int8_t *ksrc = a.k8 + (size_t)b * a.S * hD + (size_t)j * D;
    const uint8_t *vsrc = a.v8 + ((size_t)b * D * a.h + j) * a.Spad;
    load_i8_tile<D>(sq, qsrc, t0, n, hD);
    const int t = t0 + tid;
    const float qa = t < n ? a.qs[((size_t)b * a.h + j) * a.wq + t / a.gq] * a.scale_log2 : 0.0f;
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tO = tmem + kTile;
    const uint32_t lane_S = tc::tmem_addr(tS, warp * 32, 0), lane_O = tc::tmem_addr(tO, warp * 32, 0);
    constexpr uint32_t idS = tc::idesc_f16_f32(kTile, kTile), idO = tc::idesc_f16_f32(kTile, D);
    const uint32_t aq = tc::smem_u32(sq), ak = tc::smem_u32(sk), av = tc::smem_u32(sv), ap = tc::smem_u32(sp);

    float m_run = -INFINITY, l_run = 0.0f;
    const int ntk = (n + kTile - 1) / kTile;
    int fail_at = 0;                           // 1: S product, 2: PV product, 3: last PV product
    uint64_t *fail_bar = bar_o;
    uint32_t fail_par = 0;
    for (int kt = 0; kt < ntk; ++kt) {
        const int u0 = kt * kTile;
        if (kt > 0) {                          // the previous PV product read V and P
            const bool ok = tc::mbar_wait(bar_o, (kt - 1) & 1, kWaitNs);
            if (__syncthreads_or(!ok)) { fail_at = 2; fail_bar = bar_o; fail_par = (kt - 1) & 1; break; }
            tc::fence_after_sync();
        }
        load_i8_tile<D>(sk, ksrc, u0, n, hD);
        load_v_tile<D>(sv, vsrc, (size_t)a.h * a.Spad, u0, n);
        tc::fence_smem_to_async();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int s = 0; s < D / 16; ++s)
                tc::mma_f16(tS, tc::sw128_desc_k(aq, s, kTile), tc::sw128_desc_k(ak, s, kTile), idS, s > 0);
            tc::mma_commit(bar_s);
        }
        // scales of the tile's two 64-key groups
        const size_t krow = ((size_t)b * a.h + j) * a.wk;
        const int g0 = u0 / 64;
        const float c0 = qa * a.ks[krow + g0];
        const float c1 = (g0 + 1 < a.wk) ? qa * a.ks[krow + g0 + 1] : 0.0f;
        const int nvalid = min(kTile, n - u0);
        {
            const bool ok = tc::mbar_wait(bar_s, kt & 1, kWaitNs);
            if (__syncthreads_or(!ok)) { fail_at = 1; fail_bar = bar_s; fail_par = kt & 1; break; }
        }
        tc::fence_after_sync();
        float x[kTile];
#pragma unroll
        for (int cc = 0; cc < kTile / 32; ++cc) {
            float v[32];
            tc::tmem_ld32(lane_S + cc * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) x[cc * 32 + i] = v[i];
        }
        float mt = -INFINITY;
#pragma unroll
        for (int i = 0; i < kTile; ++i) {
            const float y = i < nvalid ? x[i] * (i < 64 ? c0 : c1) : -INFINITY;
            x[i] = y;
            mt = fmaxf(mt, y);
        }
        const float m_new = fmaxf(m_run, mt);
        const float alpha = exp2f(m_run - m_new);   // 0 on the first tile
        float lsum = 0.0f;
#pragma unroll
        for (int c = 0; c < kTile / 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int x2 = 0; x2 < 4; ++x2) {
                const __half2 hp = __floats2half2_rn(exp2f(x[8 * c + 2 * x2] - m_new),
                                                     exp2f(x[8 * c + 2 * x2 + 1] - m_new));
                const float2 f = __half22float2(hp);
                lsum += f.x + f.y;
                w[x2] = *reinterpret_cast<const uint32_t *>(&hp);
            }
            *reinterpret_cast<uint4 *>(sp + tc::sw128_offset(tid, c, kTile)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        l_run = l_run * alpha + lsum;
        m_run = m_new;
        // O *= alpha for rows whose max grew (a warp-wide TMEM access)
        if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                float v[32];
                tc::tmem_ld32(lane_O + cc * 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= alpha;
                tc::tmem_st32(lane_O + cc * 32, v);
            }
            tc::tmem_st_wait();
        }
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int s = 0; s < kTile / 16; ++s)
                tc::mma_f16(tO, tc::sw128_desc_k(ap, s, kTile), tc::sw128_desc_k(av, s, D), idO,
                            (kt > 0 || s > 0) ? 1u : 0u);
            tc::mma_commit(bar_o);
        }
    }

    if (fail_at == 0) {
        const bool ok = tc::mbar_wait(bar_o, (ntk - 1) & 1, kWaitNs);
        if (__syncthreads_or(!ok)) { fail_at = 3; fail_par = (ntk - 1) & 1; }
    }
    if (fail_at == 0) {
        tc::fence_after_sync();
        const float inv_l = 1.0f / l_run;
        const float *vsc = a.vs + ((size_t)b * a.h + j) * D;
        const size_t orow = (((size_t)b * n + t) * a.h + j) * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
            float v[32];
            tc::tmem_ld32(lane_O + cc * 32, v);
            if (t < n) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = v[i] * inv_l * vsc[cc * 32 + i];
                if (a.out_dtype == ULP_F32) {
                    float4 *o = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.out) + orow + cc * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                } else {
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        if (a.out_dtype == ULP_BF16) {
                            const __nv_bfloat162 hv = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                            w[i] = *reinterpret_cast<const uint32_t *>(&hv);
                        } else {
                            const __half2 hv = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
                            w[i] = *reinterpret_cast<const uint32_t *>(&hv);
                        }
                    }
                    uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(a.out) + orow + cc * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                }
            }
        }
    } else {
        // an MMA did not complete in time: report, give it a second bounded
        // wait, then release the tensor memory
        if (tid == 0 && a.status) atomicExch(a.status, fail_at);
        tc::mbar_wait(fail_bar, fail_par, kWaitNs);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

}  // namespace ulp

using namespace ulp;

extern "C" int ulp_sage_attention(const int8_t *q8, const int8_t *k8, const uint8_t *v8, const float *q_scale,
                                  const float *k_scale, const float *v_scale, int B, int S, int h, int D,
                                  int n, int q_group, float sm_scale, void *out, int out_dtype, int *status,
                                  ulp_stream_t stream)
{
    if (B < 1 || S < 1 || h < 1) return fail(ULP_EINVAL, "sage_attention: B, S, h must be positive");
    if (D != 64 && D != 128) return fail(ULP_EINVAL, "sage_attention: head_dim must be 64 or 128 (got %d)", D);
    if (n < 1 || n > S) return fail(ULP_EINVAL, "sage_attention: n = %d outside [1, %d]", n, S);
    if (int s = check_q_group(q_group, "sage_attention")) return s;
    if (out_dtype != ULP_F32 && out_dtype != ULP_BF16 && out_dtype != ULP_FP16)
        return fail(ULP_EDTYPE, "sage_attention: out_dtype must be ULP_F32, ULP_BF16 or ULP_FP16 (got %d)", out_dtype);
    if (!(sm_scale > 0.0f) || !(sm_scale < INFINITY))
        return fail(ULP_EINVAL, "sage_attention: sm_scale must be positive and finite");
    if ((long long)B * S * h * D > (1ll << 40)) return fail(ULP_EINVAL, "sage_attention: tensors too large");
    if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(out) || !aligned4(q_scale) ||
        !aligned4(k_scale) || !aligned4(v_scale))
        return fail(ULP_EALIGN, "sage_attention: q8, k8, v8, out must be 16-byte aligned, scales 4-byte aligned");
    AttnArgs a{};
    a.q8 = q8; a.k8 = k8; a.v8 = v8;
    a.qs = q_scale; a.ks = k_scale; a.vs = v_scale;
    a.out = out; a.status = status; a.out_dtype = out_dtype;
    a.S = S; a.h = h; a.n = n; a.Spad = (S + 63) / 64 * 64; a.gq = q_group;
    a.wq = (n + q_group - 1) / q_group;
    a.wk = (n + kGK - 1) / kGK;
    a.scale_log2 = sm_scale * 1.4426950408889634f;
    const int ntq = (n + kTile - 1) / kTile;
    if (ntq > INT_MAX || h > 65535 || B > 65535) return fail(ULP_EINVAL, "sage_attention: grid too large");
    const dim3 grid((unsigned)ntq, (unsigned)h, (unsigned)B);
    const cudaStream_t st = (cudaStream_t)stream;
    if (D == 128) {
        const size_t bytes = AttnLayout<128>::bytes + 1024;
        cudaFuncSetAttribute(sage_attention_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        sage_attention_kernel<128><<<grid, kAttnThreads, bytes, st>>>(a);
    } else {
        const size_t bytes = AttnLayout<64>::bytes + 1024;
        cudaFuncSetAttribute(sage_attention_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        sage_attention_kernel<64><<<grid, kAttnThreads, bytes, st>>>(a);
    }
    return check_launch("sage_attention");
}
