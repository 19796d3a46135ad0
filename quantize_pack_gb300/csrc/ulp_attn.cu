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
// product while the softmax denominator sums the fp32 weights, so rounding P
// moves the output by at most 2^-11 of max |V|.  Scales must be positive
// (they are amax / 127).
//
// Two kernels.  The widen pass writes Q and K as fp16 [B*h, T, D] and V as
// fp16 [B*h, D, T] (T = the live prefix rounded up to 128 rows, zero past
// it) into a workspace, once per call, so the attention kernel moves every
// tile with TMA straight into the tensor core's 128-byte swizzled operand
// layout.  The attention kernel runs one CTA of eleven warps per (b, head,
// pair of 128-query tiles A and B):
//   warp 8 (TMA): the two Q tiles once, then K tiles of 128 keys into three
//     stages (a stage frees when both S products that read it complete);
//   warp 10 (TMA): V tiles into two stages (freed when both PV products
//     that read them complete);
//   warp 9 (MMA, one thread): per K tile i, O_A += P_A(i-1) V(i-1), then
//     S_A(i) = Q_A K_i^T, then the same for B; P is the A operand in tensor
//     memory, Q, K and V come from shared memory;
//   warps 0-3 (softmax of tile A) and 4-7 (tile B): one query row per
//     thread (TMEM lane = row), all 128 keys of each K tile.  A thread keeps
//     its row's running max m of the scaled logits and the running sum l of
//     the weights, and writes P = 2^(S c - m) (fp16) into tensor memory over
//     the S tile it came from.  The tensor pipe runs in order, so S(i+1)
//     overwrites that buffer only after PV(i) has read it, and the commit
//     that completes S(i+1) also covers PV(i): when a warpgroup sees S(i+1)
//     its O is settled and may be rescaled.  m moves only when the tile's
//     max exceeds it by more than 8 (log2 units), so O is rescaled rarely;
//     weights stay <= 2^8, and numerator and denominator share the same m.
// Each K and V tile is read once for 256 queries.  Every mbarrier wait is
// bounded: on a timeout the CTA records a status, every role stops, the
// tensor memory is freed and nothing is written.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <mutex>

#include "ulp_internal.cuh"
#include "ulp_tc.cuh"

namespace ulp {

namespace {

constexpr int kTile = 128;                 // queries per tile, keys per step
constexpr int kQTiles = 2;                 // query tiles per CTA, one per softmax warpgroup
constexpr int kSoftmaxThreads = 256;       // warps 0-7
constexpr int kAttnThreads = 352;          // + Q/K TMA warp 8, MMA warp 9, V TMA warp 10
constexpr int kKTmaWarp = 8, kMmaWarp = 9, kVTmaWarp = 10;
constexpr int kKStages = 3, kVStages = 2;  // shared-memory stages
constexpr uint32_t kTmemCols = 512;        // S_A, S_B: 128 columns each; O_A, O_B: D each
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr float kRescaleLog2 = 8.0f;       // max growth (log2) absorbed without rescaling O

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------ widen pass

// 4 int8 -> 4 fp16, exact: byte u = x + 128 becomes fp16 1024 + u (bits
// 0x6400 | u), minus 1152.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140), b = __byte_perm(u, 0x64646464u, 0x7362);
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    lo = *reinterpret_cast<const uint32_t *>(&ha);
    hi = *reinterpret_cast<const uint32_t *>(&hb);
}

// 2 E4M3 bytes (low 16 bits) -> fp16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16(uint32_t w)
{
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
    return (uint32_t)r.x | ((uint32_t)r.y << 16);
}

struct WidenArgs {
    const int8_t *q8, *k8;
    const uint8_t *v8;
    uint16_t *q16, *k16, *v16;             // [B*h, T, D], [B*h, T, D], [B*h, D, T]
    int S, h, D, n, T, Spad;
};

// blockIdx.z: 0 = Q, 1 = K, 2 = V; blockIdx.y = b * h + j; one thread per 16
// input bytes (T * D / 16 chunks per head for each tensor).
__global__ void __launch_bounds__(256) attn_widen_kernel(WidenArgs a)
{
    const int which = blockIdx.z, bh = blockIdx.y;
    const int b = bh / a.h, j = bh - b * a.h;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long per = (long long)a.T * a.D / 16;
    if (idx >= per) return;
    uint4 w = make_uint4(0, 0, 0, 0);
    uint4 lo, hi;
    if (which < 2) {
        const int nv = a.D / 16;
        const int t = (int)(idx / nv), cv = (int)(idx % nv);
        const int8_t *src = which == 0 ? a.q8 : a.k8;
        if (t < a.n) w = *reinterpret_cast<const uint4 *>(src + (((size_t)b * a.S + t) * a.h + j) * a.D + cv * 16);
        i8x4_to_f16(w.x, lo.x, lo.y);
        i8x4_to_f16(w.y, lo.z, lo.w);
        i8x4_to_f16(w.z, hi.x, hi.y);
        i8x4_to_f16(w.w, hi.z, hi.w);
        uint16_t *dst = (which == 0 ? a.q16 : a.k16) + ((size_t)bh * a.T + t) * a.D + cv * 16;
        reinterpret_cast<uint4 *>(dst)[0] = lo;
        reinterpret_cast<uint4 *>(dst)[1] = hi;
    } else {
        const int nv = a.T / 16;
        const int d = (int)(idx / nv), cv = (int)(idx % nv);
        const int key = cv * 16;
        if (key < a.n) {
            w = *reinterpret_cast<const uint4 *>(a.v8 + (((size_t)b * a.D + d) * a.h + j) * a.Spad + key);
            const int valid = a.n - key;   // keys past the prefix become zero
            if (valid < 16) {
                uint32_t *ww = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int keep = min(max(valid - 4 * x, 0), 4);
                    ww[x] = keep == 4 ? ww[x] : (keep == 0 ? 0u : (ww[x] & ((1u << (8 * keep)) - 1u)));
                }
            }
        }
        lo = make_uint4(e4m3x2_to_f16(w.x), e4m3x2_to_f16(w.x >> 16), e4m3x2_to_f16(w.y), e4m3x2_to_f16(w.y >> 16));
        hi = make_uint4(e4m3x2_to_f16(w.z), e4m3x2_to_f16(w.z >> 16), e4m3x2_to_f16(w.w), e4m3x2_to_f16(w.w >> 16));
        uint16_t *dst = a.v16 + ((size_t)bh * a.D + d) * a.T + key;
        reinterpret_cast<uint4 *>(dst)[0] = lo;
        reinterpret_cast<uint4 *>(dst)[1] = hi;
    }
}

// ------------------------------------------------------- attention kernel

struct AttnArgs {
    const float *qs, *ks, *vs;
    void *out;
    int *status;
    int out_dtype;
    int h, n, gq, wq, wk, ntk;
    float scale_log2;                      // sm_scale * log2(e)
};

template <int D, bool PV8>
struct AttnLayout {
    static constexpr uint32_t tBytes = kTile * D * 2;         // a Q or K tile: 128 rows x D
    static constexpr uint32_t vBytes = D * kTile * (PV8 ? 1 : 2);   // a V tile: D rows x 128 keys
    static constexpr uint32_t q0 = 0;                         // kQTiles Q tiles
    static constexpr uint32_t k0 = q0 + kQTiles * tBytes;     // kKStages K tiles
    static constexpr uint32_t v0 = k0 + kKStages * tBytes;    // kVStages V tiles
    static constexpr uint32_t bars = v0 + kVStages * vBytes;
    static constexpr uint32_t bytes = bars + 32 * 8;
};

// Barrier slots (uint64 each) after Lay::bars.
enum : int {
    kQFull = 0,
    kKFull = 1,                                        // [kKStages]
    kKEmpty = kKFull + kKStages,                       // [kKStages]
    kVFull = kKEmpty + kKStages,                       // [kVStages]
    kVEmpty = kVFull + kVStages,                       // [kVStages]
    kSFull = kVEmpty + kVStages,                       // [kQTiles]
    kPReady = kSFull + kQTiles,                        // [kQTiles]
    kOLast = kPReady + kQTiles,
    kTmemSlot = kOLast + 1,
    kAbortSlot = kTmemSlot + 1,
    kNumSlots = kAbortSlot + 1
};
static_assert(kNumSlots <= 32, "barrier area");

template <int D, bool PV8>
__global__ void __launch_bounds__(kAttnThreads, 1)
    sage_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, AttnArgs a)
{
    using Lay = AttnLayout<D, PV8>;
    extern __shared__ uint8_t dyn_smem[];
    // 1024-byte aligned base in the shared window (the swizzle is a function
    // of the address)
    const uint32_t raw = tc::smem_u32(dyn_smem);
    uint8_t *sm = dyn_smem + ((1024u - (raw & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Lay::bars);
    uint64_t *q_full = bars + kQFull, *k_full = bars + kKFull, *k_empty = bars + kKEmpty;
    uint64_t *v_full = bars + kVFull, *v_empty = bars + kVEmpty, *s_full = bars + kSFull;
    uint64_t *p_ready = bars + kPReady, *o_last = bars + kOLast;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kTmemSlot);
    volatile int *abort = reinterpret_cast<volatile int *>(bars + kAbortSlot);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * (kQTiles * kTile), j = blockIdx.y, b = blockIdx.z;
    const int bh = b * a.h + j;
    const int n = a.n, ntk = a.ntk;

    if (warp == kMmaWarp) tc::tmem_alloc(tmem_slot, kTmemCols);
    if (tid == 0) {
        tc::mbar_init(q_full, 1);
        for (int s = 0; s < kKStages; ++s) {
            tc::mbar_init(k_full + s, 1);
            tc::mbar_init(k_empty + s, 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            tc::mbar_init(v_full + s, 1);
            tc::mbar_init(v_empty + s, 1);
        }
        for (int w = 0; w < kQTiles; ++w) {
            tc::mbar_init(s_full + w, 1);
            tc::mbar_init(p_ready + w, kSoftmaxThreads / kQTiles);
        }
        tc::mbar_init(o_last, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // S_w at column 128 w, O_w at 256 + D w
    const uint32_t tS0 = tmem, tO0 = tmem + kQTiles * kTile;

    if (warp == kKTmaWarp) {
        // ------------------------------------------------------ TMA: Q, K
        if (lane == 0) {
            // the two query tiles (rows past T read as zeros)
            tc::mbar_expect_tx(q_full, kQTiles * Lay::tBytes);
            for (int w = 0; w < kQTiles; ++w)
                for (int kb = 0; kb < D / 64; ++kb)
                    tc::tma_load_3d(sm + Lay::q0 + w * Lay::tBytes + kb * (kTile * 128), &tm_q, kb * 64,
                                    t0 + w * kTile, bh, q_full);
            int last[kKStages];
            for (int s = 0; s < kKStages; ++s) last[s] = -1;
            for (int i = 0; i < ntk; ++i) {
                const int s = i % kKStages;
                // a K stage frees when both S products that read it complete
                if (i >= kKStages &&
                    !tc::mbar_wait_abortable(k_empty + s, ((i / kKStages) - 1) & 1, kWaitNs, abort))
                    break;
                tc::mbar_expect_tx(k_full + s, Lay::tBytes);
                uint8_t *kd = sm + Lay::k0 + s * Lay::tBytes;
                for (int kb = 0; kb < D / 64; ++kb)
                    tc::tma_load_3d(kd + kb * (kTile * 128), &tm_k, kb * 64, i * kTile, bh, k_full + s);
                last[s] = i;
            }
            if (*abort) {                      // let the copies in flight land
                tc::mbar_wait(q_full, 0, kWaitNs);
                for (int s = 0; s < kKStages; ++s)
                    if (last[s] >= 0) tc::mbar_wait(k_full + s, (last[s] / kKStages) & 1, kWaitNs);
            }
        }
    } else if (warp == kVTmaWarp) {
        // --------------------------------------------------------- TMA: V
        if (lane == 0) {
            int last[kVStages];
            for (int s = 0; s < kVStages; ++s) last[s] = -1;
            for (int i = 0; i < ntk; ++i) {
                const int s = i % kVStages;
                // a V stage frees when both PV products that read it complete
                if (i >= kVStages &&
                    !tc::mbar_wait_abortable(v_empty + s, ((i / kVStages) - 1) & 1, kWaitNs, abort))
                    break;
                tc::mbar_expect_tx(v_full + s, Lay::vBytes);
                uint8_t *vd = sm + Lay::v0 + s * Lay::vBytes;
                if (PV8) {
                    // the E4M3 bytes of v8 itself: D rows of 128 keys (128 B,
                    // one swizzle row); keys >= n lie outside the map: zeros
                    tc::tma_load_3d(vd, &tm_v, i * kTile, j, b * D, v_full + s);
                } else {
                    for (int c = 0; c < 2; ++c)
                        tc::tma_load_3d(vd + c * (D * 128), &tm_v, i * kTile + c * 64, 0, bh, v_full + s);
                }
                last[s] = i;
            }
            if (*abort) {
                for (int s = 0; s < kVStages; ++s)
                    if (last[s] >= 0) tc::mbar_wait(v_full + s, (last[s] / kVStages) & 1, kWaitNs);
            }
        }
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------------- MMA issuer
        // Step i (0 <= i <= ntk): for w = A, B: O_w += P_w(i-1) V(i-1) once
        // the warpgroup has written P_w(i-1), then S_w(i) = Q_w K_i^T.
        if (lane == 0) {
            // (E4M3 A and B are type 0 of kind::f8f6f4, fp16 type 0 of kind::f16:
            // the PV descriptor's bits are the same for both)
            constexpr uint32_t idS = tc::idesc_f16_f32(kTile, kTile), idO = tc::idesc_f16_f32(kTile, D);
            bool ok = tc::mbar_wait_abortable(q_full, 0, kWaitNs, abort);
            const uint32_t aq = tc::smem_u32(sm + Lay::q0);
            for (int i = 0; ok && i <= ntk; ++i) {
                const int ks = i % kKStages, vs = (i + kVStages - 1) % kVStages;
                uint32_t ak = 0, av = 0;
                if (i < ntk) {
                    if (!(ok = tc::mbar_wait_abortable(k_full + ks, (i / kKStages) & 1, kWaitNs, abort))) break;
                    ak = tc::smem_u32(sm + Lay::k0 + ks * Lay::tBytes);
                }
                if (i >= 1) {
                    if (!(ok = tc::mbar_wait_abortable(v_full + vs, ((i - 1) / kVStages) & 1, kWaitNs, abort)))
                        break;
                    av = tc::smem_u32(sm + Lay::v0 + vs * Lay::vBytes);
                }
                tc::fence_after_sync();
                for (int w = 0; w < kQTiles; ++w) {
                    const uint32_t tS = tS0 + w * kTile;
                    if (i >= 1) {
                        // A = P_w(i-1): fp16 pairs in the first 64 columns of S_w, or
                        // E4M3 quadruples in the first 32 (K = 16 or 32 keys a product)
                        if (!(ok = tc::mbar_wait_abortable(p_ready + w, (i - 1) & 1, kWaitNs, abort))) break;
                        tc::fence_after_sync();
                        if (PV8) {
#pragma unroll
                            for (int k = 0; k < kTile / 32; ++k)
                                tc::mma_f8_ts(tO0 + w * D, tS + k * 8, tc::sw128_desc_k(av, k, D), idO,
                                              (i > 1 || k > 0) ? 1u : 0u);
                        } else {
#pragma unroll
                            for (int k = 0; k < kTile / 16; ++k)
                                tc::mma_f16_ts(tO0 + w * D, tS + k * 8, tc::sw128_desc_k(av, k, D), idO,
                                               (i > 1 || k > 0) ? 1u : 0u);
                        }
                    }
                    if (i < ntk) {
                        const uint32_t aqw = aq + w * Lay::tBytes;
#pragma unroll
                        for (int k = 0; k < D / 16; ++k)
                            tc::mma_f16(tS, tc::sw128_desc_k(aqw, k, kTile), tc::sw128_desc_k(ak, k, kTile), idS,
                                        k > 0);
                        tc::mma_commit(s_full + w);
                    }
                }
                if (!ok) break;
                if (i >= 1) tc::mma_commit(v_empty + vs);
                if (i < ntk) tc::mma_commit(k_empty + ks);
            }
            // completes when every product issued above has (also after an abort)
            tc::mma_commit(o_last);
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------- softmax
        // warpgroup w = warp / 4 owns query tile w; warp % 4 picks the TMEM
        // lane quarter, so the thread's row is its lane in S_w and O_w
        const int w = warp >> 2, row = (warp & 3) * 32 + lane;
        const int t = t0 + w * kTile + row;
        const float qa = t < n ? a.qs[(size_t)bh * a.wq + t / a.gq] * a.scale_log2 : 0.0f;
        const float *ksr = a.ks + (size_t)bh * a.wk;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tS0 + w * kTile + lane_base, tO = tO0 + w * D + lane_base;
        float m_use = -INFINITY, l = 0.0f;
        bool bad = false;
        // a warp-uniform outcome, so the warp-wide TMEM accesses stay converged
        auto wait_warp = [&](uint64_t *bar, uint32_t parity) {
            return __all_sync(0xffffffffu, tc::mbar_wait_abortable(bar, parity, kWaitNs, abort)) != 0;
        };
        for (int i = 0; i < ntk; ++i) {
            const int u0 = i * kTile;
            const int gk = u0 / 64;            // the tile's two K groups (their loads
                                               // overlap the wait for S)
            const float c0 = gk < a.wk ? qa * ksr[gk] : 0.0f;
            const float c1 = gk + 1 < a.wk ? qa * ksr[gk + 1] : 0.0f;
            const int nvalid = min(n - u0, kTile);
            if (!wait_warp(s_full + w, i & 1)) {
                bad = true;
                break;
            }
            tc::fence_after_sync();
            // the row's 128 integer logits; c >= 0, so a half's max scaled
            // logit is c times its max raw logit, and each weight is
            // 2^fma(S, c, -m).  Eight independent running maxima per half keep
            // the chains short.
            float x[kTile];
            {
                uint32_t r0[32], r1[32], r2[32], r3[32];
                tc::tmem_ld32_issue(tS, r0);
                tc::tmem_ld32_issue(tS + 32, r1);
                tc::tmem_ld32_issue(tS + 64, r2);
                tc::tmem_ld32_issue(tS + 96, r3);
                tc::tmem_ld_wait(r0);
                tc::tmem_pin(r1);
                tc::tmem_pin(r2);
                tc::tmem_pin(r3);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    x[e] = __uint_as_float(r0[e]);
                    x[32 + e] = __uint_as_float(r1[e]);
                    x[64 + e] = __uint_as_float(r2[e]);
                    x[96 + e] = __uint_as_float(r3[e]);
                }
            }
            float mh[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float m8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
                if (nvalid == kTile) {
#pragma unroll
                    for (int e = 0; e < 64; ++e) m8[e & 7] = fmaxf(m8[e & 7], x[hf * 64 + e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        m8[e & 7] = hf * 64 + e < nvalid ? fmaxf(m8[e & 7], x[hf * 64 + e]) : m8[e & 7];
                }
                const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                mh[hf] = hf * 64 < nvalid ? (hf == 0 ? c0 : c1) * mx : -INFINITY;
            }
            const float mt = fmaxf(mh[0], mh[1]);
            const bool grow = mt > m_use + kRescaleLog2;   // always on the first tile
            float alpha = 1.0f;
            if (grow) {
                alpha = ex2(m_use - mt);                   // 0 on the first tile
                m_use = mt;
            }
            const float nm = -m_use;
            float ls;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const float c = hf == 0 ? c0 : c1;
                float *xh = x + hf * 64;
                uint32_t pk[32];
                if (nvalid == kTile) {
                    // exponents two at a time (packed fma.rn.f32x2: the same
                    // rounding as two fmaf), then exp2
                    const uint64_t c2 = f2pack(c, c), nm2 = f2pack(nm, nm);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        f2unpack(f2fma(f2pack(xh[2 * e], xh[2 * e + 1]), c2, nm2), xh[2 * e], xh[2 * e + 1]);
#pragma unroll
                    for (int e = 0; e < 64; ++e) xh[e] = ex2(xh[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 64; ++e) xh[e] = hf * 64 + e < nvalid ? ex2(fmaf(xh[e], c, nm)) : 0.0f;
                }
                if (PV8) {
                    // E4M3 weights (rn, satfinite; they are <= 2^8 < 448), four
                    // keys a column: S_w columns 16 hf .. 16 hf + 15
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = e4m3x4(xh[4 * e], xh[4 * e + 1], xh[4 * e + 2], xh[4 * e + 3]);
                    tc::tmem_st16u(tS + hf * 16, *reinterpret_cast<const uint32_t(*)[16]>(pk));
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const __half2 hp = __floats2half2_rn(xh[2 * e], xh[2 * e + 1]);
                        pk[e] = *reinterpret_cast<const uint32_t *>(&hp);
                    }
                    // P of this half's 64 keys over S_w columns 32 hf .. 32 hf + 31;
                    // the half's weight sum (four packed partial sums) overlaps the store
                    tc::tmem_st32u(tS + hf * 32, pk);
                }
                uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
                for (int e = 0; e < 32; ++e) acc[e & 3] = f2add(acc[e & 3], f2pack(xh[2 * e], xh[2 * e + 1]));
                float s0, s1, s2, s3, s4, s5, s6, s7;
                f2unpack(acc[0], s0, s1);
                f2unpack(acc[1], s2, s3);
                f2unpack(acc[2], s4, s5);
                f2unpack(acc[3], s6, s7);
                const float hs = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
                ls = hf == 0 ? hs : ls + hs;
            }
            l = l * alpha + ls;
            // O_w *= alpha where the max grew: S_w(i) completing means PV_w(i-1),
            // issued before it, has completed too
            if (i >= 1 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    float v[32];
                    tc::tmem_ld32(tO + cc * 32, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] *= alpha;
                    tc::tmem_st32(tO + cc * 32, v);
                }
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
            tc::mbar_arrive(p_ready + w);
        }
        if (!bad && wait_warp(o_last, 0)) {
            tc::fence_after_sync();
            const float inv_l = 1.0f / l;
            const float *vsc = a.vs + (size_t)bh * D;
            const size_t orow = (((size_t)b * n + t) * a.h + j) * D;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                float v[32];
                tc::tmem_ld32(tO + cc * 32, v);
                if (t < n) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = v[e] * inv_l * vsc[cc * 32 + e];
                    if (a.out_dtype == ULP_F32) {
                        float4 *o = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.out) + orow + cc * 32);
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                    } else {
                        uint32_t ww[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            if (a.out_dtype == ULP_BF16) {
                                const __nv_bfloat162 hv = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                                ww[e] = *reinterpret_cast<const uint32_t *>(&hv);
                            } else {
                                const __half2 hv = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
                                ww[e] = *reinterpret_cast<const uint32_t *>(&hv);
                            }
                        }
                        uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(a.out) + orow + cc * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[e] = make_uint4(ww[4 * e], ww[4 * e + 1], ww[4 * e + 2], ww[4 * e + 3]);
                    }
                }
            }
        }
    }

    // every role is done (or gave up); the MMA thread's last commit covers
    // every product it issued, so after an abort one more bounded wait on it
    // comes before the tensor memory is released
    tc::fence_before_sync();
    __syncthreads();
    if (*abort) {
        if (tid == 0 && a.status) atomicExch(a.status, 1);
        if (tid == 0) tc::mbar_wait(o_last, 0, kWaitNs);
        __syncthreads();
    }
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------ host side

// fp16 tensor [planes, rows, cols] (cols contiguous) as a 3-D map with
// boxes of 64 columns x box_rows rows and the 128-byte swizzle.
int make_map(CUtensorMap *m, void *base, uint64_t cols, uint64_t rows, uint64_t planes, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return fail(ULP_ECUDA, "sage_attention: cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[3] = {cols, rows, planes};
    const cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ULP_ECUDA, "sage_attention: tensor map encoding failed (%d)", (int)r);
    return ULP_OK;
}

// v8 [B, D, h, Spad] E4M3 as a 3-D byte map (keys, head, b * D + d) with
// boxes of 128 keys x 1 head x D channels and the 128-byte swizzle; the key
// extent is n, so keys past the live prefix read as zeros.
int make_v8_map(CUtensorMap *m, const uint8_t *v8, int B, int D, int h, int n, int Spad)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return fail(ULP_ECUDA, "sage_attention: cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[3] = {(cuuint64_t)n, (cuuint64_t)h, (cuuint64_t)B * D};
    const cuuint64_t strides[2] = {(cuuint64_t)Spad, (cuuint64_t)h * Spad};
    const cuuint32_t box[3] = {(cuuint32_t)kTile, 1, (cuuint32_t)D};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(v8), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ULP_ECUDA, "sage_attention: tensor map encoding failed (%d)", (int)r);
    return ULP_OK;
}

template <int D, bool PV8>
void launch_attention(dim3 grid, cudaStream_t st, const CUtensorMap &mq, const CUtensorMap &mk,
                      const CUtensorMap &mv, const AttnArgs &a)
{
    // one CTA per SM (it holds all 512 TMEM columns): the request is padded
    // past half of the SM's shared memory where the layout is smaller
    const size_t bytes = std::max<size_t>(AttnLayout<D, PV8>::bytes + 1024, 120 * 1024);
    cudaFuncSetAttribute(sage_attention_kernel<D, PV8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    sage_attention_kernel<D, PV8><<<grid, kAttnThreads, bytes, st>>>(mq, mk, mv, a);
}

size_t widened_bytes(int B, int h, int D, int n)
{
    const size_t T = (size_t)(n + kTile - 1) / kTile * kTile;
    return 3 * (size_t)B * h * T * D * 2;
}

}  // namespace

}  // namespace ulp

using namespace ulp;

extern "C" int ulp_sage_attention_workspace_bytes(int B, int S, int h, int D, int n, size_t *bytes)
{
    if (B < 1 || S < 1 || h < 1 || (D != 64 && D != 128) || n < 1 || n > S || !bytes)
        return fail(ULP_EINVAL, "sage_attention_workspace_bytes: bad sizes");
    *bytes = widened_bytes(B, h, D, n);
    return ULP_OK;
}

extern "C" int ulp_sage_attention(const int8_t *q8, const int8_t *k8, const uint8_t *v8, const float *q_scale,
                                  const float *k_scale, const float *v_scale, int B, int S, int h, int D,
                                  int n, int q_group, float sm_scale, void *workspace, size_t workspace_bytes,
                                  void *out, int out_dtype, int pv_precision, int *status, ulp_stream_t stream)
{
    if (B < 1 || S < 1 || h < 1) return fail(ULP_EINVAL, "sage_attention: B, S, h must be positive");
    if (D != 64 && D != 128) return fail(ULP_EINVAL, "sage_attention: head_dim must be 64 or 128 (got %d)", D);
    if (n < 1 || n > S) return fail(ULP_EINVAL, "sage_attention: n = %d outside [1, %d]", n, S);
    if (int s = check_q_group(q_group, "sage_attention")) return s;
    if (out_dtype != ULP_F32 && out_dtype != ULP_BF16 && out_dtype != ULP_FP16)
        return fail(ULP_EDTYPE, "sage_attention: out_dtype must be ULP_F32, ULP_BF16 or ULP_FP16 (got %d)",
                    out_dtype);
    if (pv_precision != ULP_PV_F16 && pv_precision != ULP_PV_E4M3)
        return fail(ULP_EINVAL, "sage_attention: pv_precision must be ULP_PV_F16 or ULP_PV_E4M3 (got %d)",
                    pv_precision);
    if (!(sm_scale > 0.0f) || !(sm_scale < INFINITY))
        return fail(ULP_EINVAL, "sage_attention: sm_scale must be positive and finite");
    if ((long long)B * S * h * D > (1ll << 40) || (long long)B * h > 65535)
        return fail(ULP_EINVAL, "sage_attention: tensors too large");
    if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(out) || !aligned16(workspace) ||
        !aligned4(q_scale) || !aligned4(k_scale) || !aligned4(v_scale))
        return fail(ULP_EALIGN, "sage_attention: q8, k8, v8, out, workspace must be 16-byte aligned, "
                                "scales 4-byte aligned");
    const size_t need = widened_bytes(B, h, D, n);
    if (workspace_bytes < need)
        return fail(ULP_EINVAL, "sage_attention: workspace of %zu bytes, %zu needed", workspace_bytes, need);
    const int T = (n + kTile - 1) / kTile * kTile;
    const int Spad = (S + 63) / 64 * 64;
    const size_t plane = (size_t)B * h * T * D;
    uint16_t *q16 = reinterpret_cast<uint16_t *>(workspace), *k16 = q16 + plane, *v16 = k16 + plane;

    const bool pv8 = pv_precision == ULP_PV_E4M3;
    CUtensorMap mq, mk, mv;
    if (int s = make_map(&mq, q16, D, T, (uint64_t)B * h, kTile)) return s;
    if (int s = make_map(&mk, k16, D, T, (uint64_t)B * h, kTile)) return s;
    if (pv8) {
        if (int s = make_v8_map(&mv, v8, B, D, h, n, Spad)) return s;
    } else {
        if (int s = make_map(&mv, v16, T, D, (uint64_t)B * h, D)) return s;
    }

    const cudaStream_t st = (cudaStream_t)stream;
    WidenArgs w{q8, k8, v8, q16, k16, v16, S, h, D, n, T, Spad};
    const long long chunks = (long long)T * D / 16;
    // blockIdx.z: Q, K (and V, unless the PV product reads v8 itself)
    const dim3 wgrid((unsigned)((chunks + 255) / 256), (unsigned)(B * h), pv8 ? 2 : 3);
    attn_widen_kernel<<<wgrid, 256, 0, st>>>(w);
    if (int s = check_launch("sage_attention (widen)")) return s;

    AttnArgs a{};
    a.qs = q_scale; a.ks = k_scale; a.vs = v_scale;
    a.out = out; a.status = status; a.out_dtype = out_dtype;
    a.h = h; a.n = n; a.gq = q_group;
    a.wq = (n + q_group - 1) / q_group;
    a.wk = (n + kGK - 1) / kGK;
    a.ntk = T / kTile;
    a.scale_log2 = sm_scale * 1.4426950408889634f;
    // a CTA per pair of query tiles; an odd last tile's partner reads zeros
    const dim3 grid((unsigned)((a.ntk + kQTiles - 1) / kQTiles), (unsigned)h, (unsigned)B);
    if (D == 128) {
        if (pv8) launch_attention<128, true>(grid, st, mq, mk, mv, a);
        else launch_attention<128, false>(grid, st, mq, mk, mv, a);
    } else {
        if (pv8) launch_attention<64, true>(grid, st, mq, mk, mv, a);
        else launch_attention<64, false>(grid, st, mq, mk, mv, a);
    }
    return check_launch("sage_attention");
}
