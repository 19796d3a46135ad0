// Internal: the raw-K boundary min/max producer's per-unit body, shared by
// its own kernel and the single-launch group step.  Not part of the ABI.
#pragma once

#include "ulp_internal.cuh"

namespace ulp {

struct MinmaxArgs {
    const uint16_t *k, *q;
    float *minmax, *qpart;
    int B, L, H, P, rank, used;
    int gq;   // Q group rows, 64 or 128
};

// 128-thread barriers of the unit's threads
struct SyncCta {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};
struct SyncNamed {   // named barrier `id` (1..15) over one 128-thread quarter of a larger CTA
    int id;
    __device__ __forceinline__ void operator()() const { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
};

template <int D>
struct MinmaxSmem {
    float smn[128 / (D / 8)][D], smx[128 / (D / 8)][D];
    float red[4];
};

// One unit (rank, b, head, e) on 128 threads (tid 0..127): e = 0 first
// touched group, e = 1 last.  `sync` is a barrier over exactly these threads.
template <int D, int DT, class Sync>
__device__ __forceinline__ void boundary_minmax_unit(const MinmaxArgs &a, int blk, int tid, MinmaxSmem<D> &sm,
                                                     Sync sync)
{
    constexpr int NV = D / 8, RL = 128 / NV, ITK = kGK / RL, ITQ = kGQ / RL;
    const int e = blk & 1; blk >>= 1;
    const int hh = blk % a.H; blk /= a.H;
    const int b = blk % a.B; blk /= a.B;
    const int rk = blk;
    const int r = a.rank >= 0 ? a.rank : rk;
    const int row0 = r * a.L;
    const int c = tid % NV, rl = tid / NV;
    const size_t HD = (size_t)a.H * D;
    const size_t off = (size_t)rk * a.B * a.L * HD + (size_t)b * a.L * HD + (size_t)hh * D + c * 8;

    // ---- K: raw min / max per channel over the live rows of the group
    const int g = e == 0 ? first_group(r, a.L, kGK) : last_group(r, a.L, kGK);
    const int lo = max(g * kGK, row0);
    const int hi = min(min(g * kGK + kGK, row0 + a.L), a.used);
    float mn[8], mx[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { mn[i] = INFINITY; mx[i] = -INFINITY; }
    {
        uint4 v[ITK];
#pragma unroll
        for (int i = 0; i < ITK; ++i) {
            const int t = g * kGK + i * RL + rl;
            if (t >= lo && t < hi) v[i] = ld_stream(a.k + off + (size_t)(t - row0) * HD);
        }
#pragma unroll
        for (int i = 0; i < ITK; ++i) {
            const int t = g * kGK + i * RL + rl;
            if (t >= lo && t < hi) {
                float f[8];
                to_f32x8<DT>(v[i], f);
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const float y = f[x] == 0.0f ? 0.0f : f[x];   // -0 -> +0
                    mn[x] = fminf(mn[x], y);
                    mx[x] = fmaxf(mx[x], y);
                }
            }
        }
    }
#pragma unroll
    for (int x = 0; x < 8; ++x) {
        sm.smn[rl][c * 8 + x] = mn[x];
        sm.smx[rl][c * 8 + x] = mx[x];
    }

    // ---- Q: partial amax over the rank's rows of its first / last Q group
    // (ITQ covers the widest group; rows past a narrower group fail the test)
    const int gq = e == 0 ? first_group(r, a.L, a.gq) : last_group(r, a.L, a.gq);
    const int qlo = max(gq * a.gq, row0), qhi = min(gq * a.gq + a.gq, row0 + a.L);
    float qa = -INFINITY;
    {
        uint4 v[ITQ];
#pragma unroll
        for (int i = 0; i < ITQ; ++i) {
            const int t = gq * a.gq + i * RL + rl;
            if (t >= qlo && t < qhi) v[i] = ld_stream(a.q + off + (size_t)(t - row0) * HD);
        }
#pragma unroll
        for (int i = 0; i < ITQ; ++i) {
            const int t = gq * a.gq + i * RL + rl;
            if (t >= qlo && t < qhi) {
                float f[8];
                to_f32x8<DT>(v[i], f);
#pragma unroll
                for (int x = 0; x < 8; ++x) qa = fmaxf(qa, fabsf(f[x]));
            }
        }
    }
    qa = warp_max(qa);
    if ((tid & 31) == 0) sm.red[tid >> 5] = qa;
    sync();

    const size_t obase = ((((size_t)rk * a.B + b) * a.H + hh) * 2 + e) * 2 * D;
    if (tid < D) {
        const int d = tid;
        float vmin = INFINITY, vmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < RL; ++i) {
            vmin = fminf(vmin, sm.smn[i][d]);
            vmax = fmaxf(vmax, sm.smx[i][d]);
        }
        a.minmax[obase + d] = vmin;
        a.minmax[obase + D + d] = vmax;
    }
    if (tid == 0) {
        const float v = fmaxf(fmaxf(sm.red[0], sm.red[1]), fmaxf(sm.red[2], sm.red[3]));
        a.qpart[(((size_t)rk * a.B + b) * a.H + hh) * 2 + e] = floor_eps(v);
    }
}

}  // namespace ulp
