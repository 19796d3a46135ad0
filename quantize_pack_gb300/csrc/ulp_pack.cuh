// Internal to the sender pack: its argument block and the boundary derive it
// folds in.  Not part of the ABI.
#pragma once

#include "ulp_internal.cuh"

namespace ulp {

struct PackArgs {
    const uint16_t *q, *k, *v, *k_mean;
    float *k_amax;
    const float *qpart;      // [P, B, H, 2]
    const float *gathered;   // [P, B, H, 2, 2, D] raw-K min/max, or null: K boundary slots read from k_amax
    const float *v_scale;    // [B, H, D]
    uint8_t *send;
    ChunkLayout lay;
    int B, L, H, P, h, rank, used, fused, layout, nq, nk;   // nq = slots(L, q_group)
    int early;   // read q, k, v, k_mean, v_scale before waiting for the preceding kernel
};

constexpr int kSlab = 128;   // rows of a slab: one 128-row group = two 64-row groups

// Page "derive_k_boundary_amax" (formula and the proof paragraph after it):
// the amax of 64-row K group g of (b, head hh), rebuilt from the raw-K
// min/max of every rank touching g:
//   max(1e-7, max_{r touching g} max_d max(rn(maxK - m_d), rn(m_d - minK))).
// A rank whose slice of g has no live row contributes the sentinels
// (+inf, -inf), i.e. -inf.  The floor is monotone, so flooring the single
// maximum gives the bits of flooring each term.  All 32 lanes of the warp
// call it; every lane gets the value.
template <int D, int DT>
__device__ __forceinline__ float derive_slot_warp(const float *gathered, const uint16_t *k_mean, int B, int H,
                                                  int L, int P, int b, int hh, int g)
{
    const int lane = threadIdx.x & 31;
    const int S = P * L;
    const int r_lo = (g * kGK) / L, r_hi = (min(g * kGK + kGK, S) - 1) / L;
    float acc = -INFINITY;
#pragma unroll
    for (int x = 0; x < D / 32; ++x) {
        const int d = lane + 32 * x;
        const uint16_t mb = k_mean[((size_t)b * H + hh) * D + d];
        const float m = DT == ULP_BF16 ? __uint_as_float((uint32_t)mb << 16) : __half2float(__ushort_as_half(mb));
        for (int rr = r_lo; rr <= r_hi; ++rr) {
            const int ee = g == first_group(rr, L, kGK) ? 0 : 1;
            const size_t base = ((((size_t)rr * B + b) * H + hh) * 2 + ee) * 2 * D;
            acc = fmaxf(acc, fmaxf(__fsub_rn(gathered[base + D + d], m), __fsub_rn(m, gathered[base + d])));
        }
    }
    return floor_eps(warp_max(acc));
}

}  // namespace ulp
