// Internal to the sender pack: its argument block, the boundary derive it
// folds in, and its per-CTA body, shared by its own kernel and the
// single-launch group step.  Not part of the ABI.
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


// Rows per CTA: a whole slab, or at D = 128 with 64-row Q groups one 64-row
// half (one K group, one Q group), so that four CTAs stay resident per SM.
// A 128-row Q group stays in one CTA: splitting it across two cost more than
// it saved (a cluster exchange of the two maxima, or each half also reading
// the other's Q rows).  Every thread holds 4 rows of 16-byte vectors per
// tensor, so a CTA has R * D / 32 threads (512 or 256).
template <int D, int GQ>
constexpr int pack_rows() { return D == 128 && GQ == 64 ? 64 : 128; }
template <int D, int GQ>
constexpr int pack_threads() { return pack_rows<D, GQ>() * D / 32; }

template <int D, int GQ>
struct PackSmem {
    uint4 vtile[pack_rows<D, GQ>() * D / 8];      // V rows of the CTA
    float red[pack_threads<D, GQ>() / 32][4];     // per-warp Q0, Q1, K0, K1 maxima
    Int8Scale scl[4];                             // Q (first / second group), K (first / second group)
    float vs[D], vr[D];                           // V channel scales and their reciprocals
};

struct Slab {
    int rk, r, b, hh, js, g, L, S, row0, ts, fk, lk, tk, gu;   // js, ts: slab slot, touched slabs
};

// The CTA's rows of one slab: R = pack_rows<D, GQ>() rows from
// tb = 128 g + R hs.  FULL = all of them belong to the rank and none is
// excluded from the K amax (so no per-row predicate is needed).  GQ = Q group
// rows: 128 (the slab's group, slot js) or 64 (the K groups).
template <int D, int DT, int GQ, bool FOLD, bool FULL>
__device__ __forceinline__ void pack_slab(const PackArgs &a, const Slab &sl, int half, PackSmem<D, GQ> &sm)
{
    constexpr int R = pack_rows<D, GQ>();     // rows of the CTA
    constexpr int NV = D / 8;                 // 16-byte vectors per row
    constexpr int RL = pack_threads<D, GQ>() / NV;   // row lanes
    constexpr int IT = R / RL;                // rows per thread
    constexpr int NW = pack_threads<D, GQ>() / 32;
    constexpr int KG = R / kGK;               // K groups of the CTA
    constexpr int NQH = R / GQ;               // Q groups of the CTA
    static_assert(IT == 4, "4 rows per thread");
    static_assert(IT % KG == 0 && RL * IT / KG == kGK, "the CTA's rows split into whole K groups");
    static_assert(GQ == 64 || GQ == 128, "Q groups of 64 or 128 rows");

    const int c = threadIdx.x % NV, rl = threadIdx.x / NV;
    const int L = sl.L, row0 = sl.row0, g = sl.g;
    const size_t HD = (size_t)a.H * D;
    const int hs = R == kSlab ? 0 : half;             // the slab's half (64-row CTAs)
    const int tb = g * kSlab + hs * R;                // the CTA's first row
    const int t_first = tb + rl;                      // row i is t_first + i * RL
    // global row t of this rank lives at in_base + t * HD
    const size_t in_base = ((size_t)sl.rk * a.B + sl.b) * L * HD - (size_t)row0 * HD + (size_t)sl.hh * D + c * 8;
    auto valid = [&](int t) { return FULL || (t >= row0 && t < row0 + L); };
    if (!a.early) pdl_wait();

    // ---- 1. V rows -> shared memory
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const int t = t_first + i * RL;
        if (valid(t)) cp_async16(&sm.vtile[(i * RL + rl) * NV + c], a.v + in_base + (size_t)t * HD);
    }
    cp_async_commit();

    // ---- 2. Q, K rows -> registers; V channel scales
    uint4 qv[IT], kv[IT];
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const int t = t_first + i * RL;
        if (valid(t)) {
            qv[i] = ld_stream(a.q + in_base + (size_t)t * HD);
            kv[i] = ld_stream(a.k + in_base + (size_t)t * HD);
        }
    }
    if (threadIdx.x < D) {
        const float s = a.v_scale[((size_t)sl.b * a.H + sl.hh) * D + threadIdx.x];
        sm.vs[threadIdx.x] = s;
        sm.vr[threadIdx.x] = __frcp_rn(s);
    }
    float m[8];
    to_f32x8<DT>(*reinterpret_cast<const uint4 *>(a.k_mean + ((size_t)sl.b * a.H + sl.hh) * D + c * 8), m);

    // ---- 3. amax: Q per Q group of the slab (all rows, or each 64-row
    // half), K per 64-row half.  Per channel pair, a running max and min of
    // the raw 16-bit values (exact); then max |Q| = max(maxQ, -minQ) and, rn
    // subtraction being monotone, max |rn(K - m)| = max(rn(maxK - m), rn(m - minK)).
    float qmax0 = -INFINITY, qmax1 = -INFINITY, kmax0 = -INFINITY, kmax1 = -INFINITY;
#pragma unroll
    for (int hq = 0; hq < NQH; ++hq) {
        Pair16<DT> pr[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) pr[x].init();
#pragma unroll
        for (int i = hq * IT / NQH; i < (hq + 1) * IT / NQH; ++i) {
            if (valid(t_first + i * RL)) {
                pr[0].add(qv[i].x);
                pr[1].add(qv[i].y);
                pr[2].add(qv[i].z);
                pr[3].add(qv[i].w);
            }
        }
        float v = -INFINITY;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const float2 hi = pair_f32<DT>(pr[x].mx), lo = pair_f32<DT>(pr[x].mn);
            v = fmaxf(v, fmaxf(fmaxf(hi.x, -lo.x), fmaxf(hi.y, -lo.y)));
        }
        if (hq == 0) qmax0 = v;
        else qmax1 = v;
    }
#pragma unroll
    for (int hk = 0; hk < KG; ++hk) {
        Pair16<DT> pr[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) pr[x].init();
#pragma unroll
        for (int i = hk * IT / KG; i < (hk + 1) * IT / KG; ++i) {
            const int t = t_first + i * RL;
            // live rows only in the partial live group
            if (FULL || (valid(t) && !(t >= a.used && t / kGK == sl.gu))) {
                pr[0].add(kv[i].x);
                pr[1].add(kv[i].y);
                pr[2].add(kv[i].z);
                pr[3].add(kv[i].w);
            }
        }
        float v = -INFINITY;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const float2 hi = pair_f32<DT>(pr[x].mx), lo = pair_f32<DT>(pr[x].mn);
            v = fmaxf(v, fmaxf(fmaxf(__fsub_rn(hi.x, m[2 * x]), __fsub_rn(m[2 * x], lo.x)),
                               fmaxf(__fsub_rn(hi.y, m[2 * x + 1]), __fsub_rn(m[2 * x + 1], lo.y))));
        }
        if (hk == 0) kmax0 = v;
        else kmax1 = v;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (a.early) pdl_wait();          // k_amax, the partials and the chunks belong to the chain
    qmax0 = warp_max(qmax0);
    if (NQH == 2) qmax1 = warp_max(qmax1);
    kmax0 = warp_max(kmax0);
    if (KG == 2) kmax1 = warp_max(kmax1);
    if (lane == 0) {
        sm.red[warp][0] = qmax0;
        sm.red[warp][1] = qmax1;
        sm.red[warp][2] = kmax0;
        sm.red[warp][3] = kmax1;
    }
    __syncthreads();

    const size_t amax_row = (((size_t)sl.rk * a.B + sl.b) * a.H + sl.hh) * a.nk;
    if (warp == 0) {
        // the rank's first/last K groups in this CTA, derived from the
        // gathered raw-K min/max when they are given (all 32 lanes; the
        // value goes to k_amax, where the K scale below reads it)
        if (FOLD) {
#pragma unroll
            for (int hk = 0; hk < KG; ++hk) {
                const int gk = 2 * g + KG * hs + hk;
                if (gk >= sl.fk && gk <= sl.lk && (gk == sl.fk || gk == sl.lk)) {
                    const float d = derive_slot_warp<D, DT>(a.gathered, a.k_mean, a.B, a.H, L, a.P, sl.b, sl.hh, gk);
                    if (lane == 0) a.k_amax[amax_row + (gk - sl.fk)] = d;
                }
            }
            __syncwarp();
        }
        qmax0 = lane < NW ? sm.red[lane][0] : -INFINITY;
        qmax1 = lane < NW ? sm.red[lane][1] : -INFINITY;
        kmax0 = lane < NW ? sm.red[lane][2] : -INFINITY;
        kmax1 = lane < NW ? sm.red[lane][3] : -INFINITY;
        qmax0 = warp_max(qmax0);
        if (NQH == 2) qmax1 = warp_max(qmax1);
        kmax0 = warp_max(kmax0);
        if (KG == 2) kmax1 = warp_max(kmax1);
        if (lane < NQH) {
            // Q group gg of this lane; its slot range and boundary test
            const int gg = (kSlab / GQ) * g + (R / GQ) * hs + lane;
            const bool touched = GQ == kSlab || (gg >= sl.fk && gg <= sl.lk);
            const bool boundary = GQ == kSlab ? (sl.js == 0 || sl.js == sl.ts - 1) : (gg == sl.fk || gg == sl.lk);
            float qs = 1.0f;                                 // a half with no row of the rank
            if (touched) {
                float qam;
                if (boundary) {                              // merge the gathered partials
                    const int rend = min(gg * GQ + GQ, sl.S);
                    qam = -INFINITY;
                    for (int rr = (gg * GQ) / L; rr <= (rend - 1) / L; ++rr) {
                        const int ee = gg == first_group(rr, L, GQ) ? 0 : 1;
                        qam = fmaxf(qam, a.qpart[(((size_t)rr * a.B + sl.b) * a.H + sl.hh) * 2 + ee]);
                    }
                } else {
                    qam = floor_eps(lane == 0 ? qmax0 : qmax1);
                }
                qs = __fdiv_rn(qam, 127.0f);
            }
            sm.scl[lane] = int8_scale(qs);
        } else if (lane >= 2 && lane < 2 + KG) {
            const int hk = lane - 2, gk = 2 * g + KG * hs + hk;
            float ks = 1.0f;
            if (gk >= sl.fk && gk <= sl.lk) {
                const int jk = gk - sl.fk;
                float kam;
                if (jk == 0 || jk == sl.tk - 1 || !a.fused) {
                    kam = a.k_amax[amax_row + jk];
                } else {
                    kam = floor_eps(hk == 0 ? kmax0 : kmax1);
                    a.k_amax[amax_row + jk] = kam;
                }
                ks = __fdiv_rn(kam, 127.0f);
            }
            sm.scl[2 + hk] = int8_scale(ks);
        }
    }
    __syncthreads();

    // ---- scale slots of the chunk
    const int p = sl.hh / a.h, j = sl.hh - p * a.h;
    const size_t cb = a.lay.bytes;
    uint8_t *chunk = a.send + (a.layout == ULP_SEND_DEST_MAJOR
                                   ? ((size_t)p * a.P + sl.r) * cb
                                   : ((size_t)(a.rank >= 0 ? 0 : sl.rk) * a.P + p) * cb);
    if (threadIdx.x < 32) {
        float *qs_out = reinterpret_cast<float *>(chunk + a.lay.qs) + ((size_t)sl.b * a.h + j) * a.nq;
        float *ks_out = reinterpret_cast<float *>(chunk + a.lay.ks) + ((size_t)sl.b * a.h + j) * a.nk;
        const int t = threadIdx.x;
        if (GQ == kSlab && t == 0 && hs == 0) qs_out[sl.js] = sm.scl[0].s;   // one writer per slab
        if (GQ != kSlab && t < NQH) {
            const int gg = (kSlab / GQ) * g + (R / GQ) * hs + t;
            if (gg >= sl.fk && gg <= sl.lk) qs_out[gg - sl.fk] = sm.scl[t].s;
        }
        if (t >= 2 && t < 2 + KG) {
            const int gk = 2 * g + KG * hs + (t - 2);
            if (gk >= sl.fk && gk <= sl.lk) ks_out[gk - sl.fk] = sm.scl[t].s;
        }
        // slots past the touched groups: the CTA of the slab's last rows
        if (sl.js == sl.ts - 1 && (R == kSlab || hs == 1)) {
            if (sl.b == a.B - 1 && j == a.h - 1) {
                // the last writer of the chunk's scale sections zeroes their
                // alignment padding, so every chunk byte is defined
                const size_t nqs = (size_t)a.B * a.h * a.nq, nks = (size_t)a.B * a.h * a.nk;
                float *qsec = reinterpret_cast<float *>(chunk + a.lay.qs);
                float *ksec = reinterpret_cast<float *>(chunk + a.lay.ks);
                if (nqs + t < (a.lay.ks - a.lay.qs) / 4) qsec[nqs + t] = 0.0f;
                if (nks + t < (a.lay.bytes - a.lay.ks) / 4) ksec[nks + t] = 0.0f;
            }
            const int tq = GQ == kSlab ? sl.ts : sl.tk;  // touched Q groups
            if (tq + t < a.nq) qs_out[tq + t] = __fdiv_rn(kEps, 127.0f);
            if (sl.tk + t < a.nk) {
                float kam;
                if (a.fused) {
                    kam = kEps;
                    a.k_amax[amax_row + sl.tk + t] = kam;
                } else {
                    kam = a.k_amax[amax_row + sl.tk + t];
                }
                ks_out[sl.tk + t] = __fdiv_rn(kam, 127.0f);
            }
        }
    }

    // ---- 4. Q codes, then K codes, from registers (8 bytes per row).  Q's
    // scale bounds every Q element of its group, and K's every live K row, so
    // only K rows at or past `used` (padding) can saturate -- or any row when
    // the caller supplied the K amax (unfused).
    const size_t hD = (size_t)a.h * D;
    // global row t of this rank goes to out_base + t * hD within a section
    uint8_t *out_base = chunk + ((size_t)sl.b * L - row0) * hD + (size_t)j * D + c * 8;
#pragma unroll
    for (int hq = 0; hq < NQH; ++hq) {
        const Int8Scale qsc = sm.scl[hq];
#pragma unroll
        for (int i = hq * IT / NQH; i < (hq + 1) * IT / NQH; ++i) {
            const int t = t_first + i * RL;
            if (valid(t)) {
                float f[8];
                to_f32x8<DT>(qv[i], f);
                *reinterpret_cast<uint2 *>(out_base + (size_t)t * hD + a.lay.q) = int8_codes8<false>(f, qsc);
            }
        }
    }
    to_f32x8<DT>(*reinterpret_cast<const uint4 *>(a.k_mean + ((size_t)sl.b * a.H + sl.hh) * D + c * 8), m);
    const bool k_sat = !a.fused || tb + R > a.used;   // CTA-uniform
#pragma unroll
    for (int hk = 0; hk < KG; ++hk) {
        const Int8Scale ksc = sm.scl[2 + hk];
#pragma unroll
        for (int i = hk * IT / KG; i < (hk + 1) * IT / KG; ++i) {
            const int t = t_first + i * RL;
            if (valid(t)) {
                float f[8];
                to_f32x8<DT>(kv[i], f);
#pragma unroll
                for (int x = 0; x < 8; x += 2)
                    f2unpack(f2sub(f2pack(f[x], f[x + 1]), f2pack(m[x], m[x + 1])), f[x], f[x + 1]);
                *reinterpret_cast<uint2 *>(out_base + (size_t)t * hD + a.lay.k) =
                    k_sat ? int8_codes8<true>(f, ksc) : int8_codes8<false>(f, ksc);
            }
        }
    }

    // ---- 5. V codes from shared memory (rows this thread copied itself)
    float vs[8], vr[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) {
        vs[x] = sm.vs[c * 8 + x];
        vr[x] = sm.vr[c * 8 + x];
    }
    cp_async_wait_all();
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const int t = t_first + i * RL;
        if (valid(t)) {
            *reinterpret_cast<uint2 *>(out_base + (size_t)t * hD + a.lay.v) =
                e4m3_codes8<DT>(sm.vtile[(i * RL + rl) * NV + c], vs, vr);
        }
    }
}

// One CTA per slab, or per 64-row half at D = 128 with 64-row Q groups
// (block index = head, slab index (times 2 plus the half), rank * B + batch).
//  1. V rows of the CTA -> shared memory with cp.async (each thread later
//     reads back only the bytes it copied, so no barrier guards them);
//  2. Q and K rows -> registers; V channel scales and their reciprocals ->
//     shared memory (one reciprocal per channel);
//  3. Q amax and the amax of the CTA's 64-row K groups: per-thread,
//     per-warp, then warp 0 merges the warps, applies the boundary rules and
//     publishes the scales;
//  4. Q/K codes from the registers; 5. V codes from shared memory.
template <int D, int DT, int GQ, bool FOLD>
__device__ __forceinline__ void pack_block(const PackArgs &a, unsigned bx, unsigned by, unsigned bz,
                                           PackSmem<D, GQ> &sm)
{
    constexpr int R = pack_rows<D, GQ>();
    Slab sl;
    sl.hh = bx;
    const int hs = R == kSlab ? 0 : (int)(by & 1u);   // the slab's half (64-row CTAs)
    sl.js = R == kSlab ? (int)by : (int)(by >> 1);
    sl.rk = bz / a.B;
    sl.b = bz - sl.rk * a.B;
    sl.r = a.rank >= 0 ? a.rank : sl.rk;
    sl.L = a.L;
    sl.S = a.P * a.L;
    sl.row0 = sl.r * a.L;
    const int fs = first_group(sl.r, a.L, kSlab);
    sl.ts = last_group(sl.r, a.L, kSlab) - fs + 1;
    if (sl.js >= sl.ts) {
        pdl_wait();
        return;
    }
    sl.g = fs + sl.js;
    sl.fk = first_group(sl.r, a.L, kGK);
    sl.lk = last_group(sl.r, a.L, kGK);
    sl.tk = sl.lk - sl.fk + 1;
    sl.gu = a.used < sl.S ? (a.used - 1) / kGK : -1;
    // FULL: the CTA's rows all belong to the rank and its K groups exclude no
    // row (written per case: the whole-slab form keeps that kernel free of spills)
    bool full;
    if (R == kSlab) {
        full = sl.g * kSlab >= sl.row0 && sl.g * kSlab + kSlab <= sl.row0 + a.L &&
               !(sl.gu >= 0 && sl.gu / 2 == sl.g);
    } else {
        const int tb = sl.g * kSlab + hs * R;
        full = tb >= sl.row0 && tb + R <= sl.row0 + a.L && sl.gu != 2 * sl.g + hs;
    }
    if (full) pack_slab<D, DT, GQ, FOLD, true>(a, sl, hs, sm);
    else pack_slab<D, DT, GQ, FOLD, false>(a, sl, hs, sm);
}

// Checks the arguments of ulp_pack (all but enable_pdl) and fills `a` and
// the launch grid.  Returns a status (ULP_OK on success).
int pack_setup(PackArgs &a, dim3 &grid, const void *q, const void *k, const void *v, const void *k_mean,
               int dtype, float *k_amax, const float *gathered_q_partial, const float *gathered_minmax,
               const float *v_scale, int B, int L, int H, int D, int rank, int world_size, int used_sequence,
               int q_group, int fused, uint8_t *send, int send_layout);

}  // namespace ulp
