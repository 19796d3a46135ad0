// Internal: unpack_for_sage's block body and argument setup, shared by its
// own kernel and the single-launch group step.  Not part of the ABI.
#pragma once

#include "ulp_internal.cuh"

namespace ulp {

constexpr int kUnpackThreads = 128;
constexpr int kCopyVecPerThread = 16;
constexpr int kCopyPiece = kUnpackThreads * kCopyVecPerThread * 16;   // bytes per copy block

struct UnpackArgs {
    const uint8_t *recv;
    int8_t *q8, *k8;
    uint8_t *v8;
    float *qs, *ks;
    ChunkLayout lay;
    int B, L, h, P, S, Spad, wq, wk, nq, nk, nd;
    int gq;                    // Q group rows, 64 or 128
    int TT, CC;                // V tiles: t-tiles of 128 rows, 64-byte column blocks
    long long nVtiles, nVblk;  // V warp tiles, V blocks
    long long pieces, nCblk;   // copy pieces per span, copy blocks
    long long nSblk;           // scale blocks
};

__device__ __forceinline__ void transpose4x4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t &b0, uint32_t &b1, uint32_t &b2, uint32_t &b3)
{
    const uint32_t t0 = __byte_perm(a0, a1, 0x5140), t1 = __byte_perm(a0, a1, 0x7362);
    const uint32_t t2 = __byte_perm(a2, a3, 0x5140), t3 = __byte_perm(a2, a3, 0x7362);
    b0 = __byte_perm(t0, t2, 0x5410);
    b1 = __byte_perm(t0, t2, 0x7632);
    b2 = __byte_perm(t1, t3, 0x5410);
    b3 = __byte_perm(t1, t3, 0x7632);
}

template <int D>
__device__ __forceinline__ void unpack_v_tile(const UnpackArgs &a, long long tile)
{
    const int lane = threadIdx.x & 31;
    const int tb = lane >> 2, cbk = lane & 3;
    const int cc = (int)(tile % a.CC); tile /= a.CC;
    const int tt = (int)(tile % a.TT); tile /= a.TT;
    const int b = (int)(tile % a.B);
    const int p = (int)(tile / a.B);
    const size_t cbytes = a.lay.bytes;
    const size_t hD = (size_t)a.h * D;
    const uint8_t *rbase = a.recv + (size_t)p * a.P * cbytes + a.lay.v + (size_t)b * a.L * hD;
    const int t0 = tt * 128 + tb * 16;
    const int col = cc * 64 + cbk * 16;

    uint32_t w[16][4];
    {
        int s = t0 / a.L, tl = t0 - s * a.L;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (t0 + i < a.S) v = ld_stream(rbase + (size_t)s * cbytes + (size_t)tl * hD + col);
            w[i][0] = v.x; w[i][1] = v.y; w[i][2] = v.z; w[i][3] = v.w;
            if (++tl == a.L) { tl = 0; ++s; }
        }
    }
    if (t0 >= a.Spad) return;
    uint8_t *obase = a.v8 + (size_t)p * a.B * D * a.h * a.Spad + t0;
#pragma unroll
    for (int qw = 0; qw < 4; ++qw) {              // 4 source columns per word
        uint32_t o[4][4];                         // [column in word][row word]
#pragma unroll
        for (int pr = 0; pr < 4; ++pr)            // 4 rows per word
            transpose4x4(w[4 * pr][qw], w[4 * pr + 1][qw], w[4 * pr + 2][qw], w[4 * pr + 3][qw],
                         o[0][pr], o[1][pr], o[2][pr], o[3][pr]);
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int c = col + 4 * qw + n;
            const int j = c / D, d = c % D;
            uint8_t *dst = obase + (((size_t)b * D + d) * a.h + j) * a.Spad;
            *reinterpret_cast<uint4 *>(dst) = make_uint4(o[n][0], o[n][1], o[n][2], o[n][3]);
        }
    }
}

// One block's work (128 threads, tid 0..127): V tiles, a Q/K copy piece or
// scale slots, by block index.  No barrier: every thread or warp works alone.
template <int D>
__device__ __forceinline__ void unpack_unit(const UnpackArgs &a, long long blk, int tid)
{
    if (blk < a.nVblk) {
        const long long tile = blk * (kUnpackThreads / 32) + (tid >> 5);
        if (tile < a.nVtiles) unpack_v_tile<D>(a, tile);
        return;
    }
    blk -= a.nVblk;
    const size_t cbytes = a.lay.bytes;
    const size_t hD = (size_t)a.h * D;
    if (blk < a.nCblk) {
        // span = (p, tensor, b, s): L*h*D contiguous bytes on both sides
        long long span = blk / a.pieces;
        const long long piece = blk % a.pieces;
        const int s = (int)(span % a.P); span /= a.P;
        const int b = (int)(span % a.B); span /= a.B;
        const int tensor = (int)(span % 2);
        const int p = (int)(span / 2);
        const size_t len = (size_t)a.L * hD;
        const uint4 *src = reinterpret_cast<const uint4 *>(
            a.recv + ((size_t)p * a.P + s) * cbytes + (tensor ? a.lay.k : a.lay.q) + (size_t)b * len);
        uint4 *dst = reinterpret_cast<uint4 *>(
            (tensor ? a.k8 : a.q8) + (size_t)p * a.B * a.S * hD + ((size_t)b * a.S + (size_t)s * a.L) * hD);
        const size_t nvec = len / 16;
        const size_t v0 = (size_t)piece * (kCopyPiece / 16) + tid;
        uint4 v[kCopyVecPerThread];
#pragma unroll
        for (int i = 0; i < kCopyVecPerThread; ++i) {
            const size_t idx = v0 + (size_t)i * kUnpackThreads;
            if (idx < nvec) v[i] = ld_stream(src + idx);
        }
#pragma unroll
        for (int i = 0; i < kCopyVecPerThread; ++i) {
            const size_t idx = v0 + (size_t)i * kUnpackThreads;
            if (idx < nvec) dst[idx] = v[i];
        }
        return;
    }
    blk -= a.nCblk;
    // scales: one thread per output slot
    const long long per = (long long)a.B * a.h * (a.wq + a.wk);
    const long long idx = blk * kUnpackThreads + tid;
    if (idx >= per * a.nd) return;
    const int p = (int)(idx / per);
    long long rem = idx % per;
    const int bj = (int)(rem / (a.wq + a.wk));
    int g = (int)(rem % (a.wq + a.wk));
    const uint8_t *rp = a.recv + (size_t)p * a.P * cbytes;
    if (g < a.wq) {
        const int s = (g * a.gq) / a.L;
        const float *src = reinterpret_cast<const float *>(rp + (size_t)s * cbytes + a.lay.qs);
        a.qs[((size_t)p * a.B * a.h + bj) * a.wq + g] = src[(size_t)bj * a.nq + (g - first_group(s, a.L, a.gq))];
    } else {
        g -= a.wq;
        const int s = (g * kGK) / a.L;
        const float *src = reinterpret_cast<const float *>(rp + (size_t)s * cbytes + a.lay.ks);
        a.ks[((size_t)p * a.B * a.h + bj) * a.wk + g] = src[(size_t)bj * a.nk + (g - first_group(s, a.L, kGK))];
    }
}

// Checks the arguments of unpack_for_sage and fills `a`; `blocks` = the
// launch's 128-thread blocks.  Returns a status (ULP_OK on success).
int unpack_setup(UnpackArgs &a, long long &blocks, const uint8_t *recv, int B, int L, int h, int D,
                 int world_size, int aligned, int scale_sequence, int q_group, int8_t *q8, int8_t *k8,
                 uint8_t *v8, float *q_scale, float *k_scale, int num_dests);

}  // namespace ulp
