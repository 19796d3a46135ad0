// Sender pack: INT8 Q/K with per-group fp32 scales and FP8 E4M3 V with the
// caller's V scale, written into the source-major chunks that the Ulysses
// all-to-all moves (page "unpack_for_sage": recv_u8 is the source-major
// buffer of chunks; Returns: the V scale remains with the caller).
//
// One CTA handles one 128-row global Q group (a "slab") of one head on one
// rank: Q, K and V rows of the slab are loaded once into registers, the Q
// amax and the amax of the slab's two 64-row K groups are reduced in the CTA,
// and the codes are written from the same registers.  Boundary groups (the
// rank's first/last touched group) take their amax from the gathered partials
// (Q) or the derived slots (K), so every input byte crosses HBM once.
#include "ulp_internal.cuh"

namespace ulp {

struct PackArgs {
    const uint16_t *q, *k, *v, *k_mean;
    float *k_amax;
    const float *qpart;    // [P, B, H, 2]
    const float *v_scale;  // [B, H, D]
    uint8_t *send;
    ChunkLayout lay;
    int B, L, H, P, h, rank, used, fused, layout, nq, nk;
};

template <int D, int DT>
__global__ void __launch_bounds__(256) pack_kernel(PackArgs a)
{
    constexpr int NV = D / 8;        // 16-byte vectors per row
    constexpr int RL = 256 / NV;     // row lanes
    constexpr int IT = kGQ / RL;     // rows per thread
    static_assert(IT % 2 == 0 && RL * IT / 2 == kGK, "slab halves must be the K groups");

    int blk = blockIdx.x;
    const int hh = blk % a.H; blk /= a.H;
    const int jq = blk % a.nq; blk /= a.nq;
    const int b = blk % a.B; blk /= a.B;
    const int rk = blk;
    const int r = a.rank >= 0 ? a.rank : rk;
    const int L = a.L, S = a.P * L, row0 = r * L;
    const int fq = first_group(r, L, kGQ), tq = last_group(r, L, kGQ) - fq + 1;
    if (jq >= tq) return;
    const int fk = first_group(r, L, kGK), lk = last_group(r, L, kGK), tk = lk - fk + 1;
    const int g = fq + jq;
    const int c = threadIdx.x % NV, rl = threadIdx.x / NV;
    const int gu = a.used < S ? (a.used - 1) / kGK : -1;
    const size_t HD = (size_t)a.H * D;
    const size_t in_off = (size_t)rk * a.B * L * HD + (size_t)b * L * HD + (size_t)hh * D + c * 8;

    // ---- load the slab (rows of this rank only)
    uint4 qv[IT], kv[IT], vv[IT];
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const int t = g * kGQ + i * RL + rl;
        if (t >= row0 && t < row0 + L) {
            const size_t o = in_off + (size_t)(t - row0) * HD;
            qv[i] = ld_stream(a.q + o);
            kv[i] = ld_stream(a.k + o);
            vv[i] = ld_stream(a.v + o);
        }
    }
    float m[8];
    to_f32x8<DT>(*reinterpret_cast<const uint4 *>(a.k_mean + ((size_t)b * a.H + hh) * D + c * 8), m);

    // ---- amax of the slab: Q over all its rows, K per 64-row half
    float qmax = -INFINITY, kmax0 = -INFINITY, kmax1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const int t = g * kGQ + i * RL + rl;
        if (t >= row0 && t < row0 + L) {
            float f[8];
            to_f32x8<DT>(qv[i], f);
#pragma unroll
            for (int x = 0; x < 8; ++x) qmax = fmaxf(qmax, fabsf(f[x]));
            if (!(t >= a.used && t / kGK == gu)) {           // live rows only in the partial group
                to_f32x8<DT>(kv[i], f);
                float km = -INFINITY;
#pragma unroll
                for (int x = 0; x < 8; ++x) km = fmaxf(km, fabsf(__fsub_rn(f[x], m[x])));
                if (i < IT / 2) kmax0 = fmaxf(kmax0, km);
                else kmax1 = fmaxf(kmax1, km);
            }
        }
    }
    __shared__ float red[8][3];
    qmax = warp_max(qmax);
    kmax0 = warp_max(kmax0);
    kmax1 = warp_max(kmax1);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[warp][0] = qmax;
        red[warp][1] = kmax0;
        red[warp][2] = kmax1;
    }
    __syncthreads();
    qmax = red[0][0];
    kmax0 = red[0][1];
    kmax1 = red[0][2];
#pragma unroll
    for (int w = 1; w < 8; ++w) {
        qmax = fmaxf(qmax, red[w][0]);
        kmax0 = fmaxf(kmax0, red[w][1]);
        kmax1 = fmaxf(kmax1, red[w][2]);
    }

    // ---- scales
    float qam;
    if (jq == 0 || jq == tq - 1) {                      // boundary: merge the gathered partials
        const int rend = min(g * kGQ + kGQ, S);
        qam = -INFINITY;
        for (int rr = (g * kGQ) / L; rr <= (rend - 1) / L; ++rr) {
            const int ee = g == first_group(rr, L, kGQ) ? 0 : 1;
            qam = fmaxf(qam, a.qpart[(((size_t)rr * a.B + b) * a.H + hh) * 2 + ee]);
        }
    } else {
        qam = floor_eps(qmax);
    }
    const float qs = __fdiv_rn(qam, 127.0f);
    const size_t amax_row = (((size_t)rk * a.B + b) * a.H + hh) * a.nk;
    float ks[2] = {1.0f, 1.0f};
#pragma unroll
    for (int hk = 0; hk < 2; ++hk) {
        const int gk = 2 * g + hk;
        if (gk < fk || gk > lk) continue;
        const int jk = gk - fk;
        float kam;
        if (jk == 0 || jk == tk - 1 || !a.fused) {
            kam = a.k_amax[amax_row + jk];
        } else {
            kam = floor_eps(hk == 0 ? kmax0 : kmax1);
            if (threadIdx.x == 0) a.k_amax[amax_row + jk] = kam;
        }
        ks[hk] = __fdiv_rn(kam, 127.0f);
    }

    const int p = hh / a.h, j = hh % a.h;
    const size_t cb = a.lay.bytes;
    uint8_t *chunk = a.send + (a.layout == ULP_SEND_DEST_MAJOR
                                   ? ((size_t)p * a.P + r) * cb
                                   : ((size_t)(a.rank >= 0 ? 0 : rk) * a.P + p) * cb);
    float *qs_out = reinterpret_cast<float *>(chunk + a.lay.qs) + ((size_t)b * a.h + j) * a.nq;
    float *ks_out = reinterpret_cast<float *>(chunk + a.lay.ks) + ((size_t)b * a.h + j) * a.nk;
    if (threadIdx.x == 0) qs_out[jq] = qs;
    if (threadIdx.x == 1 || threadIdx.x == 2) {
        const int gk = 2 * g + (threadIdx.x - 1);
        if (gk >= fk && gk <= lk) ks_out[gk - fk] = ks[threadIdx.x - 1];
    }
    if (jq == tq - 1) {                                  // slots past the touched groups
        const int t = threadIdx.x;
        if (b == a.B - 1 && j == a.h - 1) {
            // this CTA is the last writer of the chunk's scale sections: zero
            // their alignment padding so every chunk byte is defined
            const size_t nqs = (size_t)a.B * a.h * a.nq, nks = (size_t)a.B * a.h * a.nk;
            float *qsec = reinterpret_cast<float *>(chunk + a.lay.qs);
            float *ksec = reinterpret_cast<float *>(chunk + a.lay.ks);
            if (nqs + t < (a.lay.ks - a.lay.qs) / 4) qsec[nqs + t] = 0.0f;
            if (nks + t < (a.lay.bytes - a.lay.ks) / 4) ksec[nks + t] = 0.0f;
        }
        if (tq + t < a.nq) qs_out[tq + t] = __fdiv_rn(kEps, 127.0f);
        if (tk + t < a.nk) {
            float kam;
            if (a.fused) {
                kam = kEps;
                a.k_amax[amax_row + tk + t] = kam;
            } else {
                kam = a.k_amax[amax_row + tk + t];
            }
            ks_out[tk + t] = __fdiv_rn(kam, 127.0f);
        }
    }

    // ---- quantise from registers and store 8 bytes per row and tensor
    float vs[8];
    {
        const float4 *vp = reinterpret_cast<const float4 *>(a.v_scale + ((size_t)b * a.H + hh) * D + c * 8);
        const float4 v0 = vp[0], v1 = vp[1];
        vs[0] = v0.x; vs[1] = v0.y; vs[2] = v0.z; vs[3] = v0.w;
        vs[4] = v1.x; vs[5] = v1.y; vs[6] = v1.z; vs[7] = v1.w;
    }
    const size_t hD = (size_t)a.h * D;
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const int t = g * kGQ + i * RL + rl;
        if (t >= row0 && t < row0 + L) {
            const size_t o = ((size_t)b * L + (t - row0)) * hD + (size_t)j * D + c * 8;
            float f[8];
            int cq[8];
            to_f32x8<DT>(qv[i], f);
#pragma unroll
            for (int x = 0; x < 8; ++x) cq[x] = int8_code(__fdiv_rn(f[x], qs));
            *reinterpret_cast<uint2 *>(chunk + a.lay.q + o) =
                make_uint2(pack4(cq[0], cq[1], cq[2], cq[3]), pack4(cq[4], cq[5], cq[6], cq[7]));
            const float ksr = i < IT / 2 ? ks[0] : ks[1];
            to_f32x8<DT>(kv[i], f);
#pragma unroll
            for (int x = 0; x < 8; ++x) cq[x] = int8_code(__fdiv_rn(__fsub_rn(f[x], m[x]), ksr));
            *reinterpret_cast<uint2 *>(chunk + a.lay.k + o) =
                make_uint2(pack4(cq[0], cq[1], cq[2], cq[3]), pack4(cq[4], cq[5], cq[6], cq[7]));
            to_f32x8<DT>(vv[i], f);
            uint32_t w[4];
#pragma unroll
            for (int x = 0; x < 4; ++x)
                w[x] = e4m3x2(__fdiv_rn(f[2 * x], vs[2 * x]), __fdiv_rn(f[2 * x + 1], vs[2 * x + 1]));
            *reinterpret_cast<uint2 *>(chunk + a.lay.v + o) =
                make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
        }
    }
}

}  // namespace ulp

using namespace ulp;

extern "C" int ulp_pack(const void *q, const void *k, const void *v, const void *k_mean, int dtype,
                        float *k_amax, const float *gathered_q_partial, const float *v_scale, int B,
                        int L, int H, int D, int rank, int world_size, int used_sequence, int fused,
                        uint8_t *send, int send_layout, int enable_pdl, ulp_stream_t stream)
{
    if (int s = check_common(dtype, B, L, H, D, rank, world_size, used_sequence, enable_pdl)) return s;
    if (fused != 0 && fused != 1) return fail(ULP_EINVAL, "pack: fused must be 0 or 1 (got %d)", fused);
    if (send_layout != ULP_SEND_SOURCE_MAJOR && send_layout != ULP_SEND_DEST_MAJOR)
        return fail(ULP_EINVAL, "pack: send_layout must be 0 or 1 (got %d)", send_layout);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(k_mean) || !aligned4(k_amax) ||
        !aligned4(gathered_q_partial) || !aligned16(v_scale) || !aligned16(send))
        return fail(ULP_EALIGN, "pack: q, k, v, k_mean, v_scale, send must be 16-byte aligned, "
                                "k_amax and gathered_q_partial 4-byte aligned");
    const int h = H / world_size;
    PackArgs a{(const uint16_t *)q, (const uint16_t *)k, (const uint16_t *)v, (const uint16_t *)k_mean,
               k_amax, gathered_q_partial, v_scale, send, chunk_layout(B, L, h, D),
               B, L, H, world_size, h, rank,
               used_sequence < 0 ? L * world_size : used_sequence, fused, send_layout,
               slots(L, kGQ), slots(L, kGK)};
    // A shard touches at least ceil(L/G) groups, so at most one slot per
    // (b, head) is untouched; the last slab's CTA writes it.
    const int nranks = rank == ULP_ALL_RANKS ? world_size : 1;
    const long long blocks = (long long)nranks * B * a.nq * H;
    if (blocks > INT_MAX) return fail(ULP_EINVAL, "pack: grid of %lld blocks", blocks);
    const cudaStream_t st = (cudaStream_t)stream;
    if (D == 128) {
        if (dtype == ULP_BF16) pack_kernel<128, ULP_BF16><<<(unsigned)blocks, 256, 0, st>>>(a);
        else pack_kernel<128, ULP_FP16><<<(unsigned)blocks, 256, 0, st>>>(a);
    } else {
        if (dtype == ULP_BF16) pack_kernel<64, ULP_BF16><<<(unsigned)blocks, 256, 0, st>>>(a);
        else pack_kernel<64, ULP_FP16><<<(unsigned)blocks, 256, 0, st>>>(a);
    }
    return check_launch("pack");
}
