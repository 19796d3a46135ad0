// Sender pack: INT8 Q/K with per-group fp32 scales and FP8 E4M3 V with the
// caller's V scale, written into the source-major chunks that the Ulysses
// all-to-all moves (page "unpack_for_sage": recv_u8 is the source-major
// buffer of chunks; Returns: the V scale remains with the caller).
//
// Work unit: a "slab" = the rows of one 128-row global group of one head on
// one rank, one CTA each (at D = 128 with q_group = 64, one CTA per 64-row
// half: one K group and one Q group).  Q and K rows are loaded once into
// registers, V rows into shared memory; the Q amax (of the slab's one 128-row
// Q group, or of the 64-row Q groups when q_group = 64) and the amax of the
// CTA's 64-row K groups are reduced in the CTA and the codes are written from
// the same registers.
// Boundary groups (the rank's first/last touched group) take their amax from
// the gathered partials (Q) or the derived slots (K), so every input byte
// crosses HBM once.  Quotients use a correctly rounded reciprocal and
// Markstein's correction (ulp_internal.cuh), so the codes are those of the
// IEEE quotient.
#include "ulp_pack.cuh"

namespace ulp {

template <int D, int DT, int GQ, bool FOLD>
__global__ void __launch_bounds__(pack_threads<D, GQ>(), 1024 / pack_threads<D, GQ>()) pack_kernel(PackArgs a)
{
    __shared__ __align__(16) PackSmem<D, GQ> sm;
    pdl_trigger();
    pack_block<D, DT, GQ, FOLD>(a, blockIdx.x, blockIdx.y, blockIdx.z, sm);
}

template <int D, int DT, int GQ>
static cudaError_t pack_launch(dim3 grid, cudaStream_t st, bool pdl, const PackArgs &a)
{
    // the derive is a separate instantiation: its warp-0 code would otherwise
    // cost the common kernel registers
    if (a.gathered) return launch_kernel(pack_kernel<D, DT, GQ, true>, grid, dim3(pack_threads<D, GQ>()), st, pdl, a);
    return launch_kernel(pack_kernel<D, DT, GQ, false>, grid, dim3(pack_threads<D, GQ>()), st, pdl, a);
}

}  // namespace ulp

using namespace ulp;

namespace ulp {

int pack_setup(PackArgs &a, dim3 &grid, const void *q, const void *k, const void *v, const void *k_mean,
               int dtype, float *k_amax, const float *gathered_q_partial, const float *gathered_minmax,
               const float *v_scale, int B, int L, int H, int D, int rank, int world_size, int used_sequence,
               int q_group, int fused, uint8_t *send, int send_layout)
{
    if (int s = check_common(dtype, B, L, H, D, rank, world_size, used_sequence, -1)) return s;
    if (int s = check_q_group(q_group, "pack")) return s;
    if (fused != 0 && fused != 1) return fail(ULP_EINVAL, "pack: fused must be 0 or 1 (got %d)", fused);
    if (send_layout != ULP_SEND_SOURCE_MAJOR && send_layout != ULP_SEND_DEST_MAJOR)
        return fail(ULP_EINVAL, "pack: send_layout must be 0 or 1 (got %d)", send_layout);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(k_mean) || !aligned4(k_amax) ||
        !aligned4(gathered_q_partial) || !aligned16(v_scale) || !aligned16(send) ||
        (gathered_minmax && !aligned4(gathered_minmax)))
        return fail(ULP_EALIGN, "pack: q, k, v, k_mean, v_scale, send must be 16-byte aligned, "
                                "k_amax, gathered_q_partial and gathered_minmax 4-byte aligned");
    const int h = H / world_size;
    a = PackArgs{(const uint16_t *)q, (const uint16_t *)k, (const uint16_t *)v, (const uint16_t *)k_mean,
                 k_amax, gathered_q_partial, gathered_minmax, v_scale, send, chunk_layout(B, L, h, D, q_group),
                 B, L, H, world_size, h, rank,
                 used_sequence < 0 ? L * world_size : used_sequence, fused, send_layout,
                 slots(L, q_group), slots(L, kGK)};
    // A shard touches at least ceil(L/G) groups, so at most one slot per
    // (b, head) is untouched; the CTA of the last slab's last rows writes it.
    const int nranks = rank == ULP_ALL_RANKS ? world_size : 1;
    const int nslab = slots(L, kSlab);
    const int halves = D == 128 && q_group == 64 ? 2 : 1;   // CTAs per slab
    if ((long long)nslab * halves > 65535 || (long long)nranks * B > 65535)
        return fail(ULP_EINVAL, "pack: grid too large (slabs %d, ranks x batch %lld)", nslab,
                    (long long)nranks * B);
    grid = dim3((unsigned)H, (unsigned)(nslab * halves), (unsigned)(nranks * B));
    return ULP_OK;
}

}  // namespace ulp

extern "C" int ulp_pack(const void *q, const void *k, const void *v, const void *k_mean, int dtype,
                        float *k_amax, const float *gathered_q_partial, const float *gathered_minmax,
                        const float *v_scale, int B, int L, int H, int D, int rank, int world_size,
                        int used_sequence, int q_group, int fused, uint8_t *send, int send_layout,
                        int enable_pdl, ulp_stream_t stream)
{
    if (enable_pdl < -1 || enable_pdl > 2) return fail(ULP_EINVAL, "enable_pdl must be -1, 0, 1 or 2 (got %d)", enable_pdl);
    PackArgs a;
    dim3 grid;
    if (int s = pack_setup(a, grid, q, k, v, k_mean, dtype, k_amax, gathered_q_partial, gathered_minmax, v_scale,
                           B, L, H, D, rank, world_size, used_sequence, q_group, fused, send, send_layout))
        return s;
    const cudaStream_t st = (cudaStream_t)stream;
    const bool pdl = pdl_enabled(enable_pdl);
    a.early = enable_pdl == 2;
#define ULP_PACK_LAUNCH(GQ_)                                                                  \
    do {                                                                                      \
        if (D == 128) {                                                                       \
            if (dtype == ULP_BF16) pack_launch<128, ULP_BF16, GQ_>(grid, st, pdl, a);          \
            else pack_launch<128, ULP_FP16, GQ_>(grid, st, pdl, a);                           \
        } else {                                                                              \
            if (dtype == ULP_BF16) pack_launch<64, ULP_BF16, GQ_>(grid, st, pdl, a);           \
            else pack_launch<64, ULP_FP16, GQ_>(grid, st, pdl, a);                            \
        }                                                                                     \
    } while (0)
    if (q_group == 128) ULP_PACK_LAUNCH(128);
    else ULP_PACK_LAUNCH(64);
#undef ULP_PACK_LAUNCH
    return check_launch("pack");
}
