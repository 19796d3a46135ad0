// unpack_for_sage (page "flashinfer.comm._ulysses_lowp.unpack_for_sage"):
// source-major chunks -> INT8 Q/K [B, S, h, D], FP8 V transposed to
// [B, D, h, ceil(S/64)*64] with a zero tail, fp32 scales [B, h, width].
//
// One launch, three block roles:
//  - V: each warp transposes a 128-row x 64-byte tile of the [S, h*D] V
//    matrix entirely in registers (16 x 16-byte loads, a 16 x 16 byte
//    transpose with byte permutes, 16 x 16-byte stores): loads are 64-byte
//    row segments, stores 128-byte row segments of v8.
//  - Q/K: each (source, batch) block of L*h*D bytes is one contiguous run on
//    both sides; blocks copy 32 KiB pieces, 16 vectors of 16 bytes in flight
//    per thread.
//  - scales: one thread per output slot.
#include "ulp_unpack.cuh"

namespace ulp {

template <int D>
__global__ void __launch_bounds__(kUnpackThreads) unpack_kernel(UnpackArgs a)
{
    pdl_trigger();
    pdl_wait();
    unpack_unit<D>(a, blockIdx.x, threadIdx.x);
}

int unpack_setup(UnpackArgs &a, long long &blocks, const uint8_t *recv, int B, int L, int h, int D,
                 int world_size, int aligned, int scale_sequence, int q_group, int8_t *q8, int8_t *k8,
                 uint8_t *v8, float *q_scale, float *k_scale, int num_dests)
{
    if (int s = check_world(world_size)) return s;
    if (int s = check_q_group(q_group, "unpack")) return s;
    if (B < 1 || L < 1 || h < 1) return fail(ULP_EINVAL, "unpack: B, L, h must be positive (%d, %d, %d)", B, L, h);
    if (D != 64 && D != 128) return fail(ULP_EINVAL, "unpack: head_dim must be 64 or 128 (got %d)", D);
    if (num_dests < 1) return fail(ULP_EINVAL, "unpack: num_dests must be >= 1 (got %d)", num_dests);
    if (aligned < -1 || aligned > 1) return fail(ULP_EINVAL, "unpack: aligned must be -1, 0 or 1");
    if (aligned == 1 && L % 128 != 0)
        return fail(ULP_EINVAL, "unpack: aligned=True requires local_sequence %% 128 == 0 (L = %d)", L);
    if ((long long)L * world_size > INT_MAX / 2) return fail(ULP_EINVAL, "unpack: sequence too long");
    const int S = L * world_size;
    if (scale_sequence != -1 && (scale_sequence < 1 || scale_sequence > S))
        return fail(ULP_EINVAL, "unpack: scale_sequence %d outside [1, %d]", scale_sequence, S);
    if (!aligned16(recv) || !aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned4(q_scale) ||
        !aligned4(k_scale))
        return fail(ULP_EALIGN, "unpack: recv, q8, k8, v8 must be 16-byte aligned, scales 4-byte aligned");

    a = UnpackArgs{};
    a.recv = recv; a.q8 = q8; a.k8 = k8; a.v8 = v8; a.qs = q_scale; a.ks = k_scale;
    a.lay = chunk_layout(B, L, h, D, q_group);
    a.gq = q_group;
    a.B = B; a.L = L; a.h = h; a.P = world_size; a.S = S; a.Spad = (S + 63) / 64 * 64;
    const int n = scale_sequence < 0 ? S : scale_sequence;
    a.wq = (n + q_group - 1) / q_group;
    a.wk = (n + kGK - 1) / kGK;
    a.nq = slots(L, q_group);
    a.nk = slots(L, kGK);
    a.nd = num_dests;
    a.TT = (a.Spad + 127) / 128;
    a.CC = h * D / 64;
    a.nVtiles = (long long)num_dests * B * a.TT * a.CC;
    a.nVblk = (a.nVtiles + 3) / 4;
    a.pieces = ((long long)L * h * D + kCopyPiece - 1) / kCopyPiece;
    a.nCblk = (long long)num_dests * 2 * B * world_size * a.pieces;
    a.nSblk = ((long long)num_dests * B * h * (a.wq + a.wk) + kUnpackThreads - 1) / kUnpackThreads;
    blocks = a.nVblk + a.nCblk + a.nSblk;
    if (blocks > INT_MAX) return fail(ULP_EINVAL, "unpack: grid of %lld blocks", blocks);
    return ULP_OK;
}

}  // namespace ulp

using namespace ulp;

extern "C" int ulp_unpack_for_sage(const uint8_t *recv, int B, int L, int h, int D, int world_size,
                                   int aligned, int scale_sequence, int q_group, int8_t *q8,
                                   int8_t *k8, uint8_t *v8, float *q_scale, float *k_scale,
                                   int num_dests, int enable_pdl, ulp_stream_t stream)
{
    if (enable_pdl < -1 || enable_pdl > 2) return fail(ULP_EINVAL, "unpack: enable_pdl must be -1, 0, 1 or 2");
    UnpackArgs a;
    long long blocks = 0;
    if (int s = unpack_setup(a, blocks, recv, B, L, h, D, world_size, aligned, scale_sequence, q_group, q8, k8,
                             v8, q_scale, k_scale, num_dests))
        return s;
    const cudaStream_t st = (cudaStream_t)stream;
    const bool pdl = pdl_enabled(enable_pdl);
    if (D == 128) launch_kernel(unpack_kernel<128>, dim3((unsigned)blocks), dim3(kUnpackThreads), st, pdl, a);
    else launch_kernel(unpack_kernel<64>, dim3((unsigned)blocks), dim3(kUnpackThreads), st, pdl, a);
    return check_launch("unpack_for_sage");
}
