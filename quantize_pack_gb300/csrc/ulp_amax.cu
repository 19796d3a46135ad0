// K grouped amax (page "k_grouped_amax"), the raw-K boundary min/max producer
// and the boundary derive (page "derive_k_boundary_amax"); also the optional
// debug check that the rows past used_sequence are zero.
//
// The first three are reductions over at most 64 (K) or q_group <= 128 (Q) rows of one head.
// Threads own one 16-byte column vector (8 channels) and a row lane; loads are
// 16-byte and coalesced along the head's D contiguous elements; the maxima are
// fp32 fmaxf trees (exact, so order-independent).
#include "ulp_minmax.cuh"

namespace ulp {

#define ULP_DISPATCH(D, DT, ...)                                                   \
    do {                                                                           \
        if ((D) == 128 && (DT) == ULP_BF16) { constexpr int kD = 128, kDT = ULP_BF16; __VA_ARGS__; } \
        else if ((D) == 128) { constexpr int kD = 128, kDT = ULP_FP16; __VA_ARGS__; } \
        else if ((DT) == ULP_BF16) { constexpr int kD = 64, kDT = ULP_BF16; __VA_ARGS__; } \
        else { constexpr int kD = 64, kDT = ULP_FP16; __VA_ARGS__; }               \
    } while (0)

struct AmaxArgs {
    const uint16_t *k;
    const uint16_t *k_mean;
    float *out;
    int B, L, H, P, rank, nslots, used;  // used = S when there is no padding
};

// One CTA per (rank, b, head, slot).  128 threads = RL row lanes x NV vectors.
template <int D, int DT>
__global__ void __launch_bounds__(128) k_grouped_amax_kernel(AmaxArgs a)
{
    constexpr int NV = D / 8, RL = 128 / NV, IT = kGK / RL;
    pdl_trigger();
    pdl_wait();
    int blk = blockIdx.x;
    const int j = blk % a.nslots; blk /= a.nslots;
    const int hh = blk % a.H; blk /= a.H;
    const int b = blk % a.B; blk /= a.B;
    const int rk = blk;                                   // index in the rank stack
    const int r = a.rank >= 0 ? a.rank : rk;
    const int S = a.P * a.L;
    const int fk = first_group(r, a.L, kGK), lk = last_group(r, a.L, kGK);
    const int g = fk + j;
    const int c = threadIdx.x % NV, rl = threadIdx.x / NV;

    float acc = -INFINITY;
    if (g <= lk) {
        const int row0 = r * a.L;
        const int lo = max(g * kGK, row0);
        int hi = min(g * kGK + kGK, row0 + a.L);
        if (a.used < S && g == (a.used - 1) / kGK) hi = min(hi, a.used);   // live rows only
        float m[8];
        to_f32x8<DT>(*reinterpret_cast<const uint4 *>(a.k_mean + ((size_t)b * a.H + hh) * D + c * 8), m);
        const size_t HD = (size_t)a.H * D;
        const uint16_t *base = a.k + (size_t)rk * a.B * a.L * HD + (size_t)b * a.L * HD + (size_t)hh * D + c * 8;
        uint4 v[IT];
#pragma unroll
        for (int i = 0; i < IT; ++i) {
            const int t = g * kGK + i * RL + rl;
            if (t >= lo && t < hi) v[i] = ld_stream(base + (size_t)(t - row0) * HD);
        }
#pragma unroll
        for (int i = 0; i < IT; ++i) {
            const int t = g * kGK + i * RL + rl;
            if (t >= lo && t < hi) {
                float f[8];
                to_f32x8<DT>(v[i], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaxf(acc, fabsf(__fsub_rn(f[e], m[e])));
            }
        }
    }
    __shared__ float red[4];
    acc = warp_max(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float v = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        a.out[(((size_t)rk * a.B + b) * a.H + hh) * a.nslots + j] = floor_eps(v);
    }
}

// One CTA per (rank, b, head, e): e = 0 first touched group, e = 1 last.
template <int D, int DT>
__global__ void __launch_bounds__(128) boundary_minmax_kernel(MinmaxArgs a)
{
    __shared__ MinmaxSmem<D> sm;
    pdl_trigger();
    pdl_wait();
    boundary_minmax_unit<D, DT>(a, blockIdx.x, threadIdx.x, sm, SyncCta{});
}

struct DeriveArgs {
    float *amax;
    const float *gathered;
    const uint16_t *k_mean;
    int B, L, H, P, rank, nslots;
};

// One CTA of D threads per (rank, b, head, e); thread d owns channel d.
template <int D, int DT>
__global__ void __launch_bounds__(128) derive_kernel(DeriveArgs a)
{
    pdl_trigger();
    pdl_wait();
    int blk = blockIdx.x;
    const int e = blk & 1; blk >>= 1;
    const int hh = blk % a.H; blk /= a.H;
    const int b = blk % a.B; blk /= a.B;
    const int rk = blk;
    const int r = a.rank >= 0 ? a.rank : rk;
    const int fk = first_group(r, a.L, kGK), lk = last_group(r, a.L, kGK);
    if (e == 1 && lk == fk) return;                  // one boundary group: e = 0 writes it
    const int g = e == 0 ? fk : lk;
    const int S = a.P * a.L;
    const int r_lo = (g * kGK) / a.L, r_hi = (min(g * kGK + kGK, S) - 1) / a.L;
    const int d = threadIdx.x;
    const uint16_t mb = a.k_mean[((size_t)b * a.H + hh) * D + d];
    const float m = DT == ULP_BF16 ? __uint_as_float((uint32_t)mb << 16)
                                   : __half2float(__ushort_as_half(mb));
    // max over ranks of floor(max over d) == floor(max over ranks and d): the
    // floor is monotone, so one reduction gives the same bits.
    float acc = -INFINITY;
    for (int rr = r_lo; rr <= r_hi; ++rr) {
        const int ee = g == first_group(rr, a.L, kGK) ? 0 : 1;
        const size_t base = ((((size_t)rr * a.B + b) * a.H + hh) * 2 + ee) * 2 * D;
        const float mn = a.gathered[base + d], mx = a.gathered[base + D + d];
        acc = fmaxf(acc, fmaxf(__fsub_rn(mx, m), __fsub_rn(m, mn)));
    }
    __shared__ float red[4];
    acc = warp_max(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float v = red[0];
        for (int w = 1; w < D / 32; ++w) v = fmaxf(v, red[w]);
        a.amax[(((size_t)rk * a.B + b) * a.H + hh) * a.nslots + (g - fk)] = floor_eps(v);
    }
}

static int grid_of(long long blocks, unsigned *out, const char *what)
{
    if (blocks < 1 || blocks > INT_MAX) return fail(ULP_EINVAL, "%s: grid of %lld blocks", what, blocks);
    *out = (unsigned)blocks;
    return ULP_OK;
}


// ------------------------------------------------- padding-row debug check

struct PadArgs {
    const uint16_t *t[3];          // q, k, v
    unsigned long long *count;
    int B, L, HD, rank, used;
};

// Elements of a 32-bit word (two 16-bit floats) whose value is not +-0.
__device__ __forceinline__ unsigned nonzero2(uint32_t w)
{
    return ((w & 0x7FFFu) != 0u) + ((w & 0x7FFF0000u) != 0u);
}

// blockIdx.y = shard slot * B + batch; threads stride over the 16-byte
// vectors of the shard's rows at or past `used` in the three tensors.
__global__ void __launch_bounds__(256) check_padding_kernel(PadArgs a)
{
    const int z = blockIdx.y;
    const int rk = z / a.B, b = z - rk * a.B;
    const int r = a.rank >= 0 ? a.rank : rk;
    const int first = max(0, a.used - r * a.L);        // the shard's first padding row
    if (first >= a.L) return;                          // whole CTA: none here
    const int nv = a.HD / 8;                           // vectors per row
    const long long total = (long long)(a.L - first) * nv;
    unsigned cnt = 0;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long row = first + i / nv;
        const size_t off = (((size_t)rk * a.B + b) * a.L + (size_t)row) * a.HD + (size_t)(i % nv) * 8;
#pragma unroll
        for (int x = 0; x < 3; ++x) {
            const uint4 w = *reinterpret_cast<const uint4 *>(a.t[x] + off);
            cnt += nonzero2(w.x) + nonzero2(w.y) + nonzero2(w.z) + nonzero2(w.w);
        }
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if ((threadIdx.x & 31) == 0 && cnt) atomicAdd(a.count, (unsigned long long)cnt);
}

}  // namespace ulp

using namespace ulp;

extern "C" {

int ulp_k_grouped_amax(const void *k, const void *k_mean, int dtype, int B, int L, int H, int D,
                       int rank, int world_size, int used_sequence, float *out, int enable_pdl,
                       ulp_stream_t stream)
{
    if (int s = check_common(dtype, B, L, H, D, rank, world_size, used_sequence, enable_pdl)) return s;
    if (!aligned16(k) || !aligned16(k_mean) || !aligned4(out))
        return fail(ULP_EALIGN, "k_grouped_amax: k, k_mean must be 16-byte aligned, out 4-byte aligned");
    const int nranks = rank == ULP_ALL_RANKS ? world_size : 1;
    AmaxArgs a{(const uint16_t *)k, (const uint16_t *)k_mean, out, B, L, H, world_size, rank,
               slots(L, kGK), used_sequence < 0 ? L * world_size : used_sequence};
    unsigned grid = 0;
    if (int s = grid_of((long long)nranks * B * H * a.nslots, &grid, "k_grouped_amax")) return s;
    const bool pdl = pdl_enabled(enable_pdl);
    ULP_DISPATCH(D, dtype, (launch_kernel(k_grouped_amax_kernel<kD, kDT>, dim3(grid), dim3(128), (cudaStream_t)stream, pdl, a)));
    return check_launch("k_grouped_amax");
}

int ulp_boundary_minmax(const void *k, const void *q, int dtype, int B, int L, int H, int D,
                        int rank, int world_size, int used_sequence, int q_group,
                        float *minmax, float *q_partial, ulp_stream_t stream)
{
    if (int s = check_common(dtype, B, L, H, D, rank, world_size, used_sequence, -1)) return s;
    if (int s = check_q_group(q_group, "boundary_minmax")) return s;
    if (!aligned16(k) || !aligned16(q) || !aligned4(minmax) || !aligned4(q_partial))
        return fail(ULP_EALIGN, "boundary_minmax: k, q must be 16-byte aligned, minmax, q_partial 4-byte aligned");
    const int nranks = rank == ULP_ALL_RANKS ? world_size : 1;
    MinmaxArgs a{(const uint16_t *)k, (const uint16_t *)q, minmax, q_partial, B, L, H, world_size, rank,
                 used_sequence < 0 ? L * world_size : used_sequence, q_group};
    unsigned grid = 0;
    if (int s = grid_of((long long)nranks * B * H * 2, &grid, "boundary_minmax")) return s;
    ULP_DISPATCH(D, dtype, (launch_kernel(boundary_minmax_kernel<kD, kDT>, dim3(grid), dim3(128), (cudaStream_t)stream, false, a)));
    return check_launch("boundary_minmax");
}

int ulp_derive_k_boundary_amax(float *grouped_amax, const float *gathered_minmax,
                               const void *k_mean, int dtype, int B, int H, int D, int rank,
                               int local_sequence, int world_size, ulp_stream_t stream)
{
    const int L = local_sequence;
    if (int s = check_common(dtype, B, L, H, D, rank, world_size, -1, -1)) return s;
    if (!aligned4(grouped_amax) || !aligned4(gathered_minmax) || !aligned16(k_mean))
        return fail(ULP_EALIGN, "derive_k_boundary_amax: k_mean must be 16-byte aligned, fp32 buffers 4-byte aligned");
    const int nranks = rank == ULP_ALL_RANKS ? world_size : 1;
    DeriveArgs a{grouped_amax, gathered_minmax, (const uint16_t *)k_mean, B, L, H, world_size, rank,
                 slots(L, kGK)};
    unsigned grid = 0;
    if (int s = grid_of((long long)nranks * B * H * 2, &grid, "derive_k_boundary_amax")) return s;
    ULP_DISPATCH(D, dtype, (launch_kernel(derive_kernel<kD, kDT>, dim3(grid), dim3(kD), (cudaStream_t)stream, false, a)));
    return check_launch("derive_k_boundary_amax");
}

int ulp_check_padding(const void *q, const void *k, const void *v, int dtype, int B, int L, int H, int D,
                      int rank, int world_size, int used_sequence, unsigned long long *count,
                      ulp_stream_t stream)
{
    if (int s = check_common(dtype, B, L, H, D, rank, world_size, used_sequence, -1)) return s;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || ((uintptr_t)count & 7u) != 0)
        return fail(ULP_EALIGN, "check_padding: q, k, v must be 16-byte aligned, count 8-byte aligned");
    const int used = used_sequence < 0 ? L * world_size : used_sequence;
    if (used == L * world_size) return ULP_OK;        // no padding rows
    const int nranks = rank == ULP_ALL_RANKS ? world_size : 1;
    if ((long long)nranks * B > 65535) return fail(ULP_EINVAL, "check_padding: ranks x batch above 65535");
    PadArgs a{{(const uint16_t *)q, (const uint16_t *)k, (const uint16_t *)v}, count, B, L, H * D,
              rank, used};
    const long long vecs = (long long)L * H * D / 8;  // at most one shard's rows
    const unsigned gx = (unsigned)std::min<long long>((vecs + 255) / 256, 4096);
    check_padding_kernel<<<dim3(gx, (unsigned)(nranks * B)), 256, 0, (cudaStream_t)stream>>>(a);
    return check_launch("check_padding");
}

}  // extern "C"
