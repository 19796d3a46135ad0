// One step of the emulated Ulysses group from one call: either the separate
// launches the path's entry points make (chained by programmatic launch), or
// a single cooperative launch that runs:
//  1. the raw-K boundary min/max and the Q boundary partials of every rank
//     (the gathered buffers of page "derive_k_boundary_amax");
//  2. the sender pack of every rank, with the boundary derive (page
//     "derive_k_boundary_amax", formula) and the exchange folded in: the K
//     amax per 64-row group (page "k_grouped_amax"), the scales, the INT8 /
//     E4M3 codes, written straight into each destination's source-major
//     chunks (page "unpack_for_sage": recv_u8);
//  3. unpack_for_sage of every destination.
// Each phase runs the per-block body of its own kernel (boundary_minmax_unit,
// pack_block, unpack_unit) on virtual block indices, so the outputs are those
// of the three-launch step, bit for bit.  Between the phases, every CTA waits
// at a grid-wide barrier.
//
// The barrier: a cooperative launch keeps every CTA resident.  Arrivals are
// counted in a caller-owned pair of 32-bit words [arrived, generation], zero
// before the first call.  The last CTA to arrive resets the count, then
// advances the generation (release); the others wait for the new generation
// (acquire).  So the pair is ready for the next barrier and the next call.
// A CTA waits at most kBarrierNs; on a timeout it records status 2 and
// returns, and its peers time out the same way, so no call hangs (the pair
// must then be zeroed again before the next call).
#include "ulp_minmax.cuh"
#include "ulp_pack.cuh"
#include "ulp_unpack.cuh"

#include <algorithm>
#include <atomic>

namespace ulp {

namespace {

constexpr uint64_t kBarrierNs = 1000000000ull;   // 1 s

struct StepArgs {
    MinmaxArgs mm;
    PackArgs pk;
    UnpackArgs up;
    unsigned *barrier;             // [2]: arrived, generation
    int *status;                   // 0, or 2 after a barrier timeout (may be null)
    int n_mm;                      // boundary units (rank, b, head, e)
    unsigned pk_x, pk_y, pk_z;     // pack grid
    long long n_up;                // unpack blocks
};

__device__ __forceinline__ uint64_t now_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Every CTA of the grid: true once all have arrived, false after a timeout.
__device__ __forceinline__ bool grid_barrier(unsigned *bar, int *status)
{
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned gen;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(gen) : "l"(bar + 1) : "memory");
        __threadfence();                         // the CTA's writes come before its arrival
        const unsigned arrived = atomicAdd(bar, 1u);
        int good = 1;
        if (arrived == gridDim.x - 1) {
            atomicExch(bar, 0u);                 // the last one: reset the count, then release
            __threadfence();
            asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(bar + 1), "r"(gen + 1u) : "memory");
        } else {
            const uint64_t t0 = now_ns();
            for (;;) {
                unsigned g;
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(g) : "l"(bar + 1) : "memory");
                if (g != gen) break;
                if (now_ns() - t0 > kBarrierNs) {
                    good = 0;
                    break;
                }
                __nanosleep(64);
            }
        }
        if (!good && status) atomicExch(status, 2);
        ok = good;
    }
    __syncthreads();
    return ok != 0;
}

// pack_threads<D, GQ>() threads: the pack body takes the whole CTA; the
// boundary and unpack bodies take 128-thread quarters of it.
template <int D, int DT, int GQ>
__global__ void __launch_bounds__(pack_threads<D, GQ>(), 1) group_step_kernel(StepArgs s)
{
    constexpr int NQ = pack_threads<D, GQ>() / 128;
    union Smem {
        PackSmem<D, GQ> pk;
        MinmaxSmem<D> mm[NQ];
    };
    __shared__ __align__(16) Smem sm;
    const int quarter = threadIdx.x >> 7, tid = threadIdx.x & 127;

    // 1. boundary min/max and Q partials (a named barrier per quarter)
    for (int u = blockIdx.x * NQ + quarter; u < s.n_mm; u += gridDim.x * NQ)
        boundary_minmax_unit<D, DT>(s.mm, u, tid, sm.mm[quarter], SyncNamed{1 + quarter});
    if (!grid_barrier(s.barrier, s.status)) return;

    // 2. pack, derive folded, exchange folded
    const long long npk = (long long)s.pk_x * s.pk_y * s.pk_z;
    for (long long u = blockIdx.x; u < npk; u += gridDim.x) {
        const unsigned bx = (unsigned)(u % s.pk_x);
        const unsigned by = (unsigned)((u / s.pk_x) % s.pk_y);
        const unsigned bz = (unsigned)(u / ((long long)s.pk_x * s.pk_y));
        pack_block<D, DT, GQ, true>(s.pk, bx, by, bz, sm.pk);
        __syncthreads();                       // the next slab reuses the shared memory
    }
    if (!grid_barrier(s.barrier, s.status)) return;

    // 3. unpack of every destination
    for (long long u = (long long)blockIdx.x * NQ + quarter; u < s.n_up; u += (long long)gridDim.x * NQ)
        unpack_unit<D>(s.up, u, tid);
}

template <int D, int DT, int GQ>
int step_launch(const StepArgs &s, cudaStream_t st)
{
    constexpr int NT = pack_threads<D, GQ>(), NQ = NT / 128;
    // resident CTAs per SM and SM count, per device (every thread computes
    // the same values, so relaxed atomics suffice)
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ULP_ECUDA, "group_step: cudaGetDevice: %s", cudaGetErrorString(e));
    int per_sm = dev >= 0 && dev < 64 ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (per_sm == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, group_step_kernel<D, DT, GQ>, NT, 0);
        if (e != cudaSuccess || per_sm < 1)
            return fail(ULP_ECUDA, "group_step: occupancy query: %s", cudaGetErrorString(e));
        if (dev >= 0 && dev < 64) cache[dev].store(per_sm, std::memory_order_relaxed);
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(ULP_ECUDA, "group_step: SM count: %s", cudaGetErrorString(e));
    const long long want = std::max({(long long)(s.n_mm + NQ - 1) / NQ,
                                     (long long)s.pk_x * s.pk_y * s.pk_z, (s.n_up + NQ - 1) / NQ, 1ll});
    const unsigned grid = (unsigned)std::min<long long>(want, (long long)per_sm * sms);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, group_step_kernel<D, DT, GQ>, s);
    if (e != cudaSuccess) return fail(ULP_ECUDA, "group_step: launch: %s", cudaGetErrorString(e));
    return ULP_OK;
}

}  // namespace

}  // namespace ulp

using namespace ulp;

extern "C" int ulp_group_step(const void *q, const void *k, const void *v, const void *k_mean, int dtype,
                              const float *v_scale, int B, int L, int H, int D, int world_size,
                              int used_sequence, int q_group, int aligned, int scale_sequence, float *minmax,
                              float *q_partial, float *k_amax, uint8_t *recv, int8_t *q8, int8_t *k8,
                              uint8_t *v8, float *q_scale, float *k_scale, int mode, unsigned *barrier,
                              int *status, ulp_stream_t stream)
{
    const bool coop = (mode & ULP_STEP_COOPERATIVE) != 0;
    const bool derive_separate = (mode & ULP_STEP_DERIVE_SEPARATE) != 0;
    if (mode < 0 || mode > (ULP_STEP_COOPERATIVE | ULP_STEP_DERIVE_SEPARATE | ULP_STEP_UNPACK_PDL))
        return fail(ULP_EINVAL, "group_step: unknown mode bits (%d)", mode);
    if (coop && mode != ULP_STEP_COOPERATIVE)
        return fail(ULP_EINVAL, "group_step: the cooperative launch takes no other mode bit (%d)", mode);
    StepArgs s{};
    dim3 grid;
    // pack's checks cover the inputs, the sizes, k_amax, the partials, the
    // min/max buffer and recv; unpack's cover its outputs.  Everything is
    // checked before the first launch.
    if (int r = pack_setup(s.pk, grid, q, k, v, k_mean, dtype, k_amax, q_partial, minmax, v_scale, B, L, H, D,
                           ULP_ALL_RANKS, world_size, used_sequence, q_group, 1, recv, ULP_SEND_DEST_MAJOR))
        return r;
    if (!minmax || !q_partial) return fail(ULP_EINVAL, "group_step: minmax and q_partial are required");
    if (int r = unpack_setup(s.up, s.n_up, recv, B, L, H / world_size, D, world_size, aligned, scale_sequence,
                             q_group, q8, k8, v8, q_scale, k_scale, world_size))
        return r;
    if (!coop) {
        // the separate launches: boundary min/max, [derive,] pack (reading
        // its inputs before its predecessor completes: neither writes them),
        // unpack -- each entry point as its own call would make them
        const cudaStream_t st = (cudaStream_t)stream;
        if (int r = ulp_boundary_minmax(k, q, dtype, B, L, H, D, ULP_ALL_RANKS, world_size, used_sequence, q_group,
                                        minmax, q_partial, st))
            return r;
        if (derive_separate) {
            if (int r = ulp_derive_k_boundary_amax(k_amax, minmax, k_mean, dtype, B, H, D, ULP_ALL_RANKS, L,
                                                   world_size, st))
                return r;
        }
        if (int r = ulp_pack(q, k, v, k_mean, dtype, k_amax, q_partial, derive_separate ? nullptr : minmax, v_scale,
                             B, L, H, D, ULP_ALL_RANKS, world_size, used_sequence, q_group, 1, recv,
                             ULP_SEND_DEST_MAJOR, 2, st))
            return r;
        return ulp_unpack_for_sage(recv, B, L, H / world_size, D, world_size, aligned, scale_sequence, q_group, q8,
                                   k8, v8, q_scale, k_scale, world_size, (mode & ULP_STEP_UNPACK_PDL) ? 1 : 0, st);
    }
    if (!barrier || !aligned4(barrier)) return fail(ULP_EALIGN, "group_step: barrier must be a 4-byte aligned pair");
    if (status && !aligned4(status)) return fail(ULP_EALIGN, "group_step: status must be 4-byte aligned");
    s.mm = MinmaxArgs{(const uint16_t *)k, (const uint16_t *)q, minmax, q_partial, B, L, H, world_size,
                      ULP_ALL_RANKS, s.pk.used, q_group};
    s.barrier = barrier;
    s.status = status;
    s.n_mm = world_size * B * H * 2;
    s.pk_x = grid.x;
    s.pk_y = grid.y;
    s.pk_z = grid.z;
    const cudaStream_t st = (cudaStream_t)stream;
    int r;
    if (D == 128) {
        if (q_group == 128) r = dtype == ULP_BF16 ? step_launch<128, ULP_BF16, 128>(s, st) : step_launch<128, ULP_FP16, 128>(s, st);
        else r = dtype == ULP_BF16 ? step_launch<128, ULP_BF16, 64>(s, st) : step_launch<128, ULP_FP16, 64>(s, st);
    } else {
        if (q_group == 128) r = dtype == ULP_BF16 ? step_launch<64, ULP_BF16, 128>(s, st) : step_launch<64, ULP_FP16, 128>(s, st);
        else r = dtype == ULP_BF16 ? step_launch<64, ULP_BF16, 64>(s, st) : step_launch<64, ULP_FP16, 64>(s, st);
    }
    if (r) return r;
    return check_launch("group_step");
}
