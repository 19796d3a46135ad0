// k_mean_global production: the global K mean of every (batch, head,
// channel), rounded to the input dtype (page "k_grouped_amax", k_mean_global
// parameter), for an emulated Ulysses group.  One fixed summation order, so
// the bits do not depend on the launch shape:
//   block sum = fp32 sum over the live rows of a rank-local 64-row block,
//               rows in increasing order;
//   partial   = fp64 pairwise sum of a rank's block sums (zero-padded to a
//               power of two, adjacent pairs level by level): the rank's
//               all-reduce contribution; total = fp64 sum over ranks in order;
//   mean      = binary32 rounding of total / used, then the dtype (RNE).
// Kernel A: a thread sums G consecutive blocks (G = 1, 2, 4 or 8, chosen
// from the shape so the grid fills whole waves) of 4 channels and the log2 G
// lowest tree levels over them, writing one fp64 node per group of G blocks
// to the workspace; kernel B (one thread per rank and channel) finishes each
// rank's tree and the rank sum.  Reads 2 bytes per K element: HBM-bound.
#include <atomic>

#include "ulp_internal.cuh"

namespace ulp {

constexpr int kMeanBlock = 64;        // rows per block sum
constexpr int kMeanThreads = 128;
constexpr int kMeanMaxNodes = 512;    // tree leaves kernel B accepts per rank (9 levels)

struct KMeanArgs {
    const uint16_t *k;   // [P, B, L, H, D]
    double *nodes;       // [P, B, ngrp, H, D]: tree nodes over G blocks each
    void *out;           // [B, H, D] dtype
    int B, L, H, D, P, nblk, ngrp, used, dtype;
};

// Kernel A: grid (ceil(H*D/4 / 128), ngrp, P * B); a thread owns 4 channels.
template <int DT, int G>
__global__ void __launch_bounds__(kMeanThreads) kmean_blocks_kernel(KMeanArgs a)
{
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "blocks per thread");
    constexpr int LV = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;   // in-thread tree levels
    pdl_wait();
    const int HD = a.H * a.D;
    const int vec = blockIdx.x * kMeanThreads + threadIdx.x;     // 4-channel vector of the row
    if (vec * 4 >= HD) return;
    const int grp = blockIdx.y;
    const int r = blockIdx.z / a.B, b = blockIdx.z - r * a.B;
    const int row_live = max(0, a.used - r * a.L);               // rank-local rows < this are live
    const uint16_t *src = a.k + ((size_t)r * a.B + b) * a.L * HD + (size_t)vec * 4;
    // The lowest levels of the rank's pairwise tree, built as the blocks
    // arrive: lv0 holds a finished block sum waiting for its right sibling
    // (fp32), st[l] a finished level-l node waiting for its sibling (fp64);
    // each node = left child + right child.
    float lv0[4];
    double st[LV > 1 ? LV - 1 : 1][4], top[4];
#pragma unroll 1
    for (int q = 0; q < G; ++q) {
        const int t0 = (grp * G + q) * kMeanBlock;
        const int t1 = min(min(t0 + kMeanBlock, a.L), row_live);
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int t = t0; t < t1; t += 16) {
            uint2 v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (t + i < t1) v[i] = __ldcs(reinterpret_cast<const uint2 *>(src + (size_t)(t + i) * HD));
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (t + i < t1) {
                    const float2 lo = pair_f32<DT>(v[i].x), hi = pair_f32<DT>(v[i].y);
                    s[0] = __fadd_rn(s[0], lo.x);                        // rows in order
                    s[1] = __fadd_rn(s[1], lo.y);
                    s[2] = __fadd_rn(s[2], hi.x);
                    s[3] = __fadd_rn(s[3], hi.y);
                }
            }
        }
        if (LV == 0) {
#pragma unroll
            for (int x = 0; x < 4; ++x) top[x] = (double)s[x];
        } else if (!(q & 1)) {
#pragma unroll
            for (int x = 0; x < 4; ++x) lv0[x] = s[x];
        } else {
            double node[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) node[x] = __dadd_rn((double)lv0[x], (double)s[x]);
            // node is at level 1; merge with finished left siblings above it
            bool done = false;
#pragma unroll
            for (int l = 1; l < LV; ++l) {
                if (!done) {
                    if (!((q >> l) & 1)) {
#pragma unroll
                        for (int x = 0; x < 4; ++x) st[l - 1][x] = node[x];
                        done = true;
                    } else {
#pragma unroll
                        for (int x = 0; x < 4; ++x) node[x] = __dadd_rn(st[l - 1][x], node[x]);
                    }
                }
            }
            if (q == G - 1) {
#pragma unroll
                for (int x = 0; x < 4; ++x) top[x] = node[x];
            }
        }
    }
    double *dst = a.nodes + (((size_t)r * a.B + b) * a.ngrp + grp) * HD + (size_t)vec * 4;
#pragma unroll
    for (int x = 0; x < 4; ++x) dst[x] = top[x];
    // kernel B may launch once every CTA has come this far (or exited): its
    // CTAs then take no slot from kernel A's later waves, and its launch
    // overlaps A's last CTAs (it waits for A's completion before reading)
    pdl_trigger();
}

// Kernel B: CTAs of 32 * P threads, thread (rank r, lane c) finishes rank r's
// tree for channel 32 * blockIdx.x + c (the nodes zero-padded to a power of
// two, added as they arrive with a carry stack of left children per level);
// the rank-0 thread then adds the ranks in order and rounds.
template <int DT>
__global__ void __launch_bounds__(256) kmean_finish_kernel(KMeanArgs a)
{
    pdl_trigger();
    pdl_wait();
    __shared__ double part[8][32];
    const int HD = a.H * a.D;
    const int c = threadIdx.x & 31, r = threadIdx.x >> 5;
    const long long idx = (long long)blockIdx.x * 32 + c;          // over B * HD
    const bool live = idx < (long long)a.B * HD;
    const int b = live ? (int)(idx / HD) : 0, ch = live ? (int)(idx - (long long)b * HD) : 0;
    int n2 = 1;
    while (n2 < a.ngrp) n2 *= 2;
    double st[9];                                      // carry stack, n2 <= 512 (checked on the host)
#pragma unroll
    for (int l = 0; l < 9; ++l) st[l] = 0.0;
    double root = 0.0;
    if (live) {
        const double *col = a.nodes + (((size_t)r * a.B + b) * a.ngrp) * HD + ch;
        // eight nodes loaded ahead of their additions
        for (int i0 = 0; i0 < n2; i0 += 8) {
            double xs[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) xs[u] = i0 + u < a.ngrp ? col[(size_t)(i0 + u) * HD] : 0.0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u;
                if (i < n2) {
                    double x = xs[u];
                    // x is a node at level 0; merge with finished left siblings
#pragma unroll
                    for (int l = 0; l < 9; ++l) {
                        if (!((i >> l) & 1)) {
                            st[l] = x;                 // a left child waits at level l
                            break;
                        }
                        x = __dadd_rn(st[l], x);       // left + right
                    }
                    if (i == n2 - 1) root = x;     // the last leaf completes the tree
                }
            }
        }
    }
    part[r][c] = root;
    __syncthreads();
    if (r == 0 && live) {
        double total = 0.0;
        for (int rr = 0; rr < a.P; ++rr) total = __dadd_rn(total, part[rr][c]);
        const float mean = __double2float_rn(__ddiv_rn(total, (double)a.used));
        uint16_t bits;
        if (DT == ULP_BF16) bits = __bfloat16_as_ushort(__float2bfloat16_rn(mean));
        else bits = __half_as_ushort(__float2half_rn(mean));
        static_cast<uint16_t *>(a.out)[idx] = bits;
    }
}

int kmean_check(int dtype, int B, int L, int H, int D, int world_size, int used_sequence)
{
    if (int s = check_common(dtype, B, L, H, D, ULP_ALL_RANKS, world_size, used_sequence, -1)) return s;
    return ULP_OK;
}

static int kmean_blocks(int L) { return (L + kMeanBlock - 1) / kMeanBlock; }
static int kmean_groups(int L, int G) { return (kmean_blocks(L) + G - 1) / G; }

// Tree nodes for the smallest group (G = 1), which bounds every G.
size_t kmean_workspace_bytes(int B, int L, int H, int D, int world_size)
{
    return sizeof(double) * (size_t)world_size * B * kmean_groups(L, 1) * H * D;
}

template <int DT>
static void launch_blocks(int G, dim3 grid, cudaStream_t st, const KMeanArgs &a)
{
    if (G == 1) launch_kernel(kmean_blocks_kernel<DT, 1>, grid, dim3(kMeanThreads), st, false, a);
    else if (G == 2) launch_kernel(kmean_blocks_kernel<DT, 2>, grid, dim3(kMeanThreads), st, false, a);
    else if (G == 4) launch_kernel(kmean_blocks_kernel<DT, 4>, grid, dim3(kMeanThreads), st, false, a);
    else launch_kernel(kmean_blocks_kernel<DT, 8>, grid, dim3(kMeanThreads), st, false, a);
}

// Resident kernel-A CTAs per SM for group G (cached per device and dtype).
static int resident_ctas(int G, int dtype)
{
    // every thread computes the same value, so relaxed atomics suffice
    static std::atomic<int> cache[64][2][4];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    const int gi = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3, di = dtype == ULP_BF16 ? 0 : 1;
    int c = cache[dev][di][gi].load(std::memory_order_relaxed);
    if (c == 0) {
        int n = 0;
        const void *f = nullptr;
        if (dtype == ULP_BF16)
            f = G == 1 ? (const void *)kmean_blocks_kernel<ULP_BF16, 1> : G == 2 ? (const void *)kmean_blocks_kernel<ULP_BF16, 2>
              : G == 4 ? (const void *)kmean_blocks_kernel<ULP_BF16, 4> : (const void *)kmean_blocks_kernel<ULP_BF16, 8>;
        else
            f = G == 1 ? (const void *)kmean_blocks_kernel<ULP_FP16, 1> : G == 2 ? (const void *)kmean_blocks_kernel<ULP_FP16, 2>
              : G == 4 ? (const void *)kmean_blocks_kernel<ULP_FP16, 4> : (const void *)kmean_blocks_kernel<ULP_FP16, 8>;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kMeanThreads, 0) != cudaSuccess || n < 1) n = 1;
        c = n;
        cache[dev][di][gi].store(c, std::memory_order_relaxed);
    }
    return c;
}

// Blocks per kernel-A thread: the largest G whose grid fills its waves best
// (the fraction of the last wave in use), among the G that keep kernel B's
// tree within kMeanMaxNodes leaves.  Every G gives the same bits.
static int choose_group(int L, int H, int D, int P, int B, int dtype)
{
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long gx = ((long long)H * D / 4 + kMeanThreads - 1) / kMeanThreads;
    int best = 8;
    double best_eff = -1.0;
    for (int G = 8; G >= 1; G /= 2) {
        if (kmean_groups(L, G) > kMeanMaxNodes) break;
        const double ctas = (double)gx * kmean_groups(L, G) * P * B;
        const double waves = ctas / ((double)resident_ctas(G, dtype) * sms);
        const double eff = waves / ceil(waves);
        if (eff > best_eff + 0.02) {               // a smaller G must fill clearly better
            best_eff = eff;
            best = G;
        }
    }
    return best;
}

// Both launches on `stream`; `nodes` holds the tree nodes for group size G.
int kmean_launch(const void *k, int dtype, int B, int L, int H, int D, int world_size,
                 int used_sequence, int G, double *nodes, void *k_mean, cudaStream_t stream)
{
    KMeanArgs a{(const uint16_t *)k, nodes, k_mean, B, L, H, D, world_size, kmean_blocks(L),
                kmean_groups(L, G), used_sequence < 0 ? L * world_size : used_sequence, dtype};
    if (a.ngrp > kMeanMaxNodes)
        return fail(ULP_EINVAL, "k_mean_global: local_sequence %d above the %d-row maximum for this group size", L,
                    kMeanMaxNodes * G * kMeanBlock);
    const long long vecs = (long long)H * D / 4;
    const long long gx = (vecs + kMeanThreads - 1) / kMeanThreads;
    if (gx > INT_MAX || (long long)world_size * B > 65535)
        return fail(ULP_EINVAL, "k_mean_global: grid too large");
    const dim3 grid_a((unsigned)gx, (unsigned)a.ngrp, (unsigned)(world_size * B));
    const long long nb = ((long long)B * H * D + 31) / 32;
    if (nb > INT_MAX) return fail(ULP_EINVAL, "k_mean_global: grid too large");
    // kernel B is a programmatic dependent launch of kernel A, whose CTAs
    // allow it only after their work
    if (dtype == ULP_BF16) {
        launch_blocks<ULP_BF16>(G, grid_a, stream, a);
        launch_kernel(kmean_finish_kernel<ULP_BF16>, dim3((unsigned)nb), dim3(32 * world_size), stream, true, a);
    } else {
        launch_blocks<ULP_FP16>(G, grid_a, stream, a);
        launch_kernel(kmean_finish_kernel<ULP_FP16>, dim3((unsigned)nb), dim3(32 * world_size), stream, true, a);
    }
    return check_launch("k_mean_global");
}

}  // namespace ulp

using namespace ulp;

extern "C" {

int ulp_k_mean_workspace_bytes(int B, int L, int H, int D, int world_size, size_t *bytes)
{
    if (int s = check_world(world_size)) return s;
    if (B < 1 || L < 1 || H < 1 || (D != 64 && D != 128) || !bytes)
        return fail(ULP_EINVAL, "k_mean_workspace_bytes: bad sizes");
    *bytes = kmean_workspace_bytes(B, L, H, D, world_size);
    return ULP_OK;
}

int ulp_k_mean_global(const void *k, int dtype, int B, int L, int H, int D, int world_size,
                      int used_sequence, void *workspace, size_t workspace_bytes, void *k_mean,
                      ulp_stream_t stream)
{
    if (int s = kmean_check(dtype, B, L, H, D, world_size, used_sequence)) return s;
    if (!aligned16(k) || !aligned16(workspace) || !aligned16(k_mean))
        return fail(ULP_EALIGN, "k_mean_global: k, workspace, k_mean must be 16-byte aligned");
    const size_t need = kmean_workspace_bytes(B, L, H, D, world_size);
    if (workspace_bytes < need)
        return fail(ULP_EINVAL, "k_mean_global: workspace of %zu bytes, %zu needed", workspace_bytes, need);
    const int G = choose_group(L, H, D, world_size, B, dtype);
    return kmean_launch(k, dtype, B, L, H, D, world_size, used_sequence, G, (double *)workspace, k_mean,
                        (cudaStream_t)stream);
}

int ulp_k_mean_global_grouped(const void *k, int dtype, int B, int L, int H, int D, int world_size,
                              int used_sequence, int blocks_per_thread, void *workspace,
                              size_t workspace_bytes, void *k_mean, ulp_stream_t stream)
{
    if (int s = kmean_check(dtype, B, L, H, D, world_size, used_sequence)) return s;
    const int G = blocks_per_thread;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(ULP_EINVAL, "k_mean_global_grouped: blocks_per_thread must be 1, 2, 4 or 8 (got %d)", G);
    if (!aligned16(k) || !aligned16(workspace) || !aligned16(k_mean))
        return fail(ULP_EALIGN, "k_mean_global: k, workspace, k_mean must be 16-byte aligned");
    const size_t need = kmean_workspace_bytes(B, L, H, D, world_size);
    if (workspace_bytes < need)
        return fail(ULP_EINVAL, "k_mean_global: workspace of %zu bytes, %zu needed", workspace_bytes, need);
    return kmean_launch(k, dtype, B, L, H, D, world_size, used_sequence, G, (double *)workspace, k_mean,
                        (cudaStream_t)stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// k_mean_global without any allocation by the caller or the library.
//
// Some callers cannot hand this library a workspace: a host framework whose
// caching allocator has already reserved the device memory it manages, a
// plugin that may only touch the tensors it is given, or a latency-bound
// loop where a cudaMalloc (which can synchronise the device) is not allowed.
// For them the tree nodes live in one fixed, file-scope device array instead.
// The array exists on every device that loads this library, for as long as
// the library stays loaded, whether or not this entry point is ever called.

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB of tree nodes
static __device__ __align__(256) unsigned char g_kmean_scratch[kNoAllocScratchBytes];

// Device address of g_kmean_scratch per device, with the context it was
// looked up in.  Host code must not use the array's name as an address: on
// the host it only stands in for the symbol.  A device reset destroys the
// context and the module with it; the next call finds another current
// context and looks the address up again.
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
std::mutex g_scratch_mutex;
void *g_scratch_addr[128];
CUcontext g_scratch_ctx[128];

CUcontext current_context()
{
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

int scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ulp::fail(ULP_ECUDA, "k_mean_global_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 128) return ulp::fail(ULP_EINVAL, "k_mean_global_noalloc: device %d out of range", dev);
    const CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev] || !ctx || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_kmean_scratch);    // with `dev` current (sets its context up if need be)
        if (e != cudaSuccess || !p)
            return ulp::fail(ULP_ECUDA, "k_mean_global_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = current_context();
    }
    *out = g_scratch_addr[dev];
    return ULP_OK;
}

}  // namespace

extern "C" int ulp_k_mean_global_noalloc(const void *k, int dtype, int B, int L, int H, int D,
                                         int world_size, int used_sequence, void *k_mean,
                                         ulp_stream_t stream)
{
    using namespace ulp;
    if (int s = kmean_check(dtype, B, L, H, D, world_size, used_sequence)) return s;
    if (!aligned16(k) || !aligned16(k_mean))
        return fail(ULP_EALIGN, "k_mean_global_noalloc: k and k_mean must be 16-byte aligned");
    // groups of 8 blocks: the smallest node array (8 * P * B * ceil(L/512) * H * D bytes)
    const size_t need = sizeof(double) * (size_t)world_size * B * ((L + 511) / 512) * H * D;
    if (need > kNoAllocScratchBytes)
        return fail(ULP_EINVAL,
                    "k_mean_global_noalloc: this shape needs %zu bytes of scratch, the fixed "
                    "array holds %zu; use ulp_k_mean_global with a workspace",
                    need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    if (int s = scratch_address(&scratch)) return s;
    // Every tree node kernel B reads is written by kernel A of the same call,
    // so the previous call's leftovers never need clearing.
    return kmean_launch(k, dtype, B, L, H, D, world_size, used_sequence, 8, (double *)scratch, k_mean,
                        (cudaStream_t)stream);
}
