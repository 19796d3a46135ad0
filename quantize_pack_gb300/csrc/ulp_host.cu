// Host side of the ulp library: status reporting, argument checks, geometry
// queries and the emulated all-to-all.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>

#include "ulp_internal.cuh"

namespace ulp {

static thread_local std::string g_last_error;

// ------------------------------------------------------ emulated all-to-all

constexpr int kA2AThreads = 256;
constexpr int kA2AVecs = 4;   // 16-byte vectors in flight per thread

// recv[p][s] = send[s][p] over [P][P][chunk] buffers: blockIdx.y = p * P + s
// picks the destination chunk; the x blocks stride over its 16-byte vectors,
// each thread with kA2AVecs loads in flight before its stores.
__global__ void __launch_bounds__(kA2AThreads) alltoall_kernel(const uint4 *__restrict__ send,
                                                                 uint4 *__restrict__ recv, int P, size_t vecs)
{
    const int p = blockIdx.y / P, s = blockIdx.y - p * P;
    const uint4 *src = send + ((size_t)s * P + p) * vecs;
    uint4 *dst = recv + (size_t)blockIdx.y * vecs;
    const size_t step = (size_t)gridDim.x * kA2AThreads * kA2AVecs;
    for (size_t base = (size_t)blockIdx.x * kA2AThreads * kA2AVecs + threadIdx.x; base < vecs; base += step) {
        uint4 v[kA2AVecs];
#pragma unroll
        for (int i = 0; i < kA2AVecs; ++i) {
            const size_t j = base + (size_t)i * kA2AThreads;
            if (j < vecs) v[i] = ld_stream(src + j);
        }
#pragma unroll
        for (int i = 0; i < kA2AVecs; ++i) {
            const size_t j = base + (size_t)i * kA2AThreads;
            if (j < vecs) dst[j] = v[i];
        }
    }
}

int fail(int status, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

int check_launch(const char *what)
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ULP_ECUDA, "%s: %s", what, cudaGetErrorString(e));
    return ULP_OK;
}

EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool aligned16(const void *p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void *p) { return p != nullptr && ((uintptr_t)p & 3u) == 0; }

int check_world(int world_size)
{
    if (world_size != 2 && world_size != 4 && world_size != 6 && world_size != 8)
        return fail(ULP_EINVAL, "world_size must be 2, 4, 6 or 8 (got %d)", world_size);
    return ULP_OK;
}

int check_q_group(int q_group, const char *what)
{
    if (q_group != 64 && q_group != 128)
        return fail(ULP_EINVAL, "%s: q_group must be 64 or 128 (got %d)", what, q_group);
    return ULP_OK;
}

int check_common(int dtype, int B, int L, int H, int D, int rank, int world_size,
                 int used_sequence, int enable_pdl)
{
    if (dtype != ULP_BF16 && dtype != ULP_FP16)
        return fail(ULP_EDTYPE, "dtype must be ULP_BF16 or ULP_FP16 (got %d)", dtype);
    if (int s = check_world(world_size)) return s;
    if (B < 1 || L < 1 || H < 1) return fail(ULP_EINVAL, "B, L, H must be positive (%d, %d, %d)", B, L, H);
    if (D != 64 && D != 128) return fail(ULP_EINVAL, "head_dim must be 64 or 128 (got %d)", D);
    if (H % world_size != 0)
        return fail(ULP_EINVAL, "H (%d) must be a multiple of world_size (%d)", H, world_size);
    if (rank != ULP_ALL_RANKS && (rank < 0 || rank >= world_size))
        return fail(ULP_EINVAL, "rank %d outside [0, %d)", rank, world_size);
    if ((long long)L * world_size > INT_MAX / 2)
        return fail(ULP_EINVAL, "sequence length %lld too large", (long long)L * world_size);
    const int S = L * world_size;
    if (used_sequence != -1 && (used_sequence < 1 || used_sequence > S))
        return fail(ULP_EINVAL, "used_sequence %d outside [1, %d]", used_sequence, S);
    if (enable_pdl < -1 || enable_pdl > 2)
        return fail(ULP_EINVAL, "enable_pdl must be -1, 0, 1 or 2 (got %d)", enable_pdl);
    // every per-rank tensor must stay addressable with 64-bit offsets and every
    // grid within int range
    if ((double)B * S * H * D > 4.0e15) return fail(ULP_EINVAL, "tensor too large");
    return ULP_OK;
}

bool pdl_enabled(int enable_pdl)
{
    if (enable_pdl >= 1) return true;
    if (enable_pdl == 0) return false;
    // per device: 0 unknown, 1 no, 2 yes; every thread computes the same
    // value, so relaxed atomics suffice
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    int c = cached[dev].load(std::memory_order_relaxed);
    if (c == 0) {
        int major = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        c = major >= 9 ? 2 : 1;
        cached[dev].store(c, std::memory_order_relaxed);
    }
    return c == 2;
}

}  // namespace ulp

using namespace ulp;

extern "C" {

const char *ulp_last_error(void) { return g_last_error.c_str(); }

int ulp_slots(int local_sequence, int group)
{
    if (local_sequence < 1 || group < 1)
        return fail(ULP_EINVAL, "slots: L and group must be positive (%d, %d)", local_sequence, group);
    return slots(local_sequence, group);
}

int ulp_scale_widths(int n, int q_group, int *q_width, int *k_width)
{
    if (n < 1 || !q_width || !k_width) return fail(ULP_EINVAL, "scale_widths: n must be positive (%d)", n);
    if (int s = check_q_group(q_group, "scale_widths")) return s;
    *q_width = (n + q_group - 1) / q_group;
    *k_width = (n + kGK - 1) / kGK;
    return ULP_OK;
}

int ulp_chunk_offsets(int B, int L, int h, int D, int q_group, size_t offsets[5])
{
    if (B < 1 || L < 1 || h < 1 || D < 1 || !offsets)
        return fail(ULP_EINVAL, "chunk_offsets: sizes must be positive");
    if (int s = check_q_group(q_group, "chunk_offsets")) return s;
    ChunkLayout c = chunk_layout(B, L, h, D, q_group);
    offsets[0] = c.q;
    offsets[1] = c.k;
    offsets[2] = c.v;
    offsets[3] = c.qs;
    offsets[4] = c.ks;
    return ULP_OK;
}

int ulp_chunk_bytes(int B, int L, int h, int D, int q_group, size_t *chunk_bytes)
{
    if (B < 1 || L < 1 || h < 1 || D < 1 || !chunk_bytes)
        return fail(ULP_EINVAL, "chunk_bytes: sizes must be positive");
    if (int s = check_q_group(q_group, "chunk_bytes")) return s;
    *chunk_bytes = chunk_layout(B, L, h, D, q_group).bytes;
    return ULP_OK;
}

int ulp_alltoall_emulate(const uint8_t *send, uint8_t *recv, int world_size, size_t chunk_bytes,
                         ulp_stream_t stream)
{
    if (int s = check_world(world_size)) return s;
    if (chunk_bytes == 0 || chunk_bytes % 16 != 0)
        return fail(ULP_EINVAL, "chunk_bytes must be a positive multiple of 16");
    if (!aligned16(send) || !aligned16(recv)) return fail(ULP_EALIGN, "send/recv must be 16-byte aligned");
    if (send == recv) return fail(ULP_EINVAL, "alltoall: send and recv must not be the same buffer");
    const size_t vecs = chunk_bytes / 16;
    const int P = world_size;
    const size_t per_block = (size_t)kA2AThreads * kA2AVecs;   // 16 KB per block and pass
    const unsigned gx = (unsigned)std::min<size_t>(65535, (vecs + per_block - 1) / per_block);
    alltoall_kernel<<<dim3(gx, (unsigned)(P * P)), kA2AThreads, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const uint4 *>(send), reinterpret_cast<uint4 *>(recv), P, vecs);
    return check_launch("alltoall_emulate");
}

}  // extern "C"
