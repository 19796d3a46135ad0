/*
 * ulp.h -- C ABI of the GB300 (sm_103a) Ulysses low-precision quantize/pack path.
 *
 * The path feeds an INT8-QK / FP8-PV ("Sage") attention kernel after a Ulysses
 * all-to-all.  Per rank r of a Ulysses group of P ranks, rank r holds global
 * sequence rows [r*L, (r+1)*L) of Q, K, V [B, L, H, D]; after the exchange a
 * destination holds all S = P*L rows of h = H/P heads.  The entry points are:
 *
 *   ulp_k_mean_global           the step before the path: page "k_grouped_amax",
 *                               k_mean_global parameter (the global K mean)
 *   ulp_k_grouped_amax          page "flashinfer.comm._ulysses_lowp.k_grouped_amax"
 *   ulp_boundary_minmax         page "...derive_k_boundary_amax" (gathered_minmax parameter:
 *                               the raw-K boundary min/max every rank contributes)
 *   ulp_derive_k_boundary_amax  page "...derive_k_boundary_amax"
 *   ulp_pack                    the sender pack (INT8 Q/K, FP8 E4M3 V into source-major
 *                               chunks); page "...unpack_for_sage" (recv_u8 parameter,
 *                               Returns: the V scale stays with the caller)
 *   ulp_alltoall_emulate        the all-to-all of the chunks, as a device-local copy
 *   ulp_unpack_for_sage         page "...unpack_for_sage"
 *   ulp_group_step              boundary min/max + pack (exchange folded) + unpack of a
 *                               whole emulated group from one call (its launches, or one
 *                               cooperative launch)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer the caller owns; the library
 *    allocates nothing.  Across calls it keeps a thread-local last-error
 *    string, per-device lookups (launch occupancy, function attributes, the
 *    driver entry points it uses) and, for ulp_k_mean_global_noalloc, one
 *    fixed device array with its per-device address (see that entry point).
 *    Tensors are dense, row-major (C order).  Q, K, V,
 *    k_mean, v_scale, the chunk buffers and q8/k8/v8 must be 16-byte aligned;
 *    the other fp32 buffers (amax, min/max, partials, scales) 4-byte aligned.
 *  - `dtype` is ULP_BF16 or ULP_FP16 for Q/K/V/k_mean.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and runs asynchronously; a call returns once its launches are
 *    enqueued.
 *  - Return value: ULP_OK (0) or a negative status.  Arguments are validated
 *    before any launch, so a call that returns ULP_EINVAL / ULP_EDTYPE /
 *    ULP_EALIGN has enqueued nothing and left every output untouched.
 *    ULP_ECUDA reports a launch failure (cudaGetLastError after the launch).
 *    ulp_last_error() returns a message for the calling thread's last failure.
 *  - Optional integers use -1 for "None": used_sequence, scale_sequence,
 *    aligned (-1 None, 0 False, 1 True).
 *  - enable_pdl (Programmatic Dependent Launch, pages "k_grouped_amax" and
 *    "unpack_for_sage", Parameters): -1 = on where the device supports it
 *    (compute capability >= 9), 0 = off, 1 = on, 2 = on and, for ulp_pack
 *    only, the kernel may read q, k, v, k_mean and v_scale before the
 *    preceding kernel on the stream has completed (the caller guarantees that
 *    kernel does not write them).  With PDL a kernel may start while its
 *    predecessor finishes; every kernel of this library waits for its
 *    predecessor's completion before reading anything the predecessor may
 *    write and before its own first global write, so chains of these calls
 *    stay ordered.  ulp_boundary_minmax and ulp_derive_k_boundary_amax launch
 *    without PDL.
 *  - world_size is 2, 4, 6 or 8 (6: structurally supported, not validated by
 *    the method's authors); head_dim D is 64 or 128; H % world_size == 0.
 *  - rank is in [0, world_size), or ULP_ALL_RANKS: one launch covers every
 *    rank of an emulated Ulysses group held on one GPU.  Then each per-rank
 *    tensor is the stack of all ranks' tensors along a new leading axis of
 *    size world_size (written [P, ...] below).
 *
 *  - q_group is the Q group width G_Q in rows: 128 (the default width of this
 *    library; with aligned = 1, i.e. L % 128 == 0, no Q group crosses a rank)
 *    or 64 (the variant whose Q groups are the K groups, one scale width for
 *    both).  The pages print no Q width.  Every call that takes q_group must
 *    get the same value along one path; other values give ULP_EINVAL.
 *
 * Geometry (K groups of 64 rows, Q groups of q_group rows, both on the global
 * row grid): first_G(r) = (r*L)/G, last_G(r) = ((r+1)*L-1)/G; slot j of rank r is
 * global group first_G(r)+j; slots(L, G) = ceil(L/G) + (L % G != 0) bounds
 * the groups any rank touches.  Slots past the groups a rank touches hold
 * the floor value 1e-7 (amax) / rn(1e-7/127) (scale).
 *
 * Chunk layout (one source rank -> one destination; page "unpack_for_sage",
 * recv_u8 parameter: the receiver gets one source-major chunk per source; the
 * pages do not print the bytes inside a chunk, so this order is a reading of
 * this library), each section 16-byte aligned, in this order:
 *   Q int8 [B, L, h, D] | K int8 [B, L, h, D] | V e4m3 [B, L, h, D] |
 *   q_scale f32 [B, h, slots(L,q_group)] | k_scale f32 [B, h, slots(L,64)]
 * Chunk p of a source carries global heads [p*h, (p+1)*h).
 */
#ifndef ULP_H
#define ULP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void *ulp_stream_t; /* a cudaStream_t */

enum { ULP_BF16 = 0, ULP_FP16 = 1, ULP_F32 = 2 /* attention output only */ };

/* Precision of the attention's PV product (ulp_sage_attention). */
enum { ULP_PV_F16 = 0, ULP_PV_E4M3 = 1 };

enum {
    ULP_OK = 0,
    ULP_EINVAL = -1, /* argument outside its domain, inconsistent shapes, size overflow */
    ULP_EDTYPE = -2, /* dtype is neither ULP_BF16 nor ULP_FP16 */
    ULP_EALIGN = -3, /* a pointer is NULL or misaligned */
    ULP_ECUDA = -4   /* a CUDA launch or copy failed */
};

enum {
    ULP_SEND_SOURCE_MAJOR = 0, /* send[src][dst][chunk]: each rank's own send buffer */
    ULP_SEND_DEST_MAJOR = 1    /* send[dst][src][chunk]: the receivers' recv_u8 buffers */
};

#define ULP_ALL_RANKS (-1)

/* slots(L, G): per-rank slot count for groups of G rows (G = 64 for K, q_group
 * for Q): ceil(L/G) + (L % G != 0).  Page "k_grouped_amax" (Returns:
 * [B, H, slots(L, 64)]) names it without printing it; this is the plainest
 * bound in (L, G) alone.  Returns -1 (ULP_EINVAL) for L < 1 or G < 1. */
int ulp_slots(int local_sequence, int group);

/* scale_widths(n) of page "unpack_for_sage" (scale_sequence paragraph):
 * consumer scale widths for n rows, *q_width = ceil(n/q_group),
 * *k_width = ceil(n/64).  ULP_EINVAL for n < 1, a bad q_group or NULL
 * outputs. */
int ulp_scale_widths(int n, int q_group, int *q_width, int *k_width);

/* Bytes of one chunk (layout above) for batch B, shard length L, h heads per
 * destination, head dim D.  ULP_EINVAL for non-positive sizes. */
int ulp_chunk_bytes(int B, int L, int h, int D, int q_group, size_t *chunk_bytes);

/* Byte offsets of the five chunk sections: offsets[0..4] = Q, K, V,
 * q_scale, k_scale. */
int ulp_chunk_offsets(int B, int L, int h, int D, int q_group, size_t offsets[5]);

/* Bytes of the workspace ulp_k_mean_global needs: 8 * P * B * ceil(L/64) * H * D
 * (one fp64 tree node per 64-row block: the bound for every launch shape). */
int ulp_k_mean_workspace_bytes(int B, int L, int H, int D, int world_size, size_t *bytes);

/* k_mean_global production for an emulated Ulysses group (the global K mean
 * that page "k_grouped_amax" takes as k_mean_global: "rounded to the input
 * dtype").  One fixed summation order, so every implementation and launch
 * shape gives the same bits:
 *   block sum = fp32 sum of f32(K) over the live rows (global row < used) of
 *               a rank-local 64-row block, rows in increasing order;
 *   partial   = fp64 pairwise sum of a rank's block sums: zero-padded to a
 *               power of two, added in adjacent pairs level by level (the
 *               rank's all-reduce contribution); total = fp64 sum of the
 *               partials, ranks in order;
 *   k_mean    = dtype(binary32(total / used)), both roundings to nearest even.
 *   k          [P, B, L, H, D] dtype: every rank's shard
 *   workspace  device buffer of at least ulp_k_mean_workspace_bytes bytes
 *              (holds tree nodes; contents on return unspecified)
 *   k_mean     [B, H, D] dtype (output)
 * local_sequence is at most 262144 (ULP_EINVAL above). */
int ulp_k_mean_global(const void *k, int dtype, int B, int L, int H, int D, int world_size,
                      int used_sequence, void *workspace, size_t workspace_bytes, void *k_mean,
                      ulp_stream_t stream);

/* ulp_k_mean_global with the launch shape fixed: each thread of the first
 * kernel sums blocks_per_thread (1, 2, 4 or 8) consecutive 64-row blocks and
 * the lowest tree levels over them.  ulp_k_mean_global picks this number from
 * the shape and the device; every value gives the same bits (the summation
 * order above does not depend on it).  The pages have no counterpart; it
 * exists so that tests can check that every launch shape agrees.  ULP_EINVAL
 * for other values. */
int ulp_k_mean_global_grouped(const void *k, int dtype, int B, int L, int H, int D, int world_size,
                              int used_sequence, int blocks_per_thread, void *workspace,
                              size_t workspace_bytes, void *k_mean, ulp_stream_t stream);

/* ulp_k_mean_global without a workspace.  The pages have no counterpart of
 * this entry point; it exists for callers that cannot allocate device memory
 * for this call -- for example code inside a host framework whose caching
 * allocator already holds the device memory it manages, a plugin that may
 * only touch the tensors it is handed, or a latency-bound loop where a
 * cudaMalloc (which can synchronise the device) is not acceptable.
 * Same arguments and results as ulp_k_mean_global minus the workspace: the
 * tree nodes go to a fixed 8 MiB device array inside the library, which every
 * device that loads the library holds until the library is unloaded.
 *   - Shapes whose nodes need more than 8 MiB (8 * P * B * ceil(L/512) * H * D
 *     bytes) are rejected with ULP_EINVAL and a message; nothing is launched.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress, that device current) and caches it with the
 *     context it belongs to; make that first call before any stream capture
 *     on the device.  After a device reset (a new context, the module loaded
 *     again) the next call looks the address up again, and that call too
 *     should come before any capture.
 *   - Every call uses the same array and leaves its nodes there; each call
 *     writes every node it reads, so no clearing is needed.  Calls whose
 *     kernels can overlap on the GPU (other streams, other host threads) race
 *     on the array: order them on one stream or with events. */
int ulp_k_mean_global_noalloc(const void *k, int dtype, int B, int L, int H, int D, int world_size,
                              int used_sequence, void *k_mean, ulp_stream_t stream);

/* k_grouped_amax -- page "flashinfer.comm._ulysses_lowp.k_grouped_amax".
 * For each (b, head, slot j) of rank r:
 *   out[b,H,j] = max(1e-7, max |rn(f32(k[b,t,H,d]) - f32(k_mean[b,H,d]))|)
 * over the rank's rows t of global K group first_64(r)+j and all d.  With
 * used_sequence < S, the slot of the partial live group (used-1)/64 is taken
 * over live rows t < used only; all other slots (fully padded groups
 * included) keep the value over all their rows.  used_sequence = -1 or S
 * changes nothing.  Rows >= used must be zero-filled by the caller.
 *   k       [B, L, H, D] dtype     ([P, B, L, H, D] for ULP_ALL_RANKS)
 *   k_mean  [B, H, D] dtype: the global K mean rounded to dtype
 *   out     [B, H, slots(L,64)] fp32 ([P, B, H, slots] for ULP_ALL_RANKS) */
int ulp_k_grouped_amax(const void *k, const void *k_mean, int dtype, int B, int L, int H, int D,
                       int rank, int world_size, int used_sequence, float *out, int enable_pdl,
                       ulp_stream_t stream);

/* Raw-K boundary min/max of a rank -- the payload the page
 * "derive_k_boundary_amax" gathers ("AllGather #1 under stats protocol 2"):
 *   minmax[b,H,e,0,d] = min, minmax[b,H,e,1,d] = max of f32(k[b,t,H,d]) over
 *   the rank's live rows t < used of its first (e = 0) / last (e = 1) touched
 *   K group; +inf / -inf when that slice has no live row; -0 stored as +0; a
 *   rank touching one group writes it under both e.
 * Also the Q boundary partials (input of ulp_pack):
 *   q_partial[b,H,e] = max(1e-7, max |f32(q[b,t,H,d])|) over the rank's rows
 *   of its first (e = 0) / last (e = 1) touched q_group-row Q group.
 *   k, q       [B, L, H, D] dtype  ([P, ...] for ULP_ALL_RANKS)
 *   minmax     [B, H, 2, 2, D] fp32 ([P, B, H, 2, 2, D] = the gathered buffer
 *              in group-rank order, for ULP_ALL_RANKS)
 *   q_partial  [B, H, 2] fp32 ([P, B, H, 2] for ULP_ALL_RANKS) */
int ulp_boundary_minmax(const void *k, const void *q, int dtype, int B, int L, int H, int D,
                        int rank, int world_size, int used_sequence, int q_group,
                        float *minmax, float *q_partial, ulp_stream_t stream);

/* derive_k_boundary_amax -- page "flashinfer.comm._ulysses_lowp.derive_k_boundary_amax".
 * Overwrites, in place, rank r's boundary slots (its first and last touched K
 * group g) with max over every rank r' touching g of
 *   max(1e-7, max_d max(rn(maxK[r',g,d] - m[d]), rn(m[d] - minK[r',g,d])))
 * which equals the amax over the whole group (monotone rn subtraction).  Other
 * slots are left as they are.
 *   grouped_amax    [B, H, slots(L,64)] fp32, in place ([P, ...] for ULP_ALL_RANKS)
 *   gathered_minmax [P, B, H, 2, 2, D] fp32 (from ulp_boundary_minmax)
 *   k_mean          [B, H, D] dtype */
int ulp_derive_k_boundary_amax(float *grouped_amax, const float *gathered_minmax,
                               const void *k_mean, int dtype, int B, int H, int D, int rank,
                               int local_sequence, int world_size, ulp_stream_t stream);

/* Sender pack of rank r into its P chunks (layout above).  The pages print no
 * pack step: this is the producer of what page "unpack_for_sage" consumes
 * (recv_u8: source-major chunks of INT8 Q/K, FP8 E4M3 V and fp32 scales;
 * Returns: the V scale stays with the caller), with the scales of page
 * "k_grouped_amax" (Returns) and page "derive_k_boundary_amax".
 *   Q amax of q_group-row group g: max(1e-7, max |f32(q)|) over g's rows; for the
 *   rank's first/last touched Q group it is the max of gathered_q_partial over
 *   the ranks touching g, otherwise computed from the rank's own rows.
 *   K amax: k_amax slots.  The boundary slots (the rank's first/last touched
 *   K groups): with gathered_minmax given, derived in this call from it and
 *   k_mean by the formula of page "derive_k_boundary_amax" and written to
 *   k_amax (the values ulp_derive_k_boundary_amax writes); with
 *   gathered_minmax NULL, read from k_amax, which must then hold the derived
 *   values.  The other slots: fused = 0: read from k_amax (the output of
 *   ulp_k_grouped_amax); fused = 1: computed from the rank's own K rows in the
 *   same pass and written to k_amax (same values as fused = 0).
 *   scale = rn(amax / 127); q8 = sat8(rne(rn(f32(q) / qs))),
 *   k8 = sat8(rne(rn(rn(f32(k) - f32(m)) / ks))),
 *   v8 = e4m3_satfinite_rn(rn(f32(v) / v_scale[b,H,d])).
 *   q, k, v             [B, L, H, D] dtype ([P, ...] for ULP_ALL_RANKS)
 *   k_mean              [B, H, D] dtype
 *   k_amax              [B, H, slots(L,64)] fp32 ([P, ...] for ULP_ALL_RANKS)
 *   gathered_q_partial  [P, B, H, 2] fp32 (from ulp_boundary_minmax)
 *   gathered_minmax     [P, B, H, 2, 2, D] fp32 (from ulp_boundary_minmax), or NULL
 *   v_scale             [B, H, D] fp32, the caller's V scale (per global head);
 *                       positive and at least 2^-92 (smaller scales may code
 *                       inputs below 2^-102 with the wrong E4M3 value)
 *   send                ULP_SEND_SOURCE_MAJOR: [P, chunk_bytes] of this rank
 *                       ([P_src, P_dst, chunk_bytes] for ULP_ALL_RANKS);
 *                       ULP_SEND_DEST_MAJOR: [P_dst, P_src, chunk_bytes], the
 *                       receive buffers of every destination: chunk (r, p) is
 *                       written at [p][r] (the exchange folded into the stores). */
int ulp_pack(const void *q, const void *k, const void *v, const void *k_mean, int dtype,
             float *k_amax, const float *gathered_q_partial, const float *gathered_minmax,
             const float *v_scale, int B, int L, int H, int D, int rank, int world_size,
             int used_sequence, int q_group, int fused, uint8_t *send, int send_layout,
             int enable_pdl, ulp_stream_t stream);

/* The all-to-all, emulated on one GPU: recv[p][s] = send[s][p] for the
 * [P, P, chunk_bytes] buffers of all ranks (page "unpack_for_sage": recv_u8 is
 * the source-major buffer received by all-to-all), as one copy kernel.
 * chunk_bytes is a positive multiple of 16; send and recv must not overlap
 * (the same pointer gives ULP_EINVAL). */
int ulp_alltoall_emulate(const uint8_t *send, uint8_t *recv, int world_size, size_t chunk_bytes,
                         ulp_stream_t stream);

/* unpack_for_sage -- page "flashinfer.comm._ulysses_lowp.unpack_for_sage".
 * From recv_u8 [P, chunk_bytes] of one destination:
 *   q8, k8 [B, S, h, D] int8:   q8[b, s*L+t, j, d] = chunk_s.Q[b, t, j, d]
 *   v8 [B, D, h, Spad] e4m3, Spad = ceil(S/64)*64:
 *        v8[b, d, j, t] = chunk_{t/L}.V[b, t%L, j, d] for t < S, 0 for t >= S
 *   q_scale [B, h, Wq], k_scale [B, h, Wk] fp32, (Wq, Wk) = scale_widths(n),
 *        n = scale_sequence (S when -1); slot g is taken from the source that
 *        holds the group's first row.
 * aligned = 1 requires L % 128 == 0 (ULP_EINVAL otherwise); the values never
 * depend on it.  num_dests >= 1 destinations are unpacked in one launch:
 * recv is [num_dests, P, chunk_bytes] and every output gains a leading
 * num_dests axis (num_dests = 1 is the single-destination call). */
int ulp_unpack_for_sage(const uint8_t *recv, int B, int L, int h, int D, int world_size,
                        int aligned, int scale_sequence, int q_group, int8_t *q8, int8_t *k8,
                        uint8_t *v8, float *q_scale, float *k_scale, int num_dests,
                        int enable_pdl, ulp_stream_t stream);

/* Modes of ulp_group_step (bits). */
enum {
    ULP_STEP_COOPERATIVE = 1,       /* one cooperative launch (no other bit) */
    ULP_STEP_DERIVE_SEPARATE = 2,   /* separate launches: the boundary derive as its own launch */
    ULP_STEP_UNPACK_PDL = 4         /* separate launches: unpack as a programmatic dependent launch */
};

/* One step of an emulated Ulysses group (every rank, every destination) from
 * one call: ulp_boundary_minmax (ULP_ALL_RANKS), then ulp_pack with fused = 1
 * and ULP_SEND_DEST_MAJOR into recv (the all-to-all folded into the stores;
 * page "unpack_for_sage", recv_u8), with the boundary derive of page
 * "derive_k_boundary_amax" folded into pack (gathered_minmax given) or, with
 * ULP_STEP_DERIVE_SEPARATE, as ulp_derive_k_boundary_amax before it; then
 * ulp_unpack_for_sage of all P destinations (num_dests = world_size).  Every
 * output equals, bit for bit, that of those calls: minmax [P, B, H, 2, 2, D]
 * and q_partial [P, B, H, 2] as written by ulp_boundary_minmax, k_amax
 * [P, B, H, slots(L,64)] as by ulp_pack, recv [P_dst, P_src, chunk_bytes],
 * and the unpacked q8, k8, v8, q_scale, k_scale with a leading P axis.  All
 * arguments are checked before the first launch.
 *   mode without ULP_STEP_COOPERATIVE: the separate launches (three, or four
 *   with the derive), pack reading its inputs before its predecessor
 *   completes (enable_pdl = 2), unpack programmatic only with
 *   ULP_STEP_UNPACK_PDL.  One call instead of three or four, the same GPU
 *   work; barrier and status are ignored (may be NULL).
 *   mode = ULP_STEP_COOPERATIVE: one cooperative kernel runs the three phases
 *   (the derive folded) separated by grid-wide barriers.  It helps only where
 *   the host's launch rate bounds the step; in GPU time the chained launches
 *   are faster (each grid barrier costs about 2 us, and the fused kernel runs
 *   one CTA per SM).  `barrier`: two 32-bit words of device memory (4-byte
 *   aligned) that must be zero before the first call; every completed call
 *   leaves the count zero again.  Calls that may run concurrently (other
 *   streams) need their own pair.  Each barrier wait is bounded (1 s); on a
 *   timeout the kernel writes 2 to *status (a device int, or NULL) and returns
 *   early with outputs undefined, and the pair must be zeroed again before
 *   the next call.  The grid is capped by the device's occupancy so that
 *   every CTA is resident; a launch that still cannot be made gives
 *   ULP_ECUDA. */
int ulp_group_step(const void *q, const void *k, const void *v, const void *k_mean, int dtype,
                   const float *v_scale, int B, int L, int H, int D, int world_size, int used_sequence,
                   int q_group, int aligned, int scale_sequence, float *minmax, float *q_partial,
                   float *k_amax, uint8_t *recv, int8_t *q8, int8_t *k8, uint8_t *v8, float *q_scale,
                   float *k_scale, int mode, unsigned *barrier, int *status, ulp_stream_t stream);

/* Attention over the unpacked tensors of one destination -- the consumer the
 * page "unpack_for_sage" hands its outputs to (INT8 Q/K, FP8 E4M3 V, FP32
 * scales of width scale_widths(n) derived from the n rows attended over; the
 * V scale is not in the chunks, so the caller supplies it here, per that
 * page's Returns section).  The pages print no formula for it; this library's reading,
 * non-causal softmax attention over the live prefix t, u < n:
 *   Q[t] = q8[t] * q_scale[t / q_group], K[u] = k8[u] * k_scale[u / 64],
 *   V[u, d] = e4m3(v8[d, u]) * v_scale[d],
 *   O[b, t, j, :] = sum_u softmax_u(sm_scale * Q[t] . K[u]) V[u]
 * (K centred by the mean attends the same: q . m is one constant per query).
 * Computed on tensor cores with fp32 accumulation.  QK^T: fp16 operands, so
 * the integer logits are exact.  PV, by pv_precision:
 *   ULP_PV_F16:  P rounded to fp16 (relative 2^-11) and V widened to fp16
 *                (exactly); the denominator sums the fp32 weights, so rounding
 *                P moves the output by at most 2^-11 of max |V|;
 *   ULP_PV_E4M3: P rounded to E4M3 (rn; relative 2^-4 for weights >= 2^-6 of
 *                the running maximum, absolute 2^-10 below) and V read as the
 *                E4M3 bytes of v8 itself, at twice the tensor-core rate of
 *                fp16; the denominator still sums the fp32 weights, so the
 *                output moves by up to the weight-rounding error (a larger
 *                bound; see the tests).
 * A first kernel widens Q and K (and V for ULP_PV_F16) to fp16 in the
 * workspace (at least ulp_sage_attention_workspace_bytes bytes; contents on
 * return unspecified), the second runs the attention from it.
 *   q8, k8    [B, S, h, D] int8 (rows >= n are not read)
 *   v8        [B, D, h, Spad] E4M3 bytes, Spad = ceil(S/64)*64
 *   q_scale   [B, h, ceil(n/q_group)] fp32; k_scale [B, h, ceil(n/64)] fp32
 *   v_scale   [B, h, D] fp32: the caller's V scale of this destination's heads
 *   out       [B, n, h, D] of out_dtype (ULP_F32, ULP_BF16 or ULP_FP16)
 *   sm_scale  positive and finite (the usual choice is 1/sqrt(D))
 *   status    NULL, or a device int that the kernel sets to a non-zero code
 *             if a tensor-core product does not complete within about a
 *             second (the kernel then frees its tensor memory and returns
 *             without writing out); the caller clears it.
 * D is 64 or 128, 1 <= n <= S; pointers as for the other calls (16-byte
 * alignment for tensors, 4 bytes for the scales). */
int ulp_sage_attention(const int8_t *q8, const int8_t *k8, const uint8_t *v8, const float *q_scale,
                       const float *k_scale, const float *v_scale, int B, int S, int h, int D, int n,
                       int q_group, float sm_scale, void *workspace, size_t workspace_bytes,
                       void *out, int out_dtype, int pv_precision, int *status, ulp_stream_t stream);

/* Workspace bytes ulp_sage_attention needs: 6 * B * h * ceil(n/128)*128 * D
 * (Q, K, V in fp16 over the live prefix rounded up to 128 rows). */
int ulp_sage_attention_workspace_bytes(int B, int S, int h, int D, int n, size_t *bytes);

/* Debug check of a precondition of the path (page
 * "flashinfer.comm._ulysses_lowp.k_grouped_amax", Parameters: used_sequence):
 * the input rows past the live count are zero.  Counts the elements of Q, K
 * and V in global rows t >= used_sequence whose value is not +0 or -0, over
 * the shard of `rank` (or, for ULP_ALL_RANKS, over all P stacked shards), and
 * adds the count to *count, a device uint64 the caller zeroes.  Nothing is
 * launched when used_sequence is -1 or S.  -0 counts as zero: it moves no
 * amax and no code.
 *   q, k, v  [B, L, H, D] dtype ([P, B, L, H, D] for ULP_ALL_RANKS), 16-byte aligned
 *   count    device uint64, 8-byte aligned */
int ulp_check_padding(const void *q, const void *k, const void *v, int dtype, int B, int L, int H, int D,
                      int rank, int world_size, int used_sequence, unsigned long long *count,
                      ulp_stream_t stream);

/* Message of the calling thread's last failed call ("" if none). */
const char *ulp_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ULP_H */
