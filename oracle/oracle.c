/*
 * CPU oracle of the Ulysses low-precision quantize -> pack -> unpack path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg use this file.  It shares no code, header, table or
 * constant generator with the CUDA library and includes nothing from it.
 *
 * Plain, scalar, single-threaded C11.  All floating point is IEEE binary32
 * with round-to-nearest-even, no contraction (built with -ffp-contract=off),
 * `/` is the IEEE division.  Each function follows the page it names:
 *
 *   "flashinfer.comm._ulysses_lowp.k_grouped_amax"         (k_grouped_amax)
 *   "flashinfer.comm._ulysses_lowp.derive_k_boundary_amax" (derive_k_boundary_amax)
 *   "flashinfer.comm._ulysses_lowp.unpack_for_sage"        (unpack_for_sage)
 *
 * The sender pack and the raw-K boundary min/max producer are not printed on
 * the pages; the oracle states the plainest reading the pages support
 * (each reading is listed next to the function that takes it).
 *
 * Notation: P ranks, rank r owns global rows [r*L, (r+1)*L), S = P*L,
 * h = H/P heads per destination.  A global K group g is rows [64g, 64g+64),
 * a global Q group is rows [gq*g, gq*g+gq), gq = 128 (default) or 64.  A
 * rank's slot j of width G is global group first_G(r) + j,
 * first_G(r) = (r*L)/G.
 *
 * Parity status: every function here is pinned by the tests under tests/
 * (test_oracle_*.py).  Parity unpinned: the chunk byte layout, the axis
 * order of the gathered min/max buffer, the Q group width and the V-scale
 * shape are readings of this library (the pages do not fix them); they are
 * checked only indirectly, by the round-trip and P-invariance tests.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

#define GK 64  /* K group rows (k_grouped_amax: "slots(L,64)") */
/* Q group rows gq are an argument: 128 by default (reading: aligned=True <=>
 * L % 128 == 0 keeps Q groups on one rank), or 64, the variant whose Q groups
 * are the K groups (one scale width for both). */

/* The 1e-7 floor, as the binary32 value nearest to 1e-7. */
static const float EPS = 1e-7f;

/* ---------------------------------------------------------------- numbers */

/* bfloat16: the upper 16 bits of a binary32. */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* IEEE binary16 -> binary32, from the format definition (exact). */
float orc_f16_to_f32(uint16_t x)
{
    int sign = (x >> 15) & 1;
    int e = (x >> 10) & 31;
    int m = x & 1023;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static float in_f32(const uint16_t *p, size_t i, int dtype)
{
    return dtype == ORC_BF16 ? orc_bf16_to_f32(p[i]) : orc_f16_to_f32(p[i]);
}

static float maxf(float a, float b) { return a > b ? a : b; }
static float minf(float a, float b) { return a < b ? a : b; }

/* The 1e-7 floor of the pinned math (k_grouped_amax, derive_k_boundary_amax):
 * anything below 1e-7, -inf included, becomes 1e-7. */
static float floor_eps(float x) { return x < EPS ? EPS : x; }

/* Round to nearest integer, ties to even, written from the definition.
 * Valid for |y| < 2^23, which every caller guarantees. */
static float rne_int(float y)
{
    float n = floorf(y);
    float frac = y - n;            /* exact for |y| < 2^23 */
    if (frac > 0.5f) return n + 1.0f;
    if (frac < 0.5f) return n;
    return fmodf(n, 2.0f) == 0.0f ? n : n + 1.0f;
}

/* int8 code of a quotient y: round half to even, saturate to [-128, 127]. */
int8_t orc_int8_code(float y)
{
    if (y >= 128.0f) return 127;
    if (y <= -129.0f) return -128;
    float n = rne_int(y);
    if (n > 127.0f) return 127;
    if (n < -128.0f) return -128;
    return (int8_t)n;
}

/* FP8 E4M3 ("fn": no infinities, 0x7F/0xFF are NaN, largest finite 448)
 * encoder, round to nearest even, saturating to +-448 (satfinite).  The sign
 * of zero is kept.  Written from the format definition: subnormals are
 * m * 2^-9 (m = 1..7), normals (8 + m) * 2^(e-10) for e = 1..15 (m <= 6 when
 * e = 15).  Both the subnormal range and the first normal binade have the
 * step 2^-9, so one rule covers them. */
uint8_t orc_e4m3(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    float a = fabsf(x);
    if (a > 448.0f) return (uint8_t)(sign | 0x7E);

    int qexp;                                   /* step of the binade of a */
    if (a < 0.015625f) {                        /* below 2^-6 */
        qexp = -9;
    } else {
        int ex;
        frexpf(a, &ex);                         /* a = f * 2^ex, f in [0.5, 1) */
        qexp = (ex - 1) - 3;
    }
    float n = rne_int(ldexpf(a, -qexp));        /* exact scaling, then round */
    if (n == 0.0f) return sign;
    float val = ldexpf(n, qexp);                /* <= 448 since a <= 448 */
    if (val < 0.015625f) {                      /* subnormal code */
        return (uint8_t)(sign | (uint8_t)n);
    }
    int ex;
    frexpf(val, &ex);
    int E = ex - 1;                             /* val in [2^E, 2^(E+1)) */
    int mant = (int)ldexpf(val, -(E - 3)) - 8;  /* 0..7 */
    return (uint8_t)(sign | (uint8_t)((E + 7) << 3) | (uint8_t)mant);
}

/* Value of an E4M3 code (NaN for 0x7F / 0xFF). */
float orc_e4m3_decode(uint8_t c)
{
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    float v;
    if (e == 15 && m == 7) v = NAN;
    else if (e == 0) v = ldexpf((float)m, -9);
    else v = ldexpf((float)(8 + m), e - 10);
    return sign ? -v : v;
}

/* --------------------------------------------------------------- geometry */

/* slots(L, G): per-rank slot count.  Reading: ceil(L/G) + (L % G != 0), the
 * plainest bound written in (L, G) only; a shard of L rows can touch at most
 * that many global groups whatever its offset. */
int orc_slots(int L, int G) { return (L + G - 1) / G + (L % G != 0); }

static int first_group(int r, int L, int G) { return (int)(((int64_t)r * L) / G); }
static int last_group(int r, int L, int G) { return (int)(((int64_t)(r + 1) * L - 1) / G); }

static size_t a16(size_t x) { return (x + 15) & ~(size_t)15; }

/* Chunk (one source rank -> one destination rank) byte layout, in order:
 *   Q int8 [B, L, h, D] | K int8 [B, L, h, D] | V e4m3 [B, L, h, D] |
 *   q_scale f32 [B, h, slots(L,gq)] | k_scale f32 [B, h, slots(L,64)]
 * each section starting on a 16-byte boundary (a reading of this library:
 * the pages say only that recv_u8 is source-major [world_size, chunk_bytes]).
 * The alignment padding between sections is zero. */
void orc_chunk_layout(int B, int L, int h, int D, int gq, size_t *off_q, size_t *off_k,
                      size_t *off_v, size_t *off_qs, size_t *off_ks, size_t *chunk_bytes)
{
    size_t n = (size_t)B * L * h * D;
    *off_q = 0;
    *off_k = a16(n);
    *off_v = *off_k + a16(n);
    *off_qs = *off_v + a16(n);
    *off_ks = *off_qs + a16(sizeof(float) * (size_t)B * h * orc_slots(L, gq));
    *chunk_bytes = *off_ks + a16(sizeof(float) * (size_t)B * h * orc_slots(L, GK));
}

/* scale_widths(n): consumer scale-tensor widths for a sequence of n rows:
 * ceil(n/gq) Q slots and ceil(n/64) K slots. */
void orc_scale_widths(int n, int gq, int *q_width, int *k_width)
{
    *q_width = (n + gq - 1) / gq;
    *k_width = (n + GK - 1) / GK;
}

/* ------------------------------------------------------- k_mean_global */

/* k_mean_global production (the step before the path; page "k_grouped_amax",
 * k_mean_global parameter: the global K mean, rounded to the input dtype).
 * Reading of this library, one fixed order so that every implementation
 * gets the same bits:
 *   block sum  = fp32 sum of f32(K) over the live rows (t < used) of a
 *                rank-local 64-row block [64i, 64i+64) of rank r, rows in
 *                increasing order;
 *   partial_r  = fp64 pairwise sum of rank r's block sums: the blocks, padded
 *                with zeros to a power of two, are added in adjacent pairs,
 *                level by level ((b0 + b1) + (b2 + b3)) + ... (what rank r
 *                contributes to the all-reduce);
 *   total      = fp64 sum of the partials, ranks in increasing order;
 *   mean       = binary32 rounding of the fp64 quotient total / n, n = used
 *                (S when used < 0), then rounded to the dtype (nearest even).
 * Zero padding leaves the sums unchanged: no block sum or pair sum is -0.
 * k_all: [P, B, L, H, D] (every rank's shard); out: [B, H, D] dtype bits. */
static uint16_t f32_to_dtype_rne(float x, int dtype);

void orc_k_mean_global(const uint16_t *k_all, int dtype, int B, int L, int H, int D,
                       int world_size, int used, uint16_t *out)
{
    const int S = world_size * L;
    const int n = used >= 0 ? used : S;
    const int nb = (L + 63) / 64;
    int n2 = 1;
    while (n2 < nb) n2 *= 2;
    double *v = malloc(sizeof(double) * (size_t)n2);
    for (int b = 0; b < B; ++b)
        for (int hh = 0; hh < H; ++hh)
            for (int d = 0; d < D; ++d) {
                double total = 0.0;
                for (int r = 0; r < world_size; ++r) {
                    const uint16_t *k = k_all + (size_t)r * B * L * H * D;
                    for (int i = 0; i < n2; ++i) {
                        float block = 0.0f;
                        for (int tl = 64 * i; i < nb && tl < 64 * i + 64 && tl < L; ++tl) {
                            if (r * L + tl >= n) break;                    /* live rows only */
                            block += in_f32(k, (((size_t)b * L + tl) * H + hh) * D + d, dtype);
                        }
                        v[i] = (double)block;
                    }
                    for (int w = n2; w > 1; w /= 2)
                        for (int i = 0; i < w / 2; ++i) v[i] = v[2 * i] + v[2 * i + 1];
                    total += v[0];
                }
                const float mean = (float)(total / (double)n);
                out[((size_t)b * H + hh) * D + d] = f32_to_dtype_rne(mean, dtype);
            }
    free(v);
}

/* binary32 -> bfloat16 / binary16 bits, round to nearest even (finite input;
 * binary16 overflow gives infinity, underflow gives subnormals or zero). */
static uint16_t f32_to_dtype_rne(float x, int dtype)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if (dtype == ORC_BF16) {
        uint32_t lsb = (u >> 16) & 1u;
        return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
    }
    /* binary16: round |x| to a multiple of its binary16 step, from the definition */
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    float a = fabsf(x);
    if (a >= 65520.0f) return (uint16_t)(sign | 0x7C00u);   /* rounds to infinity */
    int ex;
    int qexp = a < 0x1p-14f ? -24 : (frexpf(a, &ex), (ex - 1) - 10);
    float m = rne_int(ldexpf(a, -qexp));                    /* exact scaling, then round */
    float v = ldexpf(m, qexp);
    if (v == 0.0f) return sign;
    if (v < 0x1p-14f) return (uint16_t)(sign | (uint16_t)m);  /* subnormal */
    frexpf(v, &ex);
    int E = ex - 1;
    int mant = (int)ldexpf(v, -(E - 10)) - 1024;
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)mant);
}

/* ------------------------------------------------------- k_grouped_amax */

/* k_grouped_amax, page "k_grouped_amax" (summary, used_sequence paragraph,
 * tail-padding paragraph):
 *   out[b,H,j] = max(1e-7, max over rows t of rank r in global group
 *                first_64(r)+j, and over d, of |rn(f32(K) - f32(m))|).
 * When used < S the slot of the partial live group (used-1)//64 is taken over
 * live rows t < used only; every other slot keeps the value over all its rows
 * (fully padded groups are deterministic don't-cares).  Slots past the groups
 * the rank touches hold 1e-7 (empty max, then the floor).
 * k: [B, L, H, D] of rank r; k_mean: [B, H, D]; out: [B, H, slots(L,64)].
 * used < 0 means None. */
void orc_k_grouped_amax(const uint16_t *k, const uint16_t *k_mean, int dtype, int B, int L,
                        int H, int D, int rank, int world_size, int used, float *out)
{
    const int S = world_size * L;
    const int nslots = orc_slots(L, GK);
    const int fk = first_group(rank, L, GK), lk = last_group(rank, L, GK);
    const int row0 = rank * L;
    const int correct = used >= 0 && used < S;
    const int gu = correct ? (used - 1) / GK : -1;
    for (int b = 0; b < B; ++b)
        for (int hh = 0; hh < H; ++hh)
            for (int j = 0; j < nslots; ++j) {
                int g = fk + j;
                float acc = -INFINITY;
                if (g <= lk) {
                    int lo = g * GK > row0 ? g * GK : row0;
                    int hi = g * GK + GK < row0 + L ? g * GK + GK : row0 + L;
                    if (g == gu && hi > used) hi = used;       /* live rows only */
                    for (int t = lo; t < hi; ++t)
                        for (int d = 0; d < D; ++d) {
                            float x = in_f32(k, (((size_t)b * L + (t - row0)) * H + hh) * D + d, dtype);
                            float m = in_f32(k_mean, ((size_t)b * H + hh) * D + d, dtype);
                            float c = x - m;
                            acc = maxf(acc, fabsf(c));
                        }
                }
                out[((size_t)b * H + hh) * nslots + j] = floor_eps(acc);
            }
}

/* ------------------------------------------------ boundary min/max producer */

/* Raw-K boundary min/max of rank r, the payload of "AllGather #1" (page
 * "derive_k_boundary_amax", Parameters: the gathered buffer has shape
 * [P, B, H, 2, 2, D]; a slice with only padding rows contributes min=+inf,
 * max=-inf).
 * Readings: axis 3 is e (0 = first touched K group, 1 = last), axis 4 is the
 * statistic (0 = min, 1 = max); only live rows t < used count; a rank that
 * touches one group writes it under both e; -0 is stored as +0.
 * Also the Q boundary partial amax qb[b, H, e] = max(1e-7, max |f32(Q)|) over
 * the rank's rows of its first (e=0) / last (e=1) gq-row Q group (raw Q, so
 * zero padding rows cannot raise it and used is not needed).
 * minmax: [B, H, 2, 2, D] for this rank; qb: [B, H, 2]. */
void orc_boundary_minmax(const uint16_t *k, const uint16_t *q, int dtype, int B, int L, int H,
                         int D, int rank, int world_size, int used, int gq, float *minmax,
                         float *qb)
{
    const int S = world_size * L;
    const int live = used >= 0 ? used : S;
    const int row0 = rank * L;
    for (int b = 0; b < B; ++b)
        for (int hh = 0; hh < H; ++hh)
            for (int e = 0; e < 2; ++e) {
                int g = e == 0 ? first_group(rank, L, GK) : last_group(rank, L, GK);
                int lo = g * GK > row0 ? g * GK : row0;
                int hi = g * GK + GK < row0 + L ? g * GK + GK : row0 + L;
                if (hi > live) hi = live;
                for (int d = 0; d < D; ++d) {
                    float mn = INFINITY, mx = -INFINITY;
                    for (int t = lo; t < hi; ++t) {
                        float x = in_f32(k, (((size_t)b * L + (t - row0)) * H + hh) * D + d, dtype);
                        if (x == 0.0f) x = 0.0f;   /* -0 -> +0 */
                        mn = minf(mn, x);
                        mx = maxf(mx, x);
                    }
                    size_t base = (((size_t)b * H + hh) * 2 + e) * 2 * D;
                    minmax[base + d] = mn;
                    minmax[base + D + d] = mx;
                }
                int g_q = e == 0 ? first_group(rank, L, gq) : last_group(rank, L, gq);
                int qlo = g_q * gq > row0 ? g_q * gq : row0;
                int qhi = g_q * gq + gq < row0 + L ? g_q * gq + gq : row0 + L;
                float acc = -INFINITY;
                for (int t = qlo; t < qhi; ++t)
                    for (int d = 0; d < D; ++d)
                        acc = maxf(acc, fabsf(in_f32(q, (((size_t)b * L + (t - row0)) * H + hh) * D + d, dtype)));
                qb[((size_t)b * H + hh) * 2 + e] = floor_eps(acc);
            }
}

/* ---------------------------------------------- derive_k_boundary_amax */

/* derive_k_boundary_amax, page "derive_k_boundary_amax" (formula and the
 * paragraph after it): for each of rank r's boundary K groups g (its first
 * and last touched group) and every rank r' touching g,
 *   contrib(r', g) = max(1e-7, max_d max(rn(maxK[r',g,d] - m[d]),
 *                                         rn(m[d] - minK[r',g,d])))
 * and slot g - first_64(r) becomes max over r' of contrib(r', g),
 * unconditionally.  grouped_amax: [B, H, slots(L,64)] of rank r, in place;
 * gathered: [P, B, H, 2, 2, D]. */
void orc_derive_k_boundary_amax(float *grouped_amax, const float *gathered, const uint16_t *k_mean,
                                int dtype, int B, int H, int D, int rank, int L, int world_size)
{
    const int S = world_size * L;
    const int nslots = orc_slots(L, GK);
    const int fk = first_group(rank, L, GK);
    for (int b = 0; b < B; ++b)
        for (int hh = 0; hh < H; ++hh)
            for (int e = 0; e < 2; ++e) {
                int g = e == 0 ? fk : last_group(rank, L, GK);
                int row_end = g * GK + GK < S ? g * GK + GK : S;
                int r_lo = (g * GK) / L, r_hi = (row_end - 1) / L;
                float best = -INFINITY;
                for (int rr = r_lo; rr <= r_hi; ++rr) {
                    int ee = g == first_group(rr, L, GK) ? 0 : 1;
                    size_t base = ((((size_t)rr * B + b) * H + hh) * 2 + ee) * 2 * D;
                    float acc = -INFINITY;
                    for (int d = 0; d < D; ++d) {
                        float m = in_f32(k_mean, ((size_t)b * H + hh) * D + d, dtype);
                        float up = gathered[base + D + d] - m;    /* rn(maxK - m) */
                        float dn = m - gathered[base + d];        /* rn(m - minK) */
                        acc = maxf(acc, maxf(up, dn));
                    }
                    best = maxf(best, floor_eps(acc));
                }
                grouped_amax[((size_t)b * H + hh) * nslots + (g - fk)] = best;
            }
}

/* ------------------------------------------------------------------ pack */

/* Sender pack of rank r (not printed on the pages; readings of this library):
 *  - Q amax of a gq-row global group g: max(1e-7, max |f32(Q)|) over all of
 *    g's rows, whichever ranks hold them.  A group inside rank r takes it from
 *    r's own rows; a boundary group (first/last touched) takes the max of the
 *    gathered partials qb of every rank touching g.  Slots past the touched
 *    groups hold the amax 1e-7.
 *  - K amax: the slot values of grouped_amax after derive_k_boundary_amax.
 *  - scale = rn(amax / 127) for Q and K; V scale is the caller's v_scale[b,H,d].
 *  - q8 = int8(rn(f32(q) / qs)), k8 = int8(rn(rn(f32(k) - f32(m)) / ks)),
 *    v8 = e4m3(rn(f32(v) / vs)), int8 = round half even, saturate.
 *  - chunk p (= global head H / h) receives heads [p*h, (p+1)*h), local head
 *    j = H % h, in the layout of orc_chunk_layout.
 * q, k, v: [B, L, H, D] of rank r; k_amax: [B, H, slots(L,64)];
 * gathered_qb: [P, B, H, 2]; v_scale: [B, H, D]; send: [P, chunk_bytes],
 * zero-filled here first so the alignment padding of every chunk is zero. */
void orc_pack(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *k_mean,
              int dtype, const float *k_amax, const float *gathered_qb, const float *v_scale,
              int B, int L, int H, int D, int rank, int world_size, int gq, uint8_t *send)
{
    const int P = world_size, S = P * L, h = H / P;
    const int row0 = rank * L;
    const int nq = orc_slots(L, gq), nk = orc_slots(L, GK);
    const int fq = first_group(rank, L, gq), lq = last_group(rank, L, gq);
    const int fk = first_group(rank, L, GK);
    size_t oq, ok, ov, oqs, oks, cb;
    orc_chunk_layout(B, L, h, D, gq, &oq, &ok, &ov, &oqs, &oks, &cb);
    memset(send, 0, (size_t)P * cb);

    float *qs = malloc(sizeof(float) * (size_t)nq);   /* per-slot scales of one (b, H) */
    float *ks = malloc(sizeof(float) * (size_t)nk);
    for (int b = 0; b < B; ++b)
        for (int hh = 0; hh < H; ++hh) {
            const int p = hh / h, j = hh % h;
            uint8_t *chunk = send + (size_t)p * cb;
            for (int jq = 0; jq < nq; ++jq) {
                int g = fq + jq;
                float amax;
                if (g > lq) {
                    amax = EPS;
                } else if (g == fq || g == lq) {
                    int row_end = g * gq + gq < S ? g * gq + gq : S;
                    amax = -INFINITY;
                    for (int rr = (g * gq) / L; rr <= (row_end - 1) / L; ++rr) {
                        int ee = g == first_group(rr, L, gq) ? 0 : 1;
                        amax = maxf(amax, gathered_qb[(((size_t)rr * B + b) * H + hh) * 2 + ee]);
                    }
                } else {
                    float acc = -INFINITY;
                    for (int t = g * gq; t < g * gq + gq; ++t)
                        for (int d = 0; d < D; ++d)
                            acc = maxf(acc, fabsf(in_f32(q, (((size_t)b * L + (t - row0)) * H + hh) * D + d, dtype)));
                    amax = floor_eps(acc);
                }
                qs[jq] = amax / 127.0f;
                float *dst = (float *)(chunk + oqs) + ((size_t)b * h + j) * nq + jq;
                *dst = qs[jq];
            }
            for (int jk = 0; jk < nk; ++jk) {
                ks[jk] = k_amax[((size_t)b * H + hh) * nk + jk] / 127.0f;
                float *dst = (float *)(chunk + oks) + ((size_t)b * h + j) * nk + jk;
                *dst = ks[jk];
            }
            for (int tl = 0; tl < L; ++tl) {
                int t = row0 + tl;
                float sq = qs[t / gq - fq], sk = ks[t / GK - fk];
                for (int d = 0; d < D; ++d) {
                    size_t src = (((size_t)b * L + tl) * H + hh) * D + d;
                    size_t dst = (((size_t)b * L + tl) * h + j) * D + d;
                    float xq = in_f32(q, src, dtype);
                    float xk = in_f32(k, src, dtype) - in_f32(k_mean, ((size_t)b * H + hh) * D + d, dtype);
                    float xv = in_f32(v, src, dtype);
                    chunk[oq + dst] = (uint8_t)orc_int8_code(xq / sq);
                    chunk[ok + dst] = (uint8_t)orc_int8_code(xk / sk);
                    chunk[ov + dst] = orc_e4m3(xv / v_scale[((size_t)b * H + hh) * D + d]);
                }
            }
        }
    free(qs);
    free(ks);
}

/* ------------------------------------------------------------- all-to-all */

/* The exchange of the chunks: recv[p][s] = send[s][p].  send and recv are
 * [P, P, chunk_bytes] (source-major per rank on both sides). */
void orc_alltoall(const uint8_t *send, uint8_t *recv, int world_size, size_t chunk_bytes)
{
    for (int s = 0; s < world_size; ++s)
        for (int p = 0; p < world_size; ++p)
            memcpy(recv + ((size_t)p * world_size + s) * chunk_bytes,
                   send + ((size_t)s * world_size + p) * chunk_bytes, chunk_bytes);
}

/* -------------------------------------------------------- unpack_for_sage */

/* unpack_for_sage, page "unpack_for_sage" (summary, Returns paragraphs):
 * recv: [P, chunk_bytes] source-major chunks of one destination.
 *   q8, k8 [B, S, h, D]:  q8[b, s*L + t, j, d] = chunk_s.Q[b, t, j, d]
 *   v8 [B, D, h, Spad], Spad = ceil(S/64)*64:
 *        v8[b, d, j, t] = chunk_{t/L}.V[b, t % L, j, d] for t < S, 0 for t >= S
 *   q_scale [B, h, Wq], k_scale [B, h, Wk] with (Wq, Wk) = scale_widths(n),
 *   n = scale_sequence (or S when scale_sequence < 0): slot g comes from the
 *   source holding the group's first row, s = (G*g)/L, at its slot
 *   g - first_G(s) (reading: the other toucher carries the same bytes). */
void orc_unpack_for_sage(const uint8_t *recv, int B, int L, int h, int D, int world_size,
                         int scale_sequence, int gq, int8_t *q8, int8_t *k8, uint8_t *v8,
                         float *q_scale, float *k_scale)
{
    const int P = world_size, S = P * L, Spad = (S + 63) / 64 * 64;
    const int nq = orc_slots(L, gq), nk = orc_slots(L, GK);
    size_t oq, ok, ov, oqs, oks, cb;
    orc_chunk_layout(B, L, h, D, gq, &oq, &ok, &ov, &oqs, &oks, &cb);
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < Spad; ++t)
            for (int j = 0; j < h; ++j)
                for (int d = 0; d < D; ++d) {
                    size_t vdst = (((size_t)b * D + d) * h + j) * Spad + t;
                    if (t >= S) {
                        v8[vdst] = 0;
                        continue;
                    }
                    int s = t / L, tl = t % L;
                    const uint8_t *chunk = recv + (size_t)s * cb;
                    size_t src = (((size_t)b * L + tl) * h + j) * D + d;
                    size_t dst = (((size_t)b * S + t) * h + j) * D + d;
                    q8[dst] = (int8_t)chunk[oq + src];
                    k8[dst] = (int8_t)chunk[ok + src];
                    v8[vdst] = chunk[ov + src];
                }
    int wq, wk;
    orc_scale_widths(scale_sequence >= 0 ? scale_sequence : S, gq, &wq, &wk);
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < h; ++j) {
            for (int g = 0; g < wq; ++g) {
                int s = (g * gq) / L;
                const float *src = (const float *)(recv + (size_t)s * cb + oqs);
                q_scale[((size_t)b * h + j) * wq + g] = src[((size_t)b * h + j) * nq + (g - first_group(s, L, gq))];
            }
            for (int g = 0; g < wk; ++g) {
                int s = (g * GK) / L;
                const float *src = (const float *)(recv + (size_t)s * cb + oks);
                k_scale[((size_t)b * h + j) * wk + g] = src[((size_t)b * h + j) * nk + (g - first_group(s, L, GK))];
            }
        }
}
