/* CPU oracle of the Ulysses low-precision quantize -> pack -> unpack path.
 * TEST INFRASTRUCTURE ONLY: see oracle.c for the definitions and readings. */
#ifndef ORACLE_H
#define ORACLE_H
#include <stddef.h>
#include <stdint.h>

enum { ORC_BF16 = 0, ORC_FP16 = 1 };

float orc_bf16_to_f32(uint16_t b);
float orc_f16_to_f32(uint16_t x);
int8_t orc_int8_code(float y);
uint8_t orc_e4m3(float x);
float orc_e4m3_decode(uint8_t c);

int orc_slots(int L, int G);
void orc_chunk_layout(int B, int L, int h, int D, int gq, size_t *off_q, size_t *off_k,
                      size_t *off_v, size_t *off_qs, size_t *off_ks, size_t *chunk_bytes);
void orc_scale_widths(int n, int gq, int *q_width, int *k_width);

void orc_k_mean_global(const uint16_t *k_all, int dtype, int B, int L, int H, int D,
                       int world_size, int used, uint16_t *out);
void orc_k_grouped_amax(const uint16_t *k, const uint16_t *k_mean, int dtype, int B, int L,
                        int H, int D, int rank, int world_size, int used, float *out);
void orc_boundary_minmax(const uint16_t *k, const uint16_t *q, int dtype, int B, int L, int H,
                         int D, int rank, int world_size, int used, int gq, float *minmax,
                         float *qb);
void orc_derive_k_boundary_amax(float *grouped_amax, const float *gathered, const uint16_t *k_mean,
                                int dtype, int B, int H, int D, int rank, int L, int world_size);
void orc_pack(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *k_mean,
              int dtype, const float *k_amax, const float *gathered_qb, const float *v_scale,
              int B, int L, int H, int D, int rank, int world_size, int gq, uint8_t *send);
void orc_alltoall(const uint8_t *send, uint8_t *recv, int world_size, size_t chunk_bytes);
void orc_unpack_for_sage(const uint8_t *recv, int B, int L, int h, int D, int world_size,
                         int scale_sequence, int gq, int8_t *q8, int8_t *k8, uint8_t *v8,
                         float *q_scale, float *k_scale);
#endif
