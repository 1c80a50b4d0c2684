/*
 * smoe_synth.h -- libsmoe_synth.so: on-device generator of the benchmark's
 * synthetic bf16 weights.  It is input generation only (no part of the MoE
 * method) and mirrors bit_expert_weight_gb300/synth.py bit for bit.
 */
#ifndef SMOE_SYNTH_H
#define SMOE_SYNTH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Write elements start .. start+n-1 of the stream with 64-bit key `key` as
 * bf16 bit patterns into out (device, n uint16).  Element i:
 *   z  = (2 * sum of twelve 16-bit uniforms - 12*65535) * 2^-17  (exact fp32)
 *   v  = fl32(z * (outlier ? s_out : s_norm)), 0 if zero-marked
 *   out[i - start] = bf16 round-to-nearest-even of v
 * with outlier <=> low 32 bits of word 4i+3 < t_out and zero <=> high 32
 * bits < t_zero (a threshold above 0xFFFFFFFF marks every element).
 * Returns 0, -1 on bad arguments, -4 on a CUDA launch error. */
int smoe_synth_bf16(uint16_t *out, int64_t n, int64_t start, uint64_t key, float s_norm,
                    float s_out, uint64_t t_out, uint64_t t_zero, void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* SMOE_SYNTH_H */
