/*
 * Seeded synthetic inputs generated on the device (C ABI).  Not part of the MoE computation:
 * it only fills weight planes with the same numbers the host generator
 * (routed_expert_ffn_07_b300/inputs.py) produces, because the full-size planes (tens of GB) are
 * too large to draw on the host.
 *
 * Definition (SplitMix64 used as a counter-based stream; Steele, Lea and Flood, OOPSLA 2014):
 *   mix(z): z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
 *   key(seed, layer, tensor, expert) = mix(mix(mix(mix(seed) ^ (layer+1)*0x9E3779B97F4A7C15)
 *                                          ^ (tensor+1)*0xD1B54A32D192ED03) ^ (expert+1)*0x8CB92BA72F3D8DD7)
 *   draw i of a stream = mix(key + (i+1) * 0x9E3779B97F4A7C15)            (all mod 2^64)
 * Pointers are device pointers; calls are asynchronous on `stream` (a cudaStream_t as void*).
 * Return 0 on success, 1 for invalid arguments, 2 for a CUDA launch error.
 */
#ifndef ROUTED_MOE_B300_MOE_GEN_H
#define ROUTED_MOE_B300_MOE_GEN_H
#include <stddef.h>
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

/* n_experts consecutive int4 planes of bytes_per_expert bytes (a multiple of 8) each, for
 * experts expert0 .. expert0+n_experts-1: 64-bit word i of expert e's plane = draw i of
 * key(seed, layer, tensor, e), stored little-endian.  dst must be 8-byte aligned. */
int moe_gen_int4_planes(void* dst, uint64_t seed, int layer, int tensor, int expert0, int n_experts,
                        size_t bytes_per_expert, void* stream);

/* n_experts consecutive fp16 scale planes of scales_per_expert values each:
 * value i of expert e = fp16(0.005 + 0.015 * u), u = (draw_i >> 11) * 2^-53, computed in
 * double with round-to-nearest and no fused multiply-add, then rounded to fp16. */
int moe_gen_scale_planes(void* dst, uint64_t seed, int layer, int tensor, int expert0, int n_experts,
                         size_t scales_per_expert, void* stream);

#ifdef __cplusplus
}
#endif
#endif
