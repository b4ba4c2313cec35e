/*
 * gca_synth.h -- device-side synthetic input generator (not part of GCA).
 *
 * The decode workload keeps a per-chunk K/V cache of 262144 chunks x 64
 * tokens x 12 heads x 64 dims (about 51.5 GB for K and V in bf16), too large
 * to generate on the host and copy.  This entry point fills a device buffer
 * with values from a stateless counter-based generator so that any part of
 * it can be regenerated bit-for-bit on the host:
 *
 *   h     = SplitMix64((seed << 56) ^ (tensor_id << 48) ^ (first_elem + i))
 *           (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *           generators", OOPSLA 2014: add 0x9E3779B97F4A7C15, then the
 *           two xor-shift-multiply rounds and a final xor-shift)
 *   value = (u0 + u1 + u2 + u3 - 14) / 32, u_k = (h >> 3k) & 7
 *
 * Every value is a multiple of 1/32 in [-14/32, 14/32], exact in bf16 and
 * fp32, with standard deviation about 0.143.
 */
#ifndef GCA_SYNTH_H_
#define GCA_SYNTH_H_

#include <stddef.h>
#include <stdint.h>

#include "gca.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Fill dst[0 .. n_elems) (device pointer, element type `dtype`) with the
 * values of elements first_elem .. first_elem + n_elems of the stream
 * (seed, tensor_id).  Asynchronous on `stream` (a cudaStream_t). */
gca_status_t gca_synth_fill_hash(void* dst, size_t n_elems, gca_dtype_t dtype, uint64_t seed,
                                 uint64_t tensor_id, uint64_t first_elem, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GCA_SYNTH_H_ */
