/*
 * gca_debug.h -- test-only fault injection for the device-side failure path.
 * Not part of GCA and not for production use.
 *
 * Every wait inside the library's kernels is bounded: when one runs out the
 * kernel records GCA_ERR_TIMEOUT in the status word, waits (with a bound) for
 * the copies it has already issued, and returns, so the GPU context stays
 * usable and gca_get_status() reports the error.  This entry point lets a
 * test take that path on purpose without a real hang or fault.
 */
#ifndef GCA_DEBUG_H_
#define GCA_DEBUG_H_

#include <stdint.h>

#include "gca.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gca_debug_stall_next_decode -- arm a stall for the next decode retrieval
 * launch (gca_decode_retrieve or gca_decode_retrieve_noalloc) made from the
 * calling host thread.  In that launch CTA 0 never issues (nor signals) the
 * first stage of its landmark stream, and every bounded wait of the kernel
 * gives up after `wait_ns` nanoseconds instead of the normal 2 s.  The warps
 * waiting for the withheld stage therefore run out, record GCA_ERR_TIMEOUT,
 * wait for the copies they did issue, and return; the other CTAs finish
 * normally.  The outputs of that one call are unspecified, and the next
 * gca_get_status() returns GCA_ERR_TIMEOUT.  The setting is consumed by that
 * launch (a call rejected before launching leaves it armed).
 *   wait_ns in [1000, 1000000000]; otherwise GCA_ERR_INVALID_ARG.
 */
gca_status_t gca_debug_stall_next_decode(uint64_t wait_ns);

#ifdef __cplusplus
}
#endif

#endif /* GCA_DEBUG_H_ */
