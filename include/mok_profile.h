/*
 * mok_profile.h - optional timing hooks of libmok (no counterpart in the articles; used
 * by benchmarks to attribute time to the library's kernels inside a timed region).
 *
 * When enabled on a context, every kernel launch made by later mok_plan / mok_moe_fwd /
 * mok_moe_bwd calls is bracketed by two CUDA events recorded on the launch stream.
 * Events are host-side objects; no device memory is allocated. Recording adds a few
 * microseconds per launch.
 */
#ifndef MOK_PROFILE_H_
#define MOK_PROFILE_H_

#include <stddef.h>

#include "mok.h"

#ifdef __cplusplus
extern "C" {
#endif

/* enable != 0: start recording (clears earlier records); 0: stop. */
mok_status mok_profile_enable(mok_ctx_t ctx, int enable);

/* Synchronise the recorded events and write one line per kernel name,
 * "<name> <launches> <total_ms>\n", into buf (NUL-terminated, truncated to len).
 * *total_launches receives the number of launches recorded. Records are cleared. */
mok_status mok_profile_report(mok_ctx_t ctx, char* buf, size_t len, int* total_launches);

#ifdef __cplusplus
}
#endif
#endif /* MOK_PROFILE_H_ */
