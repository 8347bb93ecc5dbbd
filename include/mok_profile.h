/*
 * mok_profile.h - optional timing hooks of libmok (no counterpart in the articles; used
 * by benchmarks to attribute time to the library's kernels inside a timed region).
 *
 * When enabled on a context, every kernel launch made by later mok_plan / mok_moe_fwd /
 * mok_moe_bwd calls is bracketed by two CUDA events recorded on the launch stream, and
 * the forward megakernel stamps its phases per CTA (%globaltimer) into a small device
 * buffer that mok_profile_enable allocates once per context (64 launches x SMs x 64 bytes;
 * freed by mok_destroy). Recording adds a few microseconds per launch.
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
 * "<name> <launches> <total_ms>\n", into buf (NUL-terminated, truncated to len), then
 * the megakernel's phases as "fwd_megakernel:<phase> <launches> <total_ms>" lines
 * (gather, gemm, gemm_spread, combine, total; measured from the kernel's first CTA start).
 * *total_launches receives the number of kernel launches recorded. Records are cleared.
 * Returns MOK_ERR_CUDA if enabling could not allocate the stamp buffer. */
mok_status mok_profile_report(mok_ctx_t ctx, char* buf, size_t len, int* total_launches);

#ifdef __cplusplus
}
#endif
#endif /* MOK_PROFILE_H_ */
