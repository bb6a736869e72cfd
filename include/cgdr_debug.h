/*
 * cgdr_debug.h -- extra entry point of libcgdr_debug.so, the index-checking build of libcgdr.
 *
 * libcgdr_debug.so is built from the same sources as libcgdr.so with CGDR_DEBUG_CHECKS: every
 * global-memory access of its kernels (tensor rows, the state, o, the gate scalars, the
 * prefill workspace) is tested against the footprint of its tensor,
 * (B-1) sb + (T-1) st + (H-1) sh + d elements, computed on the host from the call's sizes and
 * strides.  A failed test stores CGDR_ERR_BOUNDS in the call's status words (args->status, and
 * the prefill workspace word) and skips the access; a skipped copy into shared memory is
 * zero-filled or its barrier phase is completed without data, so no wait is left hanging.
 * Accesses through TMA tensor maps are bounds-checked by the hardware already (rows past the
 * tensor read as zeros).  It exports everything cgdr.h declares, plus the call below, and has
 * no counterpart in the method's description: it is a tool for checking this library.
 */
#ifndef CGDR_DEBUG_H_
#define CGDR_DEBUG_H_

#include "cgdr.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * cgdr_decode with the footprint of o that the checks use shrunk by `o_shrink` elements (from
 * the end): the decode's last o stores then fail their check, are skipped and reported as
 * CGDR_ERR_BOUNDS in args->status, while every address stays inside the caller's buffer.  It
 * shows that the checks fire.  Returns CGDR_ERR_UNSUPPORTED from a build without the checks.
 */
cgdr_status cgdr_debug_decode_shrunk_o(const cgdr_args *args, int64_t o_shrink, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CGDR_DEBUG_H_ */
