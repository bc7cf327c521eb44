/*
 * ss_testing.h - test hook of libss.so (not for production use).
 *
 * There is no counterpart on the pages: this exists so the test suite can
 * check the library's failure path without faulting or hanging a GPU.
 */
#ifndef SS_TESTING_H
#define SS_TESTING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * The next launch of ss_affine_scan, ss_selective_scan_fwd or
 * ss_selective_scan_bidir lets work unit `unit` (affine: tile index; S6:
 * sequence * chunks + chunk, chunked launches only) skip publishing its
 * look-back descriptors. Units that wait on it give up after the spin
 * timeout (ss_set_spin_timeout_ns), record SS_ERR_TIMEOUT in the workspace
 * and finish; the output of that launch is undefined. The request applies
 * to one launch and is then cleared. unit < 0 clears a pending request.
 */
void ss_testing_skip_publish_once(int64_t unit);

#ifdef __cplusplus
}
#endif

#endif /* SS_TESTING_H */
