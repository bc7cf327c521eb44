/*
 * ss_probe.h - measurement kernels of libss.so.
 *
 * The selective scan's roofline is the slower of its bytes at HBM bandwidth
 * and its exponentials at the special-function unit's rate. The HBM peak is
 * a measured copy bandwidth; this probe measures the second denominator on
 * the GPU at hand. Not part of the computation.
 */
#ifndef SS_PROBE_H
#define SS_PROBE_H

#include <stdint.h>

#include "ss.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Launches `blocks` CTAs of 256 threads; every thread runs 8 independent
 * chains of `iters` steps x <- 2^x - 1 with ex2.approx.ftz.f32 (one MUFU op
 * and one FADD per step) and writes one float to out[block * 256 + thread].
 * out: device buffer of blocks * 256 floats. Total MUFU ops:
 * blocks * 256 * 8 * iters. Time the launch with events on `stream`.
 */
ss_status ss_probe_mufu_ex2(float *out, int blocks, int iters, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SS_PROBE_H */
