// Host-side interface of the wavefront single-pass S6 forward (s6_ws.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "ss.h"
#include "ss_internal.h"

namespace ss {

// Launch shape: 32 channels per CTA, S warps (time slices of T steps each),
// R = S*T steps per block, nblk blocks per sequence.
struct WSPlan {
    int T, S, R, dgroups, nblk;
    long long ctas;
    size_t smem;
};

// Fills `out`; false if (T, S) is not a built variant or the shape exceeds
// the kernel's limits.
bool ws_make_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int T, int S,
                  WSPlan *out);
// The planner's wavefront shape for a forward call, or false when the
// channels give fewer than two CTAs per SM (the chunked kernel, which also
// splits L, is faster there).
bool ws_choose_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int sms,
                    WSPlan *out);
// One launch on `stream`; the workspace's 256-byte header receives
// device-detected errors (bounded waits on tile copies that ran out).
ss_status ws_launch(const S6Args &a, const WSPlan &pl, void *workspace, cudaStream_t stream,
                    unsigned long long timeout_ns);

}  // namespace ss
