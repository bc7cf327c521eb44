// Host-side interface of the time-parallel single-pass S6 forward (s6_tp.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "ss.h"
#include "ss_internal.h"

namespace ss {

// Launch shape of the time-parallel forward: G channels per warp, T steps
// per lane, W warps per CTA (rowW = G*W channels per CTA), R = (32/G)*T
// steps per block, nblk blocks per sequence, nsl B_t/C_t slots per block.
struct TPPlan {
    int G, T, W, rowW, S, R, dgroups, nblk, nsl;
    long long ctas;
    size_t slot_bytes, pack_bytes, smem;
};

// Fills `out` for the shape; false if (G, T, W) is not a built variant or
// the shape exceeds the kernel's limits.
bool tp_make_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int G, int T, int W,
                  TPPlan *out);
// The launch shape the planner takes for the shape on `sms` SMs; false when
// the channels give too few warps for the time-parallel pass.
bool tp_choose_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int sms,
                    TPPlan *out);
// CTAs of the plan's kernel that fit on one SM (0 if the query fails).
int tp_ctas_per_sm(const TPPlan &pl, int io_bf16);
// Two launches on `stream`: B_t / C_t packing into the workspace at
// `pack_offset` (pl.pack_bytes bytes, 256-byte aligned), then the scan. The
// workspace's 256-byte header receives device-detected errors.
ss_status tp_launch(const S6Args &a, const TPPlan &pl, void *workspace, size_t pack_offset,
                    cudaStream_t stream, unsigned long long timeout_ns);

}  // namespace ss
