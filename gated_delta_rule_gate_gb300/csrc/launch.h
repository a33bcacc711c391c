// launch.h -- host-side launchers of the CUDA kernels (internal to libgdn).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace gdn {

struct GateLaunch {
    int64_t n;
    int heads;
    int f16;
    const void *a;
    const float *dt_bias;
    const float *decay_scale;
    const void *b;
    void *decay_out;
    void *beta_out;
};

// Number of SMs of the current device (cached per device).
int sm_count();
// Sets a kernel's dynamic shared-memory limit once per (device, kernel, size).
cudaError_t smem_attr(const void *fn, int bytes);
// Resident blocks per SM of a kernel at a launch shape (at least 1; cached).
cudaError_t blocks_per_sm(const void *fn, int threads, size_t smem, int *n);

cudaError_t launch_gate(const GateLaunch &g, cudaStream_t stream);
cudaError_t launch_recurrent(const Problem &p, cudaStream_t stream);

// Chunked prefill.  `why` receives a static reason string when the problem
// falls outside what the kernel supports (the launcher then returns
// cudaErrorNotSupported without launching).
size_t chunked_workspace_bytes(const Problem &p, int chunk);
size_t chunked_workspace_min_bytes(const Problem &p, int chunk);
bool chunked_supported(const Problem &p, int chunk, const char **why);
cudaError_t launch_chunked(const Problem &p, int chunk, void *ws, size_t ws_bytes, cudaStream_t stream);

// tcgen05 chunked kernels (dk = dv = 128, every rule).  They take a workspace
// of chunked_tc_workspace_bytes() (every chunk's operand image at once), or
// down to chunked_tc_workspace_min_bytes() (one chunk per request at a time:
// the call then runs in windows of chunks, the state carried in final_state).
bool chunked_tc_eligible(const Problem &p);
size_t chunked_tc_workspace_bytes(const Problem &p);
size_t chunked_tc_workspace_min_bytes(const Problem &p);
cudaError_t launch_chunked_tc(const Problem &p, void *ws, size_t ws_bytes, cudaStream_t stream);

}  // namespace gdn
