// chunked.cu -- chunk-parallel prefill (placeholder until the kernel lands).
#include "launch.h"

namespace gdn {

size_t chunked_workspace_bytes(const Problem &, int) { return 0; }

bool chunked_supported(const Problem &, int, const char **why) {
    *why = "not built yet";
    return false;
}

cudaError_t launch_chunked(const Problem &, int, void *, size_t, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gdn
