// Process-environment checks shared by the library's entry points (host only).
#ifndef DGC_HOST_ENV_H
#define DGC_HOST_ENV_H

#include <cstdlib>

namespace dgc_host {

// True when the process belongs to a job over several GPUs (the launcher's
// WORLD_SIZE is above 1). Cluster-multicast TMA loads are a single-GPU feature
// here: every entry point that would issue them refuses such a job with
// GEMM_ERR_UNSUPPORTED before touching the device, so no multicast load is ever
// part of a multi-GPU run.
inline bool world_is_multi_gpu() {
    const char* w = std::getenv("WORLD_SIZE");
    return w && std::atoi(w) > 1;
}

}  // namespace dgc_host

#endif  // DGC_HOST_ENV_H
