// Allocation failures that leave no stale CUDA error behind.
#pragma once

#include <cuda_runtime.h>

#include "../../include/cac.h"

namespace cac {

// A failed cudaMalloc / cudaHostAlloc leaves its error code for the next
// cudaGetLastError(), which the launch checks read; clear it, so that after a
// refused allocation the next successful launch does not report it.
inline int nomem() {
    cudaGetLastError();
    return CAC_E_NOMEM;
}

}  // namespace cac
