// Host-side helpers shared by the library's translation units (defined in mfa_decode.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "mfa.h"

namespace mfa {

// Records the text of a CUDA failure for mfa_last_cuda_error() and returns MFA_ERR_CUDA.
mfa_status cuda_fail(cudaError_t e, const char* where);

// Shape, dtype and range checks of a problem description (MFA_OK, or the error to return).
mfa_status check_problem(const mfa_problem* pr);

// The attention shape of a problem that check_problem accepts: 0 MFA, 1 grouped heads,
// 2 shared latent.
int problem_shape(const mfa_problem* pr);

// True when p is a multiple of a bytes.
bool aligned(const void* p, uintptr_t a);

}  // namespace mfa
