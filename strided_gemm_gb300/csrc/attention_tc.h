// Fused attention on the tensor cores (opt-in TF32): the host side's view of
// attention_tc.cu.
#pragma once

#include <cuda_runtime.h>

#include "internal.h"

namespace sbg {

// True when the operands suit the kernel's tensor maps: Q, K and V with unit
// stride along the head dimension, 16-byte aligned bases and row / batch
// strides (a zero batch stride broadcasts), head dimension 64.
bool attention_tc_supported(const AttnProblem& a);

cudaError_t launch_attention_tc(const AttnProblem& a, cudaStream_t stream);

// Reads and clears the kernel's status word (0 when no wait ran out).
unsigned int read_and_clear_wait_status_attention_tc(cudaStream_t stream);

}  // namespace sbg
