// kda_tc.cuh -- entry points of the tensor-core (tcgen05) prefill path.
#pragma once

#include "kda_internal.cuh"

namespace kda {

// True when the tensor-core path takes these arguments (D = 128, chunk = 64,
// bf16 inputs) and this device supports it.
bool tc_prefill_applies(const kda_prefill_args& a);

// Scratch bytes the tensor-core path needs.
size_t tc_prefill_workspace(const kda_prefill_args& a);

// Enqueues the tensor-core prefill; `ws` has tc_prefill_workspace(a) bytes.
cudaError_t launch_tc_prefill(const kda_prefill_args& a, char* ws, cudaStream_t s);

}  // namespace kda
