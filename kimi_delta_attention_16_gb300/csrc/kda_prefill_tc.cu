// kda_prefill_tc.cu -- tensor-core (tcgen05) chunkwise prefill.
#include "kda_tc.cuh"

namespace kda {

bool tc_prefill_applies(const kda_prefill_args&) { return false; }

size_t tc_prefill_workspace(const kda_prefill_args&) { return 0; }

cudaError_t launch_tc_prefill(const kda_prefill_args&, char*, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace kda
