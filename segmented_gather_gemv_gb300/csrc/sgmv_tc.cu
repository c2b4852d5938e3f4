// sgmv_tc.cu -- tensor-core (tcgen05) path for segments with many rows.
#include "common.cuh"

namespace lora {

bool tc_available() { return false; }

cudaError_t launch_tc(const DeltaArgs &, int, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace lora
