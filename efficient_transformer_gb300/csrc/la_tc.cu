// la_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) kernels for bfloat16 inputs.
#include "la_internal.cuh"

namespace la {

bool tc_supported(int, int, int, int, la_dtype, int, int, int) { return false; }
cudaError_t tc_forward(const Params &, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t tc_backward(const Params &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace la
