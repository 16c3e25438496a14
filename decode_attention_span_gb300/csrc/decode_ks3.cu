// Decode kernel instance for ranks up to 48 (3 rank k-steps of 16).
#include "decode_kernel_impl.cuh"

namespace sekv {

template __global__ void decode_kernel<3>(const __grid_constant__ DecodeParams P);

const void* decode_kernel_fn_ks3() { return reinterpret_cast<const void*>(&decode_kernel<3>); }

}  // namespace sekv
