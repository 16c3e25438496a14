// Decode kernel instance for ranks up to 48 (3 rank k-steps of 16).
#include "decode_kernel_impl.cuh"

namespace sekv {

template __global__ void decode_kernel<3, false>(const __grid_constant__ DecodeParams P);
template __global__ void decode_kernel<3, true>(const __grid_constant__ DecodeParams P);

const void* decode_kernel_fn_ks3(bool mq) {
  return mq ? reinterpret_cast<const void*>(&decode_kernel<3, true>)
            : reinterpret_cast<const void*>(&decode_kernel<3, false>);
}

}  // namespace sekv
