// Decode kernel instance for ranks up to 16 (1 rank k-step of 16).
#include "decode_kernel_impl.cuh"

namespace sekv {

template __global__ void decode_kernel<1, false>(const __grid_constant__ DecodeParams P);
template __global__ void decode_kernel<1, true>(const __grid_constant__ DecodeParams P);

const void* decode_kernel_fn_ks1(bool mq) {
  return mq ? reinterpret_cast<const void*>(&decode_kernel<1, true>)
            : reinterpret_cast<const void*>(&decode_kernel<1, false>);
}

}  // namespace sekv
