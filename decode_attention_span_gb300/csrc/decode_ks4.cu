// Decode kernel instance for ranks up to 64 (4 rank k-steps of 16).
#include "decode_kernel_impl.cuh"

namespace sekv {

template __global__ void decode_kernel<4, false>(const __grid_constant__ DecodeParams P);
template __global__ void decode_kernel<4, true>(const __grid_constant__ DecodeParams P);

const void* decode_kernel_fn_ks4(bool mq) {
  return mq ? reinterpret_cast<const void*>(&decode_kernel<4, true>)
            : reinterpret_cast<const void*>(&decode_kernel<4, false>);
}

}  // namespace sekv
