// Host helpers of the decode entry points, shared by the translation units
// that launch the decode kernel.
#pragma once

#include "decode_attn.cuh"

namespace sekv {

bool config_ok(const sekv_config* cfg, sekv_status* why);
bool aligned16(const void* p);
sekv_status check_cache(const sekv_config* cfg, const sekv_layer_cache* c, bool need_store);
sekv_status fill_decode_params(const sekv_config* cfg, const sekv_layer_cache* cache,
                               const WsLayout& L, void* ws, DecodeParams& P, bool fused);
sekv_status launch_decode(const DecodeParams& P, const WsLayout& L, const sekv_config* cfg,
                          cudaStream_t stream, bool overlap);

}  // namespace sekv
