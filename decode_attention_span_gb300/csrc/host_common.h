// Host-side helpers shared by the C-ABI translation units.
#pragma once

#include <cuda.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/sekv.h"
#include "sekv_common.cuh"

namespace sekv {

int device_sm_count();
int decode_cg(const sekv_config* cfg, int sms);
int route_chunks(const sekv_config* cfg);
WsLayout ws_layout(const sekv_config* cfg, int sms);
size_t ws_cta_bytes(const WsLayout& L);
void count_launch(int n);
void reset_launches();

// Rows of row_elems elements ([groups][rows][row_elems], dense) seen as
// (x: half a row, row, half, group): a box of box_rows rows brings both
// 128-byte halves of each row in one copy, 128-byte swizzle.
bool encode_rows4d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                   uint64_t row_elems, uint64_t rows, uint64_t groups, int elem_bytes,
                   uint32_t box_rows);

size_t build_workspace_size(const sekv_config* cfg, int64_t ctx_len);

}  // namespace sekv
