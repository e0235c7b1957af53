// Entry points shared between the C-ABI translation units (api.cu, noalloc.cu); not exported.
#pragma once

#include "../../include/msa.h"

namespace msa {

// Bytes the query-major team attention needs (error word + its partial-state slots): the
// scratch of the no-allocation entry point, whatever the batch.
size_t team_attn_workspace_bytes();

// msa_sparse_attn_decode, with the block-major form of long query chunks allowed or not (the
// no-allocation entry point's fixed scratch holds only the team kernel's states).  With
// clear_error, the device error word is zeroed on the stream once every argument has passed
// validation, right before the launch (a rejected call touches nothing).
msa_status_t sparse_attn_entry(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                               const uint8_t* q, const int32_t* selection, uint16_t* out, float* lse,
                               void* workspace, size_t workspace_bytes, void* stream, bool block_major_ok,
                               bool clear_error);

}  // namespace msa
