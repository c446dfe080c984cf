// Decode attention fed by TMA (attn_decode.cu): the same arithmetic as
// launch_attn_block (bit-identical partials), with the keys and values of each
// stream read through its cache's 3-D tensor map.
#pragma once

#include "common.cuh"

namespace tfl {

// Per stream of a.rows: the tfl_kv's map over its pages (128 dims, n_kv heads,
// positions; boxes of 128 positions x 64 dims, 128-byte swizzle).
struct KvMaps {
    CUtensorMap m[kMaxStreams];
};

cudaError_t init_attn_decode_tma();
// status: the model's device status word (a bounded wait that gives up raises
// kStatusDevice); sms: the SM count of the model's device (the grid is at most
// one CTA per SM).
cudaError_t launch_attn_block_tma(const AttnDecodeArgs& a, const KvMaps& maps, int* status, int sms,
                                  cudaStream_t st, bool pdl);

}  // namespace tfl
