// Decode path, more than 8 tokens: the persistent streaming gate_up kernel
// (decode_stream.cu), used by the decode FFN launcher in place of the
// one-CTA-per-tile kernel.
#pragma once

#include "qsm_common.cuh"

namespace qsm {

// The layer's shapes fit the streaming kernel (its ring and x buffers).
bool gate_up_stream_supported(const qsm_moe_layer* L);

// gate_up + SwiGLU of every work slot (the shared expert's blocks of 8
// tokens, then the block map's blocks) into hbuf; the shared-expert gates
// into gbuf when the layer has them.
qsm_status gate_up_stream_launch(const qsm_moe_layer* L, const uint16_t* x, int T,
                                 const qsm_grouping* grp, int shared_slots, __half* hbuf,
                                 float* gbuf, float* gu_dump, int32_t* dev_status,
                                 cudaStream_t stream);

}  // namespace qsm
