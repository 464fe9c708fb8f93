// Launch descriptors of the fused attention kernels.
#pragma once

#include "common.h"

namespace psg {

// Q, K, V, O, dO, dQ, dK, dV: bfloat16 [B, T, H, 64] with the head dim
// contiguous; strides (elements) per batch, token and head.
struct AttnTensor {
    const void* ptr;
    int64_t off, sb, st, sh;
};

struct AttnParams {
    int B, T, H;
    int causal;
    float scale;
    int32_t* status;
    float* lse;        // [B, H, T] float32: row logsumexp of the scaled, masked scores
    float* delta;      // [B, H, T] float32 (backward): rowsum(dO * O)
    void* o;           // forward output / backward dQ
    int64_t o_off, o_sb, o_st, o_sh;
    const uint8_t* kmask;  // [B, T] per-key visibility (nonzero: visible) or null
    int64_t km_sb;         // its batch stride (elements); token stride 1
};

psg_status launch_attention_fwd(const AttnTensor& q, const AttnTensor& k, const AttnTensor& v, const AttnParams& p,
                                void* stream);
psg_status launch_attention_bwd(const AttnTensor& q, const AttnTensor& k, const AttnTensor& v, const AttnTensor& o,
                                const AttnTensor& dO, const AttnTensor& dq, const AttnTensor& dk,
                                const AttnTensor& dv, const AttnParams& p, void* stream);

}  // namespace psg
