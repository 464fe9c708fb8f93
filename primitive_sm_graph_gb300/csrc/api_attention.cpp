// psg_attention_fwd / psg_attention_bwd: validation and launch.
#include <cstring>

#include "api_internal.h"
#include "attention.h"

namespace psg {
namespace {

// a [B, T, H, 64] bf16 view the kernels can read with TMA: head dim
// contiguous, every other stride a multiple of 8 elements, 16-byte base
psg_status attn_view(const void* ptr, const psg_view* v, bool written, int64_t B, int64_t T, int64_t H,
                     AttnTensor* t)
{
    if (!v) return PSG_E_INVALID_ARG;
    psg_status st = check_view(v, written);
    if (st != PSG_OK) return st;
    if (v->dtype != PSG_BF16) return PSG_E_UNSUPPORTED_DTYPE;
    if (v->ndim != 4 || v->shape[0] != B || v->shape[1] != T || v->shape[2] != H) return PSG_E_INVALID_ARG;
    if (v->shape[3] != 64 || view_has_mask(v)) return PSG_E_UNSUPPORTED_LAYOUT;
    if (v->strides[3] != 1) return PSG_E_UNSUPPORTED_LAYOUT;
    for (int d = 0; d < 3; ++d)
        if (v->strides[d] % 8 != 0) return PSG_E_UNSUPPORTED_LAYOUT;
    if (B * T * H > 0 && !ptr) return PSG_E_INVALID_ARG;
    if (((uintptr_t)ptr + (uint64_t)v->offset * 2) % 16 != 0) return PSG_E_MISALIGNED;
    t->ptr = ptr;
    t->off = v->offset;
    t->sb = v->strides[0];
    t->st = v->strides[1];
    t->sh = v->strides[2];
    return PSG_OK;
}

psg_status attn_common(const psg_view* qv, float scale, int causal, AttnParams* p)
{
    if (!qv || qv->ndim != 4) return PSG_E_INVALID_ARG;
    std::memset(p, 0, sizeof(*p));
    p->B = (int)qv->shape[0];
    p->T = (int)qv->shape[1];
    p->H = (int)qv->shape[2];
    // grid limits: heads on y (65535), 2 B on z (the two backward passes)
    if (qv->shape[0] > 32767 || qv->shape[2] > 65535) return PSG_E_UNSUPPORTED_LAYOUT;
    if (qv->shape[1] > (1 << 24)) return PSG_E_UNSUPPORTED_LAYOUT;
    if (!(scale > 0.0f) || !(scale < 1e30f)) return PSG_E_INVALID_ARG;
    p->scale = scale;
    p->causal = causal ? 1 : 0;
    return PSG_OK;
}

}  // namespace
}  // namespace psg

using namespace psg;

extern "C" psg_status psg_attention_fwd(const void* q, const psg_view* qv, const void* k, const psg_view* kv,
                                        const void* v, const psg_view* vv, void* o, const psg_view* ov, float* lse,
                                        float scale, int causal, const uint8_t* key_mask, int32_t* d_status,
                                        void* stream)
{
    AttnParams p;
    psg_status st = attn_common(qv, scale, causal, &p);
    if (st != PSG_OK) return st;
    p.kmask = key_mask;
    p.km_sb = p.T;
    AttnTensor tq, tk, tv, to;
    if ((st = attn_view(q, qv, false, p.B, p.T, p.H, &tq)) != PSG_OK) return st;
    if ((st = attn_view(k, kv, false, p.B, p.T, p.H, &tk)) != PSG_OK) return st;
    if ((st = attn_view(v, vv, false, p.B, p.T, p.H, &tv)) != PSG_OK) return st;
    if ((st = attn_view(o, ov, true, p.B, p.T, p.H, &to)) != PSG_OK) return st;
    if ((int64_t)p.B * p.T * p.H > 0 && !lse) return PSG_E_INVALID_ARG;
    if ((uintptr_t)lse % 4 != 0) return PSG_E_MISALIGNED;
    p.lse = lse;
    p.status = d_status;
    p.o = o;
    p.o_off = to.off;
    p.o_sb = to.sb;
    p.o_st = to.st;
    p.o_sh = to.sh;
    return launch_attention_fwd(tq, tk, tv, p, stream);
}

extern "C" psg_status psg_attention_bwd(const void* q, const psg_view* qv, const void* k, const psg_view* kv,
                                        const void* v, const psg_view* vv, const void* o, const psg_view* ov,
                                        const void* dout, const psg_view* dov, const float* lse, float* delta,
                                        void* dq, const psg_view* dqv, void* dk, const psg_view* dkv, void* dv,
                                        const psg_view* dvv, float scale, int causal, const uint8_t* key_mask,
                                        int32_t* d_status, void* stream)
{
    AttnParams p;
    psg_status st = attn_common(qv, scale, causal, &p);
    if (st != PSG_OK) return st;
    p.kmask = key_mask;
    p.km_sb = p.T;
    AttnTensor tq, tk, tv, to, tdo, tdq, tdk, tdv;
    if ((st = attn_view(q, qv, false, p.B, p.T, p.H, &tq)) != PSG_OK) return st;
    if ((st = attn_view(k, kv, false, p.B, p.T, p.H, &tk)) != PSG_OK) return st;
    if ((st = attn_view(v, vv, false, p.B, p.T, p.H, &tv)) != PSG_OK) return st;
    if ((st = attn_view(o, ov, false, p.B, p.T, p.H, &to)) != PSG_OK) return st;
    if ((st = attn_view(dout, dov, false, p.B, p.T, p.H, &tdo)) != PSG_OK) return st;
    if ((st = attn_view(dq, dqv, true, p.B, p.T, p.H, &tdq)) != PSG_OK) return st;
    if ((st = attn_view(dk, dkv, true, p.B, p.T, p.H, &tdk)) != PSG_OK) return st;
    if ((st = attn_view(dv, dvv, true, p.B, p.T, p.H, &tdv)) != PSG_OK) return st;
    if ((int64_t)p.B * p.T * p.H > 0 && (!lse || !delta)) return PSG_E_INVALID_ARG;
    if ((uintptr_t)lse % 4 != 0 || (uintptr_t)delta % 4 != 0) return PSG_E_MISALIGNED;
    p.lse = const_cast<float*>(lse);
    p.delta = delta;
    p.status = d_status;
    return launch_attention_bwd(tq, tk, tv, to, tdo, tdq, tdk, tdv, p, stream);
}
