// psg_gather / psg_scatter_add: validation and launch planning.
#include <cstring>

#include "api_internal.h"
#include "common.h"
#include "gather_scatter.h"

namespace psg {

namespace {

// The dims after the first, as one (length, stride) pair, if they collapse.
bool row_layout(const psg_view* v, int64_t* D, int64_t* cs)
{
    int64_t len = 1, st = 1;
    bool have = false;
    for (int d = v->ndim - 1; d >= 1; --d) {
        if (v->shape[d] == 1) continue;
        if (!have) {
            len = v->shape[d];
            st = v->strides[d];
            have = true;
        } else {
            if (v->strides[d] != st * len) return false;
            len *= v->shape[d];
        }
    }
    *D = len;
    *cs = have ? st : 1;
    return true;
}

bool rest_shape_equal(const psg_view* a, const psg_view* b)
{
    if (a->ndim != b->ndim) return false;
    for (int d = 1; d < a->ndim; ++d)
        if (a->shape[d] != b->shape[d]) return false;
    return true;
}

}  // namespace

psg_status plan_gather(const void* src, const psg_view* sv, const int32_t* idx, int64_t n, void* out,
                       const psg_view* ov, int32_t* d_status, GatherLaunch* L)
{
    if (!sv || !ov || !d_status || n < 0) return PSG_E_INVALID_ARG;
    psg_status st = check_view(sv, false);
    if (st != PSG_OK) return st;
    st = check_view(ov, true);
    if (st != PSG_OK) return st;
    if (sv->ndim < 1 || !rest_shape_equal(sv, ov) || ov->shape[0] != n) return PSG_E_INVALID_ARG;
    if (sv->dtype != ov->dtype) return PSG_E_UNSUPPORTED_DTYPE;
    if (view_has_mask(sv)) return PSG_E_UNSUPPORTED_LAYOUT;
    std::memset(L, 0, sizeof(*L));
    if (!row_layout(sv, &L->D, &L->src_cs) || !row_layout(ov, &L->D, &L->out_cs)) return PSG_E_UNSUPPORTED_LAYOUT;
    if (n > 0 && (!idx || !out || !src)) return PSG_E_INVALID_ARG;
    if (!ptr_aligned(src, sv->dtype) || !ptr_aligned(out, ov->dtype) || ((uintptr_t)idx & 3)) return PSG_E_MISALIGNED;
    const int es = dtype_size(sv->dtype);
    L->src = src;
    L->out = out;
    L->idx = idx;
    L->status = d_status;
    L->n = n;
    L->V = sv->shape[0];
    L->es = es;
    L->src_offset = sv->offset;
    L->src_rs = sv->strides[0];
    L->out_offset = ov->offset;
    L->out_rs = ov->strides[0];
    const bool contig = L->src_cs == 1 && L->out_cs == 1 && (L->D * es) % 16 == 0;
    const bool al = ((uintptr_t)((const char*)src + sv->offset * es) % 16 == 0) &&
                    ((uintptr_t)((char*)out + ov->offset * es) % 16 == 0) &&
                    (L->src_rs * es) % 16 == 0 && (L->out_rs * es) % 16 == 0;
    L->vec16 = contig && al ? 1 : 0;
    return PSG_OK;
}

psg_status plan_scatter(void* dst, const psg_view* dv, const int32_t* idx, int64_t n, const void* upd,
                        const psg_view* uv, int32_t* d_status, ScatterLaunch* L)
{
    if (!dv || !uv || !d_status || n < 0 || n >= (int64_t(1) << 31)) return PSG_E_INVALID_ARG;
    psg_status st = check_view(dv, true);
    if (st != PSG_OK) return st;
    st = check_view(uv, false);
    if (st != PSG_OK) return st;
    if (dv->ndim < 1 || !rest_shape_equal(dv, uv) || uv->shape[0] != n) return PSG_E_INVALID_ARG;
    if (dv->dtype != uv->dtype) return PSG_E_UNSUPPORTED_DTYPE;
    const int dt = dv->dtype;
    if (!dtype_valid(dt)) return PSG_E_UNSUPPORTED_DTYPE;
    if (view_has_mask(uv)) return PSG_E_UNSUPPORTED_LAYOUT;
    std::memset(L, 0, sizeof(*L));
    int64_t D2;
    if (!row_layout(dv, &L->D, &L->dst_cs) || !row_layout(uv, &D2, &L->upd_cs)) return PSG_E_UNSUPPORTED_LAYOUT;
    if (n > 0 && (!idx || !dst || !upd)) return PSG_E_INVALID_ARG;
    if (!ptr_aligned(dst, dt) || !ptr_aligned(upd, dt) || ((uintptr_t)idx & 3)) return PSG_E_MISALIGNED;
    L->dst = dst;
    L->upd = upd;
    L->idx = idx;
    L->status = d_status;
    L->n = n;
    L->V = dv->shape[0];
    L->dtype = dt;
    L->dst_offset = dv->offset;
    L->dst_rs = dv->strides[0];
    L->upd_offset = uv->offset;
    L->upd_rs = uv->strides[0];
    return PSG_OK;
}

}  // namespace psg

using namespace psg;

extern "C" {

psg_status psg_gather(const void* src, const psg_view* sv, const int32_t* idx, int64_t n, void* out,
                      const psg_view* ov, int32_t* d_status, void* stream)
{
    GatherLaunch L;
    psg_status st = plan_gather(src, sv, idx, n, out, ov, d_status, &L);
    if (st != PSG_OK) return st;
    return launch_gather(L, stream);
}

size_t psg_scatter_workspace(int64_t n)
{
    return scatter_workspace_bytes(n);
}

psg_status psg_scatter_add(void* dst, const psg_view* dv, const int32_t* idx, int64_t n, const void* upd,
                           const psg_view* uv, void* workspace, size_t ws_bytes, int32_t* d_status,
                           void* stream)
{
    ScatterLaunch L;
    psg_status st = plan_scatter(dst, dv, idx, n, upd, uv, d_status, &L);
    if (st != PSG_OK) return st;
    if (n == 0) return PSG_OK;
    if (!workspace || ws_bytes < psg_scatter_workspace(n) || ((uintptr_t)workspace & 15)) return PSG_E_WORKSPACE;
    return launch_scatter(L, (unsigned long long*)workspace, stream);
}

psg_status psg_scatter_add_static(void* dst, const psg_view* dv, const int32_t* idx, int64_t n, const void* upd,
                                  const psg_view* uv, int32_t* d_status, void* stream)
{
    ScatterLaunch L;
    psg_status st = plan_scatter(dst, dv, idx, n, upd, uv, d_status, &L);
    if (st != PSG_OK) return st;
    if (n == 0) return PSG_OK;
    if (n > PSG_SCATTER_STATIC_MAX_N) return PSG_E_WORKSPACE;
    unsigned long long* keys = nullptr;
    st = static_scatter_keys(&keys);
    if (st != PSG_OK) return st;
    // every key slot the sort reads is written by this call first, so the
    // previous call's contents need no clearing
    return launch_scatter(L, keys, stream);
}

}  // extern "C"
