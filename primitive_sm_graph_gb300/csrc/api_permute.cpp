// psg_permute: validate, build the permuted View, pick the tiled transpose,
// the elementwise copy or the per-cell copy.
#include <cstring>

#include "api_internal.h"
#include "common.h"
#include "permute.h"

namespace psg {

psg_status plan_permute(const void* in, const psg_view* in_v, const int32_t* perm, void* out,
                        const psg_view* out_v, int* kind, TransposeLaunch* T, CopyLaunch* C,
                        EwPlan* E)
{
    if (!in_v || !out_v) return PSG_E_INVALID_ARG;
    psg_status st = check_view(in_v, false);
    if (st != PSG_OK) return st;
    st = check_view(out_v, true);
    if (st != PSG_OK) return st;
    const int nd = in_v->ndim;
    if (out_v->ndim != nd || (nd > 0 && !perm)) return PSG_E_INVALID_ARG;
    if (in_v->dtype != out_v->dtype) return PSG_E_UNSUPPORTED_DTYPE;
    bool seen[PSG_MAX_DIMS] = {false};
    psg_view pv = *in_v;
    for (int d = 0; d < nd; ++d) {
        const int p = perm[d];
        if (p < 0 || p >= nd || seen[p]) return PSG_E_INVALID_ARG;
        seen[p] = true;
        pv.shape[d] = in_v->shape[p];
        pv.strides[d] = in_v->strides[p];
        pv.mask_lo[d] = in_v->mask_lo[p];
        pv.mask_hi[d] = in_v->mask_hi[p];
        if (out_v->shape[d] != pv.shape[d]) return PSG_E_INVALID_ARG;
    }
    const int64_t n = view_numel(out_v);
    if (n > 0 && (!in || !out)) return PSG_E_INVALID_ARG;
    if (!ptr_aligned(in, in_v->dtype) || !ptr_aligned(out, out_v->dtype)) return PSG_E_MISALIGNED;
    const int es = dtype_size(in_v->dtype);
    const psg_view* views[2] = {out_v, &pv};
    Space sp;
    int64_t strides[2][MAXD], lo[2][MAXD], hi[2][MAXD];
    bool masked[2];
    st = build_space(views, 2, false, &sp, strides, lo, hi, masked);
    if (st != PSG_OK) return st;
    const int m = sp.nd;
    int adim = -1;
    if (!masked[1] && strides[0][m - 1] == 1 && strides[1][m - 1] != 1) {
        for (int d = 0; d < m - 1; ++d)
            if (strides[1][d] == 1) adim = d;
    }
    if (adim >= 0) {
        std::memset(T, 0, sizeof(*T));
        T->in = in;
        T->out = out;
        T->es = es;
        T->A = sp.shape[adim];
        T->I = sp.shape[m - 1];
        T->in_si = strides[1][m - 1];
        T->out_sa = strides[0][adim];
        T->in_offset = pv.offset;
        T->out_offset = out_v->offset;
        T->batch = 1;
        int nb = 0;
        for (int d = 0; d < m - 1; ++d) {
            if (d == adim) continue;
            T->bshape[nb] = sp.shape[d];
            T->in_bstride[nb] = strides[1][d];
            T->out_bstride[nb] = strides[0][d];
            T->batch *= sp.shape[d];
            ++nb;
        }
        T->nb = nb;
        *kind = 0;
        return PSG_OK;
    }
    if (in_v->dtype != PSG_F64) {
        psg_node ld;
        std::memset(&ld, 0, sizeof(ld));
        ld.op = PSG_OP_LOAD;
        ld.a = 0;
        ld.dtype = in_v->dtype;
        const void* ins[1] = {in};
        st = plan_elementwise(&ld, 1, ins, &pv, 1, out, out_v, E);
        if (st != PSG_OK) return st;
        *kind = 1;
        return PSG_OK;
    }
    std::memset(C, 0, sizeof(*C));
    C->in = in;
    C->out = out;
    C->es = es;
    C->nd = m;
    C->numel = n;
    C->in_offset = pv.offset;
    C->out_offset = out_v->offset;
    for (int d = 0; d < m; ++d) {
        C->shape[d] = sp.shape[d];
        C->in_stride[d] = strides[1][d];
        C->out_stride[d] = strides[0][d];
        C->mlo[d] = lo[1][d];
        C->mhi[d] = hi[1][d];
    }
    *kind = 2;
    return PSG_OK;
}

}  // namespace psg

using namespace psg;

extern "C" psg_status psg_permute(const void* in, const psg_view* in_v, const int32_t* perm,
                                  void* out, const psg_view* out_v, void* stream)
{
    int kind = 0;
    TransposeLaunch T;
    CopyLaunch C;
    EwPlan E;
    psg_status st = plan_permute(in, in_v, perm, out, out_v, &kind, &T, &C, &E);
    if (st != PSG_OK) return st;
    if (kind == 0) return launch_transpose(T, stream);
    if (kind == 1) return launch_elementwise(E, stream);
    return launch_copy(C, stream);
}
