// The extern "C" entry points of libpsg: argument validation, planning, and
// the hand-off to one launcher per kernel family.  Nothing here allocates
// device memory or synchronises.
#include <cstdint>
#include <cstring>

#include "api_internal.h"
#include "common.h"

namespace psg {

bool ptr_aligned(const void* p, int dt)
{
    const int es = dtype_size(dt);
    return es == 0 || ((uintptr_t)p % (uintptr_t)es) == 0;
}

void fill_operand(Operand& op, const void* ptr, const psg_view* v, const Space& sp,
                  const int64_t* st, const int64_t* lo, const int64_t* hi, bool masked)
{
    std::memset(&op, 0, sizeof(op));
    const int nd = sp.nd;
    op.ptr = ptr;
    op.dtype = v->dtype;
    op.offset = v->offset;
    op.inner_stride = st[nd - 1];
    for (int d = 0; d < nd - 1; ++d) op.outer_stride[d] = st[d];
    for (int d = 0; d < nd; ++d) {
        op.mlo[d] = lo[d];
        op.mhi[d] = hi[d];
    }
    op.mlo[MAXD - 1] = lo[nd - 1];
    op.mhi[MAXD - 1] = hi[nd - 1];
    op.mode = masked ? IN_MASKED : st[nd - 1] == 0 ? IN_UNIFORM : st[nd - 1] == 1 ? IN_CONTIG : IN_STRIDED;
}

bool same_shape(const psg_view* a, const psg_view* b)
{
    if (a->ndim != b->ndim) return false;
    for (int d = 0; d < a->ndim; ++d)
        if (a->shape[d] != b->shape[d]) return false;
    return true;
}

psg_status plan_elementwise(const psg_node* prog, int n_nodes, const void* const* in,
                            const psg_view* in_v, int n_in, void* out, const psg_view* out_v,
                            EwLaunch* L)
{
    if (!prog || n_nodes < 1 || n_nodes > PSG_MAX_NODES) return PSG_E_INVALID_ARG;
    if (n_in < 0 || n_in > PSG_MAX_INPUTS) return PSG_E_INVALID_ARG;
    if (n_in > 0 && (!in || !in_v)) return PSG_E_INVALID_ARG;
    if (!out_v) return PSG_E_INVALID_ARG;
    psg_status st = check_view(out_v, true);
    if (st != PSG_OK) return st;
    if (out_v->dtype == PSG_F64) return PSG_E_UNSUPPORTED_DTYPE;
    const int64_t n = view_numel(out_v);
    if (n > 0 && !out) return PSG_E_INVALID_ARG;
    if (!ptr_aligned(out, out_v->dtype)) return PSG_E_MISALIGNED;
    const psg_view* views[1 + PSG_MAX_INPUTS];
    views[0] = out_v;
    int dts[PSG_MAX_INPUTS];
    for (int k = 0; k < n_in; ++k) {
        st = check_view(&in_v[k], false);
        if (st != PSG_OK) return st;
        if (!same_shape(&in_v[k], out_v)) return PSG_E_INVALID_ARG;
        if (in_v[k].dtype == PSG_F64) return PSG_E_UNSUPPORTED_DTYPE;
        if (n > 0 && !in[k]) return PSG_E_INVALID_ARG;
        if (!ptr_aligned(in[k], in_v[k].dtype)) return PSG_E_MISALIGNED;
        views[1 + k] = &in_v[k];
        dts[k] = in_v[k].dtype;
    }
    std::memset(L, 0, sizeof(*L));
    int64_t strides[1 + PSG_MAX_INPUTS][MAXD], lo[1 + PSG_MAX_INPUTS][MAXD], hi[1 + PSG_MAX_INPUTS][MAXD];
    bool masked[1 + PSG_MAX_INPUTS];
    st = build_space(views, 1 + n_in, false, &L->sp, strides, lo, hi, masked);
    if (st != PSG_OK) return st;
    bool uni[PSG_MAX_INPUTS];
    for (int k = 0; k < n_in; ++k) {
        fill_operand(L->in[k], in[k], &in_v[k], L->sp, strides[1 + k], lo[1 + k], hi[1 + k], masked[1 + k]);
        uni[k] = L->in[k].mode == IN_UNIFORM;
    }
    fill_operand(L->out, out, out_v, L->sp, strides[0], lo[0], hi[0], false);
    int rdt;
    bool runi;
    st = compile_program(prog, n_nodes, dts, uni, n_in, nullptr, 0, true, &L->prog, &rdt, &runi);
    if (st != PSG_OK) return st;
    if (rdt != out_v->dtype) return PSG_E_UNSUPPORTED_DTYPE;
    L->n_in = n_in;
    L->out_uniform = runi ? 1 : 0;
    return PSG_OK;
}

}  // namespace psg

using namespace psg;

extern "C" {

psg_status psg_elementwise(const psg_node* prog, int n_nodes, const void* const* in,
                           const psg_view* in_v, int n_in, void* out, const psg_view* out_v,
                           void* stream)
{
    EwLaunch L;
    psg_status st = plan_elementwise(prog, n_nodes, in, in_v, n_in, out, out_v, &L);
    if (st != PSG_OK) return st;
    return launch_elementwise(L, stream);
}

const char* psg_status_string(int s)
{
    switch (s) {
    case PSG_OK: return "ok";
    case PSG_E_INVALID_ARG: return "invalid argument";
    case PSG_E_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case PSG_E_UNSUPPORTED_LAYOUT: return "unsupported layout";
    case PSG_E_OUT_OF_BOUNDS_VIEW: return "view reaches outside its allocation";
    case PSG_E_MISALIGNED: return "misaligned pointer";
    case PSG_E_INDEX_OUT_OF_RANGE: return "index out of range";
    case PSG_E_TIMEOUT: return "bounded device wait timed out";
    case PSG_E_CUDA: return "CUDA error";
    case PSG_E_UNSUPPORTED_PROGRAM: return "unsupported program (too long or too many live values)";
    case PSG_E_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

const char* psg_version(void) { return "psg 0.1.0 sm_103a"; }

}  // extern "C"
