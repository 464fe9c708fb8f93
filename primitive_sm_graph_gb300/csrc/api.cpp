// The extern "C" entry points of libpsg: argument validation, planning, and
// the hand-off to one launcher per kernel family.  Nothing here allocates
// device memory or synchronises.
#include <cstdint>
#include <cstring>

#include "api_internal.h"
#include "common.h"
#include "jit.h"

namespace psg {

bool ptr_aligned(const void* p, int dt)
{
    const int es = dtype_size(dt);
    return es == 0 || ((uintptr_t)p % (uintptr_t)es) == 0;
}

int fill_operand(PsgOperand& op, const void* ptr, const psg_view* v, const Space& sp,
                 const int64_t* st, const int64_t* lo, const int64_t* hi, bool masked)
{
    std::memset(&op, 0, sizeof(op));
    const int nd = sp.nd;
    op.ptr = ptr;
    op.offset = v->offset;
    op.inner_stride = st[nd - 1];
    for (int d = 0; d < nd - 1; ++d) op.outer_stride[d] = st[d];
    for (int d = 0; d < nd; ++d) {
        op.mlo[d] = lo[d];
        op.mhi[d] = hi[d];
    }
    // the inner dim's mask also sits in the last slot, where the kernels read it
    op.mlo[MAXD - 1] = lo[nd - 1];
    op.mhi[MAXD - 1] = hi[nd - 1];
    return masked ? PSG_M_MASKED : st[nd - 1] == 0 ? PSG_M_UNIFORM : st[nd - 1] == 1 ? PSG_M_CONTIG
                                                                                     : PSG_M_STRIDED;
}

int vec_mode(int mode, const PsgOperand& op, int es, const Space& sp)
{
    if (mode != PSG_M_CONTIG || op.inner_stride != 1) return mode;
    if (((uintptr_t)op.ptr + (uint64_t)op.offset * es) % 16 != 0) return mode;
    for (int d = 0; d + 1 < sp.nd; ++d)
        if (sp.shape[d] > 1 && (op.outer_stride[d] * es) % 16 != 0) return mode;
    return PSG_M_VEC;
}

bool same_shape(const psg_view* a, const psg_view* b)
{
    if (a->ndim != b->ndim) return false;
    for (int d = 0; d < a->ndim; ++d)
        if (a->shape[d] != b->shape[d]) return false;
    return true;
}

}  // namespace psg

using namespace psg;

extern "C" {

psg_status psg_elementwise(const psg_node* prog, int n_nodes, const void* const* in,
                           const psg_view* in_v, int n_in, void* out, const psg_view* out_v,
                           void* stream)
{
    EwPlan P;
    psg_status st = plan_elementwise(prog, n_nodes, in, in_v, n_in, out, out_v, &P);
    if (st != PSG_OK) return st;
    return launch_elementwise(P, stream);
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

// Test hook, not part of the ABI: plan a psg_elementwise call over dummy
// pointers and compile its kernel with NVRTC without loading or launching it
// (needs no GPU).  Returns the planning/compile status; the NVRTC log is
// copied into `log`.
extern "C" int psg_internal_compile_elementwise(const psg_node* prog, int n_nodes, const psg_view* in_v,
                                                int n_in, const psg_view* out_v, char* log, size_t log_size)
{
    const void* fake[PSG_MAX_INPUTS];
    for (int k = 0; k < PSG_MAX_INPUTS; ++k) fake[k] = (const void*)(uintptr_t)4096;
    EwPlan P;
    psg_status st = plan_elementwise(prog, n_nodes, fake, in_v, n_in, (void*)(uintptr_t)4096, out_v, &P);
    if (st != PSG_OK) return st;
    std::string l;
    st = jit_compile_only(jit_source(JIT_EW, P.spec), &l);
    if (log && log_size) {
        std::strncpy(log, l.c_str(), log_size - 1);
        log[log_size - 1] = 0;
    }
    return st;
}
