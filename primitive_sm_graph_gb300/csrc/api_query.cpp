// psg_query_launch: grid, block, dynamic shared memory and registers of the
// kernel a call would launch for a given output view (Tiki, "The architecture
// we want": register and shared-memory budgets visible before launch).  For
// the runtime-specialised calls (elementwise, reduce_rows) the kernel depends
// on the program; the query reports the kernel of the simplest program (a
// LOAD of the view's dtype, a SUM of it).
#include <cstring>

#include "api_internal.h"
#include "common.h"
#include "contract.h"
#include "launch_util.cuh"
#include "permute.h"

using namespace psg;

extern "C" psg_status psg_reduce_rows(const psg_reduce_stage*, int, const psg_node*, int, const void* const*,
                                      const psg_view*, int, void*, const psg_view*, int32_t*, void*);

namespace psg {
psg_status query_reduce(const psg_reduce_stage* stages, int n_stages, const psg_node* epi, int n_epi,
                        const psg_view* in_v, int n_in, const psg_view* out_v, int* grid, int* block,
                        int* smem, int* regs);
}

extern "C" psg_status psg_query_launch(int call, const psg_view* v, int* grid, int* block, int* smem, int* regs)
{
    if (!v || !grid || !block || !smem || !regs) return PSG_E_INVALID_ARG;
    psg_status st = check_view(v, false);
    if (st != PSG_OK) return st;
    const void* fake = (const void*)(uintptr_t)4096;
    psg_node ld;
    std::memset(&ld, 0, sizeof(ld));
    ld.op = PSG_OP_LOAD;
    ld.dtype = v->dtype;
    switch (call) {
    case PSG_CALL_ELEMENTWISE: {
        psg_view ov = *v;
        for (int d = 0; d < ov.ndim; ++d) { ov.mask_lo[d] = 0; ov.mask_hi[d] = ov.shape[d]; }
        EwPlan P;
        st = plan_elementwise(&ld, 1, &fake, v, 1, (void*)fake, &ov, &P);
        if (st != PSG_OK) return st;
        return query_elementwise(P, grid, block, smem, regs);
    }
    case PSG_CALL_REDUCE_ROWS: {
        psg_reduce_stage s;
        s.op = PSG_RED_SUM;
        s.n_nodes = 1;
        s.prologue = &ld;
        psg_view ov = *v;
        ov.ndim = v->ndim > 0 ? v->ndim - 1 : 0;
        int64_t st1 = 1;
        for (int d = ov.ndim - 1; d >= 0; --d) { ov.strides[d] = st1; st1 *= ov.shape[d]; ov.mask_lo[d] = 0; ov.mask_hi[d] = ov.shape[d]; }
        ov.offset = 0;
        ov.extent = st1;
        return query_reduce(&s, 1, nullptr, 0, v, 1, &ov, grid, block, smem, regs);
    }
    case PSG_CALL_PERMUTE: {
        int64_t tiles = 1;
        for (int d = 0; d < v->ndim; ++d) tiles *= (v->shape[d] + 63) / 64;
        query_transpose(dtype_size(v->dtype), tiles, grid, block, smem, regs);
        return PSG_OK;
    }
    case PSG_CALL_CONTRACT_BF16: {
        if (v->ndim < 2) return PSG_E_INVALID_ARG;
        const int64_t M = v->shape[v->ndim - 2];
        int64_t tiles = ((M + 127) / 128) * ((v->shape[v->ndim - 1] + 255) / 256);
        for (int d = 0; d < v->ndim - 2; ++d) tiles *= v->shape[d];
        query_contract_tc(M, tiles, grid, block, smem, regs);
        return PSG_OK;
    }
    case PSG_CALL_CONTRACT_F32_TENSOR: {
        if (v->ndim < 2) return PSG_E_INVALID_ARG;
        int64_t tiles = ((v->shape[v->ndim - 2] + 127) / 128) * ((v->shape[v->ndim - 1] + 127) / 128);
        for (int d = 0; d < v->ndim - 2; ++d) tiles *= v->shape[d];
        query_contract_tf32(tiles, grid, block, smem, regs);
        return PSG_OK;
    }
    case PSG_CALL_CONTRACT_F32: {
        if (v->ndim < 2) return PSG_E_INVALID_ARG;
        SimtParams p;
        std::memset(&p, 0, sizeof(p));
        p.ab_dtype = PSG_F32;
        p.M = v->shape[v->ndim - 2];
        p.N = v->shape[v->ndim - 1];
        p.batch = 1;
        for (int d = 0; d < v->ndim - 2; ++d) p.batch *= v->shape[d];
        query_contract_simt(p, grid, block, smem, regs);
        return PSG_OK;
    }
    case PSG_CALL_GATHER:
    case PSG_CALL_SCATTER_ADD: {
        const int64_t rows = v->ndim > 0 ? v->shape[0] : 1;
        *grid = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms() * 8);
        *block = 256;
        *smem = 0;
        *regs = -1;
        return PSG_OK;
    }
    }
    return PSG_E_INVALID_ARG;
}
