// Helpers shared by the entry points and planners.
#pragma once

#include <string>

#include "common.h"

namespace psg {

bool ptr_aligned(const void* p, int dt);
bool same_shape(const psg_view* a, const psg_view* b);
// Fill a kernel operand from a view and its iteration-space strides/masks;
// returns its addressing mode (PSG_M_*).
int fill_operand(PsgOperand& op, const void* ptr, const psg_view* v, const Space& sp,
                 const int64_t* st, const int64_t* lo, const int64_t* hi, bool masked);
// PSG_M_VEC in place of PSG_M_CONTIG when the operand's base and every row
// start are 16-byte aligned (es: element size): the kernels then move whole
// chunks with vector loads and stores and test nothing at run time.
int vec_mode(int mode, const PsgOperand& op, int es, const Space& sp);

struct EwPlan {
    PsgEwParams p;
    int n_in;
    std::string spec;  // the program-specific part of the runtime-compiled source
};
psg_status plan_elementwise(const psg_node* prog, int n_nodes, const void* const* in,
                            const psg_view* in_v, int n_in, void* out, const psg_view* out_v,
                            EwPlan* P);
psg_status launch_elementwise(const EwPlan& P, void* stream);
psg_status query_elementwise(const EwPlan& P, int* grid, int* block, int* smem, int* regs);

}  // namespace psg
