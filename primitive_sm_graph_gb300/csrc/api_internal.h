// Helpers shared by the entry points (api.cpp and the per-family API files).
#pragma once

#include "common.h"

namespace psg {

bool ptr_aligned(const void* p, int dt);
bool same_shape(const psg_view* a, const psg_view* b);
void fill_operand(Operand& op, const void* ptr, const psg_view* v, const Space& sp,
                  const int64_t* st, const int64_t* lo, const int64_t* hi, bool masked);
psg_status plan_elementwise(const psg_node* prog, int n_nodes, const void* const* in,
                            const psg_view* in_v, int n_in, void* out, const psg_view* out_v,
                            EwLaunch* L);

}  // namespace psg
