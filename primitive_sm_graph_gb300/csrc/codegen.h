// Program analysis and body generation for the runtime-specialised kernels.
#pragma once

#include <string>
#include <vector>

#include "common.h"

namespace psg {

struct ProgInfo {
    int n = 0;
    std::vector<int> dt;    // node dtype
    std::vector<int> val;   // value a node names (itself, or the source of a no-op CAST)
    std::vector<int> uni;   // uniform along the inner dim
    std::vector<int> live;  // needed by the result
    int result = 0;         // value of the last node
    int result_dtype = 0;
    bool result_uniform = false;
};

// Validate a program against the op set's dtype rules; in_dtype/in_uniform
// describe the inputs, red_dtype the reduced stage values a program may read
// (n_red = 0 forbids PSG_OP_RED).
psg_status analyze_program(const psg_node* nodes, int n, const int* in_dtype, const bool* in_uniform,
                           int n_in, const int* red_dtype, int n_red, ProgInfo* info);

// C++ source of `struct <name> { struct U; template <class C> static U uni(const
// C& c); template <class C> static void eval(const C& c, const U& u, T
// (&y)[PSG_VEC]); }`: uni() computes the program's uniform values (once per
// row), eval() the program for the PSG_VEC lanes of a chunk.
// C provides ldv<K>(arr), ld1<K>(), redf(s), redi(s).  With stash >= 0 the
// value of node `stash` (non-uniform) is read per lane from c.stashf(v) /
// c.stashi(v) instead of being computed, and whatever only fed it is dropped.
// With store_rounds the result goes only to a store that rounds float32 to a
// half width itself (round to nearest even), so a bfloat16/float16 last node
// is left unrounded; the stored bits are the same.
std::string gen_eval(const psg_node* nodes, const ProgInfo& info, const std::string& name,
                     const std::string& prefix = "", int stash = -1, bool store_rounds = false);

}  // namespace psg
