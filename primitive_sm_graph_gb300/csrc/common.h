// Internal definitions shared by the host planners.  Not part of the public
// ABI (that is include/psg.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include "jit/params.h"
#include "psg.h"

namespace psg {

constexpr int MAXD = PSG_MAXD;
constexpr int VEC = PSG_VEC;
constexpr int MAX_IN = PSG_MAXIN;
constexpr int MAX_STAGES = PSG_MAXSTAGES;

static_assert(PSG_DT_F32 == PSG_F32 && PSG_DT_BF16 == PSG_BF16 && PSG_DT_F16 == PSG_F16 &&
                  PSG_DT_F64 == PSG_F64 && PSG_DT_I32 == PSG_I32 && PSG_DT_I16 == PSG_I16 &&
                  PSG_DT_I8 == PSG_I8,
              "dtype codes of the kernels and the ABI must agree");

inline int dtype_size(int dt)
{
    switch (dt) {
    case PSG_F32: case PSG_I32: return 4;
    case PSG_BF16: case PSG_F16: case PSG_I16: return 2;
    case PSG_F64: return 8;
    case PSG_I8: return 1;
    }
    return 0;
}
inline bool dtype_valid(int dt) { return dt >= PSG_F32 && dt <= PSG_I8; }
inline bool dtype_is_int(int dt) { return dt == PSG_I32 || dt == PSG_I16 || dt == PSG_I8; }
inline bool dtype_is_float(int dt) { return dt == PSG_F32 || dt == PSG_BF16 || dt == PSG_F16; }

// Iteration space after dim collapsing: dims 0..nd-2 are "outer" (one row =
// one outer multi-index), dim nd-1 is the inner dim walked VEC cells at a time.
struct Space {
    int32_t nd;
    int32_t pad;
    int64_t shape[MAXD];
    int64_t rows;
    int64_t inner;
    int64_t chunks;
};

// view.cpp
psg_status check_view(const psg_view* v, bool for_write);
int64_t view_numel(const psg_view* v);
bool view_has_mask(const psg_view* v);
bool view_contiguous(const psg_view* v);

// Common iteration space of n views (the output first): dims ordered by the
// first view's strides (its stride-1 dim innermost) and merged where every
// view is contiguous and unmasked across the pair; keep_last keeps the views'
// last dim as the inner dim (a reduction axis).
psg_status build_space(const psg_view* const* views, int nviews, bool keep_last, Space* sp,
                       int64_t (*strides)[MAXD], int64_t (*mlo)[MAXD], int64_t (*mhi)[MAXD],
                       bool* masked);

}  // namespace psg
