// Launch descriptors of the indexed kernels.
#pragma once

#include "common.h"

namespace psg {

struct GatherLaunch {
    const void* src;
    void* out;
    const int32_t* idx;
    int32_t* status;
    int64_t n, V, D;          // rows gathered, rows of src, cells per row
    int32_t es;               // element size
    int32_t vec16;            // rows contiguous and 16-byte aligned
    int64_t src_offset, src_rs, src_cs;
    int64_t out_offset, out_rs, out_cs;
};

struct ScatterLaunch {
    void* dst;
    const void* upd;
    const int32_t* idx;
    int32_t* status;
    int64_t n, V, D;
    int32_t dtype;
    int32_t pad;
    int64_t dst_offset, dst_rs, dst_cs;
    int64_t upd_offset, upd_rs, upd_cs;
};

// Update lists up to this length are ordered by one block (stable radix sort
// of the indices in shared memory); longer ones by a multi-block bitonic sort.
constexpr int64_t kScatterPlanMaxN = 16384;

// Capacity of the static key scratch of psg_scatter_add_static (keys, after
// rounding n up to a power of two).
constexpr int64_t kStaticScatterKeys = int64_t(1) << 20;

int64_t scatter_npow2(int64_t n);
size_t scatter_workspace_bytes(int64_t n);
psg_status static_scatter_keys(unsigned long long** out);
psg_status launch_gather(const GatherLaunch& L, void* stream);
// keys: device scratch of scatter_workspace_bytes(n), 16-byte aligned
psg_status launch_scatter(const ScatterLaunch& L, unsigned long long* keys, void* stream);

}  // namespace psg
