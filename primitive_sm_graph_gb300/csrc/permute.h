// Launch descriptors of the permute kernels.
#pragma once

#include "common.h"

namespace psg {

// 2-D tiled transpose over a batch: out[b, a, i] = in[b, i, a], where a is the
// input's stride-1 dim and i the output's stride-1 dim (strides in elements).
struct TransposeLaunch {
    const void* in;
    void* out;
    int32_t es;          // element size in bytes
    int32_t nb;          // batch dims
    int64_t A, I;
    int64_t in_si;       // input stride along i
    int64_t out_sa;      // output stride along a
    int64_t in_offset, out_offset;
    int64_t batch;
    int64_t bshape[MAXD], in_bstride[MAXD], out_bstride[MAXD];
};

// Per-cell strided copy (any element size, masked reads give zeros).
struct CopyLaunch {
    const void* in;
    void* out;
    int32_t es;
    int32_t nd;
    int64_t numel;
    int64_t in_offset, out_offset;
    int64_t shape[MAXD], in_stride[MAXD], out_stride[MAXD], mlo[MAXD], mhi[MAXD];
};

psg_status launch_transpose(const TransposeLaunch& L, void* stream);
psg_status launch_copy(const CopyLaunch& L, void* stream);
void query_transpose(int es, int64_t tiles, int* grid, int* block, int* smem, int* regs);

}  // namespace psg
