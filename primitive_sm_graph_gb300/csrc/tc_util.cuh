// Helpers shared by the tensor-core kernels (sm_103a): the device helpers of
// jit/tc_device.cuh (mbarriers with bounded waits, TMA, tcgen05, CTA pairs,
// tile order) in this namespace, and the tensor-map encoder entry point.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "common.h"

namespace psg {
namespace tcu {
namespace {  // internal linkage: each kernel file gets its own copy

#include "jit/tc_device.cuh"

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    });
    return fn;
}

}  // namespace
}  // namespace tcu
}  // namespace psg
