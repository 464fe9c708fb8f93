// Launch helpers: SM count, occupancy and register counts, cached per device,
// and the launch used by every kernel of the library.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <utility>

namespace psg {

int current_device();
int num_sms();                                                 // of the current device
int max_blocks_per_sm(const void* fn, int threads, size_t smem);  // occupancy, >= 1
int kernel_regs(const void* fn);
size_t l2_bytes();
// cudaFuncSetAttribute(fn, MaxDynamicSharedMemorySize, bytes) on the current
// device, made once per (device, kernel, bytes) and remembered; the attribute
// belongs to a device, so a process that drives several GPUs sets it on each
cudaError_t set_max_dynamic_smem(const void* fn, int bytes);

// Programmatic dependent launch.  Every kernel of this library begins with
// pdl_enter(): griddepcontrol.wait holds it until the kernel before it on the
// stream has finished and that kernel's writes are visible, and only then does
// it read or write memory; griddepcontrol.launch_dependents then lets the
// next kernel be scheduled.  Launched with programmatic stream serialization,
// a kernel's launch and block scheduling overlap its predecessor's tail
// instead of following it; the data dependency is unchanged.  (A kernel that
// follows something other than a kernel, or a kernel launched without the
// attribute, waits as usual; the wait then returns at once.)
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

// true unless PSG_NO_PDL is set in the environment (read once): then every
// launch serialises in the ordinary way
bool pdl_enabled();

inline cudaLaunchConfig_t launch_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                        cudaLaunchAttribute* attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cfg;
}

// k<<<grid, block, smem, s>>>(args...) with programmatic stream serialization;
// the error is also left for cudaGetLastError(), as a <<< >>> launch does
template <typename... P, typename... A>
cudaError_t launch(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, A&&... args)
{
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config(grid, block, smem, s, attr);
    return cudaLaunchKernelEx(&cfg, k, std::forward<A>(args)...);
}

}  // namespace psg
