// Runtime specialisation: NVRTC compiles a hand-written kernel skeleton
// together with a generated program body for sm_103a; the result is cached
// for the life of the process, keyed by the full source text.
#pragma once

#include <cuda_runtime.h>

#include <string>

#include "common.h"

namespace psg {

enum JitSkeleton { JIT_EW = 0, JIT_REDUCE = 1, JIT_GEMM = 2 };

// Full source: params + prelude + `spec` (constexpr tables and bodies) + skeleton.
// JIT_GEMM: the tensor-core contraction with a fused epilogue; `spec` is the
// operand tables, a '\x01', then the program body and the kernel entry point,
// around the skeleton's device helpers, kernel bodies and epilogue context.
std::string jit_source(JitSkeleton sk, const std::string& spec);

// Compile (or fetch from the cache) the kernel `name` of skeleton `sk`
// specialised by `spec`.  The cache is keyed by (sk, spec), so a hit costs a
// hash of the short spec only.  Returns PSG_E_CUDA on a compile or load
// failure (the NVRTC log is printed to stderr when PSG_JIT_VERBOSE is set).
psg_status jit_kernel(JitSkeleton sk, const std::string& spec, const char* name, cudaKernel_t* out);

// Compile only (no device needed); for host-side checks of generated code.
psg_status jit_compile_only(const std::string& src, std::string* log);

int jit_max_blocks_per_sm(cudaKernel_t k, int threads, size_t smem);
int jit_regs(cudaKernel_t k);

}  // namespace psg
