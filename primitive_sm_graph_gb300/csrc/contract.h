// Launch descriptors of the MUL+SUM contraction kernels.
#pragma once

#include <string>

#include "common.h"

namespace psg {

#include "jit/gemm_params.h"

// The runtime-compiled part of a contraction with a fused epilogue: the
// operand tables and the program body (gen_eval's EpiProg) of the spec; the
// launcher adds the kernel entry point of the variant it runs.
struct EpiSpec {
    std::string tables, prog;
};

struct TcOperands {
    TcParams p;
    const EpiSpec* epi;         // fused epilogue program, or null
    void* ws;                   // caller workspace for split-K partials (may be null)
    size_t ws_bytes;
    const void* A;  // at the View's offset
    const void* B;
    int64_t a_ms, a_ks, a_bs;   // element strides of A along m, k, batch
    int64_t b_ns, b_ks, b_bs;
};

struct SimtParams {
    const void* A;
    const void* B;
    void* C;
    int32_t ab_dtype, c_dtype;
    int64_t M, N, K, batch;
    int64_t a_off, a_ms, a_ks, a_bs;
    int64_t b_off, b_ns, b_ks, b_bs;
    int64_t c_off, c_ms, c_ns, c_bs;
    // read windows (masks clipped to the shape; empty when the operand reads
    // nothing): A along m and k, B along n and k; cells outside the c window
    // (B's m mask, A's n mask, a batch mask) are written 0
    int64_t a_mlo, a_mhi, a_klo, a_khi;
    int64_t b_nlo, b_nhi, b_klo, b_khi;
    int64_t c_mlo, c_mhi, c_nlo, c_nhi;
};

psg_status launch_contract_tc(const TcOperands& o, void* stream);
// the JIT_GEMM spec of a fused epilogue for the single-CTA (pair false) or
// CTA-pair kernel
std::string epi_spec_source(const EpiSpec& e, bool pair);
// split-K plan of the bf16 / f16 kernel: splits (1 = none) and the
// workspace bytes they need, for an output of tiles that leaves SMs idle
int contract_tc_splits(int64_t M, int64_t N, int64_t K, int64_t batch, size_t* bytes);
// launch shape for an output of M rows in `tiles` 128 x 256 tiles: the CTA-pair
// kernel (two CTAs a 256 x 256 tile) when M > 128, else the single-CTA one
void query_contract_tc(int64_t M, int64_t tiles, int* grid, int* block, int* smem, int* regs);
// float32 operands, 3xTF32 on the tensor cores (same operand rules as the bf16 path)
psg_status launch_contract_tf32(const TcOperands& o, void* stream);
void query_contract_tf32(int64_t tiles, int* grid, int* block, int* smem, int* regs);
psg_status launch_contract_simt(const SimtParams& p, void* stream);
void query_contract_simt(const SimtParams& p, int* grid, int* block, int* smem, int* regs);

}  // namespace psg
