// Internal definitions shared by the host planner and the sm_103a kernels.
// Not part of the public ABI (that is include/psg.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include "psg.h"

#ifdef __CUDACC__
#define PSG_HD __host__ __device__
#else
#define PSG_HD
#endif

namespace psg {

// ---------------------------------------------------------------------------
// Register-form interpreter.
//
// A program (psg_node list) is compiled on the host into a short list of
// instructions over R registers.  Every register holds VEC 32-bit lanes: the
// VEC consecutive cells along the innermost dim that one thread owns.  Each
// instruction names its registers in its form id, so the kernel's switch lands
// on straight-line code whose register indices are compile-time constants: no
// per-thread dynamic indexing, no local memory.  A "scalar" instruction works
// on lane 0 only; the host sets it when every operand is uniform along the
// inner dim (a stride-0 broadcast, a constant, a reduced row value), so a
// value like LOG(b*b + 1) of an expanded column is computed once per thread
// instead of VEC times (stride-0 loops reuse their operand: Luminal IR blog,
// "ZeroStrideLoop").  BCAST copies lane 0 to all lanes where a uniform value
// meets a varying one.
// ---------------------------------------------------------------------------
constexpr int R = 6;          // registers
constexpr int VEC = 8;        // lanes (cells per thread chunk)
constexpr int MAX_INS = 96;   // instructions per program
constexpr int MAX_IN = PSG_MAX_INPUTS;
constexpr int MAX_STAGES = 4;

enum Opc : int {
    OP_NOP = 0,
    // two-register forms: r[d] = f(r[d], r[s])
    OP_MOV, OP_ADDF, OP_MULF, OP_LTF, OP_ADDI, OP_MULI, OP_LTI, OP_SEL,
    // one-register forms, in place on r[d]
    OP_NEGF, OP_NEGI, OP_EXP, OP_LOG, OP_SQRT, OP_RCP, OP_RBF16, OP_RF16, OP_F2I, OP_I2F,
    OP_W8, OP_W16, OP_PREDF, OP_PREDI, OP_CONST, OP_BCAST,
    // r[d] = input k / reduced stage value s
    OP_LD, OP_LDRED,
    OP_COUNT
};

PSG_HD constexpr int form_id(int op, int d, int s) { return (op << 6) | (d << 3) | s; }

struct Ins {
    uint16_t form;
    uint8_t scalar;
    uint8_t pad;
    uint32_t imm;  // OP_CONST bits
};

struct Program {
    int32_t n;
    int32_t out_reg;
    Ins ins[MAX_INS];
};

enum DClass { DC_FLOAT = 0, DC_INT = 1 };

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

// Host: compile a program.  in_dtype/in_uniform describe the kernel's inputs
// (uniform = constant along the thread's VEC lanes); red_dtype the reduced
// stage values a program may read (n_red = 0 forbids PSG_OP_RED).
// result_dtype receives the last node's dtype; result_uniform whether the
// result is uniform (then a BCAST is appended when bcast_result).
psg_status compile_program(const psg_node* nodes, int n, const int* in_dtype,
                           const bool* in_uniform, int n_in, const int* red_dtype, int n_red,
                           bool bcast_result, Program* out, int* result_dtype,
                           bool* result_uniform);

// ---------------------------------------------------------------------------
// Iteration space and operand descriptors after dim collapsing.
// Dims 0..nd-2 are "outer" (one row = one outer multi-index), dim nd-1 is the
// inner dim that threads walk VEC cells at a time.
// ---------------------------------------------------------------------------
constexpr int MAXD = PSG_MAX_DIMS;

enum InMode : int32_t {
    IN_UNIFORM = 0,  // inner stride 0 and no inner mask: one value per row
    IN_CONTIG = 1,   // inner stride 1, no mask: vector loads when aligned
    IN_STRIDED = 2,  // any inner stride, no mask
    IN_MASKED = 3    // has a mask somewhere: per-cell range checks
};

struct Operand {
    const void* ptr;
    int32_t dtype;
    int32_t mode;
    int64_t offset;
    int64_t inner_stride;
    int64_t outer_stride[MAXD];
    int64_t mlo[MAXD], mhi[MAXD];  // per iteration dim (IN_MASKED only)
};

struct Space {
    int32_t nd;                // iteration dims, >= 1
    int32_t pad;
    int64_t shape[MAXD];       // iteration shape
    int64_t rows;              // product of shape[0..nd-2]
    int64_t inner;             // shape[nd-1]
    int64_t chunks;            // ceil(inner / VEC)
};

// Host helpers (view.cpp)
psg_status check_view(const psg_view* v, bool for_write);
int64_t view_numel(const psg_view* v);
bool view_has_mask(const psg_view* v);
bool view_contiguous(const psg_view* v);

// Build the common iteration space of n views (outputs first), ordering dims
// by the first view's strides (its stride-1 dim innermost) and merging dims
// that are contiguous in every view.  keep_last keeps the last dim of the
// views as the inner dim (reductions).  perm_out receives, for each iteration
// dim, the original dim it came from after merging (informational).
psg_status build_space(const psg_view* const* views, int nviews, bool keep_last, Space* sp,
                       int64_t (*strides)[MAXD], int64_t (*mlo)[MAXD], int64_t (*mhi)[MAXD],
                       bool* masked);

// Launchers (one per .cu file); return PSG_E_CUDA on a launch error.
struct EwLaunch {
    Program prog;
    Space sp;
    int32_t n_in;
    int32_t out_uniform;
    Operand in[MAX_IN];
    Operand out;
};
psg_status launch_elementwise(const EwLaunch& L, void* stream);
void query_elementwise(const EwLaunch* L, int* grid, int* block, int* smem, int* regs);

}  // namespace psg
