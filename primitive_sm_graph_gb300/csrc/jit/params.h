// Launch parameters shared by the host planner and the runtime-compiled
// kernels.  Plain C types only: this file is compiled by the host compiler and
// by NVRTC (which sees it as text), so both sides agree on the layout.
#ifndef PSG_JIT_PARAMS_H
#define PSG_JIT_PARAMS_H

#define PSG_VEC 8      /* cells per thread chunk along the inner dim */
#define PSG_MAXD 8
#define PSG_MAXIN 8
#define PSG_MAXSTAGES 4

/* dtype codes: the same values as psg_dtype in psg.h */
#define PSG_DT_F32 0
#define PSG_DT_BF16 1
#define PSG_DT_F16 2
#define PSG_DT_F64 3
#define PSG_DT_I32 4
#define PSG_DT_I16 5
#define PSG_DT_I8 6

/* how an operand is addressed along the inner dim */
#define PSG_M_UNIFORM 0  /* inner stride 0, unmasked inner dim: one value per row */
#define PSG_M_CONTIG 1   /* inner stride 1, unmasked: vector loads when aligned */
#define PSG_M_STRIDED 2  /* any inner stride, unmasked */
#define PSG_M_MASKED 3   /* masked somewhere: per-cell range checks */
#define PSG_M_VEC 4      /* contiguous, every row start 16-byte aligned: vector moves only */

struct PsgOperand {
    const void* ptr;
    long long offset;
    long long inner_stride;
    long long outer_stride[PSG_MAXD];  /* per outer iteration dim */
    long long mlo[PSG_MAXD];           /* mask per iteration dim (masked mode) */
    long long mhi[PSG_MAXD];
};

/* Iteration space [shape[0] .. shape[nd-2]] rows x inner; one output. */
struct PsgEwParams {
    long long rows;
    long long inner;
    long long chunks;      /* ceil(inner / PSG_VEC) */
    long long tiles;       /* column tiles per row: work items are (row, tile) */
    long long tile_chunks; /* chunks per tile (a multiple of the group size) */
    long long shape[PSG_MAXD];
    int nd;
    int group_log2;        /* threads per row group = 1 << group_log2 */
    struct PsgOperand in[PSG_MAXIN];
    struct PsgOperand out;
};

/* device-reported status the generated kernels write (= PSG_E_TIMEOUT) */
#define PSG_DEV_E_TIMEOUT 7

/* Row reduction: every input has the iteration shape [rows.., N]; the
 * output is [rows.., N] (per-element epilogue) or [rows..] (per-row). */
struct PsgRedParams {
    long long rows;
    long long inner;       /* N, the reduced length */
    long long chunks;
    long long shape[PSG_MAXD];
    int nd;
    int team_log2;         /* threads per row = 1 << team_log2 */
    int out_per_row;       /* 1: one output per row; 0: per element */
    int pad;
    int* status;           /* device status word (PSG_E_TIMEOUT), may be null */
    long long wait_cycles; /* bound of each staged-ring wait, in SM clock cycles */
    int skip_first_copy;   /* test hook: 1 leaves every team's first ring slot unfilled */
    int pad2;
    struct PsgOperand in[PSG_MAXIN];
    struct PsgOperand out;
};

#endif
