/* Launch parameters of the tensor-core contraction kernels, shared by the
 * host planner (contract.h includes this inside namespace psg) and the
 * kernels, compiled by nvcc and, for a fused epilogue, by NVRTC.  Plain C
 * types only. */
#ifndef PSG_GEMM_PARAMS_H
#define PSG_GEMM_PARAMS_H

#ifndef PSG_DT_F32
#define PSG_DT_F32 0
#define PSG_DT_BF16 1
#define PSG_DT_F16 2
#endif

#define PSG_TC_MAX_EPI_IN 8

/* one input of a fused epilogue program, read at C's cell (b, m, n) */
struct TcEpiOperand {
    const void* ptr;           /* at the View's offset */
    long long sb, sm, sn;      /* element strides along batch, m, n */
};

struct TcParams {
    int M, N, K, batch;
    int a_kmajor, b_kmajor;     /* 1: k stride 1; 0: m (n) stride 1 */
    int num_m, num_n, num_k;    /* tile counts (filled by the launcher) */
    int c_dtype;
    int ab_dtype;               /* bf16 or f16 (tc_gemm), f32 (tc_gemm_tf32x3) */
    int splits, kb_per;         /* split-K: K-block ranges per tile (1: none) */
    float* ws;                  /* split-K partials [splits][batch][M][N] float32 */
    void* C;
    int* status;
    long long c_offset, c_rs, c_cs, c_bs;
    int tma_store;              /* 1: the epilogue writes C (or the partials) through a tensor map */
    int reduce_quad;            /* split-K reduce: 1 when C's rows take 4-cell vector moves */
    int n_epi;                  /* inputs of the fused epilogue program (0: none) */
    int pad_epi;
    struct TcEpiOperand epi[PSG_TC_MAX_EPI_IN];
};

#endif
