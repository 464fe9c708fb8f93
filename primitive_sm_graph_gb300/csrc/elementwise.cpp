// psg_elementwise: plan (views -> iteration space -> operand modes), generate
// the program body, fetch the runtime-specialised kernel, launch it.
#include <cuda_runtime.h>

#include <cstring>

#include "api_internal.h"
#include "codegen.h"
#include "jit.h"
#include "launch_util.cuh"

namespace psg {

namespace {
constexpr int EW_THREADS = 256;

constexpr int EW_BLOCKS_PER_SM = 8;  // 2048 resident threads per SM at 256 a block

int group_log2_for(int64_t chunks)
{
    int g = 0;
    while ((1 << g) < chunks && (1 << g) < EW_THREADS) ++g;
    return g;
}

// Cut rows into column tiles when there are too few rows to give every
// resident group of a full wave its own item; a tile is a multiple of the
// group size, so each thread still walks whole chunks.
void choose_tiles(int64_t rows, int64_t chunks, int gl, long long* tiles, long long* tile_chunks)
{
    const int64_t g = (int64_t)1 << gl;
    const int64_t want = (int64_t)num_sms() * EW_BLOCKS_PER_SM * (EW_THREADS >> gl);
    *tiles = 1;
    *tile_chunks = chunks > 0 ? chunks : 1;
    if (rows <= 0 || rows >= want || chunks <= g) return;
    const int64_t per_row = (want + rows - 1) / rows;
    int64_t tc = (chunks + per_row - 1) / per_row;
    tc = (tc + g - 1) / g * g;
    *tile_chunks = tc;
    *tiles = (chunks + tc - 1) / tc;
}
}  // namespace

psg_status plan_elementwise(const psg_node* prog, int n_nodes, const void* const* in,
                            const psg_view* in_v, int n_in, void* out, const psg_view* out_v,
                            EwPlan* P)
{
    if (!prog || n_nodes < 1 || n_nodes > PSG_MAX_NODES) return PSG_E_INVALID_ARG;
    if (n_in < 0 || n_in > PSG_MAX_INPUTS) return PSG_E_INVALID_ARG;
    if (n_in > 0 && (!in || !in_v)) return PSG_E_INVALID_ARG;
    if (!out_v) return PSG_E_INVALID_ARG;
    psg_status st = check_view(out_v, true);
    if (st != PSG_OK) return st;
    const int64_t n = view_numel(out_v);
    if (n > 0 && !out) return PSG_E_INVALID_ARG;
    if (!ptr_aligned(out, out_v->dtype)) return PSG_E_MISALIGNED;
    const psg_view* views[1 + PSG_MAX_INPUTS];
    views[0] = out_v;
    int dts[PSG_MAX_INPUTS];
    for (int k = 0; k < n_in; ++k) {
        st = check_view(&in_v[k], false);
        if (st != PSG_OK) return st;
        if (!same_shape(&in_v[k], out_v)) return PSG_E_INVALID_ARG;
        if (n > 0 && !in[k]) return PSG_E_INVALID_ARG;
        if (!ptr_aligned(in[k], in_v[k].dtype)) return PSG_E_MISALIGNED;
        views[1 + k] = &in_v[k];
        dts[k] = in_v[k].dtype;
    }
    std::memset(&P->p, 0, sizeof(P->p));
    Space sp;
    int64_t strides[1 + PSG_MAX_INPUTS][MAXD], lo[1 + PSG_MAX_INPUTS][MAXD], hi[1 + PSG_MAX_INPUTS][MAXD];
    bool masked[1 + PSG_MAX_INPUTS];
    st = build_space(views, 1 + n_in, false, &sp, strides, lo, hi, masked);
    if (st != PSG_OK) return st;
    bool uni[PSG_MAX_INPUTS];
    int modes[PSG_MAX_INPUTS];
    for (int k = 0; k < n_in; ++k) {
        modes[k] = fill_operand(P->p.in[k], in[k], &in_v[k], sp, strides[1 + k], lo[1 + k], hi[1 + k],
                                masked[1 + k]);
        modes[k] = vec_mode(modes[k], P->p.in[k], dtype_size(dts[k]), sp);
        uni[k] = modes[k] == PSG_M_UNIFORM;
    }
    const int out_mode = vec_mode(fill_operand(P->p.out, out, out_v, sp, strides[0], lo[0], hi[0], false),
                                  P->p.out, dtype_size(out_v->dtype), sp);
    ProgInfo I;
    st = analyze_program(prog, n_nodes, dts, uni, n_in, nullptr, 0, &I);
    if (st != PSG_OK) return st;
    if (I.result_dtype != out_v->dtype) return PSG_E_UNSUPPORTED_DTYPE;
    P->p.rows = sp.rows;
    P->p.inner = sp.inner;
    P->p.chunks = sp.chunks;
    for (int d = 0; d < MAXD; ++d) P->p.shape[d] = d < sp.nd ? sp.shape[d] : 1;
    P->p.nd = sp.nd;
    P->p.group_log2 = group_log2_for(sp.chunks);
    choose_tiles(sp.rows, sp.chunks, P->p.group_log2, &P->p.tiles, &P->p.tile_chunks);
    P->n_in = n_in;
    // the specialisation: input modes and dtypes, output dtype, the body
    std::string spec = "constexpr int kNin = " + std::to_string(n_in) + ";\n";
    std::string m = "constexpr int kInMode[] = {", d = "constexpr int kInDt[] = {";
    for (int k = 0; k < (n_in > 0 ? n_in : 1); ++k) {
        m += std::to_string(k < n_in ? modes[k] : 0) + (k + 1 < n_in ? ", " : "");
        d += std::to_string(k < n_in ? dts[k] : 0) + (k + 1 < n_in ? ", " : "");
    }
    spec += m + "};\n" + d + "};\n";
    spec += "constexpr int kOutDt = " + std::to_string(out_v->dtype) + ";\n";
    spec += "constexpr int kOutMode = " + std::to_string(out_mode) + ";\n";
    spec += std::string("constexpr bool kExact = ") + (sp.inner % PSG_VEC == 0 ? "true" : "false") + ";\n";
    spec += gen_eval(prog, I, "Body", "", -1, true);  // the result only goes to st_chunk
    P->spec = std::move(spec);
    return PSG_OK;
}

static psg_status grid_for(const EwPlan& P, cudaKernel_t k, int* grid)
{
    const int groups = EW_THREADS >> P.p.group_log2;
    const int64_t need = (P.p.rows * P.p.tiles + groups - 1) / groups;
    const int per_sm = jit_max_blocks_per_sm(k, EW_THREADS, 0);
    const int64_t cap = (int64_t)num_sms() * per_sm;
    *grid = (int)std::max<int64_t>(1, std::min<int64_t>(need, cap));
    return PSG_OK;
}

psg_status launch_elementwise(const EwPlan& P, void* stream)
{
    if (P.p.rows == 0 || P.p.inner == 0) return PSG_OK;
    cudaKernel_t k;
    psg_status st = jit_kernel(JIT_EW, P.spec, "psg_ew", &k);
    if (st != PSG_OK) return st;
    int grid;
    grid_for(P, k, &grid);
    void* args[] = {(void*)&P.p};
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config(dim3(grid), dim3(EW_THREADS), 0, (cudaStream_t)stream, attr);
    if (cudaLaunchKernelExC(&cfg, (const void*)k, args) != cudaSuccess) return PSG_E_CUDA;
    return PSG_OK;
}

psg_status query_elementwise(const EwPlan& P, int* grid, int* block, int* smem, int* regs)
{
    cudaKernel_t k;
    psg_status st = jit_kernel(JIT_EW, P.spec, "psg_ew", &k);
    if (st != PSG_OK) return st;
    grid_for(P, k, grid);
    *block = EW_THREADS;
    *smem = 0;
    *regs = jit_regs(k);
    return PSG_OK;
}

}  // namespace psg
