// psg_reduce_rows: validate stages and epilogue, build the iteration space
// (the reduced axis stays last), choose the team size and whether the row is
// cached in registers, generate the bodies, launch the specialised kernel.
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <unordered_map>
#include <mutex>

#include "api_internal.h"
#include "codegen.h"
#include "jit.h"
#include "launch_util.cuh"

namespace psg {

namespace {
constexpr int RED_THREADS = 256;      // the skeleton's launch bound (row teams)
constexpr int RED_REG_THREADS = 128;  // rows held in registers by teams of at most this many threads
constexpr int RED_COL_THREADS = 512;  // columnar layout: at most 16 members a CTA
static_assert(PSG_DEV_E_TIMEOUT == PSG_E_TIMEOUT, "device status code");
}  // namespace

namespace {

struct RedPlan {
    PsgRedParams p;
    int block;
    int smem;     // dynamic shared memory (staged mode)
    int cluster;  // CTAs per cluster (columnar layout), else 1
    std::string spec;
};

std::string int_list(const int* v, int n)
{
    std::string s = "{";
    for (int i = 0; i < (n > 0 ? n : 1); ++i) s += std::to_string(i < n ? v[i] : 0) + (i + 1 < n ? ", " : "");
    return s + "}";
}

psg_status plan_reduce(const psg_reduce_stage* stages, int n_stages, const psg_node* epilogue, int n_epi,
                       const void* const* in, const psg_view* in_v, int n_in, void* out,
                       const psg_view* out_v, RedPlan* P)
{
    if (!stages || n_stages < 1 || n_stages > MAX_STAGES) return PSG_E_INVALID_ARG;
    if (n_in < 1 || n_in > PSG_MAX_INPUTS || !in || !in_v || !out_v) return PSG_E_INVALID_ARG;
    if (n_epi < 0 || (n_epi > 0 && !epilogue)) return PSG_E_INVALID_ARG;
    const int nd = in_v[0].ndim;
    if (nd < 1) return PSG_E_INVALID_ARG;
    psg_status st;
    int dts[PSG_MAX_INPUTS];
    for (int k = 0; k < n_in; ++k) {
        st = check_view(&in_v[k], false);
        if (st != PSG_OK) return st;
        if (!same_shape(&in_v[k], &in_v[0])) return PSG_E_INVALID_ARG;
        if (in_v[k].dtype == PSG_F64) return PSG_E_UNSUPPORTED_DTYPE;
        if (view_numel(&in_v[k]) > 0 && !in[k]) return PSG_E_INVALID_ARG;
        if (!ptr_aligned(in[k], in_v[k].dtype)) return PSG_E_MISALIGNED;
        dts[k] = in_v[k].dtype;
    }
    st = check_view(out_v, true);
    if (st != PSG_OK) return st;
    if (out_v->dtype == PSG_F64) return PSG_E_UNSUPPORTED_DTYPE;
    if (view_numel(out_v) > 0 && !out) return PSG_E_INVALID_ARG;
    if (!ptr_aligned(out, out_v->dtype)) return PSG_E_MISALIGNED;
    const int64_t N = in_v[0].shape[nd - 1];
    // output form: per element [.., N], or per row [..] / [.., 1]
    bool per_row;
    bool lead_match = true;
    for (int d = 0; d < nd - 1; ++d)
        if (out_v->ndim > d && out_v->shape[d] != in_v[0].shape[d]) lead_match = false;
    if (!lead_match) return PSG_E_INVALID_ARG;
    if (out_v->ndim == nd && out_v->shape[nd - 1] == N) per_row = false;
    else if (out_v->ndim == nd && out_v->shape[nd - 1] == 1) per_row = true;
    else if (out_v->ndim == nd - 1) per_row = true;
    else return PSG_E_INVALID_ARG;
    // the output as a view over the iteration shape (stride 0 along N when per row)
    psg_view ov = in_v[0];
    ov.dtype = out_v->dtype;
    ov.offset = out_v->offset;
    ov.extent = out_v->extent;
    for (int d = 0; d < nd; ++d) {
        ov.mask_lo[d] = 0;
        ov.mask_hi[d] = ov.shape[d];
        ov.strides[d] = d < nd - 1 ? out_v->strides[d] : (per_row ? 0 : out_v->strides[nd - 1]);
    }
    const psg_view* views[1 + PSG_MAX_INPUTS];
    views[0] = &ov;
    for (int k = 0; k < n_in; ++k) views[1 + k] = &in_v[k];
    std::memset(&P->p, 0, sizeof(P->p));
    Space sp;
    int64_t strides[1 + PSG_MAX_INPUTS][MAXD], lo[1 + PSG_MAX_INPUTS][MAXD], hi[1 + PSG_MAX_INPUTS][MAXD];
    bool masked[1 + PSG_MAX_INPUTS];
    st = build_space(views, 1 + n_in, true, &sp, strides, lo, hi, masked);
    if (st != PSG_OK) return st;
    bool uni[PSG_MAX_INPUTS];
    int modes[PSG_MAX_INPUTS];
    for (int k = 0; k < n_in; ++k) {
        modes[k] = fill_operand(P->p.in[k], in[k], &in_v[k], sp, strides[1 + k], lo[1 + k], hi[1 + k],
                                masked[1 + k]);
        modes[k] = vec_mode(modes[k], P->p.in[k], dtype_size(dts[k]), sp);
        uni[k] = modes[k] == PSG_M_UNIFORM;
    }
    const int out_mode = vec_mode(fill_operand(P->p.out, out, &ov, sp, strides[0], lo[0], hi[0], false),
                                  P->p.out, dtype_size(out_v->dtype), sp);
    // float64 nodes run in psg_elementwise only: the row kernels keep 32-bit
    // running totals and register caches
    for (int s = 0; s < n_stages; ++s)
        for (int i = 0; i < stages[s].n_nodes && stages[s].prologue; ++i)
            if (stages[s].prologue[i].dtype == PSG_F64) return PSG_E_UNSUPPORTED_DTYPE;
    for (int i = 0; i < n_epi; ++i)
        if (epilogue[i].dtype == PSG_F64) return PSG_E_UNSUPPORTED_DTYPE;
    // stages
    std::string bodies;
    int sop[MAX_STAGES], sdt[MAX_STAGES];
    for (int s = 0; s < n_stages; ++s) {
        if (stages[s].op != PSG_RED_SUM && stages[s].op != PSG_RED_MAX) return PSG_E_INVALID_ARG;
        ProgInfo I;
        st = analyze_program(stages[s].prologue, stages[s].n_nodes, dts, uni, n_in, sdt, s, &I);
        if (st != PSG_OK) return st;
        sop[s] = stages[s].op;
        sdt[s] = I.result_dtype;
        bodies += gen_eval(stages[s].prologue, I, "StageBody<" + std::to_string(s) + ">", "template <>\n");
    }
    // epilogue (a per-row epilogue may read only constants and stage values)
    psg_node last_red;
    std::memset(&last_red, 0, sizeof(last_red));
    const psg_node* epi = epilogue;
    if (n_epi == 0) {
        if (!per_row) return PSG_E_INVALID_ARG;
        last_red.op = PSG_OP_RED;
        last_red.a = n_stages - 1;
        last_red.dtype = sdt[n_stages - 1];
        epi = &last_red;
        n_epi = 1;
    }
    ProgInfo E;
    st = per_row ? analyze_program(epi, n_epi, dts, uni, 0, sdt, n_stages, &E)
                 : analyze_program(epi, n_epi, dts, uni, n_in, sdt, n_stages, &E);
    if (st != PSG_OK) return st;
    if (E.result_dtype != out_v->dtype) return PSG_E_UNSUPPORTED_DTYPE;
    // which inputs the register cache holds: those that vary from row to row
    // (a row-invariant operand, like a norm's weight, stays in L1 and is
    // read again); bfloat16 rows are held packed, two cells a word
    int cache_in[PSG_MAX_INPUTS];
    int words = 0;
    for (int k = 0; k < n_in; ++k) {
        bool row_inv = modes[k] != PSG_M_MASKED;
        for (int d = 0; d + 1 < sp.nd; ++d)
            if (P->p.in[k].outer_stride[d] != 0) row_inv = false;
        cache_in[k] = !uni[k] && !row_inv;
        if (cache_in[k]) words += dts[k] == PSG_BF16 ? PSG_VEC / 2 : PSG_VEC;
    }
    // an epilogue that starts with a stage's whole program reuses that
    // stage's per-cell values (softmax: EXP(x - m) is computed once)
    int stash = -1;
    if (!per_row) {
        for (int s = n_stages - 1; s >= 0 && stash < 0; --s) {
            const int m = stages[s].n_nodes;
            if (m > n_epi || E.val[m - 1] != m - 1 || E.uni[m - 1] || !E.live[m - 1]) continue;
            bool same = true;
            for (int i = 0; i < m && same; ++i) {
                const psg_node &x = stages[s].prologue[i], &y = epi[i];
                same = x.op == y.op && x.a == y.a && x.b == y.b && x.c == y.c && x.dtype == y.dtype &&
                       std::memcmp(&x.cval, &y.cval, sizeof(double)) == 0;
            }
            if (same && m < n_epi) stash = s;
        }
    }
    // columnar layout: the rows are adjacent in memory and the reduced axis
    // is strided (a sum over a leading axis).  Every input that varies from
    // row to row must then move by 0 or 1 cell from one row to the next
    // (the last row dim), one of them by 1; inputs the rows share may be
    // contiguous along the reduced axis (every lane reads the same cells).
    bool columnar = sp.nd >= 2 && sp.rows > 1;
    bool unit_row = false;
    for (int k = 0; k < n_in && columnar; ++k) {
        if (uni[k]) continue;
        const int64_t rs = sp.shape[sp.nd - 2] > 1 ? P->p.in[k].outer_stride[sp.nd - 2] : 0;
        if (modes[k] == PSG_M_MASKED || (rs != 0 && rs != 1)) columnar = false;
        if (rs == 1 && modes[k] == PSG_M_STRIDED) unit_row = true;
        if (rs == 1 && modes[k] != PSG_M_STRIDED) columnar = false;
    }
    columnar = columnar && unit_row;
    // team of T threads per row.  A thread takes about RED_CHUNKS chunks, so
    // each issues several 16- or 32-byte loads at once and short rows fold
    // inside one warp (shuffles only); the row (and a stash) is cached in
    // registers when it fits in RED_CACHE_WORDS words per thread.
    constexpr int RED_CHUNKS = 4, RED_CHUNKS_WIDE = 8, RED_CACHE_WORDS = 64, RED_MAX_TEAM_LOG2 = 8;
    int tl = 0;
    while ((int64_t)RED_CHUNKS << tl < sp.chunks && tl < RED_MAX_TEAM_LOG2) ++tl;
    // staged mode: when every input that changes from row to row is
    // contiguous, 16-byte aligned at every row start and at least
    // RED_STAGE_MIN_BYTES a row, the rows come through a shared-memory ring of
    // kNS slots per team filled by bulk copies (kNS - 1 rows in flight while
    // the team computes); the stages and the epilogue read them from there.
    constexpr int RED_STAGED_MAX_CHUNKS = 16, RED_STAGE_MIN_BYTES = 512;
    // the ring is kept near RED_SMEM_PREF a block so that three blocks fit an
    // SM: more teams in flight beat a deeper ring (RMSNorm: 26.2 us with two
    // blocks of 3-slot rings, 25.3 us with three blocks of 2-slot rings)
    constexpr int64_t RED_SMEM_PREF = 72 * 1024, RED_SMEM_MAX = 200 * 1024;
    int staged_in[PSG_MAX_INPUTS] = {0}, seg_off[PSG_MAX_INPUTS] = {0}, row_bytes[PSG_MAX_INPUTS] = {0},
        in_size[PSG_MAX_INPUTS] = {0};
    int64_t stage_bytes = 0, tx_bytes = 0;
    bool staged = words > 0 && !columnar;
    for (int k = 0; k < n_in; ++k) {
        in_size[k] = dtype_size(dts[k]);
        if (!cache_in[k]) continue;
        const int es = in_size[k];
        const bool dt_ok = dts[k] == PSG_F32 || dts[k] == PSG_I32 || dts[k] == PSG_BF16 || dts[k] == PSG_F16;
        bool ok = dt_ok && (modes[k] == PSG_M_CONTIG || modes[k] == PSG_M_VEC) && P->p.in[k].inner_stride == 1 &&
                  ((uintptr_t)in[k] + (uint64_t)P->p.in[k].offset * es) % 16 == 0 && (sp.inner * es) % 16 == 0;
        for (int d = 0; d + 1 < sp.nd && ok; ++d)
            if (sp.shape[d] > 1 && (P->p.in[k].outer_stride[d] * es) % 16 != 0) ok = false;
        if (!ok) staged = false;
        staged_in[k] = 1;
        seg_off[k] = (int)stage_bytes;
        row_bytes[k] = (int)(sp.inner * es);
        stage_bytes += (sp.chunks * PSG_VEC * es + 127) / 128 * 128;
        tx_bytes += sp.inner * es;
    }
    if (tx_bytes < RED_STAGE_MIN_BYTES) staged = false;
    // a staged row longer than a warp's RED_CHUNKS chunks gives each thread
    // RED_CHUNKS_WIDE chunks (it reads them from shared memory, so registers
    // do not grow), and the per-row costs (the fold across warps, the row's
    // uniform values) are shared by more cells (measured: RMSNorm over 4096
    // bf16 cells a row, 28.7 us with 128-thread teams of 4 chunks, 25.3 us
    // with 64-thread teams of 8)
    if (staged && tl > 5) {
        int tw = 5;
        while ((int64_t)RED_CHUNKS_WIDE << tw < sp.chunks && tw < RED_MAX_TEAM_LOG2) ++tw;
        const int64_t tms = RED_THREADS >> tw;  // its smallest ring must fit, else keep tl
        if (((tms * 4 * 8 + 127) / 128 * 128) + tms * 2 * stage_bytes <= RED_SMEM_MAX) tl = tw;
    }
    // a staged row set too wide for a 2-slot ring per team at this team size
    // (many inputs a row): larger teams, fewer of them a block, until the ring
    // fits RED_SMEM_PREF or a team has one chunk a thread.  (Measured on the
    // GPT block's 4-stage RMSNorm backward, 7 inputs over 512-cell rows:
    // without this the rows streamed from global memory once per stage.)
    auto bar_for = [](int64_t tms) { return (tms * 4 * 8 + 127) / 128 * 128; };
    while (staged && tl < RED_MAX_TEAM_LOG2 && ((int64_t)1 << tl) < sp.chunks &&
           bar_for(RED_THREADS >> tl) + (int64_t)(RED_THREADS >> tl) * 2 * stage_bytes > RED_SMEM_PREF)
        ++tl;
    const int T = 1 << tl;
    const int64_t ch_per = (sp.chunks + T - 1) / T > 0 ? (sp.chunks + T - 1) / T : 1;
    if (ch_per > RED_STAGED_MAX_CHUNKS) staged = false;
    const int teams = RED_THREADS >> tl;
    int ns = 4;
    const int64_t bar_bytes = ((int64_t)teams * 4 * 8 + 127) / 128 * 128;
    while (ns > 2 && bar_bytes + teams * ns * stage_bytes > RED_SMEM_PREF) --ns;
    if (bar_bytes + teams * ns * stage_bytes > RED_SMEM_MAX) staged = false;
    // a row that one warp holds in registers (a team of at most 32 threads,
    // the row cached in RED_CACHE_WORDS words a thread) skips the ring: the
    // loads go out at once and nothing waits on a barrier (measured on the
    // softmax rows of 4096 x 1024 float32: 14.3 us against 16.4 us staged
    // for one launch, 10.2 against 12.5 back to back; the GPT block's step
    // unchanged)
    if (staged && tl <= 5 && ch_per * words <= RED_CACHE_WORDS) staged = false;
    if (!staged) {
        for (int k = 0; k < n_in; ++k) staged_in[k] = 0;
        stage_bytes = tx_bytes = 0;
        ns = 1;
    } else {
        for (int k = 0; k < n_in; ++k) cache_in[k] = 0;  // the ring holds the row
        words = 0;
    }
    P->smem = staged ? (int)(bar_bytes + teams * ns * stage_bytes) : 0;
    if (stash >= 0 && ch_per * (words + PSG_VEC) > RED_CACHE_WORDS) stash = -1;
    const int kch = columnar ? 0 : ch_per * words <= RED_CACHE_WORDS || staged ? (int)ch_per : 0;
    if (kch == 0) stash = -1;
    const int stash_node = stash >= 0 ? stages[stash].n_nodes - 1 : -1;
    // the stash may overwrite the cached row in place when nothing reads the
    // row after the stash stage: that stage is the last, the epilogue reads
    // no cached input past the stash (the values only the stash needed are
    // dropped), and the row is one 32-bit input (its words match the
    // stash's).  The row and the stash then share one set of registers.
    int stash_alias = -1;
    if (stash >= 0 && stash == n_stages - 1 && !staged) {
        int cached = -1, ncached = 0;
        for (int k = 0; k < n_in; ++k)
            if (cache_in[k]) { cached = k; ++ncached; }
        if (ncached == 1 && dtype_size(dts[cached]) == 4) {
            std::vector<char> need(n_epi, 0);
            need[n_epi - 1] = 1;
            bool reads = false;
            for (int i = n_epi - 1; i >= 0; --i) {
                if (!need[i]) continue;
                const psg_node& x = epi[i];
                if (i == stash_node) continue;  // read from the stash, its operands not needed
                if (x.op == PSG_OP_LOAD) {
                    if (x.a == cached && !E.uni[i]) reads = true;
                    continue;
                }
                if (x.op == PSG_OP_CONST || x.op == PSG_OP_RED) continue;
                const int nops = x.op == PSG_OP_WHERE ? 3 : (x.op == PSG_OP_NEG || x.op == PSG_OP_EXP ||
                                                             x.op == PSG_OP_LOG || x.op == PSG_OP_SQRT ||
                                                             x.op == PSG_OP_RECIP || x.op == PSG_OP_CAST) ? 1 : 2;
                const int ops[3] = {x.a, x.b, x.c};
                for (int o = 0; o < nops; ++o)
                    if (ops[o] >= 0 && ops[o] < i) need[ops[o]] = 1;
            }
            if (!reads) stash_alias = cached;
        }
    }
    // Rows held in registers by teams of at most 128 threads run in blocks of
    // 128 (RED_REG_THREADS): the register file then divides in finer steps.
    // Resident blocks the launch bound asks registers for: what the ring
    // leaves room for in staged mode; with the row in registers, as many as
    // leave each thread its cached words and stash plus about 40 working
    // registers; else 4; columnar, 512 threads an SM, so the unrolled stream
    // keeps its loads in registers.  Measured on one GB300 over the softmax
    // rows of 4096 x 1024 float32 (-Xptxas -v: no spill at 72 registers):
    // 256-thread blocks with 50 working registers (3 blocks, 76 registers)
    // took 8.8 us a launch back to back; 128-thread blocks with 40 (7 blocks,
    // 72 registers) 7.95 us; with 32 (8 blocks, 64 registers) 8.55 us; the
    // GPT block's replayed step 0.538, 0.534 and 0.541 ms.  One launch after
    // an L2 flush took 12.3-12.5 us in every case.
    const bool reg_rows = !staged && !columnar && kch > 0 && (1 << tl) <= RED_REG_THREADS;
    const int row_block = reg_rows ? RED_REG_THREADS : RED_THREADS;
    int min_blocks = 4;
    if (staged) {
        min_blocks = (int)((227 * 1024) / (P->smem + 1024));
        min_blocks = min_blocks < 1 ? 1 : min_blocks > 4 ? 4 : min_blocks;
    } else if (kch > 0) {
        const int est = kch * words + (stash >= 0 && stash_alias < 0 ? kch * PSG_VEC : 0) + 40;
        min_blocks = std::max(1, std::min(4 * RED_THREADS / row_block, 65536 / (row_block * est)));
    }
    // columnar: 32 rows a CTA and up to 16 members (warps), as many as keep
    // RED_COL_MIN_CHUNKS chunks each; a cluster of C CTAs (a power of two up
    // to 8) shares the rows when the row groups alone would leave most SMs
    // idle and every member still keeps RED_COL_MIN_CHUNKS chunks
    constexpr int RED_COL_MIN_CHUNKS = 2;
    int col_members = RED_COL_THREADS / 32;
    while (col_members > 1 && sp.chunks < (int64_t)col_members * RED_COL_MIN_CHUNKS) col_members >>= 1;
    // vectorised columnar layout (kColVec): one stage, one output per row,
    // two row dims at most collapsed to one, rows in whole groups of PSG_VEC,
    // and every input float-typed and either moving one cell a row (read as
    // aligned 16-byte vectors of PSG_VEC rows) or not moving with the row at
    // all (read once for the PSG_VEC rows).  Then a thread holds eight rows:
    // for the GPT block's RMSNorm weight gradients (512 sums of 8192 rows,
    // three inputs) one load moves 16 or 32 bytes instead of 2 or 4.
    constexpr int VEC_RT = 4;  // row threads a warp: 32 rows a CTA, 8 slots of the reduced axis a warp
    int vec_row[PSG_MAX_INPUTS] = {0};
    bool colvec = columnar && n_stages == 1 && per_row && sp.nd == 2 && sp.rows % PSG_VEC == 0;
    for (int k = 0; k < n_in && colvec; ++k) {
        const int es = dtype_size(dts[k]);
        if (dts[k] != PSG_F32 && dts[k] != PSG_BF16 && dts[k] != PSG_F16) colvec = false;
        const int64_t rs = P->p.in[k].outer_stride[0];
        if (rs == 1) {
            vec_row[k] = 1;
            if (uni[k] || ((uintptr_t)in[k] + (uint64_t)P->p.in[k].offset * es) % 16 != 0 ||
                (P->p.in[k].inner_stride * es) % 16 != 0)
                colvec = false;
        } else if (rs != 0) {
            colvec = false;
        }
    }
    if (colvec) {
        col_members = RED_COL_THREADS / 32;
        while (col_members > 1 && sp.inner < (int64_t)col_members * (32 / VEC_RT) * 2) col_members >>= 1;
    }
    const int block = columnar ? 32 * col_members : row_block;
    if (!columnar && (block >> tl) < 1) return PSG_E_INVALID_ARG;  // a block holds whole teams
    if (columnar) min_blocks = std::max(1, 512 / block);
    int cluster = 1;
    if (columnar) {
        const int64_t groups = (sp.rows + 31) / 32;
        auto deep_enough = [&](int c) {  // every member still keeps two cells (chunks) of the reduced axis
            return colvec ? sp.inner >= (int64_t)col_members * (32 / VEC_RT) * c * 2
                          : sp.chunks >= (int64_t)col_members * c * 2 * RED_COL_MIN_CHUNKS;
        };
        while (cluster < 8 && groups * cluster * 2 <= (int64_t)num_sms() && deep_enough(cluster))
            cluster *= 2;
    }
    P->cluster = cluster;
    bodies += gen_eval(epi, E, "Epi", "", stash_node, true);  // the result only goes to a store
    P->block = block;
    P->p.rows = sp.rows;
    P->p.inner = sp.inner;
    P->p.chunks = sp.chunks;
    for (int d = 0; d < MAXD; ++d) P->p.shape[d] = d < sp.nd ? sp.shape[d] : 1;
    P->p.nd = sp.nd;
    P->p.team_log2 = columnar ? -1 : tl;  // -1: columnar teams (32 a block)
    P->p.out_per_row = per_row ? 1 : 0;
    std::string spec = "constexpr int kNin = " + std::to_string(n_in) + ";\n";
    spec += "constexpr int kInMode[] = " + int_list(modes, n_in) + ";\n";
    spec += "constexpr int kInDt[] = " + int_list(dts, n_in) + ";\n";
    spec += "constexpr int kOutDt = " + std::to_string(out_v->dtype) + ";\n";
    spec += "constexpr int kOutMode = " + std::to_string(out_mode) + ";\n";
    spec += "constexpr int kNstages = " + std::to_string(n_stages) + ";\n";
    spec += "constexpr int kStageOp[] = " + int_list(sop, n_stages) + ";\n";
    spec += "constexpr int kStageDt[] = " + int_list(sdt, n_stages) + ";\n";
    spec += "constexpr int kCH = " + std::to_string(kch) + ";\n";
    spec += "constexpr int kCacheIn[] = " + int_list(cache_in, n_in) + ";\n";
    spec += "constexpr int kStash = " + std::to_string(stash) + ";\n";
    spec += "constexpr int kStashAlias = " + std::to_string(stash_alias) + ";\n";
    spec += "constexpr int kMinBlocks = " + std::to_string(min_blocks) + ";\n";
    const bool exact = kch > 0 && sp.inner % PSG_VEC == 0 && sp.chunks == (int64_t)kch * T;
    spec += "constexpr bool kExact = " + std::string(exact ? "true" : "false") + ";\n";
    spec += "constexpr int kStaged = " + std::to_string(staged ? 1 : 0) + ";\n";
    spec += "constexpr int kNS = " + std::to_string(ns) + ";\n";
    spec += "constexpr int kStageBytes = " + std::to_string(stage_bytes) + ";\n";
    spec += "constexpr int kBarBytes = " + std::to_string(staged ? bar_bytes : 0) + ";\n";
    spec += "constexpr u32 kTxBytes = " + std::to_string(tx_bytes) + "u;\n";
    spec += "constexpr int kStagedIn[] = " + int_list(staged_in, n_in) + ";\n";
    spec += "constexpr int kSegOff[] = " + int_list(seg_off, n_in) + ";\n";
    spec += "constexpr u32 kRowBytes[] = " + int_list(row_bytes, n_in) + ";\n";
    spec += "constexpr int kInSize[] = " + int_list(in_size, n_in) + ";\n";
    spec += "constexpr int kPerRow = " + std::to_string(per_row ? 1 : 0) + ";\n";
    spec += "constexpr int kColumnar = " + std::to_string(columnar ? 1 : 0) + ";\n";
    spec += "constexpr int kColVec = " + std::to_string(colvec ? 1 : 0) + ";\n";
    spec += "constexpr int kVecRT = " + std::to_string(VEC_RT) + ";\n";
    spec += "constexpr int kVecRow[] = " + int_list(vec_row, n_in) + ";\n";
    spec += "constexpr int kBlockThreads = " + std::to_string(block) + ";\n";
    spec += "constexpr int kCluster = " + std::to_string(cluster) + ";\n";
    spec += "constexpr int kStreamUnroll = " + std::to_string(columnar ? 4 : 1) + ";\n";
    spec += cluster > 1 ? "#define PSG_CLUSTER_DIMS __cluster_dims__(" + std::to_string(cluster) + ", 1, 1)\n"
                        : "#define PSG_CLUSTER_DIMS\n";
    spec += "template <int S> struct StageBody;\n";
    spec += bodies;
    P->spec = std::move(spec);
    return PSG_OK;
}

psg_status grid_for(const RedPlan& P, cudaKernel_t k, int* grid)
{
    const int teams = P.p.team_log2 < 0 ? 32 : P.block >> P.p.team_log2;
    const int64_t need = (P.p.rows + teams - 1) / teams;
    const int per_sm = jit_max_blocks_per_sm(k, P.block, (size_t)P.smem);
    // whole clusters: every CTA of a cluster walks the same row groups
    const int64_t cap = std::max<int64_t>(1, (int64_t)num_sms() * (per_sm > 0 ? per_sm : 1) / P.cluster);
    *grid = (int)(std::max<int64_t>(1, std::min<int64_t>(need, cap)) * P.cluster);
    return PSG_OK;
}

// A staged kernel's ring needs more than the default 48 KB of dynamic shared
// memory: opt in once per (kernel, device).
psg_status allow_smem(cudaKernel_t k, int bytes)
{
    if (bytes <= 48 * 1024) return PSG_OK;
    static std::mutex mu;
    static std::unordered_map<uint64_t, int> done;
    const uint64_t key = (uint64_t)(uintptr_t)k ^ ((uint64_t)current_device() << 56);
    std::lock_guard<std::mutex> g(mu);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return PSG_OK;
    if (cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return PSG_E_CUDA;
    done[key] = bytes;
    return PSG_OK;
}

}  // namespace

psg_status query_reduce(const psg_reduce_stage* stages, int n_stages, const psg_node* epi, int n_epi,
                        const psg_view* in_v, int n_in, const psg_view* out_v, int* grid, int* block,
                        int* smem, int* regs)
{
    const void* fake[PSG_MAX_INPUTS];
    for (int k = 0; k < PSG_MAX_INPUTS; ++k) fake[k] = (const void*)(uintptr_t)4096;
    RedPlan P;
    psg_status st = plan_reduce(stages, n_stages, epi, n_epi, fake, in_v, n_in, (void*)(uintptr_t)4096, out_v, &P);
    if (st != PSG_OK) return st;
    cudaKernel_t k;
    st = jit_kernel(JIT_REDUCE, P.spec, "psg_reduce", &k);
    if (st != PSG_OK) return st;
    st = allow_smem(k, P.smem);
    if (st != PSG_OK) return st;
    grid_for(P, k, grid);
    *block = P.block;
    *smem = P.smem;
    *regs = jit_regs(k);
    return PSG_OK;
}

}  // namespace psg

using namespace psg;

extern "C" psg_status psg_reduce_rows(const psg_reduce_stage* stages, int n_stages, const psg_node* epilogue,
                                      int n_epi, const void* const* in, const psg_view* in_v, int n_in,
                                      void* out, const psg_view* out_v, int32_t* d_status, void* stream)
{
    RedPlan P;
    psg_status st = plan_reduce(stages, n_stages, epilogue, n_epi, in, in_v, n_in, out, out_v, &P);
    if (st != PSG_OK) return st;
    if (P.p.rows == 0) return PSG_OK;
    P.p.status = d_status;
    P.p.wait_cycles = 2000000000ll;  // about a second at the SM clock
    P.p.skip_first_copy = 0;
    // Test hook, not part of the ABI: PSG_TEST_RING_TIMEOUT=1 (read at each
    // call) leaves the first ring slot of every staged team unfilled and
    // bounds each wait by about a millisecond, so that the wait gives up,
    // PSG_E_TIMEOUT reaches d_status and the kernel still ends after its
    // copies in flight have landed.
    if (const char* t = std::getenv("PSG_TEST_RING_TIMEOUT"); t && t[0] == '1') {
        P.p.wait_cycles = 2000000ll;
        P.p.skip_first_copy = 1;
    }
    cudaKernel_t k;
    st = jit_kernel(JIT_REDUCE, P.spec, "psg_reduce", &k);
    if (st != PSG_OK) return st;
    st = allow_smem(k, P.smem);
    if (st != PSG_OK) return st;
    int grid;
    grid_for(P, k, &grid);
    void* args[] = {(void*)&P.p};
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg =
        launch_config(dim3(grid), dim3(P.block), (size_t)P.smem, (cudaStream_t)stream, attr);
    if (cudaLaunchKernelExC(&cfg, (const void*)k, args) != cudaSuccess) return PSG_E_CUDA;
    return PSG_OK;
}

// Test hook, not part of the ABI: plan a psg_reduce_rows call over dummy
// pointers and compile its kernel without a GPU.
extern "C" int psg_internal_compile_reduce(const psg_reduce_stage* stages, int n_stages, const psg_node* epilogue,
                                           int n_epi, const psg_view* in_v, int n_in, const psg_view* out_v,
                                           char* log, size_t log_size)
{
    const void* fake[PSG_MAX_INPUTS];
    for (int k = 0; k < PSG_MAX_INPUTS; ++k) fake[k] = (const void*)(uintptr_t)4096;
    RedPlan P;
    psg_status st = plan_reduce(stages, n_stages, epilogue, n_epi, fake, in_v, n_in, (void*)(uintptr_t)4096,
                                out_v, &P);
    if (st != PSG_OK) return st;
    std::string l;
    st = jit_compile_only(jit_source(JIT_REDUCE, P.spec), &l);
    if (log && log_size) {
        std::strncpy(log, l.c_str(), log_size - 1);
        log[log_size - 1] = 0;
    }
    return st;
}
