// psg_contract: matmul as SUM over the last dim of MUL(Av, Bv).  The roles of
// the dims come from the Views themselves: Av is broadcast along n (stride 0)
// and Bv along m, exactly the two stride-0 loops of the broadcast form.
#include <algorithm>
#include <cstring>

#include "api_internal.h"
#include "codegen.h"
#include "common.h"
#include "contract.h"
#include "jit.h"

namespace psg {

namespace {

struct Batch {
    int nb;                       // batch dims kept (after dropping size 1)
    int64_t shape[MAXD], sa[MAXD], sb[MAXD], sc[MAXD];
    bool masked;                  // a batch dim is masked: every dim kept, one launch per index
    int64_t lo[MAXD], hi[MAXD];   // the window both operands read along each batch dim
};

// [lo, hi): the indices of dim d a View reads (its mask clipped to the shape)
void window(const psg_view* v, int d, int64_t& lo, int64_t& hi)
{
    lo = std::max<int64_t>(v->mask_lo[d], 0);
    hi = std::min<int64_t>(v->mask_hi[d], v->shape[d]);
    if (hi < lo) hi = lo;
}

// true when some dim's window is empty: the View reads nothing at all
bool reads_nothing(const psg_view* v)
{
    for (int d = 0; d < v->ndim; ++d) {
        int64_t lo, hi;
        window(v, d, lo, hi);
        if (hi == lo) return true;
    }
    return false;
}

// Merge batch dims that are contiguous for A, B and C alike.
void collapse_batch(Batch& B)
{
    int n = 0;
    for (int d = 0; d < B.nb; ++d) {
        if (B.shape[d] == 1) continue;
        if (n > 0 && B.sa[n - 1] == B.sa[d] * B.shape[d] && B.sb[n - 1] == B.sb[d] * B.shape[d] &&
            B.sc[n - 1] == B.sc[d] * B.shape[d]) {
            B.shape[n - 1] *= B.shape[d];
            B.sa[n - 1] = B.sa[d];
            B.sb[n - 1] = B.sb[d];
            B.sc[n - 1] = B.sc[d];
        } else {
            B.shape[n] = B.shape[d];
            B.sa[n] = B.sa[d];
            B.sb[n] = B.sb[d];
            B.sc[n] = B.sc[d];
            ++n;
        }
    }
    B.nb = n;
}

bool al16(const void* p, int64_t off_elems, int es) { return ((uintptr_t)p + (uintptr_t)(off_elems * es)) % 16 == 0; }

// The fused epilogue of the tensor-core path: validates the program and its
// inputs against C, fills the kernel's operand descriptors and writes the
// spec pieces.  dm, dn: the dims of m and n in C's index space; nb_dims:
// C's leading (batch) dims, which must merge into one stride for every input
// as they did for A, B and C.
psg_status plan_epilogue(const psg_epilogue* E, const psg_view* Cv, int dm, int dn, int nb_dims, int64_t batch,
                         TcParams& p, EpiSpec& spec)
{
    const int n = E->n_nodes, nin = E->n_in;
    if (!E->prog || n < 1 || n > PSG_MAX_NODES || nin < 0 || nin > PSG_MAX_INPUTS || nin > PSG_TC_MAX_EPI_IN)
        return PSG_E_INVALID_ARG;
    if (nin > 0 && (!E->in || !E->in_v)) return PSG_E_INVALID_ARG;
    // ACC becomes the stashed value: the first ACC node reads it, any later
    // one is a no-op CAST of the first
    std::vector<psg_node> nodes(E->prog, E->prog + n);
    int acc = -1;
    for (int i = 0; i < n; ++i) {
        psg_node& x = nodes[i];
        if (x.op == PSG_OP_LOAD && (x.a < 0 || x.a >= nin)) return PSG_E_INVALID_ARG;
        if (x.op == PSG_OP_RED) return PSG_E_INVALID_ARG;
        if (x.dtype == PSG_F64) return PSG_E_UNSUPPORTED_DTYPE;
        if (x.op != PSG_OP_ACC) continue;
        if (x.dtype != PSG_F32) return PSG_E_UNSUPPORTED_DTYPE;
        if (acc < 0) {
            acc = i;
            x.op = PSG_OP_LOAD;
            x.a = nin;
        } else {
            x.op = PSG_OP_CAST;
            x.a = acc;
        }
    }
    int dts[PSG_MAX_INPUTS + 1];
    bool uni[PSG_MAX_INPUTS + 1];
    int modes[PSG_TC_MAX_EPI_IN] = {};
    const int64_t M = Cv->shape[dm], N = Cv->shape[dn];
    for (int k = 0; k < nin; ++k) {
        const psg_view* v = &E->in_v[k];
        if (v->ndim != Cv->ndim || !same_shape(v, Cv)) return PSG_E_INVALID_ARG;
        if (!dtype_valid(v->dtype) || v->dtype == PSG_F64) return PSG_E_UNSUPPORTED_DTYPE;
        if (view_has_mask(v)) return PSG_E_UNSUPPORTED_LAYOUT;
        psg_status st = check_view(v, false);
        if (st != PSG_OK) return st;
        if (M * N * batch > 0 && !E->in[k]) return PSG_E_INVALID_ARG;
        if (!ptr_aligned(E->in[k], v->dtype)) return PSG_E_MISALIGNED;
        // the batch dims that are not 1 merge into one stride, as for A, B and C
        int64_t sb = 0;
        int last = -1;
        for (int d = 0; d < nb_dims; ++d) {
            if (v->shape[d] == 1) continue;
            if (last >= 0 && v->strides[last] != v->strides[d] * v->shape[d]) return PSG_E_UNSUPPORTED_LAYOUT;
            last = d;
            sb = v->strides[d];
        }
        const int es = dtype_size(v->dtype);
        TcEpiOperand& o = p.epi[k];
        o.ptr = (const char*)E->in[k] + v->offset * es;
        o.sb = sb;
        o.sm = M > 1 ? v->strides[dm] : 0;
        o.sn = N > 1 ? v->strides[dn] : 0;
        const bool al = ((uintptr_t)o.ptr % 16) == 0 && (o.sm * es) % 16 == 0 && (batch <= 1 || (o.sb * es) % 16 == 0);
        modes[k] = o.sn == 0 ? 0 : (o.sn == 1 && al && dtype_is_float(v->dtype)) ? 1 : 2;  // EPI_ROW / VEC / STRIDED
        dts[k] = v->dtype;
        uni[k] = o.sn == 0;
    }
    dts[nin] = PSG_F32;
    uni[nin] = false;
    ProgInfo I;
    psg_status st = analyze_program(nodes.data(), n, dts, uni, nin + 1, nullptr, 0, &I);
    if (st != PSG_OK) return st;
    if (I.result_dtype != Cv->dtype) return PSG_E_UNSUPPORTED_DTYPE;
    p.n_epi = nin;
    std::string dl = "constexpr int kEpiDt[8] = {", ml = "constexpr int kEpiMode[8] = {";
    for (int k = 0; k < 8; ++k) {
        dl += std::to_string(k < nin ? dts[k] : 0) + (k < 7 ? ", " : "};\n");
        ml += std::to_string(k < nin ? modes[k] : 0) + (k < 7 ? ", " : "};\n");
    }
    spec.tables = dl + ml + "constexpr int kEpiN = " + std::to_string(nin) + ";\n";
    // a half-width C is rounded by the store itself (the same bits)
    spec.prog = gen_eval(nodes.data(), I, "EpiProg", "", acc, Cv->dtype != PSG_F32);
    return PSG_OK;
}

}  // namespace

psg_status plan_contract(const void* A, const psg_view* Av, const void* Bp, const psg_view* Bv, void* C,
                         const psg_view* Cv, const psg_epilogue* epi, EpiSpec* espec, int32_t* d_status,
                         bool* use_tc, TcOperands* T, SimtParams* S, Batch* bt)
{
    if (!Av || !Bv || !Cv) return PSG_E_INVALID_ARG;
    const int r = Av->ndim;
    if (r < 3 || r > 6 || Bv->ndim != r) return PSG_E_INVALID_ARG;
    psg_status st = check_view(Av, false);
    if (st != PSG_OK) return st;
    st = check_view(Bv, false);
    if (st != PSG_OK) return st;
    st = check_view(Cv, true);
    if (st != PSG_OK) return st;
    if (!same_shape(Av, Bv)) return PSG_E_INVALID_ARG;
    const bool masked = view_has_mask(Av) || view_has_mask(Bv);
    const int dm = r - 3, dn = r - 2, dk = r - 1;
    const int64_t M = Av->shape[dm], N = Av->shape[dn], K = Av->shape[dk];
    // the broadcast form: A constant along n, B constant along m
    if ((N > 1 && Av->strides[dn] != 0) || (M > 1 && Bv->strides[dm] != 0)) return PSG_E_UNSUPPORTED_LAYOUT;
    // C: [batch.., M, N] or [batch.., M, N, 1]
    const bool kept = Cv->ndim == r;
    if (!(Cv->ndim == r - 1 || (kept && Cv->shape[r - 1] == 1))) return PSG_E_INVALID_ARG;
    for (int d = 0; d < r - 1; ++d)
        if (Cv->shape[d] != Av->shape[d]) return PSG_E_INVALID_ARG;
    const int adt = Av->dtype, cdt = Cv->dtype;
    if (Bv->dtype != adt) return PSG_E_UNSUPPORTED_DTYPE;
    auto is_float = [](int t) { return t == PSG_BF16 || t == PSG_F16 || t == PSG_F32; };
    auto is_int = [](int t) { return t == PSG_I32 || t == PSG_I16 || t == PSG_I8; };
    // float32-accumulated floats store to any of them; float64 to float64;
    // the integers (uint32 wraparound total) to any integer width
    if (!((is_float(adt) && is_float(cdt)) || (adt == PSG_F64 && cdt == PSG_F64) || (is_int(adt) && is_int(cdt))))
        return PSG_E_UNSUPPORTED_DTYPE;
    const int64_t numel = M * N * K;
    if (numel > 0 && (!A || !Bp)) return PSG_E_INVALID_ARG;
    if (M * N > 0 && !C) return PSG_E_INVALID_ARG;
    if (!ptr_aligned(A, adt) || !ptr_aligned(Bp, adt) || !ptr_aligned(C, cdt)) return PSG_E_MISALIGNED;
    if (M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return PSG_E_UNSUPPORTED_LAYOUT;
    bt->nb = r - 3;
    bt->masked = false;
    for (int d = 0; d < bt->nb; ++d) {
        bt->shape[d] = Av->shape[d];
        bt->sa[d] = Av->strides[d];
        bt->sb[d] = Bv->strides[d];
        bt->sc[d] = Cv->strides[d];
        int64_t alo, ahi, blo, bhi;
        window(Av, d, alo, ahi);
        window(Bv, d, blo, bhi);
        bt->lo[d] = std::max(alo, blo);
        bt->hi[d] = std::max(bt->lo[d], std::min(ahi, bhi));
        if (bt->lo[d] > 0 || bt->hi[d] < bt->shape[d]) bt->masked = true;
    }
    if (!bt->masked) collapse_batch(*bt);
    const int64_t a_ms = Av->strides[dm], a_ks = Av->strides[dk];
    const int64_t b_ns = Bv->strides[dn], b_ks = Bv->strides[dk];
    const int64_t c_ms = Cv->strides[dm], c_ns = Cv->strides[dn];
    const int64_t batch = bt->nb == 1 ? bt->shape[0] : 1;
    // tensor-core paths, one (collapsed) batch dim, TMA-addressable operands:
    // bf16 (one MMA per term) and float32 with K >= TF32X3_MIN_K (three TF32
    // MMAs per term; shorter K keeps the exact-product FP32-pipe kernel,
    // whose only error is the reduction order)
    constexpr int64_t TF32X3_MIN_K = 256;
    bool tc = (adt == PSG_BF16 || adt == PSG_F16 || (adt == PSG_F32 && K >= TF32X3_MIN_K)) && bt->nb <= 1 && K > 0 &&
              !masked;
    const int es = dtype_size(adt), q16 = 16 / es;  // elements per 16 bytes
    auto tma_ok = [&](const void* base, int64_t off, int64_t s_mn, int64_t s_k, int64_t mn, int64_t s_b, bool& kmaj) {
        if (s_k == 1 && s_mn % q16 == 0 && s_mn >= K) kmaj = true;
        else if (s_mn == 1 && s_k % q16 == 0 && s_k >= mn) kmaj = false;
        else return false;
        if (batch > 1 && (s_b % q16 != 0 || s_b <= 0)) return false;
        return al16(base, off, es);
    };
    bool akm = true, bkm = true;
    tc = tc && tma_ok(A, Av->offset, a_ms, a_ks, M, bt->nb ? bt->sa[0] : 0, akm);
    tc = tc && tma_ok(Bp, Bv->offset, b_ns, b_ks, N, bt->nb ? bt->sb[0] : 0, bkm);
    *use_tc = tc;
    const bool has_epi = epi && epi->n_nodes > 0;
    if (has_epi) {
        // the epilogue runs in the bf16 / f16 tensor-core kernel only
        if (!tc || adt == PSG_F32 || bt->masked || bt->nb > 1) return PSG_E_UNSUPPORTED_LAYOUT;
        if (!is_float(cdt)) return PSG_E_UNSUPPORTED_DTYPE;
    }
    if (tc) {
        std::memset(T, 0, sizeof(*T));
        T->p.M = (int)M;
        T->p.N = (int)N;
        T->p.K = (int)K;
        T->p.batch = (int)batch;
        T->p.a_kmajor = akm ? 1 : 0;
        T->p.b_kmajor = bkm ? 1 : 0;
        T->p.c_dtype = cdt;
        T->p.ab_dtype = adt;
        T->p.C = C;
        T->p.status = d_status;
        T->p.c_offset = Cv->offset;
        T->p.c_rs = c_ms;
        T->p.c_cs = c_ns;
        T->p.c_bs = bt->nb ? bt->sc[0] : 0;
        T->A = (const char*)A + Av->offset * es;
        T->B = (const char*)Bp + Bv->offset * es;
        T->a_ms = a_ms;
        T->a_ks = a_ks;
        T->a_bs = bt->nb ? bt->sa[0] : 0;
        T->b_ns = b_ns;
        T->b_ks = b_ks;
        T->b_bs = bt->nb ? bt->sb[0] : 0;
        if (has_epi) {
            st = plan_epilogue(epi, Cv, dm, dn, r - 3, batch, T->p, *espec);
            if (st != PSG_OK) return st;
            T->epi = espec;
        }
    }
    std::memset(S, 0, sizeof(*S));
    S->A = A;
    S->B = Bp;
    S->C = C;
    S->ab_dtype = adt;
    S->c_dtype = cdt;
    S->M = M;
    S->N = N;
    S->K = K;
    S->batch = batch;
    S->a_off = Av->offset;
    S->a_ms = a_ms;
    S->a_ks = a_ks;
    S->a_bs = bt->nb == 1 ? bt->sa[0] : 0;
    S->b_off = Bv->offset;
    S->b_ns = b_ns;
    S->b_ks = b_ks;
    S->b_bs = bt->nb == 1 ? bt->sb[0] : 0;
    S->c_off = Cv->offset;
    S->c_ms = c_ms;
    S->c_ns = c_ns;
    S->c_bs = bt->nb == 1 ? bt->sc[0] : 0;
    // read windows and the window of cells that are not zero by a mask
    window(Av, dm, S->a_mlo, S->a_mhi);
    window(Av, dk, S->a_klo, S->a_khi);
    window(Bv, dn, S->b_nlo, S->b_nhi);
    window(Bv, dk, S->b_klo, S->b_khi);
    window(Bv, dm, S->c_mlo, S->c_mhi);
    window(Av, dn, S->c_nlo, S->c_nhi);
    // a View with an empty window along any dim reads nothing (and its
    // offset is unchecked): it loads no element at all
    if (reads_nothing(Av)) S->a_mlo = S->a_mhi = 0;
    if (reads_nothing(Bv)) S->b_nlo = S->b_nhi = 0;
    return PSG_OK;
}

}  // namespace psg

using namespace psg;

namespace {

psg_status contract_impl(const void* A, const psg_view* Av, const void* B, const psg_view* Bv, void* C,
                         const psg_view* Cv, const psg_epilogue* epi, void* ws, size_t ws_bytes, int32_t* d_status,
                         void* stream)
{
    bool tc;
    TcOperands T;
    SimtParams S;
    Batch bt;
    EpiSpec espec;
    psg_status st = plan_contract(A, Av, B, Bv, C, Cv, epi, &espec, d_status, &tc, &T, &S, &bt);
    if (st != PSG_OK) return st;
    // a fused epilogue needs the whole total of a cell in one place: no split K
    const bool has_epi = epi && epi->n_nodes > 0;
    T.ws = has_epi ? nullptr : ws;
    T.ws_bytes = has_epi ? 0 : ws_bytes;
    if (S.M == 0 || S.N == 0) return PSG_OK;
    // (an empty SUM, K == 0, is its identity: every cell 0 through the SIMT kernel)
    if (bt.nb <= 1 && !bt.masked) {
        if (!tc) return launch_contract_simt(S, stream);
        return S.ab_dtype == PSG_F32 ? launch_contract_tf32(T, stream) : launch_contract_tc(T, stream);
    }
    // several batch dims that do not merge, or a masked batch dim: one launch
    // per batch index (an index outside a batch window reads nothing, writes 0)
    int64_t count = 1;
    for (int d = 0; d < bt.nb; ++d) count *= bt.shape[d];
    for (int64_t i = 0; i < count; ++i) {
        int64_t rem = i, oa = 0, ob = 0, oc = 0;
        bool inside = true;
        for (int d = bt.nb - 1; d >= 0; --d) {
            const int64_t x = rem % bt.shape[d];
            rem /= bt.shape[d];
            oa += x * bt.sa[d];
            ob += x * bt.sb[d];
            oc += x * bt.sc[d];
            inside = inside && (!bt.masked || (x >= bt.lo[d] && x < bt.hi[d]));
        }
        SimtParams s1 = S;
        if (!inside) s1.a_mlo = s1.a_mhi = s1.b_nlo = s1.b_nhi = s1.c_mlo = s1.c_mhi = 0;
        s1.a_off += oa;
        s1.b_off += ob;
        s1.c_off += oc;
        s1.batch = 1;
        st = launch_contract_simt(s1, stream);
        if (st != PSG_OK) return st;
    }
    return PSG_OK;
}

}  // namespace

extern "C" psg_status psg_contract(const void* A, const psg_view* Av, const void* B, const psg_view* Bv, void* C,
                                   const psg_view* Cv, const psg_epilogue* epilogue, int32_t* d_status, void* stream)
{
    return contract_impl(A, Av, B, Bv, C, Cv, epilogue, nullptr, 0, d_status, stream);
}

extern "C" psg_status psg_contract_ws(const void* A, const psg_view* Av, const void* B, const psg_view* Bv, void* C,
                                      const psg_view* Cv, const psg_epilogue* epilogue, void* workspace,
                                      size_t ws_bytes, int32_t* d_status, void* stream)
{
    return contract_impl(A, Av, B, Bv, C, Cv, epilogue, workspace, ws_bytes, d_status, stream);
}

extern "C" size_t psg_contract_workspace(const psg_view* Av, const psg_view* Bv, const psg_view* Cv)
{
    // shapes and dtypes decide the split; pointers and strides only decide
    // whether the tensor-core kernel runs at all (if not, nothing is used)
    if (!Av || !Bv || !Cv || Av->ndim < 3 || Av->ndim > 6 || Bv->ndim != Av->ndim) return 0;
    if (Av->dtype != Bv->dtype || (Av->dtype != PSG_BF16 && Av->dtype != PSG_F16)) return 0;
    const int r = Av->ndim;
    int64_t batch = 1;
    for (int d = 0; d < r - 3; ++d) batch *= Av->shape[d];
    const int64_t M = Av->shape[r - 3], N = Av->shape[r - 2], K = Av->shape[r - 1];
    if (batch <= 0 || M <= 0 || N <= 0 || K <= 0 || M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return 0;
    size_t bytes = 0;
    contract_tc_splits(M, N, K, batch, &bytes);
    return bytes;
}

// Test hook, not part of the ABI: plan a psg_contract call with an epilogue
// over dummy pointers and compile both variants of its kernel (single CTA
// and CTA pair) without a GPU.
extern "C" int psg_internal_compile_contract_epilogue(const psg_view* Av, const psg_view* Bv, const psg_view* Cv,
                                                      const psg_epilogue* epi, char* log, size_t log_size)
{
    const void* fake[PSG_MAX_INPUTS];
    for (int k = 0; k < PSG_MAX_INPUTS; ++k) fake[k] = (const void*)(uintptr_t)4096;
    psg_epilogue e = *epi;
    e.in = fake;
    bool tc;
    TcOperands T;
    SimtParams S;
    Batch bt;
    EpiSpec espec;
    const void* p = (const void*)(uintptr_t)4096;
    psg_status st = plan_contract(p, Av, p, Bv, (void*)p, Cv, &e, &espec, nullptr, &tc, &T, &S, &bt);
    if (st != PSG_OK) return st;
    std::string l;
    for (int pair = 0; pair < 2 && st == PSG_OK; ++pair)
        st = jit_compile_only(jit_source(JIT_GEMM, epi_spec_source(espec, pair != 0)), &l);
    if (log && log_size) {
        std::strncpy(log, l.c_str(), log_size - 1);
        log[log_size - 1] = 0;
    }
    return st;
}
