// Host compiler from a postfix psg_node program to register-form instructions.
//
// The node semantics are those of limn's op set ("The op set"): each node
// rounds to its own dtype, float16/bfloat16 compute in float32, narrow ints
// wrap.  Registers hold float32 values (for the three float dtypes) or
// sign-extended int32 values (for the three int dtypes), so a CAST that only
// widens (bf16->f32, i8->i32, ...) moves nothing and is compiled away.
//
// Allocation is a linear scan over the nodes in order: a value lives in one
// register from its definition to its last use; a two-register instruction
// overwrites its first operand, so an operand still needed later is copied
// first.  Uniform values (constant along the inner dim) are computed on lane 0
// only and broadcast where they meet a varying value.
#include <cmath>
#include <cstring>
#include <vector>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.h"

namespace psg {

namespace {

uint32_t round_const_bits(double v, int dt)
{
    if (dtype_is_int(dt)) {
        int64_t i = std::isnan(v) ? 0 : (int64_t)v;
        uint32_t u = (uint32_t)(uint64_t)i;
        if (dt == PSG_I16) u = (uint32_t)(int32_t)(int16_t)(uint16_t)(u & 0xffffu);
        if (dt == PSG_I8) u = (uint32_t)(int32_t)(int8_t)(uint8_t)(u & 0xffu);
        return u;
    }
    float f = (float)v;
    if (dt == PSG_BF16) f = __bfloat162float(__float2bfloat16_rn(f));
    if (dt == PSG_F16) f = __half2float(__float2half_rn(f));
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
}

struct Emitter {
    Program* P;
    int n = 0;
    bool overflow = false;
    void emit(int op, int d, int s, bool scalar, uint32_t imm = 0)
    {
        if (n >= MAX_INS) { overflow = true; return; }
        Ins& in = P->ins[n++];
        in.form = (uint16_t)form_id(op, d, s);
        in.scalar = scalar ? 1 : 0;
        in.pad = 0;
        in.imm = imm;
    }
};

// narrowing step after a value is computed in 32 bits
int round_op_for(int dt)
{
    switch (dt) {
    case PSG_BF16: return OP_RBF16;
    case PSG_F16: return OP_RF16;
    case PSG_I16: return OP_W16;
    case PSG_I8: return OP_W8;
    }
    return OP_NOP;
}

}  // namespace

psg_status compile_program(const psg_node* nodes, int n, const int* in_dtype,
                           const bool* in_uniform, int n_in, const int* red_dtype, int n_red,
                           bool bcast_result, Program* out, int* result_dtype,
                           bool* result_uniform)
{
    if (!nodes || n < 1 || n > PSG_MAX_NODES) return PSG_E_INVALID_ARG;
    std::vector<int> dt(n), val(n), uni(n);
    // ---- validate, and find aliases (CASTs that change no register bits) --
    for (int i = 0; i < n; ++i) {
        const psg_node& x = nodes[i];
        if (!dtype_valid(x.dtype)) return PSG_E_UNSUPPORTED_DTYPE;
        if (x.dtype == PSG_F64) return PSG_E_UNSUPPORTED_DTYPE;
        dt[i] = x.dtype;
        val[i] = i;
        auto opnd = [&](int k) { return k >= 0 && k < i; };
        switch (x.op) {
        case PSG_OP_LOAD:
            if (x.a < 0 || x.a >= n_in) return PSG_E_INVALID_ARG;
            if (in_dtype[x.a] != x.dtype) return PSG_E_UNSUPPORTED_DTYPE;
            uni[i] = in_uniform[x.a];
            break;
        case PSG_OP_CONST:
            uni[i] = 1;
            break;
        case PSG_OP_RED:
            if (x.a < 0 || x.a >= n_red) return PSG_E_INVALID_ARG;
            if (red_dtype[x.a] != x.dtype) return PSG_E_UNSUPPORTED_DTYPE;
            uni[i] = 1;
            break;
        case PSG_OP_NEG:
            if (!opnd(x.a) || dt[x.a] != x.dtype) return PSG_E_INVALID_ARG;
            uni[i] = uni[x.a];
            break;
        case PSG_OP_EXP: case PSG_OP_LOG: case PSG_OP_SQRT: case PSG_OP_RECIP:
            if (!opnd(x.a) || dt[x.a] != x.dtype) return PSG_E_INVALID_ARG;
            if (!dtype_is_float(x.dtype)) return PSG_E_UNSUPPORTED_DTYPE;
            uni[i] = uni[x.a];
            break;
        case PSG_OP_CAST: {
            if (!opnd(x.a)) return PSG_E_INVALID_ARG;
            int s = dt[x.a], d = x.dtype;
            uni[i] = uni[x.a];
            bool alias = false;
            if (s == d) alias = true;
            else if (dtype_is_float(s) && d == PSG_F32) alias = true;   // bf16/f16 -> f32 exact
            else if (dtype_is_int(s) && dtype_is_int(d) && dtype_size(d) >= dtype_size(s)) alias = true;
            if (alias) val[i] = val[x.a];
            break;
        }
        case PSG_OP_ADD: case PSG_OP_MUL: case PSG_OP_CMPLT:
            if (!opnd(x.a) || !opnd(x.b)) return PSG_E_INVALID_ARG;
            if (dt[x.a] != x.dtype || dt[x.b] != x.dtype) return PSG_E_INVALID_ARG;
            uni[i] = uni[x.a] && uni[x.b];
            break;
        case PSG_OP_WHERE:
            if (!opnd(x.a) || !opnd(x.b) || !opnd(x.c)) return PSG_E_INVALID_ARG;
            if (dt[x.b] != x.dtype || dt[x.c] != x.dtype) return PSG_E_INVALID_ARG;
            uni[i] = uni[x.a] && uni[x.b] && uni[x.c];
            break;
        default:
            return PSG_E_INVALID_ARG;
        }
    }
    // ---- liveness over underlying values, only nodes the result needs -----
    std::vector<char> live(n, 0);
    live[n - 1] = 1;
    for (int i = n - 1; i >= 0; --i) {
        if (!live[i]) continue;
        const psg_node& x = nodes[i];
        switch (x.op) {
        case PSG_OP_NEG: case PSG_OP_EXP: case PSG_OP_LOG: case PSG_OP_SQRT:
        case PSG_OP_RECIP: case PSG_OP_CAST: live[x.a] = 1; break;
        case PSG_OP_ADD: case PSG_OP_MUL: case PSG_OP_CMPLT: live[x.a] = live[x.b] = 1; break;
        case PSG_OP_WHERE: live[x.a] = live[x.b] = live[x.c] = 1; break;
        default: break;
        }
    }
    std::vector<int> last(n, -1);
    auto use = [&](int node, int at) { int v = val[node]; if (at > last[v]) last[v] = at; };
    for (int i = 0; i < n; ++i) {
        if (!live[i] || val[i] != i) continue;
        const psg_node& x = nodes[i];
        switch (x.op) {
        case PSG_OP_NEG: case PSG_OP_EXP: case PSG_OP_LOG: case PSG_OP_SQRT:
        case PSG_OP_RECIP: case PSG_OP_CAST: use(x.a, i); break;
        case PSG_OP_ADD: case PSG_OP_MUL: case PSG_OP_CMPLT: use(x.a, i); use(x.b, i); break;
        case PSG_OP_WHERE: use(x.a, i); use(x.b, i); use(x.c, i); break;
        default: break;
        }
    }
    const int result = val[n - 1];
    last[result] = n;  // the result lives to the end

    // ---- allocate and emit -------------------------------------------------
    std::memset(out, 0, sizeof(Program));
    Emitter E{out};
    int reg_of[PSG_MAX_NODES];
    int holder[R];       // value held by each register, -1 = free
    bool bc[R];          // register's lanes all equal lane 0 (uniform value broadcast)
    for (int k = 0; k < R; ++k) { holder[k] = -1; bc[k] = false; }
    auto alloc = [&](int v) -> int {
        for (int k = 0; k < R; ++k)
            if (holder[k] < 0) { holder[k] = v; bc[k] = false; return k; }
        return -1;
    };
    auto release_if_dead = [&](int v, int at) {
        if (last[v] == at) {
            int k = reg_of[v];
            if (k >= 0 && holder[k] == v) holder[k] = -1;
        }
    };
    // make a register (holding a uniform value) safe to read on every lane
    auto need_bcast = [&](int k) { if (!bc[k]) { E.emit(OP_BCAST, k, 0, false); bc[k] = true; } };
    // register for node i's result, overwriting operand value v when v dies here
    auto target_from = [&](int v, int i) -> int {
        int k = reg_of[v];
        if (last[v] == i) { holder[k] = i; return k; }
        int t = alloc(i);
        if (t < 0) return -1;
        E.emit(OP_MOV, t, k, uni[v] != 0);
        bc[t] = false;
        return t;
    };
    for (int i = 0; i < PSG_MAX_NODES; ++i) reg_of[i] = -1;

    for (int i = 0; i < n; ++i) {
        if (!live[i] || val[i] != i) continue;
        const psg_node& x = nodes[i];
        const bool sc = uni[i] != 0;
        int d = -1;
        switch (x.op) {
        case PSG_OP_LOAD:
            d = alloc(i);
            if (d < 0) return PSG_E_UNSUPPORTED_PROGRAM;
            E.emit(OP_LD, d, x.a, sc);
            break;
        case PSG_OP_CONST:
            d = alloc(i);
            if (d < 0) return PSG_E_UNSUPPORTED_PROGRAM;
            E.emit(OP_CONST, d, 0, true, round_const_bits(x.cval, x.dtype));
            break;
        case PSG_OP_RED:
            d = alloc(i);
            if (d < 0) return PSG_E_UNSUPPORTED_PROGRAM;
            E.emit(OP_LDRED, d, x.a, true);
            break;
        case PSG_OP_NEG: case PSG_OP_EXP: case PSG_OP_LOG: case PSG_OP_SQRT:
        case PSG_OP_RECIP: {
            int a = val[x.a];
            d = target_from(a, i);
            if (d < 0) return PSG_E_UNSUPPORTED_PROGRAM;
            int op = x.op == PSG_OP_NEG ? (dtype_is_int(x.dtype) ? OP_NEGI : OP_NEGF)
                   : x.op == PSG_OP_EXP ? OP_EXP : x.op == PSG_OP_LOG ? OP_LOG
                   : x.op == PSG_OP_SQRT ? OP_SQRT : OP_RCP;
            E.emit(op, d, 0, sc);
            if (round_op_for(x.dtype) != OP_NOP) E.emit(round_op_for(x.dtype), d, 0, sc);
            break;
        }
        case PSG_OP_CAST: {
            int a = val[x.a];
            int s = dt[x.a], t = x.dtype;
            d = target_from(a, i);
            if (d < 0) return PSG_E_UNSUPPORTED_PROGRAM;
            if (dtype_is_float(s) && dtype_is_int(t)) {
                E.emit(OP_F2I, d, 0, sc);
                if (round_op_for(t) != OP_NOP) E.emit(round_op_for(t), d, 0, sc);
            } else if (dtype_is_int(s) && dtype_is_float(t)) {
                E.emit(OP_I2F, d, 0, sc);
                if (round_op_for(t) != OP_NOP) E.emit(round_op_for(t), d, 0, sc);
            } else {  // narrowing within a class
                E.emit(round_op_for(t), d, 0, sc);
            }
            break;
        }
        case PSG_OP_ADD: case PSG_OP_MUL: case PSG_OP_CMPLT: {
            int a = val[x.a], b = val[x.b];
            bool comm = x.op != PSG_OP_CMPLT;
            // overwrite a dying operand; for commutative ops prefer a dying
            // varying operand so no broadcast of the target is needed
            if (comm && a != b && last[b] == i && (last[a] != i || (uni[a] && !uni[b])))
                std::swap(a, b);
            d = target_from(a, i);
            if (d < 0) return PSG_E_UNSUPPORTED_PROGRAM;
            int sreg = (a == b) ? d : reg_of[b];
            if (!sc) {
                if (uni[a]) need_bcast(d);
                if (uni[b] && sreg != d) need_bcast(sreg);
            }
            bool isint = dtype_is_int(x.dtype);
            int op = x.op == PSG_OP_ADD ? (isint ? OP_ADDI : OP_ADDF)
                   : x.op == PSG_OP_MUL ? (isint ? OP_MULI : OP_MULF) : (isint ? OP_LTI : OP_LTF);
            E.emit(op, d, sreg, sc);
            if (x.op != PSG_OP_CMPLT && round_op_for(x.dtype) != OP_NOP)
                E.emit(round_op_for(x.dtype), d, 0, sc);
            if (b != a) release_if_dead(b, i);
            break;
        }
        case PSG_OP_WHERE: {
            int c = val[x.a], xv = val[x.b], yv = val[x.c];
            int creg = reg_of[c];
            E.emit(dtype_is_int(dt[x.a]) ? OP_PREDI : OP_PREDF, creg, 0, uni[c] != 0);
            d = target_from(xv, i);
            if (d < 0) return PSG_E_UNSUPPORTED_PROGRAM;
            int yreg = (yv == xv) ? d : reg_of[yv];
            if (!sc) {
                if (uni[xv]) need_bcast(d);
                if (uni[yv] && yreg != d) need_bcast(yreg);
            }
            E.emit(OP_SEL, d, yreg, sc);
            if (c != xv) release_if_dead(c, i);
            if (yv != xv && yv != c) release_if_dead(yv, i);
            break;
        }
        }
        reg_of[i] = d;
        holder[d] = i;
        bc[d] = false;
        if (E.overflow) return PSG_E_UNSUPPORTED_PROGRAM;
    }
    int rr = reg_of[result];
    if (bcast_result && uni[result]) need_bcast(rr);
    if (E.overflow) return PSG_E_UNSUPPORTED_PROGRAM;
    out->n = E.n;
    out->out_reg = rr;
    *result_dtype = dt[n - 1];
    *result_uniform = uni[result] != 0;
    return PSG_OK;
}

}  // namespace psg
