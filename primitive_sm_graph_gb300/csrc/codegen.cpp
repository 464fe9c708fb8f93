// Program analysis and code generation for the runtime-specialised kernels.
//
// A psg_node program is validated against the op set's dtype rules (limn, "The
// op set"), CASTs that move no bits (widening bf16/f16 -> f32, i8/i16 -> wider
// ints) become aliases, dead nodes are dropped, and every remaining node
// becomes one typed C++ statement that rounds into the node's own dtype.
// Nodes whose operands are all uniform along the inner dim (constants,
// reduced row values, stride-0 inputs) are emitted once per chunk, outside
// the lane loop: a stride-0 loop reuses its operand instead of recomputing it
// (Luminal IR blog, "ZeroStrideLoop").
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "codegen.h"

namespace psg {

namespace {

uint32_t const_bits(double v, int dt)
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

std::string fmt(const char* f, ...) __attribute__((format(printf, 1, 2)));
std::string fmt(const char* f, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, f);
    vsnprintf(buf, sizeof(buf), f, ap);
    va_end(ap);
    return buf;
}

const char* ctype(int dt) { return dtype_is_int(dt) ? "int" : dt == PSG_F64 ? "double" : "float"; }

// round a 32-bit value expression into dtype dt
std::string wrap(int dt, const std::string& e)
{
    switch (dt) {
    case PSG_BF16: return "rbf(" + e + ")";
    case PSG_F16: return "rh(" + e + ")";
    case PSG_I16: return "w16(" + e + ")";
    case PSG_I8: return "w8(" + e + ")";
    }
    return e;
}

}  // namespace

psg_status analyze_program(const psg_node* nodes, int n, const int* in_dtype, const bool* in_uniform,
                           int n_in, const int* red_dtype, int n_red, ProgInfo* I)
{
    if (!nodes || n < 1 || n > PSG_MAX_NODES) return PSG_E_INVALID_ARG;
    I->n = n;
    I->dt.assign(n, 0);
    I->val.assign(n, 0);
    I->uni.assign(n, 0);
    I->live.assign(n, 0);
    for (int i = 0; i < n; ++i) {
        const psg_node& x = nodes[i];
        if (!dtype_valid(x.dtype)) return PSG_E_UNSUPPORTED_DTYPE;
        I->dt[i] = x.dtype;
        I->val[i] = i;
        auto opnd = [&](int k) { return k >= 0 && k < i; };
        switch (x.op) {
        case PSG_OP_LOAD:
            if (x.a < 0 || x.a >= n_in) return PSG_E_INVALID_ARG;
            if (in_dtype[x.a] != x.dtype) return PSG_E_UNSUPPORTED_DTYPE;
            I->uni[i] = in_uniform[x.a];
            break;
        case PSG_OP_CONST:
            I->uni[i] = 1;
            break;
        case PSG_OP_RED:
            if (x.a < 0 || x.a >= n_red) return PSG_E_INVALID_ARG;
            if (red_dtype[x.a] != x.dtype) return PSG_E_UNSUPPORTED_DTYPE;
            I->uni[i] = 1;
            break;
        case PSG_OP_NEG:
            if (!opnd(x.a) || I->dt[x.a] != x.dtype) return PSG_E_INVALID_ARG;
            I->uni[i] = I->uni[x.a];
            break;
        case PSG_OP_EXP: case PSG_OP_LOG: case PSG_OP_SQRT: case PSG_OP_RECIP:
            if (!opnd(x.a) || I->dt[x.a] != x.dtype) return PSG_E_INVALID_ARG;
            if (!dtype_is_float(x.dtype) && x.dtype != PSG_F64) return PSG_E_UNSUPPORTED_DTYPE;
            I->uni[i] = I->uni[x.a];
            break;
        case PSG_OP_CAST: {
            if (!opnd(x.a)) return PSG_E_INVALID_ARG;
            const int s = I->dt[x.a], d = x.dtype;
            I->uni[i] = I->uni[x.a];
            bool alias = s == d || (dtype_is_float(s) && d == PSG_F32) ||
                         (dtype_is_int(s) && dtype_is_int(d) && dtype_size(d) >= dtype_size(s));
            if (alias) I->val[i] = I->val[x.a];
            break;
        }
        case PSG_OP_ADD: case PSG_OP_MUL: case PSG_OP_CMPLT:
            if (!opnd(x.a) || !opnd(x.b)) return PSG_E_INVALID_ARG;
            if (I->dt[x.a] != x.dtype || I->dt[x.b] != x.dtype) return PSG_E_INVALID_ARG;
            I->uni[i] = I->uni[x.a] && I->uni[x.b];
            break;
        case PSG_OP_WHERE:
            if (!opnd(x.a) || !opnd(x.b) || !opnd(x.c)) return PSG_E_INVALID_ARG;
            if (I->dt[x.b] != x.dtype || I->dt[x.c] != x.dtype) return PSG_E_INVALID_ARG;
            I->uni[i] = I->uni[x.a] && I->uni[x.b] && I->uni[x.c];
            break;
        default:
            return PSG_E_INVALID_ARG;
        }
    }
    I->live[n - 1] = 1;
    for (int i = n - 1; i >= 0; --i) {
        if (!I->live[i]) continue;
        const psg_node& x = nodes[i];
        switch (x.op) {
        case PSG_OP_NEG: case PSG_OP_EXP: case PSG_OP_LOG: case PSG_OP_SQRT:
        case PSG_OP_RECIP: case PSG_OP_CAST: I->live[x.a] = 1; break;
        case PSG_OP_ADD: case PSG_OP_MUL: case PSG_OP_CMPLT: I->live[x.a] = I->live[x.b] = 1; break;
        case PSG_OP_WHERE: I->live[x.a] = I->live[x.b] = I->live[x.c] = 1; break;
        default: break;
        }
    }
    I->result = I->val[n - 1];
    I->result_dtype = I->dt[n - 1];
    I->result_uniform = I->uni[I->result] != 0;
    return PSG_OK;
}

std::string gen_eval(const psg_node* nodes, const ProgInfo& I, const std::string& name,
                     const std::string& prefix, int stash, bool store_rounds)
{
    const int n = I.n;
    // with a stashed node, liveness restarts from the result with that node
    // as a leaf: what only fed it is not computed again
    std::vector<int> live = I.live;
    if (stash >= 0) {
        live.assign(n, 0);
        live[n - 1] = 1;
        for (int i = n - 1; i >= 0; --i) {
            if (!live[i] || i == stash) continue;
            const psg_node& x = nodes[i];
            switch (x.op) {
            case PSG_OP_NEG: case PSG_OP_EXP: case PSG_OP_LOG: case PSG_OP_SQRT:
            case PSG_OP_RECIP: case PSG_OP_CAST: live[x.a] = 1; break;
            case PSG_OP_ADD: case PSG_OP_MUL: case PSG_OP_CMPLT: live[x.a] = live[x.b] = 1; break;
            case PSG_OP_WHERE: live[x.a] = live[x.b] = live[x.c] = 1; break;
            default: break;
            }
        }
    }
    auto ref = [&](int j) {
        const int v = I.val[j];
        return std::string(I.uni[v] ? "u" : "x") + std::to_string(v);
    };
    std::string head, uni_part, loop_part;
    std::vector<char> loaded(PSG_MAX_INPUTS, 0);
    for (int i = 0; i < n; ++i) {
        if (!live[i] || I.val[i] != i) continue;
        const psg_node& x = nodes[i];
        const int dt = x.dtype;
        const bool isint = dtype_is_int(dt);
        // the last node feeds only the store; a half-width store rounds to
        // nearest-even itself, which gives the same bits as rounding here
        const bool rounded_by_store = store_rounds && i == n - 1 && (dt == PSG_BF16 || dt == PSG_F16);
        auto wrap = [&](int d, const std::string& ex) { return rounded_by_store ? ex : psg::wrap(d, ex); };
        std::string e;
        if (i == stash) {
            loop_part += fmt("            const %s x%d = %s;\n", ctype(dt), i, isint ? "c.stashi(v)" : "c.stashf(v)");
            continue;
        }
        switch (x.op) {
        case PSG_OP_LOAD:
            if (I.uni[i]) {
                e = fmt("c.template ld1<%d>()", x.a);
            } else {
                if (!loaded[x.a]) {
                    head += fmt("        typename VT<%d>::T in%d[PSG_VEC];\n        c.template ldv<%d>(in%d);\n",
                                dt, x.a, x.a, x.a);
                    loaded[x.a] = 1;
                }
                e = fmt("in%d[v]", x.a);
            }
            break;
        case PSG_OP_CONST: {
            if (dt == PSG_F64) {
                uint64_t b64;
                std::memcpy(&b64, &x.cval, 8);
                e = fmt("__longlong_as_double(0x%016llxll)", (unsigned long long)b64);
                break;
            }
            const uint32_t b = const_bits(x.cval, dt);
            e = isint ? fmt("(int)%d", (int32_t)b) : fmt("__uint_as_float(0x%08xu)", b);
            break;
        }
        case PSG_OP_RED:
            e = fmt(isint ? "c.redi(%d)" : "c.redf(%d)", x.a);
            break;
        case PSG_OP_NEG:
            e = isint ? wrap(dt, "negi(" + ref(x.a) + ")") : (dt == PSG_F64 ? "negd(" : "negf(") + ref(x.a) + ")";
            break;
        // float64 nodes compute natively in double (limn, "The op set", the
        // dtype paragraph): the C library's exp and log, correctly rounded
        // sqrt, reciprocal, add and multiply
        case PSG_OP_EXP: e = dt == PSG_F64 ? "exp(" + ref(x.a) + ")" : wrap(dt, "psg_exp(" + ref(x.a) + ")"); break;
        case PSG_OP_LOG: e = dt == PSG_F64 ? "log(" + ref(x.a) + ")" : wrap(dt, "logf(" + ref(x.a) + ")"); break;
        case PSG_OP_SQRT:
            e = dt == PSG_F64 ? "__dsqrt_rn(" + ref(x.a) + ")" : wrap(dt, "__fsqrt_rn(" + ref(x.a) + ")");
            break;
        case PSG_OP_RECIP:
            e = dt == PSG_F64 ? "__drcp_rn(" + ref(x.a) + ")" : wrap(dt, "__frcp_rn(" + ref(x.a) + ")");
            break;
        case PSG_OP_CAST: {
            const int s = I.dt[x.a];
            // float64 to a narrower float rounds to float32 first, then (for a
            // half width) to the half width, as the oracle's CAST does
            if (s == PSG_F64 && dtype_is_int(dt)) e = wrap(dt, "__double2int_rz(" + ref(x.a) + ")");
            else if (s == PSG_F64 && dt != PSG_F64) e = wrap(dt, "__double2float_rn(" + ref(x.a) + ")");
            else if (dtype_is_int(s) && dt == PSG_F64) e = "__int2double_rn(" + ref(x.a) + ")";
            else if (dt == PSG_F64) e = "(double)" + ref(x.a);
            else if (dtype_is_float(s) && dtype_is_int(dt)) e = wrap(dt, "__float2int_rz(" + ref(x.a) + ")");
            else if (dtype_is_int(s) && dtype_is_float(dt)) e = wrap(dt, "__int2float_rn(" + ref(x.a) + ")");
            else e = wrap(dt, ref(x.a));
            break;
        }
        case PSG_OP_ADD:
            e = wrap(dt, (isint ? "addi(" : dt == PSG_F64 ? "__dadd_rn(" : "__fadd_rn(") + ref(x.a) + ", " + ref(x.b) + ")");
            break;
        case PSG_OP_MUL:
            e = wrap(dt, (isint ? "muli(" : dt == PSG_F64 ? "__dmul_rn(" : "__fmul_rn(") + ref(x.a) + ", " + ref(x.b) + ")");
            break;
        case PSG_OP_CMPLT:
            e = "(" + ref(x.a) + " < " + ref(x.b) + (isint ? " ? 1 : 0)" : dt == PSG_F64 ? " ? 1.0 : 0.0)" : " ? 1.0f : 0.0f)");
            break;
        case PSG_OP_WHERE: {
            const int cdt = I.dt[x.a];
            const bool cint = dtype_is_int(cdt);
            e = "((" + ref(x.a) + (cint ? " != 0" : cdt == PSG_F64 ? " != 0.0" : " != 0.0f") + ") ? " + ref(x.b) + " : " + ref(x.c) + ")";
            break;
        }
        }
        const std::string stmt = fmt("%s %s%d = ", ctype(dt), I.uni[i] ? "u" : "x", i) + e + ";\n";
        if (I.uni[i]) uni_part += "        const " + stmt;
        else loop_part += "            const " + stmt;
    }
    // uniform values are computed once per row by uni() and handed to eval()
    // for every chunk of that row
    std::vector<int> uvals;
    for (int i = 0; i < n; ++i)
        if (live[i] && I.val[i] == i && I.uni[i] && i != stash) uvals.push_back(i);
    const std::string rt = ctype(I.result_dtype);
    std::string s;
    s += prefix + "struct " + name + " {\n";
    s += "    struct U {\n";
    for (int i : uvals) s += fmt("        %s u%d;\n", ctype(I.dt[i]), i);
    if (uvals.empty()) s += "        int none;\n";
    s += "    };\n";
    s += "    template <class C>\n";
    s += "    __device__ __forceinline__ static U uni(const C& c)\n    {\n";
    s += uni_part;
    s += "        U r;\n";
    for (int i : uvals) s += fmt("        r.u%d = u%d;\n", i, i);
    if (uvals.empty()) s += "        r.none = 0;\n";
    s += "        return r;\n    }\n";
    s += "    template <class C>\n";
    s += "    __device__ __forceinline__ static void eval(const C& c, const U& u, " + rt + " (&y)[PSG_VEC])\n    {\n";
    for (int i : uvals) s += fmt("        const %s u%d = u.u%d;\n", ctype(I.dt[i]), i, i);
    if (I.result_uniform) {
        s += fmt("#pragma unroll\n        for (int v = 0; v < PSG_VEC; ++v) y[v] = u%d;\n", I.result);
    } else {
        s += head;
        s += "#pragma unroll\n        for (int v = 0; v < PSG_VEC; ++v) {\n";
        s += loop_part;
        s += fmt("            y[v] = x%d;\n        }\n", I.result);
    }
    s += "    }\n};\n";
    return s;
}

}  // namespace psg
