// Device side of the register-form interpreter (see common.h for the design).
// Every case below is straight-line code over compile-time register indices.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.h"

namespace psg {

// ---- lane functions (bit-level in and out) --------------------------------
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

struct FAdd { __device__ uint32_t operator()(uint32_t a, uint32_t b) const { return f2u(__fadd_rn(u2f(a), u2f(b))); } };
struct FMul { __device__ uint32_t operator()(uint32_t a, uint32_t b) const { return f2u(__fmul_rn(u2f(a), u2f(b))); } };
struct FLt  { __device__ uint32_t operator()(uint32_t a, uint32_t b) const { return u2f(a) < u2f(b) ? 0x3f800000u : 0u; } };
struct IAdd { __device__ uint32_t operator()(uint32_t a, uint32_t b) const { return a + b; } };
struct IMul { __device__ uint32_t operator()(uint32_t a, uint32_t b) const { return a * b; } };
struct ILt  { __device__ uint32_t operator()(uint32_t a, uint32_t b) const { return (int32_t)a < (int32_t)b ? 1u : 0u; } };
struct Mov  { __device__ uint32_t operator()(uint32_t, uint32_t b) const { return b; } };

struct FNeg { __device__ uint32_t operator()(uint32_t a) const { return a ^ 0x80000000u; } };
struct INeg { __device__ uint32_t operator()(uint32_t a) const { return 0u - a; } };
struct FExp { __device__ uint32_t operator()(uint32_t a) const { return f2u(expf(u2f(a))); } };
struct FLog { __device__ uint32_t operator()(uint32_t a) const { return f2u(logf(u2f(a))); } };
struct FSqrt { __device__ uint32_t operator()(uint32_t a) const { return f2u(__fsqrt_rn(u2f(a))); } };
struct FRcp { __device__ uint32_t operator()(uint32_t a) const { return f2u(__frcp_rn(u2f(a))); } };
struct RBf16 { __device__ uint32_t operator()(uint32_t a) const { return f2u(__bfloat162float(__float2bfloat16_rn(u2f(a)))); } };
struct RF16 { __device__ uint32_t operator()(uint32_t a) const { return f2u(__half2float(__float2half_rn(u2f(a)))); } };
// float -> int32: truncate, NaN -> 0, saturate (cvt.rzi.s32.f32 semantics)
struct F2I { __device__ uint32_t operator()(uint32_t a) const { return (uint32_t)__float2int_rz(u2f(a)); } };
struct I2F { __device__ uint32_t operator()(uint32_t a) const { return f2u(__int2float_rn((int32_t)a)); } };
struct W8  { __device__ uint32_t operator()(uint32_t a) const { return (uint32_t)(int32_t)(int8_t)(uint8_t)(a & 0xffu); } };
struct W16 { __device__ uint32_t operator()(uint32_t a) const { return (uint32_t)(int32_t)(int16_t)(uint16_t)(a & 0xffffu); } };

typedef uint32_t RegFile[R][VEC];

template <int D, int S, class F>
__device__ __forceinline__ void op2(RegFile& r, bool sc, F f)
{
    if (sc) {
        r[D][0] = f(r[D][0], r[S][0]);
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) r[D][v] = f(r[D][v], r[S][v]);
    }
}

template <int D, class F>
__device__ __forceinline__ void op1(RegFile& r, bool sc, F f)
{
    if (sc) {
        r[D][0] = f(r[D][0]);
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) r[D][v] = f(r[D][v]);
    }
}

template <int D, int S>
__device__ __forceinline__ void sel(RegFile& r, bool sc, uint32_t p)
{
    if (sc) {
        r[D][0] = (p & 1u) ? r[D][0] : r[S][0];
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) r[D][v] = ((p >> v) & 1u) ? r[D][v] : r[S][v];
    }
}

template <int D>
__device__ __forceinline__ uint32_t pred(const RegFile& r, bool sc, bool is_int)
{
    if (sc) {
        bool t = is_int ? (r[D][0] != 0u) : (u2f(r[D][0]) != 0.0f);
        return t ? 0xffu : 0u;  // a uniform condition selects every lane alike
    }
    uint32_t p = 0;
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        bool t = is_int ? (r[D][v] != 0u) : (u2f(r[D][v]) != 0.0f);  // NaN != 0 is true
        p |= (t ? 1u : 0u) << v;
    }
    return p;
}

template <int D>
__device__ __forceinline__ void bcast(RegFile& r)
{
#pragma unroll
    for (int v = 1; v < VEC; ++v) r[D][v] = r[D][0];
}

template <int D>
__device__ __forceinline__ void setc(RegFile& r, bool sc, uint32_t imm)
{
    r[D][0] = imm;
    if (!sc) {
#pragma unroll
        for (int v = 1; v < VEC; ++v) r[D][v] = imm;
    }
}

// Src must provide: template <int K> uint32_t in(int lane) const  (0 for
//                   K beyond the inputs it holds), and uint32_t red(int s) const.
template <int D, int K, class Src>
__device__ __forceinline__ void ld(RegFile& r, bool sc, const Src& src)
{
    if (sc) {
        r[D][0] = src.template in<K>(0);
    } else {
#pragma unroll
        for (int v = 0; v < VEC; ++v) r[D][v] = src.template in<K>(v);
    }
}

template <int D, class Src>
__device__ __forceinline__ void ldred(RegFile& r, bool sc, const Src& src, int s)
{
    uint32_t x = src.red(s);
    r[D][0] = x;
    if (!sc) {
#pragma unroll
        for (int v = 1; v < VEC; ++v) r[D][v] = x;
    }
}

#define PSG_C2(OPC, D, S, CALL) case form_id(OPC, D, S): CALL; break;
#define PSG_C2_S(OPC, D, F)                                                            \
    PSG_C2(OPC, D, 0, (op2<D, 0>(r, sc, F{}))) PSG_C2(OPC, D, 1, (op2<D, 1>(r, sc, F{}))) \
    PSG_C2(OPC, D, 2, (op2<D, 2>(r, sc, F{}))) PSG_C2(OPC, D, 3, (op2<D, 3>(r, sc, F{}))) \
    PSG_C2(OPC, D, 4, (op2<D, 4>(r, sc, F{}))) PSG_C2(OPC, D, 5, (op2<D, 5>(r, sc, F{})))
#define PSG_CASES2(OPC, F)                                                             \
    PSG_C2_S(OPC, 0, F) PSG_C2_S(OPC, 1, F) PSG_C2_S(OPC, 2, F) PSG_C2_S(OPC, 3, F)    \
    PSG_C2_S(OPC, 4, F) PSG_C2_S(OPC, 5, F)

#define PSG_SEL_S(D)                                                                   \
    PSG_C2(OP_SEL, D, 0, (sel<D, 0>(r, sc, p))) PSG_C2(OP_SEL, D, 1, (sel<D, 1>(r, sc, p))) \
    PSG_C2(OP_SEL, D, 2, (sel<D, 2>(r, sc, p))) PSG_C2(OP_SEL, D, 3, (sel<D, 3>(r, sc, p))) \
    PSG_C2(OP_SEL, D, 4, (sel<D, 4>(r, sc, p))) PSG_C2(OP_SEL, D, 5, (sel<D, 5>(r, sc, p)))

#define PSG_C1(OPC, D, CALL) case form_id(OPC, D, 0): CALL; break;
#define PSG_CASES1(OPC, F)                                                             \
    PSG_C1(OPC, 0, (op1<0>(r, sc, F{}))) PSG_C1(OPC, 1, (op1<1>(r, sc, F{})))           \
    PSG_C1(OPC, 2, (op1<2>(r, sc, F{}))) PSG_C1(OPC, 3, (op1<3>(r, sc, F{})))           \
    PSG_C1(OPC, 4, (op1<4>(r, sc, F{}))) PSG_C1(OPC, 5, (op1<5>(r, sc, F{})))
#define PSG_CASES1X(OPC, T)                                                            \
    PSG_C1(OPC, 0, T(0)) PSG_C1(OPC, 1, T(1)) PSG_C1(OPC, 2, T(2)) PSG_C1(OPC, 3, T(3))   \
    PSG_C1(OPC, 4, T(4)) PSG_C1(OPC, 5, T(5))

#define PSG_LD_K(D, K) PSG_C2(OP_LD, D, K, (ld<D, K>(r, sc, src)))
#define PSG_LD_D(D)                                                                    \
    PSG_LD_K(D, 0) PSG_LD_K(D, 1) PSG_LD_K(D, 2) PSG_LD_K(D, 3) PSG_LD_K(D, 4)         \
    PSG_LD_K(D, 5) PSG_LD_K(D, 6) PSG_LD_K(D, 7)

#define PSG_T_PREDF(D) (p = pred<D>(r, sc, false))
#define PSG_T_PREDI(D) (p = pred<D>(r, sc, true))
#define PSG_T_CONST(D) (setc<D>(r, sc, in.imm))
#define PSG_T_BCAST(D) (bcast<D>(r))
#define PSG_T_LDRED(D) (ldred<D>(r, sc, src, 0))

// Run a compiled program.
template <class Src>
__device__ __forceinline__ void run_program(const Ins* __restrict__ prog, int n, RegFile& r,
                                            const Src& src)
{
    uint32_t p = 0;
    for (int i = 0; i < n; ++i) {
        const Ins in = prog[i];
        const bool sc = in.scalar != 0;
        switch (in.form) {
            PSG_CASES2(OP_MOV, Mov)
            PSG_CASES2(OP_ADDF, FAdd)
            PSG_CASES2(OP_MULF, FMul)
            PSG_CASES2(OP_LTF, FLt)
            PSG_CASES2(OP_ADDI, IAdd)
            PSG_CASES2(OP_MULI, IMul)
            PSG_CASES2(OP_LTI, ILt)
            PSG_SEL_S(0) PSG_SEL_S(1) PSG_SEL_S(2) PSG_SEL_S(3) PSG_SEL_S(4) PSG_SEL_S(5)
            PSG_CASES1(OP_NEGF, FNeg)
            PSG_CASES1(OP_NEGI, INeg)
            PSG_CASES1(OP_EXP, FExp)
            PSG_CASES1(OP_LOG, FLog)
            PSG_CASES1(OP_SQRT, FSqrt)
            PSG_CASES1(OP_RCP, FRcp)
            PSG_CASES1(OP_RBF16, RBf16)
            PSG_CASES1(OP_RF16, RF16)
            PSG_CASES1(OP_F2I, F2I)
            PSG_CASES1(OP_I2F, I2F)
            PSG_CASES1(OP_W8, W8)
            PSG_CASES1(OP_W16, W16)
            PSG_CASES1X(OP_PREDF, PSG_T_PREDF)
            PSG_CASES1X(OP_PREDI, PSG_T_PREDI)
            PSG_CASES1X(OP_CONST, PSG_T_CONST)
            PSG_CASES1X(OP_BCAST, PSG_T_BCAST)
            PSG_LD_D(0) PSG_LD_D(1) PSG_LD_D(2) PSG_LD_D(3) PSG_LD_D(4) PSG_LD_D(5)
            // LDRED: the stage index lives in the low bits (s field)
#define PSG_LDRED_DS(D, S) case form_id(OP_LDRED, D, S): ldred<D>(r, sc, src, S); break;
#define PSG_LDRED_D(D) PSG_LDRED_DS(D, 0) PSG_LDRED_DS(D, 1) PSG_LDRED_DS(D, 2) PSG_LDRED_DS(D, 3)
            PSG_LDRED_D(0) PSG_LDRED_D(1) PSG_LDRED_D(2) PSG_LDRED_D(3) PSG_LDRED_D(4) PSG_LDRED_D(5)
#undef PSG_LDRED_D
#undef PSG_LDRED_DS
            default: break;
        }
    }
}

// Read the result register's lane v (compile-time register choice via switch).
__device__ __forceinline__ uint32_t result_lane(const RegFile& r, int reg, int v)
{
    switch (reg) {
    case 0: return r[0][v];
    case 1: return r[1][v];
    case 2: return r[2][v];
    case 3: return r[3][v];
    case 4: return r[4][v];
    default: return r[5][v];
    }
}

// Copy the result register into out[VEC] (lane indices compile-time).
__device__ __forceinline__ void result_vec(const RegFile& r, int reg, uint32_t (&out)[VEC])
{
#define PSG_RV(K) case K: _Pragma("unroll") for (int v = 0; v < VEC; ++v) out[v] = r[K][v]; break;
    switch (reg) {
        PSG_RV(0) PSG_RV(1) PSG_RV(2) PSG_RV(3) PSG_RV(4) default: PSG_RV(5)
    }
#undef PSG_RV
}

// ---- storage conversion (value registers hold f32 or sign-extended int32) --
__device__ __forceinline__ uint32_t load_cell(const void* p, int64_t off, int dt)
{
    switch (dt) {
    case PSG_F32:
    case PSG_I32: return __ldg((const uint32_t*)p + off);
    case PSG_BF16: return ((uint32_t)__ldg((const unsigned short*)p + off)) << 16;
    case PSG_F16: return f2u(__half2float(__ushort_as_half(__ldg((const unsigned short*)p + off))));
    case PSG_I16: return (uint32_t)(int32_t)(int16_t)__ldg((const unsigned short*)p + off);
    case PSG_I8: return (uint32_t)(int32_t)__ldg((const signed char*)p + off);
    }
    return 0;
}

__device__ __forceinline__ void store_cell(void* p, int64_t off, int dt, uint32_t v)
{
    switch (dt) {
    case PSG_F32:
    case PSG_I32: ((uint32_t*)p)[off] = v; break;
    case PSG_BF16: ((unsigned short*)p)[off] = (unsigned short)(v >> 16); break;  // value is bf16-exact
    case PSG_F16: ((unsigned short*)p)[off] = __half_as_ushort(__float2half_rn(u2f(v))); break;
    case PSG_I16: ((unsigned short*)p)[off] = (unsigned short)(v & 0xffffu); break;
    case PSG_I8: ((unsigned char*)p)[off] = (unsigned char)(v & 0xffu); break;
    }
}

}  // namespace psg
