// Device helpers of the runtime-specialised kernels (compiled by NVRTC for
// sm_103a, no system headers).  Values are computed as float (for float32,
// bfloat16 and float16 nodes) or int (for the three int widths); every node
// rounds into its own dtype, as a node of the op graph does (limn, "The op
// set": half widths are storage, narrow ints wrap).
typedef unsigned int u32;
typedef unsigned short u16;
typedef long long i64;

// Programmatic dependent launch: wait until the kernel before this one on the
// stream has finished and its writes are visible, then let the next kernel be
// scheduled.  First statement of every kernel; the host launches with
// programmatic stream serialization, so a launch overlaps its predecessor's
// tail and the data dependency is unchanged.
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- per-node rounding -------------------------------------------------
__device__ __forceinline__ float rbf(float x)  // float32 -> bfloat16 (RNE) -> float32
{
    u16 h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(x));
    return __uint_as_float(((u32)h) << 16);
}
__device__ __forceinline__ float rh(float x)   // float32 -> float16 (RNE) -> float32
{
    u16 h;
    float r;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(x));
    asm("cvt.f32.f16 %0, %1;" : "=f"(r) : "h"(h));
    return r;
}
__device__ __forceinline__ float h2f(u16 h)
{
    float r;
    asm("cvt.f32.f16 %0, %1;" : "=f"(r) : "h"(h));
    return r;
}
__device__ __forceinline__ u16 f2h(float x)  // float32 -> float16 bits (round to nearest even)
{
    u16 h;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(x));
    return h;
}
// NEG of a float flips the sign bit and nothing else (-0 for +0, NaN stays
// NaN); done on the bits so no floating-point rewrite can drop a zero's sign
__device__ __forceinline__ float negf(float x)
{
    u32 r;
    asm("xor.b32 %0, %1, 0x80000000;" : "=r"(r) : "r"(__float_as_uint(x)));
    return __uint_as_float(r);
}
// NEG of a float64: the sign bit flipped
__device__ __forceinline__ double negd(double x)
{
    return __longlong_as_double(__double_as_longlong(x) ^ (long long)0x8000000000000000ull);
}
__device__ __forceinline__ int w8(int x) { return (int)(signed char)(x & 0xff); }
__device__ __forceinline__ int w16(int x) { return (int)(short)(x & 0xffff); }
// EXP: exp(x) = 2^(x log2 e).  The product x * log2 e is carried as an
// unevaluated sum t + tl: t = RN(x * L2E_HI), the exact rounding error of
// that product from one FMA (Dekker's TwoProduct), plus x times the float32
// remainder of log2 e, so tl holds everything t lost (|tl| <= 2^-16 for any
// result that is not 0 or inf).  2^t comes from the hardware base-2
// approximation and 2^tl = 1 + tl ln 2 to first order (the next term is
// below 2^-33), applied with one FMA.  Results below the normal range are
// formed 2^64 higher and scaled down once at the end, so they round once
// into the subnormals; t outside (-160, 128) (0, inf, NaN) takes 2^t as is.
// The base-2 step flushes subnormals, which changes no result: its input
// is subnormal only when |t| < 2^-126 (2^t rounds to 1 either way), and its
// output only when t < -190, where exp underflows to 0 regardless.  (The
// flushing form is the shorter instruction sequence: the C2 chain's EXP
// cells run 8% faster.)  No branch.  The error is the base-2 approximation's plus one rounding;
// the tests hold it to 8 float32 ulps of the C library's expf.
__device__ __forceinline__ float psg_exp(float x)
{
    const float L2E_HI = __uint_as_float(0x3fb8aa3bu);  // log2(e) rounded to float32
    const float L2E_LO = __uint_as_float(0x32a57060u);  // log2(e) - L2E_HI, rounded
    const float LN2 = __uint_as_float(0x3f317218u);     // ln 2 rounded to float32
    const float t = __fmul_rn(x, L2E_HI);
    const float tl = __fmaf_rn(x, L2E_LO, __fmaf_rn(x, L2E_HI, -t));
    const bool sub = t < -125.0f;
    const float ts = sub ? __fadd_rn(t, 64.0f) : t;     // exact: t is a multiple of 2^-17 there
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(ts));
    const float rc = __fmaf_rn(r, __fmul_rn(tl, LN2), r);
    const float v = t > -160.0f && t < 128.0f ? rc : r;
    return sub ? __fmul_rn(v, __uint_as_float(0x1f800000u) /* 2^-64 */) : v;
}

__device__ __forceinline__ int addi(int a, int b) { return (int)((u32)a + (u32)b); }
__device__ __forceinline__ int muli(int a, int b) { return (int)((u32)a * (u32)b); }
__device__ __forceinline__ int negi(int a) { return (int)(0u - (u32)a); }

// ---- value type of a dtype ----------------------------------------------
template <int DT> struct VT { typedef float T; };
template <> struct VT<PSG_DT_F64> { typedef double T; };
template <> struct VT<PSG_DT_I32> { typedef int T; };
template <> struct VT<PSG_DT_I16> { typedef int T; };
template <> struct VT<PSG_DT_I8> { typedef int T; };

// one cell, widened
template <int DT>
__device__ __forceinline__ typename VT<DT>::T ld_cell(const void* p, i64 o)
{
    if constexpr (DT == PSG_DT_F32) return __ldg((const float*)p + o);
    else if constexpr (DT == PSG_DT_F64) return __ldg((const double*)p + o);
    else if constexpr (DT == PSG_DT_BF16) return __uint_as_float(((u32)__ldg((const u16*)p + o)) << 16);
    else if constexpr (DT == PSG_DT_F16) return h2f(__ldg((const u16*)p + o));
    else if constexpr (DT == PSG_DT_I32) return __ldg((const int*)p + o);
    else if constexpr (DT == PSG_DT_I16) return (int)__ldg((const short*)p + o);
    else return (int)__ldg((const signed char*)p + o);
}

template <int DT>
__device__ __forceinline__ void st_cell(void* p, i64 o, typename VT<DT>::T v)
{
    if constexpr (DT == PSG_DT_F32) ((float*)p)[o] = v;
    else if constexpr (DT == PSG_DT_F64) ((double*)p)[o] = v;
    else if constexpr (DT == PSG_DT_BF16) {
        u16 h;
        asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
        ((u16*)p)[o] = h;
    }
    else if constexpr (DT == PSG_DT_F16) ((u16*)p)[o] = f2h(v);
    else if constexpr (DT == PSG_DT_I32) ((int*)p)[o] = v;
    else if constexpr (DT == PSG_DT_I16) ((short*)p)[o] = (short)v;
    else ((signed char*)p)[o] = (signed char)v;
}

// PSG_VEC cells of a row starting at column col0: vector loads when the run
// is full and 16-byte aligned (8-byte for int8), else cell by cell.
template <int DT, int MODE>
__device__ __forceinline__ void ld_chunk(const PsgOperand& op, i64 roff, bool rok, i64 col0,
                                         int nvalid, typename VT<DT>::T (&d)[PSG_VEC])
{
    typedef typename VT<DT>::T T;
    if constexpr (MODE == PSG_M_UNIFORM) {
        const T x = ld_cell<DT>(op.ptr, roff);
#pragma unroll
        for (int v = 0; v < PSG_VEC; ++v) d[v] = x;
    } else if constexpr (MODE == PSG_M_CONTIG || MODE == PSG_M_VEC) {
        const i64 b = roff + col0;
        if constexpr (DT == PSG_DT_F32 || DT == PSG_DT_I32) {
            const T* q = (const T*)op.ptr + b;
            if (nvalid == PSG_VEC && (MODE == PSG_M_VEC || (((unsigned long long)q) & 15) == 0)) {
                const uint4 x = __ldg((const uint4*)q), y = __ldg((const uint4*)q + 1);
                const u32 w[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
                for (int v = 0; v < PSG_VEC; ++v) {
                    if constexpr (DT == PSG_DT_F32) d[v] = __uint_as_float(w[v]);
                    else d[v] = (int)w[v];
                }
                return;
            }
        } else if constexpr (DT == PSG_DT_F64) {
            const double* q = (const double*)op.ptr + b;
            if (nvalid == PSG_VEC && (MODE == PSG_M_VEC || (((unsigned long long)q) & 15) == 0)) {
#pragma unroll
                for (int u = 0; u < PSG_VEC / 2; ++u) {
                    const double2 x = __ldg((const double2*)q + u);
                    d[2 * u] = x.x;
                    d[2 * u + 1] = x.y;
                }
                return;
            }
        } else if constexpr (DT == PSG_DT_I8) {
            const signed char* q = (const signed char*)op.ptr + b;
            if (nvalid == PSG_VEC && (MODE == PSG_M_VEC || (((unsigned long long)q) & 7) == 0)) {
                const uint2 x = __ldg((const uint2*)q);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    d[v] = (int)(signed char)((x.x >> (8 * v)) & 0xffu);
                    d[4 + v] = (int)(signed char)((x.y >> (8 * v)) & 0xffu);
                }
                return;
            }
        } else {
            const u16* q = (const u16*)op.ptr + b;
            if (nvalid == PSG_VEC && (MODE == PSG_M_VEC || (((unsigned long long)q) & 15) == 0)) {
                const uint4 x = __ldg((const uint4*)q);
                const u32 w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const u16 lo = (u16)(w[v] & 0xffffu), hi = (u16)(w[v] >> 16);
                    if constexpr (DT == PSG_DT_BF16) {
                        d[2 * v] = __uint_as_float(((u32)lo) << 16);
                        d[2 * v + 1] = __uint_as_float(((u32)hi) << 16);
                    } else if constexpr (DT == PSG_DT_F16) {
                        d[2 * v] = h2f(lo);
                        d[2 * v + 1] = h2f(hi);
                    } else {
                        d[2 * v] = (int)(short)lo;
                        d[2 * v + 1] = (int)(short)hi;
                    }
                }
                return;
            }
        }
#pragma unroll
        for (int v = 0; v < PSG_VEC; ++v) d[v] = v < nvalid ? ld_cell<DT>(op.ptr, b + v) : (T)0;
    } else if constexpr (MODE == PSG_M_STRIDED) {
#pragma unroll
        for (int v = 0; v < PSG_VEC; ++v)
            d[v] = v < nvalid ? ld_cell<DT>(op.ptr, roff + (col0 + v) * op.inner_stride) : (T)0;
    } else {
        const i64 lo = op.mlo[PSG_MAXD - 1], hi = op.mhi[PSG_MAXD - 1];
#pragma unroll
        for (int v = 0; v < PSG_VEC; ++v) {
            const i64 c = col0 + v;
            const bool ok = rok && v < nvalid && c >= lo && c < hi;
            d[v] = ok ? ld_cell<DT>(op.ptr, roff + c * op.inner_stride) : (T)0;
        }
    }
}

// lane 0 only (the cell at col0), for operands uniform along the inner dim
template <int DT, int MODE>
__device__ __forceinline__ typename VT<DT>::T ld_first(const PsgOperand& op, i64 roff, bool rok, i64 col0)
{
    if constexpr (MODE == PSG_M_UNIFORM) return ld_cell<DT>(op.ptr, roff);
    else if constexpr (MODE == PSG_M_MASKED) {
        const bool ok = rok && col0 >= op.mlo[PSG_MAXD - 1] && col0 < op.mhi[PSG_MAXD - 1];
        return ok ? ld_cell<DT>(op.ptr, roff + col0 * op.inner_stride) : (typename VT<DT>::T)0;
    } else return ld_cell<DT>(op.ptr, roff + col0 * op.inner_stride);
}

// store PSG_VEC cells; vector stores for contiguous, full, aligned runs
// (MODE == PSG_M_VEC: known aligned, nothing is tested)
template <int DT, int MODE>
__device__ __forceinline__ void st_chunk(const PsgOperand& op, i64 roff, i64 col0, int nvalid,
                                         const typename VT<DT>::T (&y)[PSG_VEC])
{
    if ((MODE == PSG_M_VEC || op.inner_stride == 1) && nvalid == PSG_VEC) {
        const i64 b = roff + col0;
        if constexpr (DT == PSG_DT_F32 || DT == PSG_DT_I32) {
            u32* q = (u32*)op.ptr + b;
            if (MODE == PSG_M_VEC || (((unsigned long long)q) & 15) == 0) {
                u32 w[8];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    if constexpr (DT == PSG_DT_F32) w[v] = __float_as_uint(y[v]);
                    else w[v] = (u32)y[v];
                }
                ((uint4*)q)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                ((uint4*)q)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                return;
            }
        } else if constexpr (DT == PSG_DT_F64) {
            double* q = (double*)op.ptr + b;
            if (MODE == PSG_M_VEC || (((unsigned long long)q) & 15) == 0) {
#pragma unroll
                for (int u = 0; u < PSG_VEC / 2; ++u) ((double2*)q)[u] = make_double2(y[2 * u], y[2 * u + 1]);
                return;
            }
        } else if constexpr (DT == PSG_DT_BF16 || DT == PSG_DT_F16 || DT == PSG_DT_I16) {
            u16* q = (u16*)op.ptr + b;
            if (MODE == PSG_M_VEC || (((unsigned long long)q) & 15) == 0) {
                u32 w[4];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    // half widths: one round-to-nearest-even conversion per pair
                    if constexpr (DT == PSG_DT_BF16)
                        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[v]) : "f"(y[2 * v + 1]), "f"(y[2 * v]));
                    else if constexpr (DT == PSG_DT_F16)
                        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w[v]) : "f"(y[2 * v + 1]), "f"(y[2 * v]));
                    else w[v] = ((u32)y[2 * v] & 0xffffu) | ((u32)y[2 * v + 1] << 16);
                }
                *(uint4*)q = make_uint4(w[0], w[1], w[2], w[3]);
                return;
            }
        }
#pragma unroll
        for (int v = 0; v < PSG_VEC; ++v) st_cell<DT>((void*)op.ptr, b + v, y[v]);
        return;
    }
#pragma unroll
    for (int v = 0; v < PSG_VEC; ++v)
        if (v < nvalid) st_cell<DT>((void*)op.ptr, roff + (col0 + v) * op.inner_stride, y[v]);
}

// Offsets of a row: decompose the row index over the outer dims.
template <int NIN>
__device__ __forceinline__ void row_offsets(const PsgOperand* in, const PsgOperand& out, const i64* shape,
                                            int nd, i64 row, i64 (&roff)[NIN > 0 ? NIN : 1],
                                            bool (&rok)[NIN > 0 ? NIN : 1], const int* modes, i64& ooff)
{
#pragma unroll
    for (int k = 0; k < NIN; ++k) {
        roff[k] = in[k].offset;
        rok[k] = true;
    }
    ooff = out.offset;
    i64 rem = row;
    for (int d = nd - 2; d >= 0; --d) {
        i64 i;
        if (d > 0) {
            const i64 q = rem / shape[d];
            i = rem - q * shape[d];
            rem = q;
        } else {
            i = rem;
        }
        ooff += i * out.outer_stride[d];
#pragma unroll
        for (int k = 0; k < NIN; ++k) {
            roff[k] += i * in[k].outer_stride[d];
            if (modes[k] == PSG_M_MASKED) rok[k] = rok[k] && i >= in[k].mlo[d] && i < in[k].mhi[d];
        }
    }
}
