/*
 * Plain CPU oracle for the primitive-op graph hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test suite, the smoke check and the bench's
 * cpu_baseline / reference arm do.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Design (limn, "Three rules hold it together": the numpy device interprets
 * the graph one call per node, no fusion, and is the reference every backend
 * is diffed against):
 *   - one plain loop nest per primitive node, sequential ascending index order;
 *   - every node rounds its result to its own dtype;
 *   - float16 / bfloat16 are storage widths: values are widened to float32 to
 *     compute, and a reduce keeps a float32 running total and rounds once at
 *     the end (limn, section "The op set", the dtype paragraph);
 *   - float64 computes natively in double;
 *   - narrow ints wrap modulo 2^width (same paragraph).
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math (no FMA contraction, so a
 * MUL node followed by an ADD node rounds twice, as two nodes do).
 *
 * Threading: the optional OpenMP team splits OUTPUT cells only; every cell is
 * computed start to finish by one thread in the serial order, so the result
 * is bit-identical to the serial run (limn, "Backends", the c-device
 * paragraph on OpenMP).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dtype codes of this oracle (its own numbering) */
enum { O_F32 = 0, O_BF16 = 1, O_F16 = 2, O_F64 = 3, O_I32 = 4, O_I16 = 5, O_I8 = 6 };
/* unary opcodes */
enum { U_NEG = 0, U_EXP = 1, U_LOG = 2, U_SQRT = 3, U_RECIP = 4 };
/* binary opcodes */
enum { B_ADD = 0, B_MUL = 1, B_CMPLT = 2 };
/* reduce opcodes */
enum { R_SUM = 0, R_MAX = 1 };

static int o_size(int dt)
{
    switch (dt) {
    case O_F32: case O_I32: return 4;
    case O_BF16: case O_F16: case O_I16: return 2;
    case O_F64: return 8;
    case O_I8: return 1;
    }
    return 0;
}
static int o_is_int(int dt) { return dt == O_I32 || dt == O_I16 || dt == O_I8; }

/* ---- scalar conversions ------------------------------------------------ */

/* float32 -> bfloat16, round to nearest even; NaN stays a (quiet) NaN. */
static uint16_t f32_to_bf16_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}
static float bf16_bits_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* load an element of a float-family dtype (not f64) widened to float32 */
static float ld_f(int dt, const void* p, int64_t i)
{
    switch (dt) {
    case O_F32: return ((const float*)p)[i];
    case O_BF16: return bf16_bits_to_f32(((const uint16_t*)p)[i]);
    case O_F16: return (float)((const _Float16*)p)[i];
    }
    return NAN;
}
/* store a float32 value into a float-family dtype (not f64), rounding RNE */
static void st_f(int dt, void* p, int64_t i, float v)
{
    switch (dt) {
    case O_F32: ((float*)p)[i] = v; break;
    case O_BF16: ((uint16_t*)p)[i] = f32_to_bf16_bits(v); break;
    case O_F16: ((_Float16*)p)[i] = (_Float16)v; break;
    }
}
/* load an integer element, sign-extended */
static int32_t ld_i(int dt, const void* p, int64_t i)
{
    switch (dt) {
    case O_I32: return ((const int32_t*)p)[i];
    case O_I16: return ((const int16_t*)p)[i];
    case O_I8: return ((const int8_t*)p)[i];
    }
    return 0;
}
/* store an integer, wrapping modulo 2^width (two's complement) */
static void st_i(int dt, void* p, int64_t i, uint32_t v)
{
    switch (dt) {
    case O_I32: ((int32_t*)p)[i] = (int32_t)v; break;
    case O_I16: ((int16_t*)p)[i] = (int16_t)(uint16_t)(v & 0xffffu); break;
    case O_I8: ((int8_t*)p)[i] = (int8_t)(uint8_t)(v & 0xffu); break;
    }
}
/* float -> int32 conversion reading: truncate toward zero, NaN -> 0,
 * saturate to the int32 range; narrower targets then wrap. */
static uint32_t f_to_i32(double v)
{
    if (v != v) return 0u;
    if (v >= 2147483647.0) return (uint32_t)INT32_MAX;
    if (v <= -2147483648.0) return (uint32_t)INT32_MIN;
    return (uint32_t)(int32_t)v;
}

/* ---- VIEW: materialise (shape, strides, offset, mask) ------------------- */

/* Element with multi-index i reads base[offset + sum_d i_d*strides_d] when
 * mask_lo_d <= i_d < mask_hi_d for every d, else a zero of the dtype
 * (limn, "Three rules": a View is (shape, strides, offset, mask); "Reading
 * the schedule": a padded read is a range check that folds to a literal zero).
 * Returns 0, or -1 if a read falls outside [0, base_len). */
int orc_view_read(int dt, const void* base, int64_t base_len, int ndim, const int64_t* shape,
                  const int64_t* strides, int64_t offset, const int64_t* mlo, const int64_t* mhi,
                  void* out)
{
    int es = o_size(dt);
    int64_t n = 1;
    for (int d = 0; d < ndim; ++d) n *= shape[d];
    int64_t idx[16];
    for (int d = 0; d < ndim; ++d) idx[d] = 0;
    const char* b = (const char*)base;
    char* o = (char*)out;
    for (int64_t e = 0; e < n; ++e) {
        int inside = 1;
        int64_t off = offset;
        for (int d = 0; d < ndim; ++d) {
            if (idx[d] < mlo[d] || idx[d] >= mhi[d]) inside = 0;
            off += idx[d] * strides[d];
        }
        if (inside) {
            if (off < 0 || off >= base_len) return -1;
            memcpy(o + e * es, b + off * es, (size_t)es);
        } else {
            memset(o + e * es, 0, (size_t)es);
        }
        for (int d = ndim - 1; d >= 0; --d) { /* odometer, last dim fastest */
            if (++idx[d] < shape[d]) break;
            idx[d] = 0;
        }
    }
    return 0;
}

/* ---- elementwise nodes ------------------------------------------------- */

/* NEG EXP LOG SQRT RECIP on one dtype.  Returns -2 for an op the dtype lacks. */
int orc_unary(int op, int dt, const void* x, void* y, int64_t n, int nthreads)
{
    if (o_is_int(dt) && op != U_NEG) return -2;
    if (dt == O_F64) {
        const double* xd = (const double*)x;
        double* yd = (double*)y;
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
        for (int64_t i = 0; i < n; ++i) {
            double v = xd[i], r = 0;
            switch (op) {
            case U_NEG: r = -v; break;
            case U_EXP: r = exp(v); break;
            case U_LOG: r = log(v); break;
            case U_SQRT: r = sqrt(v); break;
            case U_RECIP: r = 1.0 / v; break;
            }
            yd[i] = r;
        }
        return 0;
    }
    if (o_is_int(dt)) {
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
        for (int64_t i = 0; i < n; ++i) st_i(dt, y, i, 0u - (uint32_t)ld_i(dt, x, i));
        return 0;
    }
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float v = ld_f(dt, x, i), r = 0;
        switch (op) {
        case U_NEG: r = -v; break;
        case U_EXP: r = expf(v); break;
        case U_LOG: r = logf(v); break;
        case U_SQRT: r = sqrtf(v); break;
        case U_RECIP: r = 1.0f / v; break;
        }
        st_f(dt, y, i, r);
    }
    return 0;
}

/* CAST between any two of the seven dtypes. */
int orc_cast(int dts, const void* x, int dtd, void* y, int64_t n, int nthreads)
{
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        if (o_is_int(dts)) {
            int32_t v = ld_i(dts, x, i);
            if (o_is_int(dtd)) st_i(dtd, y, i, (uint32_t)v);
            else if (dtd == O_F64) ((double*)y)[i] = (double)v;
            else st_f(dtd, y, i, (float)v); /* int -> f32 (RN), then the target width */
        } else if (dts == O_F64) {
            double v = ((const double*)x)[i];
            if (o_is_int(dtd)) st_i(dtd, y, i, f_to_i32(v));
            else if (dtd == O_F64) ((double*)y)[i] = v;
            else st_f(dtd, y, i, (float)v);
        } else {
            float v = ld_f(dts, x, i);
            if (o_is_int(dtd)) st_i(dtd, y, i, f_to_i32((double)v));
            else if (dtd == O_F64) ((double*)y)[i] = (double)v;
            else st_f(dtd, y, i, v);
        }
    }
    return 0;
}

/* ADD MUL CMPLT with both operands and the result in one dtype.
 * CMPLT yields 1 or 0 of that dtype; a NaN operand compares false. */
int orc_binary(int op, int dt, const void* a, const void* b, void* y, int64_t n, int nthreads)
{
    if (dt == O_F64) {
        const double* ad = (const double*)a;
        const double* bd = (const double*)b;
        double* yd = (double*)y;
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
        for (int64_t i = 0; i < n; ++i) {
            double u = ad[i], v = bd[i];
            yd[i] = op == B_ADD ? u + v : op == B_MUL ? u * v : (u < v ? 1.0 : 0.0);
        }
        return 0;
    }
    if (o_is_int(dt)) {
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
        for (int64_t i = 0; i < n; ++i) {
            int32_t u = ld_i(dt, a, i), v = ld_i(dt, b, i);
            uint32_t r = op == B_ADD ? (uint32_t)u + (uint32_t)v
                       : op == B_MUL ? (uint32_t)u * (uint32_t)v
                                     : (uint32_t)(u < v ? 1 : 0);
            st_i(dt, y, i, r);
        }
        return 0;
    }
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float u = ld_f(dt, a, i), v = ld_f(dt, b, i);
        float r = op == B_ADD ? u + v : op == B_MUL ? u * v : (u < v ? 1.0f : 0.0f);
        st_f(dt, y, i, r);
    }
    return 0;
}

/* WHERE: c != 0 (a NaN condition counts as nonzero) selects x, else y. */
int orc_where(int dtc, const void* c, int dt, const void* x, const void* y, void* out, int64_t n,
              int nthreads)
{
    int es = o_size(dt);
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        int t;
        if (o_is_int(dtc)) t = ld_i(dtc, c, i) != 0;
        else if (dtc == O_F64) t = ((const double*)c)[i] != 0.0;
        else t = ld_f(dtc, c, i) != 0.0f; /* NaN != 0 is true */
        memcpy((char*)out + i * es, (const char*)(t ? x : y) + i * es, (size_t)es);
    }
    return 0;
}

/* ---- reduce nodes ------------------------------------------------------ */

/* MAX of two floats: NaN propagates; on a tie between +0 and -0 the result is
 * +0; the identity is -inf (never 0: Litmus, "The corpus", reduction_init). */
static float fmax_step(float acc, float x)
{
    if (acc != acc) return acc;
    if (x != x || x > acc || (x == acc && !signbit(x))) return x;
    return acc;
}
static double dmax_step(double acc, double x)
{
    if (acc != acc) return acc;
    if (x != x || x > acc || (x == acc && !signbit(x))) return x;
    return acc;
}

/* SUM or MAX over the last dim of a contiguous [rows, cols] array, folding
 * j = 0, 1, ... in order; float32 running total for float16/bfloat16/float32,
 * rounded once into the dtype at the end.  Output [rows]. */
int orc_reduce(int op, int dt, const void* x, int64_t rows, int64_t cols, void* out, int nthreads)
{
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t base = r * cols;
        if (dt == O_F64) {
            const double* xd = (const double*)x;
            double acc = op == R_SUM ? 0.0 : -INFINITY;
            for (int64_t j = 0; j < cols; ++j)
                acc = op == R_SUM ? acc + xd[base + j] : dmax_step(acc, xd[base + j]);
            ((double*)out)[r] = acc;
        } else if (o_is_int(dt)) {
            uint32_t acc = op == R_SUM ? 0u
                         : (uint32_t)(dt == O_I32 ? INT32_MIN : dt == O_I16 ? INT16_MIN : INT8_MIN);
            for (int64_t j = 0; j < cols; ++j) {
                int32_t v = ld_i(dt, x, base + j);
                if (op == R_SUM) acc += (uint32_t)v;
                else if (v > (int32_t)acc) acc = (uint32_t)v;
            }
            st_i(dt, out, r, acc);
        } else {
            float acc = op == R_SUM ? 0.0f : -INFINITY;
            for (int64_t j = 0; j < cols; ++j) {
                float v = ld_f(dt, x, base + j);
                acc = op == R_SUM ? acc + v : fmax_step(acc, v);
            }
            st_f(dt, out, r, acc);
        }
    }
    return 0;
}

/* ---- fused MUL+SUM loop (Luminal IR blog, "Naive Matrix Multiplication") --
 * C[i,j] = sum over k ascending of A[i,k]*B[k,j]: the product rounds (a MUL
 * node), then the running total rounds (an ADD into a float32 accumulator),
 * which is exactly what the literal broadcast-MUL node followed by a SUM node
 * computes, in the same k order.  A is [M,K] and B is [K,N], both row-major
 * (the blog's loop indexes B as B[k*p + j]).  Output rounded to dtc once. */
int orc_matmul(int dtab, const void* A, const void* B, int dtc, void* C, int64_t M, int64_t N,
               int64_t K, int nthreads)
{
    if (o_is_int(dtab)) {
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
        for (int64_t i = 0; i < M; ++i)
            for (int64_t j = 0; j < N; ++j) {
                uint32_t acc = 0;
                for (int64_t k = 0; k < K; ++k)
                    acc += (uint32_t)ld_i(dtab, A, i * K + k) * (uint32_t)ld_i(dtab, B, k * N + j);
                st_i(dtc, C, i * N + j, acc);
            }
        return 0;
    }
    if (dtab == O_F64) {
        const double* a = (const double*)A;
        const double* b = (const double*)B;
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
        for (int64_t i = 0; i < M; ++i)
            for (int64_t j = 0; j < N; ++j) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double p = a[i * K + k] * b[k * N + j];
                    acc = acc + p;
                }
                ((double*)C)[i * N + j] = acc;
            }
        return 0;
    }
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                float p = ld_f(dtab, A, i * K + k) * ld_f(dtab, B, k * N + j);
                acc = acc + p;
            }
            st_f(dtc, C, i * N + j, acc);
        }
    return 0;
}

/* The same loop with B stored transposed (BT[j*K + k] = B[k*N + j]): the
 * products and the k order are those of orc_matmul, so the bits are too; only
 * the memory walk is friendlier to a CPU cache. */
int orc_matmul_bt(int dtab, const void* A, const void* BT, int dtc, void* C, int64_t M, int64_t N,
                  int64_t K, int nthreads)
{
    if (dtab == O_F64) {
        const double* a = (const double*)A;
        const double* b = (const double*)BT;
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
        for (int64_t i = 0; i < M; ++i)
            for (int64_t j = 0; j < N; ++j) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double p = a[i * K + k] * b[j * K + k];
                    acc = acc + p;
                }
                ((double*)C)[i * N + j] = acc;
            }
        return 0;
    }
    if (o_is_int(dtab)) return -2;
    float* af = (float*)malloc((size_t)(M * K) * sizeof(float));
    float* bf = (float*)malloc((size_t)(N * K) * sizeof(float));
    if (!af || !bf) { free(af); free(bf); return -1; }
    for (int64_t e = 0; e < M * K; ++e) af[e] = ld_f(dtab, A, e);
    for (int64_t e = 0; e < N * K; ++e) bf[e] = ld_f(dtab, BT, e);
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                float p = af[i * K + k] * bf[j * K + k];
                acc = acc + p;
            }
            st_f(dtc, C, i * N + j, acc);
        }
    free(af);
    free(bf);
    return 0;
}

/* The same loop for a list of sampled output cells (ii[s], jj[s]); the
 * float32 total is returned unrounded in acc[s] and also |a||b| summed in
 * absum[s] (the magnitude the reduction-order bound is stated against). */
int orc_matmul_cells(int dtab, const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                     const int64_t* ii, const int64_t* jj, int64_t ns, float* acc, double* absum,
                     int nthreads)
{
    (void)M;
#pragma omp parallel for num_threads(nthreads) if (nthreads > 1) schedule(static)
    for (int64_t s = 0; s < ns; ++s) {
        int64_t i = ii[s], j = jj[s];
        float t = 0.0f;
        double m = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            float a = ld_f(dtab, A, i * K + k), b = ld_f(dtab, B, k * N + j);
            float p = a * b;
            t = t + p;
            m += fabs((double)a * (double)b);
        }
        acc[s] = t;
        absum[s] = m;
    }
    return 0;
}

/* ---- indexed nodes ----------------------------------------------------- */

/* GATHER rows: out[n,:] = src[idx[n],:] for src [V, D] row-major.  An index
 * outside [0, V) is an error: that row is zero-filled and the count of bad
 * indices is returned. */
int64_t orc_gather_rows(int dt, const void* src, int64_t V, int64_t D, const int32_t* idx,
                        int64_t n, void* out)
{
    int es = o_size(dt);
    int64_t bad = 0;
    for (int64_t r = 0; r < n; ++r) {
        int64_t v = idx[r];
        if (v < 0 || v >= V) {
            memset((char*)out + r * D * es, 0, (size_t)(D * es));
            ++bad;
        } else {
            memcpy((char*)out + r * D * es, (const char*)src + v * D * es, (size_t)(D * es));
        }
    }
    return bad;
}

/* SCATTER-add rows: for n = 0, 1, ... in order, dst[idx[n],:] += upd[n,:].
 * Float destinations keep a float32 running total per cell starting from the
 * cell's value and round once into the dtype at the end (float64 in double);
 * integers wrap.  A bad index skips its row and is counted. */
int64_t orc_scatter_add_rows(int dt, void* dst, int64_t V, int64_t D, const int32_t* idx, int64_t n,
                             const void* upd)
{
    int64_t bad = 0;
    if (dt == O_F64) {
        double* d = (double*)dst;
        const double* u = (const double*)upd;
        for (int64_t r = 0; r < n; ++r) {
            int64_t v = idx[r];
            if (v < 0 || v >= V) { ++bad; continue; }
            for (int64_t c = 0; c < D; ++c) d[v * D + c] = d[v * D + c] + u[r * D + c];
        }
        return bad;
    }
    if (o_is_int(dt)) {
        for (int64_t r = 0; r < n; ++r) {
            int64_t v = idx[r];
            if (v < 0 || v >= V) { ++bad; continue; }
            for (int64_t c = 0; c < D; ++c)
                st_i(dt, dst, v * D + c,
                     (uint32_t)ld_i(dt, dst, v * D + c) + (uint32_t)ld_i(dt, upd, r * D + c));
        }
        return bad;
    }
    float* acc = (float*)malloc((size_t)(V * D) * sizeof(float));
    if (!acc) return -1;
    for (int64_t e = 0; e < V * D; ++e) acc[e] = ld_f(dt, dst, e);
    for (int64_t r = 0; r < n; ++r) {
        int64_t v = idx[r];
        if (v < 0 || v >= V) { ++bad; continue; }
        for (int64_t c = 0; c < D; ++c) acc[v * D + c] = acc[v * D + c] + ld_f(dt, upd, r * D + c);
    }
    for (int64_t e = 0; e < V * D; ++e) st_f(dt, dst, e, acc[e]);
    free(acc);
    return bad;
}

/* AdamW with decoupled weight decay, one step over one tensor, in float32,
 * every operation rounded in this order (the reading of limn's optimizer as
 * an ASSIGN graph; the arithmetic is Loshchilov & Hutter's AdamW in the
 * order torch.optim.AdamW applies it):
 *   p1 = p * (1 - lr*wd)
 *   m' = b1*m + (1-b1)*g          v' = b2*v + (1-b2)*(g*g)
 *   denom = sqrt(v') / sqrt(1 - b2t) + eps
 *   p' = p1 - (lr / (1 - b1t)) * (m' / denom)
 * b1t = b1^t and b2t = b2^t are the running products after this step.
 * p and g have dtype dt (f32 / bf16 / f16 storage, float32 compute; p'
 * rounds once into dt); m, v are float32. */
void orc_adamw(int dt, void* p, const void* g, float* m, float* v, int64_t n, float lr, float b1, float b2,
               float eps, float wd, float b1t, float b2t)
{
    const float decay = 1.0f - lr * wd;
    const float c1 = 1.0f - b1, c2 = 1.0f - b2;
    const float bc1 = 1.0f - b1t, bc2s = sqrtf(1.0f - b2t);
    const float step = lr / bc1;
    for (int64_t i = 0; i < n; ++i) {
        const float pi = ld_f(dt, p, i), gi = ld_f(dt, g, i);
        const float p1 = pi * decay;
        const float mi = b1 * m[i] + c1 * gi;
        const float g2 = gi * gi;
        const float vi = b2 * v[i] + c2 * g2;
        const float denom = sqrtf(vi) / bc2s + eps;
        const float upd = mi / denom;
        st_f(dt, p, i, p1 - step * upd);
        m[i] = mi;
        v[i] = vi;
    }
}

int orc_omp_max_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
