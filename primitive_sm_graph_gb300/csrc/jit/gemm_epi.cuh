// A fused epilogue program in the tensor-core contraction (compiled by NVRTC
// only, after gemm_body.cuh and the spec's operand tables kEpiDt[] and
// kEpiMode[]).  The program's nodes come from gen_eval: ACC, the cell's
// float32 total, is read as the stashed value; LOAD k reads epilogue input k
// at the same cell (b, m, n) of C.  Each node rounds into its own dtype, as a
// node of the op graph does; the last one is rounded by C's store.
//
// Operand modes (kEpiMode): EPI_ROW is constant along n (stride 0: read once
// per row), EPI_VEC has unit n stride with every 8-cell chunk 16-byte
// aligned (vector loads), EPI_STRIDED is anything else (one load a cell).
#define EPI_ROW 0
#define EPI_VEC 1
#define EPI_STRIDED 2

// Inputs fetched ahead: half-width EPI_VEC operands, one 16-byte word per
// 8-cell chunk of a 64-column slice, at most two of them (the registers of
// two slices in flight); other inputs load inside the program.
__host__ __device__ constexpr bool epi_raw_ok(int k)
{
    return k < kEpiN && kEpiMode[k] == EPI_VEC && (kEpiDt[k] == PSG_DT_BF16 || kEpiDt[k] == PSG_DT_F16);
}
__host__ __device__ constexpr int epi_raw_slot(int k)
{
    int s = 0;
    for (int j = 0; j < k; ++j)
        if (epi_raw_ok(j)) ++s;
    return epi_raw_ok(k) && s < 2 ? s : -1;
}
__host__ __device__ constexpr int epi_raw_count()
{
    int s = 0;
    for (int k = 0; k < 8; ++k)
        if (epi_raw_slot(k) >= 0) ++s;
    return s;
}
constexpr int kEpiRaw = epi_raw_count();
struct EpiRaw {
    uint4 w[kEpiRaw > 0 ? kEpiRaw : 1][64 / PSG_VEC];
};

struct EpiCtx {
    const TcParams& p;
    int b, m, col0;     // the cell (b, m, col0 .. col0 + PSG_VEC - 1) of C
    const float* acc;   // the float32 totals of those PSG_VEC cells
    const EpiRaw* raw;  // the slice's fetched words (chunk q), or null
    int q;

    // one value of a row-constant operand
    template <int K>
    __device__ __forceinline__ typename VT<kEpiDt[K]>::T ld1() const
    {
        const TcEpiOperand& o = p.epi[K];
        return ld_cell<kEpiDt[K]>(o.ptr, (i64)b * o.sb + (i64)m * o.sm);
    }
    // PSG_VEC consecutive cells along n (0 past C's last column)
    template <int K>
    __device__ __forceinline__ void ldv(typename VT<kEpiDt[K]>::T (&out)[PSG_VEC]) const
    {
        constexpr int DT = kEpiDt[K];
        const TcEpiOperand& o = p.epi[K];
        const i64 base = (i64)b * o.sb + (i64)m * o.sm;
        const int left = p.N - col0;
        if constexpr (kEpiMode[K] == EPI_VEC && (DT == PSG_DT_BF16 || DT == PSG_DT_F16)) {
            if (left >= PSG_VEC) {
                uint4 w;
                if constexpr (epi_raw_slot(K) >= 0) w = raw->w[epi_raw_slot(K)][q];
                else w = __ldg((const uint4*)((const u16*)o.ptr + base + col0));
                const u32 ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int v = 0; v < PSG_VEC; ++v) {
                    const u32 h = (ws[v >> 1] >> ((v & 1) * 16)) & 0xffffu;
                    out[v] = DT == PSG_DT_BF16 ? __uint_as_float(h << 16) : h2f((u16)h);
                }
                return;
            }
        } else if constexpr (kEpiMode[K] == EPI_VEC && DT == PSG_DT_F32) {
            if (left >= PSG_VEC) {
                const float4 lo = __ldg((const float4*)((const float*)o.ptr + base + col0));
                const float4 hi = __ldg((const float4*)((const float*)o.ptr + base + col0) + 1);
                out[0] = lo.x; out[1] = lo.y; out[2] = lo.z; out[3] = lo.w;
                out[4] = hi.x; out[5] = hi.y; out[6] = hi.z; out[7] = hi.w;
                return;
            }
        }
#pragma unroll
        for (int v = 0; v < PSG_VEC; ++v)
            out[v] = v < left ? ld_cell<DT>(o.ptr, base + (i64)(col0 + v) * o.sn) : (typename VT<DT>::T)0;
    }
    __device__ __forceinline__ float stashf(int v) const { return acc[v]; }
    __device__ __forceinline__ int stashi(int v) const { return 0; }
};

// The epilogue class of gemm_body.cuh for a generated program Prog.
template <class Prog>
struct EpiJit {
    static constexpr bool active = true;
    typedef typename Prog::U U;
    typedef EpiRaw Raw;
    __device__ __forceinline__ static U row_uni(const TcParams& p, int b, int m)
    {
        const EpiCtx c{p, b, m, 0, nullptr, nullptr, 0};
        return Prog::uni(c);
    }
    // an L2 prefetch of row m's contiguous (EPI_VEC) inputs over `cols`
    // columns from n0, one request per 128-byte line
    __device__ __forceinline__ static void prefetch_l2(const TcParams& p, int b, int m, int n0, int cols)
    {
        if (m >= p.M || n0 >= p.N) return;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k >= kEpiN || kEpiMode[k] != EPI_VEC) continue;
            const TcEpiOperand& o = p.epi[k];
            const int es = kEpiDt[k] == PSG_DT_F32 ? 4 : 2;  // EPI_VEC inputs are float-typed
            const char* row = (const char*)o.ptr + ((i64)b * o.sb + (i64)m * o.sm + n0) * es;
            const int span = (p.N - n0 < cols ? p.N - n0 : cols) * es;
            for (int off = 0; off < span; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
        }
    }
    // the fetched inputs' words of the 64-column slice at n0
    __device__ __forceinline__ static void fetch(const TcParams& p, int b, int m, int n0, EpiRaw& r)
    {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int s = epi_raw_slot(k);
            if (s < 0) continue;
            const TcEpiOperand& o = p.epi[k];
            const u16* row = (const u16*)o.ptr + (i64)b * o.sb + (i64)m * o.sm;
#pragma unroll
            for (int q = 0; q < 64 / PSG_VEC; ++q) {
                const int col0 = n0 + q * PSG_VEC;
                r.w[s][q] = p.N - col0 >= PSG_VEC ? __ldg((const uint4*)(row + col0)) : make_uint4(0, 0, 0, 0);
            }
        }
    }
    __device__ __forceinline__ static void apply(const TcParams& p, const U& u, int b, int m, int n0,
                                                 uint32_t (&rr)[2][32], const EpiRaw& raw)
    {
#pragma unroll
        for (int q = 0; q < 64 / PSG_VEC; ++q) {
            float acc[PSG_VEC];
#pragma unroll
            for (int v = 0; v < PSG_VEC; ++v) acc[v] = __uint_as_float(rr[q >> 2][(q & 3) * PSG_VEC + v]);
            const EpiCtx c{p, b, m, n0 + q * PSG_VEC, acc, &raw, q};
            float y[PSG_VEC];
            Prog::eval(c, u, y);
#pragma unroll
            for (int v = 0; v < PSG_VEC; ++v) rr[q >> 2][(q & 3) * PSG_VEC + v] = __float_as_uint(y[v]);
        }
    }
};
