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

struct EpiCtx {
    const TcParams& p;
    int b, m, col0;     // the cell (b, m, col0 .. col0 + PSG_VEC - 1) of C
    const float* acc;   // the float32 totals of those PSG_VEC cells

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
                const uint4 w = __ldg((const uint4*)((const u16*)o.ptr + base + col0));
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
    __device__ __forceinline__ static U row_uni(const TcParams& p, int b, int m)
    {
        const EpiCtx c{p, b, m, 0, nullptr};
        return Prog::uni(c);
    }
    __device__ __forceinline__ static void apply(const TcParams& p, const U& u, int b, int m, int n0,
                                                 uint32_t (&rr)[2][32])
    {
#pragma unroll
        for (int q = 0; q < 64 / PSG_VEC; ++q) {
            float acc[PSG_VEC];
#pragma unroll
            for (int v = 0; v < PSG_VEC; ++v) acc[v] = __uint_as_float(rr[q >> 2][(q & 3) * PSG_VEC + v]);
            const EpiCtx c{p, b, m, n0 + q * PSG_VEC, acc};
            float y[PSG_VEC];
            Prog::eval(c, u, y);
#pragma unroll
            for (int v = 0; v < PSG_VEC; ++v) rr[q >> 2][(q & 3) * PSG_VEC + v] = __float_as_uint(y[v]);
        }
    }
};
