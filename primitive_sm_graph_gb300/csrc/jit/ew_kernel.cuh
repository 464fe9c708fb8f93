// Fused elementwise kernel skeleton (runtime-specialised per program).
//
// limn ("Backends") runs one thread per output cell; here one thread owns a
// chunk of PSG_VEC consecutive cells along the innermost dim, so contiguous
// operands move with 128-bit loads and stores and an expanded (stride-0)
// operand is read once per chunk.  Row offsets come from one multi-index
// decomposition per work item; within a row the View's index is col * stride.
// A block is split into row groups of a power-of-two size so short rows still
// fill it; long rows are cut into column tiles so that few rows (a fully
// contiguous space collapses to one) still spread over every SM.  A work item
// is one (row, tile) pair and the grid is persistent (a multiple of the SM
// count).
//
// kExact: the row length is a multiple of PSG_VEC, so every chunk is whole.
//
// The including source defines kNin, kInMode[], kInDt[], kOutDt, kExact and
// struct Body { template <class C> static void eval(const C&, T (&y)[PSG_VEC]); }.

struct EwCtx {
    const PsgEwParams& p;
    const i64 (&roff)[kNin > 0 ? kNin : 1];
    const bool (&rok)[kNin > 0 ? kNin : 1];
    i64 col0;
    int nvalid;
    template <int K>
    __device__ __forceinline__ void ldv(typename VT<kInDt[K]>::T (&d)[PSG_VEC]) const
    {
        ld_chunk<kInDt[K], kInMode[K]>(p.in[K], roff[K], rok[K], col0, nvalid, d);
    }
    template <int K>
    __device__ __forceinline__ typename VT<kInDt[K]>::T ld1() const
    {
        return ld_first<kInDt[K], kInMode[K]>(p.in[K], roff[K], rok[K], col0);
    }
};

extern "C" __global__ void __launch_bounds__(256) psg_ew(const __grid_constant__ PsgEwParams p)
{
    pdl_enter();
    const int gs = 1 << p.group_log2;
    const int groups = 256 >> p.group_log2;
    const int grp = threadIdx.x >> p.group_log2;
    const int lane = threadIdx.x & (gs - 1);
    const i64 items = p.rows * p.tiles;
    for (i64 it = (i64)blockIdx.x * groups + grp; it < items; it += (i64)gridDim.x * groups) {
        const i64 row = p.tiles == 1 ? it : it / p.tiles;
        const i64 c0 = (it - row * p.tiles) * p.tile_chunks;
        const i64 c1 = c0 + p.tile_chunks < p.chunks ? c0 + p.tile_chunks : p.chunks;
        i64 roff[kNin > 0 ? kNin : 1];
        bool rok[kNin > 0 ? kNin : 1];
        i64 ooff;
        row_offsets<kNin>(p.in, p.out, p.shape, p.nd, row, roff, rok, kInMode, ooff);
        if (c0 + lane >= c1) continue;
        const EwCtx cu{p, roff, rok, 0, PSG_VEC};
        const typename Body::U u = Body::uni(cu);  // the row's uniform values, once
        for (i64 ch = c0 + lane; ch < c1; ch += gs) {
            const i64 col0 = ch * PSG_VEC;
            const i64 left = p.inner - col0;
            const int nvalid = kExact || left >= PSG_VEC ? PSG_VEC : (int)left;
            const EwCtx c{p, roff, rok, col0, nvalid};
            typename VT<kOutDt>::T y[PSG_VEC];
            Body::eval(c, u, y);
            st_chunk<kOutDt, kOutMode>(p.out, ooff, col0, nvalid, y);
        }
    }
}
