// Row reduction skeleton (runtime-specialised per set of stage programs).
//
// A team of T = 1 << team_log2 threads (T <= 256, the block size) owns one
// row of length N (the last dim; limn, "Reading the schedule": a reduce is a
// cut and elementwise work fuses into it).  Each thread holds chunks lane,
// lane+T, ... of PSG_VEC cells.  When the row fits (kCH chunks per thread,
// kCH > 0) the inputs are loaded once into registers and every stage and the
// epilogue read them from there, so the row costs one HBM read and one
// write; otherwise every stage streams the row again.  A stage folds its
// prologue values per thread, then across the warp with shuffles and across
// the team's warps through shared memory in a fixed order (the same bits
// every run).  Within a thread each
// of the PSG_VEC lane slots keeps its own running value, so the fold is
// PSG_VEC short chains and a three-level tree instead of one long chain.
// The running total is float32 (int32 for ints) and rounds into the stage
// dtype once (limn, "The op set": a reduce keeps its running total in
// float32).
//
// Only inputs that change from row to row are cached (kCacheIn); bfloat16
// cells are held packed, two to a word.  When the epilogue begins with the
// whole program of stage kStash, that stage keeps its per-cell values
// (the stash) and the epilogue reads them instead of computing them again.
//
// kExact: every thread's kCH chunks are whole and inside the row, so no
// chunk needs a range check.
//
// kColumnar: the reduced axis is strided and the rows sit next to each other
// in memory (a sum over the leading axis of a row-major tensor).  A team is
// then one thread in each warp of the block (its member index is the warp)
// and the block's 32 teams are 32 adjacent rows, so one warp's load of a
// cell index covers 32 adjacent cells.  With kCluster > 1 a thread-block
// cluster shares the rows: CTA rank c holds members c*M .. c*M + M - 1 and
// every CTA folds all members' partials, read from each rank's shared
// memory in rank order, so each gets the same total.
//
// The including source defines kNin, kInMode[], kInDt[], kOutDt, kNstages,
// kStageOp[], kStageDt[], kCH, kExact, kCacheIn[], kStash, kPerRow, the
// staged-mode constants, StageBody<S> and Epi.

template <int V> struct IC { static constexpr int value = V; };
template <int J, int N, class F>
__device__ __forceinline__ void sfor(F& f)
{
    if constexpr (J < N) {
        f(IC<J>{});
        sfor<J + 1, N>(f);
    }
}

#define PSG_RED_SUM 0
#define PSG_RED_MAX 1
constexpr int kNinP = kNin > 0 ? kNin : 1;
constexpr int kCHP = kCH > 0 ? kCH : 1;

// MAX: NaN propagates, +0 beats -0 on a tie, so any order gives the same
// bits.  max.NaN gives a NaN when either operand is one and treats -0 as
// below +0 (checked on this hardware for both operand orders, and by the
// signed-zero tests across every fold layout).
__device__ __forceinline__ float fmax_step(float acc, float x)
{
    float m;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(m) : "f"(acc), "f"(x));
    return m;
}

template <int OP, int DT>
struct Fold {
    typedef typename VT<DT>::T T;
    static __device__ __forceinline__ T identity()
    {
        if constexpr (OP == PSG_RED_SUM) return (T)0;
        else if constexpr (DT == PSG_DT_I32) return (int)0x80000000;
        else if constexpr (DT == PSG_DT_I16) return -32768;
        else if constexpr (DT == PSG_DT_I8) return -128;
        else return __uint_as_float(0xff800000u);  // -inf
    }
    static __device__ __forceinline__ T step(T acc, T x)
    {
        if constexpr (OP == PSG_RED_SUM) {
            if constexpr (DT == PSG_DT_I32 || DT == PSG_DT_I16 || DT == PSG_DT_I8) return addi(acc, x);
            else return __fadd_rn(acc, x);
        } else {
            if constexpr (DT == PSG_DT_I32 || DT == PSG_DT_I16 || DT == PSG_DT_I8) return x > acc ? x : acc;
            else return fmax_step(acc, x);
        }
    }
    // the total rounds into the stage dtype once
    static __device__ __forceinline__ T finish(T v)
    {
        if constexpr (DT == PSG_DT_BF16) return rbf(v);
        else if constexpr (DT == PSG_DT_F16) return rh(v);
        else if constexpr (DT == PSG_DT_I16) return w16(v);
        else if constexpr (DT == PSG_DT_I8) return w8(v);
        else return v;
    }
};

__device__ __forceinline__ u32 as_bits(float x) { return __float_as_uint(x); }
__device__ __forceinline__ u32 as_bits(int x) { return (u32)x; }
template <class T> __device__ __forceinline__ T from_bits(u32 b);
template <> __device__ __forceinline__ float from_bits<float>(u32 b) { return __uint_as_float(b); }
template <> __device__ __forceinline__ int from_bits<int>(u32 b) { return (int)b; }

// ---- staged rows: shared-memory ring filled by bulk copies ---------------
__device__ __forceinline__ u32 smem_addr(const void* p) { return (u32)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(unsigned long long* b, u32 count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* b, u32 bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(unsigned long long* b, u32 parity)
{
    u32 ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
constexpr long long kWaitCycles = 2000000000ll;  // about one second
// true when the phase completed; false once `limit` cycles have passed
// (PSG_E_TIMEOUT goes to the status word)
__device__ __noinline__ bool mbar_wait(unsigned long long* b, u32 parity, int* status, long long limit)
{
    const long long t0 = clock64();
    for (u32 i = 0;; ++i) {
        if (mbar_try(b, parity)) return true;
        if ((i & 7) == 7 && clock64() - t0 > limit) {
            if (status) atomicCAS(status, 0, PSG_DEV_E_TIMEOUT);
            return false;
        }
    }
}
// one contiguous global range -> shared memory, completing on mbarrier b
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, u32 bytes, unsigned long long* b)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(b))
                 : "memory");
}
// the PSG_VEC cells at col0 of a staged row segment (16-byte shared loads)
template <int DT>
__device__ __forceinline__ void ld_staged(const unsigned char* seg, i64 col0, typename VT<DT>::T (&d)[PSG_VEC])
{
    if constexpr (DT == PSG_DT_F32 || DT == PSG_DT_I32) {
        const uint4* q = (const uint4*)(seg + col0 * 4);
        const uint4 x = q[0], y = q[1];
        const u32 w[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
        for (int v = 0; v < PSG_VEC; ++v) {
            if constexpr (DT == PSG_DT_F32) d[v] = __uint_as_float(w[v]);
            else d[v] = (int)w[v];
        }
    } else {
        const uint4 x = *(const uint4*)(seg + col0 * 2);
        const u32 w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            if constexpr (DT == PSG_DT_BF16) {
                d[2 * v] = __uint_as_float(w[v] << 16);
                d[2 * v + 1] = __uint_as_float(w[v] & 0xffff0000u);
            } else {
                d[2 * v] = h2f((u16)(w[v] & 0xffffu));
                d[2 * v + 1] = h2f((u16)(w[v] >> 16));
            }
        }
    }
}

struct RedCtx {
    const PsgRedParams& p;
    const i64 (&roff)[kNinP];
    const bool (&rok)[kNinP];
    const u32 (&cache)[kNinP][kCHP][PSG_VEC];
    const u32 (&stash)[kCHP][PSG_VEC];
    const u32 (&red)[PSG_MAXSTAGES];
    const unsigned char* sb;  // the row's stage in shared memory (staged mode)
    i64 col0;
    int nvalid;
    int j;  // chunk slot (compile-time after unrolling)
    template <int K>
    __device__ __forceinline__ void ldv(typename VT<kInDt[K]>::T (&d)[PSG_VEC]) const
    {
        typedef typename VT<kInDt[K]>::T T;
        if constexpr (kStaged && kStagedIn[K]) {
            ld_staged<kInDt[K]>(sb + kSegOff[K], col0, d);
        } else if constexpr (kCH > 0 && kCacheIn[K] && kInDt[K] == PSG_DT_BF16) {
#pragma unroll
            for (int w = 0; w < PSG_VEC / 2; ++w) {
                d[2 * w] = __uint_as_float(cache[K][j][w] << 16);
                d[2 * w + 1] = __uint_as_float(cache[K][j][w] & 0xffff0000u);
            }
        } else if constexpr (kCH > 0 && kCacheIn[K]) {
#pragma unroll
            for (int v = 0; v < PSG_VEC; ++v) d[v] = from_bits<T>(cache[K][j][v]);
        } else {
            ld_chunk<kInDt[K], kInMode[K]>(p.in[K], roff[K], rok[K], col0, nvalid, d);
        }
    }
    template <int K>
    __device__ __forceinline__ typename VT<kInDt[K]>::T ld1() const
    {
        return ld_first<kInDt[K], kInMode[K]>(p.in[K], roff[K], rok[K], col0);
    }
    __device__ __forceinline__ float redf(int s) const { return __uint_as_float(red[s]); }
    __device__ __forceinline__ int redi(int s) const { return (int)red[s]; }
    __device__ __forceinline__ float stashf(int v) const { return __uint_as_float(stash[j][v]); }
    __device__ __forceinline__ int stashi(int v) const { return (int)stash[j][v]; }
};

// ---- columnar teams: fold across warps (and the cluster's CTAs) ----------
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ u32 ld_rank(const u32* p, int rank)
{
    u32 a, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
// v: this member's partial for row (threadIdx.x & 31); sm: [M * 32] words,
// cpart: [32].  Warp 0 folds the CTA's members 0, 1, .. in order; then every
// thread folds the ranks' CTA totals 0, 1, .. in order: one tree for all.
template <int OP, int DT>
__device__ __forceinline__ typename VT<DT>::T col_fold(typename VT<DT>::T v, u32* sm, u32* cpart)
{
    typedef Fold<OP, DT> F;
    typedef typename VT<DT>::T T;
    constexpr int MM = kBlockThreads / 32;  // members per CTA at the launch bound
    const int M = blockDim.x >> 5, t = threadIdx.x & 31;
    sm[(threadIdx.x >> 5) * 32 + t] = as_bits(v);
    __syncthreads();
    if (threadIdx.x < 32) {
        u32 part[MM];  // every partial loaded before the first add
#pragma unroll
        for (int m = 0; m < MM; ++m) part[m] = m < M ? sm[m * 32 + t] : 0u;
        T r = from_bits<T>(part[0]);
#pragma unroll
        for (int m = 1; m < MM; ++m)
            if (m < M) r = F::step(r, from_bits<T>(part[m]));
        cpart[t] = as_bits(r);
    }
    if constexpr (kCluster > 1) cluster_sync_all();
    else __syncthreads();
    u32 q[kCluster];
#pragma unroll
    for (int c = 0; c < kCluster; ++c) q[c] = kCluster > 1 ? ld_rank(cpart + t, c) : cpart[t];
    T r = from_bits<T>(q[0]);
#pragma unroll
    for (int c = 1; c < kCluster; ++c) r = F::step(r, from_bits<T>(q[c]));
    // nobody rewrites sm or cpart (or leaves the cluster) while another still reads them
    if constexpr (kCluster > 1) cluster_sync_all();
    else __syncthreads();
    return r;
}

// ---- kColVec: columnar rows eight to a thread ------------------------------
// A thread's PSG_VEC lanes are eight adjacent rows (the cells next to each
// other in memory), and a chunk is one index r of the reduced axis: an input
// that moves with the row is read as one 16-byte (32-byte for float32) vector
// at r, an input that does not is read once and shared by the lanes.  A warp
// holds kVecRT row threads (kVecRT * 8 rows) by 32 / kVecRT slots of the
// reduced axis; the members of a row group are those slots over the CTA's
// warps and the cluster's CTAs.  One stage, one output per row.
constexpr int kVecRS = 32 / kVecRT;

template <int DT>
__device__ __forceinline__ void ld_rowvec(const void* p, i64 o, typename VT<DT>::T (&d)[PSG_VEC])
{
    if constexpr (DT == PSG_DT_F32) {
        const uint4* q = (const uint4*)((const float*)p + o);
        const uint4 a = __ldg(q), b = __ldg(q + 1);
        const u32 w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int v = 0; v < PSG_VEC; ++v) d[v] = __uint_as_float(w[v]);
    } else {
        const uint4 a = __ldg((const uint4*)((const u16*)p + o));
        const u32 w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            if constexpr (DT == PSG_DT_BF16) {
                d[2 * v] = __uint_as_float(w[v] << 16);
                d[2 * v + 1] = __uint_as_float(w[v] & 0xffff0000u);
            } else {
                d[2 * v] = h2f((u16)(w[v] & 0xffffu));
                d[2 * v + 1] = h2f((u16)(w[v] >> 16));
            }
        }
    }
}

struct VecCtx {
    const PsgRedParams& p;
    const i64 (&roff)[kNinP];  // each input's offset at the thread's first row, r = 0
    i64 r;
    const u32* red;
    template <int K>
    __device__ __forceinline__ void ldv(typename VT<kInDt[K]>::T (&d)[PSG_VEC]) const
    {
        const i64 o = roff[K] + r * p.in[K].inner_stride;
        if constexpr (kVecRow[K]) {
            ld_rowvec<kInDt[K]>(p.in[K].ptr, o, d);
        } else {
            const typename VT<kInDt[K]>::T x = ld_cell<kInDt[K]>(p.in[K].ptr, o);
#pragma unroll
            for (int v = 0; v < PSG_VEC; ++v) d[v] = x;
        }
    }
    template <int K>
    __device__ __forceinline__ typename VT<kInDt[K]>::T ld1() const
    {
        return ld_cell<kInDt[K]>(p.in[K].ptr, roff[K]);
    }
    __device__ __forceinline__ float redf(int s) const { return __uint_as_float(red[s]); }
    __device__ __forceinline__ int redi(int s) const { return (int)red[s]; }
    __device__ __forceinline__ float stashf(int) const { return 0.0f; }
    __device__ __forceinline__ int stashi(int) const { return 0; }
};

// fold: [warps][kVecRT][PSG_VEC] words; cpart: [kVecRT][PSG_VEC] = 32 words
__device__ __forceinline__ void colvec_body(const PsgRedParams& p, u32* fold, u32* cpart)
{
    typedef Fold<kStageOp[0], kStageDt[0]> F;
    typedef typename VT<kStageDt[0]>::T T;
    const int warp = threadIdx.x >> 5, l = threadIdx.x & 31;
    const int rt = l % kVecRT, rs = l / kVecRT;
    const int W = blockDim.x >> 5;
    const int rank = kCluster > 1 ? (int)(blockIdx.x % kCluster) : 0;
    const i64 member = ((i64)rank * W + warp) * kVecRS + rs;
    const i64 TM = (i64)kCluster * W * kVecRS;  // members of a row group
    const i64 rows_cta = (i64)kVecRT * PSG_VEC;
    const i64 groups = (p.rows + rows_cta - 1) / rows_cta;
    const u32 nored[PSG_MAXSTAGES] = {0u, 0u, 0u, 0u};
    for (i64 g = blockIdx.x / kCluster; g < groups; g += gridDim.x / kCluster) {
        const i64 j0 = g * rows_cta + (i64)rt * PSG_VEC;
        const bool active = j0 < p.rows;  // rows come in whole groups of PSG_VEC
        i64 roff[kNinP];
        bool rok[kNinP];
        i64 ooff = 0;
        if (active) {
            row_offsets<kNin>(p.in, p.out, p.shape, p.nd, j0, roff, rok, kInMode, ooff);
        } else {
#pragma unroll
            for (int k = 0; k < kNinP; ++k) roff[k] = 0;
        }
        T accv[PSG_VEC];
#pragma unroll
        for (int v = 0; v < PSG_VEC; ++v) accv[v] = F::identity();
        if (active) {
            const VecCtx cu{p, roff, 0, nored};
            const typename StageBody<0>::U u = StageBody<0>::uni(cu);
            i64 r = member;
            // four reduced indices at a time: their loads all go out together
            for (; r + 3 * TM < p.inner; r += 4 * TM) {
                T y[4][PSG_VEC];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const VecCtx c{p, roff, r + q * TM, nored};
                    StageBody<0>::eval(c, u, y[q]);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int v = 0; v < PSG_VEC; ++v) accv[v] = F::step(accv[v], y[q][v]);
            }
            for (; r < p.inner; r += TM) {
                const VecCtx c{p, roff, r, nored};
                T y[PSG_VEC];
                StageBody<0>::eval(c, u, y);
#pragma unroll
                for (int v = 0; v < PSG_VEC; ++v) accv[v] = F::step(accv[v], y[v]);
            }
        }
        // one fixed tree, the same bits on every run: the warp's slots by
        // shuffles (xor 4, 8, 16), then the CTA's warps in order, then the
        // cluster's CTAs in rank order; lane rt * PSG_VEC + v of warp 0 owns
        // row j0(rt) + v from the second level on
#pragma unroll
        for (int off = kVecRT; off < 32; off <<= 1)
#pragma unroll
            for (int v = 0; v < PSG_VEC; ++v)
                accv[v] = F::step(accv[v], from_bits<T>(__shfl_xor_sync(0xffffffffu, as_bits(accv[v]), off, 32)));
        if (rs == 0) {
#pragma unroll
            for (int v = 0; v < PSG_VEC; ++v) fold[(warp * kVecRT + rt) * PSG_VEC + v] = as_bits(accv[v]);
        }
        __syncthreads();
        constexpr int MW = kBlockThreads / 32;  // warps at the launch bound
        if (warp == 0) {
            u32 part[MW];  // every warp's partial loaded before the first add
#pragma unroll
            for (int m = 0; m < MW; ++m) part[m] = m < W ? fold[m * 32 + l] : 0u;
            T a = from_bits<T>(part[0]);
#pragma unroll
            for (int m = 1; m < MW; ++m)
                if (m < W) a = F::step(a, from_bits<T>(part[m]));
            cpart[l] = as_bits(a);
        }
        if constexpr (kCluster > 1) cluster_sync_all();
        else __syncthreads();
        const int ort = l / PSG_VEC, ov = l % PSG_VEC;  // the row this lane of warp 0 finishes
        const i64 oj = g * rows_cta + (i64)ort * PSG_VEC + ov;
        if (rank == 0 && warp == 0 && oj < p.rows) {
            T a = from_bits<T>(kCluster > 1 ? ld_rank(cpart + l, 0) : cpart[l]);
#pragma unroll
            for (int c = 1; c < kCluster; ++c) a = F::step(a, from_bits<T>(ld_rank(cpart + l, c)));
            const u32 red1[PSG_MAXSTAGES] = {as_bits(F::finish(a)), 0u, 0u, 0u};
            i64 ro2[kNinP];
            bool rk2[kNinP];
            i64 oo2 = 0;
            row_offsets<kNin>(p.in, p.out, p.shape, p.nd, oj, ro2, rk2, kInMode, oo2);
            const VecCtx ce{p, ro2, 0, red1};
            typename VT<kOutDt>::T y[PSG_VEC];
            Epi::eval(ce, Epi::uni(ce), y);
            st_cell<kOutDt>((void*)p.out.ptr, oo2, y[0]);
        }
        // nobody rewrites fold or cpart while another CTA of the cluster reads them
        if constexpr (kCluster > 1) cluster_sync_all();
        else __syncthreads();
    }
}

// fold v across the team (threads [team*T, team*T + T) of the block)
template <int OP, int DT>
__device__ __forceinline__ typename VT<DT>::T team_fold(typename VT<DT>::T v, int team_log2, u32* sm)
{
    typedef Fold<OP, DT> F;
    const int T = 1 << team_log2;
    const int width = T < 32 ? T : 32;
    for (int off = width >> 1; off > 0; off >>= 1) {
        const u32 o = __shfl_xor_sync(0xffffffffu, as_bits(v), off, 32);
        v = F::step(v, from_bits<typename VT<DT>::T>(o));
    }
    if (T > 32) {
        const int warp = threadIdx.x >> 5;
        const int W = T >> 5;
        const int team = threadIdx.x >> team_log2;
        if ((threadIdx.x & 31) == 0) sm[warp] = as_bits(v);
        __syncthreads();
        v = from_bits<typename VT<DT>::T>(sm[team * W]);
        for (int w = 1; w < W; ++w) v = F::step(v, from_bits<typename VT<DT>::T>(sm[team * W + w]));
        __syncthreads();
    }
    return v;
}

// the stash's registers: its own array, or the cached row of input A
template <int A, int NIN, int CH>
__device__ __forceinline__ u32 (&stash_ref(u32 (&cache)[NIN][CH][PSG_VEC], u32 (&own)[A >= 0 ? 1 : CH][PSG_VEC]))[CH][PSG_VEC]
{
    if constexpr (A >= 0) return cache[A];
    else return own;
}

extern "C" __global__ void __launch_bounds__(kBlockThreads, kMinBlocks) PSG_CLUSTER_DIMS psg_reduce(
    const __grid_constant__ PsgRedParams p)
{
    pdl_enter();
    __shared__ u32 sm[kColumnar ? kBlockThreads : 32];
    __shared__ u32 cpart[kColumnar ? 32 : 1];
    if constexpr (kColVec) {
        colvec_body(p, sm, cpart);
        return;
    }
    extern __shared__ __align__(128) unsigned char dsm[];  // staged mode: barriers, then the ring
    // members of a team (T), teams of a block, this thread's team and member index (lane)
    const int T = kColumnar ? (int)(blockDim.x >> 5) * kCluster : 1 << p.team_log2;
    const int teams = kColumnar ? 32 : (int)(blockDim.x >> p.team_log2);
    const int team = kColumnar ? (int)(threadIdx.x & 31) : (int)(threadIdx.x >> p.team_log2);
    const int lane = kColumnar ? (int)(blockIdx.x % kCluster) * (int)(blockDim.x >> 5) + (int)(threadIdx.x >> 5)
                               : (int)(threadIdx.x & (T - 1));
    unsigned long long* bars = (unsigned long long*)dsm;  // [teams][kNS]
    unsigned char* ring = dsm + kBarBytes;                 // [teams][kNS][kStageBytes]
    if constexpr (kStaged) {
        if (threadIdx.x < teams * kNS) mbar_init(&bars[threadIdx.x], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        __syncthreads();
    }
    // iteration it gives team `team` the row first + it * step + team; every
    // team of the block runs the same number of iterations, so the barriers
    // inside team_fold (and the staged ring's) are reached by all threads
    const i64 step = (i64)(gridDim.x / kCluster) * teams;
    const i64 first = (i64)(blockIdx.x / kCluster) * teams;
    const i64 niter = first < p.rows ? (p.rows - first + step - 1) / step : 0;
    // a staged wait gave up: this thread stops waiting (and, as the team's
    // issuing lane, stops filling the ring) and the kernel ends in bounded time
    bool dead = false;
    // ring slots lane 0 has filled, and the phase parity of each one's last
    // fill: every copy the team issued lands before the kernel may exit
    u32 armed = 0, armed_ph = 0;
    // staged mode: one lane of the team fills ring slot it % kNS with the
    // row of iteration it (one bulk copy per staged input)
    auto issue = [&](i64 it) {
        const i64 row = first + it * step + team;
        if (lane != 0 || row >= p.rows || dead) return;
        if (p.skip_first_copy && it == 0) return;  // test hook: a slot nothing fills
        i64 ro[kNinP];
        bool rk[kNinP];
        i64 oo;
        row_offsets<kNin>(p.in, p.out, p.shape, p.nd, row, ro, rk, kInMode, oo);
        const int slot = (int)(it % kNS);
        unsigned long long* b = &bars[team * kNS + slot];
        unsigned char* dst = ring + (size_t)(team * kNS + slot) * kStageBytes;
        // the team's reads of this slot (generic proxy) come before the copy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(b, kTxBytes);
        armed |= 1u << slot;
        armed_ph = (armed_ph & ~(1u << slot)) | ((u32)((it / kNS) & 1) << slot);
        auto cp = [&](auto kt) {
            constexpr int K = decltype(kt)::value;
            if constexpr (kStagedIn[K])
                bulk_g2s(dst + kSegOff[K], (const char*)p.in[K].ptr + ro[K] * kInSize[K], kRowBytes[K], b);
        };
        sfor<0, kNin>(cp);
    };
    if constexpr (kStaged) {
        for (i64 it = 0; it < kNS - 1 && it < niter; ++it) issue(it);
    }
    for (i64 it = 0; it < niter; ++it) {
        const i64 row = first + it * step + team;
        const bool active = row < p.rows;
        i64 roff[kNinP];
        bool rok[kNinP];
        i64 ooff = 0;
        if (active) {
            row_offsets<kNin>(p.in, p.out, p.shape, p.nd, row, roff, rok, kInMode, ooff);
        } else {
#pragma unroll
            for (int k = 0; k < kNinP; ++k) { roff[k] = 0; rok[k] = false; }
        }
        const unsigned char* sb = nullptr;
        if constexpr (kStaged) {
            if (it + kNS - 1 < niter) issue(it + kNS - 1);
            const int slot = (int)(it % kNS);
            sb = ring + (size_t)(team * kNS + slot) * kStageBytes;
            if (active && !dead)
                dead = !mbar_wait(&bars[team * kNS + slot], (u32)((it / kNS) & 1), p.status, p.wait_cycles);
        }
        // register-cache mode: load the row once
        u32 cache[kNinP][kCHP][PSG_VEC];
        if constexpr (kCH > 0) {
#pragma unroll
            for (int j = 0; j < kCH; ++j) {
                const i64 ch = lane + (i64)j * T;
                const i64 col0 = ch * PSG_VEC;
                const i64 left = p.inner - col0;
                const int nvalid = !active ? 0 : kExact ? PSG_VEC : left <= 0 ? 0 : left < PSG_VEC ? (int)left : PSG_VEC;
                auto ldk = [&](auto kt) {
                    constexpr int K = decltype(kt)::value;
                    if constexpr (kCacheIn[K]) {
                        typename VT<kInDt[K]>::T d[PSG_VEC];
                        if (nvalid > 0) ld_chunk<kInDt[K], kInMode[K]>(p.in[K], roff[K], rok[K], col0, nvalid, d);
                        if constexpr (kInDt[K] == PSG_DT_BF16) {
#pragma unroll
                            for (int w = 0; w < PSG_VEC / 2; ++w)
                                cache[K][j][w] = nvalid > 0 ? (__float_as_uint(d[2 * w]) >> 16) |
                                                                  (__float_as_uint(d[2 * w + 1]) & 0xffff0000u)
                                                            : 0u;
                        } else {
#pragma unroll
                            for (int v = 0; v < PSG_VEC; ++v) cache[K][j][v] = nvalid > 0 ? as_bits(d[v]) : 0u;
                        }
                    }
                };
                sfor<0, kNin>(ldk);
            }
        }
        u32 red[PSG_MAXSTAGES] = {0u, 0u, 0u, 0u};
        // the stash, or (kStashAlias >= 0) the cached row it overwrites
        u32 stash_own[kStashAlias >= 0 ? 1 : kCHP][PSG_VEC];
        u32 (&stash)[kCHP][PSG_VEC] = stash_ref<kStashAlias>(cache, stash_own);
        auto stage = [&](auto st) {
            constexpr int S = decltype(st)::value;
            constexpr int OP = kStageOp[S];
            constexpr int DT = kStageDt[S];
            typedef Fold<OP, DT> F;
            // one running value per lane slot v: PSG_VEC independent chains
            // (short dependency chains), folded in a fixed tree at the end
            typename VT<DT>::T accv[PSG_VEC];
#pragma unroll
            for (int v = 0; v < PSG_VEC; ++v) accv[v] = F::identity();
            const int nch = kCH > 0 ? kCH : (int)((p.chunks - lane + T - 1) / T);
            typename StageBody<S>::U u;
            if (active) {
                const RedCtx cu{p, roff, rok, cache, stash, red, sb, 0, PSG_VEC, 0};
                u = StageBody<S>::uni(cu);  // the row's uniform values, once
            }
            // streaming: the member's whole chunks first, kStreamUnroll at a
            // time with no range checks, so their loads can all go out together
            int jj0 = 0;
            if constexpr (kCH == 0 && kStreamUnroll > 1) {
                const i64 whole = p.inner / PSG_VEC;  // chunks entirely inside the row
                const int nw = active && lane < whole ? (int)((whole - lane + T - 1) / T) : 0;
                for (; jj0 + kStreamUnroll <= nw; jj0 += kStreamUnroll) {
#pragma unroll
                    for (int q = 0; q < kStreamUnroll; ++q) {
                        const i64 col0 = (lane + (i64)(jj0 + q) * T) * PSG_VEC;
                        const RedCtx c{p, roff, rok, cache, stash, red, sb, col0, PSG_VEC, 0};
                        typename VT<DT>::T y[PSG_VEC];
                        StageBody<S>::eval(c, u, y);
#pragma unroll
                        for (int v = 0; v < PSG_VEC; ++v) accv[v] = F::step(accv[v], y[v]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < (kCH > 0 ? kCH : 1); ++j) {
                for (int jj = (kCH > 0 ? j : jj0); jj < (kCH > 0 ? j + 1 : nch); ++jj) {
                    const i64 ch = lane + (i64)jj * T;
                    const i64 col0 = ch * PSG_VEC;
                    const i64 left = p.inner - col0;
                    if (!active || (!kExact && left <= 0)) continue;
                    const int nvalid = kExact ? PSG_VEC : left < PSG_VEC ? (int)left : PSG_VEC;
                    const RedCtx c{p, roff, rok, cache, stash, red, sb, col0, nvalid, j};
                    typename VT<DT>::T y[PSG_VEC];
                    StageBody<S>::eval(c, u, y);
                    if constexpr (S == kStash) {
#pragma unroll
                        for (int v = 0; v < PSG_VEC; ++v) stash[j][v] = as_bits(y[v]);
                    }
#pragma unroll
                    for (int v = 0; v < PSG_VEC; ++v)
                        if (kExact || v < nvalid) accv[v] = F::step(accv[v], y[v]);
                }
            }
#pragma unroll
            for (int w = PSG_VEC / 2; w > 0; w >>= 1) {
#pragma unroll
                for (int v = 0; v < w; ++v) accv[v] = F::step(accv[v], accv[v + w]);
            }
            typename VT<DT>::T acc;
            if constexpr (kColumnar) acc = col_fold<OP, DT>(accv[0], sm, cpart);
            else acc = team_fold<OP, DT>(accv[0], p.team_log2, sm);
            red[S] = as_bits(F::finish(acc));
        };
        sfor<0, kNstages>(stage);
        if (active) {
            if constexpr (kPerRow) {
                if (lane == 0) {
                    const RedCtx c{p, roff, rok, cache, stash, red, sb, 0, 1, 0};
                    typename VT<kOutDt>::T y[PSG_VEC];
                    Epi::eval(c, Epi::uni(c), y);
                    st_cell<kOutDt>((void*)p.out.ptr, ooff, y[0]);
                }
            } else {
                const int nch = kCH > 0 ? kCH : (int)((p.chunks - lane + T - 1) / T);
                const RedCtx cu{p, roff, rok, cache, stash, red, sb, 0, PSG_VEC, 0};
                const typename Epi::U u = Epi::uni(cu);  // the row's uniform values, once
#pragma unroll
                for (int j = 0; j < (kCH > 0 ? kCH : 1); ++j) {
                    for (int jj = (kCH > 0 ? j : 0); jj < (kCH > 0 ? j + 1 : nch); ++jj) {
                        const i64 ch = lane + (i64)jj * T;
                        const i64 col0 = ch * PSG_VEC;
                        const i64 left = p.inner - col0;
                        if (!kExact && left <= 0) continue;
                        const int nvalid = kExact ? PSG_VEC : left < PSG_VEC ? (int)left : PSG_VEC;
                        const RedCtx c{p, roff, rok, cache, stash, red, sb, col0, nvalid, j};
                        typename VT<kOutDt>::T y[PSG_VEC];
                        Epi::eval(c, u, y);
                        st_chunk<kOutDt, kOutMode>(p.out, ooff, col0, nvalid, y);
                    }
                }
            }
        }
        // staged mode: every thread is done with this slot before it is refilled
        if constexpr (kStaged) __syncthreads();
    }
    // staged mode: the last fill of every slot has landed before the block's
    // shared memory goes away (at once when every wait succeeded; after a
    // wait gave up, the copies still in flight are waited for, bounded)
    if constexpr (kStaged) {
        if (lane == 0) {
            for (int s = 0; s < kNS; ++s) {
                if (!(armed & (1u << s))) continue;
                const long long t0 = clock64();
                while (!mbar_try(&bars[team * kNS + s], (armed_ph >> s) & 1u) && clock64() - t0 < kWaitCycles) {
                }
            }
        }
    }
}
