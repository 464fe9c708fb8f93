// The bf16 / f16 MUL+SUM contraction kernels on the tensor cores (sm_103a):
// constants, the epilogue and the bodies of the single-CTA kernel and the
// CTA-pair kernel, templated on the epilogue.  Compiled two ways: by nvcc
// inside the library (contract_tc.cu, with EpiNone: C is the float32 total
// rounded once) and by NVRTC as text, ahead of a generated epilogue program
// (a residual add, a ReLU, a cast: elementwise work fused into the
// contraction that produces its operand, limn, "Reading the schedule").  No
// #include here; the includer provides the integer types, CUtensorMap,
// TcParams and the helpers of tc_device.cuh.
//
// An epilogue class Epi has `static constexpr bool active`, a type U (its
// per-row values) and, when active, row_uni(p, b, m) -> U and
// apply(p, u, b, m, n0, rr): rr holds the float32 totals of row m, columns
// n0 .. n0 + 63, as bits, and receives the program's values the same way.

struct EpiNone {
    static constexpr bool active = false;
    struct U {};
    struct Raw {};
};

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int B_BYTES = BN * BK * 2;             // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 48 KB
constexpr int TMEM_COLS = 512;                   // two 128 x 256 f32 accumulators
// warps 2 .. 9: warp w reads TMEM lanes 32 (w % 4) .. + 31 (the rows it may
// access), and the two warps of a lane quadrant take one half of the tile's
// columns each, so eight warps issue the epilogue's instructions (with four,
// one warp a scheduler, a fused program's per-cell work outlasted the next
// tile's products)
constexpr int EPI_WARPS = 8;
constexpr int EPI_COLS = BN / 2;                 // columns of a tile one epilogue warp takes
constexpr int THREADS = 64 + 32 * EPI_WARPS;
// the epilogue stages 32 rows x 128 bytes at a time, one slot a warp; the
// staging area follows the operand ring (so a tensor-core operand read past
// the last stage stays inside the allocation), the barriers follow it
constexpr int EPI_CHUNK = 4096;
constexpr int STAGING_BYTES = EPI_WARPS * EPI_CHUNK;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STAGING_BYTES + 256;

struct Bars {
    uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], drain;
    uint32_t tmem_base;
    int32_t abort;
};

__device__ __forceinline__ void mma_bf16(uint32_t dtmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t accum)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(dtmem), "l"(ad), "l"(bd), "r"(idesc), "r"(accum));
}
// two float32 values (bits) rounded to nearest even into a pair of bfloat16
// (bf) or float16 halves, lo in the low half
__device__ __forceinline__ uint32_t pack_half2(bool bf, uint32_t lo, uint32_t hi)
{
    uint32_t w;
    if (bf) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(__uint_as_float(hi)), "f"(__uint_as_float(lo)));
    else asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(__uint_as_float(hi)), "f"(__uint_as_float(lo)));
    return w;
}

// One TMEM load's 32 columns of row m (n0 = the first column) into C, or, under
// split-K, into this K range's float32 partials; rows and columns outside C
// are skipped.
__device__ __forceinline__ void epi_store32(const TcParams& p, const uint32_t (&r)[32], int m, int64_t crow, int n0,
                                            int sp, int b)
{
    if (m >= p.M) return;
    if (p.splits > 1) {
        // split-K: this K range's float32 total, summed later in split order
        float* dst = p.ws + (((int64_t)sp * p.batch + b) * p.M + m) * p.N + n0;
        if (n0 + 32 <= p.N && ((uintptr_t)dst & 15) == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                ((uint4*)dst)[j] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
        } else {
            for (int j = 0; j < 32; ++j)
                if (n0 + j < p.N) dst[j] = __uint_as_float(r[j]);
        }
    } else if (p.c_dtype == PSG_DT_BF16 || p.c_dtype == PSG_DT_F16) {
        const bool bf = p.c_dtype == PSG_DT_BF16;
        uint16_t* dst = (uint16_t*)p.C + crow + n0;
        if (p.c_cs == 1 && n0 + 32 <= p.N && ((uintptr_t)dst & 15) == 0) {
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = pack_half2(bf, r[2 * j], r[2 * j + 1]);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                ((uint4*)dst)[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        } else {
            uint16_t* C = (uint16_t*)p.C;
            for (int j = 0; j < 32; ++j)
                if (n0 + j < p.N) C[crow + (int64_t)(n0 + j) * p.c_cs] = (uint16_t)(pack_half2(bf, r[j], r[j]) & 0xffffu);
        }
    } else {
        float* dst = (float*)p.C + crow + n0;
        if (p.c_cs == 1 && n0 + 32 <= p.N && ((uintptr_t)dst & 15) == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                ((uint4*)dst)[j] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
        } else {
            float* C = (float*)p.C;
            for (int j = 0; j < 32; ++j)
                if (n0 + j < p.N) C[crow + (int64_t)(n0 + j) * p.c_cs] = __uint_as_float(r[j]);
        }
    }
}

// One accumulator's rows row0 .. row0 + 31 (this warp's 32 TMEM lanes, tm
// their first column) over columns c_lo .. c_lo + EPI_COLS - 1 of the tile,
// whose first column is n_base: 64 columns per pair of TMEM loads, rounded
// once into the output dtype (float32 partials under split-K).  With
// p.tma_store every 32 x 128-byte piece is written into the warp's
// 128B-swizzled staging slot and leaves in one TMA store (the tensor clips
// rows and columns past its edge); otherwise each lane stores its own row.
template <class Epi>
__device__ __forceinline__ void epilogue_rows(const TcParams& p, const CUtensorMap* tmap_c, uint8_t* slot,
                                              uint32_t& nst, uint32_t tm, int row0, int n_base, int c_lo, int sp,
                                              int b, int lane)
{
    const int m = row0 + lane;
    const int64_t crow = p.c_offset + (int64_t)b * p.c_bs + (int64_t)m * p.c_rs;
    const bool f32out = p.splits > 1 || p.c_dtype == PSG_DT_F32;
    const int z = p.splits > 1 ? sp * p.batch + b : b;
    // a fused epilogue program: its values that are uniform along the row,
    // once per row
    typename Epi::U eu;
    // the program's inputs for a 64-column slice are fetched one slice ahead
    // into registers, so their loads are in flight while the slice before is
    // computed and stored (not one load latency per 8 columns)
    // (the slice loop stays rolled: unrolled, its code no longer fits the
    // instruction cache and every contraction's epilogue slows down)
    typename Epi::Raw raw, next;
    if constexpr (Epi::active) {
        if (m < p.M) {
            eu = Epi::row_uni(p, b, m);
            Epi::fetch(p, b, m, n_base + c_lo, raw);
        }
    }
#pragma unroll 1
    for (int c2 = c_lo; c2 < c_lo + EPI_COLS; c2 += 64) {
        if constexpr (Epi::active) {
            if (c2 + 64 < c_lo + EPI_COLS && m < p.M) Epi::fetch(p, b, m, n_base + c2 + 64, next);
        }
        uint32_t rr[2][32];
        __syncwarp();  // tcgen05.ld is warp-collective: reach it converged
        tmem_ld32_nowait(tm + (uint32_t)c2, rr[0]);
        tmem_ld32_nowait(tm + (uint32_t)c2 + 32u, rr[1]);
        tmem_ld_wait();
        // the fused epilogue replaces each float32 total by the program's
        // value (rounded as its nodes round) before the store rounds it into C
        if constexpr (Epi::active) {
            if (m < p.M) Epi::apply(p, eu, b, m, n_base + c2, rr, raw);
            raw = next;
        }
        if (!p.tma_store) {
#pragma unroll
            for (int h = 0; h < 2; ++h) epi_store32(p, rr[h], m, crow, n_base + c2 + 32 * h, sp, b);
            continue;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (h == 1 && !f32out) break;  // 64 half-width columns fill one 128-byte row
            uint32_t w[32];
            if (f32out) {
#pragma unroll
                for (int j = 0; j < 32; ++j) w[j] = rr[h][j];
            } else if (p.c_dtype == PSG_DT_BF16) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[j])
                        : "f"(__uint_as_float(rr[j >> 4][(2 * j + 1) & 31])), "f"(__uint_as_float(rr[j >> 4][(2 * j) & 31])));
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w[j])
                        : "f"(__uint_as_float(rr[j >> 4][(2 * j + 1) & 31])), "f"(__uint_as_float(rr[j >> 4][(2 * j) & 31])));
            }
            if (nst >= 1) {  // the store that last read the slot is done reading it
                if (lane == 0) bulk_wait_read0();
                __syncwarp();
            }
            const uint32_t row = smem_u32(slot) + (uint32_t)lane * 128u;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                             ::"r"(row + (uint32_t)((u ^ (lane & 7)) << 4)), "r"(w[4 * u]), "r"(w[4 * u + 1]),
                               "r"(w[4 * u + 2]), "r"(w[4 * u + 3])
                             : "memory");
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                // a box wholly past the tensor's edge is not issued; the group is
                // committed either way, so the slot accounting above holds
                const int x = n_base + c2 + 32 * h;
                if (row0 < p.M && x < p.N) tma_store_3d(tmap_c, slot, x, row0, z);
                bulk_commit();
            }
            ++nst;
        }
    }
}

// The single-CTA kernel's body; Epi is EpiNone or a fused epilogue program.
template <class Epi>
__device__ __forceinline__ void tc_gemm_body(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                                             const CUtensorMap& tmap_c, const TcParams& p)
{
    extern __shared__ uint8_t smem_raw[];
    // swizzled tiles need 1024-byte alignment of their shared-memory address
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* staging = smem + STAGES * STAGE_BYTES;
    Bars* bars = (Bars*)(staging + STAGING_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total = p.num_m * p.num_n * p.batch;
    const int units = total * p.splits;  // (tile, K range) work units

    // set-up that touches no global memory runs before the wait on the
    // previous kernel: barriers, TMEM, the tensor maps' descriptor fetch
    if (threadIdx.x == 0) {
        prefetch_map(&tmap_a);
        prefetch_map(&tmap_b);
        if (p.tma_store) prefetch_map(&tmap_c);
        for (int s = 0; s < STAGES; ++s) {
            bar_init(&bars->full[s], 1);
            bar_init(&bars->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            bar_init(&bars->tfull[a], 1);
            bar_init(&bars->tempty[a], EPI_WARPS);
        }
        bar_init(&bars->drain, 1);
        bars->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&bars->tmem_base)), "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_enter();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_ph = 0;  // per-stage flags / parity of the last arm
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const int t = u / p.splits, sp = u - t * p.splits;
                const int kb0 = sp * p.kb_per, kb1 = min(p.num_k, kb0 + p.kb_per);
                int b, mb, nb;
                tile_coords(p.num_m, p.num_n, t, b, mb, nb);
                const int m0 = mb * BM, n0 = nb * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!bar_wait(&bars->empty[stage], ph ^ 1u, &bars->abort, p.status)) { ok = false; break; }
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    uint8_t* sb = sa + A_BYTES;
                    bar_expect_tx(&bars->full[stage], STAGE_BYTES);
                    const int k0 = kb * BK;
                    if (p.a_kmajor) {
                        tma_load_3d(sa, &tmap_a, &bars->full[stage], k0, m0, b);
                    } else {
                        tma_load_3d(sa, &tmap_a, &bars->full[stage], m0, k0, b);
                        tma_load_3d(sa + 8192, &tmap_a, &bars->full[stage], m0 + 64, k0, b);
                    }
                    if (p.b_kmajor) {
                        tma_load_3d(sb, &tmap_b, &bars->full[stage], k0, n0, b);
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            tma_load_3d(sb + i * 8192, &tmap_b, &bars->full[stage], n0 + 64 * i, k0, b);
                    }
                    armed |= 1u << stage;
                    armed_ph = (armed_ph & ~(1u << stage)) | (ph << stage);
                    if (++stage == STAGES) { stage = 0; ph ^= 1u; }
                }
            }
            // every copy this CTA issued lands before the CTA may exit
            for (int s = 0; s < STAGES; ++s)
                if (armed & (1u << s)) {
                    const long long t0 = clock64();
                    while (!bar_try(&bars->full[s], (armed_ph >> s) & 1u) && clock64() - t0 < WAIT_CYCLES) {
                    }
                }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            // instruction descriptor: f32 accumulate, A and B both bf16 (1) or both f16 (0),
            // M = 128, N = 256
            const uint32_t ab = p.ab_dtype == PSG_DT_F16 ? 0u : 1u;
            const uint32_t idesc = (1u << 4) | (ab << 7) | (ab << 10) | ((p.a_kmajor ? 0u : 1u) << 15) |
                                   ((p.b_kmajor ? 0u : 1u) << 16) | ((uint32_t)(BN >> 3) << 17) |
                                   ((uint32_t)(BM >> 4) << 24);
            // K-major: 8-row groups 1024 B apart, a K step of 16 is 32 B; MN-major:
            // 64-wide MN atoms 8 KB apart, 8-row K groups 1024 B apart, a K step of
            // 16 rows is 2 KB
            const uint32_t a_lbo = p.a_kmajor ? 16u : 8192u, b_lbo = p.b_kmajor ? 16u : 8192u;
            const uint32_t a_step = p.a_kmajor ? 2u : 128u, b_step = p.b_kmajor ? 2u : 128u;
            int stage = 0;
            uint32_t ph = 0;
            uint32_t aph[2] = {0u, 0u};
            bool ok = true;
            int local = 0;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++local) {
                const int kb0 = (u % p.splits) * p.kb_per, kb1 = min(p.num_k, kb0 + p.kb_per);
                const int acc = local & 1;
                if (!bar_wait(&bars->tempty[acc], aph[acc] ^ 1u, &bars->abort, p.status)) break;
                tc_fence_after();
                const uint32_t dtm = tmem + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!bar_wait(&bars->full[stage], ph, &bars->abort, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    const uint64_t ad = sdesc(sa, a_lbo, 1024u), bd = sdesc(sb, b_lbo, 1024u);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_bf16(dtm, ad + (uint64_t)(k * a_step), bd + (uint64_t)(k * b_step), idesc,
                                 (kb != kb0 || k != 0) ? 1u : 0u);
                    mma_commit(&bars->empty[stage]);  // frees the stage when these MMAs finish
                    if (++stage == STAGES) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
                mma_commit(&bars->tfull[acc]);  // accumulator ready for the epilogue
                aph[acc] ^= 1u;
            }
            // every MMA issued by this CTA completes before TMEM is freed
            mma_commit(&bars->drain);
            const long long t0 = clock64();
            while (!bar_try(&bars->drain, 0u) && clock64() - t0 < WAIT_CYCLES) {
            }
        }
    } else {
        // ---------------- epilogue: TMEM -> registers -> global ----------------
        const int q = warp & 3;  // TMEM lanes 32q .. 32q+31 belong to this warp
        const int c_lo = ((warp - 2) >> 2) * EPI_COLS;  // and these columns of each tile
        uint8_t* slot = staging + (warp - 2) * EPI_CHUNK;
        uint32_t nst = 0;
        uint32_t aph[2] = {0u, 0u};
        int local = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++local) {
            const int t = u / p.splits, sp = u - t * p.splits;
            const int acc = local & 1;
            int b, mb, nb;
            tile_coords(p.num_m, p.num_n, t, b, mb, nb);
            // the epilogue program's inputs for this tile head for L2 while the products run
            if constexpr (Epi::active) Epi::prefetch_l2(p, b, mb * BM + q * 32 + lane, nb * BN + c_lo, EPI_COLS);
            if (!bar_wait(&bars->tfull[acc], aph[acc], &bars->abort, p.status)) break;
            aph[acc] ^= 1u;
            tc_fence_after();
            epilogue_rows<Epi>(p, &tmap_c, slot, nst, tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN),
                               mb * BM + q * 32, nb * BN, c_lo, sp, b, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive(&bars->tempty[acc]);
        }
        if (lane == 0) bulk_wait_all();  // staged stores done before the CTA's shared memory goes away
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
}

// ---- CTA-pair variant: one 256 x 256 tile over two SMs ---------------------
//
// A cluster of two CTAs computes a 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256): each CTA holds 128 rows of the
// A slice and 128 columns of the B slice in its own shared memory, and its
// own 128 rows of the float32 accumulator in its TMEM.  Per 64-deep K slice a
// CTA loads 32 KB where the single-CTA tile loads 48 KB for the same 128 x 256
// outputs, so operand traffic from L2 per product drops by a third and the
// ring holds six stages.  The leader (rank 0) issues every MMA; both CTAs'
// copies count on the leader's full barrier (cta_group::2 bulk tensor
// copies), the MMA commits arrive on both CTAs' barriers (multicast), and
// both CTAs' epilogue warps free an accumulator on the leader's barrier.
constexpr int P_BM = 256;                              // rows of a pair tile (128 a CTA)
constexpr int P_HN = BN / 2;                           // columns of B a CTA holds
constexpr int P_STAGES = 6;
constexpr int P_A_BYTES = 128 * BK * 2;                // 16 KB
constexpr int P_B_BYTES = P_HN * BK * 2;               // 16 KB
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;   // 32 KB
constexpr int P_SMEM_BYTES = 1024 + P_STAGES * P_STAGE_BYTES + STAGING_BYTES + 256;

struct PairBars {
    uint64_t full[P_STAGES], empty[P_STAGES], tfull[2], tempty[2], drain;
    uint32_t tmem_base;
    int32_t abort;
};

__device__ __forceinline__ void mma_bf16_pair(uint32_t dtmem, uint64_t ad, uint64_t bd, uint32_t idesc,
                                              uint32_t accum)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(dtmem), "l"(ad), "l"(bd), "r"(idesc), "r"(accum));
}

// The CTA-pair kernel's body (launched in clusters of two CTAs).
template <class Epi>
__device__ __forceinline__ void tc_gemm2_body(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                                              const CUtensorMap& tmap_c, const TcParams& p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* staging = smem + P_STAGES * P_STAGE_BYTES;
    PairBars* bars = (PairBars*)(staging + STAGING_BYTES);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int cid = (int)(blockIdx.x >> 1), ncl = (int)(gridDim.x >> 1);
    const int total = p.num_m * p.num_n * p.batch;  // num_m counts 256-row blocks here
    const int units = total * p.splits;

    if (threadIdx.x == 0) {
        prefetch_map(&tmap_a);
        prefetch_map(&tmap_b);
        if (p.tma_store) prefetch_map(&tmap_c);
        for (int s = 0; s < P_STAGES; ++s) {
            bar_init(&bars->full[s], 1);
            bar_init(&bars->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            bar_init(&bars->tfull[a], 1);
            bar_init(&bars->tempty[a], 2 * EPI_WARPS);
        }
        bar_init(&bars->drain, 1);
        bars->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&bars->tmem_base)), "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    // both CTAs' barriers exist and both TMEM allocations are done before any
    // copy signals the leader or any MMA writes the peer
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    pdl_enter();  // nothing above touched global memory
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        if (lane == 0) {
            const uint32_t full0 = smem_in_rank(&bars->full[0], 0);  // the leader's full barriers
            int stage = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_ph = 0;
            bool ok = true;
            for (int u = cid; u < units && ok; u += ncl) {
                const int t = u / p.splits, sp = u - t * p.splits;
                const int kb0 = sp * p.kb_per, kb1 = min(p.num_k, kb0 + p.kb_per);
                int b, mb, nb;
                tile_coords(p.num_m, p.num_n, t, b, mb, nb);
                const int m0 = mb * P_BM + (int)rank * 128, n0 = nb * BN + (int)rank * P_HN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!bar_wait(&bars->empty[stage], ph ^ 1u, &bars->abort, p.status)) { ok = false; break; }
                    uint8_t* sa = smem + stage * P_STAGE_BYTES;
                    uint8_t* sb = sa + P_A_BYTES;
                    const uint32_t fb = full0 + (uint32_t)(stage * 8);
                    if (leader) bar_expect_tx(&bars->full[stage], 2 * P_STAGE_BYTES);  // both CTAs' bytes
                    const int k0 = kb * BK;
                    if (p.a_kmajor) {
                        tma_load_3d_pair(sa, &tmap_a, fb, k0, m0, b);
                    } else {
                        tma_load_3d_pair(sa, &tmap_a, fb, m0, k0, b);
                        tma_load_3d_pair(sa + 8192, &tmap_a, fb, m0 + 64, k0, b);
                    }
                    if (p.b_kmajor) {
                        tma_load_3d_pair(sb, &tmap_b, fb, k0, n0, b);
                    } else {
                        tma_load_3d_pair(sb, &tmap_b, fb, n0, k0, b);
                        tma_load_3d_pair(sb + 8192, &tmap_b, fb, n0 + 64, k0, b);
                    }
                    armed |= 1u << stage;
                    armed_ph = (armed_ph & ~(1u << stage)) | (ph << stage);
                    if (++stage == P_STAGES) { stage = 0; ph ^= 1u; }
                }
            }
            // the leader's full barriers count both CTAs' copies: once each
            // armed stage completed, every copy of the pair has landed
            if (leader)
                for (int s = 0; s < P_STAGES; ++s)
                    if (armed & (1u << s)) bar_wait_drain(&bars->full[s], (armed_ph >> s) & 1u);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (leader only) ----------------
        if (leader && lane == 0) {
            // f32 accumulate, A and B both bf16 (1) or both f16 (0), M = 256, N = 256
            const uint32_t ab = p.ab_dtype == PSG_DT_F16 ? 0u : 1u;
            const uint32_t idesc = (1u << 4) | (ab << 7) | (ab << 10) | ((p.a_kmajor ? 0u : 1u) << 15) |
                                   ((p.b_kmajor ? 0u : 1u) << 16) | ((uint32_t)(BN >> 3) << 17) |
                                   ((uint32_t)(P_BM >> 4) << 24);
            const uint32_t a_lbo = p.a_kmajor ? 16u : 8192u, b_lbo = p.b_kmajor ? 16u : 8192u;
            const uint32_t a_step = p.a_kmajor ? 2u : 128u, b_step = p.b_kmajor ? 2u : 128u;
            int stage = 0;
            uint32_t ph = 0;
            uint32_t aph[2] = {0u, 0u};
            bool ok = true;
            int local = 0;
            for (int u = cid; u < units && ok; u += ncl, ++local) {
                const int kb0 = (u % p.splits) * p.kb_per, kb1 = min(p.num_k, kb0 + p.kb_per);
                const int acc = local & 1;
                if (!bar_wait(&bars->tempty[acc], aph[acc] ^ 1u, &bars->abort, p.status)) break;
                tc_fence_after();
                const uint32_t dtm = tmem + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!bar_wait(&bars->full[stage], ph, &bars->abort, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * P_STAGE_BYTES);
                    const uint32_t sb = sa + P_A_BYTES;
                    const uint64_t ad = sdesc(sa, a_lbo, 1024u), bd = sdesc(sb, b_lbo, 1024u);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_bf16_pair(dtm, ad + (uint64_t)(k * a_step), bd + (uint64_t)(k * b_step), idesc,
                                      (kb != kb0 || k != 0) ? 1u : 0u);
                    mma_commit_pair(&bars->empty[stage]);  // frees the stage in both CTAs
                    if (++stage == P_STAGES) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair(&bars->tfull[acc]);  // both halves of the accumulator are ready
                aph[acc] ^= 1u;
            }
            mma_commit_pair_local(&bars->drain);
            bar_wait_drain(&bars->drain, 0u);
        }
    } else {
        // ---------------- epilogue (both CTAs): this CTA's 128 rows ----------------
        const int q = warp & 3;
        const int c_lo = ((warp - 2) >> 2) * EPI_COLS;
        uint8_t* slot = staging + (warp - 2) * EPI_CHUNK;
        uint32_t nst = 0;
        const uint32_t tempty0 = smem_in_rank(&bars->tempty[0], 0);
        uint32_t aph[2] = {0u, 0u};
        int local = 0;
        for (int u = cid; u < units; u += ncl, ++local) {
            const int t = u / p.splits, sp = u - t * p.splits;
            const int acc = local & 1;
            int b, mb, nb;
            tile_coords(p.num_m, p.num_n, t, b, mb, nb);
            if constexpr (Epi::active)
                Epi::prefetch_l2(p, b, mb * P_BM + (int)rank * 128 + q * 32 + lane, nb * BN + c_lo, EPI_COLS);
            if (!bar_wait(&bars->tfull[acc], aph[acc], &bars->abort, p.status)) break;
            aph[acc] ^= 1u;
            tc_fence_after();
            epilogue_rows<Epi>(p, &tmap_c, slot, nst, tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN),
                               mb * P_BM + (int)rank * 128 + q * 32, nb * BN, c_lo, sp, b, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive_cluster(tempty0 + (uint32_t)(acc * 8));
        }
        if (lane == 0) bulk_wait_all();
    }
    // the leader's MMAs read this CTA's shared memory and write its TMEM: no
    // CTA frees either before both are done
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
}

