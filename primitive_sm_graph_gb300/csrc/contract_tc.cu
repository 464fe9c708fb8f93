// bf16 MUL+SUM contraction on the 5th-generation tensor cores (sm_103a).
//
// C[b, m, n] = sum_k A[b, m, k] * B[b, k, n]: limn lowers a matmul to a
// broadcast MUL and a SUM over k that fuse into one kernel ("Reading the
// schedule": a whole matmul is one kernel); the broadcast is the stride-0
// loop of the Luminal IR blog ("Naive Matrix Multiplication").  Here the
// MUL+SUM of one 128x256 output tile runs as a chain of
// tcgen05.mma.cta_group::1.kind::f16 (bf16 inputs, float32 accumulate in
// TMEM), fed by TMA.
//
// Warp roles (320 threads, one CTA per SM, persistent over tiles):
//   warp 0  TMA producer: one elected lane streams 64-deep K slices of A and
//           B into a 4-stage shared-memory ring (128B-swizzled tiles);
//   warp 1  MMA issuer: allocates all 512 TMEM columns (two 128x256 f32
//           accumulators), one lane issues 4 MMAs (K = 16 each) per stage and
//           commits the stage back to the producer;
//   warps 2-9 epilogue: two warps per 32 TMEM lanes (rows), each taking
//           128 of the tile's 256 columns; a warp reads 64 columns with two
//           tcgen05.ld before one wait, rounds to the output dtype once and
//           stores, while the MMA warp fills the other accumulator.
// Every wait on an mbarrier gives up after about a second: the CTA then sets
// PSG_E_TIMEOUT in the caller's status word, drains its own copies and MMAs,
// frees TMEM and returns.  No TMA multicast is used: each CTA loads its own
// tiles.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "contract.h"
#include "launch_util.cuh"
#include "tc_util.cuh"

namespace psg {

namespace {

using namespace tcu;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int B_BYTES = BN * BK * 2;             // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 48 KB
constexpr int TMEM_COLS = 512;                   // two 128 x 256 f32 accumulators
constexpr int EPI_WARPS = 4;                     // warps 2 .. 5
constexpr int THREADS = 64 + 32 * EPI_WARPS;
// the epilogue stages 32 rows x 128 bytes at a time, two slots a warp; the
// staging area follows the operand ring (so a tensor-core operand read past
// the last stage stays inside the allocation), the barriers follow it
constexpr int EPI_CHUNK = 4096;
constexpr int STAGING_BYTES = EPI_WARPS * 2 * EPI_CHUNK;
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
    } else if (p.c_dtype == PSG_BF16) {
        __nv_bfloat16* dst = (__nv_bfloat16*)p.C + crow + n0;
        if (p.c_cs == 1 && n0 + 32 <= p.N && ((uintptr_t)dst & 15) == 0) {
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const __nv_bfloat162 hv = __floats2bfloat162_rn(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                w[j] = *(const uint32_t*)&hv;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                ((uint4*)dst)[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        } else {
            __nv_bfloat16* C = (__nv_bfloat16*)p.C;
            for (int j = 0; j < 32; ++j)
                if (n0 + j < p.N) C[crow + (int64_t)(n0 + j) * p.c_cs] = __float2bfloat16_rn(__uint_as_float(r[j]));
        }
    } else if (p.c_dtype == PSG_F16) {
        __half* C = (__half*)p.C;
        for (int j = 0; j < 32; ++j)
            if (n0 + j < p.N) C[crow + (int64_t)(n0 + j) * p.c_cs] = __float2half_rn(__uint_as_float(r[j]));
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
// their first column) over the tile's BN columns, which start at column
// n_base: 64 columns per pair of TMEM loads, rounded once into the output
// dtype (float32 partials under split-K).  With p.tma_store every 32 x
// 128-byte piece is written into one of the warp's two 128B-swizzled staging
// slots and leaves in one TMA store (the tensor clips rows and columns past
// its edge); otherwise each lane stores its own row.
__device__ __forceinline__ void epilogue_rows(const TcParams& p, const CUtensorMap* tmap_c, uint8_t* slots,
                                              uint32_t& nst, uint32_t tm, int row0, int n_base, int sp, int b,
                                              int lane)
{
    const int m = row0 + lane;
    const int64_t crow = p.c_offset + (int64_t)b * p.c_bs + (int64_t)m * p.c_rs;
    const bool f32out = p.splits > 1 || p.c_dtype == PSG_F32;
    const int z = p.splits > 1 ? sp * p.batch + b : b;
    for (int c2 = 0; c2 < BN; c2 += 64) {
        uint32_t rr[2][32];
        __syncwarp();  // tcgen05.ld is warp-collective: reach it converged
        tmem_ld32_nowait(tm + (uint32_t)c2, rr[0]);
        tmem_ld32_nowait(tm + (uint32_t)c2 + 32u, rr[1]);
        tmem_ld_wait();
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
            } else if (p.c_dtype == PSG_BF16) {
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
            uint8_t* slot = slots + (nst & 1u) * EPI_CHUNK;
            if (nst >= 2) {  // the store that last read this slot is done reading it
                if (lane == 0) bulk_wait_read1();
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

__global__ void __launch_bounds__(THREADS, 1) tc_gemm(const __grid_constant__ CUtensorMap tmap_a,
                                                      const __grid_constant__ CUtensorMap tmap_b,
                                                      const __grid_constant__ CUtensorMap tmap_c,
                                                      const __grid_constant__ TcParams p)
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
            const uint32_t ab = p.ab_dtype == PSG_F16 ? 0u : 1u;
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
        uint8_t* slots = staging + (warp - 2) * 2 * EPI_CHUNK;
        uint32_t nst = 0;
        uint32_t aph[2] = {0u, 0u};
        int local = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++local) {
            const int t = u / p.splits, sp = u - t * p.splits;
            const int acc = local & 1;
            if (!bar_wait(&bars->tfull[acc], aph[acc], &bars->abort, p.status)) break;
            aph[acc] ^= 1u;
            tc_fence_after();
            int b, mb, nb;
            tile_coords(p.num_m, p.num_n, t, b, mb, nb);
            epilogue_rows(p, &tmap_c, slots, nst, tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN),
                          mb * BM + q * 32, nb * BN, sp, b, lane);
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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    tc_gemm2(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
             const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ TcParams p)
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
            const uint32_t ab = p.ab_dtype == PSG_F16 ? 0u : 1u;
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
        uint8_t* slots = staging + (warp - 2) * 2 * EPI_CHUNK;
        uint32_t nst = 0;
        const uint32_t tempty0 = smem_in_rank(&bars->tempty[0], 0);
        uint32_t aph[2] = {0u, 0u};
        int local = 0;
        for (int u = cid; u < units; u += ncl, ++local) {
            const int t = u / p.splits, sp = u - t * p.splits;
            const int acc = local & 1;
            if (!bar_wait(&bars->tfull[acc], aph[acc], &bars->abort, p.status)) break;
            aph[acc] ^= 1u;
            tc_fence_after();
            int b, mb, nb;
            tile_coords(p.num_m, p.num_n, t, b, mb, nb);
            epilogue_rows(p, &tmap_c, slots, nst, tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN),
                          mb * P_BM + (int)rank * 128 + q * 32, nb * BN, sp, b, lane);
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

// C = sum over the splits, in split order, of the float32 partials, rounded
// once into C's dtype.  With p.reduce_quad (every row of C contiguous and
// 4-cell aligned: N % 4 == 0, unit column stride, 16-byte aligned partials)
// a thread adds four adjacent cells with 16-byte loads and divides its index
// once per four cells.
__global__ void __launch_bounds__(256) splitk_reduce(const __grid_constant__ TcParams p)
{
    pdl_enter();
    const int64_t cells = (int64_t)p.batch * p.M * p.N;
    const int64_t stride = cells;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    if (p.reduce_quad) {
        const int64_t nq = p.N / 4, quads = cells / 4;
        for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < quads; q += step) {
            const int64_t bm = q / nq;
            const int64_t n = (q - bm * nq) * 4, e = q * 4;
            float4 acc = *(const float4*)(p.ws + e);
            for (int s = 1; s < p.splits; ++s) {
                const float4 v = *(const float4*)(p.ws + e + s * stride);
                acc.x = __fadd_rn(acc.x, v.x);
                acc.y = __fadd_rn(acc.y, v.y);
                acc.z = __fadd_rn(acc.z, v.z);
                acc.w = __fadd_rn(acc.w, v.w);
            }
            const int64_t m = bm % p.M, b = bm / p.M;
            const int64_t o = p.c_offset + b * p.c_bs + m * p.c_rs + n;
            if (p.c_dtype == PSG_F32) {
                *(float4*)((float*)p.C + o) = acc;
            } else if (p.c_dtype == PSG_F16) {
                const __half2 lo = __floats2half2_rn(acc.x, acc.y), hi = __floats2half2_rn(acc.z, acc.w);
                *(uint2*)((__half*)p.C + o) = make_uint2(*(const uint32_t*)&lo, *(const uint32_t*)&hi);
            } else {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
                *(uint2*)((__nv_bfloat16*)p.C + o) = make_uint2(*(const uint32_t*)&lo, *(const uint32_t*)&hi);
            }
        }
        return;
    }
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < cells; e += step) {
        float acc = p.ws[e];
        for (int s = 1; s < p.splits; ++s) acc = __fadd_rn(acc, p.ws[e + s * stride]);
        const int64_t n = e % p.N, bm = e / p.N, m = bm % p.M, b = bm / p.M;
        const int64_t o = p.c_offset + b * p.c_bs + m * p.c_rs + n * p.c_cs;
        if (p.c_dtype == PSG_F32) ((float*)p.C)[o] = acc;
        else if (p.c_dtype == PSG_F16) ((__half*)p.C)[o] = __float2half_rn(acc);
        else ((__nv_bfloat16*)p.C)[o] = __float2bfloat16_rn(acc);
    }
}

// launch of splitk_reduce: the quad path when C's rows allow it
void launch_splitk_reduce(TcParams p, void* stream)
{
    const int es = dtype_size(p.c_dtype);
    const bool quad = p.N % 4 == 0 && p.c_cs == 1 && ((uintptr_t)p.ws & 15) == 0 &&
                      (((uintptr_t)p.C + (uint64_t)p.c_offset * es) % (4 * es)) == 0 && (p.c_rs * es) % (4 * es) == 0 &&
                      (p.batch == 1 || (p.c_bs * es) % (4 * es) == 0);
    p.reduce_quad = quad ? 1 : 0;
    const int64_t cells = (int64_t)p.batch * p.M * p.N;
    const int64_t work = quad ? cells / 4 : cells;
    const int rgrid = (int)std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, (int64_t)num_sms() * 8));
    launch(splitk_reduce, rgrid, 256, 0, (cudaStream_t)stream, p);
}

// 3-D tensor map over a bf16 or f16 operand: dims {inner, outer, batch}.
bool make_map(CUtensorMap* map, const void* base, int64_t inner, int64_t outer, int64_t batch, int64_t outer_stride,
              int64_t batch_stride, uint32_t box_inner, uint32_t box_outer, bool f16)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)batch};
    cuuint64_t strides[2] = {(cuuint64_t)(outer_stride * 2), (cuuint64_t)(batch_stride * 2)};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of the epilogue's destination, 32 rows x 128 bytes a box,
// 128B-swizzled: C itself, or under split-K the float32 partials
// [splits][batch][M][N].  Sets p.tma_store; false (direct stores) when C's
// layout cannot be described (a strided column, a row pitch or base that is
// not a multiple of 16 bytes).
void make_out_map(CUtensorMap* map, TcParams& p)
{
    p.tma_store = 0;
    std::memset(map, 0, sizeof(*map));
    auto enc = encode_fn();
    if (!enc) return;
    const bool partials = p.splits > 1;
    const int es = partials ? 4 : dtype_size(p.c_dtype);
    const CUtensorMapDataType dt = partials || p.c_dtype == PSG_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : p.c_dtype == PSG_F16          ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const void* base;
    int64_t rs, bs, nz;
    if (partials) {
        base = p.ws;
        rs = p.N;
        bs = (int64_t)p.M * p.N;
        nz = (int64_t)p.splits * p.batch;
    } else {
        if (p.c_cs != 1) return;
        base = (const char*)p.C + p.c_offset * es;
        rs = p.M > 1 ? p.c_rs : p.N;
        bs = p.batch > 1 ? p.c_bs : rs * p.M;
        nz = p.batch;
    }
    if (((uintptr_t)base & 15) != 0 || rs < p.N || (rs * es) % 16 != 0 || bs <= 0 || (bs * es) % 16 != 0) return;
    cuuint64_t dims[3] = {(cuuint64_t)p.N, (cuuint64_t)p.M, (cuuint64_t)nz};
    cuuint64_t strides[2] = {(cuuint64_t)(rs * es), (cuuint64_t)(bs * es)};
    cuuint32_t box[3] = {(cuuint32_t)(128 / es), 32, 1};
    cuuint32_t ones[3] = {1, 1, 1};
    if (enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
        p.tma_store = 1;
}

}  // namespace

int contract_tc_splits(int64_t M, int64_t N, int64_t K, int64_t batch, size_t* bytes)
{
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN) * batch;
    const int64_t num_k = (K + BK - 1) / BK;
    const int64_t sms = num_sms();
    *bytes = 0;
    // only when the output's tiles leave most SMs idle and K is long enough
    // (K >= 1024) that each split keeps at least 8 K blocks: the float32
    // partials then cost little next to the products
    if (tiles * 2 > sms || num_k < 16) return 1;
    int64_t s = std::min<int64_t>(std::min<int64_t>(sms / tiles, num_k / 8), 16);
    if (s < 2) return 1;
    const int64_t per = (num_k + s - 1) / s;
    s = (num_k + per - 1) / per;  // no empty range
    *bytes = (size_t)(s * batch * M * N * 4);
    return (int)s;
}

namespace {

// The CTA-pair kernel takes outputs of more than one 128-row block over
// K >= 1024, or over K >= 512 when the single-CTA tiles make two waves or more
// (measured on GB300: 8192 x 8192 x 2048 in 164 us against 194 us single-CTA;
// 8192 x 2048 x 512 in 18.7 us against 20.1 us; 8192 x 512 x 512, one wave,
// 8.2 us against 7.8 us).  PSG_GEMM_KERNEL=single or =pair in the environment forces one of
// them (pair still needs M > 128).
bool use_pair(const TcParams& p)
{
    if (p.M <= BM) return false;
    const char* f = std::getenv("PSG_GEMM_KERNEL");
    if (f && f[0] == 's') return false;
    if (f && f[0] == 'p') return true;
    const int64_t tiles = (int64_t)((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN) * p.batch;
    return p.K >= 1024 || (p.K >= 512 && tiles >= 2 * (int64_t)num_sms());
}

// clusters of two tc_gemm2 CTAs that fit on the device at once (per device)
int pair_clusters()
{
    constexpr int MAX_DEV = 64;
    static std::mutex mu;
    static int cached[MAX_DEV];
    const int d = current_device();
    std::lock_guard<std::mutex> g(mu);
    if (cached[d] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * num_sms());
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = P_SMEM_BYTES;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, (const void*)tc_gemm2, &cfg) != cudaSuccess || n < 1) n = num_sms() / 2;
        cached[d] = n;
    }
    return cached[d];
}

psg_status launch_pair(const TcOperands& o, TcParams p, int64_t a_bs, int64_t b_bs, void* stream)
{
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute((const void*)tc_gemm2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        P_SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return PSG_E_CUDA;
    CUtensorMap ma, mb;
    const bool f16 = p.ab_dtype == PSG_F16;
    // a CTA holds 128 rows of A and 128 columns of B per 64-deep K slice
    bool ok = p.a_kmajor ? make_map(&ma, o.A, p.K, p.M, p.batch, o.a_ms, a_bs, 64, 128, f16)
                         : make_map(&ma, o.A, p.M, p.K, p.batch, o.a_ks, a_bs, 64, 64, f16);
    ok = ok && (p.b_kmajor ? make_map(&mb, o.B, p.K, p.N, p.batch, o.b_ns, b_bs, 64, P_HN, f16)
                           : make_map(&mb, o.B, p.N, p.K, p.batch, o.b_ks, b_bs, 64, 64, f16));
    if (!ok) return PSG_E_CUDA;
    p.num_m = (p.M + P_BM - 1) / P_BM;
    p.num_n = (p.N + BN - 1) / BN;
    p.num_k = (p.K + BK - 1) / BK;
    p.kb_per = (p.num_k + p.splits - 1) / p.splits;
    CUtensorMap mc;
    make_out_map(&mc, p);
    const int64_t units = (int64_t)p.num_m * p.num_n * p.batch * p.splits;
    const int clusters = (int)std::min<int64_t>(units, pair_clusters());
    launch(tc_gemm2, 2 * clusters, THREADS, P_SMEM_BYTES, (cudaStream_t)stream, ma, mb, mc, p);
    if (p.splits > 1) launch_splitk_reduce(p, stream);
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

}  // namespace

psg_status launch_contract_tc(const TcOperands& o, void* stream)
{
    TcParams p = o.p;
    p.splits = 1;
    p.ws = nullptr;
    if (o.ws) {
        size_t need = 0;
        const int s = contract_tc_splits(p.M, p.N, p.K, p.batch, &need);
        if (s > 1 && need <= o.ws_bytes && ((uintptr_t)o.ws & 15) == 0) {
            p.splits = s;
            p.ws = (float*)o.ws;
        }
    }
    if (p.M == 0 || p.N == 0 || p.batch == 0) return PSG_OK;
    CUtensorMap ma, mb;
    // batch strides of a single batch are never used; keep them a legal multiple of 16 bytes
    const int64_t a_bs = p.batch > 1 ? o.a_bs : (p.a_kmajor ? o.a_ms * p.M : o.a_ks * p.K);
    const int64_t b_bs = p.batch > 1 ? o.b_bs : (p.b_kmajor ? o.b_ns * p.N : o.b_ks * p.K);
    if (use_pair(p)) return launch_pair(o, p, a_bs, b_bs, stream);
    const bool f16 = p.ab_dtype == PSG_F16;
    bool ok = p.a_kmajor ? make_map(&ma, o.A, p.K, p.M, p.batch, o.a_ms, a_bs, 64, 128, f16)
                         : make_map(&ma, o.A, p.M, p.K, p.batch, o.a_ks, a_bs, 64, 64, f16);
    ok = ok && (p.b_kmajor ? make_map(&mb, o.B, p.K, p.N, p.batch, o.b_ns, b_bs, 64, 256, f16)
                           : make_map(&mb, o.B, p.N, p.K, p.batch, o.b_ks, b_bs, 64, 64, f16));
    if (!ok) return PSG_E_CUDA;
    p.num_m = (p.M + BM - 1) / BM;
    p.num_n = (p.N + BN - 1) / BN;
    p.num_k = (p.K + BK - 1) / BK;
    p.kb_per = (p.num_k + p.splits - 1) / p.splits;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute((const void*)tc_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return PSG_E_CUDA;
    CUtensorMap mc;
    make_out_map(&mc, p);
    const int64_t units = (int64_t)p.num_m * p.num_n * p.batch * p.splits;
    const int grid = (int)std::min<int64_t>(units, num_sms());
    launch(tc_gemm, grid, THREADS, SMEM_BYTES, (cudaStream_t)stream, ma, mb, mc, p);
    if (p.splits > 1) launch_splitk_reduce(p, stream);
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

void query_contract_tc(int64_t M, int64_t tiles, int* grid, int* block, int* smem, int* regs)
{
    TcParams p = {};
    p.M = (int)std::min<int64_t>(M, 1 << 30);
    p.K = 1 << 30;  // the query has no K: report the kernel a long K takes
    if (use_pair(p)) {
        *grid = 2 * (int)std::min<int64_t>((tiles + 1) / 2, pair_clusters());
        *block = THREADS;
        *smem = P_SMEM_BYTES;
        *regs = kernel_regs((const void*)tc_gemm2);
        return;
    }
    *grid = (int)std::min<int64_t>(tiles, num_sms());
    *block = THREADS;
    *smem = SMEM_BYTES;
    *regs = kernel_regs((const void*)tc_gemm);
}

}  // namespace psg
