// float32 MUL+SUM contraction on the 5th-generation tensor cores (sm_103a),
// as three TF32 products per term (the 3xTF32 split of Ootomo & Yokota,
// "Recovering single precision accuracy from Tensor Cores while surpassing
// the FP32 theoretical peak performance", 2022).
//
// C[b, m, n] = sum_k A[b, m, k] * B[b, k, n] (limn, "Reading the schedule":
// a whole matmul is one kernel; Luminal IR blog, "Naive Matrix
// Multiplication": the broadcast MUL and the SUM over k).  Every float32
// operand x is split into hi = x with its low 13 mantissa bits cleared (a
// TF32 value) and lo = x - hi (exact in float32, then read as TF32), and
//     a * b ~= hi_a * hi_b + hi_a * lo_b + lo_a * hi_b
// accumulates in float32 in TMEM; the dropped lo_a * lo_b and the TF32
// reading of lo leave a relative error of a few 2^-20 per product, inside
// the reduction-order bound 2 * gamma_{K-1} * sum |a b| for the K this path
// is used at (the planner sends short K to the FP32-pipe kernel).
//
// Warp roles (448 threads, one CTA per SM, persistent over 128x128 tiles):
//   warp 0      TMA producer: 32-deep K slices of A and B, as stored (K- or
//               MN-major, no swizzle), into a 2-stage raw ring;
//   warp 1      MMA issuer: allocates 256 TMEM columns (two 128x128 f32
//               accumulators) and issues 3 tcgen05.mma.kind::tf32 per K = 8;
//   warps 2-5   epilogue: tcgen05.ld, one rounding into C's dtype, stores;
//   warps 6-13  converters: raw tile -> hi / lo tiles, K-major with the
//               128-byte swizzle, in a 2-stage ring the MMAs read.
// Every mbarrier wait is bounded (about a second): the CTA then sets
// PSG_E_TIMEOUT in the status word, drains its copies and MMAs, frees TMEM
// and returns.  No TMA multicast.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "contract.h"
#include "launch_util.cuh"
#include "tc_util.cuh"

namespace psg {

namespace {

using namespace tcu;

constexpr int BM = 128, BN = 128, BKF = 32;      // tile, K slice (float32 elements = 128 bytes)
constexpr int RS = 2, CS = 2;                    // raw and converted ring depths
constexpr int TILE_BYTES = 128 * BKF * 4;        // 16 KB: one 128 x 32 float32 tile
constexpr int RAW_STAGE = 2 * TILE_BYTES;        // raw A, raw B
constexpr int CONV_STAGE = 4 * TILE_BYTES;       // hi A, lo A, hi B, lo B
constexpr int TMEM_COLS = 2 * BN;                // two 128 x 128 f32 accumulators
constexpr int CONV_WARPS = 8;
constexpr int THREADS = (6 + CONV_WARPS) * 32;
constexpr int SMEM_BYTES = 1024 + CS * CONV_STAGE + RS * RAW_STAGE + 512 + 1024;

struct Bars {
    uint64_t raw_full[RS], raw_empty[RS], conv_full[CS], conv_empty[CS], tfull[2], tempty[2], drain;
    uint32_t tmem_base;
    int32_t abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

__device__ __forceinline__ void mma_tf32(uint32_t dtmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t accum)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(dtmem), "l"(ad), "l"(bd), "r"(idesc), "r"(accum));
}

// x -> (hi, lo): hi keeps the TF32 bits of x, lo = x - hi exactly; a
// non-finite x is its own hi with lo = 0 (so inf and NaN pass through)
__device__ __forceinline__ void split1(float x, float& hi, float& lo)
{
    const uint32_t u = __float_as_uint(x);
    const bool fin = (u & 0x7f800000u) != 0x7f800000u;
    hi = __uint_as_float(fin ? (u & 0xffffe000u) : u);
    lo = fin ? __fsub_rn(x, hi) : 0.0f;
}

// One 128 x 32 float32 tile from its raw TMA layout into the hi and lo
// tiles (K-major: row r = m or n, 32 k values in 128 bytes, 8-row groups of
// 1024 bytes, 16-byte chunk c of row r stored at chunk c ^ (r % 8)).
// kmajor raw: [r][32 k]; MN-major raw: [32 k][128 r].  `ct` is the thread's
// index among the converter threads; each thread handles 4 chunks.
__device__ __forceinline__ void convert_tile(const float* __restrict__ raw, uint8_t* hi_t, uint8_t* lo_t, bool kmajor,
                                             int ct)
{
    constexpr int NT = CONV_WARPS * 32;
    constexpr int NJ = (128 * 8) / NT;
    // explicit shared-memory loads and stores (the tiles are shared memory;
    // a generic access would take the slower generic path), every load of
    // the thread issued before the first split
    const uint32_t rs = smem_u32(raw), hs = smem_u32(hi_t), ls = smem_u32(lo_t);
    float x[NJ][4];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int i = ct + NT * j;
        if (kmajor) {
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(x[j][0]), "=f"(x[j][1]), "=f"(x[j][2]), "=f"(x[j][3])
                         : "r"(rs + (uint32_t)(((i >> 3) * BKF + (i & 7) * 4) * 4)));
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                asm volatile("ld.shared.f32 %0, [%1];"
                             : "=f"(x[j][q])
                             : "r"(rs + (uint32_t)((((i >> 7) * 4 + q) * 128 + (i & 127)) * 4)));
        }
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int i = ct + NT * j;
        const int r = kmajor ? i >> 3 : i & 127, c = kmajor ? i & 7 : i >> 7;
        float h[4], l[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) split1(x[j][q], h[q], l[q]);
        const uint32_t off = (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(hs + off), "f"(h[0]), "f"(h[1]), "f"(h[2]), "f"(h[3])
                     : "memory");
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(ls + off), "f"(l[0]), "f"(l[1]), "f"(l[2]), "f"(l[3])
                     : "memory");
    }
}

__global__ void __launch_bounds__(THREADS, 1) tc_gemm_tf32x3(const __grid_constant__ CUtensorMap tmap_a,
                                                             const __grid_constant__ CUtensorMap tmap_b,
                                                             const __grid_constant__ TcParams p)
{
    pdl_enter();
    extern __shared__ uint8_t smem_raw[];
    // swizzled tiles need 1024-byte alignment of their shared-memory address
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* conv = smem;                          // CS x [hiA | loA | hiB | loB]
    uint8_t* raw = smem + CS * CONV_STAGE;         // RS x [A | B]
    Bars* bars = (Bars*)(raw + RS * RAW_STAGE);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total = p.num_m * p.num_n * p.batch;

    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            bar_init(&bars->raw_full[s], 1);
            bar_init(&bars->raw_empty[s], CONV_WARPS);
        }
        for (int s = 0; s < CS; ++s) {
            bar_init(&bars->conv_full[s], CONV_WARPS);
            bar_init(&bars->conv_empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            bar_init(&bars->tfull[a], 1);
            bar_init(&bars->tempty[a], 4);
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
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer: raw tiles as stored ----------------
        if (lane == 0) {
            int rs = 0;
            uint32_t ph = 0, armed = 0, armed_ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                int b, mb, nb;
                tile_coords(p.num_m, p.num_n, t, b, mb, nb);
                const int m0 = mb * BM, n0 = nb * BN;
                for (int kb = 0; kb < p.num_k; ++kb) {
                    if (!bar_wait(&bars->raw_empty[rs], ph ^ 1u, &bars->abort, p.status)) { ok = false; break; }
                    uint8_t* ra = raw + rs * RAW_STAGE;
                    bar_expect_tx(&bars->raw_full[rs], RAW_STAGE);
                    const int k0 = kb * BKF;
                    if (p.a_kmajor) tma_load_3d(ra, &tmap_a, &bars->raw_full[rs], k0, m0, b);
                    else tma_load_3d(ra, &tmap_a, &bars->raw_full[rs], m0, k0, b);
                    if (p.b_kmajor) tma_load_3d(ra + TILE_BYTES, &tmap_b, &bars->raw_full[rs], k0, n0, b);
                    else tma_load_3d(ra + TILE_BYTES, &tmap_b, &bars->raw_full[rs], n0, k0, b);
                    armed |= 1u << rs;
                    armed_ph = (armed_ph & ~(1u << rs)) | (ph << rs);
                    if (++rs == RS) { rs = 0; ph ^= 1u; }
                }
            }
            // every copy this CTA issued lands before the CTA may exit
            for (int s = 0; s < RS; ++s)
                if (armed & (1u << s)) bar_wait_drain(&bars->raw_full[s], (armed_ph >> s) & 1u);
        }
    } else if (warp >= 6) {
        // ---------------- converters: raw -> hi / lo (K-major, swizzled) ----------------
        const int ct = threadIdx.x - 6 * 32;
        int rs = 0, cs = 0;
        uint32_t rph = 0, cph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            for (int kb = 0; kb < p.num_k; ++kb) {
                if (!bar_wait(&bars->raw_full[rs], rph, &bars->abort, p.status)) { ok = false; break; }
                if (!bar_wait(&bars->conv_empty[cs], cph ^ 1u, &bars->abort, p.status)) { ok = false; break; }
                const float* ra = (const float*)(raw + rs * RAW_STAGE);
                uint8_t* cv = conv + cs * CONV_STAGE;
                convert_tile(ra, cv, cv + TILE_BYTES, p.a_kmajor != 0, ct);
                convert_tile(ra + 128 * BKF, cv + 2 * TILE_BYTES, cv + 3 * TILE_BYTES, p.b_kmajor != 0, ct);
                // the tiles just written (generic proxy) are read by the MMAs (async proxy)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    bar_arrive(&bars->conv_full[cs]);
                    bar_arrive(&bars->raw_empty[rs]);
                }
                if (++rs == RS) { rs = 0; rph ^= 1u; }
                if (++cs == CS) { cs = 0; cph ^= 1u; }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            // instruction descriptor: f32 accumulate, TF32 A and B, both K-major, M = 128, N = 128
            const uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                   ((uint32_t)(BM >> 4) << 24);
            int cs = 0;
            uint32_t cph = 0;
            uint32_t aph[2] = {0u, 0u};
            bool ok = true;
            int local = 0;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++local) {
                const int acc = local & 1;
                if (!bar_wait(&bars->tempty[acc], aph[acc] ^ 1u, &bars->abort, p.status)) break;
                tc_fence_after();
                const uint32_t dtm = tmem + (uint32_t)(acc * BN);
                for (int kb = 0; kb < p.num_k; ++kb) {
                    if (!bar_wait(&bars->conv_full[cs], cph, &bars->abort, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t base = smem_u32(conv + cs * CONV_STAGE);
                    const uint64_t ahi = sdesc(base, 16u, 1024u), alo = sdesc(base + TILE_BYTES, 16u, 1024u);
                    const uint64_t bhi = sdesc(base + 2 * TILE_BYTES, 16u, 1024u);
                    const uint64_t blo = sdesc(base + 3 * TILE_BYTES, 16u, 1024u);
                    // K = 8 TF32 values = 32 bytes per MMA: the start address moves by 2 (16-byte units)
#pragma unroll
                    for (int k = 0; k < BKF / 8; ++k) {
                        const uint64_t o = (uint64_t)(2 * k);
                        mma_tf32(dtm, alo + o, bhi + o, idesc, (kb | k) != 0 ? 1u : 0u);
                        mma_tf32(dtm, ahi + o, blo + o, idesc, 1u);
                        mma_tf32(dtm, ahi + o, bhi + o, idesc, 1u);
                    }
                    mma_commit(&bars->conv_empty[cs]);  // frees the stage when these MMAs finish
                    if (++cs == CS) { cs = 0; cph ^= 1u; }
                }
                if (!ok) break;
                mma_commit(&bars->tfull[acc]);
                aph[acc] ^= 1u;
            }
            // every MMA issued by this CTA completes before TMEM is freed
            mma_commit(&bars->drain);
            bar_wait_drain(&bars->drain, 0u);
        }
    } else {
        // ---------------- epilogue (warps 2-5): TMEM -> registers -> global ----------------
        const int q = warp & 3;  // TMEM lanes 32q .. 32q+31 belong to this warp
        uint32_t aph[2] = {0u, 0u};
        int local = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++local) {
            const int acc = local & 1;
            if (!bar_wait(&bars->tfull[acc], aph[acc], &bars->abort, p.status)) break;
            aph[acc] ^= 1u;
            tc_fence_after();
            int b, mb, nb;
            tile_coords(p.num_m, p.num_n, t, b, mb, nb);
            const int m = mb * BM + q * 32 + lane;
            const int64_t crow = p.c_offset + (int64_t)b * p.c_bs + (int64_t)m * p.c_rs;
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                __syncwarp();  // tcgen05.ld is warp-collective: reach it converged
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + c), r);
                const int n0 = nb * BN + c;
                if (m < p.M) {
                    if (p.c_dtype == PSG_BF16) {
                        __nv_bfloat16* C = (__nv_bfloat16*)p.C;
                        for (int j = 0; j < 32; ++j)
                            if (n0 + j < p.N)
                                C[crow + (int64_t)(n0 + j) * p.c_cs] = __float2bfloat16_rn(__uint_as_float(r[j]));
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
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive(&bars->tempty[acc]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
}

// 3-D tensor map over a float32 operand as stored: dims {inner, outer,
// batch}, no swizzle (the converters read it as plain rows).
bool make_map_f32(CUtensorMap* map, const void* base, int64_t inner, int64_t outer, int64_t batch,
                  int64_t outer_stride, int64_t batch_stride, uint32_t box_inner, uint32_t box_outer)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)batch};
    cuuint64_t strides[2] = {(cuuint64_t)(outer_stride * 4), (cuuint64_t)(batch_stride * 4)};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

psg_status launch_contract_tf32(const TcOperands& o, void* stream)
{
    TcParams p = o.p;
    if (p.M == 0 || p.N == 0 || p.batch == 0) return PSG_OK;
    CUtensorMap ma, mb;
    // batch strides of a single batch are never used; keep them a legal multiple of 16 bytes
    const int64_t a_bs = p.batch > 1 ? o.a_bs : (p.a_kmajor ? o.a_ms * p.M : o.a_ks * p.K);
    const int64_t b_bs = p.batch > 1 ? o.b_bs : (p.b_kmajor ? o.b_ns * p.N : o.b_ks * p.K);
    bool ok = p.a_kmajor ? make_map_f32(&ma, o.A, p.K, p.M, p.batch, o.a_ms, a_bs, BKF, BM)
                         : make_map_f32(&ma, o.A, p.M, p.K, p.batch, o.a_ks, a_bs, BM, BKF);
    ok = ok && (p.b_kmajor ? make_map_f32(&mb, o.B, p.K, p.N, p.batch, o.b_ns, b_bs, BKF, BN)
                           : make_map_f32(&mb, o.B, p.N, p.K, p.batch, o.b_ks, b_bs, BN, BKF));
    if (!ok) return PSG_E_CUDA;
    p.num_m = (p.M + BM - 1) / BM;
    p.num_n = (p.N + BN - 1) / BN;
    p.num_k = (p.K + BKF - 1) / BKF;
    if (set_max_dynamic_smem((const void*)tc_gemm_tf32x3, SMEM_BYTES) != cudaSuccess) return PSG_E_CUDA;
    const int64_t tiles = (int64_t)p.num_m * p.num_n * p.batch;
    const int grid = (int)std::min<int64_t>(tiles, num_sms());
    launch(tc_gemm_tf32x3, grid, THREADS, SMEM_BYTES, (cudaStream_t)stream, ma, mb, p);
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

void query_contract_tf32(int64_t tiles, int* grid, int* block, int* smem, int* regs)
{
    *grid = (int)std::min<int64_t>(tiles, num_sms());
    *block = THREADS;
    *smem = SMEM_BYTES;
    *regs = kernel_regs((const void*)tc_gemm_tf32x3);
}

}  // namespace psg
