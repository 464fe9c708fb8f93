// Fused scaled dot-product attention on the 5th-generation tensor cores
// (sm_103a), for one key block: T <= 256 keys, head dim 64, bfloat16.
//
// limn's fused attention op ("The op set": one node for the whole softmax
// attention that saves L = logsumexp for its backward, instead of the
// composed T x T score tensors) and Tiki's FlashAttention target ("Write the
// attention kernel at the algorithm level").  Per (batch, head, 128-query
// tile) one CTA, two resident a SM:
//   S = Q K^T           tcgen05.mma.kind::f16, M 128, N <= 256, K 64 -> TMEM
//   P = exp(scale S - m) per query row (two threads a row, one per half of
//       the keys; masked keys 0), l = its float32 sum, L = m + log l; P
//       rounded to bf16 and written back into TMEM over the S columns its
//       thread has read
//   O = P V / l         tcgen05.mma with A (= P) from TMEM, M 128, N 64,
//                       K <= 256 -> TMEM, scaled, bf16
// With a causal mask a query tile needs keys up to its last query only:
// the copies and both products stop there.  K and V arrive as the same TMA
// box (128 keys x 64, 128-byte swizzle): the K-major B operand of S = Q K^T
// and the MN-major B operand of O = P V.
//
// Backward (two passes, deterministic: every gradient cell is accumulated by
// one CTA in a fixed order, no atomics), with D = rowsum(dO * O):
//   pass K/V (per 128-key tile, over the query tiles):
//     S^T = K Q^T, P^T = exp(scale S^T - L), dP^T = V dO^T,
//     dS^T = P^T (dP^T - D), dV = P^T dO, dK = scale dS^T Q
//   pass Q (per 128-query tile, over the key tiles):
//     S = Q K^T, P = exp(scale S - L), dP = dO V^T, dS = P (dP - D),
//     dQ = scale dS K
// Every mbarrier wait is bounded (about a second; PSG_E_TIMEOUT in the
// status word, then the CTA drains and frees TMEM).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "attention.h"
#include "launch_util.cuh"
#include "tc_util.cuh"

namespace psg {

namespace {

using namespace tcu;

constexpr int QT = 128;                     // queries (or keys) per tile
constexpr int KB = 256;                     // keys per block (the whole key range)
constexpr int HD = 64;                      // head dim
constexpr int ROW_BYTES = HD * 2;           // 128: one swizzle row
constexpr int Q_BYTES = QT * ROW_BYTES;     // 16 KB
constexpr int KV_BYTES = KB * ROW_BYTES;    // 32 KB
constexpr int FWD_THREADS = 320;            // warp 0 TMA, warp 1 MMA, warps 2-9 two per query row
constexpr int FWD_SMEM = 1024 + Q_BYTES + 2 * KV_BYTES + 256 + 4 * QT * 4;
constexpr int FWD_TMEM = 256;
// TMEM columns: S in [0, 256); P (bf16 pairs) of keys 0..127 at 0, of keys
// 128..255 at FWD_P1 (each over S its own threads have read); O at FWD_O
// (S of keys 192..255, read before P is ready)
constexpr uint32_t FWD_P1 = 128, FWD_O = 192;

struct FwdBars {
    uint64_t full, s_full, p_ready, o_full, drain;
    uint32_t tmem_base;
    int32_t abort;
};

// tcgen05.mma with the A operand in TMEM (K-major: a row a lane, two bf16 a column)
__device__ __forceinline__ void mma_f16_ts(uint32_t dtmem, uint32_t atmem, uint64_t bd, uint32_t idesc,
                                           uint32_t accum)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
        ::"r"(dtmem), "r"(atmem), "l"(bd), "r"(idesc), "r"(accum));
}

// the 8 softmax warps only
__device__ __forceinline__ void rows_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// key j of batch b is not hidden by the per-key mask (limn, "The op set":
// masking is a flag per key that composes with causal)
// 2^x, the hardware base-2 approximation (subnormal results flush to 0, as
// __expf's do): the score path works in the log2 domain, x = S c - m with
// c = scale log2(e), so each score costs one FFMA and this
__device__ __forceinline__ float ex2(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
constexpr float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
          "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
          "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ bool key_on(const AttnParams& p, int b, int j)
{
    return !p.kmask || p.kmask[(int64_t)b * p.km_sb + j] != 0;
}

__device__ __forceinline__ void mma_f16(uint32_t dtmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t accum)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(dtmem), "l"(ad), "l"(bd), "r"(idesc), "r"(accum));
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
        "[%2];"
        ::"r"(smem_u32(dst)), "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// instruction descriptor: f32 accumulate, bf16 A and B, A K-major
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *(const uint32_t*)&h;
}

__global__ void __launch_bounds__(FWD_THREADS, 2) attn_fwd(const __grid_constant__ CUtensorMap tq,
                                                           const __grid_constant__ CUtensorMap tk,
                                                           const __grid_constant__ CUtensorMap tv,
                                                           const __grid_constant__ AttnParams p)
{
    pdl_enter();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sq = smem;                       // [128 q][64 d]
    uint8_t* sk = sq + Q_BYTES;               // [256 keys][64 d], two 128-key boxes
    uint8_t* sv = sk + KV_BYTES;              // [256 keys][64 d]
    FwdBars* bars = (FwdBars*)(sv + KV_BYTES);
    float* red_m = (float*)((uint8_t*)bars + 256);  // [2 halves][128 rows]
    float* red_l = red_m + 2 * QT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a 1-D grid, rank-major, longest tile first (as in attn_fwd_long)
    const int nq = (p.T + QT - 1) / QT;
    const int hb = blockIdx.x % (p.H * p.B), rank = blockIdx.x / (p.H * p.B);
    const int h = hb % p.H, b = hb / p.H;
    const int qt = p.causal ? nq - 1 - rank : rank;
    const int q0 = qt * QT;
    // keys any query of this tile sees; MMA steps of 16 keys past them read zeros
    const int kv_end = p.causal ? min(p.T, q0 + QT) : p.T;
    const int kv_pad = (kv_end + 15) & ~15;
    const int nkb = (kv_end + QT - 1) / QT;  // 128-key boxes to load (1 or 2)

    if (threadIdx.x == 0) {
        bar_init(&bars->full, 1);
        bar_init(&bars->s_full, 1);
        bar_init(&bars->p_ready, 8);
        bar_init(&bars->o_full, 1);
        bar_init(&bars->drain, 1);
        bars->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&bars->tmem_base)), "r"(FWD_TMEM));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            bar_expect_tx(&bars->full, Q_BYTES + 2 * nkb * Q_BYTES);
            tma_load_4d(sq, &tq, &bars->full, 0, q0, h, b);
            for (int kb = 0; kb < nkb; ++kb) {
                tma_load_4d(sk + kb * Q_BYTES, &tk, &bars->full, 0, kb * QT, h, b);
                tma_load_4d(sv + kb * Q_BYTES, &tv, &bars->full, 0, kb * QT, h, b);
            }
            bar_wait_drain(&bars->full, 0u);  // the copies land before this CTA may exit
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = bar_wait(&bars->full, 0u, &bars->abort, p.status);
            if (ok) {
                tc_fence_after();
                // S = Q K^T: A = Q (K-major), B = K (K-major, N = kv_pad keys); K step 16 = 32 bytes
                const uint64_t ad = sdesc(smem_u32(sq), 16u, 1024u), bd = sdesc(smem_u32(sk), 16u, 1024u);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k)
                    mma_f16(tmem, ad + 2u * k, bd + 2u * k, idesc_bf16(QT, kv_pad, false), k > 0 ? 1u : 0u);
                mma_commit(&bars->s_full);
                ok = bar_wait(&bars->p_ready, 0u, &bars->abort, p.status);
            }
            if (ok) {
                tc_fence_after();
                // O = P V: A = P from TMEM (8 columns a 16-key step), B = V (MN-major:
                // rows = keys, 8-row groups 1024 B apart; a 16-key step is 2 KB)
                const uint64_t vd = sdesc(smem_u32(sv), 8192u, 1024u);
                for (int ks = 0; ks < kv_pad / 16; ++ks) {
                    const uint32_t pa = tmem + (ks < 8 ? 8u * ks : FWD_P1 + 8u * (ks - 8));
                    mma_f16_ts(tmem + FWD_O, pa, vd + 128u * ks, idesc_bf16(QT, HD, true), ks > 0 ? 1u : 0u);
                }
                mma_commit(&bars->o_full);
            }
            mma_commit(&bars->drain);
            bar_wait_drain(&bars->drain, 0u);
        }
    } else {
        // rows: warp w owns TMEM lanes 32 (w % 4) .. + 31 (the query rows) and
        // the keys of half (w - 2) / 4
        const int half = (warp - 2) >> 2;
        const int g = warp & 3;
        const int r = 32 * g + lane;
        const int i = q0 + r;
        const uint32_t trow = tmem + ((uint32_t)(32 * g) << 16);
        const int c_beg = QT * half, c_end = min(c_beg + QT, kv_pad);
        const uint32_t pcol = half ? FWD_P1 : 0u;
        // ok stays warp-uniform: the TMEM loads and stores below are warp-collective
        bool ok = __all_sync(0xffffffffu, bar_wait(&bars->s_full, 0u, &bars->abort, p.status));
        tc_fence_after();
        const int kmax = p.causal ? min(i + 1, p.T) : p.T;  // keys 0 .. kmax-1 are visible
        // the warp's smallest kmax: 32-key groups below it need no per-key tests
        const int kmin_w = p.kmask ? 0 : (p.causal ? min(q0 + 32 * g + 1, p.T) : p.T);
        // scores in the log2 domain: m is the max of S c, c = scale log2(e)
        const float c2 = p.scale * LOG2E;
        float m = -INFINITY;
        if (ok) {
            for (int c = c_beg; c < c_end; c += 32) {
                uint32_t s[32];
                __syncwarp();
                tmem_ld32(trow + (uint32_t)c, s);
                const bool full = c + 32 <= kmin_w;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (full || (c + j < kmax && key_on(p, b, c + j))) m = fmaxf(m, __uint_as_float(s[j]) * c2);
            }
        }
        red_m[half * QT + r] = m;
        rows_sync();
        m = fmaxf(red_m[r], red_m[QT + r]);  // the row's max, the same in both halves
        float l = 0.0f;
        if (ok) {
            for (int c = c_beg; c < c_end; c += 32) {
                uint32_t s[32];
                __syncwarp();
                tmem_ld32(trow + (uint32_t)c, s);
                uint32_t w[16];
                const bool full = c + 32 <= kmin_w;
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    // l sums the float32 weights (L = (m + log2 l) ln 2 is the
                    // row's logsumexp); P is rounded to bf16 only as the MMA operand
                    const bool v0 = full || (c + j < kmax && key_on(p, b, c + j));
                    const bool v1 = full || (c + j + 1 < kmax && key_on(p, b, c + j + 1));
                    const float e0 = v0 ? ex2(fmaf(__uint_as_float(s[j]), c2, -m)) : 0.0f;
                    const float e1 = v1 ? ex2(fmaf(__uint_as_float(s[j + 1]), c2, -m)) : 0.0f;
                    l += e0;
                    l += e1;
                    w[j >> 1] = pack_bf16(e0, e1);
                }
                // columns (c - c_beg) / 2 .. + 15 of the half's P: S this thread has read
                tmem_st16(trow + pcol + (uint32_t)((c - c_beg) >> 1), w);
            }
            tmem_wait_st();
        }
        red_l[half * QT + r] = l;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) bar_arrive(&bars->p_ready);
        rows_sync();
        l = red_l[r] + red_l[QT + r];  // first half, then second: one order in both
        if (ok) ok = __all_sync(0xffffffffu, bar_wait(&bars->o_full, 0u, &bars->abort, p.status));
        tc_fence_after();
        if (ok) {
            uint32_t o[32];
            __syncwarp();  // every lane reaches the collective load
            tmem_ld32(trow + FWD_O + 32u * half, o);
            if (i < p.T) {
                // a query that sees no key at all (every key masked): O = 0, L = -inf
                const float inv = l > 0.0f ? 1.0f / l : 0.0f;
                if (half == 0) p.lse[((int64_t)b * p.H + h) * p.T + i] = l > 0.0f ? m * LN2 + logf(l) : -INFINITY;
                __nv_bfloat16* dst = (__nv_bfloat16*)p.o + p.o_off + (int64_t)b * p.o_sb + (int64_t)i * p.o_st +
                                     (int64_t)h * p.o_sh + 32 * half;
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    w[j] = pack_bf16(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    ((uint4*)dst)[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(FWD_TMEM));
}

// ---- forward over many key blocks: an online softmax ----------------------
// For T > 256 a query tile walks its key blocks of 128 (Tiki, "Write the
// attention kernel at the algorithm level": the running max m, denominator
// l and weighted sum a, rescaled as the max grows).  Per block j:
//   S_j = Q K_j^T                          (tcgen05.mma -> TMEM columns 0..127)
//   m' = max(m, max_k scale S_j), alpha = exp(m - m')
//   P_j = exp(scale S_j - m')             (bf16, back into TMEM over the S
//                                          columns its thread has read)
//   l = alpha l + rowsum(P_j), O_j = P_j V_j (a fresh TMEM accumulator,
//                                          columns 128..191)
//   a = alpha a + O_j                      (float32, in the row threads'
//                                          registers: 32 head-dim columns each)
// and at the end O = a / l, L = m + log l (a query with no visible key: O = 0,
// L = -inf).  K and V blocks come through a two-slot ring.  Roles as in the
// one-block kernel: warp 0 TMA, warp 1 MMA, warps 2-9 two threads a query row
// (one per 64-key half of a block, and per 32-column half of the head dim).
constexpr int LKV_SLOT = 2 * Q_BYTES;  // a K block and a V block: 32 KB
constexpr int LFWD_SMEM = 1024 + Q_BYTES + 2 * LKV_SLOT + 256 + 2 * 2 * QT * 4 + 2 * QT * 4;
constexpr uint32_t LFWD_O = 128;       // TMEM: S and P in 0..127, O_j in 128..191

struct LFwdBars {
    uint64_t q_full, kv_full[2], kv_empty[2], s_full, p_ready, o_full, drain;
    uint32_t tmem_base;
    int32_t abort;
};

__global__ void __launch_bounds__(FWD_THREADS, 2) attn_fwd_long(const __grid_constant__ CUtensorMap tq,
                                                                const __grid_constant__ CUtensorMap tk,
                                                                const __grid_constant__ CUtensorMap tv,
                                                                const __grid_constant__ AttnParams p)
{
    pdl_enter();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sq = smem;                        // [128 q][64 d]
    uint8_t* skv = sq + Q_BYTES;               // [2 slots][K block, V block]
    LFwdBars* bars = (LFwdBars*)(skv + 2 * LKV_SLOT);
    float* red_m = (float*)((uint8_t*)bars + 256);  // [2 blocks (parity)][2 halves][128 rows]
    float* red_l = red_m + 2 * 2 * QT;               // [2 halves][128 rows]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nall = (p.T + QT - 1) / QT;
    // a 1-D grid in order of decreasing work: rank r takes query tile
    // nall - 1 - r (causal: the tile that walks the most key blocks first)
    // of every head and batch, so the short tiles fill the tail
    const int hb = blockIdx.x % (p.H * p.B), rank = blockIdx.x / (p.H * p.B);
    const int h = hb % p.H, b = hb / p.H;
    const int qt = p.causal ? nall - 1 - rank : rank;
    const int q0 = qt * QT;
    const int nblk = p.causal ? min(qt + 1, nall) : nall;  // key blocks any query of the tile sees

    if (threadIdx.x == 0) {
        bar_init(&bars->q_full, 1);
        for (int s = 0; s < 2; ++s) {
            bar_init(&bars->kv_full[s], 1);
            bar_init(&bars->kv_empty[s], 1);
        }
        bar_init(&bars->s_full, 1);
        bar_init(&bars->p_ready, 8);
        bar_init(&bars->o_full, 1);
        bar_init(&bars->drain, 1);
        bars->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&bars->tmem_base)), "r"(FWD_TMEM));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            bar_expect_tx(&bars->q_full, Q_BYTES);
            tma_load_4d(sq, &tq, &bars->q_full, 0, q0, h, b);
            uint32_t armed = 0, armed_ph = 0;
            for (int j = 0; j < nblk; ++j) {
                const int s = j & 1;
                // a slot is refilled once the products of the block before in it are done
                if (j >= 2 && !bar_wait(&bars->kv_empty[s], (uint32_t)(((j >> 1) - 1) & 1), &bars->abort, p.status))
                    break;
                uint8_t* slot = skv + s * LKV_SLOT;
                bar_expect_tx(&bars->kv_full[s], 2 * Q_BYTES);
                tma_load_4d(slot, &tk, &bars->kv_full[s], 0, j * QT, h, b);
                tma_load_4d(slot + Q_BYTES, &tv, &bars->kv_full[s], 0, j * QT, h, b);
                armed |= 1u << s;
                armed_ph = (armed_ph & ~(1u << s)) | ((uint32_t)((j >> 1) & 1) << s);
            }
            // every copy this CTA issued lands before it may exit
            bar_wait_drain(&bars->q_full, 0u);
            for (int s = 0; s < 2; ++s)
                if (armed & (1u << s)) bar_wait_drain(&bars->kv_full[s], (armed_ph >> s) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = bar_wait(&bars->q_full, 0u, &bars->abort, p.status);
            const uint64_t ad = sdesc(smem_u32(sq), 16u, 1024u);
            for (int j = 0; j < nblk && ok; ++j) {
                const int s = j & 1;
                ok = bar_wait(&bars->kv_full[s], (uint32_t)((j >> 1) & 1), &bars->abort, p.status);
                // S_j goes over P_{j-1}: the product that reads it has completed
                if (ok && j > 0) ok = bar_wait(&bars->o_full, (uint32_t)((j - 1) & 1), &bars->abort, p.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t sk = smem_u32(skv + s * LKV_SLOT);
                const uint64_t bd = sdesc(sk, 16u, 1024u);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k)
                    mma_f16(tmem, ad + 2u * k, bd + 2u * k, idesc_bf16(QT, QT, false), k > 0 ? 1u : 0u);
                mma_commit(&bars->s_full);
                // P_j is written and the running O rescaled by the row threads
                ok = bar_wait(&bars->p_ready, (uint32_t)(j & 1), &bars->abort, p.status);
                if (!ok) break;
                tc_fence_after();
                // O += P_j V_j (the first block overwrites): A = P from TMEM (keys
                // 0..63 in columns 0..31, keys 64..127 in columns 64..95, 8
                // columns a 16-key step), B = V MN-major
                const uint64_t vd = sdesc(sk + Q_BYTES, 8192u, 1024u);
#pragma unroll
                for (int ks = 0; ks < QT / 16; ++ks) {
                    const uint32_t pa = tmem + (ks < 4 ? 8u * ks : 64u + 8u * (ks - 4));
                    mma_f16_ts(tmem + LFWD_O, pa, vd + 128u * ks, idesc_bf16(QT, HD, true), (j > 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(&bars->o_full);
                mma_commit(&bars->kv_empty[s]);  // K_j and V_j read once these complete
            }
            mma_commit(&bars->drain);
            bar_wait_drain(&bars->drain, 0u);
        }
    } else {
        // warp w owns TMEM lanes 32 (w % 4) .. + 31 (the query rows), the keys
        // 64 half .. + 63 of every block and head-dim columns 32 half .. + 31
        const int half = (warp - 2) >> 2;
        const int g = warp & 3;
        const int r = 32 * g + lane;
        const int i = q0 + r;
        const uint32_t trow = tmem + ((uint32_t)(32 * g) << 16);
        // scores in the log2 domain: m is the running max of S c, c = scale log2(e)
        const float c2 = p.scale * LOG2E;
        float m = -INFINITY, lh = 0.0f;
        bool ok = true;
        for (int j = 0; j < nblk; ++j) {
            ok = ok && __all_sync(0xffffffffu, bar_wait(&bars->s_full, (uint32_t)(j & 1), &bars->abort, p.status));
            tc_fence_after();
            const int kb = j * QT + 64 * half;  // this thread's first key of the block
            // every key of the thread's 64 visible to every row of its warp:
            // no per-key tests (all blocks but the diagonal and the ragged last)
            const bool full = kb + 63 < p.T && (!p.causal || kb + 63 <= q0 + 32 * g) && !p.kmask;
            // the thread's 64 scores: two loads and one wait a pass (the
            // softmax pass reads them again rather than hold 64 registers
            // across the exchange of the block max)
            float mb = -INFINITY;
            if (ok) {
                uint32_t sv0[32], sv1[32];
                __syncwarp();
                tmem_ld32_nowait(trow + 64u * half, sv0);
                tmem_ld32_nowait(trow + 64u * half + 32u, sv1);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int kj = kb + c, kj1 = kb + 32 + c;
                    if (full || (kj < p.T && (!p.causal || kj <= i) && key_on(p, b, kj)))
                        mb = fmaxf(mb, __uint_as_float(sv0[c]) * c2);
                    if (full || (kj1 < p.T && (!p.causal || kj1 <= i) && key_on(p, b, kj1)))
                        mb = fmaxf(mb, __uint_as_float(sv1[c]) * c2);
                }
            }
            float* rm = red_m + (j & 1) * 2 * QT;
            rm[half * QT + r] = mb;
            rows_sync();
            const float mn = fmaxf(m, fmaxf(rm[r], rm[QT + r]));  // the running max, the same in both halves
            const float alpha = m == -INFINITY ? 0.0f : ex2(m - mn);
            float lb = 0.0f;
            if (ok) {
                // P over the S columns 64 half .. + 31, 32 keys at a time (the
                // second group's scores are read before the first group's P
                // goes over them)
                auto p32 = [&](const uint32_t (&sx)[32], int k0, uint32_t col) {
                    uint32_t w[16];
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        float e[2];
#pragma unroll
                        for (int x = 0; x < 2; ++x) {
                            const int kj = k0 + c + x;
                            const bool vis = full || (kj < p.T && (!p.causal || kj <= i) && key_on(p, b, kj));
                            e[x] = vis ? ex2(fmaf(__uint_as_float(sx[c + x]), c2, -mn)) : 0.0f;
                            lb += e[x];
                        }
                        w[c >> 1] = pack_bf16(e[0], e[1]);
                    }
                    tmem_st16(trow + col, w);
                };
                uint32_t sv0[32], sv1[32];
                __syncwarp();
                tmem_ld32(trow + 64u * half, sv0);
                tmem_ld32_nowait(trow + 64u * half + 32u, sv1);
                p32(sv0, kb, 64u * half);
                tmem_ld_wait();
                p32(sv1, kb + 32, 64u * half + 16u);
                // the running O (this thread's 32 head-dim columns) takes the
                // new max before P_j V_j adds to it: once the product of the
                // block before has completed, and only when some row's max moved
                if (j > 0) ok = __all_sync(0xffffffffu, bar_wait(&bars->o_full, (uint32_t)((j - 1) & 1), &bars->abort,
                                                                 p.status));
                tc_fence_after();
                if (ok && j > 0 && !__all_sync(0xffffffffu, alpha == 1.0f)) {
                    uint32_t o[32];
                    tmem_ld32(trow + LFWD_O + 32u * half, o);
#pragma unroll
                    for (int d = 0; d < 32; ++d) o[d] = __float_as_uint(__uint_as_float(o[d]) * alpha);
                    tmem_st32(trow + LFWD_O + 32u * half, o);
                }
                tmem_wait_st();
            }
            lh = lh * alpha + lb;
            m = mn;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive(&bars->p_ready);
        }
        // the last product done: O holds sum_j P_j V_j, every block at the final max
        float a[32];
        if (ok && nblk > 0)
            ok = __all_sync(0xffffffffu, bar_wait(&bars->o_full, (uint32_t)((nblk - 1) & 1), &bars->abort, p.status));
        tc_fence_after();
        if (ok) {
            uint32_t o[32];
            tmem_ld32(trow + LFWD_O + 32u * half, o);
#pragma unroll
            for (int d = 0; d < 32; ++d) a[d] = __uint_as_float(o[d]);
        }
        // l: the two key halves' sums, first half then second (one order in both threads)
        red_l[half * QT + r] = lh;
        rows_sync();
        const float l = red_l[r] + red_l[QT + r];
        if (ok && i < p.T) {
            const float inv = l > 0.0f ? 1.0f / l : 0.0f;
            // L = ln(sum exp(scale S)) = (m + log2 l) ln 2
            if (half == 0) p.lse[((int64_t)b * p.H + h) * p.T + i] = l > 0.0f ? m * LN2 + logf(l) : -INFINITY;
            __nv_bfloat16* dst = (__nv_bfloat16*)p.o + p.o_off + (int64_t)b * p.o_sb + (int64_t)i * p.o_st +
                                 (int64_t)h * p.o_sh + 32 * half;
            uint32_t w[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) w[x] = pack_bf16(a[2 * x] * inv, a[2 * x + 1] * inv);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                ((uint4*)dst)[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(FWD_TMEM));
}

// ---- backward ---------------------------------------------------------------
// Both passes, one CTA per (128-row tile of its own operands, head, batch),
// two resident a SM.  The streamed operand tiles come through a ring of two
// tile slots (the producer refills a slot once the second products of the
// tile in it have completed) and are taken 64 rows (a sub-tile) at a time:
//   pass K/V (KV): own K, V (rows = keys); streamed Q, dO (columns = queries)
//     S^T = K Q^T, dP^T = V dO^T, P^T = exp(scale S^T - L), dS^T = P^T (dP^T - D)
//     dV += P^T dO, dK += dS^T Q            (dK scaled by `scale` at the end)
//   pass Q: own Q, dO (rows = queries); streamed K, V (columns = keys)
//     S = Q K^T, dP = dO V^T, P = exp(scale S - L), dS = P (dP - D)
//     dQ += dS K                            (scaled by `scale` at the end)
// TMEM columns (256): S 0-63, dP 64-127, dV 128-191, dK or dQ 192-255.  P and
// dS (bf16 pairs) go back into TMEM over the S and dP columns their own
// thread has read (half h of the columns at 32 h .. 32 h + 15), and the
// second products take them as the A operand from TMEM.  Two threads share a
// row, one per half of the sub-tile's 64 columns; each gradient cell is
// accumulated by one CTA in a fixed order (no atomics).
constexpr int T_BYTES = QT * ROW_BYTES;     // 16 KB: a 128-row tile of one operand
constexpr int SUB = 64;                     // streamed rows a sub-tile
constexpr int BWD_THREADS = 320;            // warp 0 TMA, warp 1 MMA, warps 2-9 two per row
constexpr int BWD_SMEM = 1024 + 6 * T_BYTES + 256;
constexpr int BWD_TMEM = 256;
constexpr uint32_t BWD_DP = 64, BWD_ACC0 = 128, BWD_ACC1 = 192;

struct BwdBars {
    uint64_t full[2], empty[2], mm1, ready, mm2, drain;
    uint32_t tmem_base;
    int32_t abort;
};

// D[b, h, t] = sum_d dO[b, t, h, d] * O[b, t, h, d] (float32 total of exact
// bf16 products, folded in a fixed order): 8 lanes per row, 16 bytes of O
// and dO per lane, a 3-level shuffle fold inside the 8-lane group
__global__ void __launch_bounds__(256) attn_delta(const __grid_constant__ AttnTensor o,
                                                  const __grid_constant__ AttnTensor dO,
                                                  const __grid_constant__ AttnParams p)
{
    pdl_enter();
    const int64_t rows = (int64_t)p.B * p.T * p.H;
    const int sub = threadIdx.x & 7, grp = (threadIdx.x & 31) >> 3;
    // warp-uniform loop over groups of 4 rows (the shuffles need every lane)
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * 4; r0 < rows; r0 += warps * 4) {
        const int64_t r = r0 + grp;
        const bool ok = r < rows;
        float v = 0.0f;
        int b = 0, t = 0, h = 0;
        if (ok) {
            h = (int)(r % p.H);
            t = (int)((r / p.H) % p.T);
            b = (int)(r / ((int64_t)p.H * p.T));
            const uint4 x =
                ((const uint4*)((const __nv_bfloat16*)o.ptr + o.off + b * o.sb + t * o.st + h * o.sh))[sub];
            const uint4 y =
                ((const uint4*)((const __nv_bfloat16*)dO.ptr + dO.off + b * dO.sb + t * dO.st + h * dO.sh))[sub];
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float x0 = __uint_as_float(xs[u] << 16), x1 = __uint_as_float(xs[u] & 0xffff0000u);
                const float y0 = __uint_as_float(ys[u] << 16), y1 = __uint_as_float(ys[u] & 0xffff0000u);
                v = __fadd_rn(v, __fadd_rn(__fmul_rn(x0, y0), __fmul_rn(x1, y1)));
            }
        }
        for (int off = 4; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off, 8));
        if (ok && sub == 0) p.delta[((int64_t)b * p.H + h) * p.T + t] = v;
    }
}

// store 32 float32 accumulator columns (scaled) of row `row` as bf16, at
// head-dim columns c0 .. c0 + 31
__device__ __forceinline__ void store_row32(const AttnTensor& t, int b, int row, int h, int c0,
                                            const uint32_t (&x)[32], float scale)
{
    __nv_bfloat16* dst =
        (__nv_bfloat16*)t.ptr + t.off + (int64_t)b * t.sb + (int64_t)row * t.st + (int64_t)h * t.sh + c0;
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        w[j] = pack_bf16(__uint_as_float(x[2 * j]) * scale, __uint_as_float(x[2 * j + 1]) * scale);
#pragma unroll
    for (int u = 0; u < 4; ++u) ((uint4*)dst)[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
}

template <bool KV>
__device__ __forceinline__ void attn_bwd_pass(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                              const CUtensorMap& tdo, const AttnTensor& g0, const AttnTensor& g1,
                                              const AttnParams& p, int b, int h, int rank)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* own0 = smem;                   // KV: K, Q: Q  [128 rows][64]
    uint8_t* own1 = own0 + T_BYTES;         // KV: V, Q: dO
    uint8_t* st0 = own1 + T_BYTES;          // KV: Q, Q: K  [2 slots][128 rows][64]
    uint8_t* st1 = st0 + 2 * T_BYTES;       // KV: dO, Q: V
    BwdBars* bars = (BwdBars*)(st1 + 2 * T_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntile = (p.T + QT - 1) / QT;
    // own tile by rank of decreasing work: causal, a key tile sees the query
    // tiles from its own on (the first key tile the most), a query tile the
    // key tiles up to its own (the last query tile the most)
    const int ot = KV || !p.causal ? rank : ntile - 1 - rank;
    const int r0 = ot * QT;  // first own row (key in KV, query in Q)
    // streamed tiles: KV, the query tiles that see these keys; Q, the key tiles these queries see
    const int it0 = KV ? (p.causal ? ot : 0) : 0;
    const int it1 = KV ? ntile : (p.causal ? min(ot + 1, ntile) : ntile);
    const int nst = 2 * (it1 - it0);  // sub-tiles

    if (threadIdx.x == 0) {
        bar_init(&bars->full[0], 1);
        bar_init(&bars->full[1], 1);
        bar_init(&bars->empty[0], 1);
        bar_init(&bars->empty[1], 1);
        bar_init(&bars->mm1, 1);
        bar_init(&bars->ready, 8);
        bar_init(&bars->mm2, 1);
        bar_init(&bars->drain, 1);
        bars->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&bars->tmem_base)), "r"(BWD_TMEM));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            const CUtensorMap* m_own0 = KV ? &tk : &tq;
            const CUtensorMap* m_own1 = KV ? &tv : &tdo;
            const CUtensorMap* m_st0 = KV ? &tq : &tk;
            const CUtensorMap* m_st1 = KV ? &tdo : &tv;
            uint32_t armed = 0, armed_ph = 0;  // slots filled, and the parity of each one's last fill
            for (int t = it0; t < it1; ++t) {
                const int u = t - it0, slot = u & 1;
                // a slot is refilled once the tile before in it has been used up
                if (u >= 2 && !bar_wait(&bars->empty[slot], (uint32_t)(((u >> 1) - 1) & 1), &bars->abort, p.status))
                    break;
                uint64_t* fb = &bars->full[slot];
                bar_expect_tx(fb, (u == 0 ? 4u : 2u) * T_BYTES);
                if (u == 0) {
                    tma_load_4d(own0, m_own0, fb, 0, r0, h, b);
                    tma_load_4d(own1, m_own1, fb, 0, r0, h, b);
                }
                tma_load_4d(st0 + slot * T_BYTES, m_st0, fb, 0, t * QT, h, b);
                tma_load_4d(st1 + slot * T_BYTES, m_st1, fb, 0, t * QT, h, b);
                armed |= 1u << slot;
                armed_ph = (armed_ph & ~(1u << slot)) | ((uint32_t)((u >> 1) & 1) << slot);
            }
            // the copies land before this CTA may exit
            for (int s = 0; s < 2; ++s)
                if (armed & (1u << s)) bar_wait_drain(&bars->full[s], (armed_ph >> s) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            const uint64_t a0 = sdesc(smem_u32(own0), 16u, 1024u), a1 = sdesc(smem_u32(own1), 16u, 1024u);
            for (int st = 0; st < nst && ok; ++st) {
                const int t = st >> 1, s = st & 1, slot = t & 1;
                if (s == 0) ok = bar_wait(&bars->full[slot], (uint32_t)((t >> 1) & 1), &bars->abort, p.status);
                // the previous sub-tile's second products have read P and dS (S and dP columns)
                if (ok && st > 0) ok = bar_wait(&bars->mm2, (uint32_t)((st - 1) & 1), &bars->abort, p.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t sub = smem_u32(st0 + slot * T_BYTES) + (uint32_t)(s * SUB * ROW_BYTES);
                const uint32_t sub1 = smem_u32(st1 + slot * T_BYTES) + (uint32_t)(s * SUB * ROW_BYTES);
                const uint64_t b0 = sdesc(sub, 16u, 1024u), b1 = sdesc(sub1, 16u, 1024u);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k) {
                    mma_f16(tmem, a0 + 2u * k, b0 + 2u * k, idesc_bf16(QT, SUB, false), k > 0 ? 1u : 0u);
                    mma_f16(tmem + BWD_DP, a1 + 2u * k, b1 + 2u * k, idesc_bf16(QT, SUB, false), k > 0 ? 1u : 0u);
                }
                mma_commit(&bars->mm1);
                ok = bar_wait(&bars->ready, (uint32_t)(st & 1), &bars->abort, p.status);
                if (!ok) break;
                tc_fence_after();
                // KV: dV += P^T dO_sub, dK += dS^T Q_sub; Q: dQ += dS K_sub.  B MN-major
                // (rows = the sub-tile's streamed rows; a 16-row K step is 2 KB)
                const uint64_t n0 = sdesc(sub, 8192u, 1024u), n1 = sdesc(sub1, 8192u, 1024u);
#pragma unroll
                for (int ks = 0; ks < SUB / 16; ++ks) {
                    const uint32_t col = 32u * (ks >> 1) + 8u * (ks & 1);  // half ks / 2, 8 columns a step
                    const uint32_t acc = (st > 0 || ks > 0) ? 1u : 0u;
                    if (KV) mma_f16_ts(tmem + BWD_ACC0, tmem + col, n1 + 128u * ks, idesc_bf16(QT, HD, true), acc);
                    mma_f16_ts(tmem + BWD_ACC1, tmem + BWD_DP + col, n0 + 128u * ks, idesc_bf16(QT, HD, true), acc);
                }
                mma_commit(&bars->mm2);
                // the tile's last products: its slot is free once they complete
                if (s == 1) mma_commit(&bars->empty[slot]);
            }
            mma_commit(&bars->drain);
            bar_wait_drain(&bars->drain, 0u);
        }
    } else {
        // rows: warp w owns TMEM lanes 32 (w % 4) .. + 31 and half (w - 2) / 4 of each sub-tile's columns
        const int half = (warp - 2) >> 2;
        const int g = warp & 3;
        const int r = 32 * g + lane;
        const int row = r0 + r;  // KV: key j; Q: query i
        const uint32_t trow = tmem + ((uint32_t)(32 * g) << 16);
        const int64_t lbase = ((int64_t)b * p.H + h) * p.T;
        // P = exp(scale S - L) = 2^(S c - L log2 e), c = scale log2(e): one FFMA
        // and one base-2 step a score
        const float c2 = p.scale * LOG2E;
        float Lr = 0.0f, Dr = 0.0f;
        if (!KV && row < p.T) {
            Lr = p.lse[lbase + row] * LOG2E;
            Dr = p.delta[lbase + row];
        }
        const int w_lo = r0 + 32 * g, w_hi = w_lo + 31;  // this warp's own rows
        bool ok = true;
        for (int st = 0; st < nst; ++st) {
            const int t = st >> 1, s = st & 1;
            // KV pass: L and D of the 32 queries this warp's columns cover,
            // one per lane (loaded before the wait), handed out by shuffles
            float Lq = 0.0f, Dq = 0.0f;
            if (KV) {
                const int iq = (it0 + t) * QT + SUB * s + 32 * half + lane;
                if (iq < p.T) {
                    Lq = __ldg(p.lse + lbase + iq) * LOG2E;
                    Dq = __ldg(p.delta + lbase + iq);
                }
            }
            // the 32 streamed rows this thread's columns cover; every pair with
            // the warp's own rows visible: no per-pair tests
            const int o_lo = (it0 + t) * QT + SUB * s + 32 * half, o_hi = o_lo + 31;
            const bool full = o_hi < p.T && w_hi < p.T && !p.kmask &&
                              (!p.causal || (KV ? w_hi <= o_lo : o_hi <= w_lo));
            ok = ok && __all_sync(0xffffffffu, bar_wait(&bars->mm1, (uint32_t)(st & 1), &bars->abort, p.status));
            tc_fence_after();
            if (ok) {
#pragma unroll
                for (int cc = 0; cc < 32; cc += 16) {
                    uint32_t sv[16], dp[16], wp[8], ws[8];
                    __syncwarp();
                    tmem_ld16(trow + 32u * half + cc, sv);
                    tmem_ld16(trow + BWD_DP + 32u * half + cc, dp);
#pragma unroll
                    for (int u = 0; u < 16; u += 2) {
                        float pv[2], dsv[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int c = SUB * s + 32 * half + cc + u + e;  // streamed row within its tile
                            const int other = (it0 + t) * QT + c;
                            const int i = KV ? other : row, j = KV ? row : other;
                            const bool vis = full || (i < p.T && j < p.T && (!p.causal || j <= i) && key_on(p, b, j));
                            const float L = KV ? __shfl_sync(0xffffffffu, Lq, cc + u + e) : Lr;
                            const float D = KV ? __shfl_sync(0xffffffffu, Dq, cc + u + e) : Dr;
                            const float pe = vis ? ex2(fmaf(__uint_as_float(sv[u + e]), c2, -L)) : 0.0f;
                            pv[e] = pe;
                            dsv[e] = pe * (__uint_as_float(dp[u + e]) - D);
                        }
                        wp[u >> 1] = pack_bf16(pv[0], pv[1]);
                        ws[u >> 1] = pack_bf16(dsv[0], dsv[1]);
                    }
                    // over the S and dP columns this thread has just read
                    if (KV) tmem_st8(trow + 32u * half + (cc >> 1), wp);
                    tmem_st8(trow + BWD_DP + 32u * half + (cc >> 1), ws);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive(&bars->ready);
        }
        // the last sub-tile's second products are done: the gradients are complete
        if (ok && nst > 0)
            ok = __all_sync(0xffffffffu, bar_wait(&bars->mm2, (uint32_t)((nst - 1) & 1), &bars->abort, p.status));
        tc_fence_after();
        if (ok) {
            // (every tile has at least one streamed tile: nst >= 2 for T >= 1)
            uint32_t x[32];
            __syncwarp();
            if (KV) {
                tmem_ld32(trow + BWD_ACC0 + 32u * half, x);
                if (row < p.T) store_row32(g0, b, row, h, 32 * half, x, 1.0f);
            }
            tmem_ld32(trow + BWD_ACC1 + 32u * half, x);
            if (row < p.T) store_row32(KV ? g1 : g0, b, row, h, 32 * half, x, p.scale);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(BWD_TMEM));
}

// both passes in one grid (z < B: pass K/V of batch z, else pass Q of batch
// z - B), so the two kinds of CTA fill each other's tails
__global__ void __launch_bounds__(BWD_THREADS, 2) attn_bwd(const __grid_constant__ CUtensorMap tq,
                                                           const __grid_constant__ CUtensorMap tk,
                                                           const __grid_constant__ CUtensorMap tv,
                                                           const __grid_constant__ CUtensorMap tdo,
                                                           const __grid_constant__ AttnTensor dq,
                                                           const __grid_constant__ AttnTensor dk,
                                                           const __grid_constant__ AttnTensor dv,
                                                           const __grid_constant__ AttnParams p)
{
    pdl_enter();
    // a 1-D grid, rank-major: every (head, pass, batch) of rank 0 (the
    // longest tiles) first
    const int per = p.H * 2 * p.B;
    const int rank = (int)blockIdx.x / per, rest = (int)blockIdx.x - rank * per;
    const int h = rest % p.H, z = rest / p.H;
    if (z < p.B) attn_bwd_pass<true>(tq, tk, tv, tdo, dv, dk, p, z, h, rank);
    else attn_bwd_pass<false>(tq, tk, tv, tdo, dq, dq, p, z - p.B, h, rank);
}

// 4-D tensor map over a [B, T, H, 64] bfloat16 operand: dims {64, T, H, B},
// box {64, rows, 1, 1}, 128-byte swizzle (one 128-byte row per token).
bool make_map_attn(CUtensorMap* map, const AttnTensor& t, int T, int H, int B, uint32_t rows)
{
    auto enc = encode_fn();
    if (!enc) return false;
    const void* base = (const char*)t.ptr + t.off * 2;
    cuuint64_t dims[4] = {(cuuint64_t)HD, (cuuint64_t)T, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)(t.st * 2), (cuuint64_t)(t.sh * 2), (cuuint64_t)(t.sb * 2)};
    cuuint32_t box[4] = {(cuuint32_t)HD, rows, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

psg_status launch_attention_fwd(const AttnTensor& q, const AttnTensor& k, const AttnTensor& v, const AttnParams& p,
                                void* stream)
{
    if (p.B == 0 || p.T == 0 || p.H == 0) return PSG_OK;
    CUtensorMap mq, mk, mv;
    if (!make_map_attn(&mq, q, p.T, p.H, p.B, QT) || !make_map_attn(&mk, k, p.T, p.H, p.B, QT) ||
        !make_map_attn(&mv, v, p.T, p.H, p.B, QT))
        return PSG_E_CUDA;
    const dim3 grid((unsigned)((p.T + QT - 1) / QT), (unsigned)p.H, (unsigned)p.B);
    if (p.T > KB) {
        // more keys than one block: the online softmax over 128-key blocks
        if (set_max_dynamic_smem((const void*)attn_fwd_long, LFWD_SMEM) != cudaSuccess) return PSG_E_CUDA;
        const int64_t nlong = (int64_t)grid.x * p.H * p.B;
        if (nlong > 0x7fffffffll) return PSG_E_UNSUPPORTED_LAYOUT;  // one 1-D grid holds every tile
        const dim3 lgrid((unsigned)nlong);
        launch(attn_fwd_long, lgrid, FWD_THREADS, LFWD_SMEM, (cudaStream_t)stream, mq, mk, mv, p);
        return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
    }
    if (set_max_dynamic_smem((const void*)attn_fwd, FWD_SMEM) != cudaSuccess) return PSG_E_CUDA;
    const int64_t nshort = (int64_t)grid.x * p.H * p.B;
    if (nshort > 0x7fffffffll) return PSG_E_UNSUPPORTED_LAYOUT;
    launch(attn_fwd, dim3((unsigned)nshort), FWD_THREADS, FWD_SMEM, (cudaStream_t)stream, mq, mk, mv, p);
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

psg_status launch_attention_bwd(const AttnTensor& q, const AttnTensor& k, const AttnTensor& v, const AttnTensor& o,
                                const AttnTensor& dO, const AttnTensor& dq, const AttnTensor& dk,
                                const AttnTensor& dv, const AttnParams& p, void* stream)
{
    if (p.B == 0 || p.T == 0 || p.H == 0) return PSG_OK;
    cudaStream_t s = (cudaStream_t)stream;
    CUtensorMap mq, mk, mv, mdo;
    if (!make_map_attn(&mq, q, p.T, p.H, p.B, QT) || !make_map_attn(&mk, k, p.T, p.H, p.B, QT) ||
        !make_map_attn(&mv, v, p.T, p.H, p.B, QT) || !make_map_attn(&mdo, dO, p.T, p.H, p.B, QT))
        return PSG_E_CUDA;
    if (set_max_dynamic_smem((const void*)attn_bwd, BWD_SMEM) != cudaSuccess) return PSG_E_CUDA;
    const int64_t rows = (int64_t)p.B * p.T * p.H;
    const int dgrid = (int)std::min<int64_t>((rows + 31) / 32, (int64_t)num_sms() * 16);  // 32 rows a block
    launch(attn_delta, dgrid, 256, 0, s, o, dO, p);
    const int64_t tiles = (p.T + QT - 1) / QT;
    if (tiles * p.H * 2 * p.B > 0x7fffffffll) return PSG_E_UNSUPPORTED_LAYOUT;  // one 1-D grid holds every tile
    const dim3 grid((unsigned)(tiles * p.H * 2 * p.B));
    launch(attn_bwd, grid, BWD_THREADS, BWD_SMEM, s, mq, mk, mv, mdo, dq, dk, dv, p);
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

}  // namespace psg
