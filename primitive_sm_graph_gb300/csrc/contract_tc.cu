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
//   warps 2-9 epilogue: two warps per 32 TMEM lanes (rows), each over half
//           of the tile's 256 columns; a warp reads 64 columns with two
//           tcgen05.ld before one wait, rounds to the output dtype once and
//           stores (through a 128B-swizzled staging slot and a TMA store when
//           C's layout allows), while the MMA warp fills the other
//           accumulator.
// The CTA-pair kernel further down keeps these roles over two SMs.
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
#include "jit.h"
#include "launch_util.cuh"
#include "tc_util.cuh"

namespace psg {

namespace {

using namespace tcu;

#include "jit/gemm_body.cuh"

__global__ void __launch_bounds__(THREADS, 1) tc_gemm(const __grid_constant__ CUtensorMap tmap_a,
                                                      const __grid_constant__ CUtensorMap tmap_b,
                                                      const __grid_constant__ CUtensorMap tmap_c,
                                                      const __grid_constant__ TcParams p)
{
    tc_gemm_body<EpiNone>(tmap_a, tmap_b, tmap_c, p);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    tc_gemm2(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
             const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ TcParams p)
{
    tc_gemm2_body<EpiNone>(tmap_a, tmap_b, tmap_c, p);
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

}  // namespace

std::string epi_spec_source(const EpiSpec& e, bool pair)
{
    std::string body = e.prog;
    if (pair)
        body += "extern \"C\" __global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)\n"
                "psg_gemm2_epi(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,\n"
                "              const __grid_constant__ CUtensorMap tc, const __grid_constant__ TcParams p)\n"
                "{\n    tc_gemm2_body<EpiJit<EpiProg>>(ta, tb, tc, p);\n}\n";
    else
        body += "extern \"C\" __global__ void __launch_bounds__(THREADS, 1)\n"
                "psg_gemm_epi(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,\n"
                "             const __grid_constant__ CUtensorMap tc, const __grid_constant__ TcParams p)\n"
                "{\n    tc_gemm_body<EpiJit<EpiProg>>(ta, tb, tc, p);\n}\n";
    return e.tables + '\x01' + body;
}

namespace {

// The kernel specialised for a fused epilogue program (compiled at the first
// call with this program and variant, then cached): the single-CTA body or
// the CTA-pair body with the generated program as its epilogue.
psg_status epi_kernel(const EpiSpec& e, bool pair, cudaKernel_t* k)
{
    return jit_kernel(JIT_GEMM, epi_spec_source(e, pair), pair ? "psg_gemm2_epi" : "psg_gemm_epi", k);
}

// launch of a runtime-compiled contraction kernel with its three tensor maps
psg_status launch_epi(cudaKernel_t k, int grid, int smem, CUtensorMap& ma, CUtensorMap& mb, CUtensorMap& mc,
                      TcParams& p, void* stream)
{
    if (set_max_dynamic_smem((const void*)k, smem) != cudaSuccess) return PSG_E_CUDA;
    void* args[] = {(void*)&ma, (void*)&mb, (void*)&mc, (void*)&p};
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config(dim3(grid), dim3(THREADS), (size_t)smem, (cudaStream_t)stream, attr);
    return cudaLaunchKernelExC(&cfg, (const void*)k, args) == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

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
    cudaKernel_t ek = nullptr;
    if (o.epi) {
        const psg_status st = epi_kernel(*o.epi, true, &ek);
        if (st != PSG_OK) return st;
    } else if (set_max_dynamic_smem((const void*)tc_gemm2, P_SMEM_BYTES) != cudaSuccess) {
        return PSG_E_CUDA;
    }
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
    if (ek) return launch_epi(ek, 2 * clusters, P_SMEM_BYTES, ma, mb, mc, p, stream);
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
    cudaKernel_t ek = nullptr;
    if (o.epi) {
        const psg_status st = epi_kernel(*o.epi, false, &ek);
        if (st != PSG_OK) return st;
    } else if (set_max_dynamic_smem((const void*)tc_gemm, SMEM_BYTES) != cudaSuccess) {
        return PSG_E_CUDA;
    }
    CUtensorMap mc;
    make_out_map(&mc, p);
    const int64_t units = (int64_t)p.num_m * p.num_n * p.batch * p.splits;
    const int grid = (int)std::min<int64_t>(units, num_sms());
    if (ek) return launch_epi(ek, grid, SMEM_BYTES, ma, mb, mc, p, stream);
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
