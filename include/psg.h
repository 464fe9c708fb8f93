/*
 * psg.h -- C ABI of the primitive-op graph hot path on GB300 (sm_103a).
 *
 * The library executes the data-parallel kernels of a lazy graph over a closed
 * set of primitive ops (limn, "The op set": sources, VIEW, NEG EXP LOG SQRT
 * RECIP CAST, ADD MUL CMPLT, WHERE, SUM MAX, GATHER SCATTER) on tensors laid
 * out by a View (limn, "Three rules hold it together": shape, strides, offset,
 * mask).  Five call families:
 *   psg_elementwise   a fused elementwise chain over Views;
 *   psg_reduce_rows   SUM/MAX row reductions with fused prologue/epilogue;
 *   psg_permute       CONTIGUOUS of a permuted View (tiled transpose);
 *   psg_contract      matmul as a broadcast MUL followed by a SUM over k,
 *                     with an optional fused elementwise epilogue;
 *   psg_contract_ws   the same with a split-K workspace (psg_contract_workspace);
 *   psg_gather / psg_scatter_add   the indexed ops along dim 0.
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory: every pointer argument named as device memory must point to memory
 *   the CUDA device can address (cudaMalloc / torch CUDA tensors).  The caller
 *   owns every buffer, workspace and stream; the library never synchronises
 *   and allocates no device memory at run time.  Its one fixed device array
 *   is the key scratch of psg_scatter_add_static, part of the library image.
 * State: psg_elementwise and psg_reduce_rows compile a kernel per distinct
 *   program (NVRTC, on first use) and keep it in a process-wide cache that
 *   only grows, guarded by a mutex; per-device attribute caches likewise.
 *   Nothing else persists between calls.
 * Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  Every
 *   call only enqueues work on it and returns.
 * Errors: host-side validation happens before any launch and returns a
 *   psg_status; nothing is launched when it is not PSG_OK.  Errors found on the
 *   device (a GATHER index out of range, a bounded wait that gave up) are
 *   written as a psg_status code into the caller's `d_status` word (device
 *   memory, zeroed by the caller) and read after a synchronise.  The library
 *   never traps.  An unsupported dtype, layout or program returns its own
 *   code; no call silently runs a different implementation (Tiki, "Compile
 *   model code": unsupported contracts raise a typed error).
 * Empty sizes: a call whose result has no cells (a zero-length dim of the
 *   output, an empty batch, sequence or head axis, no GATHER/SCATTER rows)
 *   returns PSG_OK and writes nothing; its pointers may then be null.  A
 *   reduction over an empty axis gives the fold's identity: SUM 0, MAX -inf
 *   for floats and the dtype's minimum for integers, then the epilogue.  A
 *   contraction over K = 0 writes 0 (the empty SUM) in C's dtype.
 * Thread safety: calls may be made from several host threads at once.
 * Launches: every kernel is launched with programmatic stream serialization
 *   and waits (griddepcontrol.wait) for the kernel before it on the stream
 *   before touching memory, so a launch overlaps only its predecessor's tail;
 *   results are the same bits either way.  Environment: PSG_NO_PDL (any
 *   value, read once) launches without the attribute; PSG_GEMM_KERNEL=single
 *   or =pair picks the bf16/f16 contraction kernel (single CTA or CTA pair)
 *   where both apply.
 */
#ifndef PSG_H
#define PSG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PSG_OK = 0,
    PSG_E_INVALID_ARG = 1,          /* null pointer, bad count, shapes that disagree */
    PSG_E_UNSUPPORTED_DTYPE = 2,    /* dtype combination this call does not implement */
    PSG_E_UNSUPPORTED_LAYOUT = 3,   /* view layout this call does not implement */
    PSG_E_OUT_OF_BOUNDS_VIEW = 4,   /* a reachable element lies outside [0, extent) */
    PSG_E_MISALIGNED = 5,           /* pointer not aligned to its element size */
    PSG_E_INDEX_OUT_OF_RANGE = 6,   /* device-reported: GATHER/SCATTER index outside [0, V) */
    PSG_E_TIMEOUT = 7,              /* device-reported: a bounded wait gave up */
    PSG_E_CUDA = 8,                 /* a CUDA runtime call or launch failed */
    PSG_E_UNSUPPORTED_PROGRAM = 9,  /* program too long / needs too many live values */
    PSG_E_WORKSPACE = 10            /* workspace missing or too small */
} psg_status;

/* The seven dtypes (limn, "The op set", dtype paragraph).  float16/bfloat16
 * are storage widths: kernels widen them to float32 to compute and reductions
 * keep float32 running totals, rounding once at the end. */
typedef enum {
    PSG_F32 = 0, PSG_BF16 = 1, PSG_F16 = 2, PSG_F64 = 3, PSG_I32 = 4, PSG_I16 = 5, PSG_I8 = 6
} psg_dtype;

#define PSG_MAX_DIMS 8

/* A View (limn, "Three rules hold it together"): the element with
 * multi-index (i_0 .. i_{ndim-1}), 0 <= i_d < shape[d], reads
 *     base[offset + sum_d i_d * strides[d]]
 * when mask_lo[d] <= i_d < mask_hi[d] for every d, and reads a zero of the
 * dtype otherwise (a padded read; limn, "Reading the schedule").
 * Units are elements, not bytes.  strides[d] >= 0 (0 = expand/broadcast; a
 * step other than 1 has no View behind it, so there are no negative strides).
 * offset may be negative when masking keeps every reachable read in range.
 * extent = number of elements in the allocation `base` points to; every
 * reachable (unmasked) element must lie in [0, extent), or the call returns
 * PSG_E_OUT_OF_BOUNDS_VIEW.  A View that is written must be injective (no
 * stride-0 dim of size > 1, no overlapping dims) and unmasked.
 * ndim 0 is a scalar (one element). */
typedef struct {
    int32_t ndim;
    int32_t dtype; /* psg_dtype */
    int64_t shape[PSG_MAX_DIMS];
    int64_t strides[PSG_MAX_DIMS];
    int64_t offset;
    int64_t mask_lo[PSG_MAX_DIMS];
    int64_t mask_hi[PSG_MAX_DIMS];
    int64_t extent;
} psg_view;

/* Program nodes.  A program is an array of nodes in topological order; a
 * node's operands name earlier nodes by index; the last node is the result.
 * Every node carries the dtype of its value and rounds to it (the per-node
 * semantics of limn's numpy device).  Operand dtype rules (validated):
 *   NEG EXP LOG SQRT RECIP: operand dtype == node dtype (EXP LOG SQRT RECIP
 *       float only);  ADD MUL CMPLT: both operands have the node dtype; CMPLT
 *       yields 1 or 0 of that dtype (a NaN operand compares false);
 *   WHERE(a=cond, b=x, c=y): cond any dtype, true when nonzero (NaN is
 *       nonzero); x, y have the node dtype;
 *   CAST(a): any dtype -> node dtype (float->float round to nearest even;
 *       float->int truncates toward zero with NaN -> 0 and saturation to the
 *       int32 range, then wraps to the width; int->float converts to float32
 *       and rounds to the width; int->int wraps);
 *   LOAD(a=input index): the node dtype must equal that input's view dtype;
 *   CONST: value cval rounded into the node dtype;
 *   RED(a=stage index): (psg_reduce_rows only) the reduced value of an
 *       earlier stage, in that stage's dtype;
 *   ACC: (psg_contract's epilogue only) the cell's float32 total, the SUM
 *       over k before any rounding into C; node dtype PSG_F32.
 * float64 nodes (PSG_F64, every op above) run in psg_elementwise, each
 * rounded to double; psg_reduce_rows and psg_contract's epilogue refuse them
 * (PSG_E_UNSUPPORTED_DTYPE). */
typedef enum {
    PSG_OP_LOAD = 0, PSG_OP_CONST = 1, PSG_OP_RED = 2,
    PSG_OP_NEG = 3, PSG_OP_EXP = 4, PSG_OP_LOG = 5, PSG_OP_SQRT = 6, PSG_OP_RECIP = 7,
    PSG_OP_CAST = 8, PSG_OP_ADD = 9, PSG_OP_MUL = 10, PSG_OP_CMPLT = 11, PSG_OP_WHERE = 12,
    PSG_OP_ACC = 13
} psg_op;

typedef struct {
    int32_t op;    /* psg_op */
    int32_t a, b, c;
    int32_t dtype; /* psg_dtype of the node's value */
    int32_t reserved;
    double cval;   /* PSG_OP_CONST only */
} psg_node;

#define PSG_MAX_NODES 64
#define PSG_MAX_INPUTS 8

/* ---------------------------------------------------------------------------
 * psg_elementwise -- realise a fused elementwise chain (limn, "Reading the
 * schedule": elementwise work fuses into one kernel; "Backends": one thread
 * per output cell, here 8 cells per thread with 128-bit loads).
 *   out[i] = prog(in_0[i], ..., in_{n_in-1}[i])   for every multi-index i of
 *   out_v's shape.
 * prog/n_nodes: host memory, 1..PSG_MAX_NODES nodes (no PSG_OP_RED).
 * in[k]: device pointers; in_v[k]: host array of n_in (<= PSG_MAX_INPUTS)
 *   views, each with out_v's ndim and shape (broadcasting is a stride-0 dim).
 * out/out_v: device pointer and its view (unmasked, injective); its dtype must
 *   equal the last node's dtype.  `out` must not overlap any input unless the
 *   two views are identical.
 * Returns PSG_OK or a validation error; the kernel itself cannot fail.
 * ------------------------------------------------------------------------- */
psg_status psg_elementwise(const psg_node* prog, int n_nodes, const void* const* in,
                           const psg_view* in_v, int n_in, void* out, const psg_view* out_v,
                           void* stream);

/* ---------------------------------------------------------------------------
 * psg_reduce_rows -- SUM/MAX over the last dim with fused prologue and
 * epilogue (limn, "Reading the schedule": a reduce is a cut and elementwise
 * work fuses into it; "The op set", the dtype paragraph: float32 running
 * totals, rounded once).  One team of threads folds each row; a row is not
 * split across blocks, so very few very long rows use few SMs.
 *
 * Every input view has the iteration shape [R_0 .. R_{d-2}, N]; the last dim
 * is the reduced one.  Stages run in order; stage s computes, for every row r,
 *     red_s[r] = fold_{j=0..N-1} prologue_s(r, j)
 * with SUM (identity 0) or MAX (identity -inf; NaN propagates; +0 wins a tie
 * with -0).  The fold keeps a float32 total for float dtypes (int32 wrapping
 * total for ints) and rounds to the stage dtype (the prologue result dtype)
 * once.  A prologue may read inputs, constants and earlier stages' values
 * (PSG_OP_RED a=s).  After the stages:
 *   - if out_v's last dim is N: out[r, j] = epilogue(r, j) per element
 *     (softmax: two stages, MAX then SUM(EXP(x - m)), epilogue e * RECIP(s));
 *   - if out_v's last dim is 1 (keepdim) or out_v drops it: out[r] =
 *     epilogue(r) evaluated once per row, where the epilogue may read only
 *     constants and stage values; with n_epi == 0 out[r] = red_{last}[r].
 * The sum of N values deviates from the exact sum by at most
 * gamma_{N-1} * sum |x_j| in any association order (Litmus, "ToleranceBound",
 * the reduction_order term), which is the tolerance this call is tested to.
 * stages: host array of n_stages (1..4) stage descriptors, each pointing to a
 *   host program.  epilogue: host program or NULL.
 * d_status: device int32 or NULL.  When contiguous rows are staged through
 *   shared memory by bulk copies, a copy that has not landed after about a
 *   second makes the kernel write PSG_E_TIMEOUT there, stop waiting and
 *   finish (its outputs are then undefined).
 * ------------------------------------------------------------------------- */
typedef enum { PSG_RED_SUM = 0, PSG_RED_MAX = 1 } psg_red_op;

typedef struct {
    int32_t op;             /* psg_red_op */
    int32_t n_nodes;
    const psg_node* prologue;
} psg_reduce_stage;

psg_status psg_reduce_rows(const psg_reduce_stage* stages, int n_stages, const psg_node* epilogue,
                           int n_epi, const void* const* in, const psg_view* in_v, int n_in,
                           void* out, const psg_view* out_v, int32_t* d_status, void* stream);

/* ---------------------------------------------------------------------------
 * psg_permute -- CONTIGUOUS(VIEW(permute(perm)) of in): out[i_0..i_{n-1}] =
 * in[j] with j_{perm[d]} = i_d (limn, "Three rules": permute is a View;
 * "Reading the schedule": a copy is a cut).  A 2-D transpose takes the tiled
 * shared-memory path (Tiki, "What works today": swizzled transpose).
 * perm: host array of in_v->ndim distinct dims.  out_v: shape[d] =
 * in_v->shape[perm[d]], same dtype, unmasked and injective (contiguous is the
 * fast path).  Bit-exact: only bytes move.
 * ------------------------------------------------------------------------- */
psg_status psg_permute(const void* in, const psg_view* in_v, const int32_t* perm, void* out,
                       const psg_view* out_v, void* stream);

/* ---------------------------------------------------------------------------
 * psg_contract -- matmul as MUL of two broadcast Views followed by a SUM over
 * the last dim (limn, "Reading the schedule": a whole matmul is one kernel and
 * the (M,N,1) result aliases the (M,N) sink; Luminal IR blog, "Naive Matrix
 * Multiplication": the broadcast is a stride-0 loop):
 *     C[b.., m, n] = sum_{k ascending in the reference} Av[b.., m, n, k] * Bv[b.., m, n, k]
 * Av, Bv: views of rank 3..6 with shape [batch.., M, N, K]; Av's stride along
 *   N must be 0 and Bv's stride along M must be 0 (A broadcast over n, B over
 *   m), batch strides are free.  Cv: shape [batch.., M, N] (or with a
 *   trailing 1), injective.
 * Masks (padded operands) are allowed on Av and Bv: a masked element is a
 *   zero factor.  A's mask along m and k and B's along n and k zero the
 *   loaded factor (so 0 * inf is NaN, as in the broadcast product); a mask
 *   across the other operand's broadcast axis (A's along n, B's along m) or
 *   along a batch dim writes the cell 0, which is the sum of its zero
 *   products whenever the other operand is finite.  Masked operands take the
 *   FP32-pipe kernel (a masked batch dim: one launch per batch index).
 * dtypes: A and B of one type: PSG_BF16 or PSG_F16 (tensor cores, float32
 *   accumulate in TMEM, exact products) or PSG_F32 (K >= 256 and 16-byte
 *   aligned operands: tensor cores as 3xTF32, hi*hi + hi*lo + lo*hi with a
 *   few 2^-20 relative error per product; otherwise float32 FMA on the FP32
 *   pipes); C PSG_F32, PSG_BF16 or PSG_F16 (rounded once, RNE).  PSG_F64
 *   operands sum in float64 in k order into a PSG_F64 C.  PSG_I32 / PSG_I16 /
 *   PSG_I8 operands sum in uint32 with wraparound into an integer C of any
 *   of those widths (stored modulo 2^width: the ints wrap).  Operands the
 *   tensor cores cannot address (strides not 16-byte multiples, several
 *   batch dims that do not merge) take the FP32-pipe kernel.  Any other
 *   dtype pairing returns PSG_E_UNSUPPORTED_DTYPE.
 * The total deviates from the sequential float32 loop by at most
 * 2 * gamma_{K-1} * sum_k |a_k b_k| (Litmus, "ToleranceBound"); for the
 * 3xTF32 path that bound absorbs the product error at the K it is used at.
 * epilogue: NULL (or n_nodes == 0) stores each total rounded once into C.
 *   Otherwise every cell of C is the epilogue program's value at that cell
 *   (limn, "Reading the schedule": elementwise work fuses into the kernel
 *   that produces its operand, so a residual add, a ReLU or a cast after the
 *   contraction costs no trip through memory):
 *       C[b.., m, n] = prog(ACC = the cell's float32 total,
 *                           LOAD k = epilogue->in[k] read through in_v[k] at (b.., m, n))
 *   Each node rounds into its own dtype as in psg_elementwise; the last
 *   node's dtype must be C's.  The epilogue runs in the bf16 / f16 tensor-
 *   core kernel only (A and B bf16 or f16, TMA-addressable, batch dims that
 *   merge for every operand): any other contraction with an epilogue
 *   returns PSG_E_UNSUPPORTED_LAYOUT, as does a masked epilogue input.
 *   The first call with a new program compiles its kernel (NVRTC, cached
 *   for the process, as psg_elementwise does).  C may be an epilogue input
 *   only through an identical View (an in-place update).
 * d_status: device int32 or NULL; receives PSG_E_TIMEOUT if a pipeline wait in
 *   the tensor-core kernel gave up (the output is then invalid).
 * ------------------------------------------------------------------------- */
typedef struct {
    const psg_node* prog;      /* host program, 1..PSG_MAX_NODES nodes (ACC, LOAD, CONST and elementwise ops) */
    int32_t n_nodes;
    int32_t n_in;              /* 0..PSG_MAX_INPUTS */
    const void* const* in;     /* host array of n_in device pointers */
    const psg_view* in_v;      /* host array of n_in views, each of C's shape, unmasked */
} psg_epilogue;

psg_status psg_contract(const void* A, const psg_view* Av, const void* B, const psg_view* Bv,
                        void* C, const psg_view* Cv, const psg_epilogue* epilogue, int32_t* d_status,
                        void* stream);

/* ---------------------------------------------------------------------------
 * psg_contract_workspace / psg_contract_ws -- psg_contract with a caller
 * workspace that lets the bf16 / f16 tensor-core kernel split K when the
 * output has too few 128x256 tiles to occupy the GPU (a weight gradient:
 * small M x N, long K).  Each split sums its own range of K blocks into a
 * float32 partial; a second launch adds the partials in split order and
 * rounds once into C.  The result is deterministic (the split count depends
 * only on the shapes and the GPU's SM count) and within psg_contract's bound:
 * it is still a float32 sum of the same K exact products.
 * psg_contract_workspace: bytes of device workspace psg_contract_ws would use
 *   for these views (0 when it would not split; also 0 for invalid views).
 * psg_contract_ws: as psg_contract; workspace: device memory, 16-byte aligned,
 *   owned by the caller, not read before it is written, free again once the
 *   stream passes the call.  NULL or fewer than the queried bytes runs the
 *   unsplit kernel, and so does a call with an epilogue program.
 * ------------------------------------------------------------------------- */
size_t psg_contract_workspace(const psg_view* Av, const psg_view* Bv, const psg_view* Cv);
psg_status psg_contract_ws(const void* A, const psg_view* Av, const void* B, const psg_view* Bv,
                           void* C, const psg_view* Cv, const psg_epilogue* epilogue, void* workspace,
                           size_t ws_bytes, int32_t* d_status, void* stream);

/* ---------------------------------------------------------------------------
 * psg_gather -- GATHER along dim 0 (limn, "The op set"; nn.Embedding is the
 * use, "nn, optim and checkpoints"):  out[n, ...] = src[idx[n], ...].
 * sv: view of src with shape [V, ...]; idx: device int32[n]; ov: view of out
 * with shape [n, ...] (unmasked, injective), same dtype.  An index outside
 * [0, V) zero-fills its row and writes PSG_E_INDEX_OUT_OF_RANGE to d_status
 * (device int32, required).
 * ------------------------------------------------------------------------- */
psg_status psg_gather(const void* src, const psg_view* sv, const int32_t* idx, int64_t n, void* out,
                      const psg_view* ov, int32_t* d_status, void* stream);

/* ---------------------------------------------------------------------------
 * psg_scatter_add -- SCATTER-add along dim 0 (limn, "The op set"; "Backends":
 * a scatter's colliding adds stay in order), deterministic:
 *     for n = 0, 1, .. n-1 in order:  dst[idx[n], ...] += upd[n, ...]
 * Float destinations keep a float32 running total per cell, starting from the
 * cell's value, and round into the dtype once; ints wrap.  Colliding rows are
 * added in ascending n, so two runs give the same bits (no float atomics).
 * dv: view of dst [V, ...] (contiguous rows); uv: view of upd [n, ...]; both
 * one dtype, any of the seven (f64 keeps a float64 total; i32, i16 and i8
 * add in 32-bit wrapping arithmetic and keep the low bits, which is the
 * wrap of the width).  An index outside [0, V) skips its row and
 * writes PSG_E_INDEX_OUT_OF_RANGE to d_status (device int32, required).
 * workspace: device memory of at least psg_scatter_workspace(n) bytes,
 *   256-byte aligned, owned by the caller, free for reuse once the stream has
 *   passed this call.
 * ------------------------------------------------------------------------- */
size_t psg_scatter_workspace(int64_t n);
psg_status psg_scatter_add(void* dst, const psg_view* dv, const int32_t* idx, int64_t n,
                           const void* upd, const psg_view* uv, void* workspace, size_t ws_bytes,
                           int32_t* d_status, void* stream);

/* ---------------------------------------------------------------------------
 * psg_scatter_add_static -- the same deterministic SCATTER-add as
 * psg_scatter_add, for callers that cannot allocate device memory: code that
 * runs after a memory pool has reserved the whole GPU and hands out no more,
 * or paths that must not allocate at all (a step being recorded for replay,
 * a loop with a fixed memory budget).  It takes no workspace; its scratch
 * (the sort keys) is one fixed array inside this library's device image, of
 * PSG_SCATTER_STATIC_MAX_N 64-bit keys (8 MiB), which every GPU that loads
 * the library holds until the process exits.  The pages have no counterpart
 * to this call.
 *   - n must be <= PSG_SCATTER_STATIC_MAX_N, else PSG_E_WORKSPACE and nothing
 *     is launched; the other arguments and errors are those of
 *     psg_scatter_add.
 *   - It calls no device allocator of any kind.  The first call on a device
 *     looks up the array's device address once (with that device current)
 *     and caches it; make that first call before any stream capture.
 *   - Every call shares the one array and leaves its keys there; each call
 *     rewrites every key it reads, so nothing needs clearing between calls.
 *     Two calls that run on the GPU at the same time (different streams
 *     without ordering between them) race on the array and give wrong sums:
 *     order them on one stream.
 * ------------------------------------------------------------------------- */
#define PSG_SCATTER_STATIC_MAX_N (1 << 20)
psg_status psg_scatter_add_static(void* dst, const psg_view* dv, const int32_t* idx, int64_t n,
                                  const void* upd, const psg_view* uv, int32_t* d_status,
                                  void* stream);

/* ---------------------------------------------------------------------------
 * psg_attention_fwd / psg_attention_bwd -- fused scaled dot-product attention
 * (limn, "The op set": the fused attention op that saves L = logsumexp for
 * its backward and a two-pass deterministic backward, in place of the
 * composed T x T score tensors; masking is a flag per key that composes with
 * causal; Tiki, "Write the attention kernel at the algorithm level": the
 * running max, denominator and weighted sum, and the FlashAttention backward
 * dS = P * (dO V^T - D)).
 *
 * Per batch b and head h, with S = scale * Q K^T and key j visible to query
 * i unless j > i (causal) or key_mask[b, j] == 0:
 *     L[b,h,i] = log sum_{visible j} exp(S[i,j]),  O = exp(S - L) V over the
 *     visible keys (a query with no visible key: O = 0, L = -inf);
 *     D[i] = sum_d dO[i,d] O[i,d],  P = exp(S - L) (0 where hidden),
 *     dS = P * (dO V^T - D),  dV = P^T dO,  dQ = scale * dS K,
 *     dK = scale * dS^T Q.
 * Views: Q, K, V, O, dO, dQ, dK, dV are bf16 [B, T, H, 64] (head dim
 * contiguous; batch, token and head strides multiples of 8 elements; base
 * 16-byte aligned; no mask).  B <= 32767, H <= 65535, T <= 2^24; other
 * shapes return PSG_E_UNSUPPORTED_LAYOUT.  T <= 256 keys take one key block
 * per head; longer sequences walk 128-key blocks with a running max and sum.
 * key_mask: device bytes [B, T] (row-major; nonzero = visible) or NULL (every
 * key visible).  S and dP are float32 sums of exact bf16 products; P and dS
 * are rounded to bf16 before the second products.  lse: device float32
 * [B, H, T], written by fwd and read by bwd.  delta: device float32 [B, H, T]
 * scratch of bwd (caller-owned).  scale > 0.  A bounded wait that gives up
 * writes PSG_E_TIMEOUT into d_status.
 * ------------------------------------------------------------------------- */
psg_status psg_attention_fwd(const void* q, const psg_view* qv, const void* k, const psg_view* kv,
                             const void* v, const psg_view* vv, void* o, const psg_view* ov, float* lse,
                             float scale, int causal, const uint8_t* key_mask, int32_t* d_status, void* stream);
psg_status psg_attention_bwd(const void* q, const psg_view* qv, const void* k, const psg_view* kv,
                             const void* v, const psg_view* vv, const void* o, const psg_view* ov,
                             const void* dout, const psg_view* dov, const float* lse, float* delta,
                             void* dq, const psg_view* dqv, void* dk, const psg_view* dkv, void* dv,
                             const psg_view* dvv, float scale, int causal, const uint8_t* key_mask,
                             int32_t* d_status, void* stream);

/* ---------------------------------------------------------------------------
 * psg_adamw_step -- one AdamW step (decoupled weight decay) over a list of
 * tensors in one launch (limn, "nn, optim and checkpoints": optimizer steps
 * as ASSIGN graphs over the parameters, beta**t kept on the device).
 * Per element, in float32, each operation rounded in this order:
 *     p1 = p * (1 - lr*wd);  m' = b1*m + (1-b1)*g;  v' = b2*v + (1-b2)*(g*g)
 *     p' = p1 - (lr / (1 - b1^t)) * (m' / (sqrt(v') / sqrt(1 - b2^t) + eps))
 * where b^t are the running products after this step; p' rounds once into
 * the parameter dtype (RNE).  tensors: host array of n_tensors entries; p
 * and g (device) share `dtype` (PSG_F32, PSG_BF16 or PSG_F16); m and v are
 * float32 device arrays of numel elements, updated in place.  d_beta_pow:
 * device float32 [2] = {b1^t, b2^t} before the step ({1, 1} at the start);
 * the call advances it.  Tensors are processed 32 per launch, then one
 * single-thread launch advances d_beta_pow.
 * ------------------------------------------------------------------------- */
typedef struct {
    void* p;            /* parameters (dtype), updated in place */
    const void* g;      /* gradients (dtype) */
    float* m;           /* first moment, float32 */
    float* v;           /* second moment, float32 */
    int64_t numel;
} psg_adamw_tensor;

psg_status psg_adamw_step(const psg_adamw_tensor* tensors, int n_tensors, int dtype, float lr, float beta1,
                          float beta2, float eps, float weight_decay, float* d_beta_pow, int32_t* d_status,
                          void* stream);

/* ---------------------------------------------------------------------------
 * psg_query_launch -- the launch a call would make, before making it (Tiki,
 * "The architecture we want": register and shared-memory budgets visible
 * before launch).  call: one of psg_call; v: the output view the call would
 * write (for PSG_CALL_CONTRACT: Cv).  Writes grid (blocks), block (threads),
 * dynamic shared memory bytes and registers per thread of the kernel chosen.
 * A float32 contraction runs on the tensor cores as 3xTF32 when K >= 256
 * and both operands are TMA-addressable (PSG_CALL_CONTRACT_F32_TENSOR),
 * else on the FP32 pipes (PSG_CALL_CONTRACT_F32).
 * ------------------------------------------------------------------------- */
typedef enum {
    PSG_CALL_ELEMENTWISE = 0, PSG_CALL_REDUCE_ROWS = 1, PSG_CALL_PERMUTE = 2,
    PSG_CALL_CONTRACT_BF16 = 3, PSG_CALL_CONTRACT_F32 = 4, PSG_CALL_GATHER = 5,
    PSG_CALL_SCATTER_ADD = 6, PSG_CALL_CONTRACT_F32_TENSOR = 7
} psg_call;

psg_status psg_query_launch(int call, const psg_view* v, int* grid, int* block, int* smem,
                            int* regs);

/* Human-readable name of a status code (static storage). */
const char* psg_status_string(int status);

/* Library version string (static storage). */
const char* psg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PSG_H */
