/*
 * pgg.h -- C ABI of the GB300 (sm_103a) fused MoE permute + grouped-matmul
 * backward, input gradient only.
 *
 * Operation (page "MoeInitRoutingGroupedMatmulGrad design", section
 * "数学定义和公式", element-wise gradient formula):
 *
 *     d_x[b, k] = sum_{i : batch(i) = b} sum_n gradY[i, n] * weight[g(i), k, n]
 *
 *   gradY  [M, N]     upstream gradient d_y in expanded (expert-sorted) order,
 *                     M = batch * topK                       (section "输入输出")
 *   weight [G, K, N]  expert weights, same dtype as gradY     (section "输入输出")
 *   g(i)              expert whose block of rows holds row i; block g has
 *                     groupList[g] rows (counts, not a cumulative sum; a count
 *                     of 0 is an empty expert)         (sections "输入输出", "约束")
 *   batch(i)          original_pos(i) / topK, original_pos = b * topK + j
 *                     (section "数学定义和公式", Step 2)
 *   expandedRowIdx    int64 [L], L == M. rowIdxType 0 (gather form): entry i is
 *                     the original position of expanded row i. rowIdxType 1
 *                     (scatter form): entry p is the expanded row of original
 *                     position p                 (section "输入输出", note 1)
 *   out               FP32 [batch, K], always FP32 whatever the input dtype
 *                     (section "输入输出", note 2; section 2.6.2)
 *
 * The [M, K] intermediate d_y @ weight^T is never materialised (section 1.1).
 * The result is bitwise identical from run to run: the topK contributions to
 * each out element are added in increasing expanded-row order (section 2.4.1
 * asks for deterministic computation).
 *
 * Conventions shared by every call below:
 *   - All tensors are dense and row-major. Device pointers are addresses in the
 *     current CUDA device's memory; the caller owns every buffer and keeps it
 *     alive until the work on `stream` has finished. The library allocates no
 *     memory and keeps no state between calls except per-device cached device
 *     attributes and the test hooks at the end of this file.
 *   - Calls only enqueue work on `stream` (NULL = legacy default stream) and
 *     never synchronise. Inputs are not modified.
 *   - Every kernel except the one that resets the workspace header (the first
 *     of a routing or index-validation stage) is launched with programmatic
 *     stream serialization: its CTAs may be scheduled while the previous
 *     kernel in the stream (the library's own, or the caller's) drains, and it
 *     waits for that kernel's completion before it reads any memory, so stream
 *     order is kept exactly.
 *   - Host-detected errors are returned synchronously and nothing is enqueued.
 *   - Device-detected errors (bad index, groupList sum, not a permutation,
 *     a wait that ran out) are written to the status word, the first uint32 of
 *     the workspace: 0 means success, otherwise one of PGG_ERR_INDEX ..
 *     PGG_ERR_TIMEOUT. Read it after the stream has finished. When routing
 *     validation fails, `out` is zero-filled instead of computed.
 *   - Alignment: gradY and weight must be aligned to their element size,
 *     out to 4 bytes, expandedRowIdx and groupList to 8 bytes, and the
 *     workspace to 256 bytes; otherwise PGG_ERR_ALIGN. Any N and K are
 *     accepted. When N * sizeof(dtype) is a multiple of 16 bytes and gradY
 *     and weight are 16-byte aligned, the grouped GEMM runs on the tensor
 *     cores with its operands streamed by the tensor-memory-access unit,
 *     which needs both. Otherwise, for 16-bit dtypes with an even N and
 *     gradY and weight 4-byte aligned, it still runs on the tensor cores,
 *     with the operands copied 4 bytes at a time by gather warps (plan
 *     variant 5; same tiles, same bits as variant 0 where both apply). In
 *     every other case (fp32 rows that are not a multiple of 16 bytes, odd
 *     N, 2-byte aligned pointers) it runs on the FP32 pipes (plan variant
 *     3), with the same ordered scatter-add and the same determinism. For
 *     the same call the tensor-core and FP32-pipe paths may differ in the
 *     last bits of the GEMM sums, never from run to run.
 */
#ifndef PGG_H
#define PGG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* pgg_stream_t;

/* Input dtype of gradY and weight (section "输入输出": FLOAT / FLOAT16 / BF16). */
typedef enum { PGG_F32 = 0, PGG_F16 = 1, PGG_BF16 = 2 } pgg_dtype;

typedef enum {
  PGG_OK = 0,
  PGG_ERR_NULL = 1,      /* a required pointer is NULL */
  PGG_ERR_SHAPE = 2,     /* sizes violate the constraint table (L != M, M != batch*topK, ...) */
  PGG_ERR_ATTR = 3,      /* topK <= 0, batch <= 0, or rowIdxType not in {0, 1} */
  PGG_ERR_DTYPE = 4,     /* dtype not in pgg_dtype */
  PGG_ERR_WORKSPACE = 5, /* workspace smaller than pgg_dx_workspace_size reports */
  PGG_ERR_CUDA = 6,      /* a CUDA runtime/driver call failed (launch, tensor map, device query) */
  PGG_ERR_ALIGN = 7,     /* pointer or row-stride alignment, see above */
  /* device-detected, written to the status word: */
  PGG_ERR_INDEX = 16,    /* an expandedRowIdx entry outside [0, M) */
  PGG_ERR_GROUPSUM = 17, /* a negative groupList entry, or sum(groupList) != M */
  PGG_ERR_NOT_PERM = 18, /* expandedRowIdx is not a permutation of [0, M) */
  PGG_ERR_TIMEOUT = 19,  /* a bounded wait inside a kernel ran out (no hang; result invalid) */
  PGG_ERR_CHECK = 20     /* checked build only (libpgg_checks.so, compiled with -DPGG_CHECKS):
                            a device bounds check on an index read from the routing tables
                            failed; the access was kept in bounds, the result is invalid */
} pgg_status;

/*
 * Workspace bytes pgg_dx_execute needs for these sizes (the two-phase
 * get-workspace-size / execute convention of section 2.2.2). Pure host code:
 * no CUDA call. Arguments as for pgg_dx_execute; L is the length of
 * expandedRowIdx. The figure grows as 12*M + 4*batch*ceil(K/128) bytes plus a
 * few KB; it is independent of N and never holds an [M, K] array.
 * Returns PGG_OK and writes *workspace_bytes, or a host error code.
 */
int pgg_dx_workspace_size(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L,
                          int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                          size_t* workspace_bytes);

/*
 * Computes out[batch, K] (FP32, fully overwritten) from gradY, weight,
 * expandedRowIdx and groupList as defined at the top of this file.
 *
 *   gradY          device, [M, N] of `dtype`
 *   weight         device, [G, K, N] of `dtype`
 *   expandedRowIdx device, int64 [L], L == M, form selected by rowIdxType
 *   groupList      device, int64 [G], per-expert row counts (sum must be M)
 *   M, N, K, G     sizes; M == batch * topK, all >= 1, M < 2^31
 *   batch, topK    attributes (section "约束": both > 0)
 *   rowIdxType     0 gather form, 1 scatter form
 *   workspace      device scratch of at least pgg_dx_workspace_size bytes,
 *                  256-byte aligned, contents on entry irrelevant; holds the
 *                  status word at offset 0 after the call
 *   out            device, FP32 [batch, K]
 *   stream         CUDA stream the work is enqueued on
 *
 * Equivalent to pgg_dx_route_prep followed by pgg_dx_grouped_gemm on the same
 * workspace and stream.
 */
int pgg_dx_execute(const void* gradY, const void* weight, const int64_t* expandedRowIdx,
                   const int64_t* groupList, int64_t M, int64_t N, int64_t K, int64_t G,
                   int64_t L, int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                   void* workspace, size_t workspace_bytes, float* out, pgg_stream_t stream);

/*
 * First stage of pgg_dx_execute, exposed so that each stage can be timed on
 * its own: validates the routing on the device (writing the status word),
 * builds the per-expert row offsets (exclusive scan of groupList), the list
 * of row blocks that skips empty experts, the inverse of expandedRowIdx and,
 * per expanded row, its token and its rank among that token's rows; resets
 * the scatter-add tickets. Same arguments and errors as pgg_dx_execute,
 * without the value tensors and `out`.
 */
int pgg_dx_route_prep(const int64_t* expandedRowIdx, const int64_t* groupList, int64_t M,
                      int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch, int64_t topK,
                      int rowIdxType, pgg_dtype dtype, void* workspace, size_t workspace_bytes,
                      pgg_stream_t stream);

/*
 * Second stage of pgg_dx_execute: the persistent grouped-GEMM kernel with the
 * fused, ordered scatter-add into out. Requires a pgg_dx_route_prep with the
 * same sizes, routing and workspace earlier on the same stream (or otherwise
 * ordered before it). If the status word is non-zero on entry the kernel
 * zero-fills out and returns. Same arguments and errors as pgg_dx_execute.
 */
int pgg_dx_grouped_gemm(const void* gradY, const void* weight, const int64_t* expandedRowIdx,
                        const int64_t* groupList, int64_t M, int64_t N, int64_t K, int64_t G,
                        int64_t L, int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                        void* workspace, size_t workspace_bytes, float* out,
                        pgg_stream_t stream);

/* How pgg_dx_execute will run a problem of these sizes (host only, no CUDA call). */
typedef struct {
  int32_t variant;          /* 0 = wide row blocks on CTA pairs (tensor-bound), 1 = narrow row
                               blocks (weight streaming), 2 = wide row blocks on single CTAs,
                               3 = FP32-pipe kernel (rows of N * sizeof(dtype) bytes that are
                               not a multiple of 16), 4 = owner kernel (each CTA pair owns a
                               block of d_x: few experts per token, 16-bit dtypes; falls back
                               to variant 0 when an expert's rows are not in increasing original
                               position), 5 = variant 0 with its operands copied by gather
                               warps (16-bit rows of an even length that is not a multiple of
                               8 elements); pgg_dx_execute also takes variant 5 (4-byte aligned,
                               16-bit, even N) or else 3 when gradY or weight is not 16-byte
                               aligned */
  int32_t rows_per_block;   /* expanded rows per tile: the MMA N extent (variant 4: tokens per
                               slab) */
  int32_t k_per_block;      /* output columns per CTA and tile (128; a CTA pair covers 256) */
  int32_t stages;           /* shared-memory pipeline depth */
  int32_t k_blocks;         /* ceil(K / k_per_block) */
  int32_t band_k_blocks;    /* k-blocks per band of the tile order */
  int64_t max_row_blocks;   /* upper bound on row blocks: ceil(M/rows_per_block) + G */
  size_t workspace_bytes;   /* as pgg_dx_workspace_size */
  int32_t threads;          /* threads per CTA of the grouped-GEMM kernel */
  int32_t smem_bytes;       /* dynamic shared memory per CTA */
  int32_t cta_pair;         /* 1: clusters of two CTAs share each tile (tcgen05 cta_group::2) */
} pgg_plan_info;

int pgg_dx_plan(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch,
                int64_t topK, int rowIdxType, pgg_dtype dtype, pgg_plan_info* info);

/* Human-readable name of a pgg_status code (static string). */
const char* pgg_status_string(int status);

/*
 * Test hooks (process-wide; not needed in normal use).
 * pgg_debug_set_wait_limit_ns: time limit of every bounded wait inside the
 *   kernels (default 2e9 ns). 0 restores the default.
 * pgg_debug_set_ticket_bias: added to the ticket count each ordered
 *   scatter-add waits for; a positive bias makes every wait of a row with
 *   rank > 0 run out, which exercises the PGG_ERR_TIMEOUT path. 0 = off.
 * pgg_debug_force_variant: -1 = automatic (default), 0 .. 5 = force the
 *   variant reported by pgg_dx_plan (2, 4 and 5 exist for the 16-bit dtypes
 *   only, 5 for an even N only; rows that are not a multiple of 16 bytes
 *   take variant 5 when they can, else 3).
 * pgg_debug_set_band_k_blocks: k-blocks per band of the tile order (0 =
 *   automatic). The result does not depend on it, bit for bit: only the time
 *   order of the tiles changes, never the order of the additions.
 * pgg_debug_set_hold_release: non-zero makes the epilogue of the owner d_x
 *   variant, of the forward and of the weight-gradient kernels withhold its
 *   first release of an accumulator, so that the MMA thread's bounded wait
 *   for it runs out: exercises PGG_ERR_TIMEOUT in those kernels (every CTA
 *   role gives up, drains its copies and MMAs and frees tensor memory). A CTA
 *   pair with fewer than three tiles never waits for that release. 0 = off.
 */
void pgg_debug_set_wait_limit_ns(uint64_t ns);
void pgg_debug_set_ticket_bias(uint32_t bias);
void pgg_debug_force_variant(int variant);
void pgg_debug_set_band_k_blocks(int k_blocks);
void pgg_debug_set_hold_release(int hold);

/*
 * pgg_dx_execute for callers that cannot allocate device memory. (The pages
 * have no counterpart of this call; it is a service of this library.)
 *
 * Who needs it: code that has no allocator at hand when the gradient is due
 * -- a plugin inside a framework that owns all device memory, a serving or
 * real-time runtime that reserved HBM up front and forbids cudaMalloc later,
 * plain C code without an allocator handle. Such a caller passes the same
 * inputs and `out` as to pgg_dx_execute, but no workspace: the call uses a
 * fixed 8 MiB scratch array that the library's CUDA module reserves on every
 * device that loads the library, held until the process exits. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 *   status  optional device pointer (may be NULL); after the work on `stream`
 *           has finished it holds the device-detected status word that
 *           pgg_dx_execute would have left at the start of its workspace.
 *
 * Returns PGG_ERR_WORKSPACE when pgg_dx_workspace_size for these sizes exceeds
 * 8 MiB (8388608 bytes; e.g. M = 108000, K = 7168 needs 4.3 MB), and
 * otherwise what pgg_dx_execute returns.
 *
 * Each call looks up the scratch array's device address (cudaGetSymbolAddress)
 * on the current device, so the address stays valid after cudaDeviceReset;
 * only a call made while `stream` is being captured reuses the address that
 * the previous call on the device looked up, so make the first call on a
 * device before any stream capture on it. Every call on a device shares the one
 * array, and each call re-initialises what it needs, so leftover contents from
 * the previous call do no harm -- but two calls whose work overlaps on the GPU
 * (for example on two streams without ordering between them) race on the
 * array and give wrong results. Order such calls on one stream.
 */
int pgg_dx_execute_static_scratch(const void* gradY, const void* weight,
                                  const int64_t* expandedRowIdx, const int64_t* groupList,
                                  int64_t M, int64_t N, int64_t K, int64_t G, int64_t L,
                                  int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                                  float* out, uint32_t* status, pgg_stream_t stream);

/*
 * ---------------------------------------------------------------------------
 * Weight gradient (the companion operator; page "MoeInitRoutingGroupedMatmulGrad
 * design", section 1.2 "为何不计算 d_weight", item 3: a separate grouped matmul
 * expanded_x^T @ d_y per expert; section 1.1: the forward's MoeInitRouting
 * lays out the token rows by expert, expanded_x[i] = x[batch(i)]):
 *
 *     dweight[g, k, n] = sum_{expanded rows i of expert g} x[batch(i), k] * gradY[i, n]
 *
 *   x              device, [batch, K] of `dtype`: the forward input in original
 *                  token order. expanded_x is never materialised: its rows are
 *                  gathered from x by token. (A caller that kept expanded_x
 *                  [M, K] instead passes it as x with batch = M, topK = 1 and
 *                  expandedRowIdx = 0 .. M-1, groupList unchanged.)
 *   gradY          device, [M, N] of `dtype`, expanded order
 *   expandedRowIdx, groupList, M, N, K, G, L, batch, topK, rowIdxType, dtype:
 *                  as for pgg_dx_execute
 *   out_dtype      dtype of dweight: `dtype` (the page sizes d_weight in the
 *                  input precision) or PGG_F32; else PGG_ERR_DTYPE. Accumulation
 *                  is always FP32; a 16-bit output is rounded to nearest even.
 *   workspace      at least pgg_dw_workspace_size bytes, 256-byte aligned;
 *                  status word at offset 0 as for pgg_dx_execute
 *   dweight        device, [G, K, N] of out_dtype, fully overwritten; an expert
 *                  with no rows gets zeros; zero-filled when the routing
 *                  validation fails
 *
 * Each element is produced by one tile with a fixed order of additions (the
 * expert's rows in increasing order, in MMA blocks of 16), so the result is
 * bitwise repeatable. Runs on the tensor cores when dtype is 16-bit, K and N
 * are multiples of 8 and x, gradY, dweight are 16-byte aligned (variant 0);
 * also on the tensor cores, with the gradY rows copied 4 bytes at a time by
 * the gather warps and dweight written with 4-byte stores, when N is even but
 * not a multiple of 8 (or gradY / dweight are only 4-byte aligned) while K is
 * a multiple of 8 and x is 16-byte aligned (variant 5); otherwise on the FP32
 * pipes (variant 3, also forced by pgg_debug_force_variant(3)). Alignment: x
 * and gradY aligned to their element size, dweight to its element size.
 */
int pgg_dw_workspace_size(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L,
                          int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                          size_t* workspace_bytes);

int pgg_dw_execute(const void* x, const void* gradY, const int64_t* expandedRowIdx,
                   const int64_t* groupList, int64_t M, int64_t N, int64_t K, int64_t G,
                   int64_t L, int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                   pgg_dtype out_dtype, void* workspace, size_t workspace_bytes, void* dweight,
                   pgg_stream_t stream);

/*
 * Second stage of pgg_dw_execute, exposed so that the kernel can be timed on
 * its own: the weight-gradient kernel alone, on a workspace prepared by
 * pgg_dx_route_prep with the same sizes and routing (the routing step is the
 * same for both gradients). Same arguments and errors as pgg_dw_execute.
 */
int pgg_dw_grouped_gemm(const void* x, const void* gradY, const int64_t* expandedRowIdx,
                        const int64_t* groupList, int64_t M, int64_t N, int64_t K, int64_t G,
                        int64_t L, int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                        pgg_dtype out_dtype, void* workspace, size_t workspace_bytes,
                        void* dweight, pgg_stream_t stream);

/*
 * How pgg_dw_execute runs these sizes with 16-byte aligned pointers: variant 0
 * (tensor cores: k_per_block = 128 output rows, 256 output columns, 64
 * reduction rows per stage), 5 (the same with the gradY rows gathered by
 * warps: N even, not a multiple of 8) or 3 (FP32 pipes: 64 rows, 128
 * columns, 32 rows per step); k_blocks and band_k_blocks hold the k and n
 * blocks per expert.
 */
int pgg_dw_plan(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch,
                int64_t topK, int rowIdxType, pgg_dtype dtype, pgg_plan_info* info);

/*
 * ---------------------------------------------------------------------------
 * Forward (the operation these are the gradients of; page
 * "MoeInitRoutingGroupedMatmulGrad design", sections 1.1 and 1.2, forward
 * chain: MoeInitRouting(x) -> expanded_x, GroupedMatmul(expanded_x, weight)
 * -> y):
 *
 *     y[i, n] = sum_k x[batch(i), k] * weight[g(i), k, n]      (i in expanded order)
 *
 *   x              device, [batch, K] of `dtype`, original token order; the rows
 *                  of expanded_x are gathered from it by the routing, never
 *                  materialised
 *   weight         device, [G, K, N] of `dtype`
 *   expandedRowIdx, groupList, M, N, K, G, L, batch, topK, rowIdxType, dtype:
 *                  as for pgg_dx_execute
 *   out_dtype      dtype of y: `dtype` or PGG_F32 (else PGG_ERR_DTYPE); FP32
 *                  accumulation, one round-to-nearest-even for 16-bit outputs
 *   workspace      at least pgg_fwd_workspace_size bytes, 256-byte aligned;
 *                  status word at offset 0 as for pgg_dx_execute
 *   y              device, [M, N] of out_dtype, expanded order, fully
 *                  overwritten; zero-filled when the routing validation fails
 *
 * Each element is one dot product over k in a fixed order: bitwise
 * repeatable. Tensor cores when dtype is 16-bit, K and N are multiples of 8
 * and x, weight, y are 16-byte aligned (variant 0); also on the tensor cores,
 * with the weight rows copied 4 bytes at a time by the gather warps and y
 * written with 4-byte stores, when N is even but not a multiple of 8 (or
 * weight / y are only 4-byte aligned) while K is a multiple of 8 and x is
 * 16-byte aligned (variant 5); otherwise the FP32 pipes (variant 3, also forced
 * by pgg_debug_force_variant(3)). x and weight aligned to their element size,
 * y to its element size.
 */
int pgg_fwd_workspace_size(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L,
                           int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                           size_t* workspace_bytes);

int pgg_fwd_execute(const void* x, const void* weight, const int64_t* expandedRowIdx,
                    const int64_t* groupList, int64_t M, int64_t N, int64_t K, int64_t G,
                    int64_t L, int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                    pgg_dtype out_dtype, void* workspace, size_t workspace_bytes, void* y,
                    pgg_stream_t stream);

/*
 * The two stages of pgg_fwd_execute, exposed so that each can be timed on its
 * own: the routing step (validation, expert offsets, row blocks of up to 256
 * rows, tokens) and the forward kernel on the workspace it prepared. Same
 * arguments and errors as pgg_fwd_execute (the routing step without the value
 * tensors and y).
 */
int pgg_fwd_route_prep(const int64_t* expandedRowIdx, const int64_t* groupList, int64_t M,
                       int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch, int64_t topK,
                       int rowIdxType, pgg_dtype dtype, void* workspace, size_t workspace_bytes,
                       pgg_stream_t stream);

int pgg_fwd_grouped_gemm(const void* x, const void* weight, const int64_t* expandedRowIdx,
                         const int64_t* groupList, int64_t M, int64_t N, int64_t K, int64_t G,
                         int64_t L, int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                         pgg_dtype out_dtype, void* workspace, size_t workspace_bytes, void* y,
                         pgg_stream_t stream);

/*
 * How pgg_fwd_execute runs these sizes with 16-byte aligned pointers: variant
 * 0 (tensor cores on CTA pairs: row blocks of rows_per_block = 256 expanded
 * rows x 256 n, k_per_block = 64 per stage), 5 (the same with the weight rows
 * gathered by warps: N even, not a multiple of 8) or 3 (FP32 pipes: 64 rows x
 * 128 n, 32 k per step; also when x holds 64 GiB or more, batch * K / 8 >=
 * 2^32 - 1, since the tensor-core kernel addresses x rows with 32-bit offsets
 * in 16-byte units); band_k_blocks holds the n blocks per row block.
 */
int pgg_fwd_plan(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch,
                 int64_t topK, int rowIdxType, pgg_dtype dtype, pgg_plan_info* info);

/*
 * ---------------------------------------------------------------------------
 * Probs-weighted unpermute backward (page "NPU DeepSeek-V3.2-Exp TileLang
 * operator practice", section moe_token_unpermute_grad). For the combine that
 * follows the expert matmul, out[b] = sum_j prob[b, j] * permuted[row(b, j)]:
 *
 *     perm_grad[row(b, j), h] = d_out[b, h] * prob[b, j]        (prob = 1 when probs is NULL)
 *     probs_grad[b, j]        = sum_h d_out[b, h] * permuted[row(b, j), h]
 *
 * with row(b, j) the expanded row of original position b * topK + j, read from
 * expandedRowIdx in the rowIdxType form (0 gather, 1 scatter, as above). No
 * experts are involved. perm_grad is the gradY of pgg_dx_execute and
 * pgg_dw_execute.
 *
 *   permuted       device, [M, H] of `dtype` (may be NULL when probs is NULL)
 *   d_out          device, [batch, H] of `dtype`
 *   probs          device, [batch, topK] of `dtype`, or NULL (plain scatter copy)
 *   probs_grad_dtype  `dtype` or PGG_F32 (the dot products accumulate in FP32)
 *   workspace      pgg_unpermute_grad_workspace_size bytes, 256-byte aligned;
 *                  status word at offset 0 (PGG_ERR_INDEX / PGG_ERR_NOT_PERM
 *                  zero-fill both outputs)
 *   perm_grad      device, [M, H] of `dtype`, fully overwritten
 *   probs_grad     device, [batch, topK], required with probs
 *
 * perm_grad is d_out * prob rounded once to `dtype`; each probs_grad is one
 * FP32 sum in a fixed order: bitwise repeatable. All pointers aligned to their
 * element size; 16-byte vector access when H * sizeof(dtype) is a multiple of
 * 16 and the row pointers are 16-byte aligned.
 */
int pgg_unpermute_grad_workspace_size(int64_t M, int64_t batch, int64_t topK,
                                      size_t* workspace_bytes);

int pgg_unpermute_grad(const void* permuted, const void* d_out, const void* probs,
                       const int64_t* expandedRowIdx, int64_t M, int64_t H, int64_t batch,
                       int64_t topK, int rowIdxType, pgg_dtype dtype, pgg_dtype probs_grad_dtype,
                       void* workspace, size_t workspace_bytes, void* perm_grad, void* probs_grad,
                       pgg_stream_t stream);

/*
 * The same call in two stream-ordered stages, for callers that validate the
 * routing once and apply it to several tensors, and for timing the kernel
 * alone. pgg_unpermute_grad is exactly prep followed by apply.
 *   pgg_unpermute_grad_prep   index validation and the inverse map, into the
 *                             workspace (status word at offset 0).
 *   pgg_unpermute_grad_apply  the unpermute kernel; reads the workspace that a
 *                             prep of the same expandedRowIdx (same M, batch,
 *                             topK, rowIdxType) filled earlier on the stream.
 *                             Its arguments and checks are those of
 *                             pgg_unpermute_grad.
 */
int pgg_unpermute_grad_prep(const int64_t* expandedRowIdx, int64_t M, int64_t batch, int64_t topK,
                            int rowIdxType, void* workspace, size_t workspace_bytes,
                            pgg_stream_t stream);

int pgg_unpermute_grad_apply(const void* permuted, const void* d_out, const void* probs,
                             const int64_t* expandedRowIdx, int64_t M, int64_t H, int64_t batch,
                             int64_t topK, int rowIdxType, pgg_dtype dtype,
                             pgg_dtype probs_grad_dtype, void* workspace, size_t workspace_bytes,
                             void* perm_grad, void* probs_grad, pgg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PGG_H */
