// Internal definitions shared by the host planner and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "pgg.h"

#include <utility>

namespace pgg {

// Output columns (problem K) per tile. They are the 128 accumulator lanes of
// one tensor-memory tile.
constexpr int kKBlock = 128;
// Bytes of one operand row inside a pipeline stage: one 128-byte swizzle atom
// along the reduction dimension (64 half-precision or 32 fp32 elements).
constexpr int kRowBytes = 128;
// d_y is read through five tensor maps whose boxes are 16, 32, 64, 128 and
// 256 rows high; each tile takes one copy per k step with the smallest box
// that covers its rows (the number of copies, not their size, limits the copy
// engine here).
constexpr int kDyMaps = 5;
constexpr int kDyMinRows = 16;

struct DyMaps {
  CUtensorMap box[kDyMaps];  // box[j]: 16 << j rows x one 128-byte row segment
};

// Status codes written by the kernels (same values as pgg_status).
constexpr uint32_t kStIndex = 16, kStGroupSum = 17, kStNotPerm = 18, kStTimeout = 19;
constexpr uint32_t kStCheck = 20;  // a device bounds check failed (checked build only)

// Start of the workspace. The status word comes first (documented in pgg.h).
struct alignas(16) WsHeader {
  uint32_t status;        // first device-detected error, 0 = ok
  uint32_t sched_next;    // dynamic tile counter of the grouped-GEMM kernel
  uint32_t n_row_blocks;  // number of non-empty row blocks
  uint32_t timeout_site;  // where a bounded wait ran out, or (checked build) where a
                          // bounds check failed (diagnostic)
  uint32_t unsorted;      // 1: some expert's rows are not in increasing original position
  uint32_t pad[11];
};
static_assert(sizeof(WsHeader) == 64, "header size");

// Device bounds checks of the checked build (compiled with -DPGG_CHECKS).
// check_index returns i when 0 <= i < n. Otherwise it records PGG_ERR_CHECK in
// the status word (the first error wins; `site` goes to timeout_site) and
// returns 0, so that the access stays inside the buffer and the kernel's
// control flow, barriers and bounded waits are unchanged: nothing traps and
// nothing hangs, and the caller reads the status word. The default build
// compiles the check away and returns i.
#ifdef __CUDACC__
__device__ __forceinline__ int64_t check_index(WsHeader* hdr, int64_t i, int64_t n,
                                               uint32_t site) {
#ifdef PGG_CHECKS
  if (i >= 0 && i < n) return i;
  if (atomicCAS(&hdr->status, 0u, kStCheck) == 0u) hdr->timeout_site = site;
  return 0;
#else
  (void)hdr;
  (void)n;
  (void)site;
  return i;
#endif
}

// The same for a condition: records PGG_ERR_CHECK and returns false when `ok`
// is false (the caller then substitutes values that keep every access in
// bounds); always true in the default build.
__device__ __forceinline__ bool check_ok(WsHeader* hdr, bool ok, uint32_t site) {
#ifdef PGG_CHECKS
  if (!ok && atomicCAS(&hdr->status, 0u, kStCheck) == 0u) hdr->timeout_site = site;
  return ok;
#else
  (void)hdr;
  (void)ok;
  (void)site;
  return true;
#endif
}
#endif

// 1 in the checked build.
#ifdef PGG_CHECKS
constexpr int kCheckedBuild = 1;
#else
constexpr int kCheckedBuild = 0;
#endif

struct Layout {
  size_t hdr, off, rbstart, rblist, inv, rowinfo, tickets, seg, total;
  int64_t n_tickets;  // batch * k_blocks, rounded up to a multiple of 4
};

// Largest token slab of the owner variant of the d_x kernel (gmm_dx_owner.cu).
constexpr int kMaxSlabTokens = 224;  // owner variant; tensor memory columns 480-511 stay free

struct Plan {
  int variant;         // 0 wide row blocks on CTA pairs, 1 narrow row blocks, 2 wide on single
                       // CTAs, 3 FP32-pipe kernel, 4 owner kernel, 5 variant 0 with operands
                       // gathered by warps (rows the tensor-memory-access unit cannot stream)
  int pair;            // 1: CTA-pair tiles of 256 k
  int dtype;           // pgg_dtype
  int rows_per_block;  // MMA N extent
  int stages;
  int threads;
  int smem_bytes;
  int k_blocks;
  int band_k_blocks;
  int k_units;     // k_blocks, or k-block pairs for CTA-pair tiles
  int band_units;
  int64_t max_row_blocks;
  int64_t M, N, K, G, batch, topK;
  int row_idx_type;
  int nk;  // reduction steps: ceil(N / elements per 128-byte row)
  int slab_tokens;  // owner variant: tokens per slab (<= kMaxSlabTokens); 0 otherwise
  int n_slabs;      // owner variant: ceil(batch / slab_tokens); 0 otherwise
  Layout layout;
};

// Per-row record written by the routing kernels: token and rank of the
// expanded row among that token's rows (by increasing expanded index).
struct RowInfo {
  int32_t token;
  int32_t rank;
};

struct GemmArgs {
  const void* dy;         // [M, N] dtype (read directly by the gathered-operand variant)
  const void* w;          // [G, K, N] dtype (read directly by the gathered-operand variant)
  int64_t N;
  const int4* rblist;     // {expert, first row, rows, 0} per row block
  const RowInfo* rowinfo; // [M]
  uint32_t* tickets;      // [batch * k_blocks]
  WsHeader* hdr;
  float* out;             // [batch, K]
  int64_t K;
  int64_t batch;
  int64_t M, G, max_row_blocks;  // bounds of the routing tables (checked build)
  int32_t k_blocks;    // ceil(K / 128): ticket columns
  int32_t k_units;     // k blocks per row block in the tile order (pairs: k-block pairs)
  int32_t band_units;  // k units per band of the tile order
  int32_t nk;
  uint32_t ticket_bias;
  int32_t vec_rows;  // 1: epilogue writes 512-byte row segments with v4 stores / reductions
                     // (needs K % 4 == 0); 0: one 128-byte scalar store / reduction per warp
  int32_t only_if_unsorted;  // 1: the owner kernel ran first; do the work only if it could not
  uint64_t wait_limit_ns;
};

// Arguments of the owner variant of the d_x kernel (gmm_dx_owner.cu).
struct OwnerArgs {
  const int64_t* off;     // [G + 1] first expanded row of each expert
  const int32_t* seg;     // [G][n_slabs + 1] first row of expert g with token >= slab * T
  const RowInfo* rowinfo; // [M]
  WsHeader* hdr;
  float* out;             // [batch, K]
  int64_t M, K, G, batch;
  int32_t n_slabs;
  int32_t slab_tokens;  // T
  int32_t k_units;  // ceil(K / 256): k ranges of a CTA pair
  int32_t nk;       // reduction steps: ceil(N / 128) when wide, else ceil(N / 64)
  int32_t wide;     // 1: stages of two 64-n panels (N a multiple of 64)
  int32_t tma_out;  // 1: d_x written by TMA stores (K % 4 == 0, out 16-byte aligned)
  int32_t hold_release;  // test hook: 1 = the epilogue never frees accumulator 0 after its
                         // first chunk (the bounded waits then run out); 0 in normal use
  uint64_t wait_limit_ns;
};

// Tensor maps of the owner kernel: the d_x kernel's (d_y boxes of 16 << j rows,
// weight {N, K, G}); for wide stages, weight {64, K, N / 64, G} with boxes
// {64, 128, 2, 1} and d_y {64, M, N / 64} with boxes {64, 64, 2}; for TMA
// write-out, d_x {K, batch} fp32 with boxes {32, 32}.
struct OwnerMaps {
  DyMaps dy;
  CUtensorMap tw;
  CUtensorMap tw4;
  CUtensorMap dy3;
  CUtensorMap tout;
};

// Arguments of the FP32-pipe kernel used when the operands cannot be streamed
// by the tensor-memory-access unit (row bytes not a multiple of 16, or a
// pointer not 16-byte aligned).
struct SimtArgs {
  const void* dy;         // [M, N] dtype
  const void* w;          // [G, K, N] dtype
  const int4* rblist;     // {expert, first row, rows, 0} per row block (any row count)
  const RowInfo* rowinfo; // [M]
  uint32_t* tickets;      // [batch * k_blocks]
  WsHeader* hdr;
  float* out;             // [batch, K]
  int64_t N;
  int64_t K;
  int64_t batch;
  int64_t M, G, max_row_blocks;  // bounds of the routing tables (checked build)
  int32_t k_blocks;
  uint32_t ticket_bias;
  int32_t vec_out;  // 1: K % 4 == 0 and out 16-byte aligned (16-byte stores / reductions)
  uint64_t wait_limit_ns;
};

// Arguments of the weight-gradient kernels (gmm_dw.cu, gmm_dw_simt.cu).
struct DwArgs {
  const void* x;           // [batch, K] dtype: the forward input, original token order
  const void* dy;          // [M, N] dtype, expanded order
  const int64_t* off;      // [G + 1] first expanded row of each expert (routing step)
  const RowInfo* rowinfo;  // [M] token of each expanded row (routing step)
  WsHeader* hdr;
  void* out;               // [G, K, N] in the output dtype
  int64_t M, N, K, G, batch;
  int32_t k_blocks;  // output rows (k) blocks per expert
  int32_t n_blocks;  // output column (n) blocks per expert
  int32_t out_f32;   // 1: out is fp32; 0: out has the input dtype
  int32_t dy_3d;     // tensor-core kernel: d_y map is 3-D {64 n, rows, n / 64} (N % 64 == 0)
  int32_t gather_dy;  // tensor-core kernel: 1 = d_y rows copied by the gather warps (4-byte
                      // cp.async) and the output written with 4-byte stores (N even, N * 2
                      // not a multiple of 16); 0 = TMA for both
  int32_t hold_release;  // test hook (tensor-core kernel): 1 = each epilogue warp keeps its
                         // first accumulator release back; 0 in normal use
  uint64_t wait_limit_ns;
};

// Arguments of the forward kernels (gmm_fwd.cu, gmm_fwd_simt.cu).
struct FwdArgs {
  const void* x;           // [batch, K] dtype: the forward input, original token order
  const void* w;           // [G, K, N] dtype (read directly by the FP32-pipe kernel)
  const int4* rblist;      // {expert, first row, rows, 0} per row block (routing step)
  const RowInfo* rowinfo;  // [M] token of each expanded row
  WsHeader* hdr;
  void* out;               // y [M, N] in the output dtype, expanded order
  int64_t M, N, K;
  int64_t G, batch, max_row_blocks;  // bounds of the routing tables (checked build)
  int32_t n_blocks;  // output column blocks per row block
  int32_t out_f32;   // 1: y is fp32; 0: y has the input dtype
  int32_t gather_w;  // tensor-core kernel: 1 = weight rows copied by the gather warps (4-byte
                     // cp.async) and y written with 4-byte stores (N even, N * 2 not a
                     // multiple of 16); 0 = TMA for both
  int32_t hold_release;  // test hook (tensor-core kernel): 1 = each epilogue warp keeps its
                         // first accumulator release back; 0 in normal use
  uint64_t wait_limit_ns;
};

// Arguments of the probs-weighted unpermute backward (unpermute_grad.cu).
struct UnpermArgs {
  const void* perm;       // [M, H] dtype (with probs)
  const void* dout;       // [batch, H] dtype
  const void* probs;      // [batch, topK] dtype, or null
  const int64_t* idx;     // [M] expandedRowIdx
  const int32_t* inv;     // [M] inverse of idx (index prep)
  WsHeader* hdr;
  void* perm_grad;        // [M, H] dtype
  void* probs_grad;       // [batch, topK] in the probs-grad dtype, or null
  int64_t M, H, batch, topK;
  int32_t row_idx_type;
  int32_t probs_grad_f32;  // 1: probs_grad is fp32; 0: it has the input dtype
};

// Launches `kern` with the programmatic-serialization attribute: its CTAs may
// be scheduled while the previous kernel in the stream drains, and every such
// kernel calls griddepcontrol.wait (ptx::griddep_wait) before it reads
// anything, so the previous kernel's results are complete and visible by then.
// cluster_x > 1 adds that cluster dimension.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, unsigned cluster_x, Args&&... args) {
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace pgg
