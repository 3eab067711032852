// C ABI of the fused MoE permute + grouped-matmul backward (include/pgg.h):
// argument validation (the constraint table and infershape checks of the page
// "MoeInitRoutingGroupedMatmulGrad design", sections "约束" and 2.3), the
// execution plan and workspace layout, tensor-map encoding, and the launches.

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "pgg.h"
#include "pgg_internal.h"

namespace pgg {

cudaError_t launch_route_prep(const Plan& plan, const int64_t* idx, const int64_t* group_list,
                              void* workspace, int num_sms, cudaStream_t stream);
cudaError_t launch_grouped_gemm(int dtype, int variant, const DyMaps& tdy,
                                const CUtensorMap& tw, const GemmArgs& args, int max_ctas,
                                cudaStream_t stream);
bool kernel_config(int dtype, int variant, int* rows, int* stages, int* threads, int* smem,
                   int* pair);
void simt_config(int* rows, int* stages, int* threads, int* smem);
cudaError_t launch_simt(int dtype, const SimtArgs& a, int64_t max_tiles, int num_sms,
                        cudaStream_t stream);
int dw_smem_bytes();
int dw_threads();
int dw_stage_rows();
int dw_stages();
void dw_tiles(int64_t K, int64_t N, int* k_blocks, int* n_blocks);
cudaError_t launch_dw(int dtype, const CUtensorMap& tm_dy, const CUtensorMap& tm_out,
                      const DwArgs& a, int num_sms, cudaStream_t stream);
void dw_simt_tiles(int64_t K, int64_t N, int* k_blocks, int* n_blocks);
int dw_simt_smem_bytes();
cudaError_t launch_dw_simt(int dtype, const DwArgs& a, int vec, int num_sms, cudaStream_t stream);
int fwd_smem_bytes();
int fwd_threads();
int fwd_rows_per_block();
int fwd_stages();
void fwd_tiles(int64_t N, int* n_blocks);
cudaError_t launch_fwd(int dtype, const CUtensorMap& tm_w, const FwdArgs& a, int64_t max_tiles,
                       int num_sms, cudaStream_t stream);
void fwd_simt_tiles(int64_t N, int* n_blocks);
int fwd_simt_smem_bytes();
cudaError_t launch_fwd_simt(int dtype, const FwdArgs& a, int vec, int64_t max_tiles, int num_sms,
                            cudaStream_t stream);
int owner_smem_bytes(bool wide);
int owner_stages(bool wide);
int owner_threads();
cudaError_t launch_owner(int dtype, const OwnerMaps& m, const OwnerArgs& a, int num_sms,
                         cudaStream_t stream);
cudaError_t launch_index_prep(const int64_t* idx, int64_t M, int row_idx_type, int32_t* inv,
                              WsHeader* hdr, int num_sms, cudaStream_t stream);
cudaError_t launch_unpermute_grad(int dtype, const UnpermArgs& a, bool vec, bool pairs,
                                  int num_sms, cudaStream_t stream);

namespace {

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};
std::atomic<uint32_t> g_ticket_bias{0};
std::atomic<int> g_hold_release{0};
std::atomic<int> g_force_variant{-1};
std::atomic<int> g_band_k_blocks{0};

constexpr int64_t kInt32Max = 2147483647;
constexpr int kVariantSimt = 3;    // FP32-pipe kernel (gmm_dx_simt.cu)
constexpr int kVariantOwner = 4;   // slab-owner kernel (gmm_dx_owner.cu), ticketed fallback
constexpr int kVariantGather = 5;  // ticketed pair kernel, operands copied by gather warps

// Token slab of the owner variant: about 112 rows of each expert per slab
// when the routing is even (G * T / topK rows), so that most experts take one
// MMA of N <= 128; a multiple of 32 in [32, 256].
int owner_slab_tokens(int64_t G, int64_t topK) {
  int64_t t = 112 * G / topK / 32 * 32;
  if (t < 32) t = 32;
  if (t > kMaxSlabTokens) t = kMaxSlabTokens;
  return static_cast<int>(t);
}

// The owner variant pays off when its slabs hold about 112 rows of each
// expert (so its MMAs are wide: few experts per token), for 16-bit inputs,
// and when there are enough (slab, 256-k) units to fill the GPU.
bool owner_fits(int64_t K, int64_t G, int64_t batch, int64_t topK, int dtype) {
  if (dtype == PGG_F32) return false;
  if (112 * G > static_cast<int64_t>(kMaxSlabTokens) * topK) return false;
  const int64_t T = owner_slab_tokens(G, topK);
  const int64_t slabs = (batch + T - 1) / T;
  const int64_t k_units = (K + 255) / 256;
  return slabs * k_units >= 128;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int elem_size(int dtype) { return dtype == PGG_F32 ? 4 : 2; }

// Host checks of sizes and attributes; pointers are checked by the callers.
int check_sizes(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch, int64_t topK,
                int rowIdxType, int dtype) {
  if (dtype != PGG_F32 && dtype != PGG_F16 && dtype != PGG_BF16) return PGG_ERR_DTYPE;
  if (batch <= 0 || topK <= 0 || (rowIdxType != 0 && rowIdxType != 1)) return PGG_ERR_ATTR;
  if (M <= 0 || N <= 0 || K <= 0 || G <= 0) return PGG_ERR_SHAPE;
  if (M > kInt32Max || N > kInt32Max || K > kInt32Max || G > kInt32Max) return PGG_ERR_SHAPE;
  if (L != M) return PGG_ERR_SHAPE;
  if (batch > M || topK > M || batch * topK != M) return PGG_ERR_SHAPE;
  return PGG_OK;
}

// Rows of d_y and weight that the tensor-memory-access unit can stream: their
// byte length must be a multiple of 16.
bool rows_streamable(int64_t N, int dtype) { return (N * elem_size(dtype)) % 16 == 0; }

// Rows that the gather warps of variant 5 can copy 4 bytes at a time: 16-bit
// elements, an even count per row.
bool rows_gatherable(int64_t N, int dtype) { return dtype != PGG_F32 && N % 2 == 0; }

// rows_override > 0: row blocks of that many rows (the forward's 256) instead
// of the d_x variant's.
int make_plan(int64_t M, int64_t N, int64_t K, int64_t G, int64_t batch, int64_t topK,
              int rowIdxType, int dtype, Plan* p, int rows_override = 0) {
  std::memset(p, 0, sizeof(*p));
  p->dtype = dtype;
  int variant = g_force_variant.load();
  if (variant < 0) {
    variant = (M / G < 64) ? 1 : 0;
    if (owner_fits(K, G, batch, topK, dtype)) variant = kVariantOwner;
  }
  if (variant == kVariantOwner && dtype == PGG_F32) variant = 0;
  if (variant == kVariantGather && !rows_gatherable(N, dtype)) variant = kVariantSimt;
  if (!rows_streamable(N, dtype) && variant != kVariantSimt)
    variant = rows_gatherable(N, dtype) ? kVariantGather : kVariantSimt;
  p->variant = variant;
  if (variant == kVariantSimt) {
    simt_config(&p->rows_per_block, &p->stages, &p->threads, &p->smem_bytes);
  } else if (!kernel_config(dtype, variant == kVariantOwner ? 0 : variant, &p->rows_per_block,
                            &p->stages, &p->threads, &p->smem_bytes, &p->pair)) {
    // the owner variant keeps the ticketed kernel's (variant 0) row blocks for its fallback
    return PGG_ERR_DTYPE;
  }
  p->slab_tokens = variant == kVariantOwner ? owner_slab_tokens(G, topK) : 0;
  p->n_slabs = variant == kVariantOwner
                   ? static_cast<int>((batch + p->slab_tokens - 1) / p->slab_tokens)
                   : 0;
  if (rows_override > 0) p->rows_per_block = rows_override;
  p->M = M;
  p->N = N;
  p->K = K;
  p->G = G;
  p->batch = batch;
  p->topK = topK;
  p->row_idx_type = rowIdxType;
  p->k_blocks = static_cast<int>((K + kKBlock - 1) / kKBlock);
  const int band = g_band_k_blocks.load();
  p->band_k_blocks = (band > 0 && band < p->k_blocks) ? band : p->k_blocks;
  const int elems_per_row = kRowBytes / elem_size(dtype);
  p->nk = static_cast<int>((N + elems_per_row - 1) / elems_per_row);
  p->max_row_blocks = (M + p->rows_per_block - 1) / p->rows_per_block + G;
  p->k_units = p->pair ? (p->k_blocks + 1) / 2 : p->k_blocks;
  p->band_units = p->pair ? (p->band_k_blocks + 1) / 2 : p->band_k_blocks;
  if (p->max_row_blocks * p->k_units > kInt32Max) return PGG_ERR_SHAPE;

  Layout& L = p->layout;
  size_t a = 0;
  auto take = [&](size_t bytes) {
    const size_t o = a;
    a = align_up(a + bytes, 256);
    return o;
  };
  L.hdr = take(sizeof(WsHeader));
  L.off = take(sizeof(int64_t) * static_cast<size_t>(G + 1));
  L.rbstart = take(sizeof(int32_t) * static_cast<size_t>(G + 1));
  L.rblist = take(sizeof(int4) * static_cast<size_t>(p->max_row_blocks));
  L.inv = take(sizeof(int32_t) * static_cast<size_t>(M));
  L.rowinfo = take(sizeof(RowInfo) * static_cast<size_t>(M));
  L.n_tickets = (batch * p->k_blocks + 3) / 4 * 4;
  L.tickets = take(sizeof(uint32_t) * static_cast<size_t>(L.n_tickets));
  L.seg = take(sizeof(int32_t) * static_cast<size_t>(G) * static_cast<size_t>(p->n_slabs + 1));
  L.total = a;
  return PGG_OK;
}

struct DeviceInfo {
  int num_sms = 0;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[64];

int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PGG_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev[dev].num_sms == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return PGG_ERR_CUDA;
    g_dev[dev].num_sms = sms;
  }
  *out = g_dev[dev];
  return PGG_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

CUtensorMapDataType tmap_type(int dtype) {
  if (dtype == PGG_BF16) return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (dtype == PGG_F16) return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
}

// d_y [M, N] as 2-D maps with boxes of 32, 64, 128 and 256 rows x one
// 128-byte row segment. weight [G, K, N] as a 3-D map; boxes of 1 expert x
// 128 k x one segment. Rows or columns outside the tensor read as zero. L2
// promotion: 128 bytes (one box row) for the CTA-pair tiles, where 256 bytes
// measured about 1% slower on the largest workload; 256 bytes for the others,
// whose weight streams from HBM (narrow row blocks of many small experts).
int encode_maps(const Plan& p, const void* dy, const void* w, DyMaps* tdy, CUtensorMap* tw) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PGG_ERR_CUDA;
  const cuuint64_t es = static_cast<cuuint64_t>(elem_size(p.dtype));
  const cuuint32_t box_n = static_cast<cuuint32_t>(kRowBytes / es);
  const CUtensorMapL2promotion promo = (p.pair && p.variant == 0)
                                           ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                           : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  for (int j = 0; j < kDyMaps; ++j) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.N) * es};
    cuuint32_t box[2] = {box_n, static_cast<cuuint32_t>(kDyMinRows << j)};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&tdy->box[j], tmap_type(p.dtype), 2, const_cast<void*>(dy), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PGG_ERR_CUDA;
  }
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.K),
                          static_cast<cuuint64_t>(p.G)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(p.N) * es,
                             static_cast<cuuint64_t>(p.N) * static_cast<cuuint64_t>(p.K) * es};
    cuuint32_t box[3] = {box_n, static_cast<cuuint32_t>(kKBlock), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(tw, tmap_type(p.dtype), 3, const_cast<void*>(w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PGG_ERR_CUDA;
  }
  return PGG_OK;
}

// Owner kernel stages of two 64-n panels (16-bit dtypes, N a multiple of 64):
// weight {64, K, N / 64, G} in boxes {64, 128, 2, 1}, d_y {64, M, N / 64} in
// boxes {64, 64, 2}; panels past N / 64 read as zero.
int encode_owner_wide_maps(const Plan& p, const void* dy, const void* w, OwnerMaps* m) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PGG_ERR_CUDA;
  const cuuint64_t N = static_cast<cuuint64_t>(p.N), K = static_cast<cuuint64_t>(p.K);
  {
    cuuint64_t dims[4] = {64, K, N / 64, static_cast<cuuint64_t>(p.G)};
    cuuint64_t strides[3] = {N * 2, 128, N * K * 2};
    cuuint32_t box[4] = {64, 128, 2, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (enc(&m->tw4, tmap_type(p.dtype), 4, const_cast<void*>(w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PGG_ERR_CUDA;
  }
  {
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(p.M), N / 64};
    cuuint64_t strides[2] = {N * 2, 128};
    cuuint32_t box[3] = {64, 64, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&m->dy3, tmap_type(p.dtype), 3, const_cast<void*>(dy), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PGG_ERR_CUDA;
  }
  return PGG_OK;
}

// d_x [batch, K] fp32 for the owner kernel's write-out: boxes of 32 k x 32
// tokens, no swizzle; stores past K or batch are clipped.
int encode_owner_out_map(const Plan& p, float* out, CUtensorMap* m) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PGG_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(p.batch)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.K) * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, out, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? PGG_OK
             : PGG_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Common front half of every entry point that enqueues work.
int prepare(const void* gradY, const void* weight, const int64_t* idx, const int64_t* gl,
            bool need_values, int64_t M, int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch,
            int64_t topK, int rowIdxType, int dtype, void* ws, size_t ws_bytes, const float* out,
            Plan* plan) {
  if (!idx || !gl || !ws) return PGG_ERR_NULL;
  if (need_values && (!gradY || !weight || !out)) return PGG_ERR_NULL;
  int rc = check_sizes(M, N, K, G, L, batch, topK, rowIdxType, dtype);
  if (rc != PGG_OK) return rc;
  rc = make_plan(M, N, K, G, batch, topK, rowIdxType, dtype, plan);
  if (rc != PGG_OK) return rc;
  if (!aligned(ws, 256) || !aligned(idx, 8) || !aligned(gl, 8)) return PGG_ERR_ALIGN;
  const uintptr_t es = static_cast<uintptr_t>(elem_size(dtype));
  if (need_values && (!aligned(gradY, es) || !aligned(weight, es) || !aligned(out, 4)))
    return PGG_ERR_ALIGN;
  if (ws_bytes < plan->layout.total) return PGG_ERR_WORKSPACE;
  return PGG_OK;
}

int run_route_prep(const Plan& plan, const int64_t* idx, const int64_t* gl, void* ws,
                   cudaStream_t stream) {
  DeviceInfo di;
  if (device_info(&di) != PGG_OK) return PGG_ERR_CUDA;
  return launch_route_prep(plan, idx, gl, ws, di.num_sms, stream) == cudaSuccess ? PGG_OK
                                                                                   : PGG_ERR_CUDA;
}

// The FP32-pipe kernel: any row length and element-aligned pointers. It runs
// on the row blocks the routing step built, whatever their height.
int run_simt(const Plan& plan, const void* gradY, const void* weight, void* ws, float* out,
             const DeviceInfo& di, cudaStream_t stream) {
  char* w = static_cast<char*>(ws);
  SimtArgs a;
  a.dy = gradY;
  a.w = weight;
  a.rblist = reinterpret_cast<const int4*>(w + plan.layout.rblist);
  a.rowinfo = reinterpret_cast<const RowInfo*>(w + plan.layout.rowinfo);
  a.tickets = reinterpret_cast<uint32_t*>(w + plan.layout.tickets);
  a.hdr = reinterpret_cast<WsHeader*>(w + plan.layout.hdr);
  a.out = out;
  a.N = plan.N;
  a.K = plan.K;
  a.batch = plan.batch;
  a.M = plan.M;
  a.G = plan.G;
  a.max_row_blocks = plan.max_row_blocks;
  a.k_blocks = plan.k_blocks;
  a.ticket_bias = g_ticket_bias.load();
  a.vec_out = (plan.K % 4 == 0 && aligned(out, 16)) ? 1 : 0;
  a.wait_limit_ns = g_wait_limit_ns.load();
  return launch_simt(plan.dtype, a, plan.max_row_blocks * plan.k_blocks, di.num_sms, stream) ==
                 cudaSuccess
             ? PGG_OK
             : PGG_ERR_CUDA;
}

int run_grouped_gemm(const Plan& plan, const void* gradY, const void* weight, void* ws, float* out,
                     cudaStream_t stream) {
  DeviceInfo di;
  if (device_info(&di) != PGG_OK) return PGG_ERR_CUDA;
  if (plan.variant == kVariantSimt) return run_simt(plan, gradY, weight, ws, out, di, stream);
  // Operands the tensor-memory-access unit cannot stream (rows, or pointers
  // not 16-byte aligned): copied by gather warps when their rows and pointers
  // allow 4-byte copies, else the FP32-pipe kernel. Every plan's row blocks
  // have at most 256 rows, which both kernels take.
  const bool gather = plan.variant == kVariantGather || !aligned(gradY, 16) ||
                      !aligned(weight, 16);
  if (gather && !(rows_gatherable(plan.N, plan.dtype) && aligned(gradY, 4) && aligned(weight, 4)))
    return run_simt(plan, gradY, weight, ws, out, di, stream);
  DyMaps tdy;
  const bool owner = plan.variant == kVariantOwner && !gather;
  CUtensorMap tw;
  std::memset(&tdy, 0, sizeof(tdy));
  std::memset(&tw, 0, sizeof(tw));
  int rc = gather ? PGG_OK : encode_maps(plan, gradY, weight, &tdy, &tw);
  if (rc != PGG_OK) return rc;
  char* w = static_cast<char*>(ws);
  GemmArgs a;
  a.dy = gradY;
  a.w = weight;
  a.N = plan.N;
  a.rblist = reinterpret_cast<const int4*>(w + plan.layout.rblist);
  a.rowinfo = reinterpret_cast<const RowInfo*>(w + plan.layout.rowinfo);
  a.tickets = reinterpret_cast<uint32_t*>(w + plan.layout.tickets);
  a.hdr = reinterpret_cast<WsHeader*>(w + plan.layout.hdr);
  a.out = out;
  a.K = plan.K;
  a.batch = plan.batch;
  a.M = plan.M;
  a.G = plan.G;
  a.max_row_blocks = plan.max_row_blocks;
  a.k_blocks = plan.k_blocks;
  a.k_units = plan.k_units;
  a.band_units = plan.band_units;
  a.nk = plan.nk;
  a.ticket_bias = g_ticket_bias.load();
  a.vec_rows = (plan.K % 4 == 0 && aligned(out, 16)) ? 1 : 0;
  a.only_if_unsorted = owner ? 1 : 0;
  a.wait_limit_ns = g_wait_limit_ns.load();
  if (owner) {
    OwnerArgs o;
    o.off = reinterpret_cast<const int64_t*>(w + plan.layout.off);
    o.seg = reinterpret_cast<const int32_t*>(w + plan.layout.seg);
    o.rowinfo = a.rowinfo;
    o.hdr = a.hdr;
    o.out = out;
    o.M = plan.M;
    o.K = plan.K;
    o.G = plan.G;
    o.batch = plan.batch;
    o.n_slabs = plan.n_slabs;
    o.slab_tokens = plan.slab_tokens;
    o.k_units = static_cast<int32_t>((plan.K + 255) / 256);
    o.nk = plan.nk;
    o.wide = 0;
    o.hold_release = g_hold_release.load() != 0 ? 1 : 0;
    o.wait_limit_ns = a.wait_limit_ns;
    OwnerMaps om;
    om.dy = tdy;
    om.tw = tw;
    std::memset(&om.tw4, 0, sizeof(om.tw4));
    std::memset(&om.dy3, 0, sizeof(om.dy3));
    std::memset(&om.tout, 0, sizeof(om.tout));
    o.tma_out = 0;
    if (plan.K % 4 == 0 && aligned(out, 16)) {
      rc = encode_owner_out_map(plan, out, &om.tout);
      if (rc != PGG_OK) return rc;
      o.tma_out = 1;
    }
    if (plan.N % 64 == 0) {
      rc = encode_owner_wide_maps(plan, gradY, weight, &om);
      if (rc != PGG_OK) return rc;
      o.wide = 1;
      o.nk = static_cast<int32_t>((plan.N + 127) / 128);
    }
    if (launch_owner(plan.dtype, om, o, di.num_sms, stream) != cudaSuccess) return PGG_ERR_CUDA;
  }
  // the ticketed kernel; after the owner kernel it works only when that one
  // could not (some expert's rows not in increasing original position)
  // the gathered-operand kernel takes the tiles of variant 0 (CTA pairs of
  // 256 k, row blocks of up to 256 rows)
  const int kernel_variant = gather ? kVariantGather : (owner ? 0 : plan.variant);
  const int k_units = gather ? (plan.k_blocks + 1) / 2 : plan.k_units;
  if (gather) {
    a.k_units = k_units;
    a.band_units = (plan.band_k_blocks + 1) / 2;
  }
  const int64_t max_ctas =
      plan.max_row_blocks * k_units * ((gather || plan.pair) ? 2 : 1);
  const int grid = static_cast<int>(max_ctas < di.num_sms ? max_ctas : di.num_sms);
  return launch_grouped_gemm(plan.dtype, kernel_variant, tdy, tw, a, grid, stream) == cudaSuccess
             ? PGG_OK
             : PGG_ERR_CUDA;
}

// ---------------------------------------------------------------- weight gradient

// The tensor-core kernel takes 16-bit inputs whose x and d_y rows are whole
// 16-byte units, with x, d_y and the output 16-byte aligned; everything else
// runs on the FP32 pipes.
bool dw_tensor_path(int dtype, int64_t N, int64_t K, const void* x, const void* dy,
                    const void* out) {
  if (g_force_variant.load() == kVariantSimt) return false;
  if (dtype == PGG_F32) return false;
  if ((K * 2) % 16 != 0 || (N * 2) % 16 != 0) return false;
  return aligned(x, 16) && aligned(dy, 16) && aligned(out, 16);
}

// The tensor-core weight gradient with the d_y rows copied by its gather
// warps (4 bytes at a time) and the output written with 4-byte stores: 16-bit
// inputs, x rows whole 16-byte units and x 16-byte aligned (gathered 16 bytes
// at a time), N even, d_y and the output 4-byte aligned.
bool dw_gather_path(int dtype, int64_t N, int64_t K, const void* x, const void* dy,
                    const void* out) {
  if (g_force_variant.load() == kVariantSimt) return false;
  if (dtype == PGG_F32) return false;
  if ((K * 2) % 16 != 0 || N % 2 != 0) return false;
  return aligned(x, 16) && aligned(dy, 4) && aligned(out, 4);
}

int check_dw(const void* x, const void* gradY, const int64_t* idx, const int64_t* gl,
             int64_t M, int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch, int64_t topK,
             int rowIdxType, int dtype, int out_dtype, void* ws, size_t ws_bytes,
             const void* dweight, Plan* plan) {
  if (!x || !gradY || !idx || !gl || !ws || !dweight) return PGG_ERR_NULL;
  int rc = check_sizes(M, N, K, G, L, batch, topK, rowIdxType, dtype);
  if (rc != PGG_OK) return rc;
  if (out_dtype != dtype && out_dtype != PGG_F32) return PGG_ERR_DTYPE;
  if (G * K > kInt32Max / 4) return PGG_ERR_SHAPE;  // tile numbers stay below 2^31
  rc = make_plan(M, N, K, G, batch, topK, rowIdxType, dtype, plan);
  if (rc != PGG_OK) return rc;
  const uintptr_t es = static_cast<uintptr_t>(elem_size(dtype));
  if (!aligned(ws, 256) || !aligned(idx, 8) || !aligned(gl, 8)) return PGG_ERR_ALIGN;
  if (!aligned(x, es) || !aligned(gradY, es) ||
      !aligned(dweight, static_cast<uintptr_t>(elem_size(out_dtype))))
    return PGG_ERR_ALIGN;
  if (ws_bytes < plan->layout.total) return PGG_ERR_WORKSPACE;
  return PGG_OK;
}

int run_dw(const Plan& plan, const void* x, const void* gradY, void* ws, void* dweight,
           int out_dtype, cudaStream_t stream) {
  DeviceInfo di;
  if (device_info(&di) != PGG_OK) return PGG_ERR_CUDA;
  char* w = static_cast<char*>(ws);
  DwArgs a;
  a.x = x;
  a.dy = gradY;
  a.off = reinterpret_cast<const int64_t*>(w + plan.layout.off);
  a.rowinfo = reinterpret_cast<const RowInfo*>(w + plan.layout.rowinfo);
  a.hdr = reinterpret_cast<WsHeader*>(w + plan.layout.hdr);
  a.out = dweight;
  a.M = plan.M;
  a.N = plan.N;
  a.K = plan.K;
  a.G = plan.G;
  a.batch = plan.batch;
  a.out_f32 = out_dtype == PGG_F32 ? 1 : 0;
  a.dy_3d = 0;
  a.gather_dy = 0;
  a.hold_release = g_hold_release.load() != 0 ? 1 : 0;
  a.wait_limit_ns = g_wait_limit_ns.load();
  if (!dw_tensor_path(plan.dtype, plan.N, plan.K, x, gradY, dweight) &&
      dw_gather_path(plan.dtype, plan.N, plan.K, x, gradY, dweight)) {
    dw_tiles(plan.K, plan.N, &a.k_blocks, &a.n_blocks);
    a.gather_dy = 1;
    CUtensorMap none;
    std::memset(&none, 0, sizeof(none));
    return launch_dw(plan.dtype, none, none, a, di.num_sms, stream) == cudaSuccess ? PGG_OK
                                                                                   : PGG_ERR_CUDA;
  }
  if (dw_tensor_path(plan.dtype, plan.N, plan.K, x, gradY, dweight)) {
    dw_tiles(plan.K, plan.N, &a.k_blocks, &a.n_blocks);
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PGG_ERR_CUDA;
    CUtensorMap tm;
    const cuuint32_t rows = static_cast<cuuint32_t>(dw_stage_rows());
    CUresult cr;
    a.dy_3d = plan.N % 64 == 0 ? 1 : 0;
    if (a.dy_3d) {
      // {64 n, rows, n-chunk}: a box of 4 chunks lands as four 64-n panels;
      // chunks past N / 64 read as zero
      cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(plan.M),
                            static_cast<cuuint64_t>(plan.N / 64)};
      cuuint64_t strides[2] = {static_cast<cuuint64_t>(plan.N) * 2, 128};
      cuuint32_t box[3] = {64, rows, 2};  // one CTA's half of the tile's 256 n
      cuuint32_t estr[3] = {1, 1, 1};
      cr = enc(&tm, tmap_type(plan.dtype), 3, const_cast<void*>(gradY), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
      cuuint64_t dims[2] = {static_cast<cuuint64_t>(plan.N), static_cast<cuuint64_t>(plan.M)};
      cuuint64_t strides[1] = {static_cast<cuuint64_t>(plan.N) * 2};
      cuuint32_t box[2] = {64, rows};
      cuuint32_t estr[2] = {1, 1};
      cr = enc(&tm, tmap_type(plan.dtype), 2, const_cast<void*>(gradY), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (cr != CUDA_SUCCESS) return PGG_ERR_CUDA;
    // the output [G, K, N] as a 3-D map, boxes of 128 bytes x 32 rows of k
    CUtensorMap tm_out;
    {
      const int oes = out_dtype == PGG_F32 ? 4 : 2;
      cuuint64_t dims[3] = {static_cast<cuuint64_t>(plan.N), static_cast<cuuint64_t>(plan.K),
                            static_cast<cuuint64_t>(plan.G)};
      cuuint64_t strides[2] = {static_cast<cuuint64_t>(plan.N) * oes,
                               static_cast<cuuint64_t>(plan.N) * static_cast<cuuint64_t>(plan.K) *
                                   oes};
      cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / oes), 32, 1};
      cuuint32_t estr[3] = {1, 1, 1};
      if (enc(&tm_out, tmap_type(out_dtype), 3, dweight, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PGG_ERR_CUDA;
    }
    return launch_dw(plan.dtype, tm, tm_out, a, di.num_sms, stream) == cudaSuccess ? PGG_OK
                                                                                   : PGG_ERR_CUDA;
  }
  dw_simt_tiles(plan.K, plan.N, &a.k_blocks, &a.n_blocks);
  const uintptr_t vec_align = out_dtype == PGG_F32 ? 16 : 8;
  const int vec = (plan.N % 4 == 0 && aligned(dweight, vec_align)) ? 1 : 0;
  return launch_dw_simt(plan.dtype, a, vec, di.num_sms, stream) == cudaSuccess ? PGG_OK
                                                                                  : PGG_ERR_CUDA;
}

// ---------------------------------------------------------------- forward

// The tensor-core forward's gather warps address an x row by its offset in
// 16-byte units, held in 32 bits (x below 64 GiB).
bool fwd_x_rows_fit(int64_t batch, int64_t K) { return batch * (K / 8) < 0xFFFFFFFFll; }

// The tensor-core forward takes 16-bit inputs whose x, weight and y rows are
// whole 16-byte units, with x, weight and y 16-byte aligned.
bool fwd_tensor_path(int dtype, int64_t N, int64_t K, int64_t batch, const void* x, const void* w,
                     const void* y) {
  if (g_force_variant.load() == kVariantSimt) return false;
  if (dtype == PGG_F32) return false;
  if ((K * 2) % 16 != 0 || (N * 2) % 16 != 0 || !fwd_x_rows_fit(batch, K)) return false;
  return aligned(x, 16) && aligned(w, 16) && aligned(y, 16);
}

// The tensor-core forward with the weight rows copied by its gather warps (4
// bytes at a time) and y written with 4-byte stores: 16-bit inputs, x rows
// whole 16-byte units and x 16-byte aligned (gathered 16 bytes at a time), N
// even, weight and y 4-byte aligned.
bool fwd_gather_path(int dtype, int64_t N, int64_t K, int64_t batch, const void* x, const void* w,
                     const void* y) {
  if (g_force_variant.load() == kVariantSimt) return false;
  if (dtype == PGG_F32) return false;
  if ((K * 2) % 16 != 0 || N % 2 != 0 || !fwd_x_rows_fit(batch, K)) return false;
  return aligned(x, 16) && aligned(w, 4) && aligned(y, 4);
}

int make_fwd_plan(int64_t M, int64_t N, int64_t K, int64_t G, int64_t batch, int64_t topK,
                  int rowIdxType, int dtype, Plan* p) {
  return make_plan(M, N, K, G, batch, topK, rowIdxType, dtype, p, fwd_rows_per_block());
}

int check_fwd(const void* x, const void* weight, const int64_t* idx, const int64_t* gl,
              bool need_values, int64_t M, int64_t N, int64_t K, int64_t G, int64_t L,
              int64_t batch, int64_t topK, int rowIdxType, int dtype, int out_dtype, void* ws,
              size_t ws_bytes, const void* y, Plan* plan) {
  if (!idx || !gl || !ws) return PGG_ERR_NULL;
  if (need_values && (!x || !weight || !y)) return PGG_ERR_NULL;
  int rc = check_sizes(M, N, K, G, L, batch, topK, rowIdxType, dtype);
  if (rc != PGG_OK) return rc;
  if (out_dtype != dtype && out_dtype != PGG_F32) return PGG_ERR_DTYPE;
  rc = make_fwd_plan(M, N, K, G, batch, topK, rowIdxType, dtype, plan);
  if (rc != PGG_OK) return rc;
  if (!aligned(ws, 256) || !aligned(idx, 8) || !aligned(gl, 8)) return PGG_ERR_ALIGN;
  const uintptr_t es = static_cast<uintptr_t>(elem_size(dtype));
  if (need_values && (!aligned(x, es) || !aligned(weight, es) ||
                      !aligned(y, static_cast<uintptr_t>(elem_size(out_dtype)))))
    return PGG_ERR_ALIGN;
  if (ws_bytes < plan->layout.total) return PGG_ERR_WORKSPACE;
  return PGG_OK;
}

int run_fwd(const Plan& plan, const void* x, const void* weight, void* ws, void* y,
            int out_dtype, cudaStream_t stream) {
  DeviceInfo di;
  if (device_info(&di) != PGG_OK) return PGG_ERR_CUDA;
  char* w = static_cast<char*>(ws);
  FwdArgs a;
  a.x = x;
  a.w = weight;
  a.rblist = reinterpret_cast<const int4*>(w + plan.layout.rblist);
  a.rowinfo = reinterpret_cast<const RowInfo*>(w + plan.layout.rowinfo);
  a.hdr = reinterpret_cast<WsHeader*>(w + plan.layout.hdr);
  a.out = y;
  a.M = plan.M;
  a.N = plan.N;
  a.K = plan.K;
  a.G = plan.G;
  a.batch = plan.batch;
  a.max_row_blocks = plan.max_row_blocks;
  a.out_f32 = out_dtype == PGG_F32 ? 1 : 0;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.gather_w = 0;
  a.hold_release = g_hold_release.load() != 0 ? 1 : 0;
  if (!fwd_tensor_path(plan.dtype, plan.N, plan.K, plan.batch, x, weight, y) &&
      fwd_gather_path(plan.dtype, plan.N, plan.K, plan.batch, x, weight, y)) {
    fwd_tiles(plan.N, &a.n_blocks);
    a.gather_w = 1;
    CUtensorMap none;
    std::memset(&none, 0, sizeof(none));
    return launch_fwd(plan.dtype, none, a, plan.max_row_blocks * a.n_blocks, di.num_sms,
                      stream) == cudaSuccess
               ? PGG_OK
               : PGG_ERR_CUDA;
  }
  if (fwd_tensor_path(plan.dtype, plan.N, plan.K, plan.batch, x, weight, y)) {
    fwd_tiles(plan.N, &a.n_blocks);
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PGG_ERR_CUDA;
    CUtensorMap tm_w;
    {
      // weight [G, K, N]: boxes of 64 n x 64 k of one expert
      cuuint64_t dims[3] = {static_cast<cuuint64_t>(plan.N), static_cast<cuuint64_t>(plan.K),
                            static_cast<cuuint64_t>(plan.G)};
      cuuint64_t strides[2] = {static_cast<cuuint64_t>(plan.N) * 2,
                               static_cast<cuuint64_t>(plan.N) * static_cast<cuuint64_t>(plan.K) *
                                   2};
      cuuint32_t box[3] = {64, 64, 1};
      cuuint32_t estr[3] = {1, 1, 1};
      if (enc(&tm_w, tmap_type(plan.dtype), 3, const_cast<void*>(weight), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PGG_ERR_CUDA;
    }
    return launch_fwd(plan.dtype, tm_w, a, plan.max_row_blocks * a.n_blocks, di.num_sms,
                      stream) == cudaSuccess
               ? PGG_OK
               : PGG_ERR_CUDA;
  }
  fwd_simt_tiles(plan.N, &a.n_blocks);
  const uintptr_t vec_align = out_dtype == PGG_F32 ? 16 : 8;
  const int vec = (plan.N % 4 == 0 && aligned(y, vec_align)) ? 1 : 0;
  return launch_fwd_simt(plan.dtype, a, vec, plan.max_row_blocks * a.n_blocks, di.num_sms,
                         stream) == cudaSuccess
             ? PGG_OK
             : PGG_ERR_CUDA;
}

}  // namespace
}  // namespace pgg

using namespace pgg;

extern "C" {

int pgg_dx_workspace_size(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch,
                          int64_t topK, int rowIdxType, pgg_dtype dtype, size_t* workspace_bytes) {
  if (!workspace_bytes) return PGG_ERR_NULL;
  int rc = check_sizes(M, N, K, G, L, batch, topK, rowIdxType, dtype);
  if (rc != PGG_OK) return rc;
  Plan plan;
  rc = make_plan(M, N, K, G, batch, topK, rowIdxType, dtype, &plan);
  if (rc != PGG_OK) return rc;
  *workspace_bytes = plan.layout.total;
  return PGG_OK;
}

int pgg_dx_plan(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch, int64_t topK,
                int rowIdxType, pgg_dtype dtype, pgg_plan_info* info) {
  if (!info) return PGG_ERR_NULL;
  int rc = check_sizes(M, N, K, G, L, batch, topK, rowIdxType, dtype);
  if (rc != PGG_OK) return rc;
  Plan p;
  rc = make_plan(M, N, K, G, batch, topK, rowIdxType, dtype, &p);
  if (rc != PGG_OK) return rc;
  info->variant = p.variant;
  info->rows_per_block = p.variant == kVariantOwner ? p.slab_tokens : p.rows_per_block;
  info->k_per_block = kKBlock;
  info->stages = p.variant == kVariantOwner ? owner_stages(p.N % 64 == 0) : p.stages;
  info->k_blocks = p.k_blocks;
  info->band_k_blocks = p.band_k_blocks;
  info->max_row_blocks = p.max_row_blocks;
  info->workspace_bytes = p.layout.total;
  info->threads = p.variant == kVariantOwner ? owner_threads() : p.threads;
  info->smem_bytes =
      p.variant == kVariantOwner ? owner_smem_bytes(p.N % 64 == 0) : p.smem_bytes;
  info->cta_pair = p.variant == kVariantOwner ? 1 : p.pair;
  return PGG_OK;
}

int pgg_dx_route_prep(const int64_t* expandedRowIdx, const int64_t* groupList, int64_t M, int64_t N,
                      int64_t K, int64_t G, int64_t L, int64_t batch, int64_t topK, int rowIdxType,
                      pgg_dtype dtype, void* workspace, size_t workspace_bytes,
                      pgg_stream_t stream) {
  Plan plan;
  int rc = prepare(nullptr, nullptr, expandedRowIdx, groupList, false, M, N, K, G, L, batch, topK,
                   rowIdxType, dtype, workspace, workspace_bytes, nullptr, &plan);
  if (rc != PGG_OK) return rc;
  return run_route_prep(plan, expandedRowIdx, groupList, workspace,
                        reinterpret_cast<cudaStream_t>(stream));
}

int pgg_dx_grouped_gemm(const void* gradY, const void* weight, const int64_t* expandedRowIdx,
                        const int64_t* groupList, int64_t M, int64_t N, int64_t K, int64_t G,
                        int64_t L, int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                        void* workspace, size_t workspace_bytes, float* out,
                        pgg_stream_t stream) {
  Plan plan;
  int rc = prepare(gradY, weight, expandedRowIdx, groupList, true, M, N, K, G, L, batch, topK,
                   rowIdxType, dtype, workspace, workspace_bytes, out, &plan);
  if (rc != PGG_OK) return rc;
  return run_grouped_gemm(plan, gradY, weight, workspace, out,
                          reinterpret_cast<cudaStream_t>(stream));
}

int pgg_dx_execute(const void* gradY, const void* weight, const int64_t* expandedRowIdx,
                   const int64_t* groupList, int64_t M, int64_t N, int64_t K, int64_t G, int64_t L,
                   int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype, void* workspace,
                   size_t workspace_bytes, float* out, pgg_stream_t stream) {
  Plan plan;
  int rc = prepare(gradY, weight, expandedRowIdx, groupList, true, M, N, K, G, L, batch, topK,
                   rowIdxType, dtype, workspace, workspace_bytes, out, &plan);
  if (rc != PGG_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = run_route_prep(plan, expandedRowIdx, groupList, workspace, s);
  if (rc != PGG_OK) return rc;
  return run_grouped_gemm(plan, gradY, weight, workspace, out, s);
}

int pgg_dw_workspace_size(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch,
                          int64_t topK, int rowIdxType, pgg_dtype dtype, size_t* workspace_bytes) {
  return pgg_dx_workspace_size(M, N, K, G, L, batch, topK, rowIdxType, dtype, workspace_bytes);
}

int pgg_dw_plan(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch, int64_t topK,
                int rowIdxType, pgg_dtype dtype, pgg_plan_info* info) {
  if (!info) return PGG_ERR_NULL;
  int rc = check_sizes(M, N, K, G, L, batch, topK, rowIdxType, dtype);
  if (rc != PGG_OK) return rc;
  Plan p;
  rc = make_plan(M, N, K, G, batch, topK, rowIdxType, dtype, &p);
  if (rc != PGG_OK) return rc;
  // 16-byte aligned pointers assumed: only the shape decides here
  alignas(16) static const char probe[16] = {0};
  const bool tc = dw_tensor_path(dtype, N, K, probe, probe, probe);
  const bool ga = !tc && dw_gather_path(dtype, N, K, probe, probe, probe);
  std::memset(info, 0, sizeof(*info));
  int kb = 0, nb = 0;
  if (tc || ga) {
    dw_tiles(K, N, &kb, &nb);
    info->variant = tc ? 0 : kVariantGather;
    info->rows_per_block = dw_stage_rows();
    info->k_per_block = 256;
    info->stages = dw_stages();
    info->cta_pair = 1;
    info->threads = dw_threads();
    info->smem_bytes = dw_smem_bytes();
  } else {
    dw_simt_tiles(K, N, &kb, &nb);
    info->variant = kVariantSimt;
    info->rows_per_block = 32;
    info->k_per_block = 64;
    info->stages = 2;
    info->threads = 128;
    info->smem_bytes = dw_simt_smem_bytes();
  }
  info->k_blocks = kb;
  info->band_k_blocks = nb;
  info->max_row_blocks = G;
  info->workspace_bytes = p.layout.total;
  return PGG_OK;
}

int pgg_dw_execute(const void* x, const void* gradY, const int64_t* expandedRowIdx,
                   const int64_t* groupList, int64_t M, int64_t N, int64_t K, int64_t G, int64_t L,
                   int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                   pgg_dtype out_dtype, void* workspace, size_t workspace_bytes, void* dweight,
                   pgg_stream_t stream) {
  Plan plan;
  int rc = check_dw(x, gradY, expandedRowIdx, groupList, M, N, K, G, L, batch, topK, rowIdxType,
                    dtype, out_dtype, workspace, workspace_bytes, dweight, &plan);
  if (rc != PGG_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = run_route_prep(plan, expandedRowIdx, groupList, workspace, s);
  if (rc != PGG_OK) return rc;
  return run_dw(plan, x, gradY, workspace, dweight, out_dtype, s);
}

int pgg_dw_grouped_gemm(const void* x, const void* gradY, const int64_t* expandedRowIdx,
                        const int64_t* groupList, int64_t M, int64_t N, int64_t K, int64_t G,
                        int64_t L, int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                        pgg_dtype out_dtype, void* workspace, size_t workspace_bytes,
                        void* dweight, pgg_stream_t stream) {
  Plan plan;
  int rc = check_dw(x, gradY, expandedRowIdx, groupList, M, N, K, G, L, batch, topK, rowIdxType,
                    dtype, out_dtype, workspace, workspace_bytes, dweight, &plan);
  if (rc != PGG_OK) return rc;
  return run_dw(plan, x, gradY, workspace, dweight, out_dtype,
                reinterpret_cast<cudaStream_t>(stream));
}

int pgg_fwd_workspace_size(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch,
                           int64_t topK, int rowIdxType, pgg_dtype dtype, size_t* workspace_bytes) {
  if (!workspace_bytes) return PGG_ERR_NULL;
  int rc = check_sizes(M, N, K, G, L, batch, topK, rowIdxType, dtype);
  if (rc != PGG_OK) return rc;
  Plan plan;
  rc = make_fwd_plan(M, N, K, G, batch, topK, rowIdxType, dtype, &plan);
  if (rc != PGG_OK) return rc;
  *workspace_bytes = plan.layout.total;
  return PGG_OK;
}

int pgg_fwd_plan(int64_t M, int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch,
                 int64_t topK, int rowIdxType, pgg_dtype dtype, pgg_plan_info* info) {
  if (!info) return PGG_ERR_NULL;
  int rc = check_sizes(M, N, K, G, L, batch, topK, rowIdxType, dtype);
  if (rc != PGG_OK) return rc;
  Plan p;
  rc = make_fwd_plan(M, N, K, G, batch, topK, rowIdxType, dtype, &p);
  if (rc != PGG_OK) return rc;
  alignas(16) static const char probe[16] = {0};
  const bool tc = fwd_tensor_path(dtype, N, K, batch, probe, probe, probe);
  const bool ga = !tc && fwd_gather_path(dtype, N, K, batch, probe, probe, probe);
  std::memset(info, 0, sizeof(*info));
  int nb = 0;
  info->rows_per_block = p.rows_per_block;
  info->max_row_blocks = p.max_row_blocks;
  info->workspace_bytes = p.layout.total;
  if (tc || ga) {
    fwd_tiles(N, &nb);
    info->variant = tc ? 0 : kVariantGather;
    info->k_per_block = 64;
    info->stages = fwd_stages();
    info->threads = fwd_threads();
    info->smem_bytes = fwd_smem_bytes();
    info->cta_pair = 1;
  } else {
    fwd_simt_tiles(N, &nb);
    info->variant = kVariantSimt;
    info->k_per_block = 32;
    info->stages = 2;
    info->threads = 128;
    info->smem_bytes = fwd_simt_smem_bytes();
  }
  info->k_blocks = static_cast<int32_t>((K + info->k_per_block - 1) / info->k_per_block);
  info->band_k_blocks = nb;
  return PGG_OK;
}

int pgg_fwd_route_prep(const int64_t* expandedRowIdx, const int64_t* groupList, int64_t M,
                       int64_t N, int64_t K, int64_t G, int64_t L, int64_t batch, int64_t topK,
                       int rowIdxType, pgg_dtype dtype, void* workspace, size_t workspace_bytes,
                       pgg_stream_t stream) {
  Plan plan;
  int rc = check_fwd(nullptr, nullptr, expandedRowIdx, groupList, false, M, N, K, G, L, batch,
                     topK, rowIdxType, dtype, dtype, workspace, workspace_bytes, nullptr, &plan);
  if (rc != PGG_OK) return rc;
  return run_route_prep(plan, expandedRowIdx, groupList, workspace,
                        reinterpret_cast<cudaStream_t>(stream));
}

int pgg_fwd_grouped_gemm(const void* x, const void* weight, const int64_t* expandedRowIdx,
                         const int64_t* groupList, int64_t M, int64_t N, int64_t K, int64_t G,
                         int64_t L, int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                         pgg_dtype out_dtype, void* workspace, size_t workspace_bytes, void* y,
                         pgg_stream_t stream) {
  Plan plan;
  int rc = check_fwd(x, weight, expandedRowIdx, groupList, true, M, N, K, G, L, batch, topK,
                     rowIdxType, dtype, out_dtype, workspace, workspace_bytes, y, &plan);
  if (rc != PGG_OK) return rc;
  return run_fwd(plan, x, weight, workspace, y, out_dtype, reinterpret_cast<cudaStream_t>(stream));
}

int pgg_fwd_execute(const void* x, const void* weight, const int64_t* expandedRowIdx,
                    const int64_t* groupList, int64_t M, int64_t N, int64_t K, int64_t G, int64_t L,
                    int64_t batch, int64_t topK, int rowIdxType, pgg_dtype dtype,
                    pgg_dtype out_dtype, void* workspace, size_t workspace_bytes, void* y,
                    pgg_stream_t stream) {
  Plan plan;
  int rc = check_fwd(x, weight, expandedRowIdx, groupList, true, M, N, K, G, L, batch, topK,
                     rowIdxType, dtype, out_dtype, workspace, workspace_bytes, y, &plan);
  if (rc != PGG_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = run_route_prep(plan, expandedRowIdx, groupList, workspace, s);
  if (rc != PGG_OK) return rc;
  return run_fwd(plan, x, weight, workspace, y, out_dtype, s);
}

// Workspace of the unpermute backward: the header, then the inverse index.
static size_t unperm_inv_offset() { return 256; }

int pgg_unpermute_grad_workspace_size(int64_t M, int64_t batch, int64_t topK,
                                      size_t* workspace_bytes) {
  if (!workspace_bytes) return PGG_ERR_NULL;
  if (batch <= 0 || topK <= 0) return PGG_ERR_ATTR;
  if (M <= 0 || M > kInt32Max || batch * topK != M) return PGG_ERR_SHAPE;
  *workspace_bytes = unperm_inv_offset() + align_up(sizeof(int32_t) * static_cast<size_t>(M), 256);
  return PGG_OK;
}

namespace {

// Host checks shared by the unpermute entry points: sizes, attributes and the
// workspace (pointers of the values are checked by the apply step).
int unperm_check(const int64_t* idx, int64_t M, int64_t batch, int64_t topK, int rowIdxType,
                 const void* workspace, size_t workspace_bytes) {
  if (!idx || !workspace) return PGG_ERR_NULL;
  if (rowIdxType != 0 && rowIdxType != 1) return PGG_ERR_ATTR;
  size_t need = 0;
  const int rc = pgg_unpermute_grad_workspace_size(M, batch, topK, &need);
  if (rc != PGG_OK) return rc;
  if (!aligned(workspace, 256) || !aligned(idx, 8)) return PGG_ERR_ALIGN;
  if (workspace_bytes < need) return PGG_ERR_WORKSPACE;
  return PGG_OK;
}

}  // namespace

int pgg_unpermute_grad_prep(const int64_t* expandedRowIdx, int64_t M, int64_t batch, int64_t topK,
                            int rowIdxType, void* workspace, size_t workspace_bytes,
                            pgg_stream_t stream) {
  int rc = unperm_check(expandedRowIdx, M, batch, topK, rowIdxType, workspace, workspace_bytes);
  if (rc != PGG_OK) return rc;
  DeviceInfo di;
  if (device_info(&di) != PGG_OK) return PGG_ERR_CUDA;
  char* w = static_cast<char*>(workspace);
  return launch_index_prep(expandedRowIdx, M, rowIdxType,
                           reinterpret_cast<int32_t*>(w + unperm_inv_offset()),
                           reinterpret_cast<WsHeader*>(w), di.num_sms,
                           reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PGG_OK
             : PGG_ERR_CUDA;
}

int pgg_unpermute_grad_apply(const void* permuted, const void* d_out, const void* probs,
                             const int64_t* expandedRowIdx, int64_t M, int64_t H, int64_t batch,
                             int64_t topK, int rowIdxType, pgg_dtype dtype,
                             pgg_dtype probs_grad_dtype, void* workspace, size_t workspace_bytes,
                             void* perm_grad, void* probs_grad, pgg_stream_t stream) {
  if (!d_out || !perm_grad) return PGG_ERR_NULL;
  if (probs && (!permuted || !probs_grad)) return PGG_ERR_NULL;
  if (dtype != PGG_F32 && dtype != PGG_F16 && dtype != PGG_BF16) return PGG_ERR_DTYPE;
  if (probs_grad_dtype != dtype && probs_grad_dtype != PGG_F32) return PGG_ERR_DTYPE;
  int rc = unperm_check(expandedRowIdx, M, batch, topK, rowIdxType, workspace, workspace_bytes);
  if (rc != PGG_OK) return rc;
  if (H <= 0 || H > kInt32Max) return PGG_ERR_SHAPE;
  const uintptr_t es = static_cast<uintptr_t>(elem_size(dtype));
  if (!aligned(d_out, es) || !aligned(perm_grad, es) ||
      (probs && (!aligned(permuted, es) || !aligned(probs, es) ||
                 !aligned(probs_grad, elem_size(probs_grad_dtype)))))
    return PGG_ERR_ALIGN;
  DeviceInfo di;
  if (device_info(&di) != PGG_OK) return PGG_ERR_CUDA;
  char* w = static_cast<char*>(workspace);
  UnpermArgs a;
  a.perm = permuted;
  a.dout = d_out;
  a.probs = probs;
  a.idx = expandedRowIdx;
  a.inv = reinterpret_cast<const int32_t*>(w + unperm_inv_offset());
  a.hdr = reinterpret_cast<WsHeader*>(w);
  a.perm_grad = perm_grad;
  a.probs_grad = probs ? probs_grad : nullptr;
  a.M = M;
  a.H = H;
  a.batch = batch;
  a.topK = topK;
  a.row_idx_type = rowIdxType;
  a.probs_grad_f32 = probs_grad_dtype == PGG_F32 ? 1 : 0;
  const bool vec = (H * static_cast<int64_t>(es)) % 16 == 0 && aligned(d_out, 16) &&
                   aligned(perm_grad, 16) && (!probs || aligned(permuted, 16));
  const bool pairs = H % 2 == 0 && aligned(d_out, 4) && aligned(perm_grad, 4) &&
                     (!probs || aligned(permuted, 4));
  return launch_unpermute_grad(dtype, a, vec, pairs, di.num_sms,
                               reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PGG_OK
             : PGG_ERR_CUDA;
}

int pgg_unpermute_grad(const void* permuted, const void* d_out, const void* probs,
                       const int64_t* expandedRowIdx, int64_t M, int64_t H, int64_t batch,
                       int64_t topK, int rowIdxType, pgg_dtype dtype, pgg_dtype probs_grad_dtype,
                       void* workspace, size_t workspace_bytes, void* perm_grad, void* probs_grad,
                       pgg_stream_t stream) {
  // every host check before anything is enqueued
  if (!d_out || !expandedRowIdx || !workspace || !perm_grad) return PGG_ERR_NULL;
  if (probs && (!permuted || !probs_grad)) return PGG_ERR_NULL;
  if (dtype != PGG_F32 && dtype != PGG_F16 && dtype != PGG_BF16) return PGG_ERR_DTYPE;
  if (probs_grad_dtype != dtype && probs_grad_dtype != PGG_F32) return PGG_ERR_DTYPE;
  int rc = unperm_check(expandedRowIdx, M, batch, topK, rowIdxType, workspace, workspace_bytes);
  if (rc != PGG_OK) return rc;
  if (H <= 0 || H > kInt32Max) return PGG_ERR_SHAPE;
  const uintptr_t es = static_cast<uintptr_t>(elem_size(dtype));
  if (!aligned(d_out, es) || !aligned(perm_grad, es) ||
      (probs && (!aligned(permuted, es) || !aligned(probs, es) ||
                 !aligned(probs_grad, elem_size(probs_grad_dtype)))))
    return PGG_ERR_ALIGN;
  rc = pgg_unpermute_grad_prep(expandedRowIdx, M, batch, topK, rowIdxType, workspace,
                               workspace_bytes, stream);
  if (rc != PGG_OK) return rc;
  return pgg_unpermute_grad_apply(permuted, d_out, probs, expandedRowIdx, M, H, batch, topK,
                                  rowIdxType, dtype, probs_grad_dtype, workspace, workspace_bytes,
                                  perm_grad, probs_grad, stream);
}

const char* pgg_status_string(int status) {
  switch (status) {
    case PGG_OK: return "ok";
    case PGG_ERR_NULL: return "null pointer";
    case PGG_ERR_SHAPE: return "shape outside the constraints";
    case PGG_ERR_ATTR: return "attribute outside the constraints (batch, topK, rowIdxType)";
    case PGG_ERR_DTYPE: return "unsupported dtype";
    case PGG_ERR_WORKSPACE: return "workspace too small";
    case PGG_ERR_CUDA: return "CUDA call failed";
    case PGG_ERR_ALIGN: return "pointer or row stride not aligned";
    case PGG_ERR_INDEX: return "expandedRowIdx entry out of range";
    case PGG_ERR_GROUPSUM: return "groupList negative or sum != M";
    case PGG_ERR_NOT_PERM: return "expandedRowIdx is not a permutation";
    case PGG_ERR_TIMEOUT: return "a bounded device wait ran out";
    case PGG_ERR_CHECK: return "a device bounds check failed (checked build)";
    default: return "unknown status";
  }
}

void pgg_debug_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns == 0 ? kDefaultWaitNs : ns);
}

void pgg_debug_set_ticket_bias(uint32_t bias) { g_ticket_bias.store(bias); }
void pgg_debug_set_hold_release(int hold) { g_hold_release.store(hold); }

void pgg_debug_force_variant(int variant) { g_force_variant.store(variant); }

void pgg_debug_set_band_k_blocks(int k_blocks) { g_band_k_blocks.store(k_blocks); }

}  // extern "C"

// ---------------------------------------------------------------------------
// Entry point for callers that cannot allocate device memory.
//
// Some callers of this library have no way to obtain scratch memory at the
// moment they need the gradient: a plugin running inside a framework that owns
// every device allocation and exposes no allocator to it, a serving or
// real-time runtime that reserves all of HBM up front and forbids cudaMalloc
// afterwards (a late allocation could fail or stall), or plain C code with no
// allocator handle at all. pgg_dx_execute_static_scratch serves them: it
// takes the same inputs and output as pgg_dx_execute but no workspace, and
// uses instead the fixed scratch array below, which the CUDA module reserves
// on every device that loads this library and keeps until the process exits.

namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB

// The device-side scratch. In host code this name is only a stand-in for the
// symbol, not a device address: its address is looked up per device below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

// Device address of g_static_scratch on the current device. A call made while
// `stream` is not being captured looks it up afresh (so an address made stale
// by cudaDeviceReset or a new primary context is never used) and remembers it
// per device; a call made during a stream capture uses the remembered address,
// so the first call on a device must come before any capture on it.
int static_scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PGG_ERR_CUDA;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  const bool capturing =
      cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!capturing) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return PGG_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  if (!g_scratch_ptr[dev]) return PGG_ERR_CUDA;
  *out = g_scratch_ptr[dev];
  return PGG_OK;
}

}  // namespace

extern "C" int pgg_dx_execute_static_scratch(const void* gradY, const void* weight,
                                             const int64_t* expandedRowIdx,
                                             const int64_t* groupList, int64_t M, int64_t N,
                                             int64_t K, int64_t G, int64_t L, int64_t batch,
                                             int64_t topK, int rowIdxType, pgg_dtype dtype,
                                             float* out, uint32_t* status, pgg_stream_t stream) {
  size_t need = 0;
  int rc = pgg_dx_workspace_size(M, N, K, G, L, batch, topK, rowIdxType, dtype, &need);
  if (rc != PGG_OK) return rc;
  if (need > kStaticScratchBytes) return PGG_ERR_WORKSPACE;
  void* scratch = nullptr;
  rc = static_scratch_address(reinterpret_cast<cudaStream_t>(stream), &scratch);
  if (rc != PGG_OK) return rc;
  rc = pgg_dx_execute(gradY, weight, expandedRowIdx, groupList, M, N, K, G, L, batch, topK,
                      rowIdxType, dtype, scratch, kStaticScratchBytes, out, stream);
  if (rc != PGG_OK || !status) return rc;
  // the status word is the first uint32 of the scratch
  return cudaMemcpyAsync(status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PGG_OK
             : PGG_ERR_CUDA;
}
