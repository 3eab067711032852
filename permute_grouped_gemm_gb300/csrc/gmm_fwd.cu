// Forward of the MoE permute + grouped matmul on tcgen05 tensor cores:
//
//     y[i, n] = sum over k of x[batch(i), k] * weight[g(i), k, n]
//
// ("MoeInitRoutingGroupedMatmulGrad design", sections 1.1 and 1.2, forward
// chain: MoeInitRouting(x) -> expanded_x, then GroupedMatmul(expanded_x,
// weight) -> y.) expanded_x is never materialised: its rows are gathered from
// x by token while they are staged. y is written in expanded order.
//
// Tile: one row block of an expert (at most 256 expanded rows, from the
// routing step's row-block list) x 256 output columns n, on a pair of CTAs
// (tcgen05 cta_group::2, MMA M = 256 rows, N = 256), reduced over K 64 at a
// time. CTA r owns rows 128 r .. 128 r + 127 of the block: their fp32
// accumulators (128 lanes x 256 columns, two buffers) live in its tensor
// memory.
//   A = x rows of the block's tokens, K-major: each CTA gathers its 128 rows x
//       64 k (one 128-byte swizzled row each) with 16-byte cp.async, one
//       producer warp per stage slot; rows past the block and k past K read
//       as 0. The tokens of a tile are loaded once.
//   B = weight[g, k0 .. k0 + 63, n], MN-major: each CTA loads its half of the
//       256 n as two 64-n panels by TMA from a 3-D map {N, K, G}. When the
//       weight rows are not a multiple of 16 bytes (N even, not a multiple of
//       8), the gather warps copy the panels instead, one 128-byte k row
//       segment per warp instruction, 4 bytes per lane, into the same
//       swizzled layout, and the epilogue writes y with 4-byte stores.
// Seven stage slots: the gathers' round trip (slot free -> rows copied ->
// slot full) is what bounds the kernel, and the shared memory in flight covers
// it. The epilogue therefore writes y straight from registers, with no
// shared-memory staging: each warp turns its 32 rows x 128 bytes into 16-byte
// blocks, transposes them within groups of eight lanes, and every warp store
// then writes four rows' full 128-byte segments. Rows past the row block
// (the next expert's rows) are not written.
//
// Warp roles per CTA: 0 TMA for the weight; 1 tensor-memory allocation and
// (even CTA) MMA issue; one gather warp per stage slot; four epilogue warps,
// one per tensor-memory lane quarter (13 warps in all, so that no SM
// sub-partition holds more than four and each thread may use 128 registers).
// Tiles are statically interleaved over the clusters. Waits are bounded; when
// one runs out the kernel records PGG_ERR_TIMEOUT, drains its copies and
// MMAs, frees tensor memory and returns.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "pgg_epilogue.cuh"
#include "pgg_gather.cuh"
#include "pgg_internal.h"
#include "pgg_ptx.cuh"

namespace pgg {
namespace {

constexpr int kFM = 128;       // expanded rows per CTA (the pair's MMA M is 256)
constexpr int kFN = 256;       // output columns n per tile (MMA N)
constexpr int kFK = 64;        // reduction (k) per stage: one 128-byte row of A
constexpr int kStages = 7;
constexpr int kPanel = kFK * 128;                // B panel: 64 k rows x 128 bytes (64 n)
constexpr int kABytes = kFM * 128;               // A: 128 rows x 128 bytes
constexpr int kBBytes = 2 * kPanel;              // B: this CTA's 128 n
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kGatherWarps = kStages;
constexpr int kEpiWarps = 4;
constexpr int kEpiWarp0 = 2 + kGatherWarps;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kTmemCols = 512;
constexpr int kAccCols = 256;

struct FwdCtl {
  uint64_t full[kStages];   // even CTA: weight bytes of both CTAs + x gathered in both (2 arrivals)
  uint64_t empty[kStages];  // each CTA: MMAs of the stage done (multicast commit)
  uint64_t tfull[2];        // each CTA: accumulator ready
  uint64_t tempty[2];       // even CTA: accumulator drained (epilogue warps x 2 CTAs)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr int kSmemBytes =
    kStages * kStageBytes + static_cast<int>(sizeof(FwdCtl)) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

__device__ __forceinline__ void raise_status(WsHeader* hdr, uint32_t code, uint32_t site) {
  if (atomicCAS(&hdr->status, 0u, code) == 0u) hdr->timeout_site = site;
}

__device__ __forceinline__ uint32_t cluster_id() { return blockIdx.x >> 1; }
__device__ __forceinline__ uint32_t n_clusters() { return gridDim.x >> 1; }

struct FTile {
  int64_t g, row0, n0;  // row0: this CTA's first expanded row
  int rows;             // this CTA's rows of the block (0 .. 128)
};

__device__ __forceinline__ FTile ftile_of(uint32_t t, const FwdArgs& a, uint32_t rank) {
  const uint32_t rb = t / static_cast<uint32_t>(a.n_blocks);
  int4 e = a.rblist[check_index(a.hdr, rb, a.max_row_blocks, 70)];
  // checked build: a row block outside the experts or rows becomes an empty one
  if (!check_ok(a.hdr,
                e.x >= 0 && e.x < a.G && e.y >= 0 && e.z >= 0 &&
                    static_cast<int64_t>(e.y) + e.z <= a.M,
                71))
    e = make_int4(0, 0, 0, 0);
  FTile x;
  x.g = e.x;
  x.row0 = static_cast<int64_t>(e.y) + kFM * rank;
  const int left = e.z - kFM * static_cast<int>(rank);
  x.rows = left < 0 ? 0 : (left > kFM ? kFM : left);
  x.n0 = static_cast<int64_t>(t - rb * static_cast<uint32_t>(a.n_blocks)) * kFN;
  return x;
}

__device__ __forceinline__ uint32_t b_bytes(const FwdArgs& a, int64_t n0, uint32_t rank) {
  const int64_t nc = n0 + 128 * rank;
  uint32_t b = 0;
  for (int j = 0; j < 2; ++j) b += (nc + 64 * j < a.N) ? static_cast<uint32_t>(kPanel) : 0u;
  return b;
}

__device__ void w_producer(uint8_t* smem, FwdCtl* ctl, const CUtensorMap* tm_w, const FwdArgs& a,
                           uint32_t total, int nks, uint32_t rank) {
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const bool leader = rank == 0;
  int stage = 0;
  uint32_t phase = 0, outstanding = 0, last_parity = 0;
  bool failed = false;
  for (uint32_t t = cluster_id(); t < total && !failed; t += n_clusters()) {
    const FTile x = ftile_of(t, a, rank);
    // gathered weight rows: the arrival carries no bytes
    const uint32_t both = a.gather_w ? 0u : b_bytes(a, x.n0, 0) + b_bytes(a, x.n0, 1);
    const int64_t nc = x.n0 + 128 * rank;
    for (int ks = 0; ks < nks; ++ks) {
      if (!ptx::mbar_wait_cluster(&ctl->empty[stage], phase ^ 1u, lim, abort)) {
        failed = true;
        break;
      }
      uint8_t* sb = smem + stage * kStageBytes + kABytes;
      const uint32_t fb = ptx::mapa(&ctl->full[stage], 0);
      if (leader) ptx::mbar_arrive_expect_tx(&ctl->full[stage], both);
      for (int j = 0; j < 2 && !a.gather_w; ++j)
        if (nc + 64 * j < a.N)
          ptx::tma_load_3d_pair(sb + j * kPanel, tm_w, fb, static_cast<int32_t>(nc + 64 * j),
                                ks * kFK, static_cast<int32_t>(x.g));
      outstanding |= 1u << stage;
      last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (failed) {
    ctl->abort = 1;
    raise_status(a.hdr, kStTimeout, 22);
  }
  if (leader) {
    int no_abort = 0;
    for (int s = 0; s < kStages; ++s)
      if (outstanding & (1u << s))
        ptx::mbar_wait_cluster(&ctl->full[s], (last_parity >> s) & 1u, lim, &no_abort);
  }
}

// Tokens of this CTA's rows lane, lane + 32, lane + 64, lane + 96 of a tile
// (-1 past the block).
__device__ __forceinline__ void tile_tokens(const FTile& x, const FwdArgs& a, int lane,
                                            int32_t (&tok)[4]) {
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const int r = lane + 32 * h;
    tok[h] = r < x.rows ? static_cast<int32_t>(check_index(
                              a.hdr, a.rowinfo[check_index(a.hdr, x.row0 + r, a.M, 72)].token,
                              a.batch, 73))
                        : -1;
  }
}

// Gather warp w fills stage slot w: the CTA's stages w, w + S, ... (stage q
// = tile q / nks, k block q % nks). Rows lane >> 3 + 4 j, 16-byte chunk lane & 7.
template <int DT>
__device__ void x_gatherer(uint8_t* smem, FwdCtl* ctl, const FwdArgs& a, uint32_t total, int nks,
                           uint32_t rank) {
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int w = (threadIdx.x >> 5) - 2;
  const int lane = threadIdx.x & 31;
  const int c = lane & 7;
  const char* xb = static_cast<const char*>(a.x);
  const uint32_t sa_slot = ptx::smem_addr(smem + w * kStageBytes);
  const uint32_t full = ptx::mapa(&ctl->full[w], 0);
  uint32_t phase = 0;
  bool failed = false;
  // position of the warp's next stage in the sequence: tile index j (t =
  // cluster + j * clusters) and k block
  uint32_t j = static_cast<uint32_t>(w / nks);
  int kb = w % nks;
  uint32_t tok_tile = 0xFFFFFFFFu;
  // this lane's rows (lane >> 3) + 4 q of the current tile: the x row's
  // offset in 16-byte units, or kNoRow past the block
  constexpr uint32_t kNoRow = 0xFFFFFFFFu;
  const uint32_t row_units = static_cast<uint32_t>(a.K / 8);
  uint32_t row16[kFM / 4];
  FTile x;
  while (true) {
    const uint32_t t = cluster_id() + j * n_clusters();
    if (t >= total) break;
    if (t != tok_tile) {
      x = ftile_of(t, a, rank);
      int32_t tok[4];
      tile_tokens(x, a, lane, tok);
#pragma unroll
      for (int q = 0; q < kFM / 4; ++q) {
        const int rr = (lane >> 3) + 4 * q;
        const int32_t tk = __shfl_sync(0xFFFFFFFFu, tok[rr >> 5], rr & 31);
        row16[q] = tk >= 0 ? static_cast<uint32_t>(tk) * row_units : kNoRow;
      }
      tok_tile = t;
    }
    if (!ptx::mbar_wait_cluster(&ctl->empty[w], phase ^ 1u, lim, abort)) {
      failed = true;
      break;
    }
    const int64_t k = static_cast<int64_t>(kb) * kFK + c * 8;
    const bool k_ok = k < a.K;
    const char* xk = xb + k * 2;
#pragma unroll
    for (int q = 0; q < kFM / 4; ++q) {
      const int rr = (lane >> 3) + 4 * q;
      const bool ok = k_ok && row16[q] != kNoRow;
      const void* src = ok ? static_cast<const void*>(xk + (static_cast<uint64_t>(row16[q]) << 4))
                           : static_cast<const void*>(xb);
      ptx::cp_async_16(sa_slot + rr * 128 + ((c ^ (rr & 7)) << 4), src, ok ? 16u : 0u);
    }
    if (a.gather_w) {
      // the weight panels: k rows kb * 64 .. + 63 of expert g, this CTA's 128
      // n from x.n0 + 128 rank, copied as wide as each row's alignment allows,
      // zeros outside K and N
      const char* wb = static_cast<const char*>(a.w);
      const int64_t k0 = static_cast<int64_t>(kb) * kFK;
      const int64_t kn = a.K - k0 < kFK ? a.K - k0 : kFK;
#pragma unroll 1
      for (int p = 0; p < 2; ++p) {
        const int64_t n = x.n0 + 128 * rank + 64 * p;
        const int64_t left = (a.N - n) * 2;
        const int seg = left < 0 ? 0 : (left < 128 ? static_cast<int>(left) : 128);
        gather_rows_sw128(sa_slot + kABytes + p * kPanel, wb + ((x.g * a.K + k0) * a.N + n) * 2,
                          a.N * 2, kFK, kn < 0 ? 0 : static_cast<int>(kn), seg, a.hdr, lane, 0,
                          1);
      }
    }
    ptx::cp_async_commit();
    ptx::cp_async_wait<0>();
    ptx::fence_proxy_async_smem();
    __syncwarp();
    // the even CTA's own rows go to its own MMA thread: CTA scope suffices
    if (lane == 0) {
      if (rank == 0)
        ptx::mbar_arrive(&ctl->full[w]);
      else
        ptx::mbar_arrive_remote(full);
    }
    phase ^= 1u;
    kb += kStages;
    while (kb >= nks) {
      kb -= nks;
      ++j;
    }
  }
  ptx::cp_async_wait<0>();
  if (failed) {
    ctl->abort = 1;
    if (lane == 0) raise_status(a.hdr, kStTimeout, 23);
  }
}

template <int DT>
__device__ void mma_issuer(uint8_t* smem, FwdCtl* ctl, uint32_t tmem_base, const FwdArgs& a,
                           uint32_t total, int nks) {
  constexpr uint32_t kFmt = DT == PGG_BF16 ? 1u : 0u;
  // A (x rows) K-major, B (weight) MN-major
  constexpr uint32_t idesc = ptx::idesc_make(kFmt, 2 * kFM, kFN) | (1u << 16);
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  int stage = 0, acc = 0;
  uint32_t phase = 0, aph = 0;
  bool issued = false, failed = false;
  for (uint32_t t = cluster_id(); t < total && !failed; t += n_clusters()) {
    if (!ptx::mbar_wait_cluster(&ctl->tempty[acc], aph ^ 1u, lim, abort)) {
      failed = true;
      break;
    }
    ptx::tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
    for (int ks = 0; ks < nks; ++ks) {
      if (!ptx::mbar_wait_cluster(&ctl->full[stage], phase, lim, abort)) {
        failed = true;
        break;
      }
      ptx::tc_fence_after_sync();
      const uint32_t sa = ptx::smem_addr(smem + stage * kStageBytes);
      const uint64_t da = ptx::sdesc_sw128(sa);
      const uint64_t db = ptx::sdesc_sw128_mn(sa + kABytes, kPanel);
#pragma unroll
      for (int kk = 0; kk < kFK / 16; ++kk) {
        const uint64_t a_off = static_cast<uint64_t>((kk * 32) >> 4);         // 16 k: 32 bytes
        const uint64_t b_off = static_cast<uint64_t>((kk * 16 * 128) >> 4);   // 16 k rows
        ptx::mma_f16_pair(d_tmem, da + a_off, db + b_off, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
      }
      issued = true;
      ptx::mma_commit_pair(&ctl->empty[stage], 0x3);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (failed) break;
    ptx::mma_commit_pair(&ctl->tfull[acc], 0x3);
    acc ^= 1;
    if (acc == 0) aph ^= 1u;
  }
  if (failed) {
    ctl->abort = 1;
    raise_status(a.hdr, kStTimeout, 24);
  }
  if (issued) {
    int no_abort = 0;
    ptx::mma_commit_pair(&ctl->drain, 0x1);
    ptx::mbar_wait(&ctl->drain, 0u, lim, &no_abort);
  }
}

template <int DT>
__device__ void epilogue(FwdCtl* ctl, uint32_t tmem_base, const FwdArgs& a, uint32_t total,
                         uint32_t rank) {
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;  // accumulator lanes (rows) 32 q .. 32 q + 31
  const int e = warp - kEpiWarp0;
  constexpr int kSpan = kFN / (kEpiWarps / 4);  // accumulator columns this warp writes
  const int col0 = (e / 4) * kSpan;
  const bool f32 = a.out_f32 != 0;
  const int oes = f32 ? 4 : 2;
  const int cols = 128 / oes;
  const uint32_t tempty0 = ptx::mapa(&ctl->tempty[0], 0);
  const uint32_t tempty1 = ptx::mapa(&ctl->tempty[1], 0);
  int acc = 0;
  uint32_t aph = 0;
  bool held = a.hold_release != 0;  // (test hook: the first release is withheld)
  for (uint32_t t = cluster_id(); t < total; t += n_clusters()) {
    const FTile x = ftile_of(t, a, rank);
    const int valid = x.rows - 32 * quarter;  // rows of this warp's 32 that exist
    const bool ok = ptx::mbar_wait_cluster(&ctl->tfull[acc], aph, lim, abort);
    if (!__all_sync(0xFFFFFFFFu, ok)) {
      if (lane == 0) {
        ctl->abort = 1;
        raise_status(a.hdr, kStTimeout, 25);
      }
      break;
    }
    ptx::tc_fence_after_sync();
    const uint32_t t_lane =
        tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) + static_cast<uint32_t>(acc * kAccCols);
    const int64_t row_w = x.row0 + 32 * quarter;  // first expanded row of this warp
#pragma unroll 1
    for (int c0 = col0; c0 < col0 + kSpan && x.n0 + c0 < a.N && valid > 0; c0 += cols) {
      uint4 b[8];
      chunk_blocks<DT>(t_lane + static_cast<uint32_t>(c0), f32, b);
      // rows past the block belong to the next expert and are not written
      store_chunk(b, static_cast<char*>(a.out), row_w, valid, a.N, x.n0 + c0, oes, a.gather_w != 0,
                  lane);
    }
    ptx::tc_fence_before_sync();
    __syncwarp();
    // tensor memory changes hands (the output goes out through global memory,
    // not to the MMA thread): CTA scope
    if (lane == 0 && !held) ptx::mbar_arrive_remote_cta(acc ? tempty1 : tempty0);
    held = false;
    acc ^= 1;
    if (acc == 0) aph ^= 1u;
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 1)
    gmm_fwd_kernel(const __grid_constant__ CUtensorMap tm_w, const FwdArgs a) {
  ptx::griddep_wait();  // launched with programmatic serialization: predecessors done
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  auto* ctl = reinterpret_cast<FwdCtl*>(smem + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();

  // Routing validation failed: the result is defined as zeros.
  const uint32_t st = a.hdr->status;
  if (st == kStIndex || st == kStGroupSum || st == kStNotPerm) {
    const int64_t n = a.M * a.N;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < n;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      if (a.out_f32)
        static_cast<float*>(a.out)[q] = 0.0f;
      else
        static_cast<uint16_t*>(a.out)[q] = 0;
    }
    return;
  }
  const uint32_t total = a.hdr->n_row_blocks * static_cast<uint32_t>(a.n_blocks);
  const int nks = static_cast<int>((a.K + kFK - 1) / kFK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&ctl->full[s], 3);
      ptx::mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl->tfull[b], 1);
      ptx::mbar_init(&ctl->tempty[b], 2 * kEpiWarps);
    }
    ptx::mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0 && !a.gather_w) ptx::tma_prefetch_desc(&tm_w);
  if (warp == 1) {
    ptx::tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) w_producer(smem, ctl, &tm_w, a, total, nks, rank);
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) mma_issuer<DT>(smem, ctl, tmem_base, a, total, nks);
  } else if (warp < kEpiWarp0) {
    x_gatherer<DT>(smem, ctl, a, total, nks, rank);
  } else {
    epilogue<DT>(ctl, tmem_base, a, total, rank);
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

int fwd_smem_bytes() { return kSmemBytes; }
int fwd_threads() { return kThreads; }
int fwd_rows_per_block() { return 2 * kFM; }
int fwd_stages() { return kStages; }

void fwd_tiles(int64_t N, int* n_blocks) { *n_blocks = static_cast<int>((N + kFN - 1) / kFN); }

cudaError_t launch_fwd(int dtype, const CUtensorMap& tm_w, const FwdArgs& a, int64_t max_tiles,
                       int num_sms, cudaStream_t stream) {
  void (*kern)(const CUtensorMap, const FwdArgs) = nullptr;
  if (dtype == PGG_BF16)
    kern = gmm_fwd_kernel<PGG_BF16>;
  else if (dtype == PGG_F16)
    kern = gmm_fwd_kernel<PGG_F16>;
  else
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int64_t want = max_tiles < num_sms / 2 ? max_tiles : num_sms / 2;
  if (want < 1) want = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * want), 1, 1);
  int clusters = 0;
  err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (err != cudaSuccess) return err;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  return launch_pdl(kern, dim3(static_cast<unsigned>(2 * (clusters < want ? clusters : want))),
                    dim3(kThreads), static_cast<size_t>(kSmemBytes), stream, 2, tm_w, a);
}

}  // namespace pgg
