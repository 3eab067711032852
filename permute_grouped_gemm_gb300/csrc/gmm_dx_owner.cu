// Owner variant of the fused d_x backward ("MoeInitRoutingGroupedMatmulGrad
// design", section "数学定义和公式": d_x[b, k] = sum over the token's rows i of
// sum_n d_y[i, n] * weight[g(i), k, n]), for problems with few experts.
//
// A CTA pair owns a block of d_x outright: a slab of T tokens (T <= 256, set
// by the host so that a slab holds about 112 rows of each expert) x 256 k
// (128 per CTA). It walks the experts in increasing order; for each expert it
// takes the expert's rows whose tokens lie in the slab (one contiguous range
// when each expert's rows are in increasing original position, which the
// routing step checks), computes C = weight[g] d_y[rows]^T for its 256 k on
// the tensor cores (cta_group::2, M = 256 k, N = rows rounded up to 32 and at
// most 128, TMA for both operands, accumulators in tensor memory), and adds
// each row into a shared-memory copy of the slab's d_x block. Each epilogue
// thread owns one d_x column k of the slab, for every token: it alone reads,
// adds and writes that column, in program order, in increasing expanded index
// (increasing expert, then increasing row within the expert), which is the
// order of additions of the ticketed kernel, with no tickets, no barriers
// between threads and no atomics. A token's first row (rank 0) stores, later
// rows load, add and store; two rows of one token inside one expert are
// adjacent and carried in a register. When the slab is done each thread
// writes its column to d_x once.
//
// When some expert's rows are not in increasing original position the kernel
// leaves at once and the ticketed kernel, launched after it, does the work.
//
// Warp roles per CTA: 0 TMA; 1 tensor-memory allocation and (even CTA) MMA
// issue; 2-5 epilogue. Units (slab, k range) are statically interleaved over
// the clusters. Waits are bounded; when one runs out the kernel records
// PGG_ERR_TIMEOUT, drains its copies and MMAs, frees tensor memory and
// returns.

#include <cstdint>

#include "pgg_internal.h"
#include "pgg_ptx.cuh"

namespace pgg {
namespace {

constexpr int kOK = 128;          // k per CTA (the pair's MMA M is 256)
constexpr int kMaxRows = 128;     // rows per chunk (MMA N)
constexpr int kStages = 4;
constexpr int kABytes = kOK * kRowBytes;              // weight: 128 k x 128 bytes
constexpr int kBBytes = (kMaxRows / 2) * kRowBytes;   // this CTA's half of the rows
constexpr int kStageBytes = kABytes + kBBytes;
// slab accumulators: per epilogue warp [kMaxSlabTokens + 1 tokens][32 k] fp32;
// the last row takes the stores of the padding rows of a chunk
constexpr int kAccRows = kMaxSlabTokens + 1;
constexpr int kAccBytes = 4 * kAccRows * 32 * 4;
constexpr int kThreads = 32 * 6;
constexpr int kTmemCols = 256;
constexpr int kAccCols = 128;

struct OwnCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr int kSmemBytes =
    kStages * kStageBytes + kAccBytes + static_cast<int>(sizeof(OwnCtl)) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

__device__ __forceinline__ void raise_status(WsHeader* hdr, uint32_t code, uint32_t site) {
  if (atomicCAS(&hdr->status, 0u, code) == 0u) hdr->timeout_site = site;
}

__device__ __forceinline__ uint32_t cluster_id() { return blockIdx.x >> 1; }
__device__ __forceinline__ uint32_t n_clusters() { return gridDim.x >> 1; }

// MMA N for a chunk of R rows: a multiple of 32 (each CTA stages half).
__device__ __forceinline__ int mma_n(int R) { return (R + 31) / 32 * 32; }

// Walks the chunks of one unit (slab s, k range): experts in increasing
// order, each expert's slab rows in pieces of at most 256.
struct ChunkIt {
  const OwnerArgs* a;
  int64_t s;
  int64_t g;
  int64_t r0, r_end;
  __device__ void start(const OwnerArgs* args, int64_t slab) {
    a = args;
    s = slab;
    g = -1;
    r0 = r_end = 0;
    next_expert();
  }
  __device__ void next_expert() {
    while (++g < a->G) {
      const int32_t* row = a->seg + g * (a->n_slabs + 1);
      r0 = row[s];
      r_end = row[s + 1];
      if (r0 < r_end) return;
    }
  }
  __device__ bool valid() const { return g < a->G; }
  __device__ int rows() const {
    const int64_t left = r_end - r0;
    return static_cast<int>(left < kMaxRows ? left : kMaxRows);
  }
  __device__ void next() {
    r0 += rows();
    if (r0 >= r_end) next_expert();
  }
};

__device__ void producer(uint8_t* smem, OwnCtl* ctl, const DyMaps* dy, const CUtensorMap* tw,
                         const OwnerArgs& a, uint32_t n_units, uint32_t rank) {
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const bool leader = rank == 0;
  int stage = 0;
  uint32_t phase = 0, outstanding = 0, last_parity = 0;
  bool failed = false;
  for (uint32_t u = cluster_id(); u < n_units && !failed; u += n_clusters()) {
    const int64_t slab = u / a.k_units;
    const int32_t k0 = static_cast<int32_t>((u % a.k_units) * 2 * kOK + kOK * rank);
    ChunkIt c;
    for (c.start(&a, slab); c.valid() && !failed; c.next()) {
      const int nm = mma_n(c.rows());
      const int half = nm / 2;  // this CTA's rows: 16, 32, 48 or 64
      const uint32_t tx = 2u * static_cast<uint32_t>(kABytes + half * kRowBytes);
      const int32_t brow = static_cast<int32_t>(c.r0 + rank * half);
      for (int ks = 0; ks < a.nk; ++ks) {
        if (!ptx::mbar_wait_cluster(&ctl->empty[stage], phase ^ 1u, lim, abort)) {
          failed = true;
          break;
        }
        uint8_t* sa = smem + stage * kStageBytes;
        const uint32_t fb = ptx::mapa(&ctl->full[stage], 0);
        if (leader) ptx::mbar_arrive_expect_tx(&ctl->full[stage], tx);
        ptx::tma_load_3d_pair(sa, tw, fb, ks * 64, k0, static_cast<int32_t>(c.g));
        // the rows in boxes of 64, 32 and 16 rows (each box lands on a
        // 1024-byte boundary, so the 128-byte swizzle stays in phase)
        for (int r = 0; r < half;) {
          const int j = half - r >= 64 ? 2 : (half - r >= 32 ? 1 : 0);
          ptx::tma_load_2d_pair(sa + kABytes + r * kRowBytes, &dy->box[j], fb, ks * 64, brow + r);
          r += kDyMinRows << j;
        }
        outstanding |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }
  if (failed) {
    ctl->abort = 1;
    raise_status(a.hdr, kStTimeout, 32);
  }
  if (leader) {
    int no_abort = 0;
    for (int s = 0; s < kStages; ++s)
      if (outstanding & (1u << s))
        ptx::mbar_wait_cluster(&ctl->full[s], (last_parity >> s) & 1u, lim, &no_abort);
  }
}

template <int DT>
__device__ void mma_issuer(uint8_t* smem, OwnCtl* ctl, uint32_t tmem_base, const OwnerArgs& a,
                           uint32_t n_units) {
  constexpr uint32_t kFmt = DT == PGG_BF16 ? 1u : 0u;
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  int stage = 0, acc = 0;
  uint32_t phase = 0, aph = 0;
  bool issued = false, failed = false;
  for (uint32_t u = cluster_id(); u < n_units && !failed; u += n_clusters()) {
    ChunkIt c;
    for (c.start(&a, u / a.k_units); c.valid() && !failed; c.next()) {
      const uint32_t idesc = ptx::idesc_make(kFmt, 2 * kOK, static_cast<uint32_t>(mma_n(c.rows())));
      if (!ptx::mbar_wait_cluster(&ctl->tempty[acc], aph ^ 1u, lim, abort)) {
        failed = true;
        break;
      }
      ptx::tc_fence_after_sync();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
      for (int ks = 0; ks < a.nk; ++ks) {
        if (!ptx::mbar_wait_cluster(&ctl->full[stage], phase, lim, abort)) {
          failed = true;
          break;
        }
        ptx::tc_fence_after_sync();
        const uint32_t sa = ptx::smem_addr(smem + stage * kStageBytes);
        const uint64_t da = ptx::sdesc_sw128(sa);
        const uint64_t db = ptx::sdesc_sw128(sa + kABytes);
#pragma unroll
        for (int kk = 0; kk < kRowBytes / 32; ++kk) {
          const uint64_t koff = static_cast<uint64_t>((kk * 32) >> 4);
          ptx::mma_f16_pair(d_tmem, da + koff, db + koff, idesc, (ks | kk) != 0 ? 1u : 0u);
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
  }
  if (failed) {
    ctl->abort = 1;
    raise_status(a.hdr, kStTimeout, 34);
  }
  if (issued) {
    int no_abort = 0;
    ptx::mma_commit_pair(&ctl->drain, 0x1);
    ptx::mbar_wait(&ctl->drain, 0u, lim, &no_abort);
  }
}

// Row flags of the epilogue: bits 0-8 the accumulator row (the token within
// the slab, or kMaxSlabTokens for a padding row).
constexpr int kRowMask = 0x1FF;
constexpr int kRowFirst = 1 << 9;  // the token's first row: store, no load
constexpr int kRowDup = 1 << 10;   // same token as the row before, in this batch: carry

// Epilogue warp q (of 4) owns accumulator lanes 32 q .. 32 q + 31: one d_x
// column k each, for every token of the slab. Its accumulator block acc_q is
// [kAccRows][32 k] fp32 in shared memory.
__device__ void epilogue(OwnCtl* ctl, float* acc_q, uint32_t tmem_base, const OwnerArgs& a,
                         uint32_t n_units, uint32_t rank) {
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const uint32_t tempty0 = ptx::mapa(&ctl->tempty[0], 0);
  const uint32_t tempty1 = ptx::mapa(&ctl->tempty[1], 0);
  const int64_t K = a.K;
  const int T = a.slab_tokens;
  int acc = 0;
  uint32_t aph = 0;
  bool stop = false;
  for (uint32_t u = cluster_id(); u < n_units && !stop; u += n_clusters()) {
    const int64_t slab = u / a.k_units;
    const int64_t tok0 = slab * T;
    const int64_t k =
        static_cast<int64_t>(u % a.k_units) * 2 * kOK + kOK * rank + 32 * quarter + lane;
    ChunkIt c;
    for (c.start(&a, slab); c.valid(); c.next()) {
      const int R = c.rows();
      // lane j of info[b] describes row 32 b + j of the chunk (read before the
      // accumulator is ready: it does not depend on the MMA)
      int info[kMaxRows / 32];
#pragma unroll
      for (int b = 0; b < kMaxRows / 32; ++b) {
        int f = kMaxSlabTokens;
        const int r = 32 * b + lane;
        if (r < R) {
          const RowInfo ri = a.rowinfo[c.r0 + r];
          const int64_t t = static_cast<int64_t>(ri.token) - tok0;
          if (t >= 0 && t < T) f = static_cast<int>(t) | (ri.rank == 0 ? kRowFirst : 0);
        }
        const int before = __shfl_up_sync(0xFFFFFFFFu, f, 1);
        if (lane > 0 && (f & kRowMask) != kMaxSlabTokens && ((before ^ f) & kRowMask) == 0)
          f |= kRowDup;
        info[b] = f;
      }
      const bool ok = ptx::mbar_wait_cluster(&ctl->tfull[acc], aph, lim, abort);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        if (lane == 0) {
          ctl->abort = 1;
          raise_status(a.hdr, kStTimeout, 35);
        }
        stop = true;
        break;
      }
      ptx::tc_fence_after_sync();
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) +
                              static_cast<uint32_t>(acc * kAccCols);
#pragma unroll
      for (int b = 0; b < kMaxRows / 32; ++b) {
        if (32 * b >= R) break;
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(32 * b), v);
        int row[32];
        float old[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          row[j] = __shfl_sync(0xFFFFFFFFu, info[b], j);
          old[j] = acc_q[(row[j] & kRowMask) * 32 + lane];
        }
        ptx::tmem_ld_wait();
        if (!__any_sync(0xFFFFFFFFu, info[b] & kRowDup)) {
          // distinct tokens: independent updates (-0 + x == x for every x)
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float base = (row[j] & kRowFirst) ? -0.0f : old[j];
            acc_q[(row[j] & kRowMask) * 32 + lane] = base + __uint_as_float(v[j]);
          }
        } else {
          // a token twice in a row: carry its running sum
          float carry = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = __uint_as_float(v[j]);
            const float val =
                (row[j] & kRowFirst) ? x : ((row[j] & kRowDup) ? carry + x : old[j] + x);
            acc_q[(row[j] & kRowMask) * 32 + lane] = val;
            carry = val;
          }
        }
      }
      ptx::tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_remote(acc ? tempty1 : tempty0);
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    if (stop) break;
    // the slab is done: this thread's column to d_x (every token of the
    // slab has at least one row, so every element was stored above)
    int64_t nt = a.batch - tok0;
    if (nt > T) nt = T;
    if (k < K) {
      float* dst = a.out + tok0 * K + k;
#pragma unroll 8
      for (int t = 0; t < static_cast<int>(nt); ++t) dst[t * K] = acc_q[t * 32 + lane];
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 1)
    gmm_dx_owner_kernel(const __grid_constant__ DyMaps dy, const __grid_constant__ CUtensorMap tw,
                        const OwnerArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* accs = reinterpret_cast<float*>(smem + kStages * kStageBytes);
  auto* ctl = reinterpret_cast<OwnCtl*>(smem + kStages * kStageBytes + kAccBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();

  // Routing validation failed: the result is defined as zeros. Rows not in
  // increasing position: the ticketed kernel that follows does the work.
  // (Both CTAs of a pair see the same header.)
  const uint32_t st = a.hdr->status;
  if (st == kStIndex || st == kStGroupSum || st == kStNotPerm) {
    const int64_t n = a.batch * a.K;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < n;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x)
      a.out[q] = 0.0f;
    return;
  }
  if (a.hdr->unsorted) return;
  const uint32_t n_units = static_cast<uint32_t>(a.n_slabs) * static_cast<uint32_t>(a.k_units);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&ctl->full[s], 1);
      ptx::mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl->tfull[b], 1);
      ptx::mbar_init(&ctl->tempty[b], 8);
    }
    ptx::mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int j = 0; j < kDyMaps; ++j) ptx::tma_prefetch_desc(&dy.box[j]);
    ptx::tma_prefetch_desc(&tw);
  }
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
    if (lane == 0) producer(smem, ctl, &dy, &tw, a, n_units, rank);
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) mma_issuer<DT>(smem, ctl, tmem_base, a, n_units);
  } else {
    epilogue(ctl, accs + (warp & 3) * (kAccRows * 32), tmem_base, a, n_units, rank);
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

int owner_smem_bytes() { return kSmemBytes; }
int owner_threads() { return kThreads; }

cudaError_t launch_owner(int dtype, const DyMaps& dy, const CUtensorMap& tw, const OwnerArgs& a,
                         int num_sms, cudaStream_t stream) {
  void (*kern)(const DyMaps, const CUtensorMap, const OwnerArgs) = nullptr;
  if (dtype == PGG_BF16)
    kern = gmm_dx_owner_kernel<PGG_BF16>;
  else if (dtype == PGG_F16)
    kern = gmm_dx_owner_kernel<PGG_F16>;
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
  const int64_t units = static_cast<int64_t>(a.n_slabs) * a.k_units;
  int64_t want = units < num_sms / 2 ? units : num_sms / 2;
  if (want < 1) want = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * want), 1, 1);
  int clusters = 0;
  err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (err != cudaSuccess) return err;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (clusters < want ? clusters : want)), 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, dy, tw, a);
}

}  // namespace pgg
