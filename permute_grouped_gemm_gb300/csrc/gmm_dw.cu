// Weight gradient of the MoE grouped matmul on tcgen05 tensor cores:
//
//     d_weight[g, k, n] = sum over the expanded rows i of expert g of
//                         x[batch(i), k] * d_y[i, n]
//
// ("MoeInitRoutingGroupedMatmulGrad design", section 1.2, "为何不计算
// d_weight" item 3: the separate grouped matmul expanded_x^T @ d_y; section
// 1.1: expanded_x[i] = x[batch(i)], the forward's MoeInitRouting output.)
// expanded_x is never materialised: its rows are gathered from x by token
// while they are staged.
//
// Tile: one expert g, 128 output rows k (MMA M, tensor-memory lanes) x 256
// output columns n (MMA N), reduced over the expert's rows 64 at a time. Both
// operands are MN-major (the reduction index is the outer one in memory):
//   A = x rows of the expert's tokens, 64 rows x 128 k, gathered with 16-byte
//       cp.async by four producer warps into two 64-k panels of 128-byte rows
//       in the 128-byte swizzle layout (rows past the expert's end read as 0);
//   B = d_y rows of the expert, 64 rows x 256 n, by TMA: four 64-n boxes.
// The accumulator (fp32, 256 columns, two buffers) is written by four
// epilogue warps in the output dtype (the input dtype or fp32): each lane owns
// one k and stores its row segment of n. Every output element is produced by
// exactly one tile with a fixed order of MMAs, so the result is bitwise
// repeatable. An expert with no rows gets zeros.
//
// Warp roles (320 threads): 0 TMA for d_y; 1 tensor-memory allocation and MMA
// issue; 2-5 gather of x; 6-9 epilogue. Tiles are statically interleaved over
// the persistent grid (tile = blockIdx.x + j * gridDim.x), so every role walks
// the same list without a queue. Waits are bounded; when one runs out the
// kernel records PGG_ERR_TIMEOUT, drains its copies and MMAs, frees tensor
// memory and returns.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "pgg_internal.h"
#include "pgg_ptx.cuh"

namespace pgg {
namespace {

constexpr int kDwM = 128;      // output rows k per tile (MMA M)
constexpr int kDwN = 256;      // output columns n per tile (MMA N)
constexpr int kDwRows = 64;    // reduction rows per stage
constexpr int kDwStages = 4;
constexpr int kPanel = kDwRows * 128;            // one 64-element panel: 64 rows x 128 bytes
constexpr int kABytes = 2 * kPanel;              // x: 128 k
constexpr int kBBytes = 4 * kPanel;              // d_y: 256 n
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kGatherThreads = 128;
constexpr int kGatherLag = 2;                    // cp.async groups in flight per gather thread
constexpr int kThreads = 320;
constexpr int kTmemCols = 512;                   // two 256-column accumulators
constexpr int kAccCols = 256;

static_assert(kGatherLag <= kDwStages - 1, "gather lag must leave a stage to the consumer");

struct DwCtl {
  uint64_t full_b[kDwStages];  // d_y copies landed (TMA transaction bytes)
  uint64_t full_a[kDwStages];  // x gathered (128 arrivals)
  uint64_t empty[kDwStages];   // MMAs of the stage done
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr int kSmemBytes = kDwStages * kStageBytes + static_cast<int>(sizeof(DwCtl)) + 1024;

__device__ __forceinline__ void raise_status(WsHeader* hdr, uint32_t code, uint32_t site) {
  if (atomicCAS(&hdr->status, 0u, code) == 0u) hdr->timeout_site = site;
}

struct Tile {
  int64_t g, k0, n0, row0, m;
};

__device__ __forceinline__ Tile tile_of(uint32_t t, const DwArgs& a) {
  const uint32_t per_g = static_cast<uint32_t>(a.k_blocks) * static_cast<uint32_t>(a.n_blocks);
  Tile x;
  x.g = t / per_g;
  const uint32_t rem = t - static_cast<uint32_t>(x.g) * per_g;
  x.k0 = static_cast<int64_t>(rem / a.n_blocks) * kDwM;
  x.n0 = static_cast<int64_t>(rem % a.n_blocks) * kDwN;
  x.row0 = a.off[x.g];
  x.m = a.off[x.g + 1] - x.row0;
  return x;
}

__device__ void dy_producer(uint8_t* smem, DwCtl* ctl, const CUtensorMap* tm_dy, const DwArgs& a,
                            uint32_t total) {
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  int stage = 0;
  uint32_t phase = 0, outstanding = 0, last_parity = 0;
  bool failed = false;
  for (uint32_t t = blockIdx.x; t < total && !failed; t += gridDim.x) {
    const Tile x = tile_of(t, a);
    int boxes = 0;
    for (int j = 0; j < kDwN / 64; ++j) boxes += (x.n0 + 64 * j < a.N) ? 1 : 0;
    for (int64_t r = 0; r < x.m; r += kDwRows) {
      if (!ptx::mbar_wait(&ctl->empty[stage], phase ^ 1u, lim, abort)) {
        failed = true;
        break;
      }
      uint8_t* sb = smem + stage * kStageBytes + kABytes;
      ptx::mbar_arrive_expect_tx(&ctl->full_b[stage], static_cast<uint32_t>(boxes * kPanel));
      for (int j = 0; j < boxes; ++j)
        ptx::tma_load_2d(sb + j * kPanel, tm_dy, &ctl->full_b[stage],
                         static_cast<int32_t>(x.n0 + 64 * j), static_cast<int32_t>(x.row0 + r));
      outstanding |= 1u << stage;
      last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == kDwStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (failed) {
    ctl->abort = 1;
    raise_status(a.hdr, kStTimeout, 12);
  }
  // Never leave while a copy into this CTA's shared memory may be in flight.
  int no_abort = 0;
  for (int s = 0; s < kDwStages; ++s)
    if (outstanding & (1u << s))
      ptx::mbar_wait(&ctl->full_b[s], (last_parity >> s) & 1u, lim, &no_abort);
}

// The sequence of (tile, first row) stages a CTA works through: tiles
// blockIdx.x + j * gridDim.x, experts with no rows skipped, 64 rows a stage.
struct StageIt {
  uint32_t t;
  int64_t r;
  Tile x;
  bool valid;
};

__device__ __forceinline__ void stage_seek(StageIt& s, const DwArgs& a, uint32_t total) {
  while (s.t < total) {
    s.x = tile_of(s.t, a);
    if (s.r < s.x.m) {
      s.valid = true;
      return;
    }
    s.t += gridDim.x;
    s.r = 0;
  }
  s.valid = false;
}

__device__ __forceinline__ StageIt stage_first(const DwArgs& a, uint32_t total) {
  StageIt s;
  s.t = blockIdx.x;
  s.r = 0;
  stage_seek(s, a, total);
  return s;
}

__device__ __forceinline__ StageIt stage_next(StageIt s, const DwArgs& a, uint32_t total) {
  if (!s.valid) return s;
  s.r += kDwRows;
  stage_seek(s, a, total);
  return s;
}

// Tokens of this thread's 8 rows (rr0 + 8 j) of a stage; -1 past the expert's end.
__device__ __forceinline__ void stage_tokens(const StageIt& s, const DwArgs& a, int rr0,
                                             int32_t (&tok)[kDwRows / 8]) {
#pragma unroll
  for (int j = 0; j < kDwRows / 8; ++j) {
    const int64_t r = s.r + rr0 + 8 * j;
    tok[j] = (s.valid && r < s.x.m) ? a.rowinfo[s.x.row0 + r].token : -1;
  }
}

template <int DT>
__device__ void x_gatherer(uint8_t* smem, DwCtl* ctl, const DwArgs& a, uint32_t total) {
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int gt = threadIdx.x - 64;        // 0 .. 127
  const int kc = gt & 15;                 // 16-byte chunk of the 128 k: 8 elements
  const int rr0 = gt >> 4;                // rows rr0 + 8 j
  const char* xb = static_cast<const char*>(a.x);
  int stage = 0;
  uint32_t phase = 0;
  int pend[kGatherLag + 1];
  int npend = 0;
  bool failed = false;
  // The row tokens (the gather addresses) are loaded two stages ahead, so
  // that their latency is not paid before every stage's copies.
  StageIt cur = stage_first(a, total);
  StageIt nxt = stage_next(cur, a, total);
  int32_t tok0[kDwRows / 8], tok1[kDwRows / 8], tok2[kDwRows / 8];
  stage_tokens(cur, a, rr0, tok0);
  stage_tokens(nxt, a, rr0, tok1);
  while (cur.valid) {
    const StageIt nn = stage_next(nxt, a, total);
    stage_tokens(nn, a, rr0, tok2);
    if (!ptx::mbar_wait(&ctl->empty[stage], phase ^ 1u, lim, abort)) {
      failed = true;
      break;
    }
    const int64_t k = cur.x.k0 + kc * 8;
    const bool k_ok = k < a.K;
    const uint32_t sa = ptx::smem_addr(smem + stage * kStageBytes) + (kc >> 3) * kPanel;
#pragma unroll
    for (int j = 0; j < kDwRows / 8; ++j) {
      const int rr = rr0 + 8 * j;
      const bool ok = k_ok && tok0[j] >= 0;
      const void* src = ok ? static_cast<const void*>(xb + (static_cast<int64_t>(tok0[j]) * a.K + k) * 2)
                           : static_cast<const void*>(xb);
      ptx::cp_async_16(sa + rr * 128 + (((kc & 7) ^ (rr & 7)) << 4), src, ok ? 16u : 0u);
    }
    ptx::cp_async_commit();
    pend[npend++] = stage;
    if (npend > kGatherLag) {
      // the oldest stage's copies are complete: make them visible to the
      // tensor cores, then report them
      ptx::cp_async_wait<kGatherLag>();
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(&ctl->full_a[pend[0]]);
      for (int q = 0; q < kGatherLag; ++q) pend[q] = pend[q + 1];
      --npend;
    }
    if (++stage == kDwStages) {
      stage = 0;
      phase ^= 1u;
    }
    cur = nxt;
    nxt = nn;
#pragma unroll
    for (int j = 0; j < kDwRows / 8; ++j) {
      tok0[j] = tok1[j];
      tok1[j] = tok2[j];
    }
  }
  ptx::cp_async_wait<0>();
  ptx::fence_proxy_async_smem();
  for (int q = 0; q < npend; ++q) ptx::mbar_arrive(&ctl->full_a[pend[q]]);
  if (failed) {
    ctl->abort = 1;
    raise_status(a.hdr, kStTimeout, 13);
  }
}

template <int DT>
__device__ void mma_issuer(uint8_t* smem, DwCtl* ctl, uint32_t tmem_base, const DwArgs& a,
                           uint32_t total) {
  constexpr uint32_t kFmt = DT == PGG_BF16 ? 1u : 0u;
  constexpr uint32_t idesc = ptx::idesc_make_mn(kFmt, kDwM, kDwN);
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  int stage = 0, acc = 0;
  uint32_t phase = 0, aph = 0;
  bool issued = false, failed = false;
  for (uint32_t t = blockIdx.x; t < total && !failed; t += gridDim.x) {
    const Tile x = tile_of(t, a);
    if (x.m == 0) continue;
    if (!ptx::mbar_wait(&ctl->tempty[acc], aph ^ 1u, lim, abort)) {
      failed = true;
      break;
    }
    ptx::tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
    for (int64_t r = 0; r < x.m; r += kDwRows) {
      if (!ptx::mbar_wait(&ctl->full_b[stage], phase, lim, abort) ||
          !ptx::mbar_wait(&ctl->full_a[stage], phase, lim, abort)) {
        failed = true;
        break;
      }
      ptx::tc_fence_after_sync();
      const uint32_t sa = ptx::smem_addr(smem + stage * kStageBytes);
      const uint64_t da = ptx::sdesc_sw128_mn(sa, kPanel);
      const uint64_t db = ptx::sdesc_sw128_mn(sa + kABytes, kPanel);
      const int64_t left = x.m - r;
      const int nks = left >= kDwRows ? kDwRows / 16 : static_cast<int>((left + 15) / 16);
      for (int ks = 0; ks < nks; ++ks) {
        const uint64_t koff = static_cast<uint64_t>((ks * 16 * 128) >> 4);
        ptx::mma_f16(d_tmem, da + koff, db + koff, idesc, (r > 0 || ks > 0) ? 1u : 0u);
      }
      issued = true;
      ptx::mma_commit(&ctl->empty[stage]);
      if (++stage == kDwStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (failed) break;
    ptx::mma_commit(&ctl->tfull[acc]);
    acc ^= 1;
    if (acc == 0) aph ^= 1u;
  }
  if (failed) {
    ctl->abort = 1;
    raise_status(a.hdr, kStTimeout, 14);
  }
  if (issued) {
    // Tensor memory is released only after every issued MMA has completed.
    int no_abort = 0;
    ptx::mma_commit(&ctl->drain);
    ptx::mbar_wait(&ctl->drain, 0u, lim, &no_abort);
  }
}

// 8 fp32 values -> 16 bytes of the 16-bit output dtype.
template <int DT>
__device__ __forceinline__ uint4 pack8(const uint32_t* v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(v[2 * i]), hi = __uint_as_float(v[2 * i + 1]);
    if constexpr (DT == PGG_BF16) {
      const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
      w[i] = *reinterpret_cast<const uint32_t*>(&p);
    } else {
      const __half2 p = __floats2half2_rn(lo, hi);
      w[i] = *reinterpret_cast<const uint32_t*>(&p);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int DT>
__device__ void epilogue(DwCtl* ctl, uint32_t tmem_base, const DwArgs& a, uint32_t total) {
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;  // tensor-memory lanes 32 q .. 32 q + 31 are this warp's
  const bool f32 = a.out_f32 != 0;
  int acc = 0;
  uint32_t aph = 0;
  for (uint32_t t = blockIdx.x; t < total; t += gridDim.x) {
    const Tile x = tile_of(t, a);
    const int64_t k = x.k0 + 32 * quarter + lane;
    const bool k_ok = k < a.K;
    const int64_t base = (x.g * a.K + k) * a.N + x.n0;
    if (x.m == 0) {
      if (k_ok) {
        if (f32) {
          float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + base);
          for (int c = 0; c < kDwN / 4 && x.n0 + 4 * c < a.N; ++c) o[c] = make_float4(0, 0, 0, 0);
        } else {
          uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + base);
          for (int c = 0; c < kDwN / 8 && x.n0 + 8 * c < a.N; ++c) o[c] = make_uint4(0, 0, 0, 0);
        }
      }
      continue;
    }
    const bool ok = ptx::mbar_wait(&ctl->tfull[acc], aph, lim, abort);
    if (!__all_sync(0xFFFFFFFFu, ok)) {
      if (lane == 0) {
        ctl->abort = 1;
        raise_status(a.hdr, kStTimeout, 15);
      }
      break;
    }
    ptx::tc_fence_after_sync();
    const uint32_t t_lane =
        tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) + static_cast<uint32_t>(acc * kAccCols);
#pragma unroll 1
    for (int c = 0; c < kDwN / 32; ++c) {
      uint32_t v[32];
      ptx::tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(32 * c), v);
      ptx::tmem_ld_wait();
      const int64_t n = x.n0 + 32 * c;
      if (!k_ok || n >= a.N) continue;
      if (f32) {
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + base + 32 * c);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (n + 4 * q < a.N)
            o[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                               __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
      } else {
        uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + base + 32 * c);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (n + 8 * q < a.N) o[q] = pack8<DT>(v + 8 * q);
      }
    }
    ptx::tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&ctl->tempty[acc]);
    acc ^= 1;
    if (acc == 0) aph ^= 1u;
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 1)
    gmm_dw_kernel(const __grid_constant__ CUtensorMap tm_dy, const DwArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  auto* ctl = reinterpret_cast<DwCtl*>(smem + kDwStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Routing validation failed: the result is defined as zeros.
  const uint32_t st = a.hdr->status;
  if (st == kStIndex || st == kStGroupSum || st == kStNotPerm) {
    const int64_t n = a.G * a.K * a.N;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < n;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      if (a.out_f32)
        static_cast<float*>(a.out)[q] = 0.0f;
      else
        static_cast<uint16_t*>(a.out)[q] = 0;
    }
    return;
  }
  const uint32_t total =
      static_cast<uint32_t>(a.G) * static_cast<uint32_t>(a.k_blocks) * static_cast<uint32_t>(a.n_blocks);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDwStages; ++s) {
      ptx::mbar_init(&ctl->full_b[s], 1);
      ptx::mbar_init(&ctl->full_a[s], kGatherThreads);
      ptx::mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl->tfull[b], 1);
      ptx::mbar_init(&ctl->tempty[b], 4);
    }
    ptx::mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) ptx::tma_prefetch_desc(&tm_dy);
  if (warp == 1) {
    ptx::tmem_alloc(&ctl->tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) dy_producer(smem, ctl, &tm_dy, a, total);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<DT>(smem, ctl, tmem_base, a, total);
  } else if (warp < 6) {
    x_gatherer<DT>(smem, ctl, a, total);
  } else {
    epilogue<DT>(ctl, tmem_base, a, total);
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

int dw_smem_bytes() { return kSmemBytes; }
int dw_threads() { return kThreads; }

// Tiles of 128 k x 256 n per expert.
void dw_tiles(int64_t K, int64_t N, int* k_blocks, int* n_blocks) {
  *k_blocks = static_cast<int>((K + kDwM - 1) / kDwM);
  *n_blocks = static_cast<int>((N + kDwN - 1) / kDwN);
}

cudaError_t launch_dw(int dtype, const CUtensorMap& tm_dy, const DwArgs& a, int num_sms,
                      cudaStream_t stream) {
  void (*kern)(const CUtensorMap, const DwArgs) = nullptr;
  if (dtype == PGG_BF16)
    kern = gmm_dw_kernel<PGG_BF16>;
  else if (dtype == PGG_F16)
    kern = gmm_dw_kernel<PGG_F16>;
  else
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
  if (err != cudaSuccess) return err;
  const int64_t total = a.G * a.k_blocks * a.n_blocks;
  const int64_t grid = total < num_sms ? total : num_sms;
  kern<<<static_cast<unsigned>(grid < 1 ? 1 : grid), kThreads, kSmemBytes, stream>>>(tm_dy, a);
  return cudaGetLastError();
}

}  // namespace pgg
