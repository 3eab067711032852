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
// Tile: one expert g, 256 output rows k (MMA M) x 256 output columns n (MMA
// N), on a pair of CTAs (a cluster of two; tcgen05 cta_group::2), reduced
// over the expert's rows 64 at a time. CTA r owns k rows 128 r .. 128 r + 127
// of the tile: their accumulators (fp32, 128 lanes x 256 columns, two
// buffers) live in its tensor memory. Both operands are MN-major (the
// reduction index is the outer one in memory):
//   A = x rows of the expert's tokens: each CTA gathers its 128 k of the 64
//       rows with 16-byte cp.async into two 64-k panels of 128-byte rows in the
//       128-byte swizzle layout (rows past the expert's end read as 0), one
//       producer warp per stage slot so that every slot can be in flight;
//   B = d_y rows of the expert: each CTA loads its half of the 256 n (two
//       64-n panels) by TMA, one copy through a 3-D view {64 n, rows, n / 64}
//       when N is a multiple of 64, else one 2-D box per panel. When the d_y
//       rows are not a multiple of 16 bytes (N even, not a multiple of 8),
//       the gather warps copy the panels instead, one 128-byte row segment
//       per warp instruction, 4 bytes per lane, into the same swizzled
//       layout, and the epilogue writes with 4-byte stores.
// Per SM a stage is 32 KB, so six stages fit: enough tensor work buffered to
// cover the round trip of a stage (MMA done -> slot free -> copies -> slot
// full). The even CTA issues the MMAs; completions are multicast to both.
// Every output element is produced by exactly one tile with a fixed order of
// MMAs, so the result is bitwise repeatable. An expert with no rows gets
// zeros. The epilogue warps write the output dtype (the input dtype or fp32)
// through shared memory with TMA stores.
//
// Warp roles per CTA: 0 TMA for d_y; 1 tensor-memory allocation and (even
// CTA) MMA issue; one gather warp per stage slot; eight epilogue warps. Tiles
// are statically interleaved over the clusters (tile = cluster + j *
// clusters), so every role walks the same list without a queue. Waits are
// bounded; when one runs out the kernel records PGG_ERR_TIMEOUT, drains its
// copies and MMAs, frees tensor memory and returns.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "pgg_epilogue.cuh"
#include "pgg_gather.cuh"
#include "pgg_internal.h"
#include "pgg_ptx.cuh"

namespace pgg {
namespace {

constexpr int kDwM = 128;      // output rows k per CTA (the pair's MMA M is 256)
constexpr int kDwN = 256;      // output columns n per tile (MMA N)
constexpr int kDwRows = 64;    // reduction rows per stage
constexpr int kDwStages = 6;   // shared-memory stage slots, one gather warp each
constexpr int kPanel = kDwRows * 128;            // one 64-element panel: 64 rows x 128 bytes
constexpr int kABytes = 2 * kPanel;              // x: this CTA's 128 k
constexpr int kBBytes = 2 * kPanel;              // d_y: this CTA's 128 n
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kGatherWarps = kDwStages;          // one per stage slot
constexpr int kEpiWarps = 8;                     // 4: one per lane quarter; 8: also split n in two
constexpr int kOutBufs = 1;                      // staging buffers per epilogue warp
constexpr int kEpiWarp0 = 2 + kGatherWarps;      // first epilogue warp
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kTmemCols = 512;                   // two 256-column accumulators
constexpr int kAccCols = 256;
constexpr int kOutBuf = 32 * 128;                // epilogue staging: 32 rows x 128 bytes
constexpr int kOutBytes = kEpiWarps * kOutBufs * kOutBuf;

static_assert(kDwRows == 64, "the gather lane layout assumes 64 rows per stage");

struct DwCtl {
  uint64_t full[kDwStages];    // even CTA: stage ready: d_y bytes of both CTAs (with the even
                               // CTA's expect-tx arrival) and x gathered in both (two arrivals)
  uint64_t empty[kDwStages];   // each CTA: MMAs of the stage done (multicast commit)
  uint64_t tfull[2];           // each CTA: accumulator ready (multicast commit)
  uint64_t tempty[2];          // even CTA: accumulator drained (epilogue warps x 2 CTAs)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr int kSmemBytes =
    kDwStages * kStageBytes + kOutBytes + static_cast<int>(sizeof(DwCtl)) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

__device__ __forceinline__ void raise_status(WsHeader* hdr, uint32_t code, uint32_t site) {
  if (atomicCAS(&hdr->status, 0u, code) == 0u) hdr->timeout_site = site;
}

struct Tile {
  int64_t g, k0, n0, row0, m;  // k0: this CTA's first k; n0: the tile's first n
};

__device__ __forceinline__ Tile tile_of(uint32_t t, const DwArgs& a, uint32_t rank) {
  const uint32_t per_g = static_cast<uint32_t>(a.k_blocks) * static_cast<uint32_t>(a.n_blocks);
  Tile x;
  x.g = t / per_g;
  const uint32_t rem = t - static_cast<uint32_t>(x.g) * per_g;
  x.k0 = static_cast<int64_t>(rem / a.n_blocks) * (2 * kDwM) + kDwM * rank;
  x.n0 = static_cast<int64_t>(rem % a.n_blocks) * kDwN;
  x.row0 = a.off[x.g];
  x.m = a.off[x.g + 1] - x.row0;
  return x;
}

__device__ __forceinline__ uint32_t cluster_id() { return blockIdx.x >> 1; }
__device__ __forceinline__ uint32_t n_clusters() { return gridDim.x >> 1; }

// Bytes of d_y the CTA of `rank` stages for a tile starting at n0.
__device__ __forceinline__ uint32_t b_bytes(const DwArgs& a, int64_t n0, uint32_t rank) {
  const int64_t nc = n0 + 128 * rank;
  if (a.dy_3d) return nc < a.N ? static_cast<uint32_t>(kBBytes) : 0u;
  uint32_t b = 0;
  for (int j = 0; j < 2; ++j) b += (nc + 64 * j < a.N) ? static_cast<uint32_t>(kPanel) : 0u;
  return b;
}

__device__ void dy_producer(uint8_t* smem, DwCtl* ctl, const CUtensorMap* tm_dy, const DwArgs& a,
                            uint32_t total, uint32_t rank) {
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const bool leader = rank == 0;
  int stage = 0;
  uint32_t phase = 0, outstanding = 0, last_parity = 0;
  bool failed = false;
  for (uint32_t t = cluster_id(); t < total && !failed; t += n_clusters()) {
    const Tile x = tile_of(t, a, rank);
    // gathered d_y rows: the arrival carries no bytes
    const uint32_t mine = a.gather_dy ? 0u : b_bytes(a, x.n0, rank);
    const uint32_t both = a.gather_dy ? 0u : b_bytes(a, x.n0, 0) + b_bytes(a, x.n0, 1);
    const int64_t nc = x.n0 + 128 * rank;
    for (int64_t r = 0; r < x.m; r += kDwRows) {
      if (!ptx::mbar_wait_cluster(&ctl->empty[stage], phase ^ 1u, lim, abort)) {
        failed = true;
        break;
      }
      uint8_t* sb = smem + stage * kStageBytes + kABytes;
      const uint32_t fb = ptx::mapa(&ctl->full[stage], 0);
      if (leader) ptx::mbar_arrive_expect_tx(&ctl->full[stage], both);
      if (mine) {
        if (a.dy_3d) {
          ptx::tma_load_3d_pair(sb, tm_dy, fb, 0, static_cast<int32_t>(x.row0 + r),
                                static_cast<int32_t>(nc / 64));
        } else {
          for (int j = 0; j < 2; ++j)
            if (nc + 64 * j < a.N)
              ptx::tma_load_2d_pair(sb + j * kPanel, tm_dy, fb, static_cast<int32_t>(nc + 64 * j),
                                    static_cast<int32_t>(x.row0 + r));
        }
      }
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
  // Never leave while a copy into either CTA's shared memory may be in flight:
  // the even CTA's full barriers count both CTAs' bytes; the odd CTA is held
  // by the cluster barrier at the end of the kernel.
  if (leader) {
    int no_abort = 0;
    for (int s = 0; s < kDwStages; ++s)
      if (outstanding & (1u << s))
        ptx::mbar_wait_cluster(&ctl->full[s], (last_parity >> s) & 1u, lim, &no_abort);
  }
}

// The sequence of (tile, first row) stages a CTA works through: its
// cluster's tiles, experts with no rows skipped, 64 rows a stage.
struct StageIt {
  uint32_t t;
  int64_t r;
  Tile x;
  bool valid;
};

__device__ __forceinline__ void stage_seek(StageIt& s, const DwArgs& a, uint32_t total,
                                           uint32_t rank) {
  while (s.t < total) {
    if (s.r == 0) s.x = tile_of(s.t, a, rank);
    if (s.r < s.x.m) {
      s.valid = true;
      return;
    }
    s.t += n_clusters();
    s.r = 0;
  }
  s.valid = false;
}

__device__ __forceinline__ StageIt stage_first(const DwArgs& a, uint32_t total, uint32_t rank) {
  StageIt s;
  s.t = cluster_id();
  s.r = 0;
  stage_seek(s, a, total, rank);
  return s;
}

__device__ __forceinline__ StageIt stage_next(StageIt s, const DwArgs& a, uint32_t total,
                                              uint32_t rank) {
  if (!s.valid) return s;
  s.r += kDwRows;
  if (s.r >= s.x.m) {
    s.t += n_clusters();
    s.r = 0;
  }
  stage_seek(s, a, total, rank);
  return s;
}

// Tokens of rows `lane` and `lane + 32` of a stage; -1 past the expert's end.
__device__ __forceinline__ void stage_tokens(const StageIt& s, const DwArgs& a, int lane,
                                             int32_t (&tok)[2]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int64_t r = s.r + lane + 32 * h;
    tok[h] = (s.valid && r < s.x.m)
                 ? static_cast<int32_t>(check_index(
                       a.hdr, a.rowinfo[check_index(a.hdr, s.x.row0 + r, a.M, 60)].token,
                       a.batch, 61))
                 : -1;
  }
}

// Gather warp w fills shared-memory stage slot w: the stages w, w + S, ... of
// the sequence. It issues the slot's 64 rows x 128 k as 16-byte cp.async
// copies (32 per lane), waits for its own copies, makes them visible to the
// tensor cores and reports the slot full to the even CTA; meanwhile the other
// warps have their slots in flight. The tokens of the warp's next stage are
// loaded while its copies are in flight.
template <int DT>
__device__ void x_gatherer(uint8_t* smem, DwCtl* ctl, const DwArgs& a, uint32_t total,
                           uint32_t rank) {
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int w = (threadIdx.x >> 5) - 2;   // the warp's stage slot
  const int lane = threadIdx.x & 31;
  const int kc = lane & 15;               // 16-byte chunk of the 128 k: 8 elements
  const char* xb = static_cast<const char*>(a.x);
  const uint32_t sa_slot = ptx::smem_addr(smem + w * kStageBytes) + (kc >> 3) * kPanel;
  const uint32_t full = ptx::mapa(&ctl->full[w], 0);
  uint32_t phase = 0;
  bool failed = false;
  StageIt cur = stage_first(a, total, rank);
  for (int i = 0; i < w; ++i) cur = stage_next(cur, a, total, rank);
  int32_t tok[2];
  stage_tokens(cur, a, lane, tok);
  while (cur.valid) {
    StageIt nxt = cur;
    for (int i = 0; i < kDwStages; ++i) nxt = stage_next(nxt, a, total, rank);
    if (!ptx::mbar_wait_cluster(&ctl->empty[w], phase ^ 1u, lim, abort)) {
      failed = true;
      break;
    }
    const int64_t k = cur.x.k0 + kc * 8;
    const bool k_ok = k < a.K;
#pragma unroll
    for (int j = 0; j < kDwRows / 2; ++j) {
      const int rr = (lane >> 4) + 2 * j;  // row of the stage this copy fills
      const int32_t t = __shfl_sync(0xFFFFFFFFu, tok[rr >> 5], rr & 31);
      const bool ok = k_ok && t >= 0;
      const void* src = ok ? static_cast<const void*>(xb + (static_cast<int64_t>(t) * a.K + k) * 2)
                           : static_cast<const void*>(xb);
      ptx::cp_async_16(sa_slot + rr * 128 + (((kc & 7) ^ (rr & 7)) << 4), src, ok ? 16u : 0u);
    }
    if (a.gather_dy) {
      // the d_y panels: the stage's 64 rows of the expert, this CTA's 128 n,
      // copied as wide as each row's alignment allows, zeros past the
      // expert's rows and past N
      const char* yb = static_cast<const char*>(a.dy);
      const int64_t rows_left = cur.x.m - cur.r;
      const int nrows = rows_left < kDwRows ? static_cast<int>(rows_left) : kDwRows;
      const uint32_t sb_slot = ptx::smem_addr(smem + w * kStageBytes) + kABytes;
#pragma unroll 1
      for (int p = 0; p < 2; ++p) {
        const int64_t n = cur.x.n0 + 128 * rank + 64 * p;
        const int64_t left = (a.N - n) * 2;
        const int seg = left < 0 ? 0 : (left < 128 ? static_cast<int>(left) : 128);
        gather_rows_sw128(sb_slot + p * kPanel, yb + ((cur.x.row0 + cur.r) * a.N + n) * 2,
                          a.N * 2, kDwRows, nrows, seg, a.hdr, lane, 0, 1);
      }
    }
    ptx::cp_async_commit();
    stage_tokens(nxt, a, lane, tok);
    ptx::cp_async_wait<0>();
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_remote(full);
    phase ^= 1u;
    cur = nxt;
  }
  ptx::cp_async_wait<0>();
  if (failed) {
    ctl->abort = 1;
    if (lane == 0) raise_status(a.hdr, kStTimeout, 13);
  }
}

template <int DT>
__device__ void mma_issuer(uint8_t* smem, DwCtl* ctl, uint32_t tmem_base, const DwArgs& a,
                           uint32_t total) {
  constexpr uint32_t kFmt = DT == PGG_BF16 ? 1u : 0u;
  constexpr uint32_t idesc = ptx::idesc_make_mn(kFmt, 2 * kDwM, kDwN);
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  int stage = 0, acc = 0;
  uint32_t phase = 0, aph = 0;
  bool issued = false, failed = false;
  for (uint32_t t = cluster_id(); t < total && !failed; t += n_clusters()) {
    const Tile x = tile_of(t, a, 0);
    if (x.m == 0) continue;
    if (!ptx::mbar_wait_cluster(&ctl->tempty[acc], aph ^ 1u, lim, abort)) {
      failed = true;
      break;
    }
    ptx::tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
    for (int64_t r = 0; r < x.m; r += kDwRows) {
      if (!ptx::mbar_wait_cluster(&ctl->full[stage], phase, lim, abort)) {
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
        ptx::mma_f16_pair(d_tmem, da + koff, db + koff, idesc, (r > 0 || ks > 0) ? 1u : 0u);
      }
      issued = true;
      ptx::mma_commit_pair(&ctl->empty[stage], 0x3);
      if (++stage == kDwStages) {
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
    raise_status(a.hdr, kStTimeout, 14);
  }
  if (issued) {
    // Tensor memory is released only after every issued MMA has completed.
    int no_abort = 0;
    ptx::mma_commit_pair(&ctl->drain, 0x1);
    ptx::mbar_wait(&ctl->drain, 0u, lim, &no_abort);
  }
}

// Rows of 128 bytes of the output chunk: 64 values of the 16-bit dtype or 32
// of fp32, converted from the accumulator words v.
template <int DT>
__device__ __forceinline__ void stage_row(uint8_t* buf, int row, const uint32_t* v, bool f32) {
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    uint4 q;
    if (f32)
      q = make_uint4(v[4 * p], v[4 * p + 1], v[4 * p + 2], v[4 * p + 3]);
    else
      q = pack8<DT>(v + 8 * p);
    // 128-byte swizzle: 16-byte piece p of row r sits at piece p ^ (r % 8)
    *reinterpret_cast<uint4*>(buf + row * 128 + ((p ^ (row & 7)) << 4)) = q;
  }
}

// Each epilogue warp owns 32 accumulator lanes (k) of its CTA and, with eight
// warps, half of the tile's columns. Per tile it reads the accumulator in
// chunks of 128 bytes per row (64 columns of a 16-bit output, 32 of fp32),
// converts them into a shared-memory buffer in the 128-byte swizzle layout
// and writes the 32 x 128-byte box with one TMA store (rows past K and
// columns past N are clipped by the tensor map).
template <int DT>
__device__ void epilogue(uint8_t* obuf, DwCtl* ctl, uint32_t tmem_base, const CUtensorMap* tm_out,
                         const DwArgs& a, uint32_t total, uint32_t rank) {
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;  // tensor-memory lanes 32 q .. 32 q + 31 are this warp's
  const int e = warp - kEpiWarp0;
  const int span = kDwN / (kEpiWarps / 4);      // accumulator columns this warp writes
  const int col0 = (e / 4) * span;
  const bool f32 = a.out_f32 != 0;
  const int cols = f32 ? 32 : 64;  // output columns per 128-byte chunk
  uint8_t* bufs = obuf + e * kOutBufs * kOutBuf;
  const uint32_t tempty0 = ptx::mapa(&ctl->tempty[0], 0);
  const uint32_t tempty1 = ptx::mapa(&ctl->tempty[1], 0);
  int acc = 0, nb = 0;
  uint32_t aph = 0;
  bool held = a.hold_release != 0;  // (test hook: the first release is withheld)
  for (uint32_t t = cluster_id(); t < total; t += n_clusters()) {
    const Tile x = tile_of(t, a, rank);
    const int64_t k = x.k0 + 32 * quarter + lane;
    const bool k_ok = k < a.K;
    if (x.m == 0) {
      if (k_ok && a.gather_dy) {
        // rows not 16-byte aligned: 4-byte zeros (N is even)
        const int64_t n0 = x.n0 + col0;
        uint32_t* o = reinterpret_cast<uint32_t*>(static_cast<char*>(a.out) +
                                                  ((x.g * a.K + k) * a.N + n0) * (f32 ? 4 : 2));
        const int per = f32 ? 1 : 2;  // elements per 4-byte word
        for (int c = 0; c < span / per && n0 + per * c < a.N; ++c) o[c] = 0u;
      } else if (k_ok) {
        const int64_t n0 = x.n0 + col0;
        const int64_t base = (x.g * a.K + k) * a.N + n0;
        if (f32) {
          float4* o = reinterpret_cast<float4*>(static_cast<float*>(a.out) + base);
          for (int c = 0; c < span / 4 && n0 + 4 * c < a.N; ++c) o[c] = make_float4(0, 0, 0, 0);
        } else {
          uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + base);
          for (int c = 0; c < span / 8 && n0 + 8 * c < a.N; ++c) o[c] = make_uint4(0, 0, 0, 0);
        }
      }
      continue;
    }
    const bool ok = ptx::mbar_wait_cluster(&ctl->tfull[acc], aph, lim, abort);
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
    const int32_t k_row = static_cast<int32_t>(x.k0 + 32 * quarter);
#pragma unroll 1
    for (int c0 = col0; c0 < col0 + span && x.n0 + c0 < a.N; c0 += cols) {
      uint32_t v[64];
      ptx::tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(c0),
                              *reinterpret_cast<uint32_t(*)[32]>(v));
      if (!f32)
        ptx::tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(c0 + 32),
                                *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      ptx::tmem_ld_wait();
      uint8_t* buf = bufs + (nb % kOutBufs) * kOutBuf;
      // the store issued kOutBufs chunks ago read this buffer: wait for it
      if (lane == 0) ptx::bulk_wait_read<kOutBufs - 1>();
      __syncwarp();
      stage_row<DT>(buf, lane, v, f32);
      if (a.gather_dy) {
        // rows of N * 2 (or 4) bytes that are not 16-byte multiples: 4 bytes per
        // lane, one 128-byte row segment per warp instruction, rows below K
        // and columns below N only
        __syncwarp();
        const int64_t col = x.n0 + c0 + lane * (f32 ? 1 : 2);
        const uint32_t off = ((static_cast<uint32_t>(lane) >> 2) << 4) | ((lane & 3) << 2);
        const int oes = f32 ? 4 : 2;
#pragma unroll 4
        for (int r = 0; r < 32; ++r) {
          if (k_row + r < a.K && col < a.N) {
            const uint32_t d =
                *reinterpret_cast<const uint32_t*>(buf + r * 128 + (off ^ ((r & 7) << 4)));
            char* dst = static_cast<char*>(a.out) + ((x.g * a.K + k_row + r) * a.N + col) * oes;
            *reinterpret_cast<uint32_t*>(dst) = d;
          }
        }
        __syncwarp();
        ++nb;
        continue;
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (k_row < a.K)
          ptx::tma_store_3d(tm_out, buf, static_cast<int32_t>(x.n0 + c0), k_row,
                            static_cast<int32_t>(x.g));
        ptx::bulk_commit();
      }
      ++nb;
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
  if (lane == 0) ptx::bulk_wait<0>();
  __syncwarp();
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 1)
    gmm_dw_kernel(const __grid_constant__ CUtensorMap tm_dy,
                  const __grid_constant__ CUtensorMap tm_out, const DwArgs a) {
  ptx::griddep_wait();  // launched with programmatic serialization: predecessors done
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* obuf = smem + kDwStages * kStageBytes;
  auto* ctl = reinterpret_cast<DwCtl*>(obuf + kOutBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();

  // Routing validation failed: the result is defined as zeros. (Both CTAs of
  // a pair see the same status and leave before any cluster operation.)
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
  if (warp == 0 && lane == 0) {
    if (!a.gather_dy) {
      ptx::tma_prefetch_desc(&tm_dy);
      ptx::tma_prefetch_desc(&tm_out);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();  // the peer's barriers are initialised
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) dy_producer(smem, ctl, &tm_dy, a, total, rank);
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) mma_issuer<DT>(smem, ctl, tmem_base, a, total);
  } else if (warp < kEpiWarp0) {
    x_gatherer<DT>(smem, ctl, a, total, rank);
  } else {
    epilogue<DT>(obuf, ctl, tmem_base, &tm_out, a, total, rank);
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();  // no CTA leaves while its peer may still use it
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

int dw_smem_bytes() { return kSmemBytes; }
int dw_stage_rows() { return kDwRows; }
int dw_stages() { return kDwStages; }
int dw_threads() { return kThreads; }

// Tiles of 256 k (a CTA pair) x 256 n per expert.
void dw_tiles(int64_t K, int64_t N, int* k_blocks, int* n_blocks) {
  *k_blocks = static_cast<int>((K + 2 * kDwM - 1) / (2 * kDwM));
  *n_blocks = static_cast<int>((N + kDwN - 1) / kDwN);
}

cudaError_t launch_dw(int dtype, const CUtensorMap& tm_dy, const CUtensorMap& tm_out,
                      const DwArgs& a, int num_sms, cudaStream_t stream) {
  void (*kern)(const CUtensorMap, const CUtensorMap, const DwArgs) = nullptr;
  if (dtype == PGG_BF16)
    kern = gmm_dw_kernel<PGG_BF16>;
  else if (dtype == PGG_F16)
    kern = gmm_dw_kernel<PGG_F16>;
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
  const int64_t total = a.G * a.k_blocks * a.n_blocks;
  int64_t want = total < num_sms / 2 ? total : num_sms / 2;
  if (want < 1) want = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * want), 1, 1);
  int clusters = 0;
  err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (err != cudaSuccess) return err;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  return launch_pdl(kern, dim3(static_cast<unsigned>(2 * (clusters < want ? clusters : want))),
                    dim3(kThreads), static_cast<size_t>(kSmemBytes), stream, 2, tm_dy, tm_out, a);
}

}  // namespace pgg
