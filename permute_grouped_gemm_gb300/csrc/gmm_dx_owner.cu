// Owner variant of the fused d_x backward ("MoeInitRoutingGroupedMatmulGrad
// design", section "数学定义和公式": d_x[b, k] = sum over the token's rows i of
// sum_n d_y[i, n] * weight[g(i), k, n]), for problems with few experts.
//
// A CTA pair owns a block of d_x outright: a slab of T tokens (T <= 224, set
// by the host so that a slab holds about 112 rows of each expert) x 256 k
// (128 per CTA). It walks the experts in increasing order; for each expert it
// takes the expert's rows whose tokens lie in the slab (one contiguous range
// when each expert's rows are in increasing original position, which the
// routing step checks), computes C = weight[g] d_y[rows]^T for its 256 k on
// the tensor cores (cta_group::2, M = 256 k, N = rows rounded up to 16 or 32
// and at most 128, TMA for both operands, two accumulators in tensor memory), and
// adds each row into the slab's d_x block, which also lives in tensor memory
// (columns 256 .. 256 + T: one column per token, one lane per k), so that all
// of shared memory goes to the operand pipeline. Each epilogue thread owns one
// d_x column k of the slab (its tensor-memory lane), for every token: it alone
// reads, adds and writes that column, in program order, in increasing expanded index
// (increasing expert, then increasing row within the expert), which is the
// order of additions of the ticketed kernel, with no tickets, no barriers
// between threads and no atomics. The slab block starts as -0.0, so every
// row loads, adds and stores (a token's first row gives -0 + x == x); two
// rows of one token inside one expert are adjacent and carried in a
// register. When the slab is done each thread writes its column to d_x once.
//
// When some expert's rows are not in increasing original position the kernel
// leaves at once and the ticketed kernel, launched after it, does the work.
//
// Pipeline stages: when N is a multiple of 64, each stage covers 128 n as two
// 64-n panels, loaded by one 4-D weight copy and one 3-D d_y copy (4 stages);
// otherwise 64 n (8 stages). The chunks alternate between two pipelines, one
// per accumulator, each with its own TMA thread, MMA-issuing thread and half
// of the stages: an MMA-issuing thread leaves the tensor pipe idle while it
// waits on a barrier or commits (a few hundred cycles each time), and at
// N <= 128 its eight MMAs per stage do not cover that, so the other
// pipeline's MMAs fill the gap. Each accumulator still receives its MMAs from
// one thread in a fixed order, and the epilogue takes the chunks in order, so
// the results do not depend on how the two interleave. Warp roles per CTA: 0
// and 1 TMA (pipeline 0 and 1); 2 and 3 (even CTA) MMA issue, warp 2 also
// tensor-memory allocation; 4-7 epilogue. Units (slab, k range) are
// statically interleaved over the clusters. Waits are bounded; when one runs
// out the kernel records PGG_ERR_TIMEOUT, drains its copies and MMAs, frees
// tensor memory and returns.

#include <cstdint>

#include "pgg_internal.h"
#include "pgg_ptx.cuh"

namespace pgg {
namespace {

constexpr int kOK = 128;          // k per CTA (the pair's MMA M is 256)
constexpr int kMaxRows = 128;     // rows per chunk (MMA N)
constexpr int kABytes = kOK * kRowBytes;              // weight panel: 128 k x 128 bytes
constexpr int kBBytes = (kMaxRows / 2) * kRowBytes;   // rows panel: this CTA's half of the rows
constexpr int kMaxStages = 8;

// Stage geometry: one or two 64-n panels per stage.
template <bool WIDE>
struct Geo {
  static constexpr int kPanels = WIDE ? 2 : 1;
  static constexpr int kA = kPanels * kABytes;
  static constexpr int kStageBytes = kPanels * (kABytes + kBBytes);
  static constexpr int kStages = WIDE ? 4 : kMaxStages;
  static constexpr int kRing = kStages / 2;  // stages of each pipeline
};

// Write-out staging: per epilogue warp two buffers of 32 tokens x 32 k fp32,
// stored to d_x by TMA.
constexpr int kOutBuf = 32 * 32;  // floats
constexpr int kOutBytes = 4 * 2 * kOutBuf * 4;
constexpr int kThreads = 32 * 8;
constexpr int kEpiWarp0 = 4;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 128;              // per MMA accumulator
constexpr int kSlabCol = 2 * kAccCols;     // the slab block: columns 256 .. 256 + T
constexpr int kScratchTok = 255;           // column kSlabCol + 255: padding rows' scratch
static_assert(kSlabCol + kMaxSlabTokens <= kTmemCols, "tensor memory columns");
static_assert(kMaxSlabTokens <= kScratchTok, "the scratch column lies past every slab");

struct OwnCtl {
  uint64_t full[kMaxStages];  // pipeline p uses stages p * kRing .. p * kRing + kRing - 1
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];          // per accumulator = per pipeline
  uint64_t tempty[2];
  uint64_t drain[2];
  uint32_t tmem_base;
  int abort;
};

template <bool WIDE>
constexpr int smem_bytes() {
  return Geo<WIDE>::kStages * Geo<WIDE>::kStageBytes + kOutBytes +
         static_cast<int>(sizeof(OwnCtl)) + 1024;
}
static_assert(smem_bytes<false>() <= 227 * 1024 && smem_bytes<true>() <= 227 * 1024,
              "shared memory per CTA");

__device__ __forceinline__ void raise_status(WsHeader* hdr, uint32_t code, uint32_t site) {
  if (atomicCAS(&hdr->status, 0u, code) == 0u) hdr->timeout_site = site;
}

__device__ __forceinline__ uint32_t cluster_id() { return blockIdx.x >> 1; }
__device__ __forceinline__ uint32_t n_clusters() { return gridDim.x >> 1; }

// MMA N for a chunk of R rows (each CTA stages half): a multiple of 16 with
// wide stages (whole 64-row boxes), of 32 otherwise (boxes of 16 rows or more).
template <bool WIDE>
__device__ __forceinline__ int mma_n(int R) {
  return WIDE ? (R + 15) / 16 * 16 : (R + 31) / 32 * 32;
}

// Walks the chunks of one unit (slab s, k range): experts in increasing
// order, each expert's slab rows in pieces of at most kMaxRows. The bounds of
// the next expert are loaded one expert ahead, so that moving on does not wait
// for memory.
struct ChunkIt {
  // the parameters it needs, copied into registers once (reading them through
  // a pointer to the kernel's parameters costs a memory round trip each time)
  const int32_t* seg;
  WsHeader* hdr;
  int64_t G, M;
  int32_t ns1;  // n_slabs + 1: row length of seg
  int64_t s;
  int64_t g, r0, r_end;
  int64_t ng;          // next expert, its bounds in flight
  int32_t nlo, nhi;
  __device__ void load_next() {
    ng = g + 1;
    if (ng < G) {
      const int32_t* row = seg + ng * ns1;
      nlo = row[s];
      nhi = row[s + 1];
    }
  }
  __device__ void next_expert() {
    while (true) {
      g = ng;
      if (g >= G) return;
      r0 = nlo;
      r_end = nhi;
      // checked build: bounds outside the expanded rows make the range empty
      if (!check_ok(hdr, 0 <= r0 && r0 <= r_end && r_end <= M, 30)) r0 = r_end = 0;
      load_next();
      if (r0 < r_end) return;
    }
  }
  __device__ void start(const OwnerArgs* args, int64_t slab) {
    seg = args->seg;
    hdr = args->hdr;
    G = args->G;
    M = args->M;
    ns1 = args->n_slabs + 1;
    s = slab;
    g = -1;
    r0 = r_end = 0;
    load_next();
    next_expert();
  }
  __device__ bool valid() const { return g < G; }
  __device__ int rows() const {
    const int64_t left = r_end - r0;
    return static_cast<int>(left < kMaxRows ? left : kMaxRows);
  }
  __device__ void next() {
    r0 += rows();
    if (r0 >= r_end) next_expert();
  }
};

// TMA thread of pipeline `pipe`: the operands of every other chunk (those of
// parity `pipe`), into the pipeline's stages.
template <bool WIDE>
__device__ void producer(uint8_t* smem, OwnCtl* ctl, const OwnerMaps* m, const OwnerArgs& a,
                         uint32_t n_units, uint32_t rank, int pipe) {
  using Gm = Geo<WIDE>;
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const bool leader = rank == 0;
  const int s0 = pipe * Gm::kRing;
  int stage = s0;
  uint32_t phase = 0, outstanding = 0, last_parity = 0;
  uint32_t parity = 0;  // of the chunk index
  bool failed = false;
  for (uint32_t u = cluster_id(); u < n_units && !failed; u += n_clusters()) {
    const int64_t slab = u / a.k_units;
    const int32_t k0 = static_cast<int32_t>((u % a.k_units) * 2 * kOK + kOK * rank);
    ChunkIt c;
    for (c.start(&a, slab); c.valid() && !failed; c.next(), parity ^= 1u) {
      if (parity != static_cast<uint32_t>(pipe)) continue;
      const int nm = mma_n<WIDE>(c.rows());
      const int half = nm / 2;  // this CTA's rows: a multiple of 8 (WIDE) or 16, at most 64
      // wide stages load whole 64-row boxes (the MMA reads the first half rows)
      const uint32_t tx = WIDE ? 2u * static_cast<uint32_t>(Gm::kStageBytes)
                               : 2u * static_cast<uint32_t>(kABytes + half * kRowBytes);
      const int32_t brow = static_cast<int32_t>(c.r0 + rank * half);
      for (int ks = 0; ks < a.nk; ++ks) {
        if (!ptx::mbar_wait_cluster(&ctl->empty[stage], phase ^ 1u, lim, abort)) {
          failed = true;
          break;
        }
        uint8_t* sa = smem + stage * Gm::kStageBytes;
        const uint32_t fb = ptx::mapa(&ctl->full[stage], 0);
        if (leader) ptx::mbar_arrive_expect_tx(&ctl->full[stage], tx);
        if constexpr (WIDE) {
          // panels 2 ks and 2 ks + 1 of 64 n (past N / 64 they read as zero)
          ptx::tma_load_4d_pair(sa, &m->tw4, fb, 0, k0, 2 * ks, static_cast<int32_t>(c.g));
          ptx::tma_load_3d_pair(sa + Gm::kA, &m->dy3, fb, 0, brow, 2 * ks);
        } else {
          ptx::tma_load_3d_pair(sa, &m->tw, fb, ks * 64, k0, static_cast<int32_t>(c.g));
          // the rows in boxes of 64, 32 and 16 rows (each box lands on a
          // 1024-byte boundary, so the 128-byte swizzle stays in phase)
          for (int r = 0; r < half;) {
            const int j = half - r >= 64 ? 2 : (half - r >= 32 ? 1 : 0);
            ptx::tma_load_2d_pair(sa + kABytes + r * kRowBytes, &m->dy.box[j], fb, ks * 64,
                                  brow + r);
            r += kDyMinRows << j;
          }
        }
        outstanding |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == s0 + Gm::kRing) {
          stage = s0;
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
    for (int s = s0; s < s0 + Gm::kRing; ++s)
      if (outstanding & (1u << s))
        ptx::mbar_wait_cluster(&ctl->full[s], (last_parity >> s) & 1u, lim, &no_abort);
  }
}

// MMA-issuing thread of pipeline `pipe` (even CTA): every other chunk (those
// of parity `pipe`), into accumulator `pipe`.
template <int DT, bool WIDE>
__device__ void mma_issuer(uint8_t* smem, OwnCtl* ctl, uint32_t tmem_base, const OwnerArgs& a,
                           uint32_t n_units, int pipe) {
  using Gm = Geo<WIDE>;
  constexpr uint32_t kFmt = DT == PGG_BF16 ? 1u : 0u;
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int s0 = pipe * Gm::kRing;
  const int acc = pipe;
  int stage = s0;
  uint32_t phase = 0, aph = 0;
  uint32_t parity = 0;  // of the chunk index
  bool issued = false, failed = false;
  for (uint32_t u = cluster_id(); u < n_units && !failed; u += n_clusters()) {
    ChunkIt c;
    for (c.start(&a, u / a.k_units); c.valid() && !failed; c.next(), parity ^= 1u) {
      if (parity != static_cast<uint32_t>(pipe)) continue;
      const uint32_t idesc =
          ptx::idesc_make(kFmt, 2 * kOK, static_cast<uint32_t>(mma_n<WIDE>(c.rows())));
      // (tensor memory changes hands through the tcgen05 fences around this
      // wait and the epilogue's arrivals: a CTA-scope wait suffices)
      if (!ptx::mbar_wait(&ctl->tempty[acc], aph ^ 1u, lim, abort)) {
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
        const uint32_t sa = ptx::smem_addr(smem + stage * Gm::kStageBytes);
#pragma unroll
        for (int p = 0; p < Gm::kPanels; ++p) {
          const uint64_t da = ptx::sdesc_sw128(sa + p * kABytes);
          const uint64_t db = ptx::sdesc_sw128(sa + Gm::kA + p * kBBytes);
#pragma unroll
          for (int kk = 0; kk < kRowBytes / 32; ++kk) {
            const uint64_t koff = static_cast<uint64_t>((kk * 32) >> 4);
            ptx::mma_f16_pair(d_tmem, da + koff, db + koff, idesc, (ks | p | kk) != 0 ? 1u : 0u);
          }
        }
        issued = true;
        ptx::mma_commit_pair(&ctl->empty[stage], 0x3);
        if (++stage == s0 + Gm::kRing) {
          stage = s0;
          phase ^= 1u;
        }
      }
      if (failed) break;
      ptx::mma_commit_pair(&ctl->tfull[acc], 0x3);
      aph ^= 1u;
    }
  }
  if (failed) {
    ctl->abort = 1;
    raise_status(a.hdr, kStTimeout, 34);
  }
  if (issued) {
    int no_abort = 0;
    ptx::mma_commit_pair(&ctl->drain[pipe], 0x1);
    ptx::mbar_wait(&ctl->drain[pipe], 0u, lim, &no_abort);
  }
}

// Row flags of the epilogue: bits 0-7 the token within the slab.
constexpr int kRowPad = 1 << 8;    // no row (past the chunk's end): token kScratchTok
constexpr int kRowDup = 1 << 10;   // same token as the row before, in this batch: carry

// Row records of a chunk's rows: lane j of ri[b] gets row 32 b + j (token -1
// past the chunk's end).
__device__ __forceinline__ void load_rows(const ChunkIt& c, const OwnerArgs& a, int lane,
                                          RowInfo (&ri)[kMaxRows / 32]) {
  const int R = c.rows();
#pragma unroll
  for (int b = 0; b < kMaxRows / 32; ++b) {
    const int r = 32 * b + lane;
    ri[b] = r < R ? a.rowinfo[check_index(a.hdr, c.r0 + r, a.M, 31)] : RowInfo{-1, 0};
  }
}

// 32 lanes x 32 columns of tensor memory set to x.
__device__ __forceinline__ void tmem_fill_32x32b_x32(uint32_t taddr, uint32_t x) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1,"
      " %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1};" ::"r"(
          taddr),
      "r"(x)
      : "memory");
}

// Epilogue warp q (of 4) owns tensor-memory lanes 32 q .. 32 q + 31: one d_x
// column k each, for every token of the slab.
__device__ void epilogue(OwnCtl* ctl, float* out_stage, const CUtensorMap* tout,
                         uint32_t tmem_base, const OwnerArgs& a, uint32_t n_units, uint32_t rank) {
  const uint64_t lim = a.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const uint32_t tempty0 = ptx::mapa(&ctl->tempty[0], 0);
  const uint32_t tempty1 = ptx::mapa(&ctl->tempty[1], 0);
  const int64_t K = a.K;
  const int T = a.slab_tokens;
  const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16);
  int acc = 0, obuf = 0;
  uint32_t aph = 0;
  bool stop = false;
  bool held = a.hold_release != 0;  // (test hook: the first release is withheld)
  for (uint32_t u = cluster_id(); u < n_units && !stop; u += n_clusters()) {
    const int64_t slab = u / a.k_units;
    const int64_t tok0 = slab * T;
    const int64_t k =
        static_cast<int64_t>(u % a.k_units) * 2 * kOK + kOK * rank + 32 * quarter + lane;
    // The slab block starts as -0.0 in every column, so that a token's first
    // row is added like the others (-0 + x == x for every x).
    for (int t0 = 0; t0 < T; t0 += 32)
      tmem_fill_32x32b_x32(t_lane + kSlabCol + static_cast<uint32_t>(t0), 0x80000000u);
    ptx::tmem_st_wait();
    ChunkIt c;
    c.start(&a, slab);
    // the row records of each chunk are loaded while the chunk before it is
    // added (they do not depend on the MMA)
    RowInfo ri[kMaxRows / 32];
    if (c.valid()) load_rows(c, a, lane, ri);
    while (c.valid()) {
      const int R = c.rows();
      // lane j of info[b] describes row 32 b + j of the chunk
      int info[kMaxRows / 32];
#pragma unroll
      for (int b = 0; b < kMaxRows / 32; ++b) {
        int f = kRowPad | kScratchTok;
        const int64_t t = static_cast<int64_t>(ri[b].token) - tok0;
        if (32 * b + lane < R && t >= 0 && t < T) f = static_cast<int>(t);
        const int before = __shfl_up_sync(0xFFFFFFFFu, f, 1);
        if (lane > 0 && !(f & kRowPad) && !(before & kRowPad) && ((before ^ f) & 0xFF) == 0)
          f |= kRowDup;
        info[b] = f;
      }
      ChunkIt cn = c;
      cn.next();
      if (cn.valid()) load_rows(cn, a, lane, ri);
      const bool ok = ptx::mbar_wait(&ctl->tfull[acc], aph, lim, abort);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        if (lane == 0) {
          ctl->abort = 1;
          raise_status(a.hdr, kStTimeout, 35);
        }
        stop = true;
        break;
      }
      ptx::tc_fence_after_sync();
      const uint32_t acc_col = static_cast<uint32_t>(acc * kAccCols);
      // (a loop, not unrolled: the smaller code runs faster here)
#pragma unroll 1
      for (int b = 0; b < kMaxRows / 32; ++b) {
        if (32 * b >= R) break;
        // The batch's carry flags as a warp-wide bit mask, its tokens four to
        // a 32-bit word: the per-row column arithmetic then runs on values
        // the whole warp shares (a per-row shuffle costs ~2.5x in the loads
        // and stores below).
        const int f = b == 0 ? info[0] : (b == 1 ? info[1] : (b == 2 ? info[2] : info[3]));
        const uint32_t dupm = __ballot_sync(0xFFFFFFFFu, f & kRowDup);
        uint32_t x = static_cast<uint32_t>(f & 0xFF) << (8 * (lane & 3));
        x |= __shfl_xor_sync(0xFFFFFFFFu, x, 1);
        x |= __shfl_xor_sync(0xFFFFFFFFu, x, 2);
        uint32_t pk[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) pk[w] = __shfl_sync(0xFFFFFFFFu, x, 4 * w);
        // row j's column: its token's slab column (a padding row's is the
        // scratch column, whose contents nothing reads)
        auto col = [&](int j) -> uint32_t {
          return kSlabCol + __byte_perm(pk[j >> 2], 0u, 0x4440u + static_cast<uint32_t>(j & 3));
        };
        uint32_t v[32], old[32];
        ptx::tmem_ld_32x32b_x32(t_lane + acc_col + static_cast<uint32_t>(32 * b), v);
#pragma unroll
        for (int j = 0; j < 32; ++j) old[j] = ptx::tmem_ld_32x32b_x1(t_lane + col(j));
        ptx::tmem_ld_wait_regs(v);
        ptx::tmem_ld_wait_regs(old);
        if (dupm == 0) {
          // distinct tokens: independent updates
#pragma unroll
          for (int j = 0; j < 32; ++j)
            ptx::tmem_st_32x32b_x1(t_lane + col(j),
                                   __float_as_uint(__uint_as_float(old[j]) + __uint_as_float(v[j])));
        } else {
          // a token twice in a row: carry its running sum
          float carry = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float xv = __uint_as_float(v[j]);
            const float val = ((dupm >> j) & 1u) ? carry + xv : __uint_as_float(old[j]) + xv;
            ptx::tmem_st_32x32b_x1(t_lane + col(j), __float_as_uint(val));
            carry = val;
          }
        }
        // the next batch may read what this one wrote
        ptx::tmem_st_wait();
      }
      ptx::tc_fence_before_sync();
      __syncwarp();
      // tensor memory changes hands: CTA scope (a cluster-scope release
      // cost ~1,800 cycles here)
      if (lane == 0 && !held) ptx::mbar_arrive_remote_cta(acc ? tempty1 : tempty0);
      held = false;
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
      c = cn;
    }
    if (stop) break;
    // the slab is done: this thread's column to d_x (every token of the
    // slab has at least one row, so every element was stored above), 32
    // tokens at a time: through a shared-memory buffer and a TMA store when
    // d_x rows allow it, else with 128-byte warp stores
    int64_t nt = a.batch - tok0;
    if (nt > T) nt = T;
    for (int t0 = 0; t0 < static_cast<int>(nt); t0 += 32) {
      uint32_t w[32];
      ptx::tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(kSlabCol + t0), w);
      ptx::tmem_ld_wait_regs(w);
      if (a.tma_out) {
        float* sb = out_stage + obuf * kOutBuf;
        // the store that last read this buffer (two groups ago) is done
        if (lane == 0) ptx::bulk_wait_read<1>();
        __syncwarp();
#pragma unroll
        for (int t = 0; t < 32; ++t) sb[t * 32 + lane] = __uint_as_float(w[t]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        // (a warp whose 32 columns all lie past K has nothing to store)
        if (lane == 0 && k < K) {
          ptx::tma_store_2d(tout, sb, static_cast<int32_t>(k), static_cast<int32_t>(tok0 + t0));
          ptx::bulk_commit();
        }
        obuf ^= 1;
      } else if (k < K) {
        float* dst = a.out + (tok0 + t0) * K + k;
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (t0 + t < nt) dst[t * K] = __uint_as_float(w[t]);
      }
    }
  }
  // the stores have read shared memory and written d_x before the CTA exits
  if (lane == 0) ptx::bulk_wait<0>();
  __syncwarp();
}

template <int DT, bool WIDE>
__global__ void __launch_bounds__(kThreads, 1)
    gmm_dx_owner_kernel(const __grid_constant__ OwnerMaps m, const OwnerArgs a) {
  using Gm = Geo<WIDE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* out_stage = reinterpret_cast<float*>(smem + Gm::kStages * Gm::kStageBytes);
  auto* ctl = reinterpret_cast<OwnCtl*>(smem + Gm::kStages * Gm::kStageBytes + kOutBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();

  // Launched with programmatic serialization: the routing step before this
  // kernel has finished and its memory is visible past here.
  ptx::griddep_wait();
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
    for (int s = 0; s < Gm::kStages; ++s) {
      ptx::mbar_init(&ctl->full[s], 1);
      ptx::mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl->tfull[b], 1);
      ptx::mbar_init(&ctl->tempty[b], 8);
    }
    ptx::mbar_init(&ctl->drain[0], 1);
    ptx::mbar_init(&ctl->drain[1], 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    // (both TMA threads use the same maps)
    if constexpr (WIDE) {
      ptx::tma_prefetch_desc(&m.tw4);
      ptx::tma_prefetch_desc(&m.dy3);
    } else {
      for (int j = 0; j < kDyMaps; ++j) ptx::tma_prefetch_desc(&m.dy.box[j]);
      ptx::tma_prefetch_desc(&m.tw);
    }
    if (a.tma_out) ptx::tma_prefetch_desc(&m.tout);
  }
  if (warp == 2) {
    ptx::tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp < 2) {
    if (lane == 0) producer<WIDE>(smem, ctl, &m, a, n_units, rank, warp);
  } else if (warp < kEpiWarp0) {
    if (lane == 0 && rank == 0) mma_issuer<DT, WIDE>(smem, ctl, tmem_base, a, n_units, warp - 2);
  } else {
    epilogue(ctl, out_stage + (warp & 3) * 2 * kOutBuf, &m.tout, tmem_base, a, n_units, rank);
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();
  if (warp == 2) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

int owner_smem_bytes(bool wide) { return wide ? smem_bytes<true>() : smem_bytes<false>(); }
int owner_stages(bool wide) { return wide ? Geo<true>::kStages : Geo<false>::kStages; }
int owner_threads() { return kThreads; }

// m.tw4 / m.dy3 are read when a.wide is set (N a multiple of 64), m.dy / m.tw otherwise.
cudaError_t launch_owner(int dtype, const OwnerMaps& m, const OwnerArgs& a, int num_sms,
                         cudaStream_t stream) {
  void (*kern)(const OwnerMaps, const OwnerArgs) = nullptr;
  const bool wide = a.wide != 0;
  if (dtype == PGG_BF16)
    kern = wide ? gmm_dx_owner_kernel<PGG_BF16, true> : gmm_dx_owner_kernel<PGG_BF16, false>;
  else if (dtype == PGG_F16)
    kern = wide ? gmm_dx_owner_kernel<PGG_F16, true> : gmm_dx_owner_kernel<PGG_F16, false>;
  else
    return cudaErrorInvalidValue;
  const int smem = owner_smem_bytes(wide);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
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
  return launch_pdl(kern, dim3(static_cast<unsigned>(2 * (clusters < want ? clusters : want))),
                    dim3(kThreads), static_cast<size_t>(smem), stream, 2, m, a);
}

}  // namespace pgg
