// Persistent grouped GEMM with a fused, ordered scatter-add into FP32 d_x.
//
// Computes ("MoeInitRoutingGroupedMatmulGrad design", section "数学定义和公式")
//   d_expanded_x[i, k] = sum_n d_y[i, n] * weight[g(i), k, n]        (Step 1)
//   d_x[b, k]         += d_expanded_x[i, k]  for b = original_pos(i) / topK
//                                                                     (Step 2)
// one tile at a time, so that no [M, K] array ever exists (section 1.1).
//
// Tile = (row block, k block): up to ROWS consecutive expanded rows of one
// expert and 128 consecutive output columns k. The MMA is issued with the
// weight slice as operand A (M = 128 rows of k) and the d_y rows as operand B
// (N = rows, rounded up to 16), both K-major along n, so that the accumulator
// in tensor memory holds lane = k, column = expanded row. The epilogue
// transposes 4 x 4 blocks in registers so that each lane holds four
// consecutive k of one row, and writes each row's 512-byte segment of d_x as
// 128-byte vector stores (the row's first contribution) or vector fp32
// reductions performed at L2 (later ones).
//
// Warp roles (one CTA per SM, persistent):
//   warp 0       tile scheduler + TMA producer (one lane)
//   warp 1       TMEM allocation + MMA issuer (one lane)
//   warps 2..5   epilogue: TMEM -> registers -> ordered scatter-add into d_x
//   warps 6..9   fp32 inputs only: split each staged fp32 tile into tf32
//                high and low parts for the 3-product tf32 MMA
//
// CTA pairs (the tensor-bound 16-bit variant): two CTAs of a cluster share
// one tile of 256 k x up to 256 rows. Each holds half of the weight slice
// (its 128 k) and half of the rows in its own shared memory; the even CTA
// issues tcgen05.mma.cta_group::2, which reads both halves and leaves each
// CTA's 128 accumulator lanes in that CTA's tensor memory. Per SM this halves
// the d_y bytes staged per MMA, so the shared-memory port (written by TMA,
// read by the tensor core) carries a third less traffic per flop than a
// single-CTA 128 x 256 tile. The even CTA claims tiles and forwards them to its
// peer; the peer's copies complete on the even CTA's barriers; MMA
// completions are multicast to both CTAs.
//
// Tiles are handed out by an atomic counter in increasing order of a fixed
// global numbering: bands of k blocks, then row blocks (expert-major, row
// order), then the k blocks of the band. For a fixed k block, row blocks come
// in increasing expanded-row order.
//
// Deterministic scatter-add (section 2.4.1 asks for deterministic results):
// a token's topK expanded rows are ranked by expanded index. For each (token,
// k block) a ticket counts the contributions already added. The row of rank r
// waits until the ticket reaches r, stores (rank 0) or adds (rank > 0) its 128
// values, and bumps the ticket. Every d_x element therefore receives its topK
// terms in the same order on every run, with no zero-fill pass. A row's
// predecessors lie in tiles with a smaller number (same k block, earlier row
// block) or earlier in the same tile, and tiles are only numbered once a
// running CTA has claimed them, so the wait graph has no cycle whatever the
// residency of the grid. Waits are bounded; when one runs out the kernel
// records PGG_ERR_TIMEOUT in the status word and finishes without waiting.

#include <cstdint>

#include "pgg_gather.cuh"
#include "pgg_internal.h"
#include "pgg_ptx.cuh"

namespace pgg {
namespace {

template <int DT>
struct DtTraits;
template <>
struct DtTraits<PGG_BF16> {
  static constexpr int kElem = 2;
  static constexpr uint32_t kFmt = 1;
  static constexpr bool kSplit = false;
};
template <>
struct DtTraits<PGG_F16> {
  static constexpr int kElem = 2;
  static constexpr uint32_t kFmt = 0;
  static constexpr bool kSplit = false;
};
template <>
struct DtTraits<PGG_F32> {
  static constexpr int kElem = 4;
  static constexpr uint32_t kFmt = 2;  // tf32
  static constexpr bool kSplit = true;
};

constexpr int kQueue = 4;

constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

template <int DT, int ROWS, int STAGES, bool PAIR = false, bool GATHER = false>
struct Cfg {
  static constexpr bool kSplit = DtTraits<DT>::kSplit;
  static constexpr int kElemsPerRow = kRowBytes / DtTraits<DT>::kElem;
  static constexpr int kABytes = kKBlock * kRowBytes;
  // rows of d_y this CTA stages per k step (a pair splits the tile's rows)
  static constexpr int kBRows = PAIR ? ROWS / 2 : ROWS;
  static constexpr int kBBytes = kBRows * kRowBytes;
  static constexpr int kStageBytes = (kABytes + kBBytes) * (kSplit ? 2 : 1);
  static constexpr int kAccCols = ROWS < 32 ? 32 : ROWS;
  static constexpr int kTmemCols = pow2_at_least(2 * kAccCols);  // allocation unit
  static constexpr int kWords = (ROWS + 31) / 32;
  // Epilogue warp groups of four warps (one per tensor-memory lane quarter).
  // Group g drains accumulator buffer g, so with two groups each tile's
  // epilogue has two MMA tile-times to finish. The fp32 variant keeps one
  // group (its extra warps split operands).
  static constexpr int kEpiGroups = kSplit ? 1 : 2;
  static constexpr int kEpiWarps = 4 * kEpiGroups;
  static constexpr int kXformWarps = kSplit ? 4 : 0;
  // Gathered operands: two warps per stage slot copy the slot's rows with
  // cp.async (rows whose byte length is not a multiple of 16).
  static constexpr int kWarpsPerSlot = 2;
  static constexpr int kGatherWarps = GATHER ? kWarpsPerSlot * STAGES : 0;
  static constexpr int kGatherWarp0 = 2 + kEpiWarps + kXformWarps;
  static constexpr int kThreads = 32 * (2 + kEpiWarps + kXformWarps + kGatherWarps);
  static constexpr int kMmaM = PAIR ? 2 * kKBlock : kKBlock;
  static constexpr int kNAlign = PAIR ? 32 : 16;  // MMA N granularity
  // consumers of a tile-queue slot: MMA + epilogue (+ fp32 split), and in a
  // pair the peer's producer and epilogue as well
  static constexpr uint32_t kQEmpty = PAIR ? 4 : (kSplit ? 3 : 2);
  static constexpr uint32_t kTEmpty = PAIR ? 8 : 4;  // one group's warps (of both CTAs)
  static_assert(ROWS % 32 == 0 && ROWS <= 256, "rows per block");
  static_assert(!PAIR || (!kSplit && ROWS % 64 == 0), "pairs: 16-bit inputs, rows % 64 == 0");
  static_assert(!GATHER || !kSplit, "gathered operands: 16-bit inputs");
  static_assert(kTmemCols <= 512, "tmem columns");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
};

// MMA N extent for a tile of R rows.
template <class C>
__device__ __forceinline__ int mma_n(int R) {
  const int n = (R + C::kNAlign - 1) / C::kNAlign * C::kNAlign;
  return n < C::kNAlign ? C::kNAlign : n;
}

// Rows per tensor-memory load in the epilogue (32: against 16, skewed -1.7%,
// large and unaligned -0.6%), and the bits of a row mask word they cover.
constexpr int kChunk = 32;
constexpr uint32_t kChunkMask = 0xFFFFFFFFu >> (32 - kChunk);

// Per-tile state of one epilogue group.
template <int ROWS>
struct EpiState {
  uint32_t pend[(ROWS + 31) / 32];  // rows still to be added
  uint32_t rdy[(ROWS + 31) / 32];   // rows whose turn has come in this round
  RowInfo meta[ROWS];
};

// What the gather warp of a stage slot copies (gathered-operand kernel): the
// weight rows of k block kb of expert g and `fill` rows of d_y from `row` on
// (of which the first `valid` are read, the rest zero-filled), each over the
// 64 n from n0.
struct GatherDesc {
  int32_t g;  // -1: no more stages
  int32_t row, valid, fill, kb, n0;
  int32_t pad[2];
};

template <int ROWS, int STAGES>
struct Ctl {
  uint64_t full[STAGES];   // operands landed: TMA bytes (pairs: both CTAs' bytes, even CTA's
                           // barrier), or the arrivals of the gather warps of both CTAs
  uint64_t dfull[STAGES];  // gathered operands: the slot's descriptor is posted
  uint64_t empty[STAGES];  // MMAs reading the stage completed
  uint64_t ready[STAGES];  // fp32 split done
  uint64_t tfull[2];       // accumulator complete
  uint64_t tempty[2];      // accumulator drained by the epilogue(s)
  uint64_t qfull[kQueue];
  uint64_t qempty[kQueue];
  uint64_t drain;
  int4 q[kQueue];  // {expert (-1 = stop), first row, rows, k unit}
  GatherDesc desc[STAGES];
  uint32_t tmem_base;
  int abort;
  EpiState<ROWS> epi[2];  // one per epilogue group
};

template <int DT, int ROWS, int STAGES, bool PAIR>
constexpr int smem_bytes() {
  return 1024 + STAGES * Cfg<DT, ROWS, STAGES, PAIR>::kStageBytes +
         static_cast<int>(sizeof(Ctl<ROWS, STAGES>));
}

__device__ __forceinline__ bool bar_any(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n"
      ".reg .pred p, q;\n"
      "setp.ne.u32 p, %1, 0;\n"
      "bar.red.or.pred q, %2, %3, p;\n"
      "selp.u32 %0, 1, 0, q;\n"
      "}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void raise_status(WsHeader* hdr, uint32_t code, uint32_t site) {
  if (atomicCAS(&hdr->status, 0u, code) == 0u) hdr->timeout_site = site;
}

// Index of the smallest d_y box (16 << j rows, at most CAP) that covers R rows.
template <int CAP>
__device__ __forceinline__ int dy_box(int R) {
  int j = 0;
  while ((kDyMinRows << j) < R && (kDyMinRows << j) < CAP) ++j;
  return j;
}

// Tile number -> (row block, k block). Bands of `band` k blocks; inside a band
// row-block-major, k block fastest.
__device__ __forceinline__ void decode_tile(uint32_t t, uint32_t n_rb, uint32_t kbs, uint32_t band,
                                            uint32_t* rb, uint32_t* kb) {
  const uint32_t per_band = n_rb * band;
  const uint32_t bi = t / per_band;
  const uint32_t kb_lo = bi * band;
  const uint32_t w = kbs - kb_lo < band ? kbs - kb_lo : band;
  const uint32_t rem = t - bi * per_band;
  *rb = rem / w;
  *kb = kb_lo + rem % w;
}

template <int DT, int ROWS, int STAGES, bool PAIR, bool GATHER>
__device__ void producer(uint8_t* smem, Ctl<ROWS, STAGES>* ctl, const DyMaps* dy_maps,
                         const CUtensorMap* tm_w, const GemmArgs& args, uint32_t total,
                         uint32_t rank) {
  using C = Cfg<DT, ROWS, STAGES, PAIR, GATHER>;
  const uint64_t lim = args.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const bool leader = rank == 0;
  int stage = 0, qs = 0;
  uint32_t phase = 0, qph = 0, outstanding = 0, last_parity = 0;
  const uint32_t n_rb = args.hdr->n_row_blocks;
  const uint32_t units = static_cast<uint32_t>(args.k_units);
  const uint32_t band = static_cast<uint32_t>(args.band_units);
  auto entry = [&](uint32_t t) {
    if (t >= total) return make_int4(-1, 0, 0, 0);
    uint32_t rb, ku;
    decode_tile(t, n_rb, units, band, &rb, &ku);
    int4 r = args.rblist[check_index(args.hdr, rb, args.max_row_blocks, 40)];
    // checked build: a row block outside the experts or rows becomes an empty one
    if (!check_ok(args.hdr,
                  r.x >= 0 && r.x < args.G && r.y >= 0 && r.z >= 0 && r.z <= ROWS &&
                      static_cast<int64_t>(r.y) + r.z <= args.M,
                  41))
      r = make_int4(0, 0, 0, 0);
    return make_int4(r.x, r.y, r.z, static_cast<int>(ku));
  };
  // The next tile is claimed and its row block read while the current one
  // streams, so no tile starts with a scheduler round trip.
  int4 e = make_int4(-1, 0, 0, 0);
  if (leader) e = entry(atomicAdd(&args.hdr->sched_next, 1u));
  bool failed = false;
  int stops = 0;
  while (!failed) {
    uint32_t t_next = total;
    if (leader) {
      if (e.x >= 0) t_next = atomicAdd(&args.hdr->sched_next, 1u);
      if (!ptx::mbar_wait(&ctl->qempty[qs], qph ^ 1u, lim, abort)) {
        failed = true;
        break;
      }
      ctl->q[qs] = e;
      ptx::mbar_arrive(&ctl->qfull[qs]);
      if constexpr (PAIR) {
        ptx::st_cluster_v4(ptx::mapa(&ctl->q[qs], 1), e);
        ptx::mbar_arrive_remote(ptx::mapa(&ctl->qfull[qs], 1));
      }
    } else {
      if (!ptx::mbar_wait_cluster(&ctl->qfull[qs], qph, lim, abort)) {
        failed = true;
        break;
      }
      e = ctl->q[qs];
      ptx::mbar_arrive_remote(ptx::mapa(&ctl->qempty[qs], 0));
    }
    if (++qs == kQueue) {
      qs = 0;
      qph ^= 1u;
    }
    if (e.x < 0) {
      // one stop entry per epilogue group (each group reads every other entry)
      if (leader && ++stops < C::kEpiGroups) continue;
      break;
    }
    const int nm = mma_n<C>(e.z);
    // rows of d_y this CTA stages (gathered: every row the MMA reads)
    const int b_rows = PAIR ? nm / 2 : (GATHER ? nm : e.z);
    const int bj = dy_box<C::kBRows>(b_rows);
    const uint32_t box_bytes = static_cast<uint32_t>(kDyMinRows << bj) * kRowBytes;
    const uint32_t tx = PAIR ? 2 * (C::kABytes + box_bytes) : C::kABytes + box_bytes;
    const CUtensorMap* tm_dy = &dy_maps->box[bj];
    const int kb = PAIR ? 2 * e.w + static_cast<int>(rank) : e.w;
    const int brow = e.y + (PAIR ? static_cast<int>(rank) * (nm / 2) : 0);
    int4 e_next = make_int4(-1, 0, 0, 0);
    bool have_next = false;
    for (int ks = 0; ks < args.nk; ++ks) {
      const bool ok = PAIR ? ptx::mbar_wait_cluster(&ctl->empty[stage], phase ^ 1u, lim, abort)
                           : ptx::mbar_wait(&ctl->empty[stage], phase ^ 1u, lim, abort);
      if (!ok) {
        failed = true;
        break;
      }
      uint8_t* sa = smem + stage * C::kStageBytes;
      const int32_t n0 = ks * C::kElemsPerRow;
      if constexpr (GATHER) {
        // the slot's gather warp copies the operands (the slot is free: the
        // MMAs that read it, and so the copies of its previous use, are done)
        GatherDesc& d = ctl->desc[stage];
        const int mine = e.z - (PAIR ? static_cast<int>(rank) * (nm / 2) : 0);
        d.g = e.x;
        d.row = brow;
        d.fill = b_rows;
        d.valid = mine < 0 ? 0 : (mine < b_rows ? mine : b_rows);
        d.kb = kb;
        d.n0 = n0;
        ptx::mbar_arrive(&ctl->dfull[stage]);
        (void)sa;
        (void)tx;
        (void)tm_dy;
      } else if constexpr (PAIR) {
        const uint32_t fb = ptx::mapa(&ctl->full[stage], 0);
        if (leader) ptx::mbar_arrive_expect_tx(&ctl->full[stage], tx);
        ptx::tma_load_3d_pair(sa, tm_w, fb, n0, kb * kKBlock, e.x);
        ptx::tma_load_2d_pair(sa + C::kABytes, tm_dy, fb, n0, brow);
      } else {
        ptx::mbar_arrive_expect_tx(&ctl->full[stage], tx);
        ptx::tma_load_3d(sa, tm_w, &ctl->full[stage], n0, kb * kKBlock, e.x);
        ptx::tma_load_2d(sa + C::kABytes, tm_dy, &ctl->full[stage], n0, brow);
      }
      outstanding |= 1u << stage;
      last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
      if (leader && !have_next && (ks == 1 || ks + 1 == args.nk)) {
        e_next = entry(t_next);
        have_next = true;
      }
    }
    if (leader) {
      if (!have_next) e_next = entry(t_next);
      e = e_next;
    }
  }
  if constexpr (GATHER) {
    // one stop descriptor per slot, each once the slot's last stage is consumed
    for (int i = 0; i < STAGES && !failed; ++i) {
      const bool ok = PAIR ? ptx::mbar_wait_cluster(&ctl->empty[stage], phase ^ 1u, lim, abort)
                           : ptx::mbar_wait(&ctl->empty[stage], phase ^ 1u, lim, abort);
      if (!ok) {
        failed = true;
        break;
      }
      ctl->desc[stage].g = -1;
      ptx::mbar_arrive(&ctl->dfull[stage]);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (failed) {
    ctl->abort = 1;
    raise_status(args.hdr, kStTimeout, 2);
  }
  // Gathered operands: each gather warp waits for its own copies. Otherwise
  // never leave while a copy into this CTA's shared memory may be in flight.
  // A pair's odd CTA cannot see its copies complete (they signal the even
  // CTA's barrier); the even CTA's MMA consuming the stage implies it.
  if constexpr (GATHER) return;
  int no_abort = 0;
  for (int s = 0; s < STAGES; ++s) {
    if (!(outstanding & (1u << s))) continue;
    const uint32_t par = (last_parity >> s) & 1u;
    if (!PAIR || leader)
      ptx::mbar_wait(&ctl->full[s], par, lim, &no_abort);
    else
      ptx::mbar_wait_cluster(&ctl->empty[s], par, lim, &no_abort);
  }
}

template <int DT, int ROWS, int STAGES, bool PAIR>
__device__ void mma_issuer(uint8_t* smem, Ctl<ROWS, STAGES>* ctl, uint32_t tmem_base,
                           const GemmArgs& args) {
  using C = Cfg<DT, ROWS, STAGES, PAIR>;
  const uint64_t lim = args.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  int stage = 0, qs = 0, acc = 0;
  uint32_t phase = 0, qph = 0, aph = 0;
  bool issued = false, failed = false;
  while (!failed) {
    if (!ptx::mbar_wait(&ctl->qfull[qs], qph, lim, abort)) {
      failed = true;
      break;
    }
    const int4 e = ctl->q[qs];
    ptx::mbar_arrive(&ctl->qempty[qs]);
    if (++qs == kQueue) {
      qs = 0;
      qph ^= 1u;
    }
    if (e.x < 0) break;
    const uint32_t idesc =
        ptx::idesc_make(DtTraits<DT>::kFmt, C::kMmaM, static_cast<uint32_t>(mma_n<C>(e.z)));
    const bool ok_t = PAIR ? ptx::mbar_wait_cluster(&ctl->tempty[acc], aph ^ 1u, lim, abort)
                           : ptx::mbar_wait(&ctl->tempty[acc], aph ^ 1u, lim, abort);
    if (!ok_t) {
      failed = true;
      break;
    }
    ptx::tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::kAccCols);
    for (int ks = 0; ks < args.nk; ++ks) {
      uint64_t* bar = C::kSplit ? &ctl->ready[stage] : &ctl->full[stage];
      const bool ok = PAIR ? ptx::mbar_wait_cluster(bar, phase, lim, abort)
                           : ptx::mbar_wait(bar, phase, lim, abort);
      if (!ok) {
        failed = true;
        break;
      }
      ptx::tc_fence_after_sync();
      const uint32_t sa = ptx::smem_addr(smem + stage * C::kStageBytes);
      const uint64_t a_hi = ptx::sdesc_sw128(sa);
      const uint64_t b_hi = ptx::sdesc_sw128(sa + C::kABytes);
#pragma unroll
      for (int kk = 0; kk < kRowBytes / 32; ++kk) {
        const uint64_t koff = static_cast<uint64_t>((kk * 32) >> 4);
        const uint32_t accum = (ks | kk) != 0 ? 1u : 0u;
        if constexpr (PAIR) {
          ptx::mma_f16_pair(d_tmem, a_hi + koff, b_hi + koff, idesc, accum);
        } else if constexpr (!C::kSplit) {
          ptx::mma_f16(d_tmem, a_hi + koff, b_hi + koff, idesc, accum);
        } else {
          const uint64_t a_lo = ptx::sdesc_sw128(sa + C::kABytes + C::kBBytes);
          const uint64_t b_lo = ptx::sdesc_sw128(sa + 2 * C::kABytes + C::kBBytes);
          ptx::mma_tf32(d_tmem, a_hi + koff, b_hi + koff, idesc, accum);
          ptx::mma_tf32(d_tmem, a_hi + koff, b_lo + koff, idesc, 1u);
          ptx::mma_tf32(d_tmem, a_lo + koff, b_hi + koff, idesc, 1u);
        }
      }
      issued = true;
      if constexpr (PAIR)
        ptx::mma_commit_pair(&ctl->empty[stage], 0x3);
      else
        ptx::mma_commit(&ctl->empty[stage]);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (failed) break;
    if constexpr (PAIR)
      ptx::mma_commit_pair(&ctl->tfull[acc], 0x3);
    else
      ptx::mma_commit(&ctl->tfull[acc]);
    acc ^= 1;
    if (acc == 0) aph ^= 1u;
  }
  if (failed) {
    ctl->abort = 1;
    raise_status(args.hdr, kStTimeout, 3);
  }
  if (issued) {
    // Tensor memory is released only after every issued MMA has completed.
    int no_abort = 0;
    if constexpr (PAIR)
      ptx::mma_commit_pair(&ctl->drain, 0x1);
    else
      ptx::mma_commit(&ctl->drain);
    ptx::mbar_wait(&ctl->drain, 0u, lim, &no_abort);
  }
}

template <int DT, int ROWS, int STAGES>
__device__ void transformer(uint8_t* smem, Ctl<ROWS, STAGES>* ctl, const GemmArgs& args) {
  using C = Cfg<DT, ROWS, STAGES>;
  const uint64_t lim = args.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int tt = threadIdx.x - 32 * (2 + C::kEpiWarps);
  int stage = 0, qs = 0;
  uint32_t phase = 0, qph = 0;
  while (true) {
    bool ok = ptx::mbar_wait(&ctl->qfull[qs], qph, lim, abort);
    const int4 e = ctl->q[qs];
    if (bar_any(3, 128, !ok || ctl->abort)) break;
    if (tt == 0) ptx::mbar_arrive(&ctl->qempty[qs]);
    if (++qs == kQueue) {
      qs = 0;
      qph ^= 1u;
    }
    if (e.x < 0) break;
    const int n_b4 = (kDyMinRows << dy_box<ROWS>(e.z)) * kRowBytes / 16;
    bool stop = false;
    for (int ks = 0; ks < args.nk && !stop; ++ks) {
      ok = ptx::mbar_wait(&ctl->full[stage], phase, lim, abort);
      if (bar_any(3, 128, !ok || ctl->abort)) {
        stop = true;
        break;
      }
      uint8_t* s = smem + stage * C::kStageBytes;
      uint4* a = reinterpret_cast<uint4*>(s);
      uint4* b = reinterpret_cast<uint4*>(s + C::kABytes);
      uint4* a_lo = reinterpret_cast<uint4*>(s + C::kABytes + C::kBBytes);
      uint4* b_lo = reinterpret_cast<uint4*>(s + 2 * C::kABytes + C::kBBytes);
      auto split = [](uint4* hi, uint4* lo, int i) {
        uint4 x = hi[i], h, l;
        const uint32_t m = 0xFFFFE000u;
        h.x = x.x & m; h.y = x.y & m; h.z = x.z & m; h.w = x.w & m;
        l.x = __float_as_uint(__uint_as_float(x.x) - __uint_as_float(h.x)) & m;
        l.y = __float_as_uint(__uint_as_float(x.y) - __uint_as_float(h.y)) & m;
        l.z = __float_as_uint(__uint_as_float(x.z) - __uint_as_float(h.z)) & m;
        l.w = __float_as_uint(__uint_as_float(x.w) - __uint_as_float(h.w)) & m;
        hi[i] = h;
        lo[i] = l;
      };
      for (int i = tt; i < C::kABytes / 16; i += 128) split(a, a_lo, i);
      for (int i = tt; i < n_b4; i += 128) split(b, b_lo, i);
      ptx::fence_proxy_async_smem();
      ptx::named_bar_sync(3, 128);
      if (tt == 0) ptx::mbar_arrive(&ctl->ready[stage]);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (stop) break;
  }
}

// Gather warps of stage slot `slot` (gathered-operand kernel, rows of N * 2
// bytes that are 4-byte but not 16-byte multiples), two per slot: for each
// descriptor the scheduler posts to the slot, they copy the slot's 128 weight
// rows and `fill` d_y rows, 128-byte row segments (64 n) with cp.async as wide
// as each row's alignment allows, into the layout the tensor-memory-access
// unit would have written (128-byte swizzle: 16-byte chunk c of row r at chunk
// c ^ (r % 8) of the row's 128 bytes, rows 128 bytes apart), zero-filling rows
// and columns outside the operands. Each warp then waits for its copies, makes
// them visible to the tensor cores and arrives on the slot's full barrier (the
// even CTA's, for a pair).
template <int DT, int ROWS, int STAGES, bool PAIR>
__device__ void gatherer(uint8_t* smem, Ctl<ROWS, STAGES>* ctl, const GemmArgs& args) {
  using C = Cfg<DT, ROWS, STAGES, PAIR, true>;
  using T = Cfg<DT, ROWS, STAGES, PAIR, false>;
  static_assert(C::kStageBytes == T::kStageBytes && C::kMmaM == T::kMmaM &&
                    C::kWords == T::kWords && C::kABytes == T::kABytes,
                "the gathered operands fill the stages of the TMA variant");
  const uint64_t lim = args.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int gw = (threadIdx.x >> 5) - C::kGatherWarp0;
  const int slot = gw / C::kWarpsPerSlot, part = gw % C::kWarpsPerSlot;
  const int lane = threadIdx.x & 31;
  const uint32_t sa = ptx::smem_addr(smem + slot * C::kStageBytes);
  const uint32_t sb = sa + C::kABytes;
  const char* wb = static_cast<const char*>(args.w);
  const char* yb = static_cast<const char*>(args.dy);
  const void* safe = args.hdr;  // 64-byte aligned, named by zero-filling copies only
  const int64_t N = args.N, K = args.K;
  const int64_t row_bytes = N * 2;
  uint32_t full = 0;
  if constexpr (PAIR) full = ptx::mapa(&ctl->full[slot], 0);
  uint32_t phase = 0;
  while (true) {
    if (!ptx::mbar_wait(&ctl->dfull[slot], phase, lim, abort)) {
      if (!*abort) {
        ctl->abort = 1;
        if (lane == 0) raise_status(args.hdr, kStTimeout, 7);
      }
      break;
    }
    const GatherDesc d = ctl->desc[slot];
    if (d.g < 0) break;
    const int64_t left = (N - d.n0) * 2;  // bytes of the row segment inside N
    const int seg = left < 0 ? 0 : (left < kRowBytes ? static_cast<int>(left) : kRowBytes);
    const int64_t k0 = static_cast<int64_t>(d.kb) * kKBlock;
    const int64_t kn = K - k0 < kKBlock ? K - k0 : kKBlock;  // weight rows inside K
    gather_rows_sw128(sa, wb + ((static_cast<int64_t>(d.g) * K + k0) * N + d.n0) * 2, row_bytes,
                      kKBlock, kn < 0 ? 0 : static_cast<int>(kn), seg, safe, lane, part,
                      C::kWarpsPerSlot);
    gather_rows_sw128(sb, yb + (static_cast<int64_t>(d.row) * N + d.n0) * 2, row_bytes, d.fill,
                      d.valid, seg, safe, lane, part, C::kWarpsPerSlot);
    ptx::cp_async_commit();
    ptx::cp_async_wait<0>();
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if constexpr (PAIR)
        ptx::mbar_arrive_remote(full);
      else
        ptx::mbar_arrive(&ctl->full[slot]);
    }
    phase ^= 1u;
  }
  ptx::cp_async_wait<0>();
}

// Rows of the tile whose ticket says they may be added now. Thread et looks
// after rows et and et + 128; a warp ballot forms each 32-row mask word.
template <int ROWS>
__device__ __forceinline__ void ready_rows(EpiState<ROWS>* es, const GemmArgs& args, int R,
                                           uint32_t kb, bool gave_up) {
  constexpr int kWords = (ROWS + 31) / 32;
  const int et = (threadIdx.x - 64) & 127, ew = et >> 5, lane = threadIdx.x & 31;
  const uint32_t kbs = static_cast<uint32_t>(args.k_blocks);
  bool go[2] = {false, false};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = et + 128 * h;
    if (r < R && ((es->pend[r >> 5] >> (r & 31)) & 1u)) {
      const RowInfo m = es->meta[r];
      go[h] = m.rank == 0 || gave_up;
      if (!go[h]) {
        const uint32_t have =
            ptx::ld_acquire_gpu(args.tickets + static_cast<int64_t>(m.token) * kbs + kb);
        go[h] = have >= static_cast<uint32_t>(m.rank) + args.ticket_bias;
      }
    }
  }
  const uint32_t w0 = __ballot_sync(0xffffffffu, go[0]);
  const uint32_t w1 = __ballot_sync(0xffffffffu, go[1]);
  if (lane == 0) {
    if (ew < kWords) es->rdy[ew] = w0;
    if (ew + 4 < kWords) es->rdy[ew + 4] = w1;
  }
}

// One added to the ticket at p if `on` (a predicated reduction, no branch).
__device__ __forceinline__ void red_add_one_if(uint32_t* p, uint32_t on) {
  asm volatile(
      "{\n"
      ".reg .pred q;\n"
      "setp.ne.u32 q, %1, 0;\n"
      "@q red.relaxed.gpu.global.add.u32 [%0], 1;\n"
      "}\n" ::"l"(p),
      "r"(on)
      : "memory");
}

// Four consecutive fp32 to p: stored if `st`, added at L2 if `add`, neither
// otherwise (predicated instructions, no branch).
__device__ __forceinline__ void store_or_add_v4(float* p, float4 v, bool st, bool add) {
  asm volatile(
      "{\n"
      ".reg .pred ps, pa;\n"
      "setp.ne.u32 ps, %5, 0;\n"
      "setp.ne.u32 pa, %6, 0;\n"
      "@ps st.global.v4.f32 [%0], {%1, %2, %3, %4};\n"
      "@pa red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};\n"
      "}\n" ::"l"(p),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(st ? 1u : 0u), "r"(add ? 1u : 0u)
      : "memory");
}

// Writes the ready rows without leaving registers. A tensor-memory load gives
// lane l of warp q the value of k = 32q + l for kChunk rows. Two xor-shuffle
// stages transpose every 4 x 4 block (lane bits 0-1 <-> row bits 0-1), after
// which lane l holds k = 32q + 4(l/4) .. +3 of row 4s + (l % 4). The eight lanes
// sharing a row then cover its 128 contiguous bytes of this warp's quarter, and
// one v4 store (rank 0) or v4 fp32 reduction at L2 (rank > 0) per lane writes
// four rows per warp instruction. Needs K % 4 == 0.
template <int ROWS>
__device__ __forceinline__ void write_rows_vec(const EpiState<ROWS>* es, const GemmArgs& args,
                                               uint32_t t_lane, int R, uint32_t kb, int quarter) {
  const int lane = threadIdx.x & 31;
  const int64_t K = args.K;
  const int64_t k = static_cast<int64_t>(kb) * kKBlock + 32 * quarter + 4 * (lane >> 2);
  const bool k_ok = k < K;  // K % 4 == 0: a lane's four k are all in or all out
  const bool up = (lane & 2) != 0, odd = (lane & 1) != 0;
  const int nchunks = (R + kChunk - 1) / kChunk;
  for (int c = 0; c < nchunks; ++c) {
    const int r_lo = c * kChunk;
    const uint32_t word = es->rdy[r_lo >> 5] >> (r_lo & 31);  // bits of this chunk's rows
    if ((word & kChunkMask) == 0u) continue;  // warp-uniform
    uint32_t v[kChunk];
    ptx::tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(r_lo), v);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int g = 0; g < kChunk / 4; ++g) {
      uint32_t r0 = v[4 * g], r1 = v[4 * g + 1], r2 = v[4 * g + 2], r3 = v[4 * g + 3];
      // exchange across lane bit 1 <-> row bit 1
      uint32_t t0 = __shfl_xor_sync(0xffffffffu, up ? r0 : r2, 2);
      uint32_t t1 = __shfl_xor_sync(0xffffffffu, up ? r1 : r3, 2);
      if (up) {
        r0 = t0;
        r1 = t1;
      } else {
        r2 = t0;
        r3 = t1;
      }
      // exchange across lane bit 0 <-> row bit 0
      t0 = __shfl_xor_sync(0xffffffffu, odd ? r0 : r1, 1);
      t1 = __shfl_xor_sync(0xffffffffu, odd ? r2 : r3, 1);
      if (odd) {
        r0 = t0;
        r2 = t1;
      } else {
        r1 = t0;
        r3 = t1;
      }
      // every lane issues both writes, predicated: no divergence between the
      // rows of a warp instruction (their ranks and readiness differ)
      const int j = 4 * g + (lane & 3);
      const int r = r_lo + j;  // < ROWS: a record in bounds, stale past R
      const bool wr = r < R && ((word >> j) & 1u) && k_ok;
      const RowInfo m = es->meta[r];
      float* dst = args.out + static_cast<int64_t>(m.token) * K + k;
      const float4 x = make_float4(__uint_as_float(r0), __uint_as_float(r1), __uint_as_float(r2),
                                   __uint_as_float(r3));
      store_or_add_v4(dst, x, wr && m.rank == 0, wr && m.rank != 0);
    }
  }
}

// Scalar path for K % 4 != 0: lane = k, one 128-byte store or reduction per
// row and warp.
template <int ROWS>
__device__ __forceinline__ void write_rows_scalar(const EpiState<ROWS>* es, const GemmArgs& args,
                                                  uint32_t t_lane, int R, uint32_t kb,
                                                  int quarter) {
  const int lane = threadIdx.x & 31;
  const int64_t K = args.K;
  const int64_t k = static_cast<int64_t>(kb) * kKBlock + 32 * quarter + lane;
  const bool k_ok = k < K;
  const int nchunks = (R + 31) / 32;
  for (int c = 0; c < nchunks; ++c) {
    uint32_t v[32];
    ptx::tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(c * 32), v);
    ptx::tmem_ld_wait();
    const uint32_t word = es->rdy[c];
    if (k_ok && word) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (word & (1u << j)) {
          const RowInfo m = es->meta[c * 32 + j];
          float* p = args.out + static_cast<int64_t>(m.token) * K + k;
          const float x = __uint_as_float(v[j]);
          if (m.rank == 0)
            *p = x;
          else
            ptx::red_add_f32_gpu(p, x);
        }
      }
    }
  }
}

template <int DT, int ROWS, int STAGES, bool PAIR>
__device__ void epilogue(Ctl<ROWS, STAGES>* ctl, uint32_t tmem_base, const GemmArgs& args,
                         uint32_t rank) {
  using C = Cfg<DT, ROWS, STAGES, PAIR>;
  const uint64_t lim = args.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int et = (threadIdx.x - 64) & 127;  // thread within the group
  const int grp = (threadIdx.x - 64) >> 7;   // epilogue group: drains accumulator buffer grp
  const uint32_t bar = 1u + static_cast<uint32_t>(grp);
  EpiState<ROWS>* es = &ctl->epi[grp];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;     // tensor-memory lanes this warp may read
  const uint32_t kbs = static_cast<uint32_t>(args.k_blocks);
  const bool remote = PAIR && rank != 0;  // queue and accumulator barriers live in the even CTA
  bool gave_up = false;
  // The group takes every kEpiGroups-th tile of the queue, starting at its index.
  for (uint32_t n = 0;; ++n) {
    const uint32_t i = n * C::kEpiGroups + static_cast<uint32_t>(grp);
    const int qs = static_cast<int>(i % kQueue);
    const uint32_t qph = (i / kQueue) & 1u;
    const int acc = static_cast<int>(i & 1u);
    const uint32_t aph = (i >> 1) & 1u;
    bool ok = remote ? ptx::mbar_wait_cluster(&ctl->qfull[qs], qph, lim, abort)
                     : ptx::mbar_wait(&ctl->qfull[qs], qph, lim, abort);
    const int4 e = ctl->q[qs];
    if (bar_any(bar, 128, !ok || ctl->abort)) {
      if (!ok) {
        ctl->abort = 1;
        if (et == 0) raise_status(args.hdr, kStTimeout, 4);
      }
      break;
    }
    if (et == 0) {
      if (remote)
        ptx::mbar_arrive_remote(ptx::mapa(&ctl->qempty[qs], 0));
      else
        ptx::mbar_arrive(&ctl->qempty[qs]);
    }
    if (e.x < 0) break;
    const int R = e.z, row0 = e.y;
    const uint32_t kb = PAIR ? 2u * static_cast<uint32_t>(e.w) + rank : static_cast<uint32_t>(e.w);
    const bool kb_ok = kb < kbs;  // a pair's odd half may lie beyond K
    for (int r = et; r < R; r += 128) {
      RowInfo m = args.rowinfo[check_index(args.hdr, row0 + r, args.M, 42)];
      m.token = static_cast<int32_t>(check_index(args.hdr, m.token, args.batch, 43));
      es->meta[r] = m;
    }
    if (et < C::kWords) {
      const int nr = kb_ok ? R - et * 32 : 0;
      es->pend[et] = nr >= 32 ? 0xFFFFFFFFu : (nr <= 0 ? 0u : ((1u << nr) - 1u));
    }
    ok = PAIR ? ptx::mbar_wait_cluster(&ctl->tfull[acc], aph, lim, abort)
              : ptx::mbar_wait(&ctl->tfull[acc], aph, lim, abort);
    if (bar_any(bar, 128, !ok || ctl->abort)) {
      if (!ok) {
        ctl->abort = 1;
        if (et == 0) raise_status(args.hdr, kStTimeout, 5);
      }
      break;
    }
    ptx::tc_fence_after_sync();

    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) +
                            static_cast<uint32_t>(acc * C::kAccCols);
    uint64_t t_wait0 = 0;
    // (a tile without rows, which only the checked build's substitution for a
    // bad row block makes, has nothing to wait for)
    while (kb_ok && R > 0) {
      // 1. which pending rows may go now
      ready_rows(es, args, R, kb, gave_up);
      ptx::named_bar_sync(bar, 128);
      bool any = false;
#pragma unroll
      for (int w = 0; w < C::kWords; ++w) any |= es->rdy[w] != 0u;
      if (!any) {
        if (t_wait0 == 0) t_wait0 = ptx::globaltimer();
        const bool expired = (ptx::globaltimer() - t_wait0 > lim) ||
                             *reinterpret_cast<volatile uint32_t*>(&args.hdr->status) == kStTimeout;
        if (bar_any(bar, 128, expired)) {
          gave_up = true;
          if (et == 0) raise_status(args.hdr, kStTimeout, 1);
        } else {
          __nanosleep(256);
        }
        continue;
      }
      t_wait0 = 0;  // progress: the limit counts time without any
      // 2. write the ready rows
      if (args.vec_rows)
        write_rows_vec(es, args, t_lane, R, kb, quarter);
      else
        write_rows_scalar(es, args, t_lane, R, kb, quarter);
      ptx::named_bar_sync(bar, 128);
      // 3. publish: the rows' additions happen-before the ticket bumps
      bool mine = false;
      for (int r = et; r < R; r += 128) mine |= (es->rdy[r >> 5] >> (r & 31)) & 1u;
      if (mine) {
        ptx::fence_acq_rel_gpu();
        for (int r = et; r < R; r += 128)
          red_add_one_if(args.tickets + static_cast<int64_t>(es->meta[r].token) * kbs + kb,
                         (es->rdy[r >> 5] >> (r & 31)) & 1u);
      }
      if (et < C::kWords) es->pend[et] &= ~es->rdy[et];
      ptx::named_bar_sync(bar, 128);
      bool left = false;
#pragma unroll
      for (int w = 0; w < C::kWords; ++w) left |= es->pend[w] != 0u;
      if (!left) break;
    }
    ptx::tc_fence_before_sync();
    __syncwarp();
    // The accumulator is free again. What changes hands is tensor memory,
    // ordered by the tcgen05 fences on both sides of the barrier; the rows'
    // global writes go to other tiles through the tickets, not to the MMA
    // thread. So the odd CTA arrives at CTA scope too: a cluster-scope release
    // here waits for the warp's ticket reductions to reach L2 first.
    if (lane == 0) {
      if (remote)
        ptx::mbar_arrive_remote_cta(ptx::mapa(&ctl->tempty[acc], 0));
      else
        ptx::mbar_arrive(&ctl->tempty[acc]);
    }
  }
}

template <int DT, int ROWS, int STAGES, bool PAIR, bool GATHER>
__global__ void __launch_bounds__(Cfg<DT, ROWS, STAGES, PAIR, GATHER>::kThreads, 1)
    gmm_dx_kernel(const __grid_constant__ DyMaps dy_maps, const __grid_constant__ CUtensorMap tm_w,
                  const GemmArgs args) {
  using C = Cfg<DT, ROWS, STAGES, PAIR, GATHER>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  auto* ctl = reinterpret_cast<Ctl<ROWS, STAGES>*>(smem + STAGES * C::kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;

  // Launched with programmatic serialization: the routing (or the owner
  // kernel) before this one has finished and its memory is visible past here.
  ptx::griddep_wait();
  // Routing validation failed: the result is defined as zeros. (Both CTAs of
  // a pair see the same status and leave before any cluster operation.)
  const uint32_t st = args.hdr->status;
  if (st == kStIndex || st == kStGroupSum || st == kStNotPerm) {
    const int64_t n = args.batch * args.K;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < n;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x)
      args.out[q] = 0.0f;
    return;
  }
  // After the owner kernel: nothing to do unless it had to leave the work here.
  if (args.only_if_unsorted && args.hdr->unsorted == 0) return;
  const uint32_t total = args.hdr->n_row_blocks * static_cast<uint32_t>(args.k_units);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // gathered operands: one arrival from each gather warp of the slot, in each CTA
      ptx::mbar_init(&ctl->full[s], GATHER ? C::kWarpsPerSlot * (PAIR ? 2 : 1) : 1);
      ptx::mbar_init(&ctl->empty[s], 1);
      ptx::mbar_init(&ctl->ready[s], 1);
      ptx::mbar_init(&ctl->dfull[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&ctl->tfull[a], 1);
      ptx::mbar_init(&ctl->tempty[a], C::kTEmpty);
    }
    for (int q = 0; q < kQueue; ++q) {
      ptx::mbar_init(&ctl->qfull[q], 1);
      ptx::mbar_init(&ctl->qempty[q], C::kQEmpty);
    }
    ptx::mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (!GATHER && warp == 0 && lane == 0) {
    for (int j = 0; j < kDyMaps; ++j) ptx::tma_prefetch_desc(&dy_maps.box[j]);
    ptx::tma_prefetch_desc(&tm_w);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(&ctl->tmem_base, C::kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(&ctl->tmem_base, C::kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  if constexpr (PAIR) ptx::cluster_sync();  // the peer's barriers are initialised
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0)
      producer<DT, ROWS, STAGES, PAIR, GATHER>(smem, ctl, &dy_maps, &tm_w, args, total, rank);
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) mma_issuer<DT, ROWS, STAGES, PAIR>(smem, ctl, tmem_base, args);
  } else if (warp < 2 + C::kEpiWarps) {
    epilogue<DT, ROWS, STAGES, PAIR>(ctl, tmem_base, args, rank);
  } else if (warp < C::kGatherWarp0) {
    if constexpr (C::kSplit) transformer<DT, ROWS, STAGES>(smem, ctl, args);
  } else {
    if constexpr (GATHER) gatherer<DT, ROWS, STAGES, PAIR>(smem, ctl, args);
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if constexpr (PAIR) ptx::cluster_sync();  // no CTA leaves while its peer may still use it
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    if constexpr (PAIR)
      ptx::tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else
      ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int DT, int ROWS, int STAGES, bool PAIR, bool GATHER>
cudaError_t launch_t(const DyMaps& tdy, const CUtensorMap& tw, const GemmArgs& args, int max_ctas,
                     cudaStream_t stream) {
  using C = Cfg<DT, ROWS, STAGES, PAIR, GATHER>;
  constexpr int smem = smem_bytes<DT, ROWS, STAGES, PAIR>();
  auto kern = gmm_dx_kernel<DT, ROWS, STAGES, PAIR, GATHER>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  if constexpr (!PAIR) {
    return launch_pdl(kern, dim3(static_cast<unsigned>(max_ctas)), dim3(C::kThreads), smem, stream,
                      1, tdy, tw, args);
  } else {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(2 * ((max_ctas + 1) / 2), 1, 1);
    int clusters = 0;
    err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (err != cudaSuccess) return err;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    const int want = (max_ctas + 1) / 2;
    return launch_pdl(kern, dim3(2 * static_cast<unsigned>(clusters < want ? clusters : want)),
                      dim3(C::kThreads), smem, stream, 2, tdy, tw, args);
  }
}

// (dtype, variant) -> (rows per block, stages, CTA pair, gathered operands);
// variant 5 is variant 0 with its operands copied by gather warps.
#define PGG_VARIANTS(X)                \
  X(PGG_BF16, 0, 256, 6, true, false)  \
  X(PGG_BF16, 1, 32, 10, false, false) \
  X(PGG_BF16, 2, 256, 4, false, false) \
  X(PGG_BF16, 5, 256, 6, true, true)   \
  X(PGG_F16, 0, 256, 6, true, false)   \
  X(PGG_F16, 1, 32, 10, false, false)  \
  X(PGG_F16, 2, 256, 4, false, false)  \
  X(PGG_F16, 5, 256, 6, true, true)    \
  X(PGG_F32, 0, 128, 3, false, false)  \
  X(PGG_F32, 1, 32, 4, false, false)

}  // namespace

bool kernel_config(int dtype, int variant, int* rows, int* stages, int* threads, int* smem,
                   int* pair) {
#define PGG_CFG(DT, V, R, S, P, GA)             \
  if (dtype == DT && variant == V) {            \
    *rows = R;                                  \
    *stages = S;                                \
    *threads = Cfg<DT, R, S, P, GA>::kThreads;  \
    *smem = smem_bytes<DT, R, S, P>();          \
    *pair = P ? 1 : 0;                          \
    return true;                                \
  }
  PGG_VARIANTS(PGG_CFG)
#undef PGG_CFG
  return false;
}

cudaError_t launch_grouped_gemm(int dtype, int variant, const DyMaps& tdy, const CUtensorMap& tw,
                                const GemmArgs& args, int max_ctas, cudaStream_t stream) {
#define PGG_LAUNCH(DT, V, R, S, P, GA) \
  if (dtype == DT && variant == V)     \
    return launch_t<DT, R, S, P, GA>(tdy, tw, args, max_ctas, stream);
  PGG_VARIANTS(PGG_LAUNCH)
#undef PGG_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace pgg
