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
// in tensor memory holds lane = k, column = expanded row. The epilogue moves
// each expanded row's 128 values of k into a shared-memory staging row and
// hands the 512-byte segment of d_x to the tensor-memory-access unit as one
// bulk store or bulk fp32 reduce-add (the addition happens in L2), so the
// scatter-add costs the SM a handful of instructions per row.
//
// Warp roles (one CTA per SM, persistent):
//   warp 0       tile scheduler + TMA producer (one lane)
//   warp 1       TMEM allocation + MMA issuer (one lane)
//   warps 2..5   epilogue: TMEM -> registers -> ordered scatter-add into d_x
//   warps 6..9   fp32 inputs only: split each staged fp32 tile into tf32
//                high and low parts for the 3-product tf32 MMA
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

template <int DT, int ROWS, int STAGES>
struct Cfg {
  static constexpr bool kSplit = DtTraits<DT>::kSplit;
  static constexpr int kElemsPerRow = kRowBytes / DtTraits<DT>::kElem;
  static constexpr int kABytes = kKBlock * kRowBytes;
  static constexpr int kBBytes = ROWS * kRowBytes;
  static constexpr int kStageBytes = (kABytes + kBBytes) * (kSplit ? 2 : 1);
  static constexpr int kAccCols = ROWS < 32 ? 32 : ROWS;
  static constexpr int kTmemCols = pow2_at_least(2 * kAccCols);  // allocation unit
  static constexpr int kWords = (ROWS + 31) / 32;
  static constexpr int kEpiWarps = 4;
  static constexpr int kXformWarps = kSplit ? 4 : 0;
  static constexpr int kThreads = 32 * (2 + kEpiWarps + kXformWarps);
  static_assert(ROWS % 32 == 0 && ROWS <= 256, "rows per block");
  static_assert((kTmemCols & (kTmemCols - 1)) == 0 && kTmemCols <= 512, "tmem columns");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
};

// Epilogue staging for the bulk path: rows x 128 fp32 (one 512-byte d_x row
// segment per expanded row), two buffers of kChunk rows.
constexpr int kChunk = 16;

template <int ROWS, int STAGES>
struct Ctl {
  float stg[2][kChunk][kKBlock];
  uint64_t full[STAGES];   // TMA bytes landed
  uint64_t empty[STAGES];  // MMAs reading the stage completed
  uint64_t ready[STAGES];  // fp32 split done
  uint64_t tfull[2];       // accumulator complete
  uint64_t tempty[2];      // accumulator drained by the epilogue
  uint64_t qfull[kQueue];
  uint64_t qempty[kQueue];
  uint64_t drain;
  int4 q[kQueue];  // {expert (-1 = stop), first row, rows, k block}
  uint32_t tmem_base;
  int abort;
  uint32_t pend[(ROWS + 31) / 32];
  uint32_t rdy[(ROWS + 31) / 32];
  RowInfo meta[ROWS];
};

template <int DT, int ROWS, int STAGES>
constexpr int smem_bytes() {
  return 1024 + STAGES * Cfg<DT, ROWS, STAGES>::kStageBytes + static_cast<int>(sizeof(Ctl<ROWS, STAGES>));
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

// Index of the smallest d_y box (32 << j rows, at most ROWS) that covers R rows.
template <int ROWS>
__device__ __forceinline__ int dy_box(int R) {
  int j = 0;
  while ((kDyMinRows << j) < R && (kDyMinRows << j) < ROWS) ++j;
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

template <int DT, int ROWS, int STAGES>
__device__ void producer(uint8_t* smem, Ctl<ROWS, STAGES>* ctl, const DyMaps* dy_maps,
                         const CUtensorMap* tm_w, const GemmArgs& args, uint32_t total) {
  using C = Cfg<DT, ROWS, STAGES>;
  const uint64_t lim = args.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  int stage = 0, qs = 0;
  uint32_t phase = 0, qph = 0, outstanding = 0, last_parity = 0;
  const uint32_t n_rb = args.hdr->n_row_blocks;
  const uint32_t kbs = static_cast<uint32_t>(args.k_blocks);
  const uint32_t band = static_cast<uint32_t>(args.band_k_blocks);
  auto entry = [&](uint32_t t) {
    if (t >= total) return make_int4(-1, 0, 0, 0);
    uint32_t rb, kb;
    decode_tile(t, n_rb, kbs, band, &rb, &kb);
    const int4 r = args.rblist[rb];
    return make_int4(r.x, r.y, r.z, static_cast<int>(kb));
  };
  // The next tile is claimed and its row block read while the current one
  // streams, so no tile starts with a scheduler round trip.
  int4 e = entry(atomicAdd(&args.hdr->sched_next, 1u));
  bool failed = false;
  while (!failed) {
    const uint32_t t_next = e.x >= 0 ? atomicAdd(&args.hdr->sched_next, 1u) : total;
    if (!ptx::mbar_wait(&ctl->qempty[qs], qph ^ 1u, lim, abort)) {
      failed = true;
      break;
    }
    ctl->q[qs] = e;
    ptx::mbar_arrive(&ctl->qfull[qs]);
    if (++qs == kQueue) {
      qs = 0;
      qph ^= 1u;
    }
    if (e.x < 0) break;
    const int bj = dy_box<ROWS>(e.z);
    const CUtensorMap* tm_dy = &dy_maps->box[bj];
    const uint32_t tx = C::kABytes + static_cast<uint32_t>(kDyMinRows << bj) * kRowBytes;
    int4 e_next = make_int4(-1, 0, 0, 0);
    bool have_next = false;
    for (int ks = 0; ks < args.nk; ++ks) {
      if (!ptx::mbar_wait(&ctl->empty[stage], phase ^ 1u, lim, abort)) {
        failed = true;
        break;
      }
      uint8_t* sa = smem + stage * C::kStageBytes;
      ptx::mbar_arrive_expect_tx(&ctl->full[stage], tx);
      const int32_t n0 = ks * C::kElemsPerRow;
      ptx::tma_load_3d(sa, tm_w, &ctl->full[stage], n0, e.w * kKBlock, e.x);
      ptx::tma_load_2d(sa + C::kABytes, tm_dy, &ctl->full[stage], n0, e.y);
      outstanding |= 1u << stage;
      last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
      if (ks == 1 || ks + 1 == args.nk) {
        if (!have_next) {
          e_next = entry(t_next);
          have_next = true;
        }
      }
    }
    if (!have_next) e_next = entry(t_next);
    e = e_next;
  }
  if (failed) {
    ctl->abort = 1;
    raise_status(args.hdr, kStTimeout, 2);
  }
  // Never leave while a copy into this CTA's shared memory may be in flight.
  int no_abort = 0;
  for (int s = 0; s < STAGES; ++s)
    if (outstanding & (1u << s))
      ptx::mbar_wait(&ctl->full[s], (last_parity >> s) & 1u, lim, &no_abort);
}

template <int DT, int ROWS, int STAGES>
__device__ void mma_issuer(uint8_t* smem, Ctl<ROWS, STAGES>* ctl, uint32_t tmem_base,
                           const GemmArgs& args) {
  using C = Cfg<DT, ROWS, STAGES>;
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
    uint32_t n_mma = (static_cast<uint32_t>(e.z) + 15u) & ~15u;
    if (n_mma < 16u) n_mma = 16u;
    const uint32_t idesc = ptx::idesc_make(DtTraits<DT>::kFmt, kKBlock, n_mma);
    if (!ptx::mbar_wait(&ctl->tempty[acc], aph ^ 1u, lim, abort)) {
      failed = true;
      break;
    }
    ptx::tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::kAccCols);
    for (int ks = 0; ks < args.nk; ++ks) {
      uint64_t* bar = C::kSplit ? &ctl->ready[stage] : &ctl->full[stage];
      if (!ptx::mbar_wait(bar, phase, lim, abort)) {
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
        if constexpr (!C::kSplit) {
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
      ptx::mma_commit(&ctl->empty[stage]);
      if (++stage == STAGES) {
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
    raise_status(args.hdr, kStTimeout, 3);
  }
  if (issued) {
    // Tensor memory is released only after every issued MMA has completed.
    int no_abort = 0;
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
    if (bar_any(2, 128, !ok || ctl->abort)) break;
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
      if (bar_any(2, 128, !ok || ctl->abort)) {
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
      ptx::named_bar_sync(2, 128);
      if (tt == 0) ptx::mbar_arrive(&ctl->ready[stage]);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (stop) break;
  }
}

// Rows of the tile whose ticket says they may be added now. Thread et looks
// after rows et and et + 128; a warp ballot forms each 32-row mask word.
template <int ROWS, int STAGES>
__device__ __forceinline__ void ready_rows(Ctl<ROWS, STAGES>* ctl, const GemmArgs& args, int R,
                                           uint32_t kb, bool gave_up) {
  constexpr int kWords = (ROWS + 31) / 32;
  const int et = threadIdx.x - 64, ew = et >> 5, lane = threadIdx.x & 31;
  const uint32_t kbs = static_cast<uint32_t>(args.k_blocks);
  bool go[2] = {false, false};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = et + 128 * h;
    if (r < R && ((ctl->pend[r >> 5] >> (r & 31)) & 1u)) {
      const RowInfo m = ctl->meta[r];
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
    if (ew < kWords) ctl->rdy[ew] = w0;
    if (ew + 4 < kWords) ctl->rdy[ew + 4] = w1;
  }
}

// Writes the ready rows through the tensor-memory-access unit: each warp moves
// its 32 k values of kChunk rows from tensor memory into a staging row
// [row][128 k] in shared memory; one thread per row then issues a bulk copy
// (rank 0) or bulk fp32 reduce-add (rank > 0) of the row's segment of d_x.
// Needs K % 4 == 0 (16-byte aligned segments).
template <int ROWS, int STAGES>
__device__ __forceinline__ void write_rows_bulk(Ctl<ROWS, STAGES>* ctl, const GemmArgs& args,
                                                uint32_t t_lane, int R, uint32_t kb, int quarter) {
  const int et = threadIdx.x - 64, ew = et >> 5, lane = threadIdx.x & 31;
  const int64_t K = args.K;
  const int64_t k0 = static_cast<int64_t>(kb) * kKBlock;
  const uint32_t bytes = static_cast<uint32_t>((K - k0 < kKBlock ? K - k0 : kKBlock) * 4);
  const int nchunks = (R + kChunk - 1) / kChunk;
  bool fenced = false;
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    // the warp that issued chunk c - 2 from this buffer waits for its reads
    if (c >= 2 && ew == ((c - 2) & 3)) ptx::bulk_wait_read_all();
    uint32_t v[kChunk];
    ptx::tmem_ld_32x32b_x16(t_lane + static_cast<uint32_t>(c * kChunk), v);
    ptx::tmem_ld_wait();
    ptx::named_bar_sync(1, 128);
#pragma unroll
    for (int j = 0; j < kChunk; ++j) ctl->stg[buf][j][32 * quarter + lane] = __uint_as_float(v[j]);
    ptx::fence_proxy_async_smem();
    ptx::named_bar_sync(1, 128);
    if (ew == (c & 3) && lane < kChunk) {
      const int r = c * kChunk + lane;
      if (r < R && ((ctl->rdy[r >> 5] >> (r & 31)) & 1u)) {
        const RowInfo m = ctl->meta[r];
        float* dst = args.out + static_cast<int64_t>(m.token) * K + k0;
        if (!fenced) {
          ptx::fence_proxy_async_global();
          fenced = true;
        }
        if (m.rank == 0)
          ptx::bulk_store(dst, &ctl->stg[buf][lane][0], bytes);
        else
          ptx::bulk_reduce_add_f32(dst, &ctl->stg[buf][lane][0], bytes);
      }
      ptx::bulk_commit();
    }
  }
  // every issued row is complete (performed in global memory) before its
  // ticket is published
  ptx::bulk_wait_all();
  ptx::fence_proxy_async_global();
}

// Scalar path for K % 4 != 0: lane = k, one 128-byte store or reduction per
// row and warp.
template <int ROWS, int STAGES>
__device__ __forceinline__ void write_rows_scalar(Ctl<ROWS, STAGES>* ctl, const GemmArgs& args,
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
    const uint32_t word = ctl->rdy[c];
    if (k_ok && word) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (word & (1u << j)) {
          const RowInfo m = ctl->meta[c * 32 + j];
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

template <int DT, int ROWS, int STAGES>
__device__ void epilogue(Ctl<ROWS, STAGES>* ctl, uint32_t tmem_base, const GemmArgs& args) {
  using C = Cfg<DT, ROWS, STAGES>;
  const uint64_t lim = args.wait_limit_ns;
  volatile int* abort = &ctl->abort;
  const int et = threadIdx.x - 64;  // 0..127
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;     // tensor-memory lanes this warp may read
  const uint32_t kbs = static_cast<uint32_t>(args.k_blocks);
  int qs = 0, acc = 0;
  uint32_t qph = 0, aph = 0;
  bool gave_up = false;
  while (true) {
    bool ok = ptx::mbar_wait(&ctl->qfull[qs], qph, lim, abort);
    const int4 e = ctl->q[qs];
    if (bar_any(1, 128, !ok || ctl->abort)) {
      if (!ok) {
        ctl->abort = 1;
        if (et == 0) raise_status(args.hdr, kStTimeout, 4);
      }
      break;
    }
    if (et == 0) ptx::mbar_arrive(&ctl->qempty[qs]);
    if (++qs == kQueue) {
      qs = 0;
      qph ^= 1u;
    }
    if (e.x < 0) break;
    const int R = e.z, row0 = e.y;
    const uint32_t kb = static_cast<uint32_t>(e.w);
    for (int r = et; r < R; r += 128) ctl->meta[r] = args.rowinfo[row0 + r];
    if (et < C::kWords) {
      const int n = R - et * 32;
      ctl->pend[et] = n >= 32 ? 0xFFFFFFFFu : (n <= 0 ? 0u : ((1u << n) - 1u));
    }
    ok = ptx::mbar_wait(&ctl->tfull[acc], aph, lim, abort);
    if (bar_any(1, 128, !ok || ctl->abort)) {
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
    while (true) {
      // 1. which pending rows may go now
      ready_rows(ctl, args, R, kb, gave_up);
      ptx::named_bar_sync(1, 128);
      bool any = false;
#pragma unroll
      for (int w = 0; w < C::kWords; ++w) any |= ctl->rdy[w] != 0u;
      if (!any) {
        if (t_wait0 == 0) t_wait0 = ptx::globaltimer();
        const bool expired = (ptx::globaltimer() - t_wait0 > lim) ||
                             *reinterpret_cast<volatile uint32_t*>(&args.hdr->status) == kStTimeout;
        if (bar_any(1, 128, expired)) {
          gave_up = true;
          if (et == 0) raise_status(args.hdr, kStTimeout, 1);
        } else {
          __nanosleep(256);
        }
        continue;
      }
      // 2. write the ready rows
      if (args.bulk)
        write_rows_bulk(ctl, args, t_lane, R, kb, quarter);
      else
        write_rows_scalar(ctl, args, t_lane, R, kb, quarter);
      ptx::named_bar_sync(1, 128);
      // 3. publish: the rows' additions happen-before the ticket bumps
      bool mine = false;
      for (int r = et; r < R; r += 128) mine |= (ctl->rdy[r >> 5] >> (r & 31)) & 1u;
      if (mine) {
        ptx::fence_acq_rel_gpu();
        for (int r = et; r < R; r += 128)
          if ((ctl->rdy[r >> 5] >> (r & 31)) & 1u)
            ptx::red_add_u32_gpu(args.tickets + static_cast<int64_t>(ctl->meta[r].token) * kbs + kb,
                                 1u);
      }
      if (et < C::kWords) ctl->pend[et] &= ~ctl->rdy[et];
      ptx::named_bar_sync(1, 128);
      bool left = false;
#pragma unroll
      for (int w = 0; w < C::kWords; ++w) left |= ctl->pend[w] != 0u;
      if (!left) break;
    }
    ptx::tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&ctl->tempty[acc]);
    acc ^= 1;
    if (acc == 0) aph ^= 1u;
  }
}

template <int DT, int ROWS, int STAGES>
__global__ void __launch_bounds__(Cfg<DT, ROWS, STAGES>::kThreads, 1)
    gmm_dx_kernel(const __grid_constant__ DyMaps dy_maps, const __grid_constant__ CUtensorMap tm_w,
                  const GemmArgs args) {
  using C = Cfg<DT, ROWS, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  auto* ctl = reinterpret_cast<Ctl<ROWS, STAGES>*>(smem + STAGES * C::kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Routing validation failed: the result is defined as zeros.
  const uint32_t st = args.hdr->status;
  if (st == kStIndex || st == kStGroupSum || st == kStNotPerm) {
    const int64_t n = args.batch * args.K;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < n;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x)
      args.out[q] = 0.0f;
    return;
  }
  const uint32_t total = args.hdr->n_row_blocks * static_cast<uint32_t>(args.k_blocks);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&ctl->full[s], 1);
      ptx::mbar_init(&ctl->empty[s], 1);
      ptx::mbar_init(&ctl->ready[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&ctl->tfull[a], 1);
      ptx::mbar_init(&ctl->tempty[a], C::kEpiWarps);
    }
    for (int q = 0; q < kQueue; ++q) {
      ptx::mbar_init(&ctl->qfull[q], 1);
      ptx::mbar_init(&ctl->qempty[q], C::kSplit ? 3 : 2);
    }
    ptx::mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int j = 0; j < kDyMaps; ++j) ptx::tma_prefetch_desc(&dy_maps.box[j]);
    ptx::tma_prefetch_desc(&tm_w);
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) producer<DT, ROWS, STAGES>(smem, ctl, &dy_maps, &tm_w, args, total);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<DT, ROWS, STAGES>(smem, ctl, tmem_base, args);
  } else if (warp < 2 + C::kEpiWarps) {
    epilogue<DT, ROWS, STAGES>(ctl, tmem_base, args);
  } else {
    transformer<DT, ROWS, STAGES>(smem, ctl, args);
  }

  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int DT, int ROWS, int STAGES>
cudaError_t launch_t(const DyMaps& tdy, const CUtensorMap& tw, const GemmArgs& args, int grid,
                     cudaStream_t stream) {
  using C = Cfg<DT, ROWS, STAGES>;
  constexpr int smem = smem_bytes<DT, ROWS, STAGES>();
  auto kern = gmm_dx_kernel<DT, ROWS, STAGES>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  kern<<<grid, C::kThreads, smem, stream>>>(tdy, tw, args);
  return cudaGetLastError();
}

// (dtype, variant) -> (rows per block, stages)
#define PGG_VARIANTS(X)      \
  X(PGG_BF16, 0, 256, 4)     \
  X(PGG_BF16, 1, 32, 10)     \
  X(PGG_F16, 0, 256, 4)      \
  X(PGG_F16, 1, 32, 10)      \
  X(PGG_F32, 0, 128, 3)      \
  X(PGG_F32, 1, 32, 4)

}  // namespace

bool kernel_config(int dtype, int variant, int* rows, int* stages, int* threads, int* smem) {
#define PGG_CFG(DT, V, R, S)                          \
  if (dtype == DT && variant == V) {                  \
    *rows = R;                                        \
    *stages = S;                                      \
    *threads = Cfg<DT, R, S>::kThreads;               \
    *smem = smem_bytes<DT, R, S>();                   \
    return true;                                      \
  }
  PGG_VARIANTS(PGG_CFG)
#undef PGG_CFG
  return false;
}

cudaError_t launch_grouped_gemm(int dtype, int variant, const DyMaps& tdy, const CUtensorMap& tw,
                                const GemmArgs& args, int grid, cudaStream_t stream) {
#define PGG_LAUNCH(DT, V, R, S) \
  if (dtype == DT && variant == V) return launch_t<DT, R, S>(tdy, tw, args, grid, stream);
  PGG_VARIANTS(PGG_LAUNCH)
#undef PGG_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace pgg
