// Grouped GEMM + ordered scatter-add on the FP32 pipes, for inputs the
// tensor-memory-access unit cannot stream: rows of d_y and weight whose byte
// length is not a multiple of 16 (N = 1 and N = 286 in the white-box list of
// the page "MoeInitRoutingGroupedMatmulGrad design", section 4.2.1), or
// gradY / weight pointers that are not 16-byte aligned. Any N, K and element
// alignment.
//
// Same operation, tile order and determinism as the tensor-core path (section
// "数学定义和公式", Steps 1 and 2): a persistent grid claims tiles
// (row block, k block of 128) in increasing order from the atomic counter in
// the workspace header; a tile computes
//     C[r, k] = sum_n d_y[row0 + r, n] * weight[g, k0 + k, n]
// with fp32 fused multiply-adds in increasing n, then adds each row into
// d_x[token(row), k0 .. k0 + 127] under the same (token, k block) tickets:
// the row of rank r waits until r rows of its token have been added, stores
// (rank 0) or adds (rank > 0), and bumps the ticket. A row only waits for
// rows of smaller expanded index, which lie in tiles claimed earlier or
// earlier in its own tile, so there is no wait cycle. Waits are bounded by
// the same limit as the tensor-core kernel.
//
// Tile: 64 rows x 128 k per pass (a row block of more rows is taken in passes
// of 64), 128 threads. Operands are staged as fp32 in shared memory, 32 values
// of n at a time (double-buffered, the next step's loads in flight during the
// current step's arithmetic), transposed so that a thread reads its 8 rows and
// 8 k with four 16-byte loads per n and keeps an 8 x 8 block of accumulators.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "pgg_internal.h"
#include "pgg_ptx.cuh"

namespace pgg {
namespace {

constexpr int kSRows = 64;       // rows per pass
constexpr int kSThreads = 128;   // 16 (k) x 8 (rows)
constexpr int kSNc = 32;         // reduction values staged per step
constexpr int kSMinCtas = 3;     // resident CTAs per SM the register budget is sized for
constexpr int kSAStride = kSRows + 4;    // floats per n in sA (== 4 mod 32: conflict-free stores)
constexpr int kSBStride = kKBlock + 4;   // floats per n in sB

// Element i loaded as its raw bits (zero-extended); converted to fp32 only
// when it is written to shared memory, so that the loads of the next step
// stay in flight while the current step is computed.
template <int DT>
__device__ __forceinline__ uint32_t load_raw(const void* p, int64_t i) {
  if constexpr (DT == PGG_F32)
    return __ldg(static_cast<const unsigned int*>(p) + i);
  else
    return __ldg(static_cast<const unsigned short*>(p) + i);
}
template <int DT>
__device__ __forceinline__ float raw_to_float(uint32_t r) {
  if constexpr (DT == PGG_F32)
    return __uint_as_float(r);
  else if constexpr (DT == PGG_BF16)
    return __uint_as_float(r << 16);
  else
    return __half2float(__ushort_as_half(static_cast<unsigned short>(r)));
}

__device__ __forceinline__ void raise_status(WsHeader* hdr, uint32_t code, uint32_t site) {
  if (atomicCAS(&hdr->status, 0u, code) == 0u) hdr->timeout_site = site;
}

// Adds (or, for rank 0, stores) 4 consecutive values of a d_x row.
__device__ __forceinline__ void put4(float* p, int64_t k, int64_t K, bool vec, int rank,
                                     float x0, float x1, float x2, float x3) {
  if (vec) {
    if (k < K) {
      const float4 v = make_float4(x0, x1, x2, x3);
      if (rank == 0)
        *reinterpret_cast<float4*>(p) = v;
      else
        ptx::red_add_v4_f32_gpu(p, v);
    }
    return;
  }
  const float x[4] = {x0, x1, x2, x3};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (k + c < K) {
      if (rank == 0)
        p[c] = x[c];
      else
        ptx::red_add_f32_gpu(p + c, x[c]);
    }
  }
}

constexpr int kARegs = (kSRows / 16) * (kSNc / 8);   // d_y values staged per thread per step
constexpr int kBRegs = (kKBlock / 16) * (kSNc / 8);  // weight values staged per thread per step

// Global loads of one reduction step into registers (zero outside the
// tensors). Lane (l_n, l_r) of warp w takes n = 8q + l_n and rows / k
// 16 it + 4 w + l_r: each warp instruction reads 8 consecutive n of 4 rows.
template <int DT>
__device__ __forceinline__ void stage_load(const SimtArgs& a, int64_t row0, int R, int64_t g,
                                           int64_t k0, int64_t n0, int warp, int l_n, int l_r,
                                           uint32_t (&ra)[kARegs], uint32_t (&rb)[kBRegs]) {
  const int64_t N = a.N, K = a.K;
#pragma unroll
  for (int it = 0; it < kSRows / 16; ++it) {
    const int r = it * 16 + warp * 4 + l_r;
#pragma unroll
    for (int q = 0; q < kSNc / 8; ++q) {
      const int64_t n = n0 + q * 8 + l_n;
      ra[it * (kSNc / 8) + q] = (r < R && n < N) ? load_raw<DT>(a.dy, (row0 + r) * N + n) : 0u;
    }
  }
#pragma unroll
  for (int it = 0; it < kKBlock / 16; ++it) {
    const int kk = it * 16 + warp * 4 + l_r;
#pragma unroll
    for (int q = 0; q < kSNc / 8; ++q) {
      const int64_t n = n0 + q * 8 + l_n;
      rb[it * (kSNc / 8) + q] =
          (k0 + kk < K && n < N) ? load_raw<DT>(a.w, (g * K + k0 + kk) * N + n) : 0u;
    }
  }
}

// The staged values, transposed into sA[n][row] and sB[n][k]. The strides are
// 4 mod 32 words, so the 8 n x 4 rows of a warp instruction hit 32 banks.
template <int DT>
__device__ __forceinline__ void stage_store(float* sa, float* sb, int warp, int l_n, int l_r,
                                            const uint32_t (&ra)[kARegs],
                                            const uint32_t (&rb)[kBRegs]) {
#pragma unroll
  for (int it = 0; it < kSRows / 16; ++it)
#pragma unroll
    for (int q = 0; q < kSNc / 8; ++q)
      sa[(q * 8 + l_n) * kSAStride + it * 16 + warp * 4 + l_r] =
          raw_to_float<DT>(ra[it * (kSNc / 8) + q]);
#pragma unroll
  for (int it = 0; it < kKBlock / 16; ++it)
#pragma unroll
    for (int q = 0; q < kSNc / 8; ++q)
      sb[(q * 8 + l_n) * kSBStride + it * 16 + warp * 4 + l_r] =
          raw_to_float<DT>(rb[it * (kSNc / 8) + q]);
}

struct SimtSmem {
  float a[2][kSNc * kSAStride];  // [n][row], two buffers
  float b[2][kSNc * kSBStride];  // [n][k], two buffers
};

template <int DT>
__global__ void __launch_bounds__(kSThreads, kSMinCtas) gmm_dx_simt_kernel(const SimtArgs a) {
  ptx::griddep_wait();  // launched with programmatic serialization: predecessors done
  extern __shared__ __align__(16) uint8_t simt_smem_raw[];
  SimtSmem& sm = *reinterpret_cast<SimtSmem*>(simt_smem_raw);
  float (&sA)[2][kSNc * kSAStride] = sm.a;
  float (&sB)[2][kSNc * kSBStride] = sm.b;
  __shared__ uint32_t s_tile;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  WsHeader* hdr = a.hdr;

  // Routing validation failed: the result is defined as zeros.
  const uint32_t st = hdr->status;
  if (st == kStIndex || st == kStGroupSum || st == kStNotPerm) {
    const int64_t n = a.batch * a.K;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid; q < n;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x)
      a.out[q] = 0.0f;
    return;
  }

  const uint32_t kbs = static_cast<uint32_t>(a.k_blocks);
  const uint32_t total = hdr->n_row_blocks * kbs;
  const int64_t N = a.N, K = a.K;
  const int tx = tid & 15, ty = tid >> 4;      // compute: k {4tx.., 64+4tx..}, rows 8ty..8ty+7
  const int l_n = lane & 7, l_r = lane >> 3;   // staging: 8 n x 4 rows per warp instruction
  const uint64_t lim = a.wait_limit_ns;
  bool gave_up = false;

  for (;;) {
    if (tid == 0) s_tile = atomicAdd(&hdr->sched_next, 1u);
    __syncthreads();
    const uint32_t t = s_tile;
    __syncthreads();  // every thread has read s_tile before thread 0 may claim again
    if (t >= total) break;
    const uint32_t rb = t / kbs, kb = t - rb * kbs;
    int4 e = a.rblist[check_index(hdr, rb, a.max_row_blocks, 50)];
    // checked build: a row block outside the experts or rows becomes an empty one
    if (!check_ok(hdr,
                  e.x >= 0 && e.x < a.G && e.y >= 0 && e.z >= 0 &&
                      static_cast<int64_t>(e.y) + e.z <= a.M,
                  51))
      e = make_int4(0, 0, 0, 0);
    const int64_t g = e.x;
    const int64_t k0 = static_cast<int64_t>(kb) * kKBlock;

    for (int p0 = 0; p0 < e.z; p0 += kSRows) {
      const int64_t row0 = static_cast<int64_t>(e.y) + p0;
      const int R = e.z - p0 < kSRows ? e.z - p0 : kSRows;
      float acc[8][8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

      // Software pipeline over reduction steps of kSNc values: the global
      // loads of step s + 1 are in flight (in registers) while step s is
      // computed from one shared-memory buffer; then they are written to the
      // other buffer. One barrier per step.
      uint32_t ra[kARegs], rb[kBRegs];
      stage_load<DT>(a, row0, R, g, k0, 0, warp, l_n, l_r, ra, rb);
      stage_store<DT>(sA[0], sB[0], warp, l_n, l_r, ra, rb);
      __syncthreads();
      int buf = 0;
      for (int64_t n0 = 0; n0 < N; n0 += kSNc) {
        const bool more = n0 + kSNc < N;
        if (more) stage_load<DT>(a, row0, R, g, k0, n0 + kSNc, warp, l_n, l_r, ra, rb);
        const float* pa = sA[buf];
        const float* pb = sB[buf];
#pragma unroll 4
        for (int nn = 0; nn < kSNc; ++nn) {
          const float4 a0 = *reinterpret_cast<const float4*>(&pa[nn * kSAStride + 8 * ty]);
          const float4 a1 = *reinterpret_cast<const float4*>(&pa[nn * kSAStride + 8 * ty + 4]);
          const float4 b0 = *reinterpret_cast<const float4*>(&pb[nn * kSBStride + 4 * tx]);
          const float4 b1 = *reinterpret_cast<const float4*>(&pb[nn * kSBStride + 64 + 4 * tx]);
          const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        if (more) stage_store<DT>(sA[buf ^ 1], sB[buf ^ 1], warp, l_n, l_r, ra, rb);
        __syncthreads();  // buffer buf ^ 1 is full; buffer buf may be overwritten next step
        buf ^= 1;
      }

      // Ordered scatter-add. Warp w owns rows 16w .. 16w+15 of the pass; lane
      // j < 16 tracks row 16w + j; lanes 16h .. 16h+15 hold the values of rows
      // 16w + 8h .. 16w + 8h + 7.
      const int my_row = 16 * warp + (lane & 15);
      RowInfo ri;
      ri.token = 0;
      ri.rank = 0;
      const bool tracked = lane < 16 && my_row < R;
      if (tracked) {
        ri = a.rowinfo[check_index(hdr, row0 + my_row, a.M, 52)];
        ri.token = static_cast<int32_t>(check_index(hdr, ri.token, a.batch, 53));
      }
      uint32_t pend = __ballot_sync(0xFFFFFFFFu, tracked);
      uint64_t t_wait0 = 0;
      const int half = lane >> 4;
      while (pend) {
        bool rdy = false;
        if ((pend >> lane) & 1u)
          rdy = gave_up || ri.rank == 0 ||
                ptx::ld_acquire_gpu(a.tickets + static_cast<int64_t>(ri.token) * kbs + kb) >=
                    static_cast<uint32_t>(ri.rank) + a.ticket_bias;
        const uint32_t ready = __ballot_sync(0xFFFFFFFFu, rdy);
        __syncwarp();
        if (!ready) {
          if (t_wait0 == 0) t_wait0 = ptx::globaltimer();
          bool expired = (ptx::globaltimer() - t_wait0 > lim) ||
                         *reinterpret_cast<volatile uint32_t*>(&hdr->status) == kStTimeout;
          expired = __shfl_sync(0xFFFFFFFFu, expired, 0);
          if (expired) {
            gave_up = true;
            if (lane == 0) raise_status(hdr, kStTimeout, 6);
          } else {
            __nanosleep(128);
          }
          continue;
        }
        t_wait0 = 0;  // progress: the limit counts time without any
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int j = 8 * half + i;  // row of the pass this lane writes now
          const int tok = __shfl_sync(0xFFFFFFFFu, ri.token, j);
          const int rk = __shfl_sync(0xFFFFFFFFu, ri.rank, j);
          if ((ready >> j) & 1u) {
            float* base = a.out + static_cast<int64_t>(tok) * K + k0;
            put4(base + 4 * tx, k0 + 4 * tx, K, a.vec_out, rk, acc[i][0], acc[i][1], acc[i][2],
                 acc[i][3]);
            put4(base + 64 + 4 * tx, k0 + 64 + 4 * tx, K, a.vec_out, rk, acc[i][4], acc[i][5],
                 acc[i][6], acc[i][7]);
          }
        }
        __syncwarp();
        // publish: the rows' writes happen-before the ticket bumps
        if ((ready >> lane) & 1u) {
          ptx::fence_acq_rel_gpu();
          ptx::red_add_u32_gpu(a.tickets + static_cast<int64_t>(ri.token) * kbs + kb, 1u);
        }
        pend &= ~ready;
      }
    }
  }
}

}  // namespace

void simt_config(int* rows, int* stages, int* threads, int* smem) {
  *rows = kSRows;
  *stages = 2;
  *threads = kSThreads;
  *smem = static_cast<int>(sizeof(SimtSmem) + 16);
}

cudaError_t launch_simt(int dtype, const SimtArgs& a, int64_t max_tiles, int num_sms,
                        cudaStream_t stream) {
  void (*kern)(const SimtArgs) = nullptr;
  if (dtype == PGG_F32)
    kern = gmm_dx_simt_kernel<PGG_F32>;
  else if (dtype == PGG_F16)
    kern = gmm_dx_simt_kernel<PGG_F16>;
  else if (dtype == PGG_BF16)
    kern = gmm_dx_simt_kernel<PGG_BF16>;
  else
    return cudaErrorInvalidValue;
  constexpr int smem = static_cast<int>(sizeof(SimtSmem));
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  int64_t grid = static_cast<int64_t>(num_sms) * per_sm;
  if (max_tiles < grid) grid = max_tiles;
  if (grid < 1) grid = 1;
  err = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kSThreads),
                   static_cast<size_t>(smem), stream, 1, a);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace pgg
