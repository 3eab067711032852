// Forward grouped matmul on the FP32 pipes, for inputs the tensor-core kernel
// does not take: fp32 inputs, rows of x, weight or y whose byte length is not
// a multiple of 16, or pointers that are not 16-byte aligned. Same operation
// ("MoeInitRoutingGroupedMatmulGrad design", sections 1.1 and 1.2):
//
//     y[i, n] = sum over k, in increasing k, of x[batch(i), k] * weight[g(i), k, n]
//
// Tile: a row block of one expert (taken 64 rows at a time) x 128 n, 128
// threads, each an 8 (rows) x 8 (n) block of fp32 accumulators. K is taken 32
// at a time: the x rows of the block's tokens (transposed into sA[k][row])
// and weight[g, k, n] (sB[k][n]) are loaded with element-sized loads, kept as
// raw bits in registers while the previous 32 values of k are computed, and
// converted to fp32 into one of two shared-memory buffers. Tiles are
// statically interleaved over the persistent grid.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "pgg_internal.h"
#include "pgg_ptx.cuh"

namespace pgg {
namespace {

constexpr int kRows = 64;         // rows per pass
constexpr int kCols = 128;        // n per tile
constexpr int kKc = 32;           // k per step
constexpr int kThr = 128;
constexpr int kAStride = kRows + 4;   // sA[k][row]
constexpr int kBStride = kCols + 4;   // sB[k][n]
constexpr int kARegs = (kRows / 16) * (kKc / 8);   // 16: lane (8 k x 4 rows) pattern
constexpr int kBRegs = (kKc / 4) * (kCols / 32);   // 32: lane along n

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

struct Smem {
  float a[2][kKc * kAStride];
  float b[2][kKc * kBStride];
};

// tok[it * 4 + ...]: tokens of the rows this lane loads (rows 16 it + 4 warp + l_r).
template <int DT>
__device__ __forceinline__ void load_step(const FwdArgs& a, const int32_t (&tok)[kRows / 16],
                                          int64_t g, int64_t n0, int64_t k0, int warp, int lane,
                                          uint32_t (&ra)[kARegs], uint32_t (&rb)[kBRegs]) {
  const int l_k = lane & 7, l_r = lane >> 3;
#pragma unroll
  for (int it = 0; it < kRows / 16; ++it) {
#pragma unroll
    for (int q = 0; q < kKc / 8; ++q) {
      const int64_t k = k0 + q * 8 + l_k;
      ra[it * (kKc / 8) + q] =
          (tok[it] >= 0 && k < a.K) ? load_raw<DT>(a.x, static_cast<int64_t>(tok[it]) * a.K + k)
                                    : 0u;
    }
  }
  (void)l_r;
#pragma unroll
  for (int it = 0; it < kKc / 4; ++it) {
    const int64_t k = k0 + it * 4 + warp;
#pragma unroll
    for (int h = 0; h < kCols / 32; ++h) {
      const int64_t n = n0 + 32 * h + lane;
      rb[it * (kCols / 32) + h] =
          (k < a.K && n < a.N) ? load_raw<DT>(a.w, (g * a.K + k) * a.N + n) : 0u;
    }
  }
}

template <int DT>
__device__ __forceinline__ void store_step(float* sa, float* sb, int warp, int lane,
                                           const uint32_t (&ra)[kARegs],
                                           const uint32_t (&rb)[kBRegs]) {
  const int l_k = lane & 7, l_r = lane >> 3;
#pragma unroll
  for (int it = 0; it < kRows / 16; ++it)
#pragma unroll
    for (int q = 0; q < kKc / 8; ++q)
      sa[(q * 8 + l_k) * kAStride + it * 16 + warp * 4 + l_r] =
          raw_to_float<DT>(ra[it * (kKc / 8) + q]);
#pragma unroll
  for (int it = 0; it < kKc / 4; ++it)
#pragma unroll
    for (int h = 0; h < kCols / 32; ++h)
      sb[(it * 4 + warp) * kBStride + 32 * h + lane] = raw_to_float<DT>(rb[it * (kCols / 32) + h]);
}

template <int DT>
__device__ __forceinline__ void store4(void* out, bool f32, int64_t off, int64_t n, int64_t N,
                                       bool vec, const float* v) {
  if (f32) {
    float* p = static_cast<float*>(out) + off;
    if (vec && n + 3 < N) {
      *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
      return;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (n + c < N) p[c] = v[c];
    return;
  }
  uint16_t h[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if constexpr (DT == PGG_BF16) {
      const __nv_bfloat16 b = __float2bfloat16_rn(v[c]);
      h[c] = *reinterpret_cast<const uint16_t*>(&b);
    } else {
      const __half b = __float2half_rn(v[c]);
      h[c] = *reinterpret_cast<const uint16_t*>(&b);
    }
  }
  uint16_t* p = static_cast<uint16_t*>(out) + off;
  if (vec && n + 3 < N) {
    *reinterpret_cast<uint2*>(p) = make_uint2(h[0] | (static_cast<uint32_t>(h[1]) << 16),
                                              h[2] | (static_cast<uint32_t>(h[3]) << 16));
    return;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c)
    if (n + c < N) p[c] = h[c];
}

template <int DT>
__global__ void __launch_bounds__(kThr, 3) gmm_fwd_simt_kernel(const FwdArgs a, int vec) {
  ptx::griddep_wait();  // launched with programmatic serialization: predecessors done
  extern __shared__ __align__(16) uint8_t fwd_simt_smem[];
  Smem& sm = *reinterpret_cast<Smem*>(fwd_simt_smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool f32 = a.out_f32 != 0;

  // Routing validation failed: the result is defined as zeros.
  const uint32_t st = a.hdr->status;
  if (st == kStIndex || st == kStGroupSum || st == kStNotPerm) {
    const int64_t n = a.M * a.N;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid; q < n;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      if (f32)
        static_cast<float*>(a.out)[q] = 0.0f;
      else
        static_cast<uint16_t*>(a.out)[q] = 0;
    }
    return;
  }
  const uint32_t total = a.hdr->n_row_blocks * static_cast<uint32_t>(a.n_blocks);
  const int tx = tid & 15, ty = tid >> 4;  // n {4tx.., 64+4tx..}, rows 8ty .. 8ty+7
  const int l_r = lane >> 3;
  for (uint32_t t = blockIdx.x; t < total; t += gridDim.x) {
    const uint32_t rb = t / static_cast<uint32_t>(a.n_blocks);
    int4 e = a.rblist[check_index(a.hdr, rb, a.max_row_blocks, 74)];
    // checked build: a row block outside the experts or rows becomes an empty one
    if (!check_ok(a.hdr,
                  e.x >= 0 && e.x < a.G && e.y >= 0 && e.z >= 0 &&
                      static_cast<int64_t>(e.y) + e.z <= a.M,
                  75))
      e = make_int4(0, 0, 0, 0);
    const int64_t g = e.x;
    const int64_t n0 = static_cast<int64_t>(t - rb * static_cast<uint32_t>(a.n_blocks)) * kCols;
    for (int p0 = 0; p0 < e.z; p0 += kRows) {
      const int64_t row0 = static_cast<int64_t>(e.y) + p0;
      const int R = e.z - p0 < kRows ? e.z - p0 : kRows;
      int32_t tok[kRows / 16];
#pragma unroll
      for (int it = 0; it < kRows / 16; ++it) {
        const int r = it * 16 + warp * 4 + l_r;
        tok[it] = r < R ? static_cast<int32_t>(check_index(
                              a.hdr, a.rowinfo[check_index(a.hdr, row0 + r, a.M, 76)].token,
                              a.batch, 77))
                        : -1;
      }
      float acc[8][8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
      uint32_t ra[kARegs], rb_[kBRegs];
      load_step<DT>(a, tok, g, n0, 0, warp, lane, ra, rb_);
      __syncthreads();  // earlier reads of buffer 0 are done
      store_step<DT>(sm.a[0], sm.b[0], warp, lane, ra, rb_);
      __syncthreads();
      int buf = 0;
      for (int64_t k0 = 0; k0 < a.K; k0 += kKc) {
        const bool more = k0 + kKc < a.K;
        if (more) load_step<DT>(a, tok, g, n0, k0 + kKc, warp, lane, ra, rb_);
        const float* pa = sm.a[buf];
        const float* pb = sm.b[buf];
#pragma unroll 4
        for (int kk = 0; kk < kKc; ++kk) {
          const float4 a0 = *reinterpret_cast<const float4*>(&pa[kk * kAStride + 8 * ty]);
          const float4 a1 = *reinterpret_cast<const float4*>(&pa[kk * kAStride + 8 * ty + 4]);
          const float4 b0 = *reinterpret_cast<const float4*>(&pb[kk * kBStride + 4 * tx]);
          const float4 b1 = *reinterpret_cast<const float4*>(&pb[kk * kBStride + 64 + 4 * tx]);
          const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        if (more) store_step<DT>(sm.a[buf ^ 1], sm.b[buf ^ 1], warp, lane, ra, rb_);
        __syncthreads();
        buf ^= 1;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 8 * ty + i;
        if (r >= R) continue;
        const int64_t row = (row0 + r) * a.N;
        const int64_t n_a = n0 + 4 * tx, n_b = n0 + 64 + 4 * tx;
        if (n_a < a.N) store4<DT>(a.out, f32, row + n_a, n_a, a.N, vec != 0, &acc[i][0]);
        if (n_b < a.N) store4<DT>(a.out, f32, row + n_b, n_b, a.N, vec != 0, &acc[i][4]);
      }
    }
  }
}

}  // namespace

void fwd_simt_tiles(int64_t N, int* n_blocks) {
  *n_blocks = static_cast<int>((N + kCols - 1) / kCols);
}

int fwd_simt_smem_bytes() { return static_cast<int>(sizeof(Smem)); }

// vec: N % 4 == 0 and y aligned to 4 output elements.
cudaError_t launch_fwd_simt(int dtype, const FwdArgs& a, int vec, int64_t max_tiles, int num_sms,
                            cudaStream_t stream) {
  void (*kern)(const FwdArgs, int) = nullptr;
  if (dtype == PGG_F32)
    kern = gmm_fwd_simt_kernel<PGG_F32>;
  else if (dtype == PGG_F16)
    kern = gmm_fwd_simt_kernel<PGG_F16>;
  else if (dtype == PGG_BF16)
    kern = gmm_fwd_simt_kernel<PGG_BF16>;
  else
    return cudaErrorInvalidValue;
  constexpr int smem = static_cast<int>(sizeof(Smem));
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThr, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  int64_t grid = static_cast<int64_t>(num_sms) * per_sm;
  if (max_tiles < grid) grid = max_tiles;
  if (grid < 1) grid = 1;
  err = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThr),
                   static_cast<size_t>(smem), stream, 1, a, vec);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace pgg
