// Weight gradient on the FP32 pipes, for inputs the tensor-core kernel does not
// take: fp32 inputs, rows of x or d_y whose byte length is not a multiple of
// 16, or pointers that are not 16-byte aligned. Same operation and the same
// fixed order of additions for every run:
//
//     d_weight[g, k, n] = sum over the expanded rows i of expert g, in
//                         increasing i, of x[batch(i), k] * d_y[i, n]
//
// ("MoeInitRoutingGroupedMatmulGrad design", section 1.2, "为何不计算
// d_weight" item 3, with expanded_x[i] = x[batch(i)] from section 1.1.)
//
// Tile: one expert, 64 k x 128 n, 128 threads, each an 8 (k) x 8 (n) block of
// fp32 accumulators. The expert's rows are taken 32 at a time: the x rows of
// their tokens (64 k) and the d_y rows (128 n) are loaded with element-sized
// loads, kept as raw bits in registers while the previous 32 rows are
// computed, then converted to fp32 into one of two shared-memory buffers
// (rows are the outer index in memory for both operands, so no transpose).
// Tiles are statically interleaved over the persistent grid.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "pgg_internal.h"
#include "pgg_ptx.cuh"

namespace pgg {
namespace {

constexpr int kWK = 64;           // k per tile
constexpr int kWN = 128;          // n per tile
constexpr int kWR = 32;           // reduction rows per step
constexpr int kWThreads = 128;
constexpr int kXStride = kWK + 4;   // floats per row in sX
constexpr int kDStride = kWN + 4;   // floats per row in sD
constexpr int kXRegs = (kWR / 4) * (kWK / 32);   // 16
constexpr int kDRegs = (kWR / 4) * (kWN / 32);   // 32

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

struct WTile {
  int64_t g, k0, n0, row0, m;
};

__device__ __forceinline__ WTile wtile_of(uint32_t t, const DwArgs& a) {
  const uint32_t per_g = static_cast<uint32_t>(a.k_blocks) * static_cast<uint32_t>(a.n_blocks);
  WTile x;
  x.g = t / per_g;
  const uint32_t rem = t - static_cast<uint32_t>(x.g) * per_g;
  x.k0 = static_cast<int64_t>(rem / a.n_blocks) * kWK;
  x.n0 = static_cast<int64_t>(rem % a.n_blocks) * kWN;
  x.row0 = a.off[x.g];
  x.m = a.off[x.g + 1] - x.row0;
  return x;
}

// Rows r0 .. r0 + 31 of the expert: lane l of warp w loads k = 32 h + l and
// n = 32 h + l of rows 4 it + w.
template <int DT>
__device__ __forceinline__ void wstage_load(const DwArgs& a, const WTile& x, int64_t r0, int warp,
                                            int lane, uint32_t (&rx)[kXRegs],
                                            uint32_t (&rd)[kDRegs]) {
#pragma unroll
  for (int it = 0; it < kWR / 4; ++it) {
    const int64_t r = r0 + it * 4 + warp;
    const bool row_ok = r < x.m;
    int64_t tok = 0;
    if (row_ok)
      tok = check_index(a.hdr, a.rowinfo[check_index(a.hdr, x.row0 + r, a.M, 62)].token,
                        a.batch, 63);
#pragma unroll
    for (int h = 0; h < kWK / 32; ++h) {
      const int64_t k = x.k0 + 32 * h + lane;
      rx[it * (kWK / 32) + h] = (row_ok && k < a.K) ? load_raw<DT>(a.x, tok * a.K + k) : 0u;
    }
#pragma unroll
    for (int h = 0; h < kWN / 32; ++h) {
      const int64_t n = x.n0 + 32 * h + lane;
      rd[it * (kWN / 32) + h] =
          (row_ok && n < a.N) ? load_raw<DT>(a.dy, (x.row0 + r) * a.N + n) : 0u;
    }
  }
}

template <int DT>
__device__ __forceinline__ void wstage_store(float* sx, float* sd, int warp, int lane,
                                             const uint32_t (&rx)[kXRegs],
                                             const uint32_t (&rd)[kDRegs]) {
#pragma unroll
  for (int it = 0; it < kWR / 4; ++it) {
    const int r = it * 4 + warp;
#pragma unroll
    for (int h = 0; h < kWK / 32; ++h)
      sx[r * kXStride + 32 * h + lane] = raw_to_float<DT>(rx[it * (kWK / 32) + h]);
#pragma unroll
    for (int h = 0; h < kWN / 32; ++h)
      sd[r * kDStride + 32 * h + lane] = raw_to_float<DT>(rd[it * (kWN / 32) + h]);
  }
}

struct WSmem {
  float x[2][kWR * kXStride];
  float d[2][kWR * kDStride];
};

// Stores 4 consecutive values of an output row (fp32 or the 16-bit input
// dtype), 16 / 8 bytes at once when `vec`.
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
__global__ void __launch_bounds__(kWThreads, 3) gmm_dw_simt_kernel(const DwArgs a, int vec) {
  ptx::griddep_wait();  // launched with programmatic serialization: predecessors done
  extern __shared__ __align__(16) uint8_t dw_simt_smem[];
  WSmem& sm = *reinterpret_cast<WSmem*>(dw_simt_smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool f32 = a.out_f32 != 0;

  // Routing validation failed: the result is defined as zeros.
  const uint32_t st = a.hdr->status;
  if (st == kStIndex || st == kStGroupSum || st == kStNotPerm) {
    const int64_t n = a.G * a.K * a.N;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid; q < n;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      if (f32)
        static_cast<float*>(a.out)[q] = 0.0f;
      else
        static_cast<uint16_t*>(a.out)[q] = 0;
    }
    return;
  }

  const uint32_t total =
      static_cast<uint32_t>(a.G) * static_cast<uint32_t>(a.k_blocks) * static_cast<uint32_t>(a.n_blocks);
  const int tx = tid & 15, ty = tid >> 4;  // n {4tx.., 64+4tx..}, k 8ty .. 8ty+7
  for (uint32_t t = blockIdx.x; t < total; t += gridDim.x) {
    const WTile x = wtile_of(t, a);
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    if (x.m > 0) {
      uint32_t rx[kXRegs], rd[kDRegs];
      wstage_load<DT>(a, x, 0, warp, lane, rx, rd);
      __syncthreads();  // the previous tile's reads of buffer 0 are done
      wstage_store<DT>(sm.x[0], sm.d[0], warp, lane, rx, rd);
      __syncthreads();
      int buf = 0;
      for (int64_t r0 = 0; r0 < x.m; r0 += kWR) {
        const bool more = r0 + kWR < x.m;
        if (more) wstage_load<DT>(a, x, r0 + kWR, warp, lane, rx, rd);
        const float* px = sm.x[buf];
        const float* pd = sm.d[buf];
        const int rows = x.m - r0 < kWR ? static_cast<int>(x.m - r0) : kWR;
#pragma unroll 4
        for (int r = 0; r < rows; ++r) {
          const float4 x0 = *reinterpret_cast<const float4*>(&px[r * kXStride + 8 * ty]);
          const float4 x1 = *reinterpret_cast<const float4*>(&px[r * kXStride + 8 * ty + 4]);
          const float4 d0 = *reinterpret_cast<const float4*>(&pd[r * kDStride + 4 * tx]);
          const float4 d1 = *reinterpret_cast<const float4*>(&pd[r * kDStride + 64 + 4 * tx]);
          const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          const float dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(xv[i], dv[j], acc[i][j]);
        }
        if (more) wstage_store<DT>(sm.x[buf ^ 1], sm.d[buf ^ 1], warp, lane, rx, rd);
        __syncthreads();
        buf ^= 1;
      }
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t k = x.k0 + 8 * ty + i;
      if (k >= a.K) continue;
      const int64_t row = (x.g * a.K + k) * a.N;
      const int64_t n_a = x.n0 + 4 * tx, n_b = x.n0 + 64 + 4 * tx;
      if (n_a < a.N) store4<DT>(a.out, f32, row + n_a, n_a, a.N, vec != 0, &acc[i][0]);
      if (n_b < a.N) store4<DT>(a.out, f32, row + n_b, n_b, a.N, vec != 0, &acc[i][4]);
    }
  }
}

}  // namespace

void dw_simt_tiles(int64_t K, int64_t N, int* k_blocks, int* n_blocks) {
  *k_blocks = static_cast<int>((K + kWK - 1) / kWK);
  *n_blocks = static_cast<int>((N + kWN - 1) / kWN);
}

int dw_simt_smem_bytes() { return static_cast<int>(sizeof(WSmem)); }

// vec: N % 4 == 0 and out aligned to 4 output elements (16 bytes fp32, 8 bytes 16-bit).
cudaError_t launch_dw_simt(int dtype, const DwArgs& a, int vec, int num_sms, cudaStream_t stream) {
  void (*kern)(const DwArgs, int) = nullptr;
  if (dtype == PGG_F32)
    kern = gmm_dw_simt_kernel<PGG_F32>;
  else if (dtype == PGG_F16)
    kern = gmm_dw_simt_kernel<PGG_F16>;
  else if (dtype == PGG_BF16)
    kern = gmm_dw_simt_kernel<PGG_BF16>;
  else
    return cudaErrorInvalidValue;
  constexpr int smem = static_cast<int>(sizeof(WSmem));
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const int64_t total = a.G * a.k_blocks * a.n_blocks;
  int64_t grid = static_cast<int64_t>(num_sms) * per_sm;
  if (total < grid) grid = total;
  if (grid < 1) grid = 1;
  err = launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kWThreads),
                   static_cast<size_t>(smem), stream, 1, a, vec);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace pgg
