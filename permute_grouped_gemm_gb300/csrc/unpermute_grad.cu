// Probs-weighted unpermute backward ("NPU DeepSeek-V3.2-Exp TileLang operator
// practice", section moe_token_unpermute_grad). For the combine that follows
// the expert grouped matmul, out[b] = sum_j prob[b, j] * permuted[row(b, j)],
// with row(b, j) the expanded row of original position b * topK + j:
//
//     perm_grad[row(b, j), h] = d_out[b, h] * prob[b, j]     (prob = 1 without probs)
//     probs_grad[b, j]        = sum over h of d_out[b, h] * permuted[row(b, j), h]
//
// perm_grad is the d_y that the fused d_x backward and the weight gradient
// take. Bound by HBM: d_out is read once per token (its re-reads for the
// token's topK rows hit L1 or L2), permuted is read once and perm_grad
// written once. One warp per original position (grid-stride), four 16-byte
// loads per lane in flight when the rows allow 16-byte access; the dot
// product in fp32, each lane over its own positions in increasing order, then
// a fixed shuffle tree, so that it is bitwise repeatable.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "pgg_internal.h"
#include "pgg_ptx.cuh"

namespace pgg {
namespace {

constexpr int kUThreads = 256;

template <int DT>
struct Elem;
template <>
struct Elem<PGG_F32> {
  static constexpr int kPer16 = 4;
  __device__ static float get(const void* p, int64_t i) { return static_cast<const float*>(p)[i]; }
  __device__ static void put(void* p, int64_t i, float v) { static_cast<float*>(p)[i] = v; }
};
template <>
struct Elem<PGG_F16> {
  static constexpr int kPer16 = 8;
  __device__ static float get(const void* p, int64_t i) {
    return __half2float(static_cast<const __half*>(p)[i]);
  }
  __device__ static void put(void* p, int64_t i, float v) {
    static_cast<__half*>(p)[i] = __float2half_rn(v);
  }
};
template <>
struct Elem<PGG_BF16> {
  static constexpr int kPer16 = 8;
  __device__ static float get(const void* p, int64_t i) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  }
  __device__ static void put(void* p, int64_t i, float v) {
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  }
};

// 16 bytes as floats (8 of a 16-bit dtype, 4 of fp32) and back.
template <int DT>
__device__ __forceinline__ void unpack16(const uint4& q, float* f) {
  if constexpr (DT == PGG_F32) {
    f[0] = __uint_as_float(q.x);
    f[1] = __uint_as_float(q.y);
    f[2] = __uint_as_float(q.z);
    f[3] = __uint_as_float(q.w);
  } else {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (DT == PGG_BF16) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      } else {
        const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
        const float2 t = __half22float2(h);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
      }
    }
  }
}

template <int DT>
__device__ __forceinline__ uint4 pack16(const float* f) {
  if constexpr (DT == PGG_F32) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (DT == PGG_BF16) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&p);
      } else {
        const __half2 p = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&p);
      }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// One warp per original position p = b * topK + j: it reads d_out[b] (shared
// with the token's other positions through L1), permuted[row], writes
// perm_grad[row] and reduces the dot product with a fixed shuffle tree.
template <int DT, bool PROBS, bool VEC, bool PAIRS>
__global__ void __launch_bounds__(kUThreads) unpermute_grad_kernel(const UnpermArgs a) {
  using E = Elem<DT>;
  ptx::griddep_wait();  // the index validation before this launch
  const uint32_t st = a.hdr->status;
  if (st == kStIndex || st == kStGroupSum || st == kStNotPerm) {
    const int64_t n = a.M * a.H;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t q = t0; q < n; q += stride) E::put(a.perm_grad, q, 0.0f);
    if (PROBS && a.probs_grad)
      for (int64_t q = t0; q < a.M; q += stride) {
        if (a.probs_grad_f32)
          static_cast<float*>(a.probs_grad)[q] = 0.0f;
        else
          E::put(a.probs_grad, q, 0.0f);
      }
    return;
  }
  const int lane = threadIdx.x & 31;
  const int64_t H = a.H;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kUThreads / 32);
  for (int64_t p = static_cast<int64_t>(blockIdx.x) * (kUThreads / 32) + (threadIdx.x >> 5);
       p < a.M; p += warps) {
    const int64_t b = p / a.topK;
    const int64_t row = check_index(
        a.hdr, a.row_idx_type == 0 ? static_cast<int64_t>(a.inv[p]) : a.idx[p], a.M, 80);
    const float pr = PROBS ? E::get(a.probs, p) : 1.0f;
    float dot = 0.0f;
    if constexpr (VEC) {
      constexpr int kE = E::kPer16;
      constexpr int64_t kEs = DT == PGG_F32 ? 4 : 2;  // bytes per element
      const uint4* d4 =
          reinterpret_cast<const uint4*>(static_cast<const char*>(a.dout) + b * H * kEs);
      const uint4* p4 =
          PROBS ? reinterpret_cast<const uint4*>(static_cast<const char*>(a.perm) + row * H * kEs)
                : nullptr;
      uint4* g4 = reinterpret_cast<uint4*>(static_cast<char*>(a.perm_grad) + row * H * kEs);
      const int64_t nv = H / kE;
      constexpr int kU = 4;  // vectors per lane in flight
      for (int64_t v0 = lane; v0 < nv; v0 += 32 * kU) {
        uint4 dq[kU], pq[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int64_t v = v0 + 32 * u;
          if (v < nv) {
            dq[u] = __ldg(d4 + v);
            if constexpr (PROBS) pq[u] = __ldg(p4 + v);
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int64_t v = v0 + 32 * u;
          if (v < nv) {
            float d[kE], o[kE];
            unpack16<DT>(dq[u], d);
#pragma unroll
            for (int i = 0; i < kE; ++i) o[i] = d[i] * pr;
            g4[v] = pack16<DT>(o);
            if constexpr (PROBS) {
              float x[kE];
              unpack16<DT>(pq[u], x);
#pragma unroll
              for (int i = 0; i < kE; ++i) dot = fmaf(d[i], x[i], dot);
            }
          }
        }
      }
    } else if (PAIRS) {
      // 16-bit rows of even length, 4-byte aligned: two elements per access
      const uint32_t* d2 = reinterpret_cast<const uint32_t*>(
          static_cast<const uint16_t*>(a.dout) + b * H);
      const uint32_t* p2 = PROBS ? reinterpret_cast<const uint32_t*>(
                                       static_cast<const uint16_t*>(a.perm) + row * H)
                                 : nullptr;
      uint32_t* g2 = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.perm_grad) + row * H);
      const int64_t nv = H / 2;
      constexpr int kU = 8;
      for (int64_t v0 = lane; v0 < nv; v0 += 32 * kU) {
        uint32_t dq[kU], pq[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int64_t v = v0 + 32 * u;
          if (v < nv) {
            dq[u] = __ldg(d2 + v);
            if constexpr (PROBS) pq[u] = __ldg(p2 + v);
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int64_t v = v0 + 32 * u;
          if (v < nv) {
            const uint4 dd = make_uint4(dq[u], 0, 0, 0);
            float d[8];
            unpack16<DT>(dd, d);
            float o[8] = {d[0] * pr, d[1] * pr, 0, 0, 0, 0, 0, 0};
            g2[v] = pack16<DT>(o).x;
            if constexpr (PROBS) {
              float x[8];
              unpack16<DT>(make_uint4(pq[u], 0, 0, 0), x);
              dot = fmaf(d[0], x[0], dot);
              dot = fmaf(d[1], x[1], dot);
            }
          }
        }
      }
    } else {
      for (int64_t h = lane; h < H; h += 32) {
        const float d = E::get(a.dout, b * H + h);
        E::put(a.perm_grad, row * H + h, d * pr);
        if constexpr (PROBS) dot = fmaf(d, E::get(a.perm, row * H + h), dot);
      }
    }
    if constexpr (PROBS) {
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, d);
      if (lane == 0 && a.probs_grad) {
        if (a.probs_grad_f32)
          static_cast<float*>(a.probs_grad)[p] = dot;
        else
          E::put(a.probs_grad, p, dot);
      }
    }
  }
}

template <int DT, bool PROBS>
void launch_p(const UnpermArgs& a, bool vec, bool pairs, int grid, cudaStream_t s) {
  const dim3 g(static_cast<unsigned>(grid)), b(kUThreads);
  if (vec)
    launch_pdl(unpermute_grad_kernel<DT, PROBS, true, false>, g, b, 0, s, 1, a);
  else if (pairs && DT != PGG_F32)
    launch_pdl(unpermute_grad_kernel<DT, PROBS, false, DT != PGG_F32>, g, b, 0, s, 1, a);
  else
    launch_pdl(unpermute_grad_kernel<DT, PROBS, false, false>, g, b, 0, s, 1, a);
}

template <int DT>
cudaError_t launch_t(const UnpermArgs& a, bool probs, bool vec, bool pairs, int grid,
                     cudaStream_t s) {
  if (probs)
    launch_p<DT, true>(a, vec, pairs, grid, s);
  else
    launch_p<DT, false>(a, vec, pairs, grid, s);
  return cudaGetLastError();
}

}  // namespace

// vec: H * sizeof(dtype) a multiple of 16 and perm, d_out, perm_grad 16-byte
// aligned; pairs (16-bit dtypes): H even and those pointers 4-byte aligned.
cudaError_t launch_unpermute_grad(int dtype, const UnpermArgs& a, bool vec, bool pairs,
                                  int num_sms, cudaStream_t stream) {
  int64_t grid = (a.M + kUThreads / 32 - 1) / (kUThreads / 32);
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  const bool probs = a.probs != nullptr;
  const int g = static_cast<int>(grid);
  if (dtype == PGG_F32) return launch_t<PGG_F32>(a, probs, vec, false, g, stream);
  if (dtype == PGG_F16) return launch_t<PGG_F16>(a, probs, vec, pairs, g, stream);
  if (dtype == PGG_BF16) return launch_t<PGG_BF16>(a, probs, vec, pairs, g, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pgg
