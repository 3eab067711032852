// Output path of the forward and weight-gradient epilogues: a warp's 32
// accumulator rows (tensor-memory lanes) x 128 bytes of output columns,
// converted to the output dtype and written straight from registers, so that
// no shared memory is held for staging.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "pgg.h"
#include "pgg_ptx.cuh"

namespace pgg {

// Eight fp32 values -> eight 16-bit values, each rounded to nearest even.
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

// Lane l gets its accumulator row's next 128 bytes of output as eight 16-byte
// blocks: columns c .. c + 31 of an fp32 output, c .. c + 63 of a 16-bit one
// (taddr = the warp's lane quarter at column c). At most 32 values are live.
template <int DT>
__device__ __forceinline__ void chunk_blocks(uint32_t taddr, bool f32, uint4 (&b)[8]) {
  {
    uint32_t v[32];
    ptx::tmem_ld_32x32b_x32(taddr, v);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int p = 0; p < 4; ++p)
      b[p] = f32 ? make_uint4(v[4 * p], v[4 * p + 1], v[4 * p + 2], v[4 * p + 3])
                 : pack8<DT>(v + 8 * p);
    if (f32) {
#pragma unroll
      for (int p = 4; p < 8; ++p)
        b[p] = make_uint4(v[4 * p], v[4 * p + 1], v[4 * p + 2], v[4 * p + 3]);
    }
  }
  if (!f32) {
    uint32_t v[32];
    ptx::tmem_ld_32x32b_x32(taddr + 32u, v);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int p = 0; p < 4; ++p) b[4 + p] = pack8<DT>(v + 8 * p);
  }
}

// 8 x 8 transpose of 16-byte blocks inside each group of eight lanes: lane
// 8 g + i ends with block i of the rows that lanes 8 g .. 8 g + 7 held, row
// 8 g + j in b[j]. Three butterfly steps, one per bit of the lane index.
__device__ __forceinline__ void transpose8(uint4 (&b)[8], int lane) {
#pragma unroll
  for (int s = 0; s < 3; ++s) {
    const int m = 1 << s;
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if (p & m) continue;
      const uint4 snd = hi ? b[p] : b[p | m];
      uint4 got;
      got.x = __shfl_xor_sync(0xFFFFFFFFu, snd.x, m);
      got.y = __shfl_xor_sync(0xFFFFFFFFu, snd.y, m);
      got.z = __shfl_xor_sync(0xFFFFFFFFu, snd.z, m);
      got.w = __shfl_xor_sync(0xFFFFFFFFu, snd.w, m);
      if (hi)
        b[p] = got;
      else
        b[p | m] = got;
    }
  }
}

// Writes a chunk from chunk_blocks: rows row0 + r for r < nrows of a
// row-major [*, N] output of oes-byte elements, columns col0 .. col0 +
// 128 / oes - 1, none at or past N. With `words` false the rows are whole
// 16-byte units and out is 16-byte aligned: after the transpose each warp
// store writes four rows' 128 bytes. With `words` true (rows of an even N that
// are not 16-byte multiples, out 4-byte aligned) the blocks go out 4 bytes at
// a time.
__device__ __forceinline__ void store_chunk(uint4 (&b)[8], char* out, int64_t row0, int nrows,
                                            int64_t N, int64_t col0, int oes, bool words,
                                            int lane) {
  transpose8(b, lane);
  const int bi = lane & 7, bg = lane >> 3;
  const int64_t col = col0 + bi * (16 / oes);
  if (!words) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = 8 * bg + j;
      if (r < nrows && col < N)
        *reinterpret_cast<uint4*>(out + ((row0 + r) * N + col) * oes) = b[j];
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = 8 * bg + j;
      const uint32_t w4[4] = {b[j].x, b[j].y, b[j].z, b[j].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t c = col + q * (4 / oes);
        if (r < nrows && c < N)
          *reinterpret_cast<uint32_t*>(out + ((row0 + r) * N + c) * oes) = w4[q];
      }
    }
  }
}

}  // namespace pgg
