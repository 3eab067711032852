// Copies of operand rows that the tensor-memory-access unit cannot stream
// (rows of a 16-bit operand whose byte length 2N is not a multiple of 16),
// by warps with cp.async, into the layout TMA would have written.
#pragma once

#include <cstdint>

#include "pgg_ptx.cuh"

namespace pgg {

// 8 bytes global -> shared (both 8-byte aligned), through L1; `src_bytes`
// (0 .. 8) of them are read, the rest are zero-filled.
__device__ __forceinline__ void cp_async_8(uint32_t dst_smem, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst_smem), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// 16 bytes through L1 (the 16-byte wrapper in pgg_ptx.cuh bypasses it); `src_bytes` 0 .. 16.
__device__ __forceinline__ void cp_async_16_ca(uint32_t dst_smem, const void* src,
                                               uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// Bytes [b, b + size) of a row segment of `seg` valid bytes: how many to read.
__device__ __forceinline__ uint32_t piece_bytes(int b, int size, int seg) {
  const int v = seg - b;
  return static_cast<uint32_t>(v <= 0 ? 0 : (v < size ? v : size));
}

// One residue class of rows (r = j, j + 4, j + 8, ... < nrows), every one of
// them starting at the same 16-byte phase, copied SIZE bytes per lane: 128 /
// SIZE lanes per row, 32 * SIZE / 128 rows per warp instruction. This warp
// takes every nwarps-th group of rows.
template <int SIZE>
__device__ __forceinline__ void gather_class(uint32_t dst, const char* src, int64_t row_bytes,
                                             int j, int nrows, int nvalid, int seg,
                                             const void* safe, int lane, int w, int nwarps) {
  constexpr int kLanesPerRow = 128 / SIZE;
  constexpr int kRowsPerInst = 32 / kLanesPerRow;
  const int sub = lane / kLanesPerRow;                // row of the instruction
  const int b = (lane % kLanesPerRow) * SIZE;         // byte offset in the segment
  const int cnt = nrows > j ? (nrows - j + 3) / 4 : 0;  // rows of the class
#pragma unroll 2
  for (int i0 = w * kRowsPerInst; i0 < cnt; i0 += nwarps * kRowsPerInst) {
    const int i = i0 + sub;
    if (i < cnt) {
      const int r = j + 4 * i;
      const uint32_t n = r < nvalid ? piece_bytes(b, SIZE, seg) : 0u;
      const uint32_t d = dst + r * 128 + ((((b >> 4) ^ (r & 7)) << 4) | (b & 15));
      const void* s = n ? static_cast<const void*>(src + r * row_bytes + b) : safe;
      if constexpr (SIZE == 16)
        cp_async_16_ca(d, s, n);
      else if constexpr (SIZE == 8)
        cp_async_8(d, s, n);
      else
        ptx::cp_async_4(d, s, n);
    }
  }
}

// Fills rows 0 .. nrows - 1 of a shared-memory tile in the 128-byte swizzle
// layout (16-byte chunk c of tile row r at chunk c ^ (r % 8) of the row's 128
// bytes, rows 128 bytes apart; `dst` 1024-byte aligned) with 128-byte row
// segments read from src + r * row_bytes: the first `seg` bytes of each of the
// first `nvalid` rows, zeros elsewhere. row_bytes is a multiple of 4 and src
// 4-byte aligned, so the rows' 16-byte phase repeats every four rows; each
// class of rows is copied as wide as its phase allows (16, 8 or 4 bytes per
// lane). `safe` is any 16-byte aligned address, named by the zero-filling
// copies (they read nothing). The rows are shared by `nwarps` warps, this one
// being `w`; the caller commits and waits for the copies.
__device__ __forceinline__ void gather_rows_sw128(uint32_t dst, const char* src, int64_t row_bytes,
                                                  int nrows, int nvalid, int seg, const void* safe,
                                                  int lane, int w, int nwarps) {
  const uint32_t a0 = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src)) & 15u;
  const uint32_t step = static_cast<uint32_t>(row_bytes) & 15u;
#pragma unroll 1
  for (int j = 0; j < 4; ++j) {
    const uint32_t phase = (a0 + static_cast<uint32_t>(j) * step) & 15u;
    if (phase == 0)
      gather_class<16>(dst, src, row_bytes, j, nrows, nvalid, seg, safe, lane, w, nwarps);
    else if (phase == 8)
      gather_class<8>(dst, src, row_bytes, j, nrows, nvalid, seg, safe, lane, w, nwarps);
    else
      gather_class<4>(dst, src, row_bytes, j, nrows, nvalid, seg, safe, lane, w, nwarps);
  }
}

}  // namespace pgg
