// Routing preprocess for the fused d_x backward ("MoeInitRoutingGroupedMatmulGrad
// design", sections 2.4.1 and 2.5.3: per-expert prefix tables, the flattened
// list of blocks over all non-empty experts, and the inverse of the routing
// index for rowIdxType 1).
//
// Three small launches, in stream order (for the owner variant of the d_x
// kernel the rank launch also writes the slab bounds; a fourth launch does it
// when topK > 32):
//   route_scan     (1 CTA)  exclusive scan of groupList -> off[G+1]; row-block
//                           counts and their scan -> rbstart[G+1]; the row-block
//                           list {expert, first row, rows}; header reset; the
//                           sum / sign check of groupList.
//   route_scatter  (grid)   range check of expandedRowIdx and its inverse
//                           inv[idx[q]] = q; zeroes the scatter-add tickets.
//   route_rank     (grid)   per token b: its topK expanded rows, the check that
//                           the index is a permutation, and each row's rank
//                           among the token's rows (increasing expanded index);
//                           one lane per position when topK <= 32.
//   route_owner    (grid)   owner variant only: whether each expert's rows are
//                           in increasing original position, and where each
//                           token slab starts inside each expert.
//
// The index is read as the constraint table and note 1 of section "输入输出"
// state: rowIdxType 0 maps expanded row -> original position, rowIdxType 1
// maps original position -> expanded row; original position = b * topK + j.

#include <cstdint>

#include "pgg_internal.h"
#include "pgg_ptx.cuh"

namespace pgg {

namespace {

// Exclusive scan of one int64 per thread over the block (blockDim.x <= 1024).
__device__ int64_t block_exclusive_scan(int64_t v, int64_t* total, int64_t* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  int64_t x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += y;
    }
    if (lane < nwarps) s_warp[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int64_t before = warp > 0 ? s_warp[warp - 1] : 0;
  *total = s_warp[nwarps - 1];
  __syncthreads();  // s_warp is reused by the next call
  return before + x - v;
}

__global__ void __launch_bounds__(1024) route_scan_kernel(const int64_t* __restrict__ group_list,
                                                          int64_t G, int64_t M,
                                                          int rows_per_block, WsHeader* hdr,
                                                          int64_t* __restrict__ off,
                                                          int32_t* __restrict__ rbstart,
                                                          int4* __restrict__ rblist) {
  __shared__ int64_t s_warp[32];
  __shared__ int64_t s_rows, s_blocks;
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_rows = 0;
    s_blocks = 0;
    s_bad = 0;
  }
  __syncthreads();
  for (int64_t base = 0; base < G; base += blockDim.x) {
    const int64_t g = base + tid;
    int64_t c = 0;
    if (g < G) {
      c = group_list[g];
      if (c < 0 || c > M) {
        s_bad = 1;
        c = 0;
      }
    }
    const int64_t nb = (c + rows_per_block - 1) / rows_per_block;
    int64_t tot_c, tot_b;
    const int64_t ex_c = block_exclusive_scan(c, &tot_c, s_warp);
    const int64_t ex_b = block_exclusive_scan(nb, &tot_b, s_warp);
    if (g < G) {
      off[g] = s_rows + ex_c;
      rbstart[g] = static_cast<int32_t>(s_blocks + ex_b);
    }
    __syncthreads();
    if (tid == 0) {
      s_rows += tot_c;
      s_blocks += tot_b;
    }
    __syncthreads();
  }
  const bool ok = !s_bad && s_rows == M;
  const int64_t n_rb = ok ? s_blocks : 0;
  if (tid == 0) {
    off[G] = s_rows;
    rbstart[G] = static_cast<int32_t>(s_blocks);
    hdr->status = ok ? 0u : kStGroupSum;
    hdr->sched_next = 0;
    hdr->n_row_blocks = static_cast<uint32_t>(n_rb);
    hdr->timeout_site = 0;
    hdr->unsorted = 0;
  }
  __syncthreads();
  for (int64_t e = tid; e < n_rb; e += blockDim.x) {
    // largest g with rbstart[g] <= e; it has rbstart[g + 1] > e, so it is non-empty
    int64_t lo = 0, hi = G;
    while (hi - lo > 1) {
      const int64_t mid = (lo + hi) >> 1;
      if (rbstart[mid] <= e)
        lo = mid;
      else
        hi = mid;
    }
    const int64_t j = e - rbstart[lo];
    const int64_t row0 = off[lo] + j * rows_per_block;
    const int64_t rem = off[lo + 1] - row0;
    const int64_t rows = rem < rows_per_block ? rem : rows_per_block;
    rblist[e] = make_int4(static_cast<int>(lo), static_cast<int>(row0), static_cast<int>(rows), 0);
  }
}

__global__ void route_scatter_kernel(const int64_t* __restrict__ idx, int64_t M,
                                     int32_t* __restrict__ inv, WsHeader* hdr,
                                     uint4* __restrict__ tickets4, int64_t n_tickets4) {
  ptx::griddep_wait();  // the header reset of the previous launch
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  bool bad = false;
  for (int64_t q = t0; q < M; q += stride) {
    const int64_t v = idx[q];
    if (v < 0 || v >= M)
      bad = true;
    else
      inv[v] = static_cast<int32_t>(q);
  }
  if (bad) atomicCAS(&hdr->status, 0u, kStIndex);
  for (int64_t t = t0; t < n_tickets4; t += stride) tickets4[t] = make_uint4(0, 0, 0, 0);
}

// Expanded row of original position p, or -1 if the index does not describe a
// permutation at p. Values in inv may be left over from earlier calls; a stale
// value can only pass the check if this call wrote it (see pgg_route_rank).
__device__ __forceinline__ int64_t row_of_position(const int64_t* idx, const int32_t* inv,
                                                   int64_t p, int64_t M, int row_idx_type) {
  if (row_idx_type == 0) {
    // inv[p] = q with idx[q] == p, if some q was scattered to p
    const int64_t q = inv[p];
    if (q < 0 || q >= M || idx[q] != p) return -1;
    return q;
  }
  const int64_t i = idx[p];
  if (i < 0 || i >= M || inv[i] != p) return -1;
  return i;
}

// A stale inv[p] (not written by this call) equal to q passes the type-0 check
// only if idx[q] == p, but then the scatter of this call wrote inv[p]: so every
// accepted p has a preimage, and M positions with preimages among M rows make
// the index a permutation. For type 1 inv[idx[p]] was written by this call by
// some p' with idx[p'] == idx[p]; it equals p for every p only if idx is
// injective.
__global__ void route_rank_kernel(const int64_t* __restrict__ idx, const int32_t* __restrict__ inv,
                                  int64_t batch, int64_t top_k, int64_t M, int row_idx_type,
                                  RowInfo* __restrict__ rowinfo, WsHeader* hdr) {
  ptx::griddep_wait();  // inv of the previous launch
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < batch;
       b += stride) {
    const int64_t p0 = b * top_k;
    for (int64_t j = 0; j < top_k; ++j) {
      const int64_t i = row_of_position(idx, inv, p0 + j, M, row_idx_type);
      if (i < 0) {
        bad = true;
        continue;
      }
      int32_t rank = 0;
      for (int64_t j2 = 0; j2 < top_k; ++j2) {
        const int64_t i2 = row_of_position(idx, inv, p0 + j2, M, row_idx_type);
        if (i2 >= 0 && i2 < i) ++rank;
      }
      RowInfo r;
      r.token = static_cast<int32_t>(b);
      r.rank = rank;
      rowinfo[i] = r;
    }
  }
  if (bad) atomicCAS(&hdr->status, 0u, kStNotPerm);
}

// The same, one lane per original position for topK <= 32: a token's topK
// positions sit in consecutive lanes of one warp, and each lane counts the
// token's rows below its own through shuffles.
__device__ void rank_lanes(const int64_t* __restrict__ idx, const int32_t* __restrict__ inv,
                           int64_t batch, int top_k, int64_t M, int row_idx_type,
                           RowInfo* __restrict__ rowinfo, WsHeader* hdr) {
  const int lane = threadIdx.x & 31;
  const int per_warp = 32 / top_k;  // tokens per warp
  const int slot = lane / top_k, j = lane - slot * top_k;
  const int base = slot * top_k;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  bool bad = false;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       w * per_warp < batch; w += warps) {
    const int64_t b = w * per_warp + slot;
    const bool valid = slot < per_warp && b < batch;
    const int64_t i = valid ? row_of_position(idx, inv, b * top_k + j, M, row_idx_type) : -1;
    int32_t rank = 0;
    for (int j2 = 0; j2 < top_k; ++j2) {
      const int64_t i2 = __shfl_sync(0xFFFFFFFFu, i, valid ? base + j2 : lane);
      if (i2 >= 0 && i2 < i) ++rank;
    }
    if (valid) {
      if (i < 0) {
        bad = true;
      } else {
        RowInfo r;
        r.token = static_cast<int32_t>(b);
        r.rank = rank;
        rowinfo[i] = r;
      }
    }
  }
  if (bad) atomicCAS(&hdr->status, 0u, kStNotPerm);
}

__global__ void route_rank_lanes_kernel(const int64_t* __restrict__ idx,
                                        const int32_t* __restrict__ inv, int64_t batch,
                                        int top_k, int64_t M, int row_idx_type,
                                        RowInfo* __restrict__ rowinfo, WsHeader* hdr) {
  ptx::griddep_wait();  // inv of the previous launch
  rank_lanes(idx, inv, batch, top_k, M, row_idx_type, rowinfo, hdr);
}

__global__ void header_reset_kernel(WsHeader* hdr) {
  hdr->status = 0;
  hdr->sched_next = 0;
  hdr->n_row_blocks = 0;
  hdr->timeout_site = 0;
  hdr->unsorted = 0;
}

// Original position of expanded row i (valid once the index is a permutation).
__device__ __forceinline__ int64_t position_of_row(const int64_t* idx, const int32_t* inv,
                                                   int64_t i, int row_idx_type) {
  return row_idx_type == 0 ? idx[i] : static_cast<int64_t>(inv[i]);
}

// Owner variant: (1) whether every expert's rows are in increasing original
// position (then the rows of a token slab form one contiguous range inside
// each expert); (2) seg[g][s] = first row of expert g whose position is at
// least s * slab_tokens * topK. Each row i of expert g writes the entries from
// its predecessor's slab (exclusive) to its own (inclusive); the expert's last
// row writes the rest with the expert's end, and empty experts write their
// offset everywhere. Meaningful when sorted; every write stays inside seg.
constexpr int kOffSmem = 2048;  // experts whose offsets fit in shared memory

// The owner work over rows t0, t0 + stride, ... and experts likewise. Robust
// to an index that is not a permutation (its check may run concurrently):
// positions outside [0, M) only mark the rows unsorted, and every write stays
// inside seg.
__device__ void owner_rows(const int64_t* __restrict__ idx, const int32_t* __restrict__ inv,
                           const int64_t* offs, int64_t M, int64_t G, int64_t top_k,
                           int row_idx_type, int n_slabs, int slab_tokens,
                           int32_t* __restrict__ seg, WsHeader* hdr, int64_t t0, int64_t stride) {
  const int64_t slab_rows = static_cast<int64_t>(slab_tokens) * top_k;
  const int64_t ns = n_slabs;
  bool unsorted = false;
  for (int64_t i = t0; i < M; i += stride) {
    // expert of row i: largest g with off[g] <= i
    int64_t lo = 0, hi = G;
    while (hi - lo > 1) {
      const int64_t mid = (lo + hi) >> 1;
      if (offs[mid] <= i)
        lo = mid;
      else
        hi = mid;
    }
    int32_t* row = seg + lo * (ns + 1);
    const int64_t p = position_of_row(idx, inv, i, row_idx_type);
    if (p < 0 || p >= M) {
      unsorted = true;
      continue;
    }
    const int64_t sl = p / slab_rows;
    int64_t prev = -1;
    if (i > offs[lo]) {
      const int64_t pp = position_of_row(idx, inv, i - 1, row_idx_type);
      if (pp < 0 || pp >= M || pp > p) unsorted = true;
      prev = (pp < 0 || pp >= M) ? sl : pp / slab_rows;
    }
    for (int64_t t = prev + 1; t <= sl && t <= ns; ++t) row[t] = static_cast<int32_t>(i);
    if (i + 1 == offs[lo + 1])
      for (int64_t t = sl + 1; t <= ns; ++t) row[t] = static_cast<int32_t>(i + 1);
  }
  if (unsorted) atomicOr(&hdr->unsorted, 1u);
  for (int64_t g = t0; g < G; g += stride)
    if (offs[g] == offs[g + 1])
      for (int64_t t = 0; t <= ns; ++t) seg[g * (ns + 1) + t] = static_cast<int32_t>(offs[g]);
}

// Expert offsets in shared memory when they fit (the caller syncs).
__device__ const int64_t* stage_offsets(const int64_t* off, int64_t G, int64_t* s_off) {
  if (G + 1 > kOffSmem) return off;
  for (int64_t g = threadIdx.x; g <= G; g += blockDim.x) s_off[g] = off[g];
  return s_off;
}

__global__ void route_owner_kernel(const int64_t* __restrict__ idx, const int32_t* __restrict__ inv,
                                   const int64_t* __restrict__ off, int64_t M, int64_t G,
                                   int64_t top_k, int row_idx_type, int n_slabs,
                                   int slab_tokens, int32_t* __restrict__ seg, WsHeader* hdr) {
  __shared__ int64_t s_off[kOffSmem];
  ptx::griddep_wait();  // ranks and status of the previous launch
  if (hdr->status != 0) return;  // the index is not a permutation: nothing to order
  const int64_t* offs = stage_offsets(off, G, s_off);
  __syncthreads();
  owner_rows(idx, inv, offs, M, G, top_k, row_idx_type, n_slabs, slab_tokens, seg, hdr,
             static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
             static_cast<int64_t>(gridDim.x) * blockDim.x);
}

// The lane-per-position ranks and, in the same launch, the owner work (for
// the owner variant with topK <= 32).
__global__ void route_rank_owner_kernel(const int64_t* __restrict__ idx,
                                        const int32_t* __restrict__ inv,
                                        const int64_t* __restrict__ off, int64_t batch, int top_k,
                                        int64_t M, int64_t G, int row_idx_type, int n_slabs,
                                        int slab_tokens, RowInfo* __restrict__ rowinfo,
                                        int32_t* __restrict__ seg, WsHeader* hdr) {
  __shared__ int64_t s_off[kOffSmem];
  ptx::griddep_wait();  // inv, off and the status of the previous launches
  const uint32_t st = hdr->status;  // index range or group sum already wrong: no order
  const int64_t* offs = stage_offsets(off, G, s_off);
  __syncthreads();
  rank_lanes(idx, inv, batch, top_k, M, row_idx_type, rowinfo, hdr);
  if (st == 0)
    owner_rows(idx, inv, offs, M, G, top_k, row_idx_type, n_slabs, slab_tokens, seg, hdr,
               static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
               static_cast<int64_t>(gridDim.x) * blockDim.x);
}

// Every original position must have an expanded row (see row_of_position).
__global__ void perm_check_kernel(const int64_t* __restrict__ idx, const int32_t* __restrict__ inv,
                                  int64_t M, int row_idx_type, WsHeader* hdr) {
  ptx::griddep_wait();  // inv of the previous launch
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < M; p += stride)
    if (row_of_position(idx, inv, p, M, row_idx_type) < 0) bad = true;
  if (bad) atomicCAS(&hdr->status, 0u, kStNotPerm);
}

}  // namespace

// Index validation without experts (for the unpermute backward): header
// reset, range check and inverse, permutation check. Afterwards the expanded
// row of position p is inv[p] (rowIdxType 0) or idx[p] (rowIdxType 1).
cudaError_t launch_index_prep(const int64_t* idx, int64_t M, int row_idx_type, int32_t* inv,
                              WsHeader* hdr, int num_sms, cudaStream_t stream) {
  header_reset_kernel<<<1, 1, 0, stream>>>(hdr);
  int64_t blocks = (M + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaError_t err = launch_pdl(route_scatter_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256),
                               0, stream, 1, idx, M, inv, hdr, static_cast<uint4*>(nullptr),
                               static_cast<int64_t>(0));
  if (err != cudaSuccess) return err;
  return launch_pdl(perm_check_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                    1, idx, static_cast<const int32_t*>(inv), M, row_idx_type, hdr);
}

cudaError_t launch_route_prep(const Plan& plan, const int64_t* idx, const int64_t* group_list,
                              void* workspace, int num_sms, cudaStream_t stream) {
  char* ws = static_cast<char*>(workspace);
  const Layout& L = plan.layout;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws + L.hdr);
  int64_t* off = reinterpret_cast<int64_t*>(ws + L.off);
  int32_t* rbstart = reinterpret_cast<int32_t*>(ws + L.rbstart);
  int4* rblist = reinterpret_cast<int4*>(ws + L.rblist);
  int32_t* inv = reinterpret_cast<int32_t*>(ws + L.inv);
  RowInfo* rowinfo = reinterpret_cast<RowInfo*>(ws + L.rowinfo);
  uint4* tickets4 = reinterpret_cast<uint4*>(ws + L.tickets);

  route_scan_kernel<<<1, 1024, 0, stream>>>(group_list, plan.G, plan.M, plan.rows_per_block, hdr,
                                            off, rbstart, rblist);
  const int64_t work = plan.M > plan.layout.n_tickets / 4 ? plan.M : plan.layout.n_tickets / 4;
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  // the later launches may be scheduled while their predecessor drains; each
  // waits for it (griddepcontrol.wait) before reading anything
  cudaError_t err = launch_pdl(route_scatter_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256),
                               0, stream, 1, idx, plan.M, inv, hdr, tickets4,
                               plan.layout.n_tickets / 4);
  if (err != cudaSuccess) return err;
  const int32_t* cinv = inv;
  const int64_t* coff = off;
  int32_t* seg = reinterpret_cast<int32_t*>(ws + L.seg);
  bool owner_done = false;
  if (plan.topK <= 32) {
    const int64_t per_block = 8 * (32 / plan.topK);  // tokens per 256-thread block
    int64_t rblocks = (plan.batch + per_block - 1) / per_block;
    if (plan.n_slabs > 0) {
      // ranks and slab bounds in one launch: enough blocks for the rows too
      const int64_t oblocks = (plan.M + 255) / 256;
      if (oblocks > rblocks) rblocks = oblocks;
    }
    if (rblocks > cap) rblocks = cap;
    if (rblocks < 1) rblocks = 1;
    if (plan.n_slabs > 0) {
      err = launch_pdl(route_rank_owner_kernel, dim3(static_cast<unsigned>(rblocks)), dim3(256), 0,
                       stream, 1, idx, cinv, coff, plan.batch, static_cast<int>(plan.topK), plan.M,
                       plan.G, plan.row_idx_type, plan.n_slabs, plan.slab_tokens, rowinfo, seg,
                       hdr);
      owner_done = true;
    } else {
      err = launch_pdl(route_rank_lanes_kernel, dim3(static_cast<unsigned>(rblocks)), dim3(256), 0,
                       stream, 1, idx, cinv, plan.batch, static_cast<int>(plan.topK), plan.M,
                       plan.row_idx_type, rowinfo, hdr);
    }
    if (err != cudaSuccess) return err;
  } else {
    int64_t rblocks = (plan.batch + 127) / 128;
    if (rblocks > cap) rblocks = cap;
    if (rblocks < 1) rblocks = 1;
    err = launch_pdl(route_rank_kernel, dim3(static_cast<unsigned>(rblocks)), dim3(128), 0, stream,
                     1, idx, cinv, plan.batch, plan.topK, plan.M, plan.row_idx_type, rowinfo, hdr);
    if (err != cudaSuccess) return err;
  }
  if (plan.n_slabs > 0 && !owner_done) {
    int64_t oblocks = (plan.M + 255) / 256;
    if (oblocks > cap) oblocks = cap;
    if (oblocks < 1) oblocks = 1;
    err = launch_pdl(route_owner_kernel, dim3(static_cast<unsigned>(oblocks)), dim3(256), 0, stream,
                     1, idx, cinv, coff, plan.M, plan.G, plan.topK, plan.row_idx_type,
                     plan.n_slabs, plan.slab_tokens, seg, hdr);
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

}  // namespace pgg
