// Oracle for the MoE permute + grouped-matmul backward: the input gradient d_x
// (the fused operator) and the weight gradient d_weight (its separate
// companion operator).
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or call
// this file; only the tests, the smoke check and the benchmark's CPU-baseline
// leg do. It shares no code, header, table or constant with the CUDA library.
//
// What it computes (page "MoeInitRoutingGroupedMatmulGrad design", section
// "数学定义和公式", element-wise gradient formula and its scalar form):
//
//     d_x[b, k] = sum over expanded rows i with batch(i) == b of
//                 sum over n of d_y[i, n] * weight[g(i), k, n]
//
// where g(i) is the expert whose block of the expanded order holds row i
// (groupList gives the per-expert row counts, not a cumulative sum: section
// "输入输出"), and batch(i) = original_pos(i) / topK (section "数学定义",
// Step 2). expandedRowIdx is read according to rowIdxType (section "输入输出",
// note 1): 0 = gather form, entry i holds the original position of expanded
// row i; 1 = scatter form, entry p holds the expanded row of original
// position p.
//
// The steps follow the definition directly and in this order:
//   1. every input element is widened exactly to double (fp32, fp16 and bf16
//      values are all exactly representable in double);
//   2. the expert of each expanded row is found by walking groupList;
//   3. the original-position -> expanded-row map is built from the index;
//   4. for each requested token b, for j = 0 .. topK-1 in increasing order,
//      with i the expanded row of original position b*topK + j, the dot
//      products sum_n d_y[i,n]*weight[g(i),k,n] are formed in double (n
//      ascending) and added into an accumulator row; the accumulator is the
//      output row.
// No blocking, no fusion beyond the formula, no reordering of the sum over n.
//
// Input validation mirrors the constraint table (section "约束"): batch > 0,
// topK > 0, rowIdxType in {0, 1}, M == batch * topK, every groupList entry
// >= 0 and their sum == M, expandedRowIdx a permutation of [0, M).
//
// d_weight (same page, section 1.2 "为何不计算 d_weight" item 3: a separate
// grouped matmul expanded_x^T @ d_y per expert; section 1.1: the forward's
// MoeInitRouting lays the token rows out by expert as expanded_x, so row i of
// expanded_x is row batch(i) of the forward input x):
//
//     d_weight[g, k, n] = sum over expanded rows i of expert g of
//                         x[batch(i), k] * d_y[i, n]
//
// Steps, in this order: widen every input element to double; find the expert
// of each expanded row by walking groupList and the original position of each
// row from the index; for each requested (g, k), for the rows i of expert g in
// increasing order, add x[batch(i), k] * d_y[i, n] into an accumulator row
// over n. An expert with no rows has a zero gradient.
//
// The forward that these are the gradients of (same page, section 1.1 and
// the forward chain of section 1.2: MoeInitRouting(x) -> expanded_x, then
// GroupedMatmul(expanded_x, weight) -> y, expanded_x @ weight per expert):
//
//     y[i, n] = sum over k of x[batch(i), k] * weight[g(i), k, n]
//
// Steps: widen; expert and original position of each row as above; for each
// requested expanded row i, the dot products over k (ascending) of x's row
// batch(i) with the columns of weight[g(i)].
//
// The probs-weighted unpermute backward (page "NPU DeepSeek-V3.2-Exp TileLang
// operator practice", section moe_token_unpermute_grad): the forward combine
// out[b] = sum_j prob[b, j] * permuted[row(b, j)] has the gradients
//
//     perm_grad[row(b, j), h] = d_out[b, h] * prob[b, j]       (prob = 1 without probs)
//     probs_grad[b, j]        = sum over h of d_out[b, h] * permuted[row(b, j), h]
//
// with row(b, j) the expanded row of original position b * topK + j, read from
// the index in either form as above. Steps: widen; the position -> row map;
// for each token b and j in increasing order, the scaled copy and the dot
// product over h (ascending).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

enum { kF32 = 0, kF16 = 1, kBF16 = 2 };

enum {
  kOk = 0,
  kErrNull = 1,
  kErrShape = 2,
  kErrAttr = 3,
  kErrDtype = 4,
  kErrIndex = 16,
  kErrGroupSum = 17,
  kErrNotPerm = 18,
};

// IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double decode_binary16(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1f;
  const int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = std::ldexp(static_cast<double>(f), -24);  // subnormal: f * 2^-14 * 2^-10
  } else if (e == 31) {
    v = (f == 0) ? INFINITY : NAN;
  } else {
    v = std::ldexp(static_cast<double>(1024 + f), e - 25);  // (1 + f/1024) * 2^(e-15)
  }
  return sign ? -v : v;
}

// bfloat16: the upper 16 bits of an IEEE 754 binary32.
double decode_bfloat16(uint16_t h) {
  const uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

double decode_binary32(const void* p, int64_t idx) {
  float f;
  std::memcpy(&f, static_cast<const char*>(p) + 4 * idx, sizeof f);
  return static_cast<double>(f);
}

struct Decoder {
  int dtype;
  std::vector<double> f16_table;  // all 65536 binary16 values, built by decode_binary16
  explicit Decoder(int dt) : dtype(dt) {
    if (dt == kF16) {
      f16_table.resize(65536);
      for (uint32_t h = 0; h < 65536; ++h) f16_table[h] = decode_binary16(static_cast<uint16_t>(h));
    }
  }
  double at(const void* base, int64_t idx) const {
    if (dtype == kF32) return decode_binary32(base, idx);
    const uint16_t h = static_cast<const uint16_t*>(base)[idx];
    return dtype == kF16 ? f16_table[h] : decode_bfloat16(h);
  }
};

struct Routing {
  std::vector<int64_t> group_of_row;  // g(i) for every expanded row i
  std::vector<int64_t> row_of_pos;    // expanded row of original position p
  std::vector<int64_t> pos_of_row;    // original position of expanded row i
  std::vector<int64_t> first_row;     // first expanded row of expert g (G + 1 entries)
};

// Validates the inputs against the constraint table and builds g(i) and the
// original-position -> expanded-row map.
int build_routing(const int64_t* idx, const int64_t* group_list, int64_t M, int64_t G,
                  int row_idx_type, Routing* r) {
  int64_t total = 0;
  for (int64_t g = 0; g < G; ++g) {
    if (group_list[g] < 0 || group_list[g] > M) return kErrGroupSum;
    total += group_list[g];
  }
  if (total != M) return kErrGroupSum;

  r->group_of_row.assign(M, -1);
  r->first_row.assign(G + 1, 0);
  int64_t i = 0;
  for (int64_t g = 0; g < G; ++g) {
    r->first_row[g] = i;
    for (int64_t c = 0; c < group_list[g]; ++c) r->group_of_row[i++] = g;
  }
  r->first_row[G] = i;

  for (int64_t q = 0; q < M; ++q)
    if (idx[q] < 0 || idx[q] >= M) return kErrIndex;

  r->row_of_pos.assign(M, -1);
  if (row_idx_type == 0) {
    // gather form: idx[i] = original position of expanded row i
    for (int64_t row = 0; row < M; ++row) {
      if (r->row_of_pos[idx[row]] != -1) return kErrNotPerm;
      r->row_of_pos[idx[row]] = row;
    }
  } else {
    // scatter form: idx[p] = expanded row of original position p
    std::vector<char> seen(M, 0);
    for (int64_t p = 0; p < M; ++p) {
      if (seen[idx[p]]) return kErrNotPerm;
      seen[idx[p]] = 1;
      r->row_of_pos[p] = idx[p];
    }
  }
  r->pos_of_row.assign(M, -1);
  for (int64_t p = 0; p < M; ++p) r->pos_of_row[r->row_of_pos[p]] = p;
  return kOk;
}

struct Job {
  const void* dy;
  const void* w;
  const Decoder* dec;
  const Routing* routing;
  const int64_t* tokens;
  int64_t ntokens, N, K, topK;
  double* out;
};

void run_tokens(const Job& job, int64_t t_begin, int64_t t_end) {
  const int64_t N = job.N, K = job.K;
  std::vector<double> dy_row(N);
  std::vector<double> acc(K);
  for (int64_t t = t_begin; t < t_end; ++t) {
    const int64_t b = job.tokens ? job.tokens[t] : t;
    for (int64_t k = 0; k < K; ++k) acc[k] = 0.0;
    for (int64_t j = 0; j < job.topK; ++j) {
      const int64_t i = job.routing->row_of_pos[b * job.topK + j];
      const int64_t g = job.routing->group_of_row[i];
      for (int64_t n = 0; n < N; ++n) dy_row[n] = job.dec->at(job.dy, i * N + n);
      for (int64_t k = 0; k < K; ++k) {
        const int64_t wbase = (g * K + k) * N;
        double s = 0.0;
        for (int64_t n = 0; n < N; ++n) s += dy_row[n] * job.dec->at(job.w, wbase + n);
        acc[k] += s;
      }
    }
    double* o = job.out + t * K;
    for (int64_t k = 0; k < K; ++k) o[k] = acc[k];
  }
}

struct DwJob {
  const void* x;
  const void* dy;
  const Decoder* dec;
  const Routing* routing;
  const int64_t* sel_g;
  const int64_t* sel_k;
  int64_t nsel, N, K, topK;
  double* out;
};

void run_dw_rows(const DwJob& job, int64_t s_begin, int64_t s_end) {
  const int64_t N = job.N, K = job.K;
  std::vector<double> acc(N);
  for (int64_t s = s_begin; s < s_end; ++s) {
    const int64_t g = job.sel_g ? job.sel_g[s] : s / K;
    const int64_t k = job.sel_k ? job.sel_k[s] : s % K;
    for (int64_t n = 0; n < N; ++n) acc[n] = 0.0;
    for (int64_t i = job.routing->first_row[g]; i < job.routing->first_row[g + 1]; ++i) {
      const int64_t b = job.routing->pos_of_row[i] / job.topK;
      const double xv = job.dec->at(job.x, b * K + k);
      for (int64_t n = 0; n < N; ++n) acc[n] += xv * job.dec->at(job.dy, i * N + n);
    }
    double* o = job.out + s * N;
    for (int64_t n = 0; n < N; ++n) o[n] = acc[n];
  }
}

struct FwdJob {
  const void* x;
  const void* w;
  const Decoder* dec;
  const Routing* routing;
  const int64_t* rows;
  int64_t nrows, N, K, topK;
  double* out;
};

void run_fwd_rows(const FwdJob& job, int64_t s_begin, int64_t s_end) {
  const int64_t N = job.N, K = job.K;
  std::vector<double> x_row(K);
  for (int64_t s = s_begin; s < s_end; ++s) {
    const int64_t i = job.rows ? job.rows[s] : s;
    const int64_t b = job.routing->pos_of_row[i] / job.topK;
    const int64_t g = job.routing->group_of_row[i];
    for (int64_t k = 0; k < K; ++k) x_row[k] = job.dec->at(job.x, b * K + k);
    double* o = job.out + s * N;
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += x_row[k] * job.dec->at(job.w, (g * K + k) * N + n);
      o[n] = acc;
    }
  }
}

struct UnpermJob {
  const void* perm;
  const void* dout;
  const void* probs;  // may be null
  const Decoder* dec;
  const Routing* routing;
  int64_t batch, topK, H;
  double* perm_grad;   // [M, H]
  double* probs_grad;  // [batch, topK] (only with probs)
};

void run_unperm_tokens(const UnpermJob& job, int64_t b_begin, int64_t b_end) {
  const int64_t H = job.H;
  std::vector<double> d(H);
  for (int64_t b = b_begin; b < b_end; ++b) {
    for (int64_t h = 0; h < H; ++h) d[h] = job.dec->at(job.dout, b * H + h);
    for (int64_t j = 0; j < job.topK; ++j) {
      const int64_t p = b * job.topK + j;
      const int64_t i = job.routing->row_of_pos[p];
      const double pr = job.probs ? job.dec->at(job.probs, p) : 1.0;
      double dot = 0.0;
      for (int64_t h = 0; h < H; ++h) {
        job.perm_grad[i * H + h] = d[h] * pr;
        if (job.probs) dot += d[h] * job.dec->at(job.perm, i * H + h);
      }
      if (job.probs) job.probs_grad[p] = dot;
    }
  }
}

template <class JobT, class Fn>
void run_pool(const JobT& job, int64_t count, int nthreads, Fn fn) {
  if (nthreads <= 0) nthreads = static_cast<int>(std::thread::hardware_concurrency());
  if (nthreads <= 0) nthreads = 1;
  if (nthreads > count) nthreads = static_cast<int>(count > 0 ? count : 1);
  std::vector<std::thread> pool;
  const int64_t per = (count + nthreads - 1) / nthreads;
  for (int th = 0; th < nthreads; ++th) {
    const int64_t lo = th * per;
    const int64_t hi = lo + per < count ? lo + per : count;
    if (lo >= hi) break;
    pool.emplace_back(fn, std::cref(job), lo, hi);
  }
  for (auto& t : pool) t.join();
}

}  // namespace

extern "C" {

// Widens n elements of the given dtype to double (exposed so that the tests
// can pin the decoders against independent conversions).
int oracle_decode(const void* src, int dtype, int64_t n, double* dst) {
  if (!src || !dst) return kErrNull;
  if (dtype != kF32 && dtype != kF16 && dtype != kBF16) return kErrDtype;
  Decoder dec(dtype);
  for (int64_t q = 0; q < n; ++q) dst[q] = dec.at(src, q);
  return kOk;
}

// d_x rows for the requested tokens (all tokens when tokens == NULL, then
// ntokens must equal batch). out is [ntokens, K] double, row-major.
// dy is [M, N], w is [G, K, N], both row-major in the given dtype.
int oracle_dx(const void* dy, const void* w, int dtype, const int64_t* expanded_row_idx,
              const int64_t* group_list, int64_t M, int64_t N, int64_t K, int64_t G,
              int64_t batch, int64_t topK, int row_idx_type, const int64_t* tokens,
              int64_t ntokens, double* out, int nthreads) {
  if (!dy || !w || !expanded_row_idx || !group_list || !out) return kErrNull;
  if (dtype != kF32 && dtype != kF16 && dtype != kBF16) return kErrDtype;
  if (batch <= 0 || topK <= 0 || (row_idx_type != 0 && row_idx_type != 1)) return kErrAttr;
  if (M <= 0 || N <= 0 || K <= 0 || G <= 0) return kErrShape;
  if (M != batch * topK) return kErrShape;
  if (!tokens && ntokens != batch) return kErrShape;
  for (int64_t t = 0; tokens && t < ntokens; ++t)
    if (tokens[t] < 0 || tokens[t] >= batch) return kErrShape;

  Routing routing;
  const int rc = build_routing(expanded_row_idx, group_list, M, G, row_idx_type, &routing);
  if (rc != kOk) return rc;

  Decoder dec(dtype);
  Job job{dy, w, &dec, &routing, tokens, ntokens, N, K, topK, out};
  run_pool(job, ntokens, nthreads, run_tokens);
  return kOk;
}

// Probs-weighted unpermute backward. perm [M, H] (needed only with probs),
// dout [batch, H], probs [batch, topK] or null, all in the given dtype;
// perm_grad [M, H] double; probs_grad [batch, topK] double (written only
// with probs). The index is the permutation between original positions and
// expanded rows (rowIdxType as for oracle_dx); there are no experts here.
int oracle_unpermute_grad(const void* perm, const void* dout, const void* probs, int dtype,
                          const int64_t* expanded_row_idx, int64_t M, int64_t H, int64_t batch,
                          int64_t topK, int row_idx_type, double* perm_grad, double* probs_grad,
                          int nthreads) {
  if (!dout || !expanded_row_idx || !perm_grad) return kErrNull;
  if (probs && (!perm || !probs_grad)) return kErrNull;
  if (dtype != kF32 && dtype != kF16 && dtype != kBF16) return kErrDtype;
  if (batch <= 0 || topK <= 0 || (row_idx_type != 0 && row_idx_type != 1)) return kErrAttr;
  if (M <= 0 || H <= 0) return kErrShape;
  if (M != batch * topK) return kErrShape;
  const int64_t one_group = M;
  Routing routing;
  const int rc = build_routing(expanded_row_idx, &one_group, M, 1, row_idx_type, &routing);
  if (rc != kOk) return rc;
  Decoder dec(dtype);
  UnpermJob job{perm, dout, probs, &dec, &routing, batch, topK, H, perm_grad, probs_grad};
  run_pool(job, batch, nthreads, run_unperm_tokens);
  return kOk;
}

// Forward rows y[rows[s], 0..N-1] for s < nrows (all M rows in order when
// rows == NULL, then nrows must equal M). out is [nrows, N] double. x is
// [batch, K], w is [G, K, N], both in the given dtype.
int oracle_fwd(const void* x, const void* w, int dtype, const int64_t* expanded_row_idx,
               const int64_t* group_list, int64_t M, int64_t N, int64_t K, int64_t G,
               int64_t batch, int64_t topK, int row_idx_type, const int64_t* rows, int64_t nrows,
               double* out, int nthreads) {
  if (!x || !w || !expanded_row_idx || !group_list || !out) return kErrNull;
  if (dtype != kF32 && dtype != kF16 && dtype != kBF16) return kErrDtype;
  if (batch <= 0 || topK <= 0 || (row_idx_type != 0 && row_idx_type != 1)) return kErrAttr;
  if (M <= 0 || N <= 0 || K <= 0 || G <= 0) return kErrShape;
  if (M != batch * topK) return kErrShape;
  if (!rows && nrows != M) return kErrShape;
  for (int64_t s = 0; rows && s < nrows; ++s)
    if (rows[s] < 0 || rows[s] >= M) return kErrShape;

  Routing routing;
  const int rc = build_routing(expanded_row_idx, group_list, M, G, row_idx_type, &routing);
  if (rc != kOk) return rc;

  Decoder dec(dtype);
  FwdJob job{x, w, &dec, &routing, rows, nrows, N, K, topK, out};
  run_pool(job, nrows, nthreads, run_fwd_rows);
  return kOk;
}

// d_weight rows dW[sel_g[s], sel_k[s], 0..N-1] for s < nsel (all G*K rows in
// (g, k) order when sel_g == sel_k == NULL, then nsel must equal G * K). out
// is [nsel, N] double. x is [batch, K], dy is [M, N], both in the given dtype.
int oracle_dw(const void* x, const void* dy, int dtype, const int64_t* expanded_row_idx,
              const int64_t* group_list, int64_t M, int64_t N, int64_t K, int64_t G,
              int64_t batch, int64_t topK, int row_idx_type, const int64_t* sel_g,
              const int64_t* sel_k, int64_t nsel, double* out, int nthreads) {
  if (!x || !dy || !expanded_row_idx || !group_list || !out) return kErrNull;
  if (dtype != kF32 && dtype != kF16 && dtype != kBF16) return kErrDtype;
  if (batch <= 0 || topK <= 0 || (row_idx_type != 0 && row_idx_type != 1)) return kErrAttr;
  if (M <= 0 || N <= 0 || K <= 0 || G <= 0) return kErrShape;
  if (M != batch * topK) return kErrShape;
  if ((sel_g == nullptr) != (sel_k == nullptr)) return kErrNull;
  if (!sel_g && nsel != G * K) return kErrShape;
  for (int64_t s = 0; sel_g && s < nsel; ++s)
    if (sel_g[s] < 0 || sel_g[s] >= G || sel_k[s] < 0 || sel_k[s] >= K) return kErrShape;

  Routing routing;
  const int rc = build_routing(expanded_row_idx, group_list, M, G, row_idx_type, &routing);
  if (rc != kOk) return rc;

  Decoder dec(dtype);
  DwJob job{x, dy, &dec, &routing, sel_g, sel_k, nsel, N, K, topK, out};
  run_pool(job, nsel, nthreads, run_dw_rows);
  return kOk;
}

}  // extern "C"
