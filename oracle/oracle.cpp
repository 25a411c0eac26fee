// CPU oracle for the FreeScale jagged index + embedding hot path.
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
// benchmark's CPU-baseline / reference arm may load this library.  It shares
// no code, header, table or constant with the CUDA library; it is plain,
// C++17 written from the definitions on the pages:
//
//   FreeScale: Distributed Training for Sequence Recommendation Models with
//   Minimal Scaling Cost (arXiv 2604.24073), referred to below as "FreeScale".
//
// Every function states the passage it follows.  Accumulations are in fp64.
// Each step is the plain definition of its result (sorts are std:: library
// sorts, sets are std:: set algorithms) except FBS and VBS, which are
// heuristics and are written out step by step.  These functions are
// single-threaded.  At the end of the file, *_mt variants of the steps whose
// work splits into independent pieces (samples, positions, rows) compute the
// same results on several host threads; they exist only to time the oracle
// on every core of the host, and the CPU tests prove them identical to the
// single-threaded functions.
//
// Return value of every entry point: 0 = ok, 1 = invalid argument,
// 2 = an ID outside [0, R), 3 = malformed offsets / permutation.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <numeric>
#include <thread>
#include <vector>

namespace {

typedef unsigned __int128 u128;

// bf16 <-> double.  bf16 is the upper half of an IEEE binary32.
double bf16_to_double(uint16_t h) {
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// Round a double to the nearest bf16, ties to even, in ONE rounding step:
// write |x| = m * 2^e with m in [0.5, 1), round m * 2^8 (exact in double) to
// an integer with nearbyint (default mode = to nearest, ties to even), and
// rebuild.  Values below the bf16 normal range go through binary32 first.
uint16_t double_to_bf16(double x) {
  if (std::isnan(x)) return 0x7fc0;
  if (x == 0.0) return std::signbit(x) ? 0x8000 : 0x0000;
  double ax = std::fabs(x);
  float f;
  if (ax < 1.1754943508222875e-38) {
    f = static_cast<float>(x);
  } else {
    int e = 0;
    double m = std::frexp(ax, &e);            // ax = m * 2^e, 0.5 <= m < 1
    double r = std::nearbyint(std::ldexp(m, 8));  // 128 <= r <= 256
    double v = std::ldexp(r, e - 8);
    f = static_cast<float>(x < 0 ? -v : v);   // exact: v has <= 8 significant bits
  }
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return static_cast<uint16_t>(u >> 16);
}

double read_elem(const void* base, int64_t idx, int dtype) {
  if (dtype == 0) return static_cast<double>(static_cast<const float*>(base)[idx]);
  return bf16_to_double(static_cast<const uint16_t*>(base)[idx]);
}

void write_elem(void* base, int64_t idx, int dtype, double v) {
  if (dtype == 0) {
    static_cast<float*>(base)[idx] = static_cast<float>(v);  // one RNE rounding
  } else {
    static_cast<uint16_t*>(base)[idx] = double_to_bf16(v);
  }
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// FBS partition.  FreeScale §4.1 "Partitioning Algorithms", FBS paragraph:
// sort all samples by UIH length, then deal them to the ranks zig-zag so that
// every rank gets the same number of samples.
//
// Readings (the printed index list [i, 2n-i, 2n+i, 4n-i, ...] is off by one
// in both 0- and 1-based forms):
//  * sort ascending by L, ties broken by the global index g (deterministic P,
//    FreeScale §3.1 / Algorithm 1);
//  * sorted position p lies in round rho = p / n at place k = p % n; rounds
//    alternate direction: rank = k in even rounds, n-1-k in odd rounds
//    (boustrophedon / snake);
//  * a rank lists its samples in round order;
//  * when n does not divide S the last, partial round is dealt the same way.
// Output: perm[new position] = g; rank_offsets[r] = first new position of r.
int oracle_balance_fbs(const int32_t* L, int64_t S, int32_t n, int32_t* perm, int64_t* rank_offsets) {
  if (n <= 0 || S < 0) return 1;
  for (int64_t g = 0; g < S; ++g)
    if (L[g] < 0) return 1;
  std::vector<int64_t> order(S);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) { return L[a] < L[b]; });

  std::vector<std::vector<int64_t>> mine(n);
  for (int64_t p = 0; p < S; ++p) {
    int64_t rho = p / n, k = p % n;
    int64_t r = (rho % 2 == 0) ? k : (n - 1 - k);
    mine[r].push_back(order[p]);
  }
  int64_t at = 0;
  rank_offsets[0] = 0;
  for (int32_t r = 0; r < n; ++r) {
    for (int64_t g : mine[r]) perm[at++] = static_cast<int32_t>(g);
    rank_offsets[r + 1] = at;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// VBS sample weight.  FreeScale §4.1, VBS paragraph: weight L^alpha.
// Reading: the weight is kept in fixed point, w = round_half_even(L^alpha * 2^8)
// as an unsigned 64-bit integer, so that prefix sums are exact and do not
// depend on summation order.  L^alpha is evaluated with IEEE-exact operations
// where the exponent allows it (alpha = 0.5, 1, 1.5, 2, 2.5, 3: a product of L's
// and at most one correctly rounded sqrt), otherwise with pow().
uint64_t oracle_vbs_weight(int32_t L, double alpha) {
  double x = static_cast<double>(L);
  double p;
  if (alpha == 1.0) {
    p = x;
  } else if (alpha == 1.5) {
    p = x * std::sqrt(x);
  } else if (alpha == 2.0) {
    p = x * x;
  } else if (alpha == 0.5) {
    p = std::sqrt(x);
  } else if (alpha == 2.5) {
    p = (x * x) * std::sqrt(x);
  } else if (alpha == 3.0) {
    p = (x * x) * x;
  } else {
    p = std::pow(x, alpha);
  }
  return static_cast<uint64_t>(std::nearbyint(p * 256.0));
}

// VBS partition.  FreeScale §4.1, VBS paragraph: the (globally sorted)
// samples are cut into n segments of approximately equal total weight; ranks
// may receive different numbers of samples.
// Readings:
//  * sort_by_len = 1 cuts the order sorted by (L, g) ascending, as the page
//    says; sort_by_len = 0 cuts the original rank-major order.
//  * cut rule: with P_j the exclusive prefix of the weights along the order
//    and W the total, sample j goes to rank min(n-1, floor(n * P_j / W)).
//    Segments are contiguous, may be empty, and the heaviest one weighs at
//    most W/n + max_j w_j.
//  * W == 0 (every weight zero) falls back to equal counts: rank
//    min(n-1, floor(n * j / S)).
// Output: perm = the cut order, rank_offsets[n+1], seg_weight[n].
int oracle_balance_vbs(const int32_t* L, int64_t S, int32_t n, double alpha, int32_t sort_by_len,
                       int32_t* perm, int64_t* rank_offsets, uint64_t* seg_weight) {
  if (n <= 0 || S < 0 || !(alpha >= 0.0)) return 1;
  for (int64_t g = 0; g < S; ++g)
    if (L[g] < 0) return 1;
  std::vector<int64_t> order(S);
  std::iota(order.begin(), order.end(), 0);
  if (sort_by_len)
    std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) { return L[a] < L[b]; });

  std::vector<uint64_t> w(S);
  u128 W = 0;
  for (int64_t j = 0; j < S; ++j) {
    w[j] = oracle_vbs_weight(L[order[j]], alpha);
    W += w[j];
  }
  if (W >> 64) return 1;  // total weight must fit 64 bits

  std::vector<int64_t> count(n, 0);
  for (int32_t r = 0; r < n; ++r) seg_weight[r] = 0;
  u128 P = 0;
  for (int64_t j = 0; j < S; ++j) {
    int64_t r;
    if (W == 0) {
      r = static_cast<int64_t>((static_cast<u128>(j) * static_cast<u128>(n)) / static_cast<u128>(S));
    } else {
      r = static_cast<int64_t>((P * static_cast<u128>(n)) / W);
    }
    if (r > n - 1) r = n - 1;
    count[r] += 1;
    seg_weight[r] += w[j];
    P += w[j];
    perm[j] = static_cast<int32_t>(order[j]);
  }
  rank_offsets[0] = 0;
  for (int32_t r = 0; r < n; ++r) rank_offsets[r + 1] = rank_offsets[r] + count[r];
  return 0;
}

// VBS AutoTune, the update.  FreeScale §4.1, VBS paragraph (and the AutoTune
// module of Figure 4): because L^alpha need not match the model's real
// execution time, each rank's local batch size is raised or lowered according
// to how its local execution time compares with the global average.
// Readings:
//  * the tuned quantity is a per-rank correction delta[r] (samples) to the
//    batch size the weight cut gives; it starts at 0 and persists across
//    iterations;
//  * times are integers (e.g. nanoseconds, 0 <= t < 2^53), so the comparison
//    with the average is exact: rank r is slow when t_r > avg * (1 + tol) and
//    fast when t_r < avg * (1 - tol), tol = tol_ppm / 10^6 (0 = the plain
//    comparison), evaluated as n * 10^6 * t_r against (10^6 +- tol_ppm) * sum t;
//  * the global batch is fixed (the AllGather of Algorithm 1 collects n * B
//    samples), so decrements and increments come in pairs: with k =
//    min(#slow, #fast), the k slowest ranks (time descending, lower rank first
//    on ties) lose `step` samples and the k fastest (time ascending, lower rank
//    first on ties) gain `step`; the sum of delta does not change.
int oracle_vbs_autotune(const int64_t* t, int32_t n, int64_t step, int32_t tol_ppm, int64_t* delta) {
  if (n <= 0 || step < 0 || tol_ppm < 0 || tol_ppm > 1000000) return 1;
  u128 sum = 0;
  for (int32_t r = 0; r < n; ++r) {
    if (t[r] < 0 || t[r] >= (int64_t(1) << 53)) return 1;
    sum += static_cast<u128>(t[r]);
  }
  const u128 scale = static_cast<u128>(n) * 1000000u;
  const u128 hi = sum * static_cast<u128>(1000000 + tol_ppm);
  const u128 lo = sum * static_cast<u128>(1000000 - tol_ppm);
  std::vector<int32_t> slow, fast;
  for (int32_t r = 0; r < n; ++r) {
    const u128 x = static_cast<u128>(t[r]) * scale;
    if (x > hi) slow.push_back(r);
    if (x < lo) fast.push_back(r);
  }
  std::stable_sort(slow.begin(), slow.end(), [&](int32_t a, int32_t b) { return t[a] > t[b]; });
  std::stable_sort(fast.begin(), fast.end(), [&](int32_t a, int32_t b) { return t[a] < t[b]; });
  const size_t k = std::min(slow.size(), fast.size());
  for (size_t i = 0; i < k; ++i) {
    delta[slow[i]] -= step;
    delta[fast[i]] += step;
  }
  return 0;
}

// VBS with the AutoTune correction applied.  FreeScale §4.1, VBS paragraph.
// Steps: (1) the VBS cut above gives the order and the segment ends
// e_r = rank_offsets[r+1]; (2) rank r's batch changes by delta[r], i.e. every
// segment end moves by D_r = delta[0] + ... + delta[r], the segments staying
// contiguous along the same order; (3) a correction larger than a segment can
// give cannot make a count negative: the moved ends are clamped to [0, S] and
// then made non-decreasing (each end is the largest of the ends up to it);
// (4) seg_weight is the weight of the adjusted segments.  Whenever no clamp
// acts, rank r holds exactly (its cut count + delta[r]) samples.
// delta must sum to 0 (the global batch is fixed) and |delta[r]| <= S.
int oracle_balance_vbs_tuned(const int32_t* L, int64_t S, int32_t n, double alpha, int32_t sort_by_len,
                             const int64_t* delta, int32_t* perm, int64_t* rank_offsets, uint64_t* seg_weight) {
  if (n <= 0 || S < 0) return 1;
  int64_t total = 0;
  for (int32_t r = 0; r < n; ++r) {
    if (delta[r] > S || delta[r] < -S) return 1;
    total += delta[r];
  }
  if (total != 0) return 1;
  int rc = oracle_balance_vbs(L, S, n, alpha, sort_by_len, perm, rank_offsets, seg_weight);
  if (rc != 0) return rc;
  int64_t D = 0, run_max = 0;
  for (int32_t r = 0; r < n; ++r) {
    D += delta[r];
    int64_t e = rank_offsets[r + 1] + D;
    e = std::min<int64_t>(std::max<int64_t>(e, 0), S);
    run_max = std::max(run_max, e);
    rank_offsets[r + 1] = run_max;
  }
  for (int32_t r = 0; r < n; ++r) {
    uint64_t sw = 0;
    for (int64_t j = rank_offsets[r]; j < rank_offsets[r + 1]; ++j) sw += oracle_vbs_weight(L[perm[j]], alpha);
    seg_weight[r] = sw;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Jagged sample permutation ("indexed permute").  FreeScale §3.1 Algorithm 1,
// Stage III (shuffle samples to match the partition) and §4.2: output sample k
// is input sample perm[k], with all of its IDs ([UIH | candidates]).
int oracle_permute_jagged(const int64_t* offsets, const int64_t* values, int64_t S, const int32_t* perm,
                          int64_t* out_offsets, int64_t* out_values) {
  if (S < 0) return 1;
  for (int64_t g = 0; g < S; ++g)
    if (offsets[g + 1] < offsets[g]) return 3;
  for (int64_t k = 0; k < S; ++k)
    if (perm[k] < 0 || perm[k] >= S) return 3;
  int64_t at = 0;
  out_offsets[0] = 0;
  for (int64_t k = 0; k < S; ++k) {
    int64_t g = perm[k];
    for (int64_t i = offsets[g]; i < offsets[g + 1]; ++i) out_values[at++] = values[i];
    out_offsets[k + 1] = at;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Keyed transpose.  FreeScale §4.2: jagged tensors go from the feature-major
// form (all samples of feature 0, then all samples of feature 1, ...) to the
// batch-major form (all features of sample 0, then of sample 1, ...).  Walk
// the samples b, and for each the features f, appending feature f's IDs of
// sample b (input segment f*B + b); with row_base, feature f's IDs are shifted
// by row_base[f] (rows of feature f's own table inside a stacked table).
int oracle_keyed_transpose(const int64_t* offsets, const int64_t* values, int64_t F, int64_t B,
                           const int64_t* row_base, int64_t* out_offsets, int64_t* out_values) {
  if (F < 1 || B < 0) return 1;
  for (int64_t s = 0; s < F * B; ++s)
    if (offsets[s + 1] < offsets[s]) return 3;
  int64_t at = 0;
  out_offsets[0] = 0;
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t f = 0; f < F; ++f) {
      const int64_t seg = f * B + b;
      const int64_t shift = row_base ? row_base[f] : 0;
      for (int64_t i = offsets[seg]; i < offsets[seg + 1]; ++i) out_values[at++] = values[i] + shift;
      out_offsets[b * F + f + 1] = at;
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Row-wise bucketize ("ranged dispatch").  FreeScale §3.2 (batch-major vs
// shard-major forms), Algorithm 2 line 8 (IDs AllToAll to shard-major), §4.2.
// The table is row-wise sharded into n contiguous ranges of block = ceil(R/n)
// rows (the last range is short when n does not divide R); an ID belongs to
// shard id / block.  Shard-major order is a stable sort of the batch-major
// positions by shard, so inside a shard IDs keep (source rank, position)
// order.  pos[j] is the batch-major position of shard-major entry j;
// splits[r*n + s] counts IDs of source rank r (the batch-major range
// [rank_id_offsets[r], rank_id_offsets[r+1])) that fall into shard s.
int oracle_bucketize_rowwise(const int64_t* ids, int64_t T, const int64_t* rank_id_offsets, int32_t n, int64_t R,
                             int64_t* sm_ids, int32_t* pos, int64_t* splits, int64_t* shard_offsets) {
  if (n <= 0 || R <= 0 || T < 0) return 1;
  if (rank_id_offsets[0] != 0 || rank_id_offsets[n] != T) return 3;
  for (int32_t r = 0; r < n; ++r)
    if (rank_id_offsets[r + 1] < rank_id_offsets[r]) return 3;
  for (int64_t p = 0; p < T; ++p)
    if (ids[p] < 0 || ids[p] >= R) return 2;
  const int64_t block = (R + n - 1) / n;
  std::vector<int64_t> shard(T);
  for (int64_t p = 0; p < T; ++p) shard[p] = ids[p] / block;

  std::vector<int64_t> order(T);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) { return shard[a] < shard[b]; });
  for (int64_t j = 0; j < T; ++j) {
    sm_ids[j] = ids[order[j]];
    pos[j] = static_cast<int32_t>(order[j]);
  }

  for (int64_t i = 0; i < static_cast<int64_t>(n) * n; ++i) splits[i] = 0;
  std::vector<int64_t> per_shard(n, 0);
  for (int32_t r = 0; r < n; ++r)
    for (int64_t p = rank_id_offsets[r]; p < rank_id_offsets[r + 1]; ++p) {
      splits[static_cast<int64_t>(r) * n + shard[p]] += 1;
      per_shard[shard[p]] += 1;
    }
  shard_offsets[0] = 0;
  for (int32_t s = 0; s < n; ++s) shard_offsets[s + 1] = shard_offsets[s] + per_shard[s];
  return 0;
}

// ---------------------------------------------------------------------------
// Collision / exclusive split.  FreeScale Algorithm 2 line 10
// (compute_collision on the shard-major I^i and I^{i+1}) and the notation
// paragraph after Algorithm 2: collision rows are rows of iteration i that are
// also used by iteration i+1; exclusive rows are used by one of the two only.
// Readings: collisions are counted on rows (sets), not positions; each list is
// ascending by row, which is shard-major because shards are row ranges.
//   co      = uniq(ids_t) intersect uniq(ids_next)
//   ex_t    = uniq(ids_t)    minus uniq(ids_next)
//   ex_next = uniq(ids_next) minus uniq(ids_t)
// counts = {|co|, |ex_t|, |ex_next|}; *_shard_off[k] = number of list rows
// below k * block (k = 0..n, the last one = list length).  Masks are aligned
// with the input arrays: is_co_t[j] = ids_t[j] is a collision row,
// is_co_next[j] = ids_next[j] is a collision row.  Capacity: each list holds
// at most cap_rows entries (return 1 when exceeded).
int oracle_collision_split(const int64_t* ids_t, int64_t T_t, const int64_t* ids_next, int64_t T_next, int64_t R,
                           int32_t n, int64_t* co, int64_t* ex_t, int64_t* ex_next, int64_t cap_rows,
                           int64_t* counts, int64_t* co_off, int64_t* ex_t_off, int64_t* ex_next_off,
                           uint8_t* is_co_t, uint8_t* is_co_next) {
  if (n <= 0 || R <= 0 || T_t < 0 || T_next < 0) return 1;
  for (int64_t j = 0; j < T_t; ++j)
    if (ids_t[j] < 0 || ids_t[j] >= R) return 2;
  for (int64_t j = 0; j < T_next; ++j)
    if (ids_next[j] < 0 || ids_next[j] >= R) return 2;

  std::vector<int64_t> A(ids_t, ids_t + T_t), B(ids_next, ids_next + T_next);
  std::sort(A.begin(), A.end());
  A.erase(std::unique(A.begin(), A.end()), A.end());
  std::sort(B.begin(), B.end());
  B.erase(std::unique(B.begin(), B.end()), B.end());

  std::vector<int64_t> vco, vext, vexn;
  std::set_intersection(A.begin(), A.end(), B.begin(), B.end(), std::back_inserter(vco));
  std::set_difference(A.begin(), A.end(), B.begin(), B.end(), std::back_inserter(vext));
  std::set_difference(B.begin(), B.end(), A.begin(), A.end(), std::back_inserter(vexn));
  if (static_cast<int64_t>(vco.size()) > cap_rows || static_cast<int64_t>(vext.size()) > cap_rows ||
      static_cast<int64_t>(vexn.size()) > cap_rows)
    return 1;
  std::copy(vco.begin(), vco.end(), co);
  std::copy(vext.begin(), vext.end(), ex_t);
  std::copy(vexn.begin(), vexn.end(), ex_next);
  counts[0] = static_cast<int64_t>(vco.size());
  counts[1] = static_cast<int64_t>(vext.size());
  counts[2] = static_cast<int64_t>(vexn.size());

  const int64_t block = (R + n - 1) / n;
  const std::vector<int64_t>* lists[3] = {&vco, &vext, &vexn};
  int64_t* offs[3] = {co_off, ex_t_off, ex_next_off};
  for (int l = 0; l < 3; ++l)
    for (int32_t k = 0; k <= n; ++k) {
      int64_t bound = static_cast<int64_t>(k) * block;
      offs[l][k] = std::lower_bound(lists[l]->begin(), lists[l]->end(), bound) - lists[l]->begin();
    }

  for (int64_t j = 0; j < T_t; ++j) is_co_t[j] = std::binary_search(B.begin(), B.end(), ids_t[j]) ? 1 : 0;
  for (int64_t j = 0; j < T_next; ++j) is_co_next[j] = std::binary_search(A.begin(), A.end(), ids_next[j]) ? 1 : 0;
  return 0;
}

// ---------------------------------------------------------------------------
// Embedding gather (lookup + ranged combine + merge).  FreeScale Algorithm 2
// line 12 (Lookup, then embeddings back to batch-major) and line 15 (merge of
// exclusive and collision embeddings into one batch); §2.1 (an ID list is
// turned into a sequence of embeddings: no pooling).
// out[p] = table[ids[p]] as a byte copy of one row (row_bytes bytes).  With a
// mask, only positions whose mask byte equals sel are written; the others are
// left untouched.
int oracle_emb_gather(const void* table, int64_t R, int64_t row_bytes, const int64_t* ids, int64_t T,
                      const uint8_t* mask, uint8_t sel, void* out) {
  if (R < 0 || row_bytes <= 0 || T < 0) return 1;
  const unsigned char* tb = static_cast<const unsigned char*>(table);
  unsigned char* ob = static_cast<unsigned char*>(out);
  for (int64_t p = 0; p < T; ++p) {
    if (mask && mask[p] != sel) continue;
    if (ids[p] < 0 || ids[p] >= R) return 2;
    std::memcpy(ob + p * row_bytes, tb + ids[p] * row_bytes, static_cast<size_t>(row_bytes));
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Embedding backward: gradient segment-reduce per row, then a row update.
// FreeScale Algorithm 2 lines 7 and 20 (update_embedding on exclusive and on
// collision rows), line 18 (split of the gradients into collision and
// exclusive parts) and the paragraph after it: collision rows are updated
// first so that iteration i+1 reads their new values.
//
// The pages name no optimizer.  Readings:
//  * g_r = sum over the positions p with ids[p] = r (selected by phase) of
//    grads[p], in fp64, in position order;
//  * optim 0 = SGD:               W_r <- W_r - lr * g_r;
//  * optim 1 = row-wise Adagrad:  s_r <- s_r + (1/D) sum_d g_{r,d}^2,
//                                 W_r <- W_r - lr * g_r / (sqrt(s_r) + eps),
//    (Duchi, Hazan & Singer 2011, one accumulator per row, zero initial
//    state, eps outside the square root, no weight decay);
//  * arithmetic in fp64, each result rounded once: state to binary32, weights
//    to binary32 (dtype 0) or to bfloat16 ties-to-even (dtype 1);
//  * phase 0 = every position, 1 = positions with is_co[p] == 1 (collision
//    rows), 2 = positions with is_co[p] == 0 (exclusive rows).  Collision is a
//    property of the row, so the two phases touch disjoint row sets and every
//    row of the batch is updated exactly once over the two.
// If g_out / rows_out are given, the fp64 sums g_r and their rows are written
// in ascending row order and *n_rows_out receives the number of rows.
int oracle_emb_backward(void* table, float* state, int64_t R, int32_t D, int32_t dtype, int32_t optim,
                        const int64_t* ids, const void* grads, int64_t T, const uint8_t* is_co, int32_t phase,
                        double lr, double eps, double* g_out, int64_t* rows_out, int64_t* n_rows_out) {
  if (R < 0 || D <= 0 || T < 0 || (dtype != 0 && dtype != 1) || (optim != 0 && optim != 1)) return 1;
  if (phase < 0 || phase > 2 || (phase != 0 && is_co == nullptr) || (optim == 1 && state == nullptr)) return 1;

  std::map<int64_t, std::vector<int64_t>> positions;  // row -> its positions, ascending
  for (int64_t p = 0; p < T; ++p) {
    if (phase == 1 && is_co[p] != 1) continue;
    if (phase == 2 && is_co[p] != 0) continue;
    if (ids[p] < 0 || ids[p] >= R) return 2;
    positions[ids[p]].push_back(p);
  }

  std::vector<double> g(D);
  int64_t u = 0;
  for (const auto& kv : positions) {
    const int64_t r = kv.first;
    std::fill(g.begin(), g.end(), 0.0);
    for (int64_t p : kv.second)
      for (int32_t d = 0; d < D; ++d) g[d] += read_elem(grads, p * D + d, dtype);

    if (optim == 0) {
      for (int32_t d = 0; d < D; ++d) {
        double w = read_elem(table, r * D + d, dtype);
        write_elem(table, r * D + d, dtype, w - lr * g[d]);
      }
    } else {
      double sq = 0.0;
      for (int32_t d = 0; d < D; ++d) sq += g[d] * g[d];
      double s = static_cast<double>(state[r]) + sq / static_cast<double>(D);
      state[r] = static_cast<float>(s);
      double denom = std::sqrt(s) + eps;
      for (int32_t d = 0; d < D; ++d) {
        double w = read_elem(table, r * D + d, dtype);
        write_elem(table, r * D + d, dtype, w - lr * g[d] / denom);
      }
    }
    if (g_out) {
      for (int32_t d = 0; d < D; ++d) g_out[u * D + d] = g[d];
    }
    if (rows_out) rows_out[u] = r;
    ++u;
  }
  if (n_rows_out) *n_rows_out = u;
  return 0;
}

// Helpers the tests use to read and write single bf16 values.
double oracle_bf16_to_double(uint16_t h) { return bf16_to_double(h); }
uint16_t oracle_double_to_bf16(double x) { return double_to_bf16(x); }

}  // extern "C"

// ===========================================================================
// Multi-threaded variants (for timing the oracle on all host cores).  Each
// computes exactly what the single-threaded function of the same name
// computes, with the work split into independent pieces: samples for the
// permute, positions for the gather and the masks, rows for the collision
// sets and the update.  Invalid inputs give the same return code; the outputs
// are then unspecified (the single-threaded functions may have written part
// of them, these check everything before writing).
// ===========================================================================
namespace {

// Run f(k, lo, hi) on `threads` threads over contiguous pieces of [0, n).
template <class F>
void parallel_ranges(int64_t n, int threads, F f) {
  if (threads < 1) threads = 1;
  if (n < 1) return;
  if (threads > n) threads = static_cast<int>(n);
  std::vector<std::thread> pool;
  for (int k = 0; k < threads; ++k) {
    int64_t lo = n * k / threads, hi = n * (k + 1) / threads;
    pool.emplace_back([=]() { f(k, lo, hi); });
  }
  for (auto& t : pool) t.join();
}

// Sort v on `threads` threads: each sorts one piece, then neighbouring pieces
// are merged pairwise, round after round.
template <class T>
void parallel_sort(std::vector<T>& v, int threads) {
  const int64_t n = static_cast<int64_t>(v.size());
  if (threads < 2 || n < 2) {
    std::sort(v.begin(), v.end());
    return;
  }
  if (threads > n) threads = static_cast<int>(n);
  std::vector<int64_t> cut(threads + 1);
  for (int k = 0; k <= threads; ++k) cut[k] = n * k / threads;
  parallel_ranges(threads, threads, [&](int, int64_t lo, int64_t hi) {
    for (int64_t k = lo; k < hi; ++k) std::sort(v.begin() + cut[k], v.begin() + cut[k + 1]);
  });
  for (int width = 1; width < threads; width *= 2) {
    std::vector<std::thread> pool;
    for (int k = 0; k + width < threads; k += 2 * width) {
      const int64_t a = cut[k], m = cut[k + width], b = cut[std::min(k + 2 * width, threads)];
      pool.emplace_back([&v, a, m, b]() { std::inplace_merge(v.begin() + a, v.begin() + m, v.begin() + b); });
    }
    for (auto& t : pool) t.join();
  }
}

}  // namespace

extern "C" {

// oracle_permute_jagged on several threads: the output offsets are the same
// prefix of the permuted lengths; the samples are then copied in pieces.
int oracle_permute_jagged_mt(const int64_t* offsets, const int64_t* values, int64_t S, const int32_t* perm,
                             int64_t* out_offsets, int64_t* out_values, int32_t threads) {
  if (S < 0) return 1;
  for (int64_t g = 0; g < S; ++g)
    if (offsets[g + 1] < offsets[g]) return 3;
  for (int64_t k = 0; k < S; ++k)
    if (perm[k] < 0 || perm[k] >= S) return 3;
  out_offsets[0] = 0;
  for (int64_t k = 0; k < S; ++k) out_offsets[k + 1] = out_offsets[k] + (offsets[perm[k] + 1] - offsets[perm[k]]);
  parallel_ranges(S, threads, [&](int, int64_t lo, int64_t hi) {
    for (int64_t k = lo; k < hi; ++k) {
      const int64_t g = perm[k];
      std::copy(values + offsets[g], values + offsets[g + 1], out_values + out_offsets[k]);
    }
  });
  return 0;
}

// oracle_bucketize_rowwise on several threads.  A stable sort by shard is a
// counting sort: each thread counts the shards of one contiguous range of
// positions; the start of (shard s, thread k) is the number of positions in
// shards below s plus those of shard s in the ranges of threads below k; each
// thread then writes its range in position order.
int oracle_bucketize_rowwise_mt(const int64_t* ids, int64_t T, const int64_t* rank_id_offsets, int32_t n, int64_t R,
                                int64_t* sm_ids, int32_t* pos, int64_t* splits, int64_t* shard_offsets,
                                int32_t threads) {
  if (n <= 0 || R <= 0 || T < 0) return 1;
  if (rank_id_offsets[0] != 0 || rank_id_offsets[n] != T) return 3;
  for (int32_t r = 0; r < n; ++r)
    if (rank_id_offsets[r + 1] < rank_id_offsets[r]) return 3;
  for (int64_t p = 0; p < T; ++p)
    if (ids[p] < 0 || ids[p] >= R) return 2;
  const int64_t block = (R + n - 1) / n;
  if (threads < 1) threads = 1;
  if (T > 0 && threads > T) threads = static_cast<int>(T);
  std::vector<std::vector<int64_t>> cnt(threads, std::vector<int64_t>(n, 0));
  parallel_ranges(T, threads, [&](int k, int64_t lo, int64_t hi) {
    for (int64_t p = lo; p < hi; ++p) cnt[k][ids[p] / block] += 1;
  });
  std::vector<std::vector<int64_t>> start(threads, std::vector<int64_t>(n, 0));
  int64_t at = 0;
  for (int32_t s = 0; s < n; ++s) {
    shard_offsets[s] = at;
    for (int k = 0; k < threads; ++k) {
      start[k][s] = at;
      at += cnt[k][s];
    }
  }
  shard_offsets[n] = at;
  parallel_ranges(T, threads, [&](int k, int64_t lo, int64_t hi) {
    std::vector<int64_t>& next = start[k];
    for (int64_t p = lo; p < hi; ++p) {
      const int64_t j = next[ids[p] / block]++;
      sm_ids[j] = ids[p];
      pos[j] = static_cast<int32_t>(p);
    }
  });
  for (int64_t i = 0; i < static_cast<int64_t>(n) * n; ++i) splits[i] = 0;
  parallel_ranges(n, threads, [&](int, int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r)
      for (int64_t p = rank_id_offsets[r]; p < rank_id_offsets[r + 1]; ++p) splits[r * n + ids[p] / block] += 1;
  });
  return 0;
}

// oracle_collision_split on several threads, through presence arrays over the
// rows instead of sorted unique lists: rows of t and of t+1 are marked (one
// byte per row), the three lists are the rows present in both, in t only and
// in t+1 only, in ascending order (each thread takes a range of rows, counts,
// then writes at the prefix of the counts), and the masks look rows up.
int oracle_collision_split_mt(const int64_t* ids_t, int64_t T_t, const int64_t* ids_next, int64_t T_next, int64_t R,
                              int32_t n, int64_t* co, int64_t* ex_t, int64_t* ex_next, int64_t cap_rows,
                              int64_t* counts, int64_t* co_off, int64_t* ex_t_off, int64_t* ex_next_off,
                              uint8_t* is_co_t, uint8_t* is_co_next, int32_t threads) {
  if (n <= 0 || R <= 0 || T_t < 0 || T_next < 0) return 1;
  for (int64_t j = 0; j < T_t; ++j)
    if (ids_t[j] < 0 || ids_t[j] >= R) return 2;
  for (int64_t j = 0; j < T_next; ++j)
    if (ids_next[j] < 0 || ids_next[j] >= R) return 2;
  if (threads < 1) threads = 1;
  // marks: every writer stores the same value 1, through relaxed atomics
  std::vector<std::atomic<uint8_t>> in_t(R), in_n(R);
  parallel_ranges(R, threads, [&](int, int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      in_t[r].store(0, std::memory_order_relaxed);
      in_n[r].store(0, std::memory_order_relaxed);
    }
  });
  parallel_ranges(T_t, threads, [&](int, int64_t lo, int64_t hi) {
    for (int64_t j = lo; j < hi; ++j) in_t[ids_t[j]].store(1, std::memory_order_relaxed);
  });
  parallel_ranges(T_next, threads, [&](int, int64_t lo, int64_t hi) {
    for (int64_t j = lo; j < hi; ++j) in_n[ids_next[j]].store(1, std::memory_order_relaxed);
  });
  const int pieces = static_cast<int>(std::min<int64_t>(threads, R));
  std::vector<int64_t> c[3];
  for (int l = 0; l < 3; ++l) c[l].assign(pieces + 1, 0);
  auto kind = [&](int64_t r) -> int {
    const bool a = in_t[r].load(std::memory_order_relaxed), b = in_n[r].load(std::memory_order_relaxed);
    return a && b ? 0 : (a ? 1 : (b ? 2 : -1));
  };
  parallel_ranges(R, pieces, [&](int k, int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r) {
      const int l = kind(r);
      if (l >= 0) c[l][k + 1] += 1;
    }
  });
  for (int l = 0; l < 3; ++l)
    for (int k = 0; k < pieces; ++k) c[l][k + 1] += c[l][k];
  for (int l = 0; l < 3; ++l) {
    counts[l] = c[l][pieces];
    if (counts[l] > cap_rows) return 1;
  }
  int64_t* lists[3] = {co, ex_t, ex_next};
  parallel_ranges(R, pieces, [&](int k, int64_t lo, int64_t hi) {
    int64_t at[3] = {c[0][k], c[1][k], c[2][k]};
    for (int64_t r = lo; r < hi; ++r) {
      const int l = kind(r);
      if (l >= 0) lists[l][at[l]++] = r;
    }
  });
  const int64_t block = (R + n - 1) / n;
  int64_t* offs[3] = {co_off, ex_t_off, ex_next_off};
  for (int l = 0; l < 3; ++l)
    for (int32_t k = 0; k <= n; ++k)
      offs[l][k] = std::lower_bound(lists[l], lists[l] + counts[l], static_cast<int64_t>(k) * block) - lists[l];
  parallel_ranges(T_t, threads, [&](int, int64_t lo, int64_t hi) {
    for (int64_t j = lo; j < hi; ++j) is_co_t[j] = in_n[ids_t[j]].load(std::memory_order_relaxed);
  });
  parallel_ranges(T_next, threads, [&](int, int64_t lo, int64_t hi) {
    for (int64_t j = lo; j < hi; ++j) is_co_next[j] = in_t[ids_next[j]].load(std::memory_order_relaxed);
  });
  return 0;
}

// oracle_emb_gather on several threads: positions in pieces.
int oracle_emb_gather_mt(const void* table, int64_t R, int64_t row_bytes, const int64_t* ids, int64_t T,
                         const uint8_t* mask, uint8_t sel, void* out, int32_t threads) {
  if (R < 0 || row_bytes <= 0 || T < 0) return 1;
  for (int64_t p = 0; p < T; ++p)
    if ((!mask || mask[p] == sel) && (ids[p] < 0 || ids[p] >= R)) return 2;
  const unsigned char* tb = static_cast<const unsigned char*>(table);
  unsigned char* ob = static_cast<unsigned char*>(out);
  parallel_ranges(T, threads, [&](int, int64_t lo, int64_t hi) {
    for (int64_t p = lo; p < hi; ++p) {
      if (mask && mask[p] != sel) continue;
      std::memcpy(ob + p * row_bytes, tb + ids[p] * row_bytes, static_cast<size_t>(row_bytes));
    }
  });
  return 0;
}

// oracle_emb_backward on several threads.  The selected (row, position)
// pairs are sorted (on all threads), so each row's positions are adjacent and
// ascending; the rows are then cut into pieces, and each thread sums and
// updates whole rows exactly as the single-threaded function does: fp64 sums
// in position order, one rounding per stored value.
int oracle_emb_backward_mt(void* table, float* state, int64_t R, int32_t D, int32_t dtype, int32_t optim,
                           const int64_t* ids, const void* grads, int64_t T, const uint8_t* is_co, int32_t phase,
                           double lr, double eps, int32_t threads) {
  if (R < 0 || D <= 0 || T < 0 || (dtype != 0 && dtype != 1) || (optim != 0 && optim != 1)) return 1;
  if (phase < 0 || phase > 2 || (phase != 0 && is_co == nullptr) || (optim == 1 && state == nullptr)) return 1;
  std::vector<std::pair<int64_t, int64_t>> e;  // (row, position)
  e.reserve(static_cast<size_t>(T));
  for (int64_t p = 0; p < T; ++p) {
    if (phase == 1 && is_co[p] != 1) continue;
    if (phase == 2 && is_co[p] != 0) continue;
    if (ids[p] < 0 || ids[p] >= R) return 2;
    e.emplace_back(ids[p], p);
  }
  parallel_sort(e, threads);
  // row starts, then pieces of whole rows
  std::vector<int64_t> starts;
  for (int64_t i = 0; i < static_cast<int64_t>(e.size()); ++i)
    if (i == 0 || e[i].first != e[i - 1].first) starts.push_back(i);
  const int64_t U = static_cast<int64_t>(starts.size());
  starts.push_back(static_cast<int64_t>(e.size()));
  parallel_ranges(U, threads, [&](int, int64_t lo, int64_t hi) {
    std::vector<double> g(D);
    for (int64_t u = lo; u < hi; ++u) {
      const int64_t r = e[starts[u]].first;
      std::fill(g.begin(), g.end(), 0.0);
      for (int64_t i = starts[u]; i < starts[u + 1]; ++i)
        for (int32_t d = 0; d < D; ++d) g[d] += read_elem(grads, e[i].second * D + d, dtype);
      if (optim == 0) {
        for (int32_t d = 0; d < D; ++d) {
          double w = read_elem(table, r * D + d, dtype);
          write_elem(table, r * D + d, dtype, w - lr * g[d]);
        }
      } else {
        double sq = 0.0;
        for (int32_t d = 0; d < D; ++d) sq += g[d] * g[d];
        double s = static_cast<double>(state[r]) + sq / static_cast<double>(D);
        state[r] = static_cast<float>(s);
        double denom = std::sqrt(s) + eps;
        for (int32_t d = 0; d < D; ++d) {
          double w = read_elem(table, r * D + d, dtype);
          write_elem(table, r * D + d, dtype, w - lr * g[d] / denom);
        }
      }
    }
  });
  return 0;
}

}  // extern "C"
