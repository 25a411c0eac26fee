// Jagged sample permutation ("indexed permute").
// FreeScale (arXiv 2604.24073) §3.1 Algorithm 1 Stage III (shuffle the samples
// to the ranks the partition chose) and §4.2 (jagged kernels).  On one GPU
// the AllToAll of Stage III is this device-memory permutation.
//
// Kernel 1 (one pass over the S samples): permuted lengths, their exclusive
// scan (decoupled look-back) into out_offsets, the source start of each output
// sample, and for every 4096-ID output tile the first sample that covers it.
// Kernel 2 (one pass over the T IDs, ID-balanced): each block copies a fixed
// 4096-ID window of the output, whatever the sample lengths (a 16K-ID sample
// is spread over several blocks, so long samples do not straggle).
//
// The fused permute + bucketize (FreeScale §4.2: the indexed permute and the
// ranged dispatch that prepares the IDs AllToAll, Algorithm 2 line 8) copies
// the output tiles as kernel 2 does and, as it writes each tile, counts the
// tile's IDs per shard: that is the upsweep of the bucketize's counting pass,
// so the source IDs are read once and the permuted IDs once more by the
// bucketize's downsweep (no separate read pass over the permuted IDs).
//
// The keyed transpose (FreeScale §4.2: feature-major jagged tensors to
// batch-major) is the same permutation with the source segment computed
// instead of read: output segment b*F + f is input segment f*B + b; the copy
// may add a per-feature row base to every ID (features with their own tables
// stacked in one).
#include "shard.cuh"

namespace fs {
namespace {

constexpr int kThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kThreads * kScanItems;
constexpr int kCopyItems = 16;
constexpr int kCopyTile = kThreads * kCopyItems;  // output IDs per copy tile
constexpr int64_t kShortSample = 512;  // average IDs per sample below which the segment-parallel copy runs
constexpr int64_t kManySamples = 32;   // samples in one copy tile above which its warps copy whole samples

// Source segment of output segment k: read from an array ...
struct PermArray {
  const int32_t* perm;
  __device__ __forceinline__ int64_t operator()(int64_t k) const { return perm[k]; }
};
// ... or the keyed transpose's: k = b*F + f comes from f*B + b.
struct PermTranspose {
  int64_t F, B;
  __device__ __forceinline__ int64_t operator()(int64_t k) const { return (k % F) * B + k / F; }
};

template <class Perm>
__global__ void __launch_bounds__(kThreads) permute_scan_kernel(const int64_t* offsets, int64_t S, Perm perm,
                                                                int64_t* out_offsets, int64_t* src_start,
                                                                int32_t* first_sample, int64_t n_copy_tiles,
                                                                int64_t capacity, uint64_t* status, int* tile_counter,
                                                                int32_t* err, int64_t limit, int64_t skip_tile) {
  __shared__ int64_t tmp[32];
  __shared__ int64_t s_tile;
  __shared__ int64_t s_excl;
  if (threadIdx.x == 0) s_tile = atomicAdd(tile_counter, 1);
  __syncthreads();
  const int64_t tile = s_tile;
  const int64_t base = tile * kScanTile + int64_t(threadIdx.x) * kScanItems;
  const int64_t total_in = offsets[S];
  int64_t len[kScanItems], src[kScanItems];
  int64_t sum = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int64_t k = base + i;
    len[i] = 0;
    src[i] = 0;
    if (k < S) {
      int64_t g = perm(k);
      if (g < 0 || g >= S) {
        set_err(err, FS_ERR_BAD_OFFSETS);
      } else {
        int64_t a = offsets[g], b = offsets[g + 1];
        if (b < a || a < 0 || b > total_in) {
          set_err(err, FS_ERR_BAD_OFFSETS);
        } else {
          len[i] = b - a;
          src[i] = a;
        }
      }
    }
    sum += len[i];
  }
  int64_t tot;
  int64_t ex = block_exclusive_scan<int64_t>(sum, tmp, &tot);
  if (tile == skip_tile) return;  // test hook: this tile never publishes
  if (threadIdx.x < 32) {
    uint64_t e = warp_lookback(status, 1, tile, static_cast<uint64_t>(tot), err, limit);
    if (threadIdx.x == 0) s_excl = static_cast<int64_t>(e);
  }
  __syncthreads();
  int64_t run = s_excl + ex;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int64_t k = base + i;
    if (k < S) {
      out_offsets[k] = run;
      src_start[k] = src[i];
      if (len[i] > 0) {
        // output tiles whose first position falls inside this sample
        int64_t t0 = (run + kCopyTile - 1) / kCopyTile;
        int64_t t1 = (run + len[i] + kCopyTile - 1) / kCopyTile;
        if (t1 > n_copy_tiles) t1 = n_copy_tiles;
        for (int64_t t = t0; t < t1; ++t) first_sample[t] = static_cast<int32_t>(k);
      }
    }
    run += len[i];
    if (k == S - 1) {
      out_offsets[S] = run;
      if (run > capacity) set_err(err, FS_ERR_CAPACITY);
    }
  }
}

// kBase: row_base[F] is added to every ID of an output segment k, by its
// feature k % F (a separate instantiation: the plain permute keeps its
// 64-register footprint and four resident blocks per SM).
template <bool kBase>
__global__ void __launch_bounds__(kThreads) permute_copy_kernel(const int64_t* values, const int64_t* out_offsets,
                                                                const int64_t* src_start, const int32_t* first_sample,
                                                                int64_t S, int64_t capacity, int64_t* out_values,
                                                                const int64_t* rank_offsets, int32_t n,
                                                                int64_t* rank_id_offsets, int32_t* err,
                                                                const int64_t* row_base, int64_t F) {
  if (rank_offsets && blockIdx.x == 0) {
    for (int r = threadIdx.x; r <= n; r += blockDim.x) {
      int64_t q = rank_offsets[r];
      bool bad = q < 0 || q > S || (r > 0 && rank_offsets[r - 1] > q) || (r == 0 && q != 0) || (r == n && q != S);
      if (bad) set_err(err, FS_ERR_BAD_OFFSETS);
      rank_id_offsets[r] = out_offsets[bad ? (q < 0 ? 0 : (q > S ? S : q)) : q];
    }
  }
  int64_t total = out_offsets[S];
  if (total > capacity) total = capacity;
  const int64_t ntiles = (total + kCopyTile - 1) / kCopyTile;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t j0 = t * kCopyTile;
    int64_t k = first_sample[t];
    int64_t k_hi = (t + 1 < ntiles) ? int64_t(first_sample[t + 1]) : S - 1;  // last sample touching this tile
    if (k_hi - k > kManySamples) {
      // a tile of many short samples: each warp copies whole samples (clipped
      // to the tile) instead of searching the sample of every ID
      const int64_t j1 = (j0 + kCopyTile < total) ? j0 + kCopyTile : total;
      const int lane = threadIdx.x & 31;
      for (int64_t kk = k + (threadIdx.x >> 5); kk <= k_hi; kk += kThreads / 32) {
        const int64_t d = __ldg(out_offsets + kk), e = __ldg(out_offsets + kk + 1);
        const int64_t a = d > j0 ? d : j0, z = e < j1 ? e : j1;
        if (a >= z) continue;
        const int64_t src = __ldg(src_start + kk) + (a - d);
        const int64_t add = kBase ? __ldg(row_base + kk % F) : 0;
        for (int64_t j = a + lane; j < z; j += 32) __stcs(out_values + j, __ldcs(values + src + (j - a)) + add);
      }
      continue;
    }
    int64_t srcidx[kCopyItems];
    int64_t base[kBase ? kCopyItems : 1];
#pragma unroll
    for (int i = 0; i < kCopyItems; ++i) {
      const int64_t j = j0 + int64_t(i) * kThreads + threadIdx.x;
      srcidx[i] = -1;
      if constexpr (kBase) base[i] = 0;
      if (j < total) {
        // largest k' in [k, k_hi] with out_offsets[k'] <= j
        int64_t lo = k, hi = k_hi;
        while (lo < hi) {
          int64_t mid = (lo + hi + 1) >> 1;
          if (__ldg(out_offsets + mid) <= j) lo = mid; else hi = mid - 1;
        }
        k = lo;
        srcidx[i] = __ldg(src_start + k) + (j - __ldg(out_offsets + k));
        if constexpr (kBase) base[i] = __ldg(row_base + k % F);
      }
    }
    int64_t v[kCopyItems];
#pragma unroll
    for (int i = 0; i < kCopyItems; ++i) {
      v[i] = srcidx[i] >= 0 ? __ldcs(values + srcidx[i]) : 0;
      if constexpr (kBase) v[i] += base[i];
    }
#pragma unroll
    for (int i = 0; i < kCopyItems; ++i) {
      const int64_t j = j0 + int64_t(i) * kThreads + threadIdx.x;
      if (srcidx[i] >= 0) __stcs(out_values + j, v[i]);
    }
  }
}

// Copy for short samples (segment-parallel): a warp takes groups of 32
// consecutive output samples, lane l loads sample l's destination, end,
// source and row base, then the warp copies the samples one after another,
// four IDs per lane in flight.  Writes stop at `capacity` (the scan reports
// the overflow).
constexpr int kSegUnroll = 4;
template <bool kBase>
__global__ void __launch_bounds__(kThreads) permute_seg_copy_kernel(const int64_t* values, const int64_t* out_offsets,
                                                                    const int64_t* src_start, int64_t S,
                                                                    int64_t capacity, int64_t* out_values,
                                                                    const int64_t* row_base, int64_t F) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t ngroups = (S + 31) / 32;
  for (int64_t grp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; grp < ngroups; grp += nwarps) {
    const int64_t k = grp * 32 + lane;
    int64_t d = 0, e = 0, sr = 0, b = 0;
    if (k < S) {
      d = __ldg(out_offsets + k);
      e = __ldg(out_offsets + k + 1);
      sr = __ldg(src_start + k);
      if constexpr (kBase) b = __ldg(row_base + k % F);
    }
    if (e > capacity) e = capacity;
    for (int q = 0; q < 32; ++q) {
      const int64_t dq = __shfl_sync(0xffffffffu, d, q), eq = __shfl_sync(0xffffffffu, e, q);
      const int64_t sq = __shfl_sync(0xffffffffu, sr, q);
      const int64_t bq = kBase ? __shfl_sync(0xffffffffu, b, q) : 0;
      for (int64_t j0 = dq; j0 < eq; j0 += 32 * kSegUnroll) {
        int64_t v[kSegUnroll];
#pragma unroll
        for (int u = 0; u < kSegUnroll; ++u) {
          const int64_t j = j0 + u * 32 + lane;
          v[u] = j < eq ? __ldcs(values + sq + (j - dq)) : 0;
        }
#pragma unroll
        for (int u = 0; u < kSegUnroll; ++u) {
          const int64_t j = j0 + u * 32 + lane;
          if (j < eq) __stcs(out_values + j, v[u] + bq);
        }
      }
    }
  }
}

// Fused permute + bucketize, kernel 2: blocks take chunks of
// 1 << cshift consecutive output tiles (the counting pass's chunk size) (kCopyTile == radix::kTile IDs
// each) and copy them like permute_copy_kernel; every ID written is counted
// in its shard's bin, giving the counting pass's counts[tile][shard] (exclusive
// within the chunk) and chunk_sums[chunk][shard].  Tiles past the output (up
// to ntiles_cap, the capacity's tiles) count nothing.  *T_out = the number of
// IDs written, min(out_offsets[S], capacity).
static_assert(kCopyTile == radix::kTile, "a copy tile is a counting tile");
__global__ void __launch_bounds__(kThreads) permute_count_kernel(
    const int64_t* values, const int64_t* out_offsets, const int64_t* src_start, const int32_t* first_sample,
    int64_t S, int64_t capacity, int64_t* out_values, const int64_t* rank_offsets, int32_t n, int64_t* rank_id_offsets,
    int32_t* err, shard::SrcShard sh, uint32_t* counts, uint32_t* chunk_sums, int64_t ntiles_cap, int cshift,
    int64_t* T_out) {
  __shared__ uint32_t hist[radix::kMaxBins];
  const int nb = sh.n;
  if (blockIdx.x == 0) {
    for (int r = threadIdx.x; r <= n; r += blockDim.x) {
      int64_t q = rank_offsets[r];
      bool bad = q < 0 || q > S || (r > 0 && rank_offsets[r - 1] > q) || (r == 0 && q != 0) || (r == n && q != S);
      if (bad) set_err(err, FS_ERR_BAD_OFFSETS);
      rank_id_offsets[r] = out_offsets[bad ? (q < 0 ? 0 : (q > S ? S : q)) : q];
    }
  }
  int64_t total = out_offsets[S];
  if (total > capacity) total = capacity;
  if (blockIdx.x == 0 && threadIdx.x == 0) *T_out = total;
  const int64_t ntiles = (total + kCopyTile - 1) / kCopyTile;
  // one ID written at output position j: store it, flag it if out of range, count its shard
  auto put = [&](int64_t j, int64_t v) {
    __stcs(out_values + j, v);
    if (v < 0 || v >= sh.R) set_err(err, FS_ERR_ID_RANGE);
    atomicAdd(hist + sh.digit(v, 0, 0, 0), 1u);
  };
  uint32_t run[radix::kPerT];
#pragma unroll
  for (int q = 0; q < radix::kPerT; ++q) run[q] = 0;
  for (int c = 0; c < (1 << cshift); ++c) {
    const int64_t t = (int64_t(blockIdx.x) << cshift) + c;
    if (t >= ntiles_cap) break;
    for (int d = threadIdx.x; d < nb; d += kThreads) hist[d] = 0;
    __syncthreads();
    if (t < ntiles) {
      const int64_t j0 = t * kCopyTile;
      int64_t k = first_sample[t];
      const int64_t k_hi = (t + 1 < ntiles) ? int64_t(first_sample[t + 1]) : S - 1;
      if (k_hi - k > kManySamples) {
        // many short samples: each warp copies whole samples, clipped to the tile
        const int64_t j1 = (j0 + kCopyTile < total) ? j0 + kCopyTile : total;
        const int lane = threadIdx.x & 31;
        for (int64_t kk = k + (threadIdx.x >> 5); kk <= k_hi; kk += kThreads / 32) {
          const int64_t d = __ldg(out_offsets + kk), e = __ldg(out_offsets + kk + 1);
          const int64_t a = d > j0 ? d : j0, z = e < j1 ? e : j1;
          if (a >= z) continue;
          const int64_t src = __ldg(src_start + kk) + (a - d);
          for (int64_t j = a + lane; j < z; j += 32) put(j, __ldcs(values + src + (j - a)));
        }
      } else {
        int64_t srcidx[kCopyItems];
#pragma unroll
        for (int i = 0; i < kCopyItems; ++i) {
          const int64_t j = j0 + int64_t(i) * kThreads + threadIdx.x;
          srcidx[i] = -1;
          if (j < total) {
            int64_t lo = k, hi = k_hi;  // largest k' in [k, k_hi] with out_offsets[k'] <= j
            while (lo < hi) {
              const int64_t mid = (lo + hi + 1) >> 1;
              if (__ldg(out_offsets + mid) <= j) lo = mid; else hi = mid - 1;
            }
            k = lo;
            srcidx[i] = __ldg(src_start + k) + (j - __ldg(out_offsets + k));
          }
        }
        int64_t v[kCopyItems];
#pragma unroll
        for (int i = 0; i < kCopyItems; ++i) v[i] = srcidx[i] >= 0 ? __ldcs(values + srcidx[i]) : 0;
#pragma unroll
        for (int i = 0; i < kCopyItems; ++i)
          if (srcidx[i] >= 0) put(j0 + int64_t(i) * kThreads + threadIdx.x, v[i]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < radix::kPerT; ++q) {
      const int d = threadIdx.x + q * kThreads;
      if (d < nb) {
        counts[t * nb + d] = run[q];
        run[q] += hist[d];
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int q = 0; q < radix::kPerT; ++q) {
    const int d = threadIdx.x + q * kThreads;
    if (d < nb) chunk_sums[int64_t(blockIdx.x) * nb + d] = run[q];
  }
}

__global__ void permute_empty_kernel(int64_t* out_offsets, const int64_t* rank_offsets, int32_t n,
                                     int64_t* rank_id_offsets, int32_t* err) {
  if (threadIdx.x == 0) out_offsets[0] = 0;
  if (rank_offsets)
    for (int r = threadIdx.x; r <= n; r += blockDim.x) {
      if (rank_offsets[r] != 0) set_err(err, FS_ERR_BAD_OFFSETS);
      rank_id_offsets[r] = 0;
    }
}

struct PermuteLayout {
  int64_t scan_tiles, copy_tiles;
  size_t zero_bytes() const { return align_up(size_t(scan_tiles) * sizeof(uint64_t) + 256); }
};

PermuteLayout layout(int64_t S, int64_t capacity) {
  PermuteLayout L;
  L.scan_tiles = (S + kScanTile - 1) / kScanTile;
  L.copy_tiles = (capacity + kCopyTile - 1) / kCopyTile;
  return L;
}

}  // namespace
}  // namespace fs

using namespace fs;

// The copy-tile map depends on the output capacity; the query assumes the
// worst case of one tile per 4096 IDs of a capacity up to 2^31.
extern "C" size_t fs_permute_jagged_workspace_size(int64_t S) {
  if (S < 0) return 0;
  PermuteLayout L = layout(S, int64_t(INT32_MAX));
  return L.zero_bytes() + align_up(size_t(S) * sizeof(int64_t)) + align_up(size_t(L.copy_tiles + 1) * sizeof(int32_t)) +
         256;
}

namespace fs {
namespace {

// Both calls: scan (with the permutation source P) then copy.
template <class Perm>
fs_status permute_launch(const int64_t* offsets, const int64_t* values, int64_t S, Perm P, int64_t* out_offsets,
                         int64_t* out_values, int64_t capacity, const int64_t* rank_offsets, int32_t n,
                         int64_t* rank_id_offsets, const int64_t* row_base, int64_t F, int32_t* err, void* ws,
                         size_t ws_bytes, cudaStream_t st) {
  if (S == 0) {
    permute_empty_kernel<<<1, kThreads, 0, st>>>(out_offsets, rank_offsets, n, rank_id_offsets, err);
    count_launch(1);
    return launch_status();
  }
  PermuteLayout L = layout(S, capacity);
  WsCursor cur(ws, ws_bytes);
  unsigned char* zero = cur.take<unsigned char>(L.zero_bytes());
  int64_t* src_start = cur.take<int64_t>(size_t(S));
  int32_t* first_sample = cur.take<int32_t>(size_t(L.copy_tiles + 1));
  if (!cur.ok) return FS_ERR_WORKSPACE;
  if (cudaMemsetAsync(zero, 0, L.zero_bytes(), st) != cudaSuccess) return FS_ERR_CUDA;
  int* counter = reinterpret_cast<int*>(zero);
  uint64_t* status = reinterpret_cast<uint64_t*>(zero + 256);
  permute_scan_kernel<Perm><<<unsigned(L.scan_tiles), kThreads, 0, st>>>(offsets, S, P, out_offsets, src_start,
                                                                         first_sample, L.copy_tiles, capacity, status,
                                                                         counter, err, spin_limit(), debug_skip_tile());
  int64_t grid = L.copy_tiles;
  int64_t cap = int64_t(sm_count()) * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  if (!rank_offsets && capacity <= kShortSample * S) {
    // short samples on average: one warp per group of 32 samples, no per-ID search
    auto copy = row_base ? permute_seg_copy_kernel<true> : permute_seg_copy_kernel<false>;
    copy<<<unsigned(cap), kThreads, 0, st>>>(values, out_offsets, src_start, S, capacity, out_values, row_base, F);
  } else {
    auto copy = row_base ? permute_copy_kernel<true> : permute_copy_kernel<false>;
    copy<<<unsigned(grid), kThreads, 0, st>>>(values, out_offsets, src_start, first_sample, S, capacity, out_values,
                                              rank_offsets, n, rank_id_offsets, err, row_base, F);
  }
  count_launch(2);
  return launch_status();
}

}  // namespace
}  // namespace fs

extern "C" fs_status fs_permute_jagged(const int64_t* offsets, const int64_t* values, int64_t S, const int32_t* perm,
                                       int64_t* out_offsets, int64_t* out_values, int64_t capacity,
                                       const int64_t* rank_offsets, int32_t n, int64_t* rank_id_offsets,
                                       int32_t* err, void* ws, size_t ws_bytes, fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (S < 0 || S > INT32_MAX || capacity < 0 || capacity > INT32_MAX || !out_offsets || !err)
    return FS_ERR_INVALID_ARG;
  if (S > 0 && (!offsets || !perm)) return FS_ERR_INVALID_ARG;
  if (capacity > 0 && (!values || !out_values)) return FS_ERR_INVALID_ARG;
  if (rank_offsets && (n < 1 || !rank_id_offsets)) return FS_ERR_INVALID_ARG;
  if (!aligned(out_offsets, 8) || (S > 0 && !aligned(offsets, 8)) || (out_values && !aligned(out_values, 8)) ||
      (values && !aligned(values, 8)))
    return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_permute_jagged_workspace_size(S) || !ws) return FS_ERR_WORKSPACE;
  return permute_launch(offsets, values, S, PermArray{perm}, out_offsets, out_values, capacity, rank_offsets, n,
                        rank_id_offsets, nullptr, 1, err, ws, ws_bytes, st);
}

namespace fs {
namespace {

// Workspace of the fused call: the permute's (scan status, source starts, tile
// map for `capacity` output IDs), the counting pass's for as many IDs, and the
// number of IDs written.
template <class Ws>
void take_prep_ws(int64_t S, int64_t capacity, int32_t n, Ws& ws, unsigned char** zero, int64_t** src_start,
                  int32_t** first_sample, radix::PassWs* P, int64_t** T_out) {
  const PermuteLayout L = layout(S, capacity);
  *zero = ws.template take<unsigned char>(L.zero_bytes());
  *src_start = ws.template take<int64_t>(size_t(S));
  *first_sample = ws.template take<int32_t>(size_t(L.copy_tiles + 1));
  P->ntiles = radix::num_tiles(capacity > 0 ? capacity : 1);  // at least one (empty) tile
  P->counts = ws.template take<uint32_t>(size_t(n) * size_t(P->ntiles));
  P->chunk = ws.template take<uint32_t>(size_t(n) * size_t(radix::num_chunks(P->ntiles)));
  P->totals = ws.template take<uint32_t>(radix::kMaxBins);
  P->digit_base = ws.template take<uint32_t>(radix::kMaxBins);
  P->n_valid = ws.template take<int64_t>(1);
  *T_out = ws.template take<int64_t>(1);
}

}  // namespace
}  // namespace fs

extern "C" size_t fs_permute_bucketize_workspace_size(int64_t S, int64_t capacity, int32_t n) {
  if (S < 0 || capacity < 0 || n < 1 || n > radix::kMaxBins) return 0;
  WsCounter c;
  unsigned char* z;
  int64_t *ss, *to;
  int32_t* fs;
  radix::PassWs P;
  take_prep_ws(S, capacity, n, c, &z, &ss, &fs, &P, &to);
  return c.used + 256;
}

extern "C" fs_status fs_permute_bucketize(const int64_t* offsets, const int64_t* values, int64_t S, const int32_t* perm,
                                          const int64_t* rank_offsets, int32_t n, int64_t num_rows,
                                          int64_t* out_offsets, int64_t* out_values, int64_t capacity,
                                          int64_t* rank_id_offsets, int64_t* sm_ids, int32_t* pos, int64_t* splits,
                                          int64_t* shard_offsets, int32_t* err, void* ws, size_t ws_bytes,
                                          fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (S < 0 || S > INT32_MAX || capacity < 0 || capacity > INT32_MAX || n < 1 || n > radix::kMaxBins ||
      num_rows < 1 || !out_offsets || !rank_offsets || !rank_id_offsets || !splits || !shard_offsets || !err)
    return FS_ERR_INVALID_ARG;
  if (S > 0 && (!offsets || !perm)) return FS_ERR_INVALID_ARG;
  if (capacity > 0 && (!values || !out_values || !sm_ids || !pos)) return FS_ERR_INVALID_ARG;
  if (!aligned(out_offsets, 8) || (S > 0 && !aligned(offsets, 8)) || (out_values && !aligned(out_values, 8)) ||
      (values && !aligned(values, 8)) || !aligned(rank_offsets, 8) || !aligned(rank_id_offsets, 8) ||
      (sm_ids && !aligned(sm_ids, 8)) || (pos && !aligned(pos, 4)) || !aligned(splits, 8) ||
      !aligned(shard_offsets, 8))
    return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_permute_bucketize_workspace_size(S, capacity, n) || !ws) return FS_ERR_WORKSPACE;
  WsCursor cur(ws, ws_bytes);
  unsigned char* zero;
  int64_t *src_start, *T_out;
  int32_t* first_sample;
  radix::PassWs P;
  take_prep_ws(S, capacity, n, cur, &zero, &src_start, &first_sample, &P, &T_out);
  if (!cur.ok) return FS_ERR_WORKSPACE;
  const PermuteLayout L = layout(S, capacity);
  const int64_t block = (num_rows + n - 1) / n;
  const shard::SrcShard sh{out_values, num_rows, block, 1.0f / static_cast<float>(block), n};
  int launches = 0;
  if (S == 0) {
    // no samples: empty outputs (rank_offsets must be all zero)
    permute_empty_kernel<<<1, kThreads, 0, st>>>(out_offsets, rank_offsets, n, rank_id_offsets, err);
    if (cudaMemsetAsync(P.digit_base, 0, size_t(n) * sizeof(uint32_t), st) != cudaSuccess) return FS_ERR_CUDA;
    if (cudaMemsetAsync(T_out, 0, sizeof(int64_t), st) != cudaSuccess) return FS_ERR_CUDA;
    launches = 1;
  } else {
    if (cudaMemsetAsync(zero, 0, L.zero_bytes(), st) != cudaSuccess) return FS_ERR_CUDA;
    permute_scan_kernel<PermArray><<<unsigned(L.scan_tiles), kThreads, 0, st>>>(
        offsets, S, PermArray{perm}, out_offsets, src_start, first_sample, L.copy_tiles, capacity,
        reinterpret_cast<uint64_t*>(zero + 256), reinterpret_cast<int*>(zero), err, spin_limit(), debug_skip_tile());
    const int64_t nchunks = radix::num_chunks(P.ntiles);
    const int cs = radix::chunk_shift(P.ntiles);
    permute_count_kernel<<<unsigned(nchunks), kThreads, 0, st>>>(values, out_offsets, src_start, first_sample, S,
                                                                 capacity, out_values, rank_offsets, n,
                                                                 rank_id_offsets, err, sh, P.counts, P.chunk,
                                                                 P.ntiles, cs, T_out);
    radix::chunk_scan_kernel<<<unsigned((n + 31) / 32), radix::kScanThreads, 0, st>>>(P.chunk, nchunks, n, P.totals);
    radix::digit_base_kernel<<<1, radix::kThreads, 0, st>>>(P.totals, n, P.digit_base, P.n_valid);
    const radix::PlainTiles tiles{T_out, 0, P.digit_base};
    if (num_rows < (int64_t(1) << 32)) {  // rows fit 32 bits: the lighter staging (same shard of every ID)
      const shard::SrcShard32 sh32{out_values, num_rows, block, sh.inv_block, n};
      const size_t smem = radix::downsweep_smem_bytes<uint32_t>();
      auto down = radix::downsweep_kernel<shard::SrcShard32, shard::DstShardMajor, radix::PlainTiles>;
      radix::set_smem(down, smem);
      down<<<unsigned(P.ntiles), radix::kDownThreads, smem, st>>>(sh32, shard::DstShardMajor{sm_ids, pos}, tiles, 0, 0,
                                                                  n, P.counts, P.chunk, cs);
    } else {
      const size_t smem = radix::downsweep_smem_bytes<int64_t>();
      auto down = radix::downsweep_kernel<shard::SrcShard, shard::DstShardMajor, radix::PlainTiles>;
      radix::set_smem(down, smem);
      down<<<unsigned(P.ntiles), radix::kDownThreads, smem, st>>>(sh, shard::DstShardMajor{sm_ids, pos}, tiles, 0, 0, n,
                                                              P.counts, P.chunk, cs);
    }
    launches = 5;
  }
  shard::shard_offsets_kernel<<<1, kThreads, 0, st>>>(P.digit_base, n, 0, T_out, shard_offsets);
  int64_t g = (int64_t(n) * n + kThreads - 1) / kThreads;
  if (g > int64_t(sm_count()) * 8) g = int64_t(sm_count()) * 8;
  shard::splits_kernel<<<unsigned(g < 1 ? 1 : g), kThreads, 0, st>>>(pos, shard_offsets, rank_id_offsets, n, 0, T_out,
                                                                     splits, err);
  count_launch(launches + 2);
  return launch_status();
}

extern "C" size_t fs_keyed_transpose_workspace_size(int64_t F, int64_t B) {
  if (F < 1 || B < 0 || F * B > INT32_MAX) return 0;
  return fs_permute_jagged_workspace_size(F * B);
}

extern "C" fs_status fs_keyed_transpose(const int64_t* offsets, const int64_t* values, int64_t F, int64_t B,
                                        const int64_t* row_base, int64_t* out_offsets, int64_t* out_values,
                                        int64_t capacity, int32_t* err, void* ws, size_t ws_bytes,
                                        fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (F < 1 || B < 0 || F * B > INT32_MAX || capacity < 0 || capacity > INT32_MAX || !out_offsets || !err)
    return FS_ERR_INVALID_ARG;
  const int64_t S = F * B;
  if (S > 0 && !offsets) return FS_ERR_INVALID_ARG;
  if (capacity > 0 && (!values || !out_values)) return FS_ERR_INVALID_ARG;
  if (!aligned(out_offsets, 8) || (S > 0 && !aligned(offsets, 8)) || (out_values && !aligned(out_values, 8)) ||
      (values && !aligned(values, 8)) || (row_base && !aligned(row_base, 8)))
    return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_keyed_transpose_workspace_size(F, B) || !ws) return FS_ERR_WORKSPACE;
  return permute_launch(offsets, values, S, PermTranspose{F, B}, out_offsets, out_values, capacity, nullptr, 0,
                        nullptr, row_base, F, err, ws, ws_bytes, st);
}
