// Row-wise bucketize ("ranged dispatch") into shard-major form.
// FreeScale (arXiv 2604.24073) §3.2 (batch-major vs shard-major ID forms),
// Algorithm 2 line 8 (IDs AllToAll to shard-major) and §4.2.
//
// Shard-major order is one stable counting-sort pass keyed by the shard of
// each ID (one onesweep digit pass with n digit values): per-tile warp
// multisplit, decoupled look-back across tiles, shared-memory staging so that
// the writes of every shard run are coalesced.  The send-splits matrix is
// computed afterwards from the sorted positions (inside a shard they are
// ascending, so each (source rank, shard) count is two binary searches),
// which is the local recomputation of the AllToAll metadata.
#include "onesweep.cuh"

namespace fs {
namespace {

using onesweep::kThreads;

struct SrcShard {
  using Key = int64_t;
  static constexpr bool kIndexValue = true;  // value = item index
  const int64_t* ids;
  int64_t R;
  int64_t block;
  double inv_block;
  int32_t n;
  __device__ __forceinline__ bool load(int64_t i, Key& key, uint32_t& val, int32_t* err) const {
    key = __ldcs(ids + i);
    val = static_cast<uint32_t>(i);
    if (err && (key < 0 || key >= R)) set_err(err, FS_ERR_ID_RANGE);
    return true;
  }
  __device__ __forceinline__ uint32_t digit(Key key, int, int) const {
    if (key <= 0) return 0;
    if (key >= R) return uint32_t(n - 1);
    int64_t q = static_cast<int64_t>(static_cast<double>(key) * inv_block);
    if (q * block > key) --q;
    else if ((q + 1) * block <= key) ++q;
    return q >= n ? uint32_t(n - 1) : uint32_t(q);
  }
};

struct DstShardMajor {
  int64_t* sm_ids;
  int32_t* pos;
  __device__ __forceinline__ void store(int64_t o, int64_t key, uint32_t val) const {
    __stcs(sm_ids + o, key);
    __stcs(pos + o, static_cast<int32_t>(val));
  }
};

__global__ void shard_offsets_kernel(const uint32_t* digit_offsets, int32_t n, int64_t T, int64_t* shard_offsets) {
  for (int s = threadIdx.x; s <= n; s += blockDim.x) shard_offsets[s] = (s == n) ? T : int64_t(digit_offsets[s]);
}

__device__ __forceinline__ int64_t lower_bound_i32(const int32_t* a, int64_t lo, int64_t hi, int64_t x) {
  while (lo < hi) {
    int64_t mid = (lo + hi) >> 1;
    if (int64_t(a[mid]) < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// splits[r*n + s] = #{ j in shard s : rio[r] <= pos[j] < rio[r+1] }; validates rio.
__global__ void splits_kernel(const int32_t* pos, const int64_t* shard_offsets, const int64_t* rio, int32_t n,
                              int64_t T, int64_t* splits, int32_t* err) {
  const int64_t nn = int64_t(n) * n;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nn; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / n, s = i % n;
    int64_t a = rio[r], b = rio[r + 1];
    if (a < 0 || b < a || b > T || (r == 0 && a != 0) || (r == n - 1 && b != T)) {
      set_err(err, FS_ERR_BAD_OFFSETS);
      a = a < 0 ? 0 : (a > T ? T : a);
      b = b < a ? a : (b > T ? T : b);
    }
    const int64_t lo = shard_offsets[s], hi = shard_offsets[s + 1];
    splits[i] = lower_bound_i32(pos, lo, hi, b) - lower_bound_i32(pos, lo, hi, a);
  }
}

size_t bucketize_bytes(int64_t T, int32_t n) {
  const int64_t tiles = onesweep::num_tiles(T);
  return align_up(4 * onesweep::kMaxBins * sizeof(uint32_t)) + align_up(sizeof(int64_t) + 4 * sizeof(int)) +
         align_up(size_t(tiles) * size_t(n) * sizeof(uint64_t)) + align_up(4 * onesweep::kMaxBins * sizeof(uint32_t));
}

}  // namespace
}  // namespace fs

using namespace fs;

extern "C" size_t fs_bucketize_rowwise_workspace_size(int64_t T, int32_t n) {
  if (T < 0 || n < 1) return 0;
  return bucketize_bytes(T, n) + 256;
}

extern "C" fs_status fs_bucketize_rowwise(const int64_t* ids, int64_t T, const int64_t* rank_id_offsets, int32_t n,
                                          int64_t num_rows, int64_t* sm_ids, int32_t* pos, int64_t* splits,
                                          int64_t* shard_offsets, int32_t* err, void* ws, size_t ws_bytes,
                                          fs_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T < 0 || T > INT32_MAX || n < 1 || n > onesweep::kMaxBins || num_rows < 1 || !rank_id_offsets || !splits ||
      !shard_offsets || !err)
    return FS_ERR_INVALID_ARG;
  if (T > 0 && (!ids || !sm_ids || !pos)) return FS_ERR_INVALID_ARG;
  if ((ids && !aligned(ids, 8)) || (sm_ids && !aligned(sm_ids, 8)) || (pos && !aligned(pos, 4)) ||
      !aligned(splits, 8) || !aligned(shard_offsets, 8) || !aligned(rank_id_offsets, 8))
    return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_bucketize_rowwise_workspace_size(T, n) || !ws) return FS_ERR_WORKSPACE;

  const int64_t tiles = onesweep::num_tiles(T);
  WsCursor cur(ws, ws_bytes);
  const size_t zero_bytes = align_up(4 * onesweep::kMaxBins * sizeof(uint32_t)) +
                            align_up(sizeof(int64_t) + 4 * sizeof(int)) +
                            align_up(size_t(tiles) * size_t(n) * sizeof(uint64_t));
  unsigned char* zero = cur.take<unsigned char>(zero_bytes);
  uint32_t* offs = cur.take<uint32_t>(4 * onesweep::kMaxBins);
  if (!cur.ok) return FS_ERR_WORKSPACE;
  uint32_t* hist = reinterpret_cast<uint32_t*>(zero);
  unsigned char* p = zero + align_up(4 * onesweep::kMaxBins * sizeof(uint32_t));
  int64_t* n_valid = reinterpret_cast<int64_t*>(p);
  int* counter = reinterpret_cast<int*>(p + sizeof(int64_t));
  uint64_t* status = reinterpret_cast<uint64_t*>(p + align_up(sizeof(int64_t) + 4 * sizeof(int)));
  if (cudaMemsetAsync(zero, 0, zero_bytes, st) != cudaSuccess) return FS_ERR_CUDA;

  const int64_t block = (num_rows + n - 1) / n;
  SrcShard src{ids, num_rows, block, 1.0 / static_cast<double>(block), n};
  int launches = 0;
  if (T > 0) {
    int64_t hgrid = (T + kThreads - 1) / kThreads, hcap = int64_t(sm_count()) * 8;
    if (hgrid > hcap) hgrid = hcap;
    onesweep::histogram_kernel<SrcShard><<<unsigned(hgrid), kThreads, 0, st>>>(src, T, 1, 0, n, hist, n_valid, err);
    onesweep::digit_scan_kernel<<<1, kThreads, 0, st>>>(hist, offs, n);
    const size_t smem = onesweep::pass_smem_bytes<int64_t>();
    onesweep::set_pass_smem(onesweep::pass_kernel<SrcShard, DstShardMajor>, smem);
    onesweep::pass_kernel<SrcShard, DstShardMajor><<<unsigned(tiles), kThreads, smem, st>>>(
        src, DstShardMajor{sm_ids, pos}, 0, 0, n, offs, status, counter, nullptr, T, err, spin_limit());
    launches += 3;
  } else {
    if (cudaMemsetAsync(offs, 0, size_t(n) * sizeof(uint32_t), st) != cudaSuccess) return FS_ERR_CUDA;
  }
  shard_offsets_kernel<<<1, kThreads, 0, st>>>(offs, n, T, shard_offsets);
  int64_t nn = int64_t(n) * n;
  int64_t g = (nn + kThreads - 1) / kThreads;
  if (g > int64_t(sm_count()) * 8) g = int64_t(sm_count()) * 8;
  splits_kernel<<<unsigned(g < 1 ? 1 : g), kThreads, 0, st>>>(pos, shard_offsets, rank_id_offsets, n, T, splits, err);
  count_launch(launches + 2);
  return launch_status();
}
