// Row-wise bucketize ("ranged dispatch") into shard-major form.
// FreeScale (arXiv 2604.24073) §3.2 (batch-major vs shard-major ID forms),
// Algorithm 2 line 8 (IDs AllToAll to shard-major) and §4.2.
//
// Shard-major order is one stable counting-sort pass keyed by the shard of
// each ID (n digit values): per-tile shard counts, their scan, then a per-tile
// warp multisplit with shared-memory staging so that the writes of every shard
// run are coalesced.  The send-splits matrix is
// computed afterwards from the sorted positions (inside a shard they are
// ascending, so each (source rank, shard) count is two binary searches),
// which is the local recomputation of the AllToAll metadata.
#include "radix.cuh"

namespace fs {
namespace {

using radix::kThreads;

// shard(x) = x / block.  GB300's FP64 rate is a small fraction of its FP32
// rate, so the quotient is estimated in FP32 (exact to within one for any
// x < 2^32 and quotient < 2^12) and corrected with integer products.
struct SrcShard {
  using Key = int64_t;
  static constexpr bool kIndexValue = true;  // value = item index
  static constexpr bool kFetch2 = false;
  const int64_t* ids;
  int64_t R;
  int64_t block;
  float inv_block;
  int32_t n;
  using Raw = int64_t;
  template <bool>
  __device__ __forceinline__ Raw fetch(int64_t i) const { return __ldcs(ids + i); }
  __device__ __forceinline__ bool make(Raw id, int64_t i, int, Key& key, uint32_t& val, int32_t* err) const {
    key = id;
    val = static_cast<uint32_t>(i);
    if (err && (key < 0 || key >= R)) set_err(err, FS_ERR_ID_RANGE);
    return true;
  }
  __device__ __forceinline__ uint32_t digit(Key key, int, int, int) const {
    if (key <= 0) return 0;
    if (key >= R) return uint32_t(n - 1);
    int64_t q = static_cast<int64_t>(__float2uint_rz(__fmul_rz(__ull2float_rz(uint64_t(key)), inv_block)));
    if (q * block > key) --q;
    if ((q + 1) * block <= key) ++q;
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

size_t bucketize_bytes(int64_t T, int32_t n) { return radix::pass_ws_bytes(T, n); }

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
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T < 0 || T > INT32_MAX || n < 1 || n > radix::kMaxBins || num_rows < 1 || !rank_id_offsets || !splits ||
      !shard_offsets || !err)
    return FS_ERR_INVALID_ARG;
  if (T > 0 && (!ids || !sm_ids || !pos)) return FS_ERR_INVALID_ARG;
  if ((ids && !aligned(ids, 8)) || (sm_ids && !aligned(sm_ids, 8)) || (pos && !aligned(pos, 4)) ||
      !aligned(splits, 8) || !aligned(shard_offsets, 8) || !aligned(rank_id_offsets, 8))
    return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_bucketize_rowwise_workspace_size(T, n) || !ws) return FS_ERR_WORKSPACE;

  WsCursor cur(ws, ws_bytes);
  radix::PassWs P;
  if (!radix::carve_pass_ws(T, n, cur, P)) return FS_ERR_WORKSPACE;
  const int64_t block = (num_rows + n - 1) / n;
  SrcShard src{ids, num_rows, block, 1.0f / static_cast<float>(block), n};
  int launches = 0;
  if (T > 0) {
    radix::run_pass(src, DstShardMajor{sm_ids, pos}, 0, 0, n, nullptr, T, P, err, st, &launches);
  } else {
    if (cudaMemsetAsync(P.digit_base, 0, size_t(n) * sizeof(uint32_t), st) != cudaSuccess) return FS_ERR_CUDA;
  }
  shard_offsets_kernel<<<1, kThreads, 0, st>>>(P.digit_base, n, T, shard_offsets);
  int64_t nn = int64_t(n) * n;
  int64_t g = (nn + kThreads - 1) / kThreads;
  if (g > int64_t(sm_count()) * 8) g = int64_t(sm_count()) * 8;
  splits_kernel<<<unsigned(g < 1 ? 1 : g), kThreads, 0, st>>>(pos, shard_offsets, rank_id_offsets, n, T, splits, err);
  count_launch(launches + 2);
  return launch_status();
}
