// Shard of a row and the shard-major outputs of the row-wise bucketize
// ("ranged dispatch"): FreeScale §3.2 (batch-major and shard-major ID forms),
// Algorithm 2 line 8, §4.2.  Shared by fs_bucketize_rowwise and the fused
// permute + bucketize.
#pragma once

#include "radix.cuh"

namespace fs {
namespace shard {

// shard(x) = x / block.  GB300's FP64 rate is a small fraction of its FP32
// rate, so the quotient is estimated in FP32 (exact to within one for any
// x < 2^32 and quotient < 2^12) and corrected with integer products.
struct SrcShard {
  using Key = int64_t;
  static constexpr bool kIndexValue = true;  // value = item index
  // 56 KB of shared memory (int64 keys) leave room for 3 blocks per SM anyway:
  // the downsweep takes their register budget and spills nothing
  static constexpr int kMinBlocks = 3;
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

// The same source with the IDs staged as 32-bit rows, for tables of fewer
// than 2^32 rows: the staging takes half the shared memory and the keys half
// the registers, so the downsweep fits four blocks per SM instead of three.
// An ID outside [0, R) is staged as 0 (below) or R (at or above), which has
// the shard SrcShard gives the original ID (the counting pass may use either
// source); the call reports FS_ERR_ID_RANGE, and that entry's shard-major copy
// is then the clamped value.
struct SrcShard32 {
  using Key = uint32_t;
  static constexpr bool kIndexValue = true;  // value = item index
  static constexpr int kMinBlocks = 4;
  static constexpr bool kFetch2 = false;
  const int64_t* ids;
  int64_t R;  // < 2^32
  int64_t block;
  float inv_block;
  int32_t n;
  using Raw = int64_t;
  template <bool>
  __device__ __forceinline__ Raw fetch(int64_t i) const { return __ldcs(ids + i); }
  __device__ __forceinline__ bool make(Raw id, int64_t i, int, Key& key, uint32_t& val, int32_t* err) const {
    key = id < 0 ? 0u : (id >= R ? uint32_t(R) : uint32_t(id));
    val = static_cast<uint32_t>(i);
    if (err && (id < 0 || id >= R)) set_err(err, FS_ERR_ID_RANGE);
    return true;
  }
  __device__ __forceinline__ uint32_t digit(Key key, int, int, int) const {
    if (key == 0) return 0;
    if (int64_t(key) >= R) return uint32_t(n - 1);
    int64_t q = static_cast<int64_t>(__float2uint_rz(__fmul_rz(__uint2float_rz(key), inv_block)));
    if (q * block > int64_t(key)) --q;
    if ((q + 1) * block <= int64_t(key)) ++q;
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
  __device__ __forceinline__ void store(int64_t o, uint32_t key, uint32_t val) const {
    __stcs(sm_ids + o, int64_t(key));
    __stcs(pos + o, static_cast<int32_t>(val));
  }
};

// T_dev: the item count on the device (or null: T).
static __global__ void shard_offsets_kernel(const uint32_t* digit_offsets, int32_t n, int64_t T, const int64_t* T_dev,
                                            int64_t* shard_offsets) {
  const int64_t total = T_dev ? *T_dev : T;
  for (int s = threadIdx.x; s <= n; s += blockDim.x) shard_offsets[s] = (s == n) ? total : int64_t(digit_offsets[s]);
}

static __device__ __forceinline__ int64_t lower_bound_i32(const int32_t* a, int64_t lo, int64_t hi, int64_t x) {
  while (lo < hi) {
    int64_t mid = (lo + hi) >> 1;
    if (int64_t(a[mid]) < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// splits[r*n + s] = #{ j in shard s : rio[r] <= pos[j] < rio[r+1] }; validates rio.
// T_dev: the item count on the device (or null: T).
static __global__ void splits_kernel(const int32_t* pos, const int64_t* shard_offsets, const int64_t* rio, int32_t n,
                                     int64_t T_host, const int64_t* T_dev, int64_t* splits, int32_t* err) {
  const int64_t T = T_dev ? *T_dev : T_host;
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

}  // namespace shard
}  // namespace fs
