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
#include "shard.cuh"

namespace fs {
namespace {

using radix::kThreads;
using shard::DstShardMajor;
using shard::SrcShard;

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
  int launches = 0;
  if (T > 0) {
    if (num_rows < (int64_t(1) << 32)) {  // rows fit 32 bits: the lighter staging
      const shard::SrcShard32 src{ids, num_rows, block, 1.0f / static_cast<float>(block), n};
      radix::run_pass(src, DstShardMajor{sm_ids, pos}, 0, 0, n, nullptr, T, P, err, st, &launches);
    } else {
      const SrcShard src{ids, num_rows, block, 1.0f / static_cast<float>(block), n};
      radix::run_pass(src, DstShardMajor{sm_ids, pos}, 0, 0, n, nullptr, T, P, err, st, &launches);
    }
  } else {
    if (cudaMemsetAsync(P.digit_base, 0, size_t(n) * sizeof(uint32_t), st) != cudaSuccess) return FS_ERR_CUDA;
  }
  shard::shard_offsets_kernel<<<1, kThreads, 0, st>>>(P.digit_base, n, T, nullptr, shard_offsets);
  int64_t nn = int64_t(n) * n;
  int64_t g = (nn + kThreads - 1) / kThreads;
  if (g > int64_t(sm_count()) * 8) g = int64_t(sm_count()) * 8;
  shard::splits_kernel<<<unsigned(g < 1 ? 1 : g), kThreads, 0, st>>>(pos, shard_offsets, rank_id_offsets, n, T, nullptr,
                                                                     splits, err);
  count_launch(launches + 2);
  return launch_status();
}
