// Embedding row gather into batch-major jagged output.
// FreeScale (arXiv 2604.24073) Algorithm 2 line 12 (Lookup, then the
// embeddings go back to batch-major: the ranged combine is fused here, each
// row lands directly at its batch-major position), line 15 (merge of the
// prefetched exclusive rows and the collision rows: two masked calls into one
// output buffer) and §2.1 (sequence embeddings, no pooling).
//
// Bandwidth layout: the output (T x row bytes) is written once and never
// re-read here, so it is written evict-first; table rows are read so that hot
// (Zipf head) rows stay cached.  Unmasked calls (the whole output is written)
// go through the copy engine: gather_bulk_kernel below.  Masked calls, which
// must leave unselected rows untouched, use register loads: a lane moves one
// 16-byte vector of a row, lanes of a warp cover consecutive vectors (a
// 256-byte row is 16 lanes, one warp instruction moves two rows) and each
// lane keeps 8 independent vectors in flight.
#include "bulk.cuh"
#include "fs_common.cuh"

namespace fs {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;

// Row bytes = 16 * VPR with VPR in {4, 8, 16, 32}: a warp instruction moves
// RPI = 32 / VPR whole rows (lanes [k*VPR, (k+1)*VPR) own row k), and a warp
// iteration moves RPI * U consecutive rows whose IDs (and mask bytes) one
// coalesced load brings in and shuffles out; no per-element division, U
// independent 16-byte loads in flight per lane.
template <int VPR>
__global__ void __launch_bounds__(kThreads) gather_rows_kernel(const int4* __restrict__ table, int64_t R,
                                                               const int64_t* __restrict__ ids, int64_t T,
                                                               const uint8_t* __restrict__ mask, uint8_t sel,
                                                               int4* __restrict__ out, int32_t* err) {
  constexpr int RPI = 32 / VPR;                              // rows per warp instruction
  constexpr int U = (32 / RPI) < kUnroll ? (32 / RPI) : kUnroll;
  constexpr int RPW = RPI * U;                               // rows per warp iteration, one ID per lane
  static_assert(RPW <= 32, "one lane per row ID");
  const int lane = threadIdx.x & 31;
  const int sub = lane / VPR, c = lane % VPR;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r0 = ((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * RPW; r0 < T; r0 += nwarps * RPW) {
    int64_t my_id = -1;
    if (lane < RPW && r0 + lane < T) {
      const bool take = (mask == nullptr) || (__ldg(mask + r0 + lane) == sel);
      if (take) {
        my_id = __ldcs(ids + r0 + lane);
        if (my_id < 0 || my_id >= R) {
          set_err(err, FS_ERR_ID_RANGE);
          my_id = -1;
        }
      }
    }
    int4 v[U];
    int64_t id[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      id[u] = __shfl_sync(0xffffffffu, my_id, u * RPI + sub);
      if (id[u] >= 0) v[u] = __ldg(table + id[u] * VPR + c);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (id[u] >= 0) __stcs(out + (r0 + u * RPI + sub) * VPR + c, v[u]);
  }
}

// Other row sizes that are a multiple of 16 bytes: one 16-byte vector per thread.
__global__ void __launch_bounds__(kThreads) gather_vec16_kernel(const int4* __restrict__ table, int64_t R,
                                                                int vpr /* 16-byte vectors per row */,
                                                                const int64_t* __restrict__ ids, int64_t T,
                                                                const uint8_t* __restrict__ mask, uint8_t sel,
                                                                int4* __restrict__ out, int32_t* err) {
  const int64_t total = T * vpr;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t f = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; f < total; f += stride) {
    const int64_t p = f / vpr;
    const int c = int(f - p * vpr);
    if (mask && __ldg(mask + p) != sel) continue;
    const int64_t id = __ldg(ids + p);
    if (id < 0 || id >= R) {
      set_err(err, FS_ERR_ID_RANGE);
      continue;
    }
    __stcs(out + f, __ldg(table + id * vpr + c));
  }
}

// Generic path: row bytes a multiple of 4 (or pointers not 16-byte aligned).
__global__ void __launch_bounds__(kThreads) gather_word_kernel(const uint32_t* __restrict__ table, int64_t R,
                                                               int wpr /* 4-byte words per row */,
                                                               const int64_t* __restrict__ ids, int64_t T,
                                                               const uint8_t* __restrict__ mask, uint8_t sel,
                                                               uint32_t* __restrict__ out, int32_t* err) {
  const int64_t total = T * wpr;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t f = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; f < total; f += stride) {
    const int64_t p = f / wpr;
    const int c = int(f - p * wpr);
    if (mask && __ldg(mask + p) != sel) continue;
    const int64_t id = __ldg(ids + p);
    if (id < 0 || id >= R) {
      set_err(err, FS_ERR_ID_RANGE);
      continue;
    }
    __stcs(out + f, __ldg(table + id * wpr + c));
  }
}

// Gather in shard-major order (the lookup of Algorithm 2 line 12 as each shard
// owner makes it, followed by the ranged combine back to batch-major):
// out[pos[j]] = table[sm_ids[j]] for every shard-major entry j.  Entries of
// one shard come together, so the rows a stretch of entries reads lie in one
// shard's row range; while it is being gathered, a shard's repeated rows are
// served by L2 rather than read again from DRAM.  Rows of 16 * VPR bytes, VPR
// in {4, 8, 16, 32}: lanes [k*VPR, (k+1)*VPR) move row k, U rows in flight
// per lane; whole rows are written to their scattered positions.  An ID out of
// range sets FS_ERR_ID_RANGE, a position out of [0, T) FS_ERR_BAD_OFFSETS;
// either entry is skipped.
// (three blocks per SM, as the row-sorted gather: room for the row loads and
// the next iteration's entries)
template <int VPR>
__global__ void __launch_bounds__(kThreads, 3) gather_scatter_kernel(const int4* __restrict__ table, int64_t R,
                                                                  const int64_t* __restrict__ sm_ids,
                                                                  const int32_t* __restrict__ pos, int64_t T,
                                                                  int4* __restrict__ out, int32_t* err) {
  constexpr int RPI = 32 / VPR;
  constexpr int U = (32 / RPI) < kUnroll ? (32 / RPI) : kUnroll;
  constexpr int RPW = RPI * U;
  static_assert(RPW <= 32, "one lane per entry");
  const int lane = threadIdx.x & 31;
  const int sub = lane / VPR, c = lane % VPR;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t stride = nwarps * RPW;
  // the IDs and positions of the warp's next iteration are loaded before the
  // current iteration's rows, so the entry stream's latency overlaps them
  int64_t nid = -1;
  int32_t npos = -1;
  auto load_entries = [&](int64_t e) {
    nid = -1;
    npos = -1;
    if (lane < RPW && e + lane < T) {
      nid = __ldcs(sm_ids + e + lane);
      npos = __ldcs(pos + e + lane);
    }
  };
  int64_t e0 = ((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * RPW;
  load_entries(e0);
  for (; e0 < T; e0 += stride) {
    int64_t my_id = nid;
    const int32_t my_pos = npos;
    const bool live = lane < RPW && e0 + lane < T;
    load_entries(e0 + stride);
    if (live) {
      if (my_id < 0 || my_id >= R) {
        set_err(err, FS_ERR_ID_RANGE);
        my_id = -1;
      } else if (my_pos < 0 || int64_t(my_pos) >= T) {
        set_err(err, FS_ERR_BAD_OFFSETS);
        my_id = -1;
      }
    }
    int4 v[U];
    int64_t id[U];
    int32_t p[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      id[u] = __shfl_sync(0xffffffffu, my_id, u * RPI + sub);
      p[u] = __shfl_sync(0xffffffffu, my_pos, u * RPI + sub);
      if (id[u] >= 0) v[u] = __ldg(table + id[u] * VPR + c);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (id[u] >= 0) __stcs(out + int64_t(p[u]) * VPR + c, v[u]);
  }
}

// Other row sizes, 4-byte words: thread per word of an entry's row.
__global__ void __launch_bounds__(kThreads) gather_scatter_word_kernel(const uint32_t* __restrict__ table, int64_t R,
                                                                       int wpr, const int64_t* __restrict__ sm_ids,
                                                                       const int32_t* __restrict__ pos, int64_t T,
                                                                       uint32_t* __restrict__ out, int32_t* err) {
  const int64_t total = T * wpr;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t f = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; f < total; f += stride) {
    const int64_t j = f / wpr;
    const int c = int(f - j * wpr);
    const int64_t id = __ldg(sm_ids + j);
    const int32_t p = __ldg(pos + j);
    if (id < 0 || id >= R) {
      set_err(err, FS_ERR_ID_RANGE);
      continue;
    }
    if (p < 0 || int64_t(p) >= T) {
      set_err(err, FS_ERR_BAD_OFFSETS);
      continue;
    }
    __stcs(out + int64_t(p) * wpr + c, __ldg(table + id * wpr + c));
  }
}

// Unmasked gather through the copy engine: each warp moves stages of BR
// consecutive output rows (BR * row bytes <= 2 KB).  The table rows of a stage
// arrive in a shared-memory slot by one bulk copy per row (completion counted
// in bytes on the slot's mbarrier); the whole stage then leaves by one bulk
// store to its contiguous place in the output.  A ring of NS slots keeps LA
// stages of loads in flight while one stage is stored.  Table rows are read
// with an evict-last L2 policy (hot rows are read again), the output is
// written evict-first.  A wait that exceeds wait_ns sets FS_ERR_TIMEOUT.
constexpr int kBulkStage = 2048;
template <int NS, int LA>
struct BulkRing {
  static constexpr int kWarpBytes = 128 + NS * kBulkStage;
  static constexpr int kBlockBytes = (kThreads / 32) * kWarpBytes;
  static_assert(LA >= 1 && LA <= NS - 2, "one slot is being stored while LA are loading");
};

template <int NS, int LA>
__global__ void __launch_bounds__(kThreads) gather_bulk_kernel(const char* __restrict__ table, int64_t R, int rb,
                                                               int br, const int64_t* __restrict__ ids, int64_t T,
                                                               char* __restrict__ out, int32_t* err,
                                                               uint64_t wait_ns) {
  using RG = BulkRing<NS, LA>;
  extern __shared__ __align__(128) unsigned char gsm[];
  const int lane = threadIdx.x & 31;
  unsigned char* wb = gsm + (threadIdx.x >> 5) * RG::kWarpBytes;
  const uint32_t bar0 = bulk::smem_addr(wb);
  const uint32_t data0 = bar0 + 128;
  if (lane == 0)
    for (int s = 0; s < NS; ++s) bulk::mbar_init(bar0 + 8 * s, 1);
  bulk::fence_init();
  __syncwarp();
  const uint64_t pol_in = bulk::evict_last_policy();
  const uint64_t pol_out = bulk::evict_first_policy();
  const int64_t nst = (T + br - 1) / br;
  const int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t nmine = w < nst ? (nst - 1 - w) / nw + 1 : 0;
  // ID of this lane's row in stage k (-1: none or out of range)
  auto load_id = [&](int64_t k) -> int64_t {
    if (k >= nmine) return -1;
    const int64_t r = (w + k * nw) * br + lane;
    if (lane >= br || r >= T) return -1;
    const int64_t id = __ldcs(ids + r);
    if (id < 0 || id >= R) {
      set_err(err, FS_ERR_ID_RANGE);
      return -1;
    }
    return id;
  };
  auto issue = [&](int64_t k, int64_t id) {
    if (k >= nmine) return;
    const uint32_t s = uint32_t(k % NS);
    const uint32_t bar = bar0 + 8 * s;
    const unsigned valid = __ballot_sync(0xffffffffu, id >= 0);
    if (lane == 0) bulk::arrive_expect_tx(bar, uint32_t(__popc(valid) * rb));
    __syncwarp();
    if (id >= 0) bulk::copy_g2s(data0 + s * kBulkStage + lane * rb, table + id * rb, uint32_t(rb), bar, pol_in);
  };
  for (int k = 0; k < LA; ++k) issue(k, load_id(k));
  int64_t next_id = load_id(LA);
  for (int64_t k = 0; k < nmine; ++k) {
    // the slot of stage k + LA last held stage k + LA - NS, stored at least
    // two iterations ago: at most the newest store may still be reading
    if (lane == 0) bulk::wait_group_read<NS - LA - 1>();
    __syncwarp();
    issue(k + LA, next_id);
    next_id = load_id(k + LA + 1);
    const uint32_t s = uint32_t(k % NS);
    if (!bulk::warp_wait(bar0 + 8 * s, uint32_t((k / NS) & 1), wait_ns)) {
      if (lane == 0) set_err(err, FS_ERR_TIMEOUT);
      for (int64_t j = k + 1; j <= k + LA && j < nmine; ++j)
        bulk::warp_wait(bar0 + 8 * uint32_t(j % NS), uint32_t((j / NS) & 1), wait_ns);
      break;
    }
    if (lane == 0) {
      const int64_t r0 = (w + k * nw) * br;
      const int64_t rows = (T - r0 < br) ? T - r0 : br;
      bulk::fence_async_shared();
      bulk::store_s2g(out + r0 * rb, data0 + s * kBulkStage, uint32_t(rows * rb), pol_out);
      bulk::commit_group();
    }
  }
  if (lane == 0) bulk::wait_group_all();
  __syncwarp();
  if (lane == 0)
    for (int s = 0; s < NS; ++s) bulk::mbar_inval(bar0 + 8 * s);
}

}  // namespace
}  // namespace fs

using namespace fs;

extern "C" fs_status fs_emb_gather(const void* table, int64_t num_rows, int32_t dim, fs_dtype dtype, const int64_t* ids,
                                   int64_t T, const uint8_t* mask, uint8_t sel, void* out, int32_t* err,
                                   fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T < 0 || T > INT32_MAX || num_rows < 0 || dim < 1 || (dtype != FS_F32 && dtype != FS_BF16) || !err)
    return FS_ERR_INVALID_ARG;
  if (T == 0) return FS_OK;
  if (!table || !ids || !out) return FS_ERR_INVALID_ARG;
  const int64_t row_bytes = int64_t(dim) * (dtype == FS_F32 ? 4 : 2);
  if (row_bytes % 4 != 0) return FS_ERR_INVALID_ARG;
  if (!aligned(ids, 8) || !aligned(table, 4) || !aligned(out, 4)) return FS_ERR_ALIGNMENT;
  const int sms = sm_count();
  if (!mask && row_bytes % 16 == 0 && row_bytes <= kBulkStage && aligned(table, 16) && aligned(out, 16)) {
    // unmasked: every output row is written, so whole stages go out by bulk store
    constexpr int NS = 4, LA = 2;
    using RG = BulkRing<NS, LA>;
    const int rb = int(row_bytes);
    const int br = (kBulkStage / rb) < 32 ? (kBulkStage / rb) : 32;
    auto kern = gather_bulk_kernel<NS, LA>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, RG::kBlockBytes);
    const int per_sm = (227 * 1024) / (RG::kBlockBytes + 1024);
    kern<<<unsigned(sms * per_sm), kThreads, RG::kBlockBytes, st>>>(static_cast<const char*>(table), num_rows, rb, br,
                                                                     ids, T, static_cast<char*>(out), err,
                                                                     uint64_t(spin_limit()) * 256u);
  } else if (row_bytes % 16 == 0 && aligned(table, 16) && aligned(out, 16)) {
    const int vpr = int(row_bytes / 16);
    const int4* tb = static_cast<const int4*>(table);
    int4* ob = static_cast<int4*>(out);
    const unsigned grid = unsigned(sms) * (2048 / kThreads);
    switch (vpr) {
      case 4: gather_rows_kernel<4><<<grid, kThreads, 0, st>>>(tb, num_rows, ids, T, mask, sel, ob, err); break;
      case 8: gather_rows_kernel<8><<<grid, kThreads, 0, st>>>(tb, num_rows, ids, T, mask, sel, ob, err); break;
      case 16: gather_rows_kernel<16><<<grid, kThreads, 0, st>>>(tb, num_rows, ids, T, mask, sel, ob, err); break;
      case 32: gather_rows_kernel<32><<<grid, kThreads, 0, st>>>(tb, num_rows, ids, T, mask, sel, ob, err); break;
      default: {
        const int64_t total = T * vpr;
        int64_t g = (total + kThreads - 1) / kThreads;
        if (g > int64_t(sms) * 8) g = int64_t(sms) * 8;
        gather_vec16_kernel<<<unsigned(g < 1 ? 1 : g), kThreads, 0, st>>>(tb, num_rows, vpr, ids, T, mask, sel, ob,
                                                                          err);
      }
    }
  } else {
    const int wpr = int(row_bytes / 4);
    const int64_t total = T * wpr;
    int64_t grid = (total + kThreads - 1) / kThreads;
    if (grid > int64_t(sms) * 8) grid = int64_t(sms) * 8;
    gather_word_kernel<<<unsigned(grid < 1 ? 1 : grid), kThreads, 0, st>>>(
        static_cast<const uint32_t*>(table), num_rows, wpr, ids, T, mask, sel, static_cast<uint32_t*>(out), err);
  }
  count_launch(1);
  return launch_status();
}

extern "C" fs_status fs_emb_gather_shard_major(const void* table, int64_t num_rows, int32_t dim, fs_dtype dtype,
                                               const int64_t* sm_ids, const int32_t* pos, int64_t T, void* out,
                                               int32_t* err, fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T < 0 || T > INT32_MAX || num_rows < 0 || dim < 1 || (dtype != FS_F32 && dtype != FS_BF16) || !err)
    return FS_ERR_INVALID_ARG;
  if (T == 0) return FS_OK;
  if (!table || !sm_ids || !pos || !out) return FS_ERR_INVALID_ARG;
  const int64_t row_bytes = int64_t(dim) * (dtype == FS_F32 ? 4 : 2);
  if (row_bytes % 4 != 0) return FS_ERR_INVALID_ARG;
  if (!aligned(sm_ids, 8) || !aligned(pos, 4) || !aligned(table, 4) || !aligned(out, 4)) return FS_ERR_ALIGNMENT;
  const int sms = sm_count();
  const unsigned grid = unsigned(sms) * (2048 / kThreads);
  const int vpr = (row_bytes % 16 == 0 && aligned(table, 16) && aligned(out, 16)) ? int(row_bytes / 16) : 0;
  const int4* tb = static_cast<const int4*>(table);
  int4* ob = static_cast<int4*>(out);
  switch (vpr) {
    case 4: gather_scatter_kernel<4><<<grid, kThreads, 0, st>>>(tb, num_rows, sm_ids, pos, T, ob, err); break;
    case 8: gather_scatter_kernel<8><<<grid, kThreads, 0, st>>>(tb, num_rows, sm_ids, pos, T, ob, err); break;
    case 16: gather_scatter_kernel<16><<<grid, kThreads, 0, st>>>(tb, num_rows, sm_ids, pos, T, ob, err); break;
    case 32: gather_scatter_kernel<32><<<grid, kThreads, 0, st>>>(tb, num_rows, sm_ids, pos, T, ob, err); break;
    default: {
      const int wpr = int(row_bytes / 4);
      int64_t g = (T * wpr + kThreads - 1) / kThreads;
      if (g > int64_t(sms) * 8) g = int64_t(sms) * 8;
      gather_scatter_word_kernel<<<unsigned(g < 1 ? 1 : g), kThreads, 0, st>>>(
          static_cast<const uint32_t*>(table), num_rows, wpr, sm_ids, pos, T, static_cast<uint32_t*>(out), err);
    }
  }
  count_launch(1);
  return launch_status();
}
