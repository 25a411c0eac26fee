// Embedding row gather into batch-major jagged output.
// FreeScale (arXiv 2604.24073) Algorithm 2 line 12 (Lookup, then the
// embeddings go back to batch-major: the ranged combine is fused here, each
// row lands directly at its batch-major position), line 15 (merge of the
// prefetched exclusive rows and the collision rows: two masked calls into one
// output buffer) and §2.1 (sequence embeddings, no pooling).
//
// Bandwidth layout: the output (T x row bytes) is written once and never
// re-read here, so it is written with streaming (evict-first) stores; table
// rows are read through the non-coherent path so that hot (Zipf head) rows
// stay cached in L1/L2.  A lane moves one 16-byte vector of a row; lanes of a
// warp cover consecutive vectors, so a 256-byte row is 16 lanes and one warp
// instruction moves two rows.  Each lane keeps 8 independent vectors in flight.
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

}  // namespace
}  // namespace fs

using namespace fs;

extern "C" fs_status fs_emb_gather(const void* table, int64_t num_rows, int32_t dim, fs_dtype dtype, const int64_t* ids,
                                   int64_t T, const uint8_t* mask, uint8_t sel, void* out, int32_t* err,
                                   fs_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T < 0 || T > INT32_MAX || num_rows < 0 || dim < 1 || (dtype != FS_F32 && dtype != FS_BF16) || !err)
    return FS_ERR_INVALID_ARG;
  if (T == 0) return FS_OK;
  if (!table || !ids || !out) return FS_ERR_INVALID_ARG;
  const int64_t row_bytes = int64_t(dim) * (dtype == FS_F32 ? 4 : 2);
  if (row_bytes % 4 != 0) return FS_ERR_INVALID_ARG;
  if (!aligned(ids, 8) || !aligned(table, 4) || !aligned(out, 4)) return FS_ERR_ALIGNMENT;
  const int sms = sm_count();
  if (row_bytes % 16 == 0 && aligned(table, 16) && aligned(out, 16)) {
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
