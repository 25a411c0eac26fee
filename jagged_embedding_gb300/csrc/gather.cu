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
#include "tma.cuh"

namespace fs {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;
bool g_gather_staged = false;  // 256-byte rows: bulk-copy staged kernel instead of the register path
int g_gather_variant = 0;      // 256-byte rows: unroll / L2 hint of the register path

// Row bytes = 16 * VPR with VPR in {4, 8, 16, 32}: a warp instruction moves
// RPI = 32 / VPR whole rows (lanes [k*VPR, (k+1)*VPR) own row k), and a warp
// iteration moves RPI * U consecutive rows whose IDs (and mask bytes) one
// coalesced load brings in and shuffles out; no per-element division, U
// independent 16-byte loads in flight per lane.
__device__ __forceinline__ int4 ld_row_vec(const int4* p, uint64_t pol, bool hint) {
  if (!hint) return __ldg(p);
  int4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.s32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

template <int VPR, int UNROLL = kUnroll, bool HINT = false>
__global__ void __launch_bounds__(kThreads) gather_rows_kernel(const int4* __restrict__ table, int64_t R,
                                                               const int64_t* __restrict__ ids, int64_t T,
                                                               const uint8_t* __restrict__ mask, uint8_t sel,
                                                               int4* __restrict__ out, int32_t* err) {
  constexpr int RPI = 32 / VPR;                              // rows per warp instruction
  constexpr int U = (32 / RPI) < UNROLL ? (32 / RPI) : UNROLL;
  uint64_t pol = 0;
  if constexpr (HINT) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
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
      if (id[u] >= 0) v[u] = ld_row_vec(table + id[u] * VPR + c, pol, HINT);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (id[u] >= 0) __stcs(out + (r0 + u * RPI + sub) * VPR + c, v[u]);
  }
}

// Staged gather: per warp, NST stages of 32 rows in shared memory.  Each lane
// brings one table row in with a bulk asynchronous copy (cp.async.bulk, one
// mbarrier per stage); once a stage is complete, its 32 consecutive output
// rows leave in one bulk store (or, with a mask, one bulk store per selected
// row), with an evict-first L2 policy since the output is not re-read here.
template <int RB>
struct GStaged {
  static constexpr int NST = 4;
  static constexpr int STAGE = 32 * RB;
  static constexpr int WARP_BYTES = NST * STAGE + 128;
  static constexpr int WPB_RAW = (192 * 1024) / WARP_BYTES;
  static constexpr int WPB = WPB_RAW < 1 ? 1 : (WPB_RAW > 8 ? 8 : WPB_RAW);
  static constexpr int SMEM = WPB * WARP_BYTES;
};

template <int RB>
__global__ void __launch_bounds__(GStaged<RB>::WPB * 32, 1)
    gather_staged_kernel(const unsigned char* __restrict__ table, int64_t R, const int64_t* __restrict__ ids, int64_t T,
                         const uint8_t* __restrict__ mask, uint8_t sel, unsigned char* __restrict__ out, int32_t* err,
                         int64_t limit) {
  using P = GStaged<RB>;
  constexpr int NST = P::NST;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned char* wb = smem + warp * P::WARP_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(wb + NST * P::STAGE);
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) tma::mbar_init(bars + s, 1);
    tma::fence_barrier_init();
  }
  __syncwarp();
  const uint64_t pol = tma::policy_evict_first();
  uint32_t phase = 0;
  const int64_t nbatches = (T + 31) / 32;
  const int64_t nwarps = int64_t(gridDim.x) * P::WPB;
  const int64_t first = int64_t(blockIdx.x) * P::WPB + warp;
  // batches of this warp: first, first + nwarps, ...; the k-th goes to stage k % NST
  auto issue = [&](int64_t k) {
    const int st = int(k % NST);
    const int64_t r0 = (first + k * nwarps) * 32;
    const int cnt = (T - r0 < 32) ? int(T - r0) : 32;
    int64_t id = -1;
    if (lane < cnt && (mask == nullptr || __ldg(mask + r0 + lane) == sel)) {
      id = __ldcs(ids + r0 + lane);
      if (id < 0 || id >= R) {
        set_err(err, FS_ERR_ID_RANGE);
        id = -1;
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, id >= 0);
    // a stage whose previous contents are still being stored must not be
    // overwritten: every lane commits exactly one bulk group per batch, so at
    // most NST - 1 younger groups may still be reading
    tma::bulk_wait_read<NST - 1>();
    __syncwarp();
    if (lane == 0) tma::mbar_arrive_expect_tx(bars + st, uint32_t(__popc(m)) * RB);
    __syncwarp();
    if (id >= 0) tma::bulk_g2s(wb + st * P::STAGE + lane * RB, table + id * RB, RB, bars + st);
    return m;
  };
  int64_t nmine = (first < nbatches) ? (nbatches - first + nwarps - 1) / nwarps : 0;
  unsigned pend[NST];
  for (int k = 0; k < NST && k < nmine; ++k) pend[k] = issue(k);
  for (int64_t k = 0; k < nmine; ++k) {
    const int st = int(k % NST);
    const unsigned m = pend[st];
    if (!tma::mbar_wait(bars + st, (phase >> st) & 1u, limit)) {
      if (lane == 0) set_err(err, FS_ERR_TIMEOUT);
      break;
    }
    phase ^= 1u << st;
    const int64_t r0 = (first + k * nwarps) * 32;
    const int cnt = (T - r0 < 32) ? int(T - r0) : 32;
    if (m == ((cnt == 32) ? 0xffffffffu : ((1u << cnt) - 1u))) {
      if (lane == 0) tma::bulk_s2g(out + r0 * RB, wb + st * P::STAGE, uint32_t(cnt) * RB, pol);
    } else if ((m >> lane) & 1u) {
      tma::bulk_s2g(out + (r0 + lane) * RB, wb + st * P::STAGE + lane * RB, RB, pol);
    }
    tma::bulk_commit();
    __syncwarp();
    if (k + NST < nmine) pend[st] = issue(k + NST);
  }
  tma::bulk_wait_all();
  __syncwarp();
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

extern "C" void fs_debug_gather_variant(int32_t v) {
  fs::g_gather_staged = v == 9;
  fs::g_gather_variant = v;
}

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
      case 16:
        if (g_gather_staged) {
          using P = GStaged<256>;
          cudaFuncSetAttribute(gather_staged_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, P::SMEM);
          gather_staged_kernel<256><<<unsigned(sms), P::WPB * 32, P::SMEM, st>>>(
              static_cast<const unsigned char*>(table), num_rows, ids, T, mask, sel, static_cast<unsigned char*>(out),
              err, spin_limit());
        } else if (g_gather_variant == 1) {
          gather_rows_kernel<16, 16, false><<<grid, kThreads, 0, st>>>(tb, num_rows, ids, T, mask, sel, ob, err);
        } else if (g_gather_variant == 2) {
          gather_rows_kernel<16, 8, true><<<grid, kThreads, 0, st>>>(tb, num_rows, ids, T, mask, sel, ob, err);
        } else if (g_gather_variant == 3) {
          gather_rows_kernel<16, 16, true><<<grid, kThreads, 0, st>>>(tb, num_rows, ids, T, mask, sel, ob, err);
        } else {
          gather_rows_kernel<16><<<grid, kThreads, 0, st>>>(tb, num_rows, ids, T, mask, sel, ob, err);
        }
        break;
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
