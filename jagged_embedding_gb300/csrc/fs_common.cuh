// Shared device/host helpers of the jagged library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/fs_jagged.h"

namespace fs {

// ---------------------------------------------------------------- host side

int sm_count();                        // SMs of the current device (cached per device)
int64_t spin_limit();                  // polls before a bounded wait gives up
int64_t debug_skip_tile();             // test hook: tile that never publishes (-1 = none)
void count_launch(int k = 1);          // bookkeeping for fs_launch_count()

// One NVTX range per C-ABI call, named after the call, so that a profiler's
// timeline (or `ncu --nvtx --nvtx-include`) shows which call launched which
// kernels.  With no tool attached an NVTX call is a branch on a null hook.
struct NvtxScope {
  explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
  ~NvtxScope() { nvtxRangePop(); }
  NvtxScope(const NvtxScope&) = delete;
  NvtxScope& operator=(const NvtxScope&) = delete;
};
#define FS_NVTX_RANGE() ::fs::NvtxScope fs_nvtx_scope_(__func__)

inline fs_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? FS_OK : FS_ERR_CUDA;
}

constexpr size_t align_up(size_t x, size_t a = 256) { return (x + a - 1) / a * a; }

// Bump allocator over the caller's workspace (never allocates).
struct WsCursor {
  char* base;
  size_t size;
  size_t used = 0;
  bool ok = true;
  WsCursor(void* b, size_t s) : base(static_cast<char*>(b)), size(s) {}
  template <class T>
  T* take(size_t count) {
    size_t bytes = align_up(count * sizeof(T));
    if (used + bytes > size) { ok = false; return nullptr; }
    T* p = reinterpret_cast<T*>(base + used);
    used += bytes;
    return p;
  }
};

// Same layout arithmetic, used by the *_workspace_size queries.
struct WsCounter {
  size_t used = 0;
  template <class T>
  T* take(size_t count) {
    used += align_up(count * sizeof(T));
    return nullptr;
  }
};

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------- device side

__device__ __forceinline__ void set_err(int32_t* err, int code) {
  if (*reinterpret_cast<volatile int32_t*>(err) == 0) atomicCAS(err, 0, code);
}

__device__ __forceinline__ int32_t read_err(const int32_t* err) {
  return *reinterpret_cast<const volatile int32_t*>(err);
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ uint64_t ld_volatile_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_volatile_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Single-pass chained scan status words (decoupled look-back, Merrill &
// Garland 2016): bits 63..62 = flag, bits 61..0 = value.
constexpr uint64_t kFlagAgg = 1ull << 62;
constexpr uint64_t kFlagInc = 2ull << 62;
constexpr uint64_t kValMask = (1ull << 62) - 1;

// Look-back by one full warp for one counter of tile `tile` (>= 1): publishes
// `aggregate`, walks predecessors 32 at a time until an inclusive prefix is
// found, publishes the inclusive value and returns the exclusive prefix
// (same value in every lane).  A wait that exceeds `limit` polls (or sees
// another block's error) sets FS_ERR_TIMEOUT and returns 0.
// `stride` = distance between consecutive tiles' words for this counter.
__device__ __forceinline__ uint64_t warp_lookback(uint64_t* status, int64_t stride, int64_t tile, uint64_t aggregate,
                                                  int32_t* err, int64_t limit, bool publish = true) {
  const int lane = threadIdx.x & 31;
  if (tile == 0) {
    if (lane == 0 && publish) st_volatile_u64(status, kFlagInc | aggregate);
    return 0;
  }
  if (lane == 0 && publish) st_volatile_u64(status + tile * stride, kFlagAgg | aggregate);
  uint64_t excl = 0;
  int64_t pred = tile - 1;
  int64_t polls = 0;
  while (true) {
    int64_t idx = pred - lane;
    uint64_t s = (idx >= 0) ? ld_volatile_u64(status + idx * stride) : (kFlagInc);
    uint64_t flag = s >> 62;
    unsigned not_ready = __ballot_sync(0xffffffffu, flag == 0);
    unsigned is_inc = __ballot_sync(0xffffffffu, flag == 2);
    unsigned upto = is_inc ? ((__ffs(is_inc) == 32) ? 0xffffffffu : ((2u << (__ffs(is_inc) - 1)) - 1u)) : 0xffffffffu;
    if ((not_ready & upto) == 0) {
      uint64_t v = ((1u << lane) & upto) ? (s & kValMask) : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      excl += v;
      if (is_inc) break;
      pred -= 32;
      polls = 0;
      continue;
    }
    if (++polls > limit || (polls % 1024 == 0 && read_err(err) != 0)) {
      if (lane == 0) set_err(err, FS_ERR_TIMEOUT);
      excl = 0;
      break;
    }
    __nanosleep(32);
  }
  if (lane == 0 && publish) st_volatile_u64(status + tile * stride, kFlagInc | ((excl + aggregate) & kValMask));
  return excl;
}

// Block-wide exclusive scan of one value per thread (blockDim.x <= 1024,
// multiple of 32).  `smem` needs 32 slots.  Returns exclusive prefix, sets
// *total (same in all threads).
template <class T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* smem, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) smem[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T w = (lane < nw) ? smem[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    smem[lane] = w;  // inclusive per warp
  }
  __syncthreads();
  T warp_excl = (warp == 0) ? T(0) : smem[warp - 1];
  *total = smem[nw - 1];
  T res = warp_excl + x - v;
  __syncthreads();
  return res;
}

}  // namespace fs
