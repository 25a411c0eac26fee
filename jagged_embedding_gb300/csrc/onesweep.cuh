// Device-wide stable counting-sort passes in the "onesweep" style (Adinets &
// Merrill, "Onesweep: A Faster Least Significant Digit Radix Sort for GPUs",
// 2022): one up-front histogram kernel for every digit pass, then one kernel
// per pass that ranks a tile of keys by digit inside the block (warp
// __match_any_sync multisplit), finds the tile's global offset per digit with
// a decoupled look-back over the preceding tiles, stages the tile in digit
// order in shared memory and writes it out in coalesced runs.
//
// The sources (`Src`) decide where keys and values come from (a plain array,
// a length array with the index as value, an ID array filtered by a mask ...)
// and the digit function; the sinks (`Dst`) decide what is written.
#pragma once

#include "fs_common.cuh"

namespace fs {
namespace onesweep {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 16;
constexpr int kTile = kThreads * kItems;  // 4096 keys per tile
constexpr int kMaxBins = 512;
constexpr uint32_t kSkip = 0xFFFFu;

inline int64_t num_tiles(int64_t count) { return (count + kTile - 1) / kTile; }

template <class KeyT>
constexpr size_t pass_smem_bytes() {
  size_t stage = size_t(kTile) * (sizeof(KeyT) + sizeof(uint32_t));
  size_t hist = size_t(kWarps) * kMaxBins * sizeof(uint32_t);
  size_t un = stage > hist ? stage : hist;
  return un + 2 * kMaxBins * sizeof(uint32_t) + kMaxBins * sizeof(int64_t) + 64 * sizeof(uint32_t);
}

// --------------------------------------------------------------- histogram
// hist[p * nbins_max + d] += number of valid items whose pass-p digit is d;
// *n_valid += number of valid items.  Grid-stride; block-private histograms.
template <class Src>
__global__ void __launch_bounds__(kThreads) histogram_kernel(Src src, int64_t count, int npasses, int bits, int nb,
                                                             uint32_t* hist, int64_t* n_valid, int32_t* err) {
  __shared__ uint32_t sh[4 * kMaxBins];
  __shared__ uint32_t s_valid;
  for (int j = threadIdx.x; j < npasses * nb; j += blockDim.x) sh[j] = 0;
  if (threadIdx.x == 0) s_valid = 0;
  __syncthreads();
  uint32_t my_valid = 0;
  const int lane = threadIdx.x & 31;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < count; idx += stride) {
    const unsigned act = __activemask();
    typename Src::Key k;
    uint32_t v;
    const bool ok = src.load(idx, k, v, err);
    my_valid += ok ? 1u : 0u;
    // warp-aggregated increments: one shared atomic per distinct digit of the warp
    // (Zipf-hot keys would otherwise serialise on one counter)
    for (int p = 0; p < npasses; ++p) {
      const uint32_t d = ok ? src.digit(k, p * bits, bits) : 0xFFFFFFFFu;
      const unsigned peers = __match_any_sync(act, d);
      if (ok && (__ffs(peers) - 1) == lane) atomicAdd(&sh[p * nb + d], uint32_t(__popc(peers)));
    }
  }
  for (int o = 16; o > 0; o >>= 1) my_valid += __shfl_xor_sync(0xffffffffu, my_valid, o);
  if ((threadIdx.x & 31) == 0 && my_valid) atomicAdd(&s_valid, my_valid);
  __syncthreads();
  for (int j = threadIdx.x; j < npasses * nb; j += blockDim.x) {
    uint32_t c = sh[j];
    if (c) atomicAdd(&hist[(j / nb) * kMaxBins + (j % nb)], c);
  }
  if (threadIdx.x == 0 && s_valid) atomicAdd(reinterpret_cast<unsigned long long*>(n_valid),
                                             static_cast<unsigned long long>(s_valid));
}

// Exclusive scan of each pass's digit histogram (one block per pass).
static __global__ void __launch_bounds__(kThreads) digit_scan_kernel(const uint32_t* hist, uint32_t* offsets, int nb) {
  __shared__ uint32_t tmp[32];
  const uint32_t* h = hist + blockIdx.x * kMaxBins;
  uint32_t* o = offsets + blockIdx.x * kMaxBins;
  // kThreads * 2 >= kMaxBins digits
  int d0 = threadIdx.x * 2;
  uint32_t a = d0 < nb ? h[d0] : 0, b = d0 + 1 < nb ? h[d0 + 1] : 0;
  uint32_t tot;
  uint32_t ex = block_exclusive_scan<uint32_t>(a + b, tmp, &tot);
  if (d0 < nb) o[d0] = ex;
  if (d0 + 1 < nb) o[d0 + 1] = ex + a;
}

// --------------------------------------------------------------- one pass
// Stable scatter of the valid items of [0, count) by digit (shift, bits).
// count = *count_dev if count_dev != nullptr, else count_host.
// nb = number of digit values (<= kMaxBins); status: [tiles][nb] look-back words, zeroed by the caller;
// tile_counter: zeroed int (dynamic tile order = launch order, so a tile
// only ever waits on tiles that have already started).
template <class Src, class Dst>
__global__ void __launch_bounds__(kThreads, 3) pass_kernel(Src src, Dst dst, int shift, int bits, int nb,
                                                        const uint32_t* digit_offsets, uint64_t* status,
                                                        int* tile_counter, const int64_t* count_dev,
                                                        int64_t count_host, int32_t* err, int64_t limit) {
  using KeyT = typename Src::Key;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint32_t* warp_hist = reinterpret_cast<uint32_t*>(smem_raw);                 // [kWarps][nb] (phase 1)
  KeyT* stage_k = reinterpret_cast<KeyT*>(smem_raw);                           // [kTile]      (phase 2)
  constexpr size_t stage_bytes = size_t(kTile) * (sizeof(KeyT) + sizeof(uint32_t));
  constexpr size_t hist_bytes = size_t(kWarps) * kMaxBins * sizeof(uint32_t);
  constexpr size_t un = stage_bytes > hist_bytes ? stage_bytes : hist_bytes;
  uint32_t* stage_v = reinterpret_cast<uint32_t*>(smem_raw + size_t(kTile) * sizeof(KeyT));
  uint32_t* tile_count = reinterpret_cast<uint32_t*>(smem_raw + un);
  uint32_t* local_start = tile_count + kMaxBins;
  int64_t* gbase = reinterpret_cast<int64_t*>(local_start + kMaxBins);
  uint32_t* scratch = reinterpret_cast<uint32_t*>(gbase + kMaxBins);
  __shared__ int64_t s_tile;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_tile = atomicAdd(tile_counter, 1);
  __syncthreads();
  const int64_t tile = s_tile;
  const int64_t count = count_dev ? *count_dev : count_host;
  const int64_t base = tile * kTile;
  if (base >= count) return;  // trailing tile: no later valid tile looks back at it

  // Registers per item: the key, one packed word (digit in bits 20..31, rank /
  // local position in bits 0..19) and, only for sources whose value is not the
  // item index, the value.
  KeyT key[kItems];
  uint32_t val[Src::kIndexValue ? 1 : kItems];
  uint32_t pk[kItems];
  constexpr uint32_t kSkipPk = 0xFFF00000u;
#pragma unroll
  for (int i = 0; i < kItems; ++i) {
    int64_t idx = base + int64_t(warp) * 32 * kItems + i * 32 + lane;
    uint32_t v = 0;
    bool ok = idx < count && src.load(idx, key[i], v, nullptr);
    if constexpr (!Src::kIndexValue) val[i] = v;
    pk[i] = ok ? (src.digit(key[i], shift, bits) << 20) : kSkipPk;
  }
  for (int j = threadIdx.x; j < kWarps * nb; j += kThreads) warp_hist[j] = 0;
  __syncthreads();

  // warp-level multisplit, slot by slot (slot order = position order)
  uint32_t* wh = warp_hist + warp * nb;
#pragma unroll
  for (int i = 0; i < kItems; ++i) {
    const uint32_t d = pk[i] >> 20;
    const bool skip = pk[i] == kSkipPk;
    const unsigned peers = __match_any_sync(0xffffffffu, pk[i]);
    const unsigned lt = __popc(peers & lanemask_lt());
    const uint32_t b = skip ? 0u : wh[d];
    if (!skip) pk[i] |= b + lt;
    __syncwarp();
    if (!skip && lt == 0) wh[d] = b + __popc(peers);
    __syncwarp();
  }
  __syncthreads();

  // exclusive over warps per digit, tile totals
  for (int d = threadIdx.x; d < nb; d += kThreads) {
    uint32_t run = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      uint32_t c = warp_hist[w * nb + d];
      warp_hist[w * nb + d] = run;
      run += c;
    }
    tile_count[d] = run;
  }
  __syncthreads();

  // global offset per digit: decoupled look-back over preceding tiles
  for (int d = threadIdx.x; d < nb; d += kThreads) {
    uint64_t ex = thread_lookback(status + d, nb, tile, tile_count[d], err, limit);
    gbase[d] = int64_t(digit_offsets[d]) + int64_t(ex);
  }
  // tile-local digit starts
  {
    int d0 = threadIdx.x * 2;
    uint32_t a = d0 < nb ? tile_count[d0] : 0, b = d0 + 1 < nb ? tile_count[d0 + 1] : 0;
    uint32_t tot;
    uint32_t ex = block_exclusive_scan<uint32_t>(a + b, scratch, &tot);
    if (d0 < nb) local_start[d0] = ex;
    if (d0 + 1 < nb) local_start[d0 + 1] = ex + a;
    if (threadIdx.x == 0) scratch[40] = tot;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kItems; ++i)
    if (pk[i] != kSkipPk) {
      const uint32_t d = pk[i] >> 20;
      pk[i] = local_start[d] + warp_hist[warp * nb + d] + (pk[i] & 0xFFFFFu);  // tile-local position
    }
  const uint32_t nvalid = scratch[40];
  __syncthreads();  // warp_hist is dead; its space becomes the staging area
#pragma unroll
  for (int i = 0; i < kItems; ++i)
    if (pk[i] != kSkipPk) {
      stage_k[pk[i]] = key[i];
      if constexpr (Src::kIndexValue)
        stage_v[pk[i]] = uint32_t(base + int64_t(warp) * 32 * kItems + i * 32 + lane);
      else
        stage_v[pk[i]] = val[i];
    }
  __syncthreads();
  for (uint32_t j = threadIdx.x; j < nvalid; j += kThreads) {
    KeyT k = stage_k[j];
    uint32_t d = src.digit(k, shift, bits);
    int64_t o = gbase[d] + int64_t(j - local_start[d]);
    dst.store(o, k, stage_v[j]);
  }
}

// --------------------------------------------------------------- policies

// Plain (uint32 key, uint32 value) arrays; digit = bits [shift, shift+bits).
struct SrcU32 {
  using Key = uint32_t;
  static constexpr bool kIndexValue = false;
  const uint32_t* k;
  const uint32_t* v;
  __device__ __forceinline__ bool load(int64_t i, Key& key, uint32_t& val, int32_t*) const {
    key = k[i];
    val = v[i];
    return true;
  }
  __device__ __forceinline__ uint32_t digit(Key key, int shift, int bits) const {
    return (key >> shift) & ((1u << bits) - 1u);
  }
};

struct DstU32 {
  uint32_t* k;
  uint32_t* v;
  __device__ __forceinline__ void store(int64_t o, uint32_t key, uint32_t val) const {
    k[o] = key;
    v[o] = val;
  }
};

inline int bits_for(uint64_t max_key) {
  int b = 0;
  while (b < 64 && (max_key >> b) != 0) ++b;
  return b < 1 ? 1 : b;
}

}  // namespace onesweep
}  // namespace fs

namespace fs {
namespace onesweep {

// ---------------------------------------------------------------- host driver
// LSD sort of (uint32 key, uint32 value) pairs drawn from `Src0` (items of
// [0, count) that Src0::load accepts), by the low `key_bits` bits of the key.
// Result: *out_k / *out_v, n_valid entries (n_valid stays on the device).
struct SortPlan {
  int64_t count = 0;
  int key_bits = 1, passes = 1, bits = 1, nb = 2;
  int64_t tiles = 0;
  SortPlan() = default;
  SortPlan(int64_t c, int kb) : count(c), key_bits(kb < 1 ? 1 : kb) {
    passes = (key_bits + 8) / 9;
    if (passes > 4) passes = 4;
    bits = (key_bits + passes - 1) / passes;
    nb = 1 << bits;
    tiles = num_tiles(count);
  }
  size_t zero_bytes() const {  // hist + n_valid + counters + status
    return align_up(4 * kMaxBins * sizeof(uint32_t)) + align_up(sizeof(int64_t) + 4 * sizeof(int)) +
           align_up(size_t(passes) * size_t(tiles) * nb * sizeof(uint64_t));
  }
  size_t bytes() const {
    return zero_bytes() + align_up(4 * kMaxBins * sizeof(uint32_t)) + 4 * align_up(size_t(count) * sizeof(uint32_t));
  }
};

struct SortWs {
  unsigned char* zero_base = nullptr;
  size_t zero_bytes = 0;
  uint32_t* hist = nullptr;
  int64_t* n_valid = nullptr;
  int* counters = nullptr;
  uint64_t* status = nullptr;
  uint32_t* offsets = nullptr;
  uint32_t* k[2] = {nullptr, nullptr};
  uint32_t* v[2] = {nullptr, nullptr};
};

inline bool carve_sort_ws(const SortPlan& P, WsCursor& ws, SortWs& W) {
  W.zero_bytes = P.zero_bytes();
  W.zero_base = ws.take<unsigned char>(W.zero_bytes);
  W.offsets = ws.take<uint32_t>(4 * kMaxBins);
  for (int i = 0; i < 2; ++i) {
    W.k[i] = ws.take<uint32_t>(size_t(P.count));
    W.v[i] = ws.take<uint32_t>(size_t(P.count));
  }
  if (!ws.ok) return false;
  unsigned char* p = W.zero_base;
  W.hist = reinterpret_cast<uint32_t*>(p);
  p += align_up(4 * kMaxBins * sizeof(uint32_t));
  W.n_valid = reinterpret_cast<int64_t*>(p);
  W.counters = reinterpret_cast<int*>(p + sizeof(int64_t));
  p += align_up(sizeof(int64_t) + 4 * sizeof(int));
  W.status = reinterpret_cast<uint64_t*>(p);
  return true;
}

template <class K>
inline void set_pass_smem(K kernel, size_t bytes) {
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template <class Src0>
fs_status run_sort(const Src0& src0, const SortPlan& P, const SortWs& W, int32_t* err, cudaStream_t st,
                   uint32_t** out_k, uint32_t** out_v, int* launches) {
  if (cudaMemsetAsync(W.zero_base, 0, W.zero_bytes, st) != cudaSuccess) return FS_ERR_CUDA;
  *out_k = W.k[(P.passes - 1) & 1];
  *out_v = W.v[(P.passes - 1) & 1];
  if (P.count == 0) return FS_OK;
  const int64_t lim = spin_limit();
  int64_t hgrid = (P.count + kThreads - 1) / kThreads;
  int64_t hcap = int64_t(sm_count()) * 8;
  if (hgrid > hcap) hgrid = hcap;
  histogram_kernel<Src0><<<unsigned(hgrid), kThreads, 0, st>>>(src0, P.count, P.passes, P.bits, P.nb, W.hist,
                                                               W.n_valid, err);
  digit_scan_kernel<<<P.passes, kThreads, 0, st>>>(W.hist, W.offsets, P.nb);
  *launches += 2;
  const size_t smem = pass_smem_bytes<uint32_t>();
  const size_t status_stride = size_t(P.tiles) * P.nb;
  for (int p = 0; p < P.passes; ++p) {
    DstU32 dst{W.k[p & 1], W.v[p & 1]};
    if (p == 0) {
      set_pass_smem(pass_kernel<Src0, DstU32>, smem);
      pass_kernel<Src0, DstU32><<<unsigned(P.tiles), kThreads, smem, st>>>(
          src0, dst, 0, P.bits, P.nb, W.offsets, W.status, W.counters + 0, nullptr, P.count, err, lim);
    } else {
      set_pass_smem(pass_kernel<SrcU32, DstU32>, smem);
      SrcU32 s{W.k[(p - 1) & 1], W.v[(p - 1) & 1]};
      pass_kernel<SrcU32, DstU32><<<unsigned(P.tiles), kThreads, smem, st>>>(
          s, dst, p * P.bits, P.bits, P.nb, W.offsets + p * kMaxBins, W.status + p * status_stride,
          W.counters + p, W.n_valid, 0, err, lim);
    }
    *launches += 1;
  }
  return launch_status();
}

}  // namespace onesweep
}  // namespace fs
