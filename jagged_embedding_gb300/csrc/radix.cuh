// Device-wide stable counting-sort passes (LSD radix sort, reduce-then-scan:
// Merrill & Grimshaw, "High Performance and Scalable Radix Sorting", 2011).
//
// One pass over the items of [0, count) keyed by one digit:
//   1. upsweep:    one block per chunk of kChunkTiles tiles of kTile items;
//                  per tile, the count of every digit value, written as the
//                  exclusive prefix over the chunk's earlier tiles
//                  (counts[tile][digit]); per chunk, the digit totals;
//   2. chunk scan: per digit, the exclusive prefix of the chunk totals over
//                  the chunks, and the digit totals; then the exclusive
//                  prefix of the digit totals (digit_base);
//   3. downsweep:  per tile, a stable rank of every item among the tile's items
//                  with the same digit (warp __match_any_sync multisplit, warps
//                  combined in order), staging in digit order in shared memory
//                  and coalesced writes of every digit run to
//                  digit_base[d] + chunk_base[chunk][d] + counts[tile][d] + rank.
// All count arrays are digit-minor, so every read and write of them is
// coalesced.  No block waits on another block, so nothing spins.  (A
// single-pass decoupled look-back over ~70k tiles per pass was measured on
// GB300 to be bound by the look-back chain, about 16 tiles per microsecond.)
//
// Sources (`Src`) decide where keys and values come from (a plain array, a
// length array with the index as value, an ID array filtered by a mask ...)
// and the digit function: fetch(i) only loads (so that a tile's loads are all
// in flight together), fetch2(raw) (kFetch2) the loads that depend on the
// first ones, make(raw, i, key, val, err) checks and converts.
// Sinks (`Dst`) decide what is written.
#pragma once

#include "fs_common.cuh"

namespace fs {
namespace radix {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 16;
constexpr int kTile = kThreads * kItems;  // 4096 items per tile
constexpr int kMaxBins = 1024;
constexpr int kChunkTiles = 16;  // tiles per upsweep block
constexpr int kPerT = kMaxBins / kThreads;  // digits per thread

inline int64_t num_tiles(int64_t count) { return (count + kTile - 1) / kTile; }
inline int64_t num_chunks(int64_t ntiles) { return (ntiles + kChunkTiles - 1) / kChunkTiles; }

template <class KeyT>
constexpr size_t downsweep_smem_bytes() {
  size_t stage = size_t(kTile) * (sizeof(KeyT) + sizeof(uint32_t));
  size_t hist = size_t(kWarps) * kMaxBins * sizeof(uint32_t);
  size_t un = stage > hist ? stage : hist;
  return un + 2 * kMaxBins * sizeof(uint32_t) + kMaxBins * sizeof(int64_t) + 64 * sizeof(uint32_t);
}

// Index of item i of lane `lane` in warp `warp` of tile `tile` (warp-striped,
// so a warp's slot i is 32 consecutive items; slot order = item order).
__device__ __forceinline__ int64_t item_index(int64_t tile, int warp, int i, int lane) {
  return tile * kTile + int64_t(warp) * 32 * kItems + i * 32 + lane;
}

// ------------------------------------------------------------------ upsweep
// Block c: tiles [c * kChunkTiles, ...) one after another.  Per tile, one
// block-wide histogram (all item loads issued first, then one shared-memory
// increment per item); counts[tile][d] = this chunk's count of d before the
// tile; chunk_sums[c][d] = the chunk's count of d.
template <class Src>
__global__ void __launch_bounds__(kThreads) upsweep_kernel(Src src, int shift, int bits, int nb,
                                                           const int64_t* count_dev, int64_t count_host,
                                                           uint32_t* counts, uint32_t* chunk_sums, int64_t ntiles,
                                                           int32_t* err) {
  __shared__ uint32_t hist[kMaxBins];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t chunk = blockIdx.x;
  const int64_t count = count_dev ? *count_dev : count_host;
  uint32_t run[kPerT];
#pragma unroll
  for (int j = 0; j < kPerT; ++j) run[j] = 0;
  for (int c = 0; c < kChunkTiles; ++c) {
    const int64_t tile = chunk * kChunkTiles + c;
    if (tile >= ntiles) break;
    for (int j = threadIdx.x; j < nb; j += kThreads) hist[j] = 0;
    __syncthreads();
    if (tile * kTile < count) {
      typename Src::Raw raw[kItems];
#pragma unroll
      for (int i = 0; i < kItems; ++i) {
        const int64_t idx = item_index(tile, warp, i, lane);
        if (idx < count) raw[i] = src.fetch(idx);
      }
      if constexpr (Src::kFetch2) {  // loads that depend on the first ones, all issued together
#pragma unroll
        for (int i = 0; i < kItems; ++i)
          if (item_index(tile, warp, i, lane) < count) src.fetch2(raw[i]);
      }
#pragma unroll
      for (int i = 0; i < kItems; ++i) {
        const int64_t idx = item_index(tile, warp, i, lane);
        typename Src::Key k;
        uint32_t v;
        if (idx < count && src.make(raw[i], idx, k, v, err)) atomicAdd(hist + src.digit(k, shift, bits), 1u);
      }

    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kPerT; ++j) {
      const int d = threadIdx.x + j * kThreads;
      if (d < nb) {
        counts[tile * nb + d] = run[j];
        run[j] += hist[d];
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < kPerT; ++j) {
    const int d = threadIdx.x + j * kThreads;
    if (d < nb) chunk_sums[chunk * nb + d] = run[j];
  }
}

// ------------------------------------------------------------------ scans
// Exclusive prefix of chunk_sums[0 .. nchunks)[d] over the chunks, in place,
// and totals[d].  Block b: digits [32 b, 32 b + 32), one per lane; warp w of
// the block takes a contiguous range of chunks: range sums, exclusive over the
// warps in shared memory, then each warp rescans its range.
constexpr int kScanThreads = 1024;
static __global__ void __launch_bounds__(kScanThreads) chunk_scan_kernel(uint32_t* chunk_sums, int64_t nchunks, int nb,
                                                                        uint32_t* totals) {
  __shared__ uint32_t part[32][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int d = blockIdx.x * 32 + lane;
  const int64_t per = (nchunks + 31) / 32;
  const int64_t c0 = w * per, c1 = (c0 + per < nchunks) ? c0 + per : nchunks;
  uint32_t s = 0;
  if (d < nb)
    for (int64_t c = c0; c < c1; ++c) s += chunk_sums[c * nb + d];
  part[w][lane] = s;
  __syncthreads();
  if (w == 0) {
    uint32_t run = 0;
    for (int ww = 0; ww < 32; ++ww) {
      const uint32_t t = part[ww][lane];
      part[ww][lane] = run;
      run += t;
    }
    if (d < nb) totals[d] = run;
  }
  __syncthreads();
  uint32_t run = part[w][lane];
  if (d < nb)
    for (int64_t c = c0; c < c1; ++c) {
      const uint32_t v = chunk_sums[c * nb + d];
      chunk_sums[c * nb + d] = run;
      run += v;
    }
}

// Exclusive scan of the digit totals; *n_valid = their sum.
static __global__ void __launch_bounds__(kThreads) digit_base_kernel(const uint32_t* totals, int nb, uint32_t* digit_base,
                                                              int64_t* n_valid) {
  __shared__ uint32_t tmp[32];
  constexpr int kPer = kMaxBins / kThreads;  // digits per thread
  const int d0 = threadIdx.x * kPer;
  uint32_t v[kPer], sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    v[i] = d0 + i < nb ? totals[d0 + i] : 0u;
    sum += v[i];
  }
  uint32_t tot;
  uint32_t run = block_exclusive_scan<uint32_t>(sum, tmp, &tot);
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    if (d0 + i < nb) digit_base[d0 + i] = run;
    run += v[i];
  }
  if (threadIdx.x == 0 && n_valid) *n_valid = int64_t(tot);
}

// ------------------------------------------------------------------ downsweep
template <class Src, class Dst>
__global__ void __launch_bounds__(kThreads, 4) downsweep_kernel(Src src, Dst dst, int shift, int bits, int nb,
                                                                const uint32_t* digit_base, const uint32_t* counts,
                                                                const uint32_t* chunk_base, int64_t ntiles,
                                                                const int64_t* count_dev, int64_t count_host) {
  using KeyT = typename Src::Key;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint32_t* warp_hist = reinterpret_cast<uint32_t*>(smem_raw);  // [kWarps][nb] (phase 1)
  KeyT* stage_k = reinterpret_cast<KeyT*>(smem_raw);            // [kTile]      (phase 2)
  constexpr size_t stage_bytes = size_t(kTile) * (sizeof(KeyT) + sizeof(uint32_t));
  constexpr size_t hist_bytes = size_t(kWarps) * kMaxBins * sizeof(uint32_t);
  constexpr size_t un = stage_bytes > hist_bytes ? stage_bytes : hist_bytes;
  uint32_t* stage_v = reinterpret_cast<uint32_t*>(smem_raw + size_t(kTile) * sizeof(KeyT));
  uint32_t* tile_count = reinterpret_cast<uint32_t*>(smem_raw + un);
  uint32_t* local_start = tile_count + kMaxBins;
  int64_t* gbase = reinterpret_cast<int64_t*>(local_start + kMaxBins);
  uint32_t* scratch = reinterpret_cast<uint32_t*>(gbase + kMaxBins);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t tile = blockIdx.x;
  const int64_t count = count_dev ? *count_dev : count_host;
  if (tile * kTile >= count) return;

  // this tile's offset inside every digit run: loaded first, so that these
  // reads overlap the item loads and the ranking below
  uint32_t my_off[kPerT];
#pragma unroll
  for (int i = 0; i < kPerT; ++i) {
    const int d = threadIdx.x + i * kThreads;
    my_off[i] = d < nb ? __ldg(counts + tile * nb + d) + __ldg(chunk_base + (tile / kChunkTiles) * nb + d) +
                             __ldg(digit_base + d)
                       : 0u;
  }

  // per item: the key, one packed word (digit in bits 20..31, rank / local
  // position in bits 0..19) and, only for sources whose value is not the item
  // index, the value
  KeyT key[kItems];
  uint32_t val[Src::kIndexValue ? 1 : kItems];
  uint32_t pk[kItems];
  constexpr uint32_t kSkipPk = 0xFFF00000u;
  {
    typename Src::Raw raw[kItems];
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
      const int64_t idx = item_index(tile, warp, i, lane);
      if (idx < count) raw[i] = src.fetch(idx);
    }
    if constexpr (Src::kFetch2) {
#pragma unroll
      for (int i = 0; i < kItems; ++i)
        if (item_index(tile, warp, i, lane) < count) src.fetch2(raw[i]);
    }
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
      const int64_t idx = item_index(tile, warp, i, lane);
      uint32_t v = 0;
      const bool ok = idx < count && src.make(raw[i], idx, key[i], v, nullptr);
      if constexpr (!Src::kIndexValue) val[i] = v;
      pk[i] = ok ? (src.digit(key[i], shift, bits) << 20) : kSkipPk;
    }
  }
  for (int j = threadIdx.x; j < kWarps * nb; j += kThreads) warp_hist[j] = 0;
  __syncthreads();

  // warp-level multisplit, slot by slot (slot order = item order)
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

  // exclusive over warps per digit, tile totals, global base of each digit run
#pragma unroll
  for (int i = 0; i < kPerT; ++i) {
    const int d = threadIdx.x + i * kThreads;
    if (d < nb) {
      uint32_t run = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t c = warp_hist[w * nb + d];
        warp_hist[w * nb + d] = run;
        run += c;
      }
      tile_count[d] = run;
      gbase[d] = int64_t(my_off[i]);
    }
  }
  __syncthreads();
  {
    constexpr int kPer = kMaxBins / kThreads;  // digits per thread
    const int d0 = threadIdx.x * kPer;
    uint32_t v[kPer], sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      v[i] = d0 + i < nb ? tile_count[d0 + i] : 0u;
      sum += v[i];
    }
    uint32_t tot;
    uint32_t run = block_exclusive_scan<uint32_t>(sum, scratch, &tot);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (d0 + i < nb) local_start[d0 + i] = run;
      run += v[i];
    }
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
        stage_v[pk[i]] = uint32_t(item_index(tile, warp, i, lane));
      else
        stage_v[pk[i]] = val[i];
    }
  __syncthreads();
  for (uint32_t j = threadIdx.x; j < nvalid; j += kThreads) {
    const KeyT k = stage_k[j];
    const uint32_t d = src.digit(k, shift, bits);
    dst.store(gbase[d] + int64_t(j - local_start[d]), k, stage_v[j]);
  }
}

// ------------------------------------------------------------------ policies

// Plain (uint32 key, uint32 value) arrays; digit = bits [shift, shift+bits).
struct SrcU32 {
  using Key = uint32_t;
  static constexpr bool kIndexValue = false;
  const uint32_t* k;
  const uint32_t* v;
  static constexpr bool kFetch2 = false;
  using Raw = uint2;
  __device__ __forceinline__ Raw fetch(int64_t i) const { return make_uint2(__ldcs(k + i), __ldcs(v + i)); }
  __device__ __forceinline__ bool make(const Raw& r, int64_t, Key& key, uint32_t& val, int32_t*) const {
    key = r.x;
    val = r.y;
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

// ------------------------------------------------------------------ host side

template <class K>
inline void set_smem(K kernel, size_t bytes) {
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

// Scratch of one counting-sort pass over up to `count` items with nb digit values.
struct PassWs {
  uint32_t* counts = nullptr;      // [ntiles][nb]
  uint32_t* chunk = nullptr;       // [nchunks][nb]
  uint32_t* totals = nullptr;      // [kMaxBins]
  uint32_t* digit_base = nullptr;  // [kMaxBins]
  int64_t* n_valid = nullptr;      // [1]
  int64_t ntiles = 0;
};

inline size_t pass_ws_bytes(int64_t count, int nb) {
  return align_up(size_t(nb) * size_t(num_tiles(count)) * sizeof(uint32_t)) +
         align_up(size_t(nb) * size_t(num_chunks(num_tiles(count))) * sizeof(uint32_t)) +
         2 * align_up(kMaxBins * sizeof(uint32_t)) + align_up(sizeof(int64_t));
}

inline bool carve_pass_ws(int64_t count, int nb, WsCursor& ws, PassWs& P) {
  P.ntiles = num_tiles(count);
  P.counts = ws.take<uint32_t>(size_t(nb) * size_t(P.ntiles));
  P.chunk = ws.take<uint32_t>(size_t(nb) * size_t(num_chunks(P.ntiles)));
  P.totals = ws.take<uint32_t>(kMaxBins);
  P.digit_base = ws.take<uint32_t>(kMaxBins);
  P.n_valid = ws.take<int64_t>(1);
  return ws.ok;
}

// One stable counting-sort pass (upsweep, chunk scan, digit base, downsweep).  count is
// *count_dev if given, else count_host; the grid covers count_host items.
// *P.n_valid receives the number of items the source accepted.
template <class Src, class Dst>
void run_pass(const Src& src, const Dst& dst, int shift, int bits, int nb, const int64_t* count_dev,
              int64_t count_host, const PassWs& P, int32_t* err, cudaStream_t st, int* launches) {
  if (P.ntiles == 0) {
    cudaMemsetAsync(P.n_valid, 0, sizeof(int64_t), st);
    return;
  }
  const int64_t nchunks = num_chunks(P.ntiles);
  upsweep_kernel<Src><<<unsigned(nchunks), kThreads, 0, st>>>(src, shift, bits, nb, count_dev, count_host, P.counts,
                                                              P.chunk, P.ntiles, err);
  chunk_scan_kernel<<<unsigned((nb + 31) / 32), kScanThreads, 0, st>>>(P.chunk, nchunks, nb, P.totals);
  digit_base_kernel<<<1, kThreads, 0, st>>>(P.totals, nb, P.digit_base, P.n_valid);
  const size_t smem = downsweep_smem_bytes<typename Src::Key>();
  set_smem(downsweep_kernel<Src, Dst>, smem);
  downsweep_kernel<Src, Dst><<<unsigned(P.ntiles), kThreads, smem, st>>>(src, dst, shift, bits, nb, P.digit_base,
                                                                         P.counts, P.chunk, P.ntiles, count_dev,
                                                                         count_host);
  *launches += 4;
}

// LSD sort of (uint32 key, uint32 value) pairs drawn from Src0 (the items of
// [0, count) that Src0::make accepts), by the low key_bits bits of the key,
// in passes of at most 10 bits.  Result: *out_k / *out_v, *n_valid entries
// (n_valid stays on the device).
// Digits of at most 10 bits (kMaxBins); when the key bits do not split evenly
// the wider digits go last: a key's high bits take fewer distinct values
// (rows < num_rows), so a wide high digit still has long runs per tile, while
// narrower low digits (uniformly spread) get longer runs than 10-bit ones.
struct SortPlan {
  int64_t count = 0;
  int key_bits = 1, passes = 1, nb = 2;  // nb: digit values of the widest pass
  SortPlan() = default;
  SortPlan(int64_t c, int kb) : count(c), key_bits(kb < 1 ? 1 : kb) {
    passes = (key_bits + 9) / 10;
    nb = 1 << bits(passes - 1);
  }
  int bits(int p) const {  // width of pass p
    const int base = key_bits / passes, extra = key_bits % passes;
    return base + (p >= passes - extra ? 1 : 0);
  }
  int shift(int p) const {
    int s = 0;
    for (int q = 0; q < p; ++q) s += bits(q);
    return s;
  }
  size_t bytes() const { return pass_ws_bytes(count, nb) + 4 * align_up(size_t(count) * sizeof(uint32_t)); }
};

struct SortWs {
  PassWs pass;
  uint32_t* k[2] = {nullptr, nullptr};
  uint32_t* v[2] = {nullptr, nullptr};
};

inline bool carve_sort_ws(const SortPlan& P, WsCursor& ws, SortWs& W) {
  if (!carve_pass_ws(P.count, P.nb, ws, W.pass)) return false;
  for (int i = 0; i < 2; ++i) {
    W.k[i] = ws.take<uint32_t>(size_t(P.count));
    W.v[i] = ws.take<uint32_t>(size_t(P.count));
  }
  return ws.ok;
}

// The ping-pong buffers that hold the result of run_sort (the last pass's output).
inline uint32_t* sorted_keys(const SortPlan& P, const SortWs& W) { return W.k[(P.passes - 1) & 1]; }
inline uint32_t* sorted_values(const SortPlan& P, const SortWs& W) { return W.v[(P.passes - 1) & 1]; }

template <class Src0>
fs_status run_sort(const Src0& src0, const SortPlan& P, const SortWs& W, int32_t* err, cudaStream_t st,
                   uint32_t** out_k, uint32_t** out_v, int* launches) {
  *out_k = sorted_keys(P, W);
  *out_v = sorted_values(P, W);
  if (P.count == 0) {
    if (cudaMemsetAsync(W.pass.n_valid, 0, sizeof(int64_t), st) != cudaSuccess) return FS_ERR_CUDA;
    return FS_OK;
  }
  for (int p = 0; p < P.passes; ++p) {
    DstU32 dst{W.k[p & 1], W.v[p & 1]};
    const int bits = P.bits(p), nb = 1 << bits;
    if (p == 0) {
      run_pass(src0, dst, 0, bits, nb, nullptr, P.count, W.pass, err, st, launches);
    } else {
      // later passes sort the n_valid items the first pass kept; n_valid is
      // rewritten with the same value by each pass
      SrcU32 s{W.k[(p - 1) & 1], W.v[(p - 1) & 1]};
      run_pass(s, dst, P.shift(p), bits, nb, W.pass.n_valid, P.count, W.pass, nullptr, st, launches);
    }
  }
  return launch_status();
}

}  // namespace radix
}  // namespace fs
