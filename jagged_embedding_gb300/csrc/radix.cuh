// Device-wide stable counting-sort passes (LSD radix sort, reduce-then-scan:
// Merrill & Grimshaw, "High Performance and Scalable Radix Sorting", 2011).
//
// One pass over the items of [0, count) keyed by one digit:
//   1. upsweep:    one block per chunk of 4 or 16 tiles of kTile items;
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
// and the digit function: fetch<kVal>(i) only loads (so that a tile's loads
// are all in flight together; the upsweep passes kVal = false and needs no
// value), fetch2<kVal>(raw) (kFetch2) the loads that depend on the first ones,
// make(raw, i, seg, key, val, err) checks and converts, digit(key, shift,
// bits, seg) gives the digit (seg: the tile's segment under a segment-aligned
// tiling, 0 otherwise).
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
// Tiles per counting (upsweep) block: 16, or 4 for passes of fewer than
// kSmallPassTiles tiles, so that a mid-size pass (a few thousand tiles) still
// gives every SM several blocks.  A pass's chunk size follows from its tile
// count alone (chunk_shift), so every kernel and workspace size of the pass
// agrees on it.
constexpr int64_t kSmallPassTiles = 16384;
constexpr int chunk_shift(int64_t ntiles) { return ntiles < kSmallPassTiles ? 2 : 4; }
constexpr int kPerT = kMaxBins / kThreads;  // digits per thread

constexpr int64_t num_tiles(int64_t count) { return (count + kTile - 1) / kTile; }
constexpr int64_t num_chunks(int64_t ntiles) {
  return (ntiles + (int64_t(1) << chunk_shift(ntiles)) - 1) >> chunk_shift(ntiles);
}


// Index, inside its tile, of item i of lane `lane` in warp `warp` (warp-striped,
// so a warp's slot i is 32 consecutive items; slot order = item order).
__device__ __forceinline__ int local_index(int warp, int i, int lane) { return warp * 32 * kItems + i * 32 + lane; }

// ------------------------------------------------------------------ tilings
// Which items a tile covers: [start, start + count), all in segment `seg`.
struct TileSpan {
  int64_t start;
  int32_t count;
  int32_t seg;
};

// Plain tiling: tile t covers items [t * kTile, (t + 1) * kTile) of [0, count);
// one segment; the downsweep adds digit_base[d] (the exclusive prefix of the
// digit totals) to every run of digit d.
struct PlainTiles {
  const int64_t* count_dev;  // item count on the device, or null: count_host
  int64_t count_host;
  const uint32_t* digit_base;
  __device__ __forceinline__ TileSpan span(int64_t t) const {
    const int64_t c = count_dev ? *count_dev : count_host;
    TileSpan r{t * kTile, 0, 0};
    if (r.start < c) r.count = int32_t(c - r.start < kTile ? c - r.start : kTile);
    return r;
  }
  __device__ __forceinline__ uint32_t base(int, int d) const { return __ldg(digit_base + d); }
};

// Segment-aligned tiling: the items are already grouped into nseg segments
// (segment s = items [seg_off[s], seg_off[s+1])), and the pass sorts each
// segment by the digit while keeping the segments apart.  Segment s owns tiles
// [tile_base[s], tile_base[s+1]) (ceil(size / kTile) of them), so no tile
// spans two segments.  Digits may carry a group in their top bits
// (d >> group_shift): the output is ordered by (group, segment, digit), which
// lets a key bit above the segment (the update's phase) move to the top in
// the same pass.  The downsweep adds seg_base[s][d] + group_base[g][s]:
// seg_base = (exclusive prefix of segment s's digit counts within the
// digit's group) - (global exclusive count of d over the tiles before the
// segment's first tile), group_base[g][s] = items of groups below g plus
// items of group g in segments below s (both written by seg_base_kernel and
// seg_offsets_kernel, modulo 2^32).
struct SegTiles {
  const int64_t* seg_off;     // [nseg + 1]
  const int64_t* tile_base;   // [nseg + 1]
  const int32_t* tile_seg;    // [tiles]: the tile's segment, -1 past the last (seg_map_kernel)
  const uint32_t* seg_base;   // [nseg][nb]
  const uint32_t* group_base; // [2][nseg]
  int32_t nseg;
  int32_t nb;
  int32_t group_shift;
  __device__ __forceinline__ TileSpan span(int64_t t) const {
    TileSpan r{0, 0, 0};
    const int s = __ldg(tile_seg + t);  // one load instead of a search over tile_base
    if (s < 0) return r;
    r.seg = s;
    r.start = __ldg(seg_off + s) + (t - __ldg(tile_base + s)) * kTile;
    const int64_t left = __ldg(seg_off + s + 1) - r.start;
    r.count = int32_t(left < kTile ? (left < 0 ? 0 : left) : kTile);
    return r;
  }
  __device__ __forceinline__ uint32_t base(int seg, int d) const {
    return __ldg(seg_base + size_t(seg) * nb + d) + __ldg(group_base + size_t(d >> group_shift) * nseg + seg);
  }
};

// ------------------------------------------------------------------ upsweep
// Block c: tiles [c << cshift, (c + 1) << cshift) one after another.  Per tile, one
// block-wide histogram (all item loads issued first, then one shared-memory
// increment per item); counts[tile][d] = this chunk's count of d before the
// tile; chunk_sums[c][d] = the chunk's count of d.  Empty tiles count nothing
// but still write their counts.
template <class Src, class Tiles>
__global__ void __launch_bounds__(kThreads) upsweep_kernel(Src src, Tiles tiles, int shift, int bits, int nb,
                                                           uint32_t* counts, uint32_t* chunk_sums, int64_t ntiles,
                                                           int cshift, int32_t* err) {
  __shared__ uint32_t hist[kMaxBins];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t chunk = blockIdx.x;
  uint32_t run[kPerT];
#pragma unroll
  for (int j = 0; j < kPerT; ++j) run[j] = 0;
  for (int c = 0; c < (1 << cshift); ++c) {
    const int64_t tile = (chunk << cshift) + c;
    if (tile >= ntiles) break;
    const TileSpan sp = tiles.span(tile);
    for (int j = threadIdx.x; j < nb; j += kThreads) hist[j] = 0;
    __syncthreads();
    if (sp.count > 0) {
      typename Src::Raw raw[kItems];
#pragma unroll
      for (int i = 0; i < kItems; ++i) {
        const int l = local_index(warp, i, lane);
        if (l < sp.count) raw[i] = src.template fetch<false>(sp.start + l);
      }
      if constexpr (Src::kFetch2) {  // loads that depend on the first ones, all issued together
#pragma unroll
        for (int i = 0; i < kItems; ++i)
          if (local_index(warp, i, lane) < sp.count) src.template fetch2<false>(raw[i]);
      }
#pragma unroll
      for (int i = 0; i < kItems; ++i) {
        const int l = local_index(warp, i, lane);
        typename Src::Key k;
        uint32_t v;
        if (l < sp.count && src.make(raw[i], sp.start + l, sp.seg, k, v, err))
          atomicAdd(hist + src.digit(k, shift, bits, sp.seg), 1u);
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
  // (both walks over a warp's chunks keep 8 loads in flight: the chunk counts
  // sit in L2, and one dependent load per chunk would set the pace)
  constexpr int kB = 8;
  uint32_t s = 0;
  if (d < nb) {
    int64_t c = c0;
    for (; c + kB <= c1; c += kB) {
      uint32_t v[kB];
#pragma unroll
      for (int k = 0; k < kB; ++k) v[k] = chunk_sums[(c + k) * nb + d];
#pragma unroll
      for (int k = 0; k < kB; ++k) s += v[k];
    }
    for (; c < c1; ++c) s += chunk_sums[c * nb + d];
  }
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
  if (d < nb) {
    int64_t c = c0;
    for (; c + kB <= c1; c += kB) {
      uint32_t v[kB];
#pragma unroll
      for (int k = 0; k < kB; ++k) v[k] = chunk_sums[(c + k) * nb + d];
#pragma unroll
      for (int k = 0; k < kB; ++k) {
        chunk_sums[(c + k) * nb + d] = run;
        run += v[k];
      }
    }
    for (; c < c1; ++c) {
      const uint32_t v = chunk_sums[c * nb + d];
      chunk_sums[c * nb + d] = run;
      run += v;
    }
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
// Block shape of the downsweep: kDownThreads threads, kDownItems items each
// (one tile of kTile items).  Measured alternatives (512 threads x 8 items,
// 16-bit warp counts) were no faster on the large-table passes.
constexpr int kDownThreads = kThreads;
constexpr int kDownItems = kTile / kDownThreads;
constexpr int kDownWarps = kDownThreads / 32;
constexpr int kDownPerT = kMaxBins / kDownThreads;  // digits per thread
static_assert(kDownThreads * kDownItems == kTile && kDownPerT >= 1, "downsweep shape");
using HistT = uint32_t;
constexpr int kBallotMaxBits = 8;  // widest digit the multisplit matches by ballots

// Index, inside its tile, of the downsweep's item i of lane `lane` in warp `warp`.
__device__ __forceinline__ int down_index(int warp, int i, int lane) { return warp * 32 * kDownItems + i * 32 + lane; }

// Shared memory: the per-warp digit counts during ranking, then (same space)
// the staged keys and values in tile order; behind them the tile's digit
// counts (later each run's output offset minus its tile-local start), the
// tile-local starts of the runs, and scan scratch.
template <class KeyT>
constexpr size_t downsweep_smem_bytes() {
  size_t stage = size_t(kTile) * (sizeof(KeyT) + sizeof(uint32_t));
  size_t hist = size_t(kDownWarps) * kMaxBins * sizeof(HistT);
  size_t un = stage > hist ? stage : hist;
  return un + 2 * kMaxBins * sizeof(uint32_t) + 64 * sizeof(uint32_t);
}

// Resident blocks per SM the downsweep is compiled for (its register budget:
// 64 registers a thread at 4, 85 at 3): a source may set kMinBlocks; the
// default 4 fits the 40 KB of shared memory of 32-bit keys.
template <class Src, class = void>
struct DownBlocks {
  static constexpr int value = 4;
};
template <class Src>
struct DownBlocks<Src, decltype(void(Src::kMinBlocks))> {
  static constexpr int value = Src::kMinBlocks;
};

template <class Src, class Dst, class Tiles>
__global__ void __launch_bounds__(kDownThreads, DownBlocks<Src>::value) downsweep_kernel(Src src, Dst dst, Tiles tiles,
                                                                                     int shift, int bits, int nb,
                                                                                     const uint32_t* counts,
                                                                                     const uint32_t* chunk_base,
                                                                                     int cshift) {
  using KeyT = typename Src::Key;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  HistT* warp_hist = reinterpret_cast<HistT*>(smem_raw);  // [kDownWarps][nb] (ranking)
  KeyT* stage_k = reinterpret_cast<KeyT*>(smem_raw);      // [kTile]          (staging)
  constexpr size_t stage_bytes = size_t(kTile) * (sizeof(KeyT) + sizeof(uint32_t));
  constexpr size_t hist_bytes = size_t(kDownWarps) * kMaxBins * sizeof(HistT);
  constexpr size_t un = stage_bytes > hist_bytes ? stage_bytes : hist_bytes;
  uint32_t* stage_v = reinterpret_cast<uint32_t*>(smem_raw + size_t(kTile) * sizeof(KeyT));
  uint32_t* run_off = reinterpret_cast<uint32_t*>(smem_raw + un);  // tile counts, then output offset - local start
  uint32_t* local_start = run_off + kMaxBins;
  uint32_t* scratch = local_start + kMaxBins;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t tile = blockIdx.x;
  const TileSpan sp = tiles.span(tile);
  if (sp.count <= 0) return;

  // this tile's offset inside every digit run: loaded first, so that these
  // reads overlap the item loads and the ranking below
  uint32_t my_off[kDownPerT];
#pragma unroll
  for (int i = 0; i < kDownPerT; ++i) {
    const int d = threadIdx.x + i * kDownThreads;
    my_off[i] = d < nb ? __ldg(counts + tile * nb + d) + __ldg(chunk_base + (tile >> cshift) * nb + d) +
                             tiles.base(sp.seg, d)
                       : 0u;
  }

  // per item: the key, one packed word (digit in bits 20..31, rank / local
  // position in bits 0..19) and, only for sources whose value is not the item
  // index, the value
  KeyT key[kDownItems];
  uint32_t val[Src::kIndexValue ? 1 : kDownItems];
  uint32_t pk[kDownItems];
  constexpr uint32_t kSkipPk = 0xFFF00000u;
  {
    typename Src::Raw raw[kDownItems];
#pragma unroll
    for (int i = 0; i < kDownItems; ++i) {
      const int l = down_index(warp, i, lane);
      if (l < sp.count) raw[i] = src.template fetch<true>(sp.start + l);
    }
    if constexpr (Src::kFetch2) {
#pragma unroll
      for (int i = 0; i < kDownItems; ++i)
        if (down_index(warp, i, lane) < sp.count) src.template fetch2<true>(raw[i]);
    }
#pragma unroll
    for (int i = 0; i < kDownItems; ++i) {
      const int l = down_index(warp, i, lane);
      uint32_t v = 0;
      const bool ok = l < sp.count && src.make(raw[i], sp.start + l, sp.seg, key[i], v, nullptr);
      if constexpr (!Src::kIndexValue) val[i] = v;
      pk[i] = ok ? (src.digit(key[i], shift, bits, sp.seg) << 20) : kSkipPk;
    }
  }
  for (int j = threadIdx.x; j < kDownWarps * nb; j += kDownThreads) warp_hist[j] = 0u;
  __syncthreads();

  // warp-level multisplit, slot by slot (slot order = item order)
  HistT* wh = warp_hist + warp * nb;
  // lanes with the same digit: for digits of at most 8 bits one ballot per
  // digit bit (faster there than match.any: the 256-shard bucketize pass
  // 3.36 -> 3.07 ms on 303M IDs), wider digits by match.any (10-bit passes
  // were slower with ballots)
  const int dbits = nb > 1 ? 32 - __clz(nb - 1) : 1;  // every digit is below nb
  const bool by_ballot = dbits <= kBallotMaxBits;
#pragma unroll
  for (int i = 0; i < kDownItems; ++i) {
    const uint32_t d = pk[i] >> 20;
    const bool skip = pk[i] == kSkipPk;
    unsigned peers;
    if (by_ballot) {
      const unsigned sk = __ballot_sync(0xffffffffu, skip);  // skipped items match each other only
      peers = skip ? sk : ~sk;
      // all kBallotMaxBits bits, unrolled: a kept digit is below nb, so its
      // bits from dbits up are zero, and those ballots change no kept lane's
      // peers (the skip ballot already set the skipped lanes apart)
#pragma unroll
      for (int b = 0; b < kBallotMaxBits; ++b) {
        const bool on = (d >> b) & 1u;
        const unsigned m = __ballot_sync(0xffffffffu, on);
        peers &= on ? m : ~m;
      }
    } else {
      peers = __match_any_sync(0xffffffffu, pk[i]);
    }
    const unsigned lt = __popc(peers & lanemask_lt());
    const uint32_t b = skip ? 0u : uint32_t(wh[d]);
    if (!skip) pk[i] |= b + lt;
    __syncwarp();
    if (!skip && lt == 0) wh[d] = HistT(b + __popc(peers));
    __syncwarp();
  }
  __syncthreads();

  // exclusive over warps per digit, tile totals
#pragma unroll
  for (int i = 0; i < kDownPerT; ++i) {
    const int d = threadIdx.x + i * kDownThreads;
    if (d < nb) {
      uint32_t run = 0;
#pragma unroll
      for (int w = 0; w < kDownWarps; ++w) {
        const uint32_t c = warp_hist[w * nb + d];
        warp_hist[w * nb + d] = HistT(run);
        run += c;
      }
      run_off[d] = run;
    }
  }
  __syncthreads();
  {
    constexpr int kPer = kMaxBins / kDownThreads;  // digits per thread
    const int d0 = threadIdx.x * kPer;
    uint32_t v[kPer], sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      v[i] = d0 + i < nb ? run_off[d0 + i] : 0u;
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
  // each run's output position minus its tile-local start: staged item j of
  // digit d goes to run_off[d] + j (positions < 2^31, exact modulo 2^32)
#pragma unroll
  for (int i = 0; i < kDownPerT; ++i) {
    const int d = threadIdx.x + i * kDownThreads;
    if (d < nb) run_off[d] = my_off[i] - local_start[d];
  }
#pragma unroll
  for (int i = 0; i < kDownItems; ++i)
    if (pk[i] != kSkipPk) {
      const uint32_t d = pk[i] >> 20;
      pk[i] = (d << 20) | (local_start[d] + uint32_t(warp_hist[warp * nb + d]) + (pk[i] & 0xFFFFFu));  // tile-local position
    }
  const uint32_t nvalid = scratch[40];
  __syncthreads();  // warp_hist is dead; its space becomes the staging area
#pragma unroll
  for (int i = 0; i < kDownItems; ++i)
    if (pk[i] != kSkipPk) {
      const uint32_t at = pk[i] & 0xFFFFFu;
      stage_k[at] = key[i];
      if constexpr (Src::kIndexValue)  // digit and tile-local index: no digit to recompute below
        stage_v[at] = ((pk[i] >> 20) << 12) | uint32_t(down_index(warp, i, lane));
      else
        stage_v[at] = val[i];
    }
  __syncthreads();
  for (uint32_t j = threadIdx.x; j < nvalid; j += kDownThreads) {
    const KeyT k = stage_k[j];
    const uint32_t sv = stage_v[j];
    if constexpr (Src::kIndexValue) {
      dst.store(int64_t(run_off[sv >> 12] + j), k, uint32_t(sp.start + (sv & 0xFFFu)));
    } else {
      dst.store(int64_t(run_off[src.digit(k, shift, bits, sp.seg)] + j), k, sv);
    }
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
  // the upsweep needs only the key (kVal false): the value is not loaded
  template <bool kVal>
  __device__ __forceinline__ Raw fetch(int64_t i) const { return make_uint2(__ldcs(k + i), kVal ? __ldcs(v + i) : 0u); }
  __device__ __forceinline__ bool make(const Raw& r, int64_t, int, Key& key, uint32_t& val, int32_t*) const {
    key = r.x;
    val = r.y;
    return true;
  }
  __device__ __forceinline__ uint32_t digit(Key key, int shift, int bits, int) const {
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

constexpr size_t pass_ws_bytes(int64_t count, int nb) {
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
  const PlainTiles tiles{count_dev, count_host, P.digit_base};
  const int cs = chunk_shift(P.ntiles);
  upsweep_kernel<Src, PlainTiles><<<unsigned(nchunks), kThreads, 0, st>>>(src, tiles, shift, bits, nb, P.counts,
                                                                          P.chunk, P.ntiles, cs, err);
  chunk_scan_kernel<<<unsigned((nb + 31) / 32), kScanThreads, 0, st>>>(P.chunk, nchunks, nb, P.totals);
  digit_base_kernel<<<1, kThreads, 0, st>>>(P.totals, nb, P.digit_base, P.n_valid);
  const size_t smem = downsweep_smem_bytes<typename Src::Key>();
  set_smem(downsweep_kernel<Src, Dst, PlainTiles>, smem);
  downsweep_kernel<Src, Dst, PlainTiles><<<unsigned(P.ntiles), kDownThreads, smem, st>>>(src, dst, tiles, shift, bits, nb,
                                                                                     P.counts, P.chunk, cs);
  *launches += 4;
}

// ------------------------------------------------------------------ segment-aligned passes
// Passes that sort every segment of an array already grouped into segments
// (the update's sort of shard-major IDs: one segment per shard), under
// SegTiles.  One pass = seg_map_kernel (each tile's segment), upsweep, chunk
// scan, seg_base_kernel (the digit bases of every segment), seg_offsets_kernel
// (the group bases, and the segments and tiles of the pass's output for the
// next pass), downsweep.
constexpr int kSegThreads = 1024;  // segments handled by one block: nseg <= kSegThreads

// Segment offsets of the input, made safe to tile: seg_off[s] = the running
// maximum of in[0..s] clamped to [0, count], seg_off[0] = 0, seg_off[nseg] =
// count (an input that breaks these rules sets FS_ERR_BAD_OFFSETS);
// tile_base[s] = tiles of the segments before s (ceil(size / kTile) each).
static __global__ void __launch_bounds__(kSegThreads) seg_tiles_kernel(const int64_t* in, int32_t nseg, int64_t count,
                                                                      int64_t* seg_off, int64_t* tile_base,
                                                                      int32_t* err) {
  __shared__ int64_t off[kSegThreads + 1];
  __shared__ int64_t tmp[32];
  for (int s = threadIdx.x; s <= nseg; s += blockDim.x) off[s] = in[s];
  __syncthreads();
  if (threadIdx.x == 0) {
    bool bad = off[0] != 0 || off[nseg] != count;
    int64_t run = 0;
    for (int s = 0; s <= nseg; ++s) {
      int64_t v = off[s] < 0 ? 0 : (off[s] > count ? count : off[s]);
      if (off[s] < run) bad = true;
      run = v > run ? v : run;
      off[s] = (s == 0) ? 0 : (s == nseg ? count : run);
    }
    if (bad) set_err(err, FS_ERR_BAD_OFFSETS);
  }
  __syncthreads();
  const int s = threadIdx.x;
  const int64_t n = s < nseg ? (off[s + 1] - off[s] + kTile - 1) / kTile : 0;
  int64_t total;
  const int64_t before = block_exclusive_scan<int64_t>(n, tmp, &total);
  if (s < nseg) {
    seg_off[s] = off[s];
    tile_base[s] = before;
  }
  if (s == 0) {
    seg_off[nseg] = count;
    tile_base[nseg] = total;
  }
}

// Per segment s (one block each): H[d] = global exclusive count of digit d
// over the tiles before the segment's first tile (the totals when it has
// none), the segment's digit counts c[d] = H_{s+1}[d] - H_s[d], their
// exclusive prefix within each group (groups: d >> group_shift, at most two),
// seg_base[s][d] = that prefix - H_s[d] (mod 2^32) and gtot[s][g] = the
// segment's items in group g.
static __global__ void __launch_bounds__(kThreads) seg_base_kernel(const uint32_t* counts, const uint32_t* chunk_base,
                                                              const uint32_t* totals, const int64_t* tile_base,
                                                              int32_t nseg, int nb, int group_shift, int cshift,
                                                              uint32_t* seg_base, uint32_t* gtot) {
  __shared__ uint32_t tmp[32];
  __shared__ uint32_t g0;
  const int s = blockIdx.x;
  const int64_t tiles = tile_base[nseg];
  const int64_t f0 = tile_base[s], f1 = tile_base[s + 1];
  auto G = [&](int64_t f, int d) -> uint32_t {
    return f < tiles ? counts[f * nb + d] + chunk_base[(f >> cshift) * nb + d] : totals[d];
  };
  constexpr int kPer = kMaxBins / kThreads;
  const int d0 = threadIdx.x * kPer;  // contiguous digits per thread: the scan runs in digit order
  const int gsize = 1 << group_shift;
  uint32_t h[kPer], c[kPer], sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int d = d0 + i;
    h[i] = d < nb ? G(f0, d) : 0u;
    c[i] = d < nb ? G(f1, d) - h[i] : 0u;
    sum += c[i];
  }
  if (threadIdx.x == 0) g0 = 0;
  uint32_t tot;
  uint32_t run = block_exclusive_scan<uint32_t>(sum, tmp, &tot);  // (ends with a barrier)
  uint32_t ex[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    ex[i] = run;
    if (d0 + i == gsize) g0 = run;  // items of group 0 (digits below gsize)
    run += c[i];
  }
  __syncthreads();
  const uint32_t g0tot = gsize < nb ? g0 : tot;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int d = d0 + i;
    if (d < nb) seg_base[size_t(s) * nb + d] = ex[i] - (d >= gsize ? g0tot : 0u) - h[i];
  }
  if (threadIdx.x == 0) {
    gtot[2 * s] = g0tot;
    gtot[2 * s + 1] = tot - g0tot;
  }
}

// One block of kSegThreads threads: group_base[g][s] = items of the groups
// below g plus items of group g in the segments below s; the output's
// segments (next_seg_off: the segments' valid items, in segment order) and
// their first tiles (next_tile_base) for the next pass; *n_valid = all valid
// items, *n_first = items of group 0 (when n_first is not null).
static __global__ void __launch_bounds__(kSegThreads) seg_offsets_kernel(const uint32_t* gtot, int32_t nseg,
                                                                        uint32_t* group_base, int64_t* next_seg_off,
                                                                        int64_t* next_tile_base, int64_t* n_valid,
                                                                        int64_t* n_first) {
  __shared__ int64_t tmp[32];
  const int s = threadIdx.x;
  const int64_t a = s < nseg ? int64_t(gtot[2 * s]) : 0, b = s < nseg ? int64_t(gtot[2 * s + 1]) : 0;
  int64_t ta, tb, tt;
  const int64_t ea = block_exclusive_scan<int64_t>(a, tmp, &ta);
  const int64_t eb = block_exclusive_scan<int64_t>(b, tmp, &tb);
  const int64_t et = block_exclusive_scan<int64_t>((a + b + kTile - 1) / kTile, tmp, &tt);
  if (s < nseg) {
    group_base[s] = uint32_t(ea);
    group_base[nseg + s] = uint32_t(ta + eb);
    next_seg_off[s] = ea + eb;
    next_tile_base[s] = et;
  }
  if (s == 0) {
    next_seg_off[nseg] = ta + tb;
    next_tile_base[nseg] = tt;
    *n_valid = ta + tb;
    if (n_first) *n_first = ta;
  }
}

// tile_seg[t] = the segment owning tile t of a segment-aligned tiling (the
// last segment whose first tile is <= t, so empty segments own none), -1 for
// tiles past the last segment's; the search runs over tile_base staged in
// shared memory, so the passes' tiles find their segment with one load.
static __global__ void __launch_bounds__(kSegThreads) seg_map_kernel(const int64_t* tile_base, int32_t nseg,
                                                                    int64_t max_tiles, int32_t* tile_seg) {
  __shared__ int64_t tb[kSegThreads + 1];
  for (int s = threadIdx.x; s <= nseg; s += blockDim.x) tb[s] = tile_base[s];
  __syncthreads();
  const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= max_tiles) return;
  if (t >= tb[nseg]) {
    tile_seg[t] = -1;
    return;
  }
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tb[mid] <= t) lo = mid; else hi = mid - 1;
  }
  tile_seg[t] = lo;
}

// Scratch of the segment-aligned passes over up to `count` items in nseg segments.
struct SegWs {
  int32_t nseg = 0;
  int64_t max_tiles = 0;
  uint32_t* counts = nullptr;      // [max_tiles][kMaxBins]
  uint32_t* chunk = nullptr;       // [chunks][kMaxBins]
  uint32_t* totals = nullptr;      // [kMaxBins]
  uint32_t* seg_base = nullptr;    // [nseg][kMaxBins]
  uint32_t* gtot = nullptr;        // [nseg][2]
  uint32_t* group_base = nullptr;  // [2][nseg]
  int64_t* seg_off[2] = {nullptr, nullptr};    // [nseg + 1] each: a pass's input segments
  int64_t* tile_base[2] = {nullptr, nullptr};  // [nseg + 1] each
  int32_t* tile_seg = nullptr;                 // [max_tiles]: the current pass's tile -> segment map
};

constexpr int64_t seg_max_tiles(int64_t count, int32_t nseg) { return num_tiles(count) + nseg; }

template <class Ws>
inline void take_seg_ws(int64_t count, int32_t nseg, Ws& ws, SegWs* W) {
  const int64_t mt = seg_max_tiles(count, nseg);
  uint32_t* c = ws.template take<uint32_t>(size_t(mt) * kMaxBins);
  uint32_t* ch = ws.template take<uint32_t>(size_t(num_chunks(mt)) * kMaxBins);
  uint32_t* tot = ws.template take<uint32_t>(kMaxBins);
  uint32_t* sb = ws.template take<uint32_t>(size_t(nseg) * kMaxBins);
  uint32_t* gt = ws.template take<uint32_t>(size_t(nseg) * 2);
  uint32_t* gb = ws.template take<uint32_t>(size_t(nseg) * 2);
  int64_t* so0 = ws.template take<int64_t>(size_t(nseg) + 1);
  int64_t* so1 = ws.template take<int64_t>(size_t(nseg) + 1);
  int64_t* tb0 = ws.template take<int64_t>(size_t(nseg) + 1);
  int64_t* tb1 = ws.template take<int64_t>(size_t(nseg) + 1);
  int32_t* ts = ws.template take<int32_t>(size_t(mt));
  if (W) {
    W->nseg = nseg;
    W->max_tiles = mt;
    W->counts = c;
    W->chunk = ch;
    W->totals = tot;
    W->seg_base = sb;
    W->gtot = gt;
    W->group_base = gb;
    W->seg_off[0] = so0;
    W->seg_off[1] = so1;
    W->tile_base[0] = tb0;
    W->tile_base[1] = tb1;
    W->tile_seg = ts;
  }
}

// One segment-aligned pass reading the segments in slot `in` (seg_off[in],
// tile_base[in]) and writing the next pass's segments to the other slot.
// Digit of `bits` bits, of which the bits from group_shift up are the group.
template <class Src, class Dst>
void run_seg_pass(const Src& src, const Dst& dst, int shift, int bits, int group_shift, const SegWs& W, int in,
                  int64_t* n_valid, int64_t* n_first, int32_t* err, cudaStream_t st, int* launches) {
  const int nb = 1 << bits;
  const SegTiles tiles{W.seg_off[in], W.tile_base[in], W.tile_seg, W.seg_base, W.group_base, W.nseg, nb, group_shift};
  const int64_t nchunks = num_chunks(W.max_tiles);
  const int cs = chunk_shift(W.max_tiles);
  seg_map_kernel<<<unsigned((W.max_tiles + kSegThreads - 1) / kSegThreads), kSegThreads, 0, st>>>(
      W.tile_base[in], W.nseg, W.max_tiles, W.tile_seg);
  upsweep_kernel<Src, SegTiles><<<unsigned(nchunks), kThreads, 0, st>>>(src, tiles, shift, bits, nb, W.counts,
                                                                        W.chunk, W.max_tiles, cs, err);
  chunk_scan_kernel<<<unsigned((nb + 31) / 32), kScanThreads, 0, st>>>(W.chunk, nchunks, nb, W.totals);
  seg_base_kernel<<<unsigned(W.nseg), kThreads, 0, st>>>(W.counts, W.chunk, W.totals, W.tile_base[in], W.nseg, nb,
                                                          group_shift, cs, W.seg_base, W.gtot);
  seg_offsets_kernel<<<1, kSegThreads, 0, st>>>(W.gtot, W.nseg, W.group_base, W.seg_off[1 - in],
                                                W.tile_base[1 - in], n_valid, n_first);
  const size_t smem = downsweep_smem_bytes<typename Src::Key>();
  set_smem(downsweep_kernel<Src, Dst, SegTiles>, smem);
  downsweep_kernel<Src, Dst, SegTiles><<<unsigned(W.max_tiles), kDownThreads, smem, st>>>(src, dst, tiles, shift, bits, nb,
                                                                                      W.counts, W.chunk, cs);
  *launches += 6;
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
  constexpr SortPlan() = default;
  constexpr SortPlan(int64_t c, int kb)
      : count(c), key_bits(kb < 1 ? 1 : kb), passes(((kb < 1 ? 1 : kb) + 9) / 10), nb(0) {
    nb = 1 << bits(passes - 1);
  }
  constexpr int bits(int p) const {  // width of pass p
    const int base = key_bits / passes, extra = key_bits % passes;
    return base + (p >= passes - extra ? 1 : 0);
  }
  constexpr int shift(int p) const {
    int s = 0;
    for (int q = 0; q < p; ++q) s += bits(q);
    return s;
  }
  constexpr size_t bytes() const {
    return pass_ws_bytes(count, nb) + 4 * align_up(size_t(count) * sizeof(uint32_t));
  }
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
