// Collision / exclusive row split between consecutive iterations.
// FreeScale (arXiv 2604.24073) Algorithm 2 line 10 (compute_collision on the
// shard-major I^i, I^{i+1}) and the notation paragraph after Algorithm 2.
//
// Rows are sets, so the split is computed on two presence bitmaps over the
// num_rows rows (R/8 bytes each: 12.5 MB for 100M rows, resident in the 129 MB
// L2):
//   1. mark: one pass over each ID array sets the row's bit (a load of the
//      bitmap word first, so hot rows that are already marked cost no atomic);
//   2. compact: one pass over the bitmap words with a decoupled look-back
//      scan of three popcounts (co = A&B, ex_t = A&~B, ex_next = B&~A); rows
//      come out ascending, i.e. shard-major, and the shard offsets fall out of
//      the same scan;
//   3. masks: one pass over each ID array tests the other iteration's bitmap.
#include "fs_common.cuh"

namespace fs {
namespace {

constexpr int kThreads = 256;
constexpr int kWordsPerThread = 2;  // 512 words (16384 rows) per compact tile: a 10M-row table gives 611 tiles
constexpr int kWordsPerTile = kThreads * kWordsPerThread;

__global__ void __launch_bounds__(kThreads) mark_kernel(const int64_t* ids_t, int64_t T_t, const int64_t* ids_next,
                                                        int64_t T_next, int64_t R, uint32_t* bm_t, uint32_t* bm_next,
                                                        int32_t* err) {
  const int64_t total = T_t + T_next;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const bool first = i < T_t;
    const int64_t id = first ? __ldcs(ids_t + i) : __ldcs(ids_next + (i - T_t));
    if (id < 0 || id >= R) {
      set_err(err, FS_ERR_ID_RANGE);
      continue;
    }
    uint32_t* bm = first ? bm_t : bm_next;
    const uint64_t w = uint64_t(id) >> 5;
    const uint32_t bit = 1u << (uint32_t(id) & 31u);
    if ((bm[w] & bit) == 0) atomicOr(bm + w, bit);
  }
}

// Row marking through a shared-memory window of the bitmap.  Block b takes
// the IDs [b * chunk, (b + 1) * chunk) in sub-chunks of kMarkSub; per
// sub-chunk the block finds the range of rows it touches, and when that range
// fits the window (kWinWords bitmap words: 409,600 rows) the bits are set in
// shared memory; the window's dirty words are OR-ed into the global bitmap
// only when a sub-chunk falls outside it, and at the end.  IDs in shard-major
// order (grouped by row range) stay inside one window for a whole shard, so
// the global bitmap sees one OR per dirty word instead of a load (and often
// an atomic) per ID.  A sub-chunk whose rows span more than the window is
// marked straight in global memory (load, then atomic where the bit is
// missing).  The result is the same set of bits either way.
constexpr int kMarkThreads = 256;
constexpr int kMarkItems = 8;  // per thread per sub-chunk; the next sub-chunk's 8 are in flight meanwhile
constexpr int kMarkSub = kMarkThreads * kMarkItems;
constexpr int kWinWords = 12800;  // 51.2 KB: four blocks per SM
constexpr size_t kMarkSmem = size_t(kWinWords) * sizeof(uint32_t);

__device__ __forceinline__ void block_min_max(uint32_t& lo, uint32_t& hi, uint32_t* s_lo, uint32_t* s_hi) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    s_lo[warp] = lo;
    s_hi[warp] = hi;
  }
  __syncthreads();
  lo = s_lo[0];
  hi = s_hi[0];
  for (int w = 1; w < nw; ++w) {
    lo = min(lo, s_lo[w]);
    hi = max(hi, s_hi[w]);
  }
  __syncthreads();  // s_lo / s_hi are free again
}

// Rows are below num_rows <= 2^32, so the per-ID work is 32-bit: an ID is
// checked once in 64 bits, then handled as its row; window positions are
// 32-bit word indices (rows / 32 < 2^27).
__global__ void __launch_bounds__(kMarkThreads, 4) mark_window_kernel(const int64_t* __restrict__ ids, int64_t T,
                                                                     int64_t chunk, int64_t R, uint32_t* bm,
                                                                     int32_t* err) {
  extern __shared__ uint32_t win[];  // [kWinWords]
  __shared__ uint32_t s_lo[kMarkThreads / 32], s_hi[kMarkThreads / 32];
  for (int j = threadIdx.x; j < kWinWords; j += kMarkThreads) win[j] = 0u;
  __syncthreads();
  const int64_t c0 = int64_t(blockIdx.x) * chunk;
  const int64_t c1 = (c0 + chunk < T) ? c0 + chunk : T;
  // block-uniform window state: base word (-1: no window), dirty words [dlo, dhi] relative to it
  int32_t base = -1, dlo = kWinWords, dhi = -1;
  auto flush = [&]() {
    if (base >= 0)
      for (int32_t w = dlo + int32_t(threadIdx.x); w <= dhi; w += kMarkThreads) {
        const uint32_t v = win[w];
        if (v) {
          atomicOr(bm + base + w, v);
          win[w] = 0u;
        }
      }
    dlo = kWinWords;
    dhi = -1;
  };
  int64_t nx[kMarkItems];  // the next sub-chunk's IDs, loaded while this one is marked
  auto load = [&](int64_t s0) {
    const int64_t* p = ids + s0 + threadIdx.x;
    const int64_t left = c1 - s0 - int64_t(threadIdx.x);  // this thread's items of the sub-chunk: i * kMarkThreads < left
#pragma unroll
    for (int i = 0; i < kMarkItems; ++i) nx[i] = int64_t(i) * kMarkThreads < left ? __ldcs(p + i * kMarkThreads) : -1;
  };
  if (c0 < c1) load(c0);
  for (int64_t s0 = c0; s0 < c1; s0 += kMarkSub) {
    uint32_t row[kMarkItems];
    unsigned ok = 0;  // bit i: item i is a valid ID
    uint32_t lo = 0xFFFFFFFFu, hi = 0;
    const int64_t left = c1 - s0 - int64_t(threadIdx.x);
#pragma unroll
    for (int i = 0; i < kMarkItems; ++i) {
      const int64_t id = nx[i];
      row[i] = uint32_t(id);
      if (id >= 0 && id < R) {
        ok |= 1u << i;
        lo = min(lo, row[i]);
        hi = max(hi, row[i]);
      } else if (int64_t(i) * kMarkThreads < left) {
        set_err(err, FS_ERR_ID_RANGE);
      }
    }
    if (s0 + kMarkSub < c1) load(s0 + kMarkSub);
    block_min_max(lo, hi, s_lo, s_hi);  // (also orders the previous sub-chunk's window updates before a flush)
    if (lo > hi) continue;              // no valid ID in this sub-chunk
    const int32_t lw = int32_t(lo >> 5), hw = int32_t(hi >> 5);
    if (!(base >= 0 && lw >= base && hw < base + kWinWords)) {
      flush();
      __syncthreads();
      // the new window leaves a quarter of its slack below this sub-chunk's rows and the rest
      // above (IDs grouped by row range move upwards), so later sub-chunks of the same range fit
      const int32_t slack = kWinWords - 1 - (hw - lw);
      base = slack >= 0 ? (lw - slack / 4 > 0 ? lw - slack / 4 : 0) : -1;
    }
    if (base >= 0) {
      // test before set: a Zipf-hot row's later IDs find their bit set and skip the atomic
      // (same-word shared atomics of one warp would serialize)
      uint32_t cur[kMarkItems];
#pragma unroll
      for (int i = 0; i < kMarkItems; ++i) cur[i] = (ok >> i) & 1u ? win[int32_t(row[i] >> 5) - base] : ~0u;
#pragma unroll
      for (int i = 0; i < kMarkItems; ++i) {
        const uint32_t bit = 1u << (row[i] & 31u);
        if ((cur[i] & bit) == 0) atomicOr(win + (int32_t(row[i] >> 5) - base), bit);
      }
      dlo = min(dlo, lw - base);
      dhi = max(dhi, hw - base);
    } else {
      // rows too spread for the window: every word loaded first, then an atomic where the bit
      // is missing (a stale word only costs a redundant atomic)
      uint32_t cur[kMarkItems];
#pragma unroll
      for (int i = 0; i < kMarkItems; ++i) cur[i] = (ok >> i) & 1u ? bm[row[i] >> 5] : ~0u;
#pragma unroll
      for (int i = 0; i < kMarkItems; ++i) {
        const uint32_t bit = 1u << (row[i] & 31u);
        if ((cur[i] & bit) == 0) atomicOr(bm + (row[i] >> 5), bit);
      }
    }
  }
  __syncthreads();
  flush();
}

// Blocks of the windowed mark: four per SM, each a contiguous chunk of the IDs.
void launch_mark_window(const int64_t* ids, int64_t T, int64_t R, uint32_t* bm, int32_t* err, cudaStream_t st) {
  if (T <= 0) return;
  int64_t grid = int64_t(sm_count()) * 4;
  int64_t chunk = (T + grid - 1) / grid;
  if (chunk < kMarkSub) chunk = kMarkSub;
  grid = (T + chunk - 1) / chunk;
  cudaFuncSetAttribute(mark_window_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kMarkSmem));
  mark_window_kernel<<<unsigned(grid), kMarkThreads, kMarkSmem, st>>>(ids, T, chunk, R, bm, err);
}

// Three counters packed in one 64-bit word, 21 bits each (a tile holds at most
// kWordsPerTile * 32 rows per counter).
__device__ __forceinline__ uint64_t pack3(uint32_t a, uint32_t b, uint32_t c) {
  return uint64_t(a) | (uint64_t(b) << 21) | (uint64_t(c) << 42);
}
__device__ __forceinline__ uint32_t unpack3(uint64_t v, int k) { return uint32_t((v >> (21 * k)) & 0x1FFFFFu); }

// Position of the r-th (0-based) set bit of w (w has more than r set bits):
// halves, quarters ... of the word chosen by population counts.
__device__ __forceinline__ int nth_set_bit(uint32_t w, int r) {
  int pos = 0;
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const int c = __popc(w & ((1u << half) - 1u));
    if (r >= c) {
      r -= c;
      w >>= half;
      pos += half;
    }
  }
  return pos;
}

__global__ void __launch_bounds__(kThreads) compact_kernel(const uint32_t* bm_t, const uint32_t* bm_next, int64_t nwords,
                                                           int64_t R, int32_t n, int64_t block, int64_t* co,
                                                           int64_t* ex_t, int64_t* ex_next, int64_t cap,
                                                           int64_t* counts, int64_t* co_off, int64_t* ex_t_off,
                                                           int64_t* ex_next_off, uint64_t* status, int* tile_counter,
                                                           int32_t* err, int64_t limit, int64_t skip_tile) {
  __shared__ uint64_t tmp[32];
  __shared__ int64_t s_tile;
  __shared__ int64_t s_excl[3];
  __shared__ uint32_t wpre[kWordsPerTile];   // per word of the tile: the list's set bits in earlier words
  __shared__ uint32_t wbits[kWordsPerTile];  // per word: the list's bits
  if (threadIdx.x == 0) s_tile = atomicAdd(tile_counter, 1);
  __syncthreads();
  const int64_t tile = s_tile;
  const int64_t tw0 = tile * kWordsPerTile;  // the tile's first word
  const int64_t w0 = tw0 + int64_t(threadIdx.x) * kWordsPerThread;
  uint32_t m[3][kWordsPerThread];
  uint32_t c[3] = {0, 0, 0};
#pragma unroll
  for (int i = 0; i < kWordsPerThread; ++i) {
    const int64_t w = w0 + i;
    uint32_t a = 0, b = 0;
    if (w < nwords) {
      a = bm_t[w];
      b = bm_next[w];
    }
    m[0][i] = a & b;
    m[1][i] = a & ~b;
    m[2][i] = b & ~a;
#pragma unroll
    for (int k = 0; k < 3; ++k) c[k] += __popc(m[k][i]);
  }
  uint64_t tot;
  uint64_t ex = block_exclusive_scan<uint64_t>(pack3(c[0], c[1], c[2]), tmp, &tot);
  if (tile == skip_tile) return;  // test hook: this tile never publishes
  const int warp = threadIdx.x >> 5;
  if (warp < 3) {
    uint64_t e = warp_lookback(status + warp, 3, tile, unpack3(tot, warp), err, limit);
    if ((threadIdx.x & 31) == 0) s_excl[warp] = int64_t(e);
  }
  __syncthreads();
  int64_t* lists[3] = {co, ex_t, ex_next};
  int64_t* offs[3] = {co_off, ex_t_off, ex_next_off};
  const int64_t row0 = tw0 * 32;                                           // the tile's first row
  const int64_t row_end = (tw0 + kWordsPerTile) * 32 < R ? (tw0 + kWordsPerTile) * 32 : R;
  const bool last_tile = tw0 + kWordsPerTile >= nwords;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    // words and their in-tile prefixes to shared memory
    uint32_t run = unpack3(ex, k);
#pragma unroll
    for (int i = 0; i < kWordsPerThread; ++i) {
      wpre[threadIdx.x * kWordsPerThread + i] = run;
      wbits[threadIdx.x * kWordsPerThread + i] = m[k][i];
      run += __popc(m[k][i]);
    }
    __syncthreads();
    const uint32_t cnt = unpack3(tot, k);
    const int64_t base = s_excl[k];
    int64_t* list = lists[k];
    // entry j of the tile's run of list k: the word holding it by binary search on the
    // prefixes, then its set bit by rank; consecutive threads write consecutive entries
    for (uint32_t j = threadIdx.x; j < cnt; j += kThreads) {
      int lo = 0, hi = kWordsPerTile - 1;  // the last word whose prefix is <= j
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (wpre[mid] <= j) lo = mid; else hi = mid - 1;
      }
      const int bit = nth_set_bit(wbits[lo], int(j - wpre[lo]));
      const int64_t at = base + j;
      if (at < cap) list[at] = row0 + int64_t(lo) * 32 + bit;
    }
    // shard boundaries s * block inside [row0, row_end): rows of the list below them
    const int64_t s_first = (row0 + block - 1) / block;
    for (int64_t s = s_first + threadIdx.x; s <= n && s * block < row_end; s += kThreads) {
      const int64_t rel = s * block - row0;
      const int wi = int(rel >> 5), below = int(rel & 31);
      offs[k][s] = base + wpre[wi] + __popc(wbits[wi] & ((below == 0) ? 0u : (0xFFFFFFFFu >> (32 - below))));
    }
    if (last_tile) {
      const int64_t total = base + cnt;
      if (threadIdx.x == 0) {
        counts[k] = total;
        if (total > cap) set_err(err, FS_ERR_CAPACITY);
      }
      // boundaries at or beyond R hold the full list length
      for (int64_t s = (R + block - 1) / block + threadIdx.x; s <= n; s += kThreads) offs[k][s] = total;
    }
    __syncthreads();  // wpre / wbits are rewritten for the next list
  }
}

__global__ void __launch_bounds__(kThreads) mask_kernel(const int64_t* ids_t, int64_t T_t, const int64_t* ids_next,
                                                        int64_t T_next, int64_t R, const uint32_t* bm_t,
                                                        const uint32_t* bm_next, uint8_t* is_co_t,
                                                        uint8_t* is_co_next) {
  const int64_t total = T_t + T_next;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const bool first = i < T_t;
    const int64_t j = first ? i : i - T_t;
    const int64_t id = first ? __ldcs(ids_t + j) : __ldcs(ids_next + j);
    const uint32_t* other = first ? bm_next : bm_t;
    uint8_t v = 0;
    if (id >= 0 && id < R) v = (__ldg(other + (uint64_t(id) >> 5)) >> (uint32_t(id) & 31u)) & 1u;
    if (first) is_co_t[j] = v; else is_co_next[j] = v;
  }
}

// Mask of one array only (the other mask was not requested).
__global__ void __launch_bounds__(kThreads) mask_one_kernel(const int64_t* ids, int64_t T, int64_t R,
                                                            const uint32_t* other, uint8_t* is_co) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; j < T; j += stride) {
    const int64_t id = __ldcs(ids + j);
    uint8_t v = 0;
    if (id >= 0 && id < R) v = (__ldg(other + (uint64_t(id) >> 5)) >> (uint32_t(id) & 31u)) & 1u;
    is_co[j] = v;
  }
}

struct CollLayout {
  int64_t nwords, tiles;
  size_t bitmap_bytes() const { return align_up(size_t(nwords) * sizeof(uint32_t)); }
  size_t zero_bytes() const { return 2 * bitmap_bytes() + align_up(size_t(tiles) * 3 * sizeof(uint64_t) + 256); }
};

CollLayout coll_layout(int64_t R) {
  CollLayout L;
  L.nwords = (R + 31) / 32;
  L.tiles = (L.nwords + kWordsPerTile - 1) / kWordsPerTile;
  if (L.tiles < 1) L.tiles = 1;
  return L;
}

unsigned grid_for(int64_t items) {
  int64_t g = (items + kThreads - 1) / kThreads, cap = int64_t(sm_count()) * 8;
  if (g > cap) g = cap;
  return unsigned(g < 1 ? 1 : g);
}

// compact + masks from two finished bitmaps; `status` ([tiles][3] words) and
// `counter` must be zero.  Returns the number of kernels launched.
int split_from_bitmaps(const int64_t* ids_t, int64_t T_t, const uint32_t* bm_t, const int64_t* ids_next,
                       int64_t T_next, const uint32_t* bm_next, int64_t num_rows, int32_t n, int64_t* co,
                       int64_t* ex_t, int64_t* ex_next, int64_t cap_rows, int64_t* counts, int64_t* co_shard_off,
                       int64_t* ex_t_shard_off, int64_t* ex_next_shard_off, uint8_t* is_co_t, uint8_t* is_co_next,
                       int32_t* err, uint64_t* status, int* counter, cudaStream_t st) {
  CollLayout L = coll_layout(num_rows);
  const int64_t block = (num_rows + n - 1) / n;
  int launches = 0;
  compact_kernel<<<unsigned(L.tiles), kThreads, 0, st>>>(bm_t, bm_next, L.nwords, num_rows, n, block, co, ex_t,
                                                         ex_next, cap_rows, counts, co_shard_off, ex_t_shard_off,
                                                         ex_next_shard_off, status, counter, err, spin_limit(),
                                                         debug_skip_tile());
  ++launches;
  // masks: either may be NULL (not wanted); then that pass over its IDs is skipped
  if (is_co_t && is_co_next && T_t + T_next > 0) {
    mask_kernel<<<grid_for(T_t + T_next), kThreads, 0, st>>>(ids_t, T_t, ids_next, T_next, num_rows, bm_t, bm_next,
                                                             is_co_t, is_co_next);
    ++launches;
  } else if (is_co_t && T_t > 0) {
    mask_one_kernel<<<grid_for(T_t), kThreads, 0, st>>>(ids_t, T_t, num_rows, bm_next, is_co_t);
    ++launches;
  } else if (is_co_next && T_next > 0) {
    mask_one_kernel<<<grid_for(T_next), kThreads, 0, st>>>(ids_next, T_next, num_rows, bm_t, is_co_next);
    ++launches;
  }
  return launches;
}

}  // namespace
}  // namespace fs

using namespace fs;

extern "C" size_t fs_collision_split_workspace_size(int64_t T_t, int64_t T_next, int64_t num_rows, int32_t n) {
  (void)T_t;
  (void)T_next;
  (void)n;
  if (num_rows < 1) return 0;
  return coll_layout(num_rows).zero_bytes() + 256;
}

extern "C" fs_status fs_collision_split(const int64_t* ids_t, int64_t T_t, const int64_t* ids_next, int64_t T_next,
                                        int64_t num_rows, int32_t n, int64_t* co, int64_t* ex_t, int64_t* ex_next,
                                        int64_t cap_rows, int64_t* counts, int64_t* co_shard_off,
                                        int64_t* ex_t_shard_off, int64_t* ex_next_shard_off, uint8_t* is_co_t,
                                        uint8_t* is_co_next, int32_t* err, void* ws, size_t ws_bytes,
                                        fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T_t < 0 || T_next < 0 || T_t > INT32_MAX || T_next > INT32_MAX || num_rows < 1 ||
      num_rows > (int64_t(1) << 32) || n < 1 || cap_rows < 0 || !counts || !co_shard_off || !ex_t_shard_off ||
      !ex_next_shard_off || !err)
    return FS_ERR_INVALID_ARG;
  if ((T_t > 0 && !ids_t) || (T_next > 0 && !ids_next)) return FS_ERR_INVALID_ARG;
  if (cap_rows > 0 && (!co || !ex_t || !ex_next)) return FS_ERR_INVALID_ARG;
  if ((ids_t && !aligned(ids_t, 8)) || (ids_next && !aligned(ids_next, 8)) || !aligned(counts, 8) ||
      (co && !aligned(co, 8)) || (ex_t && !aligned(ex_t, 8)) || (ex_next && !aligned(ex_next, 8)))
    return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_collision_split_workspace_size(T_t, T_next, num_rows, n) || !ws) return FS_ERR_WORKSPACE;

  CollLayout L = coll_layout(num_rows);
  WsCursor cur(ws, ws_bytes);
  unsigned char* zero = cur.take<unsigned char>(L.zero_bytes());
  if (!cur.ok) return FS_ERR_WORKSPACE;
  uint32_t* bm_t = reinterpret_cast<uint32_t*>(zero);
  uint32_t* bm_next = reinterpret_cast<uint32_t*>(zero + L.bitmap_bytes());
  unsigned char* tail = zero + 2 * L.bitmap_bytes();
  int* counter = reinterpret_cast<int*>(tail);
  uint64_t* status = reinterpret_cast<uint64_t*>(tail + 256);
  if (cudaMemsetAsync(zero, 0, L.zero_bytes(), st) != cudaSuccess) return FS_ERR_CUDA;

  int launches = 0;
  if (T_t + T_next > 0) {
    mark_kernel<<<grid_for(T_t + T_next), kThreads, 0, st>>>(ids_t, T_t, ids_next, T_next, num_rows, bm_t, bm_next,
                                                             err);
    ++launches;
  }
  launches += split_from_bitmaps(ids_t, T_t, bm_t, ids_next, T_next, bm_next, num_rows, n, co, ex_t, ex_next, cap_rows,
                                 counts, co_shard_off, ex_t_shard_off, ex_next_shard_off, is_co_t, is_co_next, err,
                                 status, counter, st);
  count_launch(launches);
  return launch_status();
}

extern "C" size_t fs_row_bitmap_words(int64_t num_rows) { return num_rows < 1 ? 0 : size_t((num_rows + 31) / 32); }

extern "C" fs_status fs_row_bitmap(const int64_t* ids, int64_t T, int64_t num_rows, uint32_t* bitmap, int32_t* err,
                                   fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T < 0 || T > INT32_MAX || num_rows < 1 || num_rows > (int64_t(1) << 32) || !bitmap || !err)
    return FS_ERR_INVALID_ARG;
  if (T > 0 && !ids) return FS_ERR_INVALID_ARG;
  if ((ids && !aligned(ids, 8)) || !aligned(bitmap, 4)) return FS_ERR_ALIGNMENT;
  if (cudaMemsetAsync(bitmap, 0, fs_row_bitmap_words(num_rows) * sizeof(uint32_t), st) != cudaSuccess)
    return FS_ERR_CUDA;
  if (T > 0) {
    launch_mark_window(ids, T, num_rows, bitmap, err, st);
    count_launch(1);
  }
  return launch_status();
}

extern "C" size_t fs_collision_split_bitmaps_workspace_size(int64_t num_rows) {
  if (num_rows < 1) return 0;
  CollLayout L = coll_layout(num_rows);
  return align_up(size_t(L.tiles) * 3 * sizeof(uint64_t) + 256) + 256;
}

extern "C" fs_status fs_collision_split_bitmaps(const int64_t* ids_t, int64_t T_t, const uint32_t* bm_t,
                                                const int64_t* ids_next, int64_t T_next, const uint32_t* bm_next,
                                                int64_t num_rows, int32_t n, int64_t* co, int64_t* ex_t,
                                                int64_t* ex_next, int64_t cap_rows, int64_t* counts,
                                                int64_t* co_shard_off, int64_t* ex_t_shard_off,
                                                int64_t* ex_next_shard_off, uint8_t* is_co_t, uint8_t* is_co_next,
                                                int32_t* err, void* ws, size_t ws_bytes, fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T_t < 0 || T_next < 0 || T_t > INT32_MAX || T_next > INT32_MAX || num_rows < 1 ||
      num_rows > (int64_t(1) << 32) || n < 1 || cap_rows < 0 || !counts || !co_shard_off || !ex_t_shard_off ||
      !ex_next_shard_off || !err || !bm_t || !bm_next)
    return FS_ERR_INVALID_ARG;
  if ((is_co_t && T_t > 0 && !ids_t) || (is_co_next && T_next > 0 && !ids_next)) return FS_ERR_INVALID_ARG;
  if (cap_rows > 0 && (!co || !ex_t || !ex_next)) return FS_ERR_INVALID_ARG;
  if ((ids_t && !aligned(ids_t, 8)) || (ids_next && !aligned(ids_next, 8)) || !aligned(counts, 8) ||
      !aligned(bm_t, 4) || !aligned(bm_next, 4) || (co && !aligned(co, 8)) || (ex_t && !aligned(ex_t, 8)) ||
      (ex_next && !aligned(ex_next, 8)))
    return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_collision_split_bitmaps_workspace_size(num_rows) || !ws) return FS_ERR_WORKSPACE;
  CollLayout L = coll_layout(num_rows);
  const size_t zb = align_up(size_t(L.tiles) * 3 * sizeof(uint64_t) + 256);
  unsigned char* zero = static_cast<unsigned char*>(ws);
  if (cudaMemsetAsync(zero, 0, zb, st) != cudaSuccess) return FS_ERR_CUDA;
  int* counter = reinterpret_cast<int*>(zero);
  uint64_t* status = reinterpret_cast<uint64_t*>(zero + 256);
  int launches = split_from_bitmaps(ids_t, T_t, bm_t, ids_next, T_next, bm_next, num_rows, n, co, ex_t, ex_next,
                                    cap_rows, counts, co_shard_off, ex_t_shard_off, ex_next_shard_off, is_co_t,
                                    is_co_next, err, status, counter, st);
  count_launch(launches);
  return launch_status();
}
