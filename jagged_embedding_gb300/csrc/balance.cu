// Sequence load balancing: FBS and VBS partitions.
// FreeScale (arXiv 2604.24073) §4.1 "Partitioning Algorithms"; §3.1 /
// Algorithm 1 (a deterministic partition function over the gathered lengths).
//
// Both partitions start from the samples ordered by (UIH length, global
// index): a stable LSD radix sort of the lengths with the index as value
// (reduce-then-scan counting passes).  FBS then deals sorted positions to ranks in snake order
// with a closed form per position; VBS scans fixed-point weights L^alpha with
// a single-pass decoupled look-back scan and cuts the prefix into n segments.
#include <mutex>

#include "radix.cuh"

namespace fs {
namespace {

using radix::kThreads;

// Length array as a sort source: key = L[g] (negative lengths flagged), value = g.
struct SrcLen {
  using Key = uint32_t;
  static constexpr bool kIndexValue = true;  // value = item index
  const int32_t* L;
  static constexpr bool kFetch2 = false;
  using Raw = int32_t;
  template <bool>
  __device__ __forceinline__ Raw fetch(int64_t i) const { return L[i]; }
  __device__ __forceinline__ bool make(Raw l, int64_t i, int, Key& key, uint32_t& val, int32_t* err) const {
    if (l < 0) {
      if (err) set_err(err, FS_ERR_INVALID_ARG);
      l = 0;
    }
    key = static_cast<uint32_t>(l);
    val = static_cast<uint32_t>(i);
    return true;
  }
  __device__ __forceinline__ uint32_t digit(Key key, int shift, int bits, int) const {
    return (key >> shift) & ((1u << bits) - 1u);
  }
};

// rank_offsets of the snake deal: F = S / n full rounds, rem = S % n samples in
// the last round, dealt left to right when F is even, right to left when odd.
__device__ __forceinline__ int64_t fbs_rank_offset(int64_t r, int64_t S, int64_t n) {
  const int64_t F = S / n, rem = S % n;
  int64_t extra_before;
  if ((F & 1) == 0) {
    extra_before = r < rem ? r : rem;                      // ranks 0..rem-1 get one more
  } else {
    int64_t first = n - rem;                               // ranks n-rem..n-1 get one more
    extra_before = r > first ? r - first : 0;
  }
  return r * F + extra_before;
}

__global__ void fbs_assign_kernel(const uint32_t* sorted_g, int64_t S, int32_t n, int32_t* perm,
                                  int64_t* rank_offsets) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t p = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; p < S; p += stride) {
    const int64_t rho = p / n, k = p % n;
    const int64_t r = (rho & 1) ? (n - 1 - k) : k;
    perm[fbs_rank_offset(r, S, n) + rho] = static_cast<int32_t>(sorted_g[p]);
  }
  for (int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; r <= n; r += stride)
    rank_offsets[r] = fbs_rank_offset(r, S, n);
}

// FBS of up to kFbsSmallMax samples in one block of 1024 threads: the (L, g)
// keys stay in registers and shared memory, and the stable LSD passes (8-bit
// digits, as many as the largest length needs: two for lengths below 65536)
// run inside the block, then the snake deal.  Same sorted order as the
// device-wide passes (a stable sort by L, ties by g), so the same perm.
constexpr int kFbsSmallThreads = 1024;
constexpr int kFbsSmallItems = 16;
constexpr int kFbsSmallMax = kFbsSmallThreads * kFbsSmallItems;  // 16384
constexpr int kFbsSmallWarps = kFbsSmallThreads / 32;
constexpr size_t kFbsSmallSmem = (2 * size_t(kFbsSmallMax) + size_t(kFbsSmallWarps) * 256 + 256 + 64) * sizeof(uint32_t);

__global__ void __launch_bounds__(kFbsSmallThreads, 1) fbs_small_kernel(const int32_t* L, int32_t S, int32_t n,
                                                                        int32_t* perm, int64_t* rank_offsets,
                                                                        int32_t* err) {
  extern __shared__ uint32_t fsm[];
  uint32_t* keys = fsm;                            // [kFbsSmallMax] one pass's output order
  uint32_t* vals = keys + kFbsSmallMax;            // [kFbsSmallMax]
  uint32_t* hist = vals + kFbsSmallMax;            // [kFbsSmallWarps][256]
  uint32_t* dstart = hist + kFbsSmallWarps * 256;  // [256]
  uint32_t* red = dstart + 256;                    // [64]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto slot = [&](int i) { return warp * 32 * kFbsSmallItems + i * 32 + lane; };  // slot order = item order
  uint32_t k[kFbsSmallItems], v[kFbsSmallItems];
  uint32_t kmax = 0;
#pragma unroll
  for (int i = 0; i < kFbsSmallItems; ++i) {
    const int g = slot(i);
    int32_t l = g < S ? L[g] : 0;
    if (l < 0) {
      set_err(err, FS_ERR_INVALID_ARG);
      l = 0;
    }
    k[i] = uint32_t(l);
    v[i] = uint32_t(g);
    kmax = k[i] > kmax ? k[i] : kmax;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t x = __shfl_xor_sync(0xffffffffu, kmax, o);
    kmax = x > kmax ? x : kmax;
  }
  if (lane == 0) red[warp] = kmax;
  __syncthreads();
  kmax = 0;
  for (int w = 0; w < kFbsSmallWarps; ++w) kmax = red[w] > kmax ? red[w] : kmax;
  const int passes = (32 - __clz(kmax) + 7) / 8;  // 0 when every length is 0: the order is g
  for (int pass = 0; pass < passes; ++pass) {
    const int shift = 8 * pass;
    for (int j = threadIdx.x; j < kFbsSmallWarps * 256; j += kFbsSmallThreads) hist[j] = 0u;
    __syncthreads();
    // warp multisplit by ballots (8-bit digits), slot by slot
    // (a warp's rank of an item among its equal digits, < 512, rides in the
    // top bits of the item's value: g < 2^14)
    uint32_t* wh = hist + warp * 256;
#pragma unroll
    for (int i = 0; i < kFbsSmallItems; ++i) {
      const bool live = slot(i) < S;
      const uint32_t d = (k[i] >> shift) & 255u;
      const unsigned lv = __ballot_sync(0xffffffffu, live);
      unsigned peers = live ? lv : ~lv;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const bool on = (d >> b) & 1u;
        const unsigned m = __ballot_sync(0xffffffffu, on);
        peers &= on ? m : ~m;
      }
      const unsigned lt = __popc(peers & lanemask_lt());
      const uint32_t base = live ? wh[d] : 0u;
      v[i] |= (base + lt) << 16;
      __syncwarp();
      if (live && lt == 0) wh[d] = base + __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    // per digit: exclusive over the warps, then over the digits
    uint32_t tot = 0;
    if (threadIdx.x < 256) {
      const int d = threadIdx.x;
      for (int w = 0; w < kFbsSmallWarps; ++w) {
        const uint32_t c = hist[w * 256 + d];
        hist[w * 256 + d] = tot;
        tot += c;
      }
    }
    // exclusive scan of the 256 digit totals by the first 8 warps
    uint32_t x = tot;
    if (warp < 8) {
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) red[32 + warp] = x;
    }
    __syncthreads();
    if (warp < 8) {
      uint32_t before = 0;
      for (int w = 0; w < warp; ++w) before += red[32 + w];
      dstart[threadIdx.x] = before + x - tot;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kFbsSmallItems; ++i)
      if (slot(i) < S) {
        const uint32_t d = (k[i] >> shift) & 255u;
        const uint32_t at = dstart[d] + hist[warp * 256 + d] + (v[i] >> 16);
        keys[at] = k[i];
        vals[at] = v[i] & 0xFFFFu;
      }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kFbsSmallItems; ++i) {
      const int p = slot(i);
      if (p < S) {
        k[i] = keys[p];
        v[i] = vals[p];
      }
    }
    __syncthreads();
  }
  // sorted position p = slot(i): the snake deal
#pragma unroll
  for (int i = 0; i < kFbsSmallItems; ++i) {
    const int64_t p = slot(i);
    if (p < S) {
      const int64_t rho = p / n, kk = p % n;
      const int64_t r = (rho & 1) ? (n - 1 - kk) : kk;
      perm[fbs_rank_offset(r, S, n) + rho] = int32_t(v[i]);
    }
  }
  for (int64_t r = threadIdx.x; r <= n; r += kFbsSmallThreads) rank_offsets[r] = fbs_rank_offset(r, S, n);
}

// ------------------------------------------------------------------- VBS

// Fixed-point weight round_half_even(256 * L^alpha); L^alpha evaluated with
// IEEE-exact operations where alpha allows (a product of L's and at most one
// correctly rounded square root), pow() otherwise.
__device__ __forceinline__ uint64_t vbs_weight(int32_t L, double alpha) {
  const double x = static_cast<double>(L < 0 ? 0 : L);
  double p;
  if (alpha == 1.0) {
    p = x;
  } else if (alpha == 1.5) {
    p = __dmul_rn(x, __dsqrt_rn(x));
  } else if (alpha == 2.0) {
    p = __dmul_rn(x, x);
  } else if (alpha == 0.5) {
    p = __dsqrt_rn(x);
  } else if (alpha == 2.5) {
    p = __dmul_rn(__dmul_rn(x, x), __dsqrt_rn(x));
  } else if (alpha == 3.0) {
    p = __dmul_rn(__dmul_rn(x, x), x);
  } else {
    p = pow(x, alpha);
  }
  return static_cast<uint64_t>(rint(__dmul_rn(p, 256.0)));
}

constexpr int kVbsItems = 8;
constexpr int kVbsTile = kThreads * kVbsItems;

// Exclusive prefix of the weights along the order (order == nullptr: identity).
// P[j] for j < S, P[S] = W.  Tiles claim their index dynamically.
__global__ void __launch_bounds__(kThreads) vbs_scan_kernel(const int32_t* L, const uint32_t* order, int64_t S,
                                                            double alpha, uint64_t* P, uint64_t* status,
                                                            int* tile_counter, int32_t* err, int64_t limit,
                                                            int64_t skip_tile) {
  __shared__ uint64_t tmp[32];
  __shared__ int64_t s_tile;
  __shared__ uint64_t s_excl;
  if (threadIdx.x == 0) s_tile = atomicAdd(tile_counter, 1);
  __syncthreads();
  const int64_t tile = s_tile;
  const int64_t base = tile * kVbsTile + int64_t(threadIdx.x) * kVbsItems;
  const uint64_t wmax = ((1ull << 62) - 1) / static_cast<uint64_t>(S > 0 ? S : 1);
  uint64_t w[kVbsItems];
  uint64_t sum = 0;
#pragma unroll
  for (int i = 0; i < kVbsItems; ++i) {
    int64_t j = base + i;
    w[i] = 0;
    if (j < S) {
      int64_t g = order ? int64_t(order[j]) : j;
      int32_t l = L[g];
      if (l < 0) set_err(err, FS_ERR_INVALID_ARG);
      w[i] = vbs_weight(l, alpha);
      if (w[i] > wmax) {
        set_err(err, FS_ERR_INVALID_ARG);
        w[i] = 0;
      }
    }
    sum += w[i];
  }
  uint64_t tot;
  uint64_t ex = block_exclusive_scan<uint64_t>(sum, tmp, &tot);
  if (tile == skip_tile) return;  // test hook: this tile never publishes
  if (threadIdx.x < 32) {
    uint64_t e = warp_lookback(status, 1, tile, tot, err, limit);
    if (threadIdx.x == 0) s_excl = e;
  }
  __syncthreads();
  uint64_t run = s_excl + ex;
#pragma unroll
  for (int i = 0; i < kVbsItems; ++i) {
    int64_t j = base + i;
    if (j < S) P[j] = run;
    run += w[i];
    if (j == S - 1) P[S] = run;
  }
}

__device__ __forceinline__ int64_t vbs_rank(uint64_t Pj, uint64_t W, int64_t j, int64_t S, int64_t n) {
  int64_t r;
  if (W == 0) {
    r = static_cast<int64_t>((static_cast<unsigned __int128>(j) * static_cast<unsigned __int128>(n)) /
                             static_cast<unsigned __int128>(S));
  } else {
    r = static_cast<int64_t>((static_cast<unsigned __int128>(Pj) * static_cast<unsigned __int128>(n)) /
                             static_cast<unsigned __int128>(W));
  }
  return r > n - 1 ? n - 1 : r;
}

__global__ void vbs_assign_kernel(const uint32_t* order, const uint64_t* P, int64_t S, int32_t n, int32_t* perm,
                                  int64_t* rank_offsets) {
  const uint64_t W = P[S];
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; j < S; j += stride) {
    perm[j] = order ? static_cast<int32_t>(order[j]) : static_cast<int32_t>(j);
    const int64_t r = vbs_rank(P[j], W, j, S, n);
    const int64_t rp = (j == 0) ? -1 : vbs_rank(P[j - 1], W, j - 1, S, n);
    for (int64_t q = rp + 1; q <= r; ++q) rank_offsets[q] = j;  // first sample of ranks rp+1..r
    if (j == S - 1)
      for (int64_t q = r + 1; q <= n; ++q) rank_offsets[q] = S;
  }
}

__global__ void vbs_segment_weight_kernel(const uint64_t* P, const int64_t* rank_offsets, int32_t n,
                                          uint64_t* seg_weight) {
  for (int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; r < n; r += int64_t(gridDim.x) * blockDim.x)
    seg_weight[r] = P[rank_offsets[r + 1]] - P[rank_offsets[r]];
}

// ------------------------------------------------------------ VBS AutoTune

constexpr int kTuneThreads = 256;
constexpr int32_t kTuneMaxRanks = 65536;
constexpr int64_t kTimeLimit = int64_t(1) << 53;

// One AutoTune update (FreeScale §4.1, VBS paragraph; Figure 4's AutoTune
// module): ranks slower than the average by more than the dead band give
// `step` samples, ranks faster than it take `step`, paired so that the global
// batch stays fixed: with k = min(#slow, #fast), the k slowest and the k
// fastest ranks move.  Every block reduces all n times itself (integer sums:
// the same in every block), then each warp decides for one rank.  A rank's
// place among the slow ones is the number of ranks with a larger time plus the
// number of lower ranks with the same time (anything slower than a slow rank
// is slow too); the fast side is the mirror image.  The warp's lanes split
// that count; the times come through shared memory in tiles of kTuneTile.
// O(n^2) comparisons in all, n <= 65536.
constexpr int kTuneTile = 2048;
constexpr int kTuneWarps = kTuneThreads / 32;  // ranks per block

__global__ void __launch_bounds__(kTuneThreads) vbs_autotune_kernel(const int64_t* t, int32_t n, int64_t step,
                                                                    int32_t tol_ppm, int64_t* delta, int32_t* err) {
  __shared__ int64_t tile[kTuneTile];
  __shared__ uint64_t part_lo[kTuneWarps], part_hi[kTuneWarps];
  __shared__ int counts[2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < 2) counts[threadIdx.x] = 0;
  // sum of the times as two exact 64-bit halves: low 32 bits and high bits of
  // each time summed apart (< 2^48 and < 2^37 for n <= 65536)
  uint64_t lo = 0, hi = 0;
  bool bad = false;
  for (int32_t q = threadIdx.x; q < n; q += kTuneThreads) {
    const int64_t x = t[q];
    bad |= (x < 0) || (x >= kTimeLimit);
    lo += static_cast<uint32_t>(x);
    hi += static_cast<uint64_t>(x) >> 32;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo += __shfl_down_sync(0xffffffffu, lo, o);
    hi += __shfl_down_sync(0xffffffffu, hi, o);
  }
  if (lane == 0) {
    part_lo[warp] = lo;
    part_hi[warp] = hi;
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_err(err, FS_ERR_INVALID_ARG);
    return;
  }
  uint64_t LO = 0, HI = 0;
#pragma unroll
  for (int w = 0; w < kTuneWarps; ++w) {
    LO += part_lo[w];
    HI += part_hi[w];
  }
  const unsigned __int128 sum = (static_cast<unsigned __int128>(HI) << 32) + LO;
  const unsigned __int128 scale = static_cast<unsigned __int128>(n) * 1000000u;
  const unsigned __int128 hi_bar = sum * static_cast<unsigned __int128>(1000000 + tol_ppm);
  const unsigned __int128 lo_bar = sum * static_cast<unsigned __int128>(1000000 - tol_ppm);
  unsigned my_slow = 0, my_fast = 0;
  for (int32_t q = threadIdx.x; q < n; q += kTuneThreads) {
    const unsigned __int128 x = static_cast<unsigned __int128>(t[q]) * scale;
    my_slow += x > hi_bar;
    my_fast += x < lo_bar;
  }
  my_slow = __reduce_add_sync(0xffffffffu, my_slow);
  my_fast = __reduce_add_sync(0xffffffffu, my_fast);
  if (lane == 0 && my_slow) atomicAdd(&counts[0], int(my_slow));
  if (lane == 0 && my_fast) atomicAdd(&counts[1], int(my_fast));
  __syncthreads();
  const int k = min(counts[0], counts[1]);
  // this warp's rank (every lane holds the same values: the branches below are warp-uniform)
  const int32_t r = blockIdx.x * kTuneWarps + warp;
  int64_t tr = 0;
  bool slow = false, active = false;
  if (r < n && k > 0) {
    tr = t[r];
    const unsigned __int128 xr = static_cast<unsigned __int128>(tr) * scale;
    slow = xr > hi_bar;
    active = slow || xr < lo_bar;
  }
  if (!__syncthreads_or(active)) return;
  unsigned place = 0;
  for (int32_t base = 0; base < n; base += kTuneTile) {
    const int32_t m = min(kTuneTile, n - base);
    __syncthreads();
    for (int i = threadIdx.x; i < m; i += kTuneThreads) tile[i] = t[base + i];
    __syncthreads();
    if (active) {
      const int32_t ties_below = r - base;  // entries i < ties_below are lower ranks
      if (slow) {
        for (int i = lane; i < m; i += 32) {
          const int64_t tq = tile[i];
          place += (tq > tr) | ((tq == tr) & (i < ties_below));
        }
      } else {
        for (int i = lane; i < m; i += 32) {
          const int64_t tq = tile[i];
          place += (tq < tr) | ((tq == tr) & (i < ties_below));
        }
      }
    }
  }
  if (active) {
    place = __reduce_add_sync(0xffffffffu, place);
    if (lane == 0 && place < unsigned(k)) delta[r] += slow ? -step : step;
  }
}

// Inclusive max-scan of one value per thread over a block (blockDim.x <= 1024,
// a multiple of 32); `smem` needs 32 slots.
__device__ __forceinline__ int64_t block_inclusive_max(int64_t v, int64_t* smem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = max(x, y);
  }
  if (lane == 31) smem[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t w = (lane < nw) ? smem[lane] : INT64_MIN;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w = max(w, y);
    }
    smem[lane] = w;
  }
  __syncthreads();
  const int64_t res = (warp == 0) ? x : max(x, smem[warp - 1]);
  __syncthreads();
  return res;
}

constexpr int kAdjustThreads = 1024;

// Apply the AutoTune correction to the VBS cut, one block: segment end r
// moves by D_r = delta[0] + ... + delta[r], is clamped to [0, S], then the ends
// are made non-decreasing (prefix maximum).  The correction must sum to 0 with
// |delta[r]| <= S; otherwise FS_ERR_INVALID_ARG and the cut is left as it was.
__global__ void __launch_bounds__(kAdjustThreads) vbs_adjust_kernel(int64_t* rank_offsets, const int64_t* delta,
                                                                    int32_t n, int64_t S, int32_t* err) {
  __shared__ int64_t smem[32];
  bool bad = false;
  int64_t part = 0;  // |part| <= (n / threads) * S < 2^62
  for (int32_t r = threadIdx.x; r < n; r += kAdjustThreads) {
    const int64_t d = delta[r];
    if (d > S || d < -S)
      bad = true;
    else
      part += d;
  }
  int64_t total;
  (void)block_exclusive_scan<int64_t>(part, smem, &total);
  bad = __syncthreads_or(bad);
  if (bad || total != 0) {
    if (threadIdx.x == 0) set_err(err, FS_ERR_INVALID_ARG);
    return;
  }
  int64_t carry = 0, run_max = 0;
  for (int32_t c0 = 0; c0 < n; c0 += kAdjustThreads) {
    const int32_t r = c0 + threadIdx.x;
    const int64_t d = r < n ? delta[r] : 0;
    int64_t chunk_sum;
    const int64_t D = carry + block_exclusive_scan<int64_t>(d, smem, &chunk_sum) + d;
    int64_t e = 0;
    if (r < n) e = min(max(rank_offsets[r + 1] + D, int64_t(0)), S);
    e = max(block_inclusive_max(e, smem), run_max);
    if (r < n) rank_offsets[r + 1] = e;
    carry += chunk_sum;
    // the chunk's last end is the running maximum for the next chunk
    if (threadIdx.x == kAdjustThreads - 1) smem[0] = e;
    __syncthreads();
    run_max = smem[0];
    __syncthreads();
  }
}

__global__ void fill_i64_kernel(int64_t* p, int64_t count, int64_t v) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < count; i += int64_t(gridDim.x) * blockDim.x)
    p[i] = v;
}

unsigned grid_for(int64_t items, int per_block = kThreads) {
  int64_t g = (items + per_block - 1) / per_block;
  int64_t cap = int64_t(sm_count()) * 8;
  if (g > cap) g = cap;
  return unsigned(g < 1 ? 1 : g);
}

constexpr int kLenKeyBits = 31;  // int32 lengths >= 0

size_t vbs_extra_bytes(int64_t S) {
  int64_t tiles = (S + kVbsTile - 1) / kVbsTile;
  return align_up(size_t(S + 1) * sizeof(uint64_t)) + align_up(size_t(tiles) * sizeof(uint64_t) + 256);
}

}  // namespace
}  // namespace fs

using namespace fs;

extern "C" size_t fs_balance_fbs_workspace_size(int64_t S, int32_t n) {
  (void)n;
  if (S < 0) return 0;
  return radix::SortPlan(S, kLenKeyBits).bytes() + 256;
}

extern "C" fs_status fs_balance_fbs(const int32_t* uih_len, int64_t S, int32_t n, int32_t* perm,
                                    int64_t* rank_offsets, int32_t* err, void* ws, size_t ws_bytes,
                                    fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (n < 1 || S < 0 || S > INT32_MAX || !rank_offsets || !err) return FS_ERR_INVALID_ARG;
  if (S > 0 && (!uih_len || !perm)) return FS_ERR_INVALID_ARG;
  if (!aligned(rank_offsets, 8) || !aligned(err, 4)) return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_balance_fbs_workspace_size(S, n) || (S > 0 && !ws)) return FS_ERR_WORKSPACE;
  int launches = 0;
  if (S == 0) {
    fill_i64_kernel<<<1, kThreads, 0, st>>>(rank_offsets, int64_t(n) + 1, 0);
    count_launch(1);
    return launch_status();
  }
  if (S <= kFbsSmallMax) {  // one block: sort and deal in shared memory
    cudaFuncSetAttribute(fbs_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kFbsSmallSmem));
    fbs_small_kernel<<<1, kFbsSmallThreads, kFbsSmallSmem, st>>>(uih_len, int32_t(S), n, perm, rank_offsets, err);
    count_launch(1);
    return launch_status();
  }
  radix::SortPlan P(S, kLenKeyBits);
  WsCursor cur(ws, ws_bytes);
  radix::SortWs W;
  if (!radix::carve_sort_ws(P, cur, W)) return FS_ERR_WORKSPACE;
  uint32_t *sk = nullptr, *sv = nullptr;
  fs_status s = radix::run_sort(SrcLen{uih_len}, P, W, err, st, &sk, &sv, &launches);
  if (s != FS_OK) return s;
  fbs_assign_kernel<<<grid_for(S > n ? S : n + 1), kThreads, 0, st>>>(sv, S, n, perm, rank_offsets);
  count_launch(launches + 1);
  return launch_status();
}

// ---------------------------------------------------------------------------
// FBS without caller workspace.  Some callers cannot allocate device memory
// at the moment they need the partition: code that runs while a memory pool
// is frozen or being torn down, a runtime whose allocator they do not own
// (for example a plugin inside another framework's process), or a step whose
// memory plan is fixed in advance.  For them this variant keeps the sort's
// scratch in a fixed array in the library's own device memory, so the call
// itself allocates nothing.
namespace fs {
namespace {

constexpr int64_t kNoAllocMaxS = int64_t(1) << 18;  // 262144 samples

// The sort's scratch for kNoAllocMaxS samples and 31-bit keys (passes of
// 7 + 8 + 8 + 8 bits: at most 256 digit values), computed by the same layout
// arithmetic that carves the workspace, so the array and the carve cannot
// drift apart; smaller S needs less.
constexpr size_t kNoAllocScratchBytes = radix::SortPlan(kNoAllocMaxS, kLenKeyBits).bytes();
static_assert(radix::SortPlan(kNoAllocMaxS, kLenKeyBits).nb == 256, "31-bit keys sort in 8-bit digits at most");
static_assert(radix::SortPlan(kNoAllocMaxS - 1, kLenKeyBits).bytes() <= kNoAllocScratchBytes,
              "the scratch need grows with S");

// Lives for as long as the library is loaded, on every device that uses it.
static __device__ __align__(256) unsigned char g_fbs_scratch[kNoAllocScratchBytes + 256];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of g_fbs_scratch on the current device.  Host code only sees
// a stand-in symbol, never a device address, so the address is looked up with
// cudaGetSymbolAddress on the first call on each device (with that device
// current) and kept for the life of the process.  A caller that resets a
// device (cudaDeviceReset) gets a new module instance there; the address kept
// from before the reset no longer belongs to it, so this entry point must not
// be called on that device after a reset.
fs_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FS_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fbs_scratch) != cudaSuccess || p == nullptr) return FS_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FS_OK;
}

}  // namespace
}  // namespace fs

extern "C" fs_status fs_balance_fbs_noalloc(const int32_t* uih_len, int64_t S, int32_t n, int32_t* perm,
                                            int64_t* rank_offsets, int32_t* err, fs_stream_t stream) {
  FS_NVTX_RANGE();
  if (S > kNoAllocMaxS) return FS_ERR_INVALID_ARG;  // beyond the fixed scratch array
  if (n < 1 || S < 0 || !rank_offsets || !err) return FS_ERR_INVALID_ARG;
  if (S > 0 && (!uih_len || !perm)) return FS_ERR_INVALID_ARG;
  void* scratch = nullptr;
  fs_status s = scratch_for_current_device(&scratch);
  if (s != FS_OK) return s;
  const size_t need = radix::SortPlan(S, kLenKeyBits).bytes();
  if (need > kNoAllocScratchBytes) return FS_ERR_INVALID_ARG;
  // every count the sort reads it has written earlier in the same call, so
  // stale contents of a previous call do no harm
  return fs_balance_fbs(uih_len, S, n, perm, rank_offsets, err, scratch, sizeof(g_fbs_scratch), stream);
}

extern "C" size_t fs_balance_vbs_workspace_size(int64_t S, int32_t n) {
  return fs_balance_fbs_workspace_size(S, n) + vbs_extra_bytes(S) + 256;
}

namespace fs {
namespace {

// The VBS cut; with batch_delta != nullptr the AutoTune correction is applied
// to the segment ends before the segment weights are taken.
fs_status vbs_run(const int32_t* uih_len, int64_t S, int32_t n, double alpha, int32_t sort_by_len,
                  const int64_t* batch_delta, int32_t* perm, int64_t* rank_offsets, uint64_t* seg_weight,
                  int32_t* err, void* ws, size_t ws_bytes, fs_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (n < 1 || S < 0 || S > INT32_MAX || !rank_offsets || !err || !seg_weight || !(alpha >= 0.0))
    return FS_ERR_INVALID_ARG;
  if (S > 0 && (!uih_len || !perm)) return FS_ERR_INVALID_ARG;
  if (!aligned(rank_offsets, 8) || !aligned(seg_weight, 8) || !aligned(err, 4)) return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_balance_vbs_workspace_size(S, n) || (S > 0 && !ws)) return FS_ERR_WORKSPACE;
  if (batch_delta && !aligned(batch_delta, 8)) return FS_ERR_ALIGNMENT;
  if (S == 0) {
    fill_i64_kernel<<<grid_for(int64_t(n) + 1), kThreads, 0, st>>>(rank_offsets, int64_t(n) + 1, 0);
    fill_i64_kernel<<<grid_for(n), kThreads, 0, st>>>(reinterpret_cast<int64_t*>(seg_weight), n, 0);
    if (batch_delta) vbs_adjust_kernel<<<1, kAdjustThreads, 0, st>>>(rank_offsets, batch_delta, n, S, err);
    count_launch(batch_delta ? 3 : 2);
    return launch_status();
  }
  int launches = 0;
  WsCursor cur(ws, ws_bytes);
  const int64_t vtiles = (S + kVbsTile - 1) / kVbsTile;
  uint64_t* P = cur.take<uint64_t>(size_t(S + 1));
  unsigned char* vzero = cur.take<unsigned char>(size_t(vtiles) * sizeof(uint64_t) + 256);
  if (!cur.ok) return FS_ERR_WORKSPACE;
  uint64_t* vstatus = reinterpret_cast<uint64_t*>(vzero + 256);
  int* vcounter = reinterpret_cast<int*>(vzero);
  if (cudaMemsetAsync(vzero, 0, size_t(vtiles) * sizeof(uint64_t) + 256, st) != cudaSuccess) return FS_ERR_CUDA;

  const uint32_t* order = nullptr;
  if (sort_by_len) {
    radix::SortPlan SP(S, kLenKeyBits);
    radix::SortWs W;
    if (!radix::carve_sort_ws(SP, cur, W)) return FS_ERR_WORKSPACE;
    uint32_t *sk = nullptr, *sv = nullptr;
    fs_status s = radix::run_sort(SrcLen{uih_len}, SP, W, err, st, &sk, &sv, &launches);
    if (s != FS_OK) return s;
    order = sv;
  }
  vbs_scan_kernel<<<unsigned(vtiles), kThreads, 0, st>>>(uih_len, order, S, alpha, P, vstatus, vcounter, err,
                                                         spin_limit(), debug_skip_tile());
  vbs_assign_kernel<<<grid_for(S), kThreads, 0, st>>>(order, P, S, n, perm, rank_offsets);
  if (batch_delta) {
    vbs_adjust_kernel<<<1, kAdjustThreads, 0, st>>>(rank_offsets, batch_delta, n, S, err);
    ++launches;
  }
  vbs_segment_weight_kernel<<<grid_for(n), kThreads, 0, st>>>(P, rank_offsets, n, seg_weight);
  count_launch(launches + 3);
  return launch_status();
}

}  // namespace
}  // namespace fs

extern "C" fs_status fs_balance_vbs(const int32_t* uih_len, int64_t S, int32_t n, double alpha, int32_t sort_by_len,
                                    int32_t* perm, int64_t* rank_offsets, uint64_t* seg_weight, int32_t* err,
                                    void* ws, size_t ws_bytes, fs_stream_t stream) {
  FS_NVTX_RANGE();
  return vbs_run(uih_len, S, n, alpha, sort_by_len, nullptr, perm, rank_offsets, seg_weight, err, ws, ws_bytes,
                 stream);
}

extern "C" fs_status fs_balance_vbs_tuned(const int32_t* uih_len, int64_t S, int32_t n, double alpha,
                                          int32_t sort_by_len, const int64_t* batch_delta, int32_t* perm,
                                          int64_t* rank_offsets, uint64_t* seg_weight, int32_t* err, void* ws,
                                          size_t ws_bytes, fs_stream_t stream) {
  FS_NVTX_RANGE();
  if (!batch_delta) return FS_ERR_INVALID_ARG;
  return vbs_run(uih_len, S, n, alpha, sort_by_len, batch_delta, perm, rank_offsets, seg_weight, err, ws, ws_bytes,
                 stream);
}

extern "C" fs_status fs_vbs_autotune(const int64_t* times, int32_t n, int64_t step, int32_t tol_ppm,
                                     int64_t* batch_delta, int32_t* err, fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (n < 1 || n > kTuneMaxRanks || step < 0 || step > INT32_MAX || tol_ppm < 0 || tol_ppm > 1000000)
    return FS_ERR_INVALID_ARG;
  if (!times || !batch_delta || !err) return FS_ERR_INVALID_ARG;
  if (!aligned(times, 8) || !aligned(batch_delta, 8) || !aligned(err, 4)) return FS_ERR_ALIGNMENT;
  const unsigned blocks = unsigned((n + kTuneWarps - 1) / kTuneWarps);
  vbs_autotune_kernel<<<blocks, kTuneThreads, 0, st>>>(times, n, step, tol_ppm, batch_delta, err);
  count_launch(1);
  return launch_status();
}
