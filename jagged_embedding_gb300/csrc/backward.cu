// Embedding backward: gradient segment-reduce per row + row update.
// FreeScale (arXiv 2604.24073) Algorithm 2 lines 7 and 20 (update_embedding
// on the exclusive / collision rows) and line 18 (split of the gradients into
// collision and exclusive parts).  The optimizer is the standard SGD or the
// row-wise Adagrad (Duchi, Hazan & Singer 2011: one accumulator per row).
//
// Pipeline (all on `stream`, sizes stay on the device):
//   1. stable LSD radix sort of (row, position) over the positions the phase
//      selects (reduce-then-scan counting passes of at most 9 bits; the first
//      pass reads the int64 IDs and the collision mask directly, so
//      unselected positions are never copied);
//   2. reduce: the sorted array is cut into fixed 2048-entry tiles, one warp
//      per tile, so a Zipf-hot row with millions of positions is spread over
//      many warps and a long tail of single-position rows costs the same per
//      entry.  A warp walks its entries in order, summing each row's gradient
//      rows in fp32 (lane l owns columns [l*EPL, (l+1)*EPL)), and updates every
//      row that starts and ends inside the tile on the spot (the table row and
//      the Adagrad state are prefetched into L2 a batch ahead).  A row that
//      crosses a tile boundary leaves its partial sums as carries;
//   3. fixup: one warp per row that crosses tile boundaries adds its carries
//      in tile order (in fp64) and updates the row.
// The summation order is fixed by the sorted order and the tiling, so results
// are bit-identical from run to run.
#include <cuda_bf16.h>

#include "radix.cuh"
#include "tma.cuh"

namespace fs {
namespace {

using radix::kThreads;
constexpr int kChunk = 2048;                 // sorted entries per reduce tile
bool g_force_unstaged = true;  // measured: the register path beats bulk-copy staging for 256-byte rows
int g_reduce_variant = 0;      // launch shape of the register path (see launch_reduce)
constexpr uint32_t kNoKey = 0xFFFFFFFFu;     // rows are < num_rows < 2^32

// Sort source: the selected positions of the batch, key = row, value = position.
struct SrcRows {
  using Key = uint32_t;
  static constexpr bool kIndexValue = true;  // value = item index
  const int64_t* ids;
  const uint8_t* is_co;
  int phase;
  int64_t R;
  __device__ __forceinline__ bool load(int64_t i, Key& key, uint32_t& val, int32_t* err) const {
    // the ID and the mask byte are loaded independently (no load-to-load dependency)
    const int64_t id = __ldcs(ids + i);
    if (phase != FS_PHASE_ALL) {
      const uint8_t m = __ldcs(is_co + i);
      if ((phase == FS_PHASE_COLLISION) ? (m != 1) : (m != 0)) return false;
    }
    if (id < 0 || id >= R) {
      if (err) set_err(err, FS_ERR_ID_RANGE);
      return false;
    }
    key = static_cast<uint32_t>(id);
    val = static_cast<uint32_t>(i);
    return true;
  }
  __device__ __forceinline__ uint32_t digit(Key key, int shift, int bits) const {
    return (key >> shift) & ((1u << bits) - 1u);
  }
};

template <int BYTES> struct Raw;
template <> struct Raw<2> { using T = unsigned short; };
template <> struct Raw<4> { using T = unsigned int; };
template <> struct Raw<8> { using T = uint2; };
template <> struct Raw<16> { using T = uint4; };

// Row slice of lane `lane`: elements [lane*EPL, lane*EPL + EPL) of row `row`.
template <bool BF16, int EPL, bool STREAM>
__device__ __forceinline__ void load_slice(const void* base, int64_t row, int lane, float (&x)[EPL]) {
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int D = 32 * EPL;
  using V = typename Raw<EPL * ESZ>::T;
  const V* p = reinterpret_cast<const V*>(static_cast<const char*>(base) + (row * D + int64_t(lane) * EPL) * ESZ);
  V v = STREAM ? __ldcs(p) : *p;
  uint32_t w[(EPL * ESZ + 3) / 4];
  if constexpr (EPL * ESZ >= 4) {
    memcpy(w, &v, EPL * ESZ);
  } else {
    w[0] = static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(&v));
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    if constexpr (BF16) {
      uint32_t h = (w[i / 2] >> ((i & 1) * 16)) & 0xFFFFu;
      x[i] = __uint_as_float(h << 16);
    } else {
      x[i] = __uint_as_float(w[i]);
    }
  }
}

template <bool BF16, int EPL>
__device__ __forceinline__ void store_slice(void* base, int64_t row, int lane, const float (&x)[EPL]) {
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int D = 32 * EPL;
  using V = typename Raw<EPL * ESZ>::T;
  uint32_t w[(EPL * ESZ + 3) / 4];
#pragma unroll
  for (int i = 0; i < (EPL * ESZ + 3) / 4; ++i) w[i] = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    if constexpr (BF16) {
      __nv_bfloat16 b = __float2bfloat16_rn(x[i]);
      uint32_t h = static_cast<uint32_t>(__bfloat16_as_ushort(b));
      w[i / 2] |= h << ((i & 1) * 16);
    } else {
      w[i] = __float_as_uint(x[i]);
    }
  }
  V v;
  if constexpr (EPL * ESZ >= 4) {
    memcpy(&v, w, EPL * ESZ);
  } else {
    unsigned short s = static_cast<unsigned short>(w[0]);
    memcpy(&v, &s, 2);
  }
  *reinterpret_cast<V*>(static_cast<char*>(base) + (row * D + int64_t(lane) * EPL) * ESZ) = v;
}

struct UpdateArgs {
  void* table;
  float* state;
  int optim;
  float lr;
  float eps;
};

// Apply the optimizer to one row with its reduced gradient (whole warp).
template <bool BF16, int EPL>
__device__ __forceinline__ void update_row(const UpdateArgs& u, uint32_t row, const float (&g)[EPL], int lane) {
  constexpr int D = 32 * EPL;
  float w[EPL];
  load_slice<BF16, EPL, false>(u.table, row, lane, w);
  if (u.optim == FS_ROWWISE_ADAGRAD) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) ss = __fmaf_rn(g[i], g[i], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    ss = __shfl_sync(0xffffffffu, ss, 0);  // one value for the whole row
    const float s = u.state[row] + ss / float(D);
    const float denom = sqrtf(s) + u.eps;
    if (lane == 0) u.state[row] = s;
#pragma unroll
    for (int i = 0; i < EPL; ++i) w[i] = w[i] - u.lr * g[i] / denom;
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) w[i] = w[i] - u.lr * g[i];
  }
  store_slice<BF16, EPL>(u.table, row, lane, w);
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

template <bool BF16, int EPL, int GROWS, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) reduce_kernel(const uint32_t* __restrict__ keys,
                                                             const uint32_t* __restrict__ vals, const int64_t* n_dev,
                                                             const void* __restrict__ grads, UpdateArgs u,
                                                             float* carry_head, float* carry_tail, uint8_t* head_cont,
                                                             uint8_t* tail_flag) {
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int D = 32 * EPL;
  constexpr int RB = D * ESZ;
  constexpr int G = GROWS;  // gradient rows in flight per warp
  const int64_t n = *n_dev;
  const int64_t ntiles = (n + kChunk - 1) / kChunk;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < ntiles; t += nwarps) {
    const int64_t s0 = t * kChunk;
    const int64_t s1 = (s0 + kChunk < n) ? s0 + kChunk : n;
    const uint32_t prev_key = s0 > 0 ? keys[s0 - 1] : kNoKey;
    const uint32_t next_key = s1 < n ? keys[s1] : kNoKey;
    uint32_t cur = keys[s0];
    bool from_prev = (cur == prev_key);
    float acc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] = 0.f;

    // keys / positions of the next batch are loaded one batch ahead
    uint32_t pre_k = (s0 + lane < s1) ? __ldcs(keys + s0 + lane) : kNoKey;
    uint32_t pre_p = (s0 + lane < s1) ? __ldcs(vals + s0 + lane) : 0u;
    for (int64_t j = s0; j < s1; j += 32) {
      const int cnt = (s1 - j < 32) ? int(s1 - j) : 32;
      const uint32_t my_k = pre_k, my_p = pre_p;
      const int64_t jn = j + 32;
      pre_k = (jn + lane < s1) ? __ldcs(keys + jn + lane) : kNoKey;
      pre_p = (jn + lane < s1) ? __ldcs(vals + jn + lane) : 0u;
      uint32_t nk = __shfl_down_sync(0xffffffffu, my_k, 1);
      const uint32_t first_next = __shfl_sync(0xffffffffu, pre_k, 0);
      if (lane == cnt - 1) nk = (j + cnt < s1) ? first_next : next_key;
      if (lane < cnt && nk != my_k) {  // a row ends at this entry: bring its table row and state to L2
        const char* rp = static_cast<const char*>(u.table) + int64_t(my_k) * RB;
#pragma unroll
        for (int b = 0; b < RB; b += 128) prefetch_l2(rp + b);
        if (u.state) prefetch_l2(u.state + my_k);
      }
      for (int e0 = 0; e0 < cnt; e0 += G) {
        float g[G][EPL];
#pragma unroll
        for (int q = 0; q < G; ++q) {
          const int e = e0 + q;
          const uint32_t p = __shfl_sync(0xffffffffu, my_p, e & 31);
          if (e < cnt) load_slice<BF16, EPL, true>(grads, p, lane, g[q]);
        }
#pragma unroll
        for (int q = 0; q < G; ++q) {
          const int e = e0 + q;
          const uint32_t k = __shfl_sync(0xffffffffu, my_k, e & 31);
          if (e < cnt) {
            if (k != cur) {
              if (from_prev) {  // the row began in an earlier tile and ends here
#pragma unroll
                for (int i = 0; i < EPL; ++i) carry_head[t * D + lane * EPL + i] = acc[i];
                if (lane == 0) head_cont[t] = 0;
              } else {
                update_row<BF16, EPL>(u, cur, acc, lane);
              }
              cur = k;
              from_prev = false;
#pragma unroll
              for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < EPL; ++i) acc[i] += g[q][i];
          }
        }
      }
    }
    // the tile's last row
    if (cur == next_key) {
      if (from_prev) {  // spans the whole tile
#pragma unroll
        for (int i = 0; i < EPL; ++i) carry_head[t * D + lane * EPL + i] = acc[i];
        if (lane == 0) {
          head_cont[t] = 1;
          tail_flag[t] = 0;
        }
      } else {  // starts here, continues in the next tile
#pragma unroll
        for (int i = 0; i < EPL; ++i) carry_tail[t * D + lane * EPL + i] = acc[i];
        if (lane == 0) tail_flag[t] = 1;
      }
    } else {
      if (from_prev) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) carry_head[t * D + lane * EPL + i] = acc[i];
        if (lane == 0) head_cont[t] = 0;
      } else {
        update_row<BF16, EPL>(u, cur, acc, lane);
      }
      if (lane == 0) tail_flag[t] = 0;
    }
  }
}

// Reduce with batched updates: within a group of G sorted entries, every row
// that ends in the group has its sum completed first (sequentially, entry by
// entry, the same order as reduce_kernel), then the table-row loads of all
// those rows are issued together and the updates applied.  A run of
// single-position rows (the Zipf tail) thus keeps up to G table rows in
// flight per warp instead of waiting for one row at a time.
template <bool BF16, int EPL, int G, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) reduce_batched_kernel(const uint32_t* __restrict__ keys,
                                                                        const uint32_t* __restrict__ vals,
                                                                        const int64_t* n_dev,
                                                                        const void* __restrict__ grads, UpdateArgs u,
                                                                        float* carry_head, float* carry_tail,
                                                                        uint8_t* head_cont, uint8_t* tail_flag) {
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int D = 32 * EPL;
  static_assert(32 % G == 0, "groups tile a batch of 32 entries");
  const int64_t n = *n_dev;
  const int64_t ntiles = (n + kChunk - 1) / kChunk;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  (void)ESZ;
  for (int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < ntiles; t += nwarps) {
    const int64_t s0 = t * kChunk;
    const int64_t s1 = (s0 + kChunk < n) ? s0 + kChunk : n;
    const uint32_t prev_key = s0 > 0 ? keys[s0 - 1] : kNoKey;
    const uint32_t next_key = s1 < n ? keys[s1] : kNoKey;
    const uint32_t first_key = keys[s0];
    bool from_prev = (first_key == prev_key);  // the open row began in an earlier tile
    float acc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] = 0.f;

    uint32_t pre_k = (s0 + lane < s1) ? __ldcs(keys + s0 + lane) : kNoKey;
    uint32_t pre_p = (s0 + lane < s1) ? __ldcs(vals + s0 + lane) : 0u;
    uint32_t last_key = first_key;
    for (int64_t j = s0; j < s1; j += 32) {
      const int cnt = (s1 - j < 32) ? int(s1 - j) : 32;
      const uint32_t my_k = pre_k, my_p = pre_p;
      const int64_t jn = j + 32;
      pre_k = (jn + lane < s1) ? __ldcs(keys + jn + lane) : kNoKey;
      pre_p = (jn + lane < s1) ? __ldcs(vals + jn + lane) : 0u;
      const uint32_t first_next = (j + cnt < s1) ? __shfl_sync(0xffffffffu, pre_k, 0) : next_key;
      // key of the entry after mine (for "a row ends at my entry")
      uint32_t nk = __shfl_down_sync(0xffffffffu, my_k, 1);
      if (lane == cnt - 1) nk = first_next;
      const bool my_end = lane < cnt && nk != my_k;
      if (my_end) {  // bring the table row and the state of a row that ends here to L2
        const char* rp = static_cast<const char*>(u.table) + int64_t(my_k) * (D * ESZ);
#pragma unroll
        for (int b = 0; b < D * ESZ; b += 128) prefetch_l2(rp + b);
        if (u.state) prefetch_l2(u.state + my_k);
      }
      const unsigned ends = __ballot_sync(0xffffffffu, my_end);
      // state of the row ending at each entry, one load per lane
      float my_state = 0.f;
      if (my_end && u.state) my_state = u.state[my_k];

      for (int e0 = 0; e0 < cnt; e0 += G) {
        float g[G][EPL];
#pragma unroll
        for (int q = 0; q < G; ++q) {
          const int e = e0 + q;
          const uint32_t p = __shfl_sync(0xffffffffu, my_p, e & 31);
          if (e < cnt) load_slice<BF16, EPL, true>(grads, p, lane, g[q]);
        }
        // sums of the rows that end in this group, in entry order
        bool upd[G];
#pragma unroll
        for (int q = 0; q < G; ++q) {
          const int e = e0 + q;
          upd[q] = false;
          if (e < cnt) {
#pragma unroll
            for (int i = 0; i < EPL; ++i) acc[i] += g[q][i];
            if ((ends >> e) & 1u) {
              const uint32_t k = __shfl_sync(0xffffffffu, my_k, e);
              if (from_prev && k == first_key) {  // began in an earlier tile: leave a carry
#pragma unroll
                for (int i = 0; i < EPL; ++i) carry_head[t * D + lane * EPL + i] = acc[i];
                if (lane == 0) head_cont[t] = 0;
                from_prev = false;
              } else {
                upd[q] = true;
#pragma unroll
                for (int i = 0; i < EPL; ++i) g[q][i] = acc[i];
              }
#pragma unroll
              for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
            }
          }
        }
        // table rows of all rows ending here, loads in flight together
        float w[G][EPL];
#pragma unroll
        for (int q = 0; q < G; ++q)
          if (upd[q]) load_slice<BF16, EPL, false>(u.table, __shfl_sync(0xffffffffu, my_k, e0 + q), lane, w[q]);
#pragma unroll
        for (int q = 0; q < G; ++q) {
          const int e = e0 + q;
          const float s_old = __shfl_sync(0xffffffffu, my_state, e & 31);
          if (upd[q]) {
            const uint32_t row = __shfl_sync(0xffffffffu, my_k, e);
            if (u.optim == FS_ROWWISE_ADAGRAD) {
              float ss = 0.f;
#pragma unroll
              for (int i = 0; i < EPL; ++i) ss = __fmaf_rn(g[q][i], g[q][i], ss);
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
              ss = __shfl_sync(0xffffffffu, ss, 0);
              const float snew = s_old + ss / float(D);
              const float denom = sqrtf(snew) + u.eps;
              if (lane == 0) u.state[row] = snew;
#pragma unroll
              for (int i = 0; i < EPL; ++i) w[q][i] = w[q][i] - u.lr * g[q][i] / denom;
            } else {
#pragma unroll
              for (int i = 0; i < EPL; ++i) w[q][i] = w[q][i] - u.lr * g[q][i];
            }
            store_slice<BF16, EPL>(u.table, row, lane, w[q]);
          }
        }
      }
      last_key = __shfl_sync(0xffffffffu, my_k, cnt - 1);
    }
    // the tile's last row, if it did not end inside the tile
    if (last_key == next_key) {
      if (from_prev) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) carry_head[t * D + lane * EPL + i] = acc[i];
        if (lane == 0) head_cont[t] = 1;
      } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) carry_tail[t * D + lane * EPL + i] = acc[i];
      }
    }
    if (lane == 0) tail_flag[t] = (last_key == next_key && !from_prev) ? 1 : 0;
  }
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Reduce with the gradient rows streamed into a per-warp shared-memory ring by
// asynchronous copies (cp.async, 16 bytes per lane, no registers held while
// in flight): the rows of groups g+1 .. g+NST-1 are on their way while group g
// is summed, so a warp keeps (NST-1) * G rows in flight even while it waits
// on a table row to update.  Same tiling, carries and summation order as
// reduce_kernel (entries in sorted order, fp32 per tile, fixed per lane).
template <bool BF16, int EPL, int G, int NST, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    reduce_async_kernel(const uint32_t* __restrict__ keys, const uint32_t* __restrict__ vals, const int64_t* n_dev,
                        const void* __restrict__ grads, UpdateArgs u, float* carry_head, float* carry_tail,
                        uint8_t* head_cont, uint8_t* tail_flag) {
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int D = 32 * EPL;
  constexpr int RB = D * ESZ;
  constexpr int CPR = RB / 16;                  // 16-byte chunks per row
  constexpr int CPL = (G * CPR + 31) / 32;      // chunks per lane per group
  static_assert(32 % G == 0, "groups tile a batch of 32 entries");
  static_assert((NST - 1) * G <= 32, "copies run at most one batch ahead");
  using V = typename Raw<EPL * ESZ>::T;
  extern __shared__ __align__(16) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned char* ring = smem + warp * (NST * G * RB);
  const char* gb = static_cast<const char*>(grads);
  const int64_t n = *n_dev;
  const int64_t ntiles = (n + kChunk - 1) / kChunk;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < ntiles; t += nwarps) {
    const int64_t s0 = t * kChunk;
    const int64_t s1 = (s0 + kChunk < n) ? s0 + kChunk : n;
    const int ne = int(s1 - s0);
    const int ngroups = (ne + G - 1) / G;
    const uint32_t prev_key = s0 > 0 ? keys[s0 - 1] : kNoKey;
    const uint32_t next_key = s1 < n ? keys[s1] : kNoKey;
    // keys / positions of two consecutive batches of 32 entries live in registers
    uint32_t bk[2], bp[2];
    bk[0] = lane < ne ? __ldcs(keys + s0 + lane) : kNoKey;
    bp[0] = lane < ne ? __ldcs(vals + s0 + lane) : 0u;
    bk[1] = 32 + lane < ne ? __ldcs(keys + s0 + 32 + lane) : kNoKey;
    bp[1] = 32 + lane < ne ? __ldcs(vals + s0 + 32 + lane) : 0u;
    int loaded_batch = 1;  // index of the batch held in slot (loaded_batch & 1)

    auto issue = [&](int g) {
      if (g < ngroups) {
        unsigned char* dst = ring + (g % NST) * (G * RB);
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int c = lane + 32 * i;
          const int cc = c < G * CPR ? c : 0;
          const int r = cc / CPR, part = cc % CPR;
          const int e = g * G + r;
          // every lane shuffles both batch slots and picks the one its entry is in
          const uint32_t p0 = __shfl_sync(0xffffffffu, bp[0], e & 31);
          const uint32_t p1 = __shfl_sync(0xffffffffu, bp[1], e & 31);
          const uint32_t p = ((e >> 5) & 1) ? p1 : p0;
          if (c < G * CPR && e < ne) cp_async16(dst + r * RB + part * 16, gb + int64_t(p) * RB + part * 16);
        }
      }
      cp_async_commit();  // one group per call, empty past the end, so wait counts stay exact
    };

    for (int g = 0; g < NST - 1; ++g) issue(g);
    uint32_t cur = __shfl_sync(0xffffffffu, bk[0], 0);
    bool from_prev = (cur == prev_key);
    float acc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] = 0.f;

    for (int g = 0; g < ngroups; ++g) {
      cp_async_wait<NST - 2>();  // group g has landed (for this lane)
      __syncwarp();              // ... and for every lane of the warp
      const unsigned char* src = ring + (g % NST) * (G * RB);
      const int bslot = ((g * G) >> 5) & 1;
      // segment ends of this group: an entry ends its row when the next key differs
#pragma unroll
      for (int r = 0; r < G; ++r) {
        const int e = g * G + r;
        if (e < ne) {
          const uint32_t k0 = __shfl_sync(0xffffffffu, bk[0], e & 31);
          const uint32_t k1 = __shfl_sync(0xffffffffu, bk[1], e & 31);
          const uint32_t k = bslot ? k1 : k0;
          if (k != cur) {
            if (from_prev) {
#pragma unroll
              for (int i = 0; i < EPL; ++i) carry_head[t * D + lane * EPL + i] = acc[i];
              if (lane == 0) head_cont[t] = 0;
            } else {
              update_row<BF16, EPL>(u, cur, acc, lane);
            }
            cur = k;
            from_prev = false;
#pragma unroll
            for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
          }
          const V v = *reinterpret_cast<const V*>(src + r * RB + lane * EPL * ESZ);
          uint32_t w[(EPL * ESZ + 3) / 4];
          if constexpr (EPL * ESZ >= 4) memcpy(w, &v, EPL * ESZ);
          else w[0] = uint32_t(*reinterpret_cast<const unsigned short*>(&v));
#pragma unroll
          for (int i = 0; i < EPL; ++i)
            acc[i] += BF16 ? __uint_as_float(((w[i / 2] >> ((i & 1) * 16)) & 0xFFFFu) << 16) : __uint_as_float(w[i]);
        }
      }
      __syncwarp();  // every lane is done with this stage before it is refilled
      // batch bookkeeping: when group g finishes a batch, the batch after the
      // next one is loaded into the slot just freed (the issue-ahead window
      // never reaches more than one batch ahead)
      if (((g + 1) * G) % 32 == 0) {
        const int finished = ((g + 1) * G) / 32 - 1;
        if (finished + 2 > loaded_batch) {
          const int nb = finished + 2;
          const int64_t base = s0 + int64_t(nb) * 32;
          bk[nb & 1] = base + lane < s1 ? __ldcs(keys + base + lane) : kNoKey;
          bp[nb & 1] = base + lane < s1 ? __ldcs(vals + base + lane) : 0u;
          loaded_batch = nb;
        }
      }
      issue(g + NST - 1);
    }
    cp_async_wait<0>();
    __syncwarp();
    // the tile's last row
    if (cur == next_key) {
      if (from_prev) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) carry_head[t * D + lane * EPL + i] = acc[i];
        if (lane == 0) {
          head_cont[t] = 1;
          tail_flag[t] = 0;
        }
      } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) carry_tail[t * D + lane * EPL + i] = acc[i];
        if (lane == 0) tail_flag[t] = 1;
      }
    } else {
      if (from_prev) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) carry_head[t * D + lane * EPL + i] = acc[i];
        if (lane == 0) head_cont[t] = 0;
      } else {
        update_row<BF16, EPL>(u, cur, acc, lane);
      }
      if (lane == 0) tail_flag[t] = 0;
    }
  }
}

// Shared-memory plan of the staged reduce: per warp NST stages, each holding
// the 32 gradient rows of one batch of sorted entries and the table rows of
// the rows that end (and get updated) in that batch, plus keys, flags and the
// stage's mbarrier.
template <bool BF16, int EPL>
struct Staged {
  static constexpr int ESZ = BF16 ? 2 : 4;
  static constexpr int D = 32 * EPL;
  static constexpr int RB = D * ESZ;
  static constexpr int NST = 3;
  static constexpr int STAGE = 2 * 32 * RB;
  static constexpr int META = NST * (32 * 4 + 32) + NST * 8;
  static constexpr int WARP_BYTES = NST * STAGE + ((META + 127) / 128) * 128;
  static constexpr int WPB_RAW = (196 * 1024) / WARP_BYTES;
  static constexpr int WPB = WPB_RAW < 1 ? 1 : (WPB_RAW > 8 ? 8 : WPB_RAW);
  static constexpr int SMEM = WPB * WARP_BYTES;
};

// Staged variant of the reduce: gradient rows and the table rows to update are
// brought into shared memory by bulk asynchronous copies (cp.async.bulk, one
// 256-byte row per lane, completion on an mbarrier), NST batches of 32 entries
// ahead of the warp that sums them.  Same tiling, carries and summation order
// as reduce_kernel.
template <bool BF16, int EPL>
__global__ void __launch_bounds__(Staged<BF16, EPL>::WPB * 32, 1)
    reduce_staged_kernel(const uint32_t* __restrict__ keys, const uint32_t* __restrict__ vals, const int64_t* n_dev,
                         const void* __restrict__ grads, UpdateArgs u, float* carry_head, float* carry_tail,
                         uint8_t* head_cont, uint8_t* tail_flag, int32_t* err, int64_t limit) {
  using P = Staged<BF16, EPL>;
  constexpr int ESZ = P::ESZ, D = P::D, RB = P::RB, NST = P::NST;
  using V = typename Raw<EPL * ESZ>::T;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned char* wb = smem + warp * P::WARP_BYTES;
  uint32_t* skeys = reinterpret_cast<uint32_t*>(wb + NST * P::STAGE);
  uint8_t* sflags = reinterpret_cast<uint8_t*>(skeys + NST * 32);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sflags + NST * 32);
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) tma::mbar_init(bars + s, 1);
    tma::fence_barrier_init();
  }
  __syncwarp();
  uint32_t phase = 0;  // bit s: parity of the next completion of stage s
  const char* gbytes = static_cast<const char*>(grads);
  const char* tbytes = static_cast<const char*>(u.table);

  const int64_t n = *n_dev;
  const int64_t ntiles = (n + kChunk - 1) / kChunk;
  const int64_t nwarps = int64_t(gridDim.x) * P::WPB;
  for (int64_t t = int64_t(blockIdx.x) * P::WPB + warp; t < ntiles; t += nwarps) {
    const int64_t s0 = t * kChunk;
    const int64_t s1 = (s0 + kChunk < n) ? s0 + kChunk : n;
    const uint32_t prev_key = s0 > 0 ? keys[s0 - 1] : kNoKey;
    const uint32_t next_key = s1 < n ? keys[s1] : kNoKey;
    const uint32_t first_key = keys[s0];
    const bool from_prev_tile = (first_key == prev_key);
    const int nb = int((s1 - s0 + 31) / 32);

    // Stage batch b: its keys / flags to shared memory, its rows in flight.
    auto issue = [&](int b) {
      const int st = b % NST;
      const int64_t j = s0 + int64_t(b) * 32;
      const int cnt = (s1 - j < 32) ? int(s1 - j) : 32;
      const uint32_t k = lane < cnt ? __ldcs(keys + j + lane) : kNoKey;
      const uint32_t p = lane < cnt ? __ldcs(vals + j + lane) : 0u;
      uint32_t nk = __shfl_down_sync(0xffffffffu, k, 1);
      if (lane == cnt - 1) nk = (j + cnt < s1) ? keys[j + cnt] : next_key;
      const bool ends = lane < cnt && nk != k;
      const bool carry = ends && from_prev_tile && k == first_key;
      const bool upd = ends && !carry;
      if (lane < cnt) {
        skeys[st * 32 + lane] = k;
        sflags[st * 32 + lane] = uint8_t((ends ? 1 : 0) | (upd ? 2 : 0));
      }
      const unsigned updm = __ballot_sync(0xffffffffu, upd);
      if (lane == 0) tma::mbar_arrive_expect_tx(bars + st, uint32_t(cnt + __popc(updm)) * RB);
      __syncwarp();
      unsigned char* gs = wb + st * P::STAGE;
      if (lane < cnt) tma::bulk_g2s(gs + lane * RB, gbytes + int64_t(p) * RB, RB, bars + st);
      if (upd) {
        tma::bulk_g2s(gs + 32 * RB + lane * RB, tbytes + int64_t(k) * RB, RB, bars + st);
        if (u.state) prefetch_l2(u.state + k);
      }
    };

    for (int b = 0; b < NST && b < nb; ++b) issue(b);
    bool from_prev = from_prev_tile;
    float acc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] = 0.f;

    for (int b = 0; b < nb; ++b) {
      const int st = b % NST;
      const int64_t j = s0 + int64_t(b) * 32;
      const int cnt = (s1 - j < 32) ? int(s1 - j) : 32;
      if (!tma::mbar_wait(bars + st, (phase >> st) & 1u, limit)) {
        if (lane == 0) set_err(err, FS_ERR_TIMEOUT);
        return;  // never seen in practice: the copies are a few microseconds long
      }
      phase ^= 1u << st;
      const unsigned char* gs = wb + st * P::STAGE;
      // Adagrad state of the rows updated in this batch, one load per lane
      const uint8_t myf = sflags[st * 32 + lane];
      float my_state = 0.f;
      if (lane < cnt && (myf & 2) && u.state) my_state = u.state[skeys[st * 32 + lane]];
      for (int e = 0; e < cnt; ++e) {
        float g[EPL];
        {
          const V v = *reinterpret_cast<const V*>(gs + e * RB + lane * EPL * ESZ);
          uint32_t w[(EPL * ESZ + 3) / 4];
          if constexpr (EPL * ESZ >= 4) memcpy(w, &v, EPL * ESZ);
          else w[0] = uint32_t(*reinterpret_cast<const unsigned short*>(&v));
#pragma unroll
          for (int i = 0; i < EPL; ++i)
            g[i] = BF16 ? __uint_as_float(((w[i / 2] >> ((i & 1) * 16)) & 0xFFFFu) << 16) : __uint_as_float(w[i]);
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc[i] += g[i];
        const uint8_t f = sflags[st * 32 + e];
        const float s_old = __shfl_sync(0xffffffffu, my_state, e);
        if (f & 1) {
          if (f & 2) {
            const uint32_t row = skeys[st * 32 + e];
            float w[EPL];
            {
              const V v = *reinterpret_cast<const V*>(gs + 32 * RB + e * RB + lane * EPL * ESZ);
              uint32_t x[(EPL * ESZ + 3) / 4];
              if constexpr (EPL * ESZ >= 4) memcpy(x, &v, EPL * ESZ);
              else x[0] = uint32_t(*reinterpret_cast<const unsigned short*>(&v));
#pragma unroll
              for (int i = 0; i < EPL; ++i)
                w[i] = BF16 ? __uint_as_float(((x[i / 2] >> ((i & 1) * 16)) & 0xFFFFu) << 16) : __uint_as_float(x[i]);
            }
            if (u.optim == FS_ROWWISE_ADAGRAD) {
              float ss = 0.f;
#pragma unroll
              for (int i = 0; i < EPL; ++i) ss = __fmaf_rn(acc[i], acc[i], ss);
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
              ss = __shfl_sync(0xffffffffu, ss, 0);
              const float snew = s_old + ss / float(D);
              const float denom = sqrtf(snew) + u.eps;
              if (lane == 0) u.state[row] = snew;
#pragma unroll
              for (int i = 0; i < EPL; ++i) w[i] = w[i] - u.lr * acc[i] / denom;
            } else {
#pragma unroll
              for (int i = 0; i < EPL; ++i) w[i] = w[i] - u.lr * acc[i];
            }
            store_slice<BF16, EPL>(u.table, row, lane, w);
          } else {  // the row began in an earlier tile and ends here
#pragma unroll
            for (int i = 0; i < EPL; ++i) carry_head[t * D + lane * EPL + i] = acc[i];
            if (lane == 0) head_cont[t] = 0;
          }
          from_prev = false;
#pragma unroll
          for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
        }
      }
      __syncwarp();
      tma::fence_proxy_async();
      if (b + NST < nb) issue(b + NST);
    }
    // the tile's last row, if it continues past the tile
    const bool open = (keys[s1 - 1] == next_key);
    if (open) {
      if (from_prev) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) carry_head[t * D + lane * EPL + i] = acc[i];
        if (lane == 0) head_cont[t] = 1;
      } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) carry_tail[t * D + lane * EPL + i] = acc[i];
      }
    }
    if (lane == 0) tail_flag[t] = (open && !from_prev) ? 1 : 0;
  }
}

// Rows that cross tile boundaries: carry of the starting tile, then the head
// carries of the following tiles in order.
template <bool BF16, int EPL>
__global__ void __launch_bounds__(kThreads) fixup_kernel(const uint32_t* __restrict__ keys, const int64_t* n_dev,
                                                         UpdateArgs u, const float* carry_head,
                                                         const float* carry_tail, const uint8_t* head_cont,
                                                         const uint8_t* tail_flag) {
  constexpr int D = 32 * EPL;
  const int64_t n = *n_dev;
  const int64_t ntiles = (n + kChunk - 1) / kChunk;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < ntiles; t += nwarps) {
    if (!tail_flag[t]) continue;
    const uint32_t row = keys[(t + 1) * kChunk - 1];
    // the chain of tile partials is summed in fp64: a Zipf-hot row can cross
    // thousands of tiles, and this keeps its error at the level of one tile's
    double acc64[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc64[i] = double(carry_tail[t * D + lane * EPL + i]);
    // the chain ends at the first following tile whose head does not continue;
    // read 32 continuation flags at a time, then sum that window's carries in
    // tile order with several loads in flight
    for (int64_t v = t + 1; v < ntiles; v += 32) {
      const uint8_t hc = (v + lane < ntiles) ? head_cont[v + lane] : uint8_t(0);
      const unsigned stop = __ballot_sync(0xffffffffu, hc == 0);
      const int last = stop ? (__ffs(stop) - 1) : 31;
      int j = 0;
      for (; j + 8 <= last + 1; j += 8) {
        float c[8][EPL];
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
          for (int i = 0; i < EPL; ++i) c[q][i] = carry_head[(v + j + q) * D + lane * EPL + i];
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
          for (int i = 0; i < EPL; ++i) acc64[i] += double(c[q][i]);
      }
      for (; j <= last; ++j)
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc64[i] += double(carry_head[(v + j) * D + lane * EPL + i]);
      if (stop) break;
    }
    float acc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] = float(acc64[i]);
    update_row<BF16, EPL>(u, row, acc, lane);
  }
}

template <bool BF16, int EPL, int G, int NST, int MINB>
void launch_async(const uint32_t* k, const uint32_t* v, const int64_t* n_dev, const void* grads, UpdateArgs u,
                  float* ch, float* ct, uint8_t* hc, uint8_t* tf, cudaStream_t st) {
  constexpr int RB = 32 * EPL * (BF16 ? 2 : 4);
  constexpr int smem = (kThreads / 32) * NST * G * RB;
  cudaFuncSetAttribute(reduce_async_kernel<BF16, EPL, G, NST, MINB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  reduce_async_kernel<BF16, EPL, G, NST, MINB><<<unsigned(sm_count()) * MINB, kThreads, smem, st>>>(
      k, v, n_dev, grads, u, ch, ct, hc, tf);
}

template <bool BF16, int EPL>
void launch_reduce(const uint32_t* k, const uint32_t* v, const int64_t* n_dev, const void* grads, UpdateArgs u,
                   float* ch, float* ct, uint8_t* hc, uint8_t* tf, int32_t* err, bool staged, cudaStream_t st) {
  const unsigned grid = unsigned(sm_count()) * (2048 / kThreads);
  if (staged) {
    using P = Staged<BF16, EPL>;
    cudaFuncSetAttribute(reduce_staged_kernel<BF16, EPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, P::SMEM);
    reduce_staged_kernel<BF16, EPL><<<unsigned(sm_count()), P::WPB * 32, P::SMEM, st>>>(
        k, v, n_dev, grads, u, ch, ct, hc, tf, err, spin_limit());
  } else {
    // (rows in flight per warp, blocks per SM): 8 x 4 fits 64 registers for any row width
    constexpr int G8 = (16 / EPL) > 8 ? 8 : (16 / EPL);
    constexpr int G16 = (32 / EPL) > 16 ? 16 : (32 / EPL);
    constexpr int G4 = (8 / EPL) > 4 ? 4 : ((8 / EPL) < 1 ? 1 : (8 / EPL));
    const unsigned sms = unsigned(sm_count());
    switch (g_reduce_variant) {
      case 1: reduce_kernel<BF16, EPL, G16, 3><<<sms * 3, kThreads, 0, st>>>(k, v, n_dev, grads, u, ch, ct, hc, tf); break;
      case 2: reduce_kernel<BF16, EPL, G16, 2><<<sms * 2, kThreads, 0, st>>>(k, v, n_dev, grads, u, ch, ct, hc, tf); break;
      case 3: reduce_kernel<BF16, EPL, G8, 6><<<sms * 6, kThreads, 0, st>>>(k, v, n_dev, grads, u, ch, ct, hc, tf); break;
      case 4: launch_async<BF16, EPL, 8, 4, 3>(k, v, n_dev, grads, u, ch, ct, hc, tf, st); break;
      case 7: reduce_batched_kernel<BF16, EPL, G8, 3><<<sms * 3, kThreads, 0, st>>>(k, v, n_dev, grads, u, ch, ct, hc, tf); break;
      case 8: reduce_batched_kernel<BF16, EPL, G8, 4><<<sms * 4, kThreads, 0, st>>>(k, v, n_dev, grads, u, ch, ct, hc, tf); break;
      case 10: reduce_batched_kernel<BF16, EPL, G8, 2><<<sms * 2, kThreads, 0, st>>>(k, v, n_dev, grads, u, ch, ct, hc, tf); break;
      case 11: reduce_batched_kernel<BF16, EPL, G4, 4><<<sms * 4, kThreads, 0, st>>>(k, v, n_dev, grads, u, ch, ct, hc, tf); break;
      case 5: launch_async<BF16, EPL, 8, 5, 2>(k, v, n_dev, grads, u, ch, ct, hc, tf, st); break;
      case 6: launch_async<BF16, EPL, 4, 8, 3>(k, v, n_dev, grads, u, ch, ct, hc, tf, st); break;
      default: reduce_kernel<BF16, EPL, G8, 4><<<sms * 4, kThreads, 0, st>>>(k, v, n_dev, grads, u, ch, ct, hc, tf); break;
    }
  }
  fixup_kernel<BF16, EPL><<<grid, kThreads, 0, st>>>(k, n_dev, u, ch, ct, hc, tf);
}

struct BwdLayout {
  radix::SortPlan plan;
  int64_t max_tiles = 0;
  size_t carry_bytes = 0, flag_bytes = 0;
};

BwdLayout bwd_layout(int64_t T, int64_t R, int32_t dim) {
  BwdLayout L;
  L.plan = radix::SortPlan(T, radix::bits_for(uint64_t(R > 0 ? R - 1 : 0)));
  L.max_tiles = (T + kChunk - 1) / kChunk;
  L.carry_bytes = align_up(size_t(L.max_tiles) * size_t(dim) * sizeof(float));
  L.flag_bytes = align_up(size_t(L.max_tiles));
  return L;
}

int epl_for(int32_t dim, fs_dtype dtype) {
  if (dim % 32 != 0) return 0;
  int e = dim / 32;
  if (e == 1 || e == 2 || e == 4) return e;
  if (e == 8 && dtype == FS_BF16) return e;
  return 0;
}

}  // namespace
}  // namespace fs

using namespace fs;

extern "C" void fs_debug_reduce_variant(int32_t v) {
  fs::g_force_unstaged = v != 9;
  fs::g_reduce_variant = v;
}

extern "C" size_t fs_emb_backward_adagrad_workspace_size(int64_t T, int64_t num_rows, int32_t dim, fs_dtype dtype) {
  (void)dtype;
  if (T < 0 || num_rows < 1 || dim < 1) return 0;
  BwdLayout L = bwd_layout(T, num_rows, dim);
  return L.plan.bytes() + 2 * L.carry_bytes + 2 * L.flag_bytes + 256;
}

extern "C" fs_status fs_emb_backward_adagrad(void* table, float* state, int64_t num_rows, int32_t dim, fs_dtype dtype,
                                             fs_optim optim, const int64_t* ids, const void* grads, int64_t T,
                                             const uint8_t* is_co, fs_phase phase, float lr, float eps, int32_t* err,
                                             void* ws, size_t ws_bytes, fs_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T < 0 || T > INT32_MAX || num_rows < 1 || num_rows >= (int64_t(1) << 32) || !err) return FS_ERR_INVALID_ARG;
  if ((dtype != FS_F32 && dtype != FS_BF16) || (optim != FS_SGD && optim != FS_ROWWISE_ADAGRAD)) return FS_ERR_INVALID_ARG;
  if (phase != FS_PHASE_ALL && phase != FS_PHASE_COLLISION && phase != FS_PHASE_EXCLUSIVE) return FS_ERR_INVALID_ARG;
  const int epl = epl_for(dim, dtype);
  if (epl == 0) return FS_ERR_INVALID_ARG;
  if (optim == FS_ROWWISE_ADAGRAD && !state) return FS_ERR_INVALID_ARG;
  if (T == 0) return FS_OK;
  if (!table || !ids || !grads || (phase != FS_PHASE_ALL && !is_co)) return FS_ERR_INVALID_ARG;
  const size_t vec = size_t(epl) * (dtype == FS_F32 ? 4 : 2);
  if (!aligned(table, vec) || !aligned(grads, vec) || !aligned(ids, 8) || (state && !aligned(state, 4)))
    return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_emb_backward_adagrad_workspace_size(T, num_rows, dim, dtype) || !ws) return FS_ERR_WORKSPACE;

  BwdLayout L = bwd_layout(T, num_rows, dim);
  WsCursor cur(ws, ws_bytes);
  radix::SortWs W;
  if (!radix::carve_sort_ws(L.plan, cur, W)) return FS_ERR_WORKSPACE;
  float* carry_head = cur.take<float>(size_t(L.max_tiles) * dim);
  float* carry_tail = cur.take<float>(size_t(L.max_tiles) * dim);
  uint8_t* head_cont = cur.take<uint8_t>(size_t(L.max_tiles));
  uint8_t* tail_flag = cur.take<uint8_t>(size_t(L.max_tiles));
  if (!cur.ok) return FS_ERR_WORKSPACE;

  int launches = 0;
  uint32_t *sk = nullptr, *sv = nullptr;
  SrcRows src{ids, is_co, int(phase), num_rows};
  fs_status s = radix::run_sort(src, L.plan, W, err, st, &sk, &sv, &launches);
  if (s != FS_OK) return s;
  UpdateArgs u{table, optim == FS_ROWWISE_ADAGRAD ? state : nullptr, int(optim), lr, eps};
  const bool bf = dtype == FS_BF16;
  // bulk copies need 16-byte aligned rows; otherwise the register-staged kernel runs
  const bool staged = aligned(grads, 16) && aligned(table, 16) && !g_force_unstaged;
#define FS_REDUCE(BF, E) launch_reduce<BF, E>(sk, sv, W.pass.n_valid, grads, u, carry_head, carry_tail, head_cont, \
                                               tail_flag, err, staged, st)
  switch (epl) {
    case 1: if (bf) FS_REDUCE(true, 1); else FS_REDUCE(false, 1); break;
    case 2: if (bf) FS_REDUCE(true, 2); else FS_REDUCE(false, 2); break;
    case 4: if (bf) FS_REDUCE(true, 4); else FS_REDUCE(false, 4); break;
    default: FS_REDUCE(true, 8); break;
  }
#undef FS_REDUCE
  count_launch(launches + 2);
  return launch_status();
}
