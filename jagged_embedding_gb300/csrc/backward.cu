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
//   2. reduce: the sorted array is cut into tiles of 256 to 2048 entries (the
//      length follows from the range's size), one warp per tile at a time, so
//      a Zipf-hot row with millions of positions is spread over many warps and
//      a long tail of single-position rows costs the same per entry.  A warp
//      walks its entries in order, summing each row's gradient rows in fp32
//      (lane l owns columns [l*EPL, (l+1)*EPL)), and updates every row that
//      starts and ends inside the tile on the spot (the table row and the
//      Adagrad state are prefetched into L2 a batch ahead).  A row that crosses
//      a tile boundary leaves its partial sums as carries;
//   3. fixup: one warp per row that crosses tile boundaries adds its carries
//      in tile order (in fp64) and updates the row.
// The summation order is fixed by the sorted order and the tiling, so results
// are bit-identical from run to run.
//
// Row-sorted path: the same sort, run as its own call before the batch's
// lookup, leaves the sorted entries in the workspace; a gather reads them
// (each distinct table row once, written to all of its positions) and the
// update then reduces them without sorting again.
#include <cuda_bf16.h>

#include <algorithm>

#include "bulk.cuh"
#include "radix.cuh"

namespace fs {
namespace {

using radix::kThreads;
// Sorted entries per reduce tile: chosen on the device from the range's size n
// so that a small range still spreads over every warp (about `target` tiles),
// between kMinChunk and kMaxChunk and a multiple of 32.  Every kernel of one
// update launch computes it from the same n and target, so they agree, and the
// result depends only on n and the launch shape: identical run to run.
constexpr int kMinChunk = 256, kMaxChunk = 2048;
__device__ __forceinline__ int64_t tile_entries(int64_t n, int64_t target) {
  int64_t c = (n + target - 1) / (target > 0 ? target : 1);
  c = (c + 31) / 32 * 32;
  return c < kMinChunk ? kMinChunk : (c > kMaxChunk ? kMaxChunk : c);
}
constexpr uint32_t kNoKey = 0xFFFFFFFFu;     // rows are < num_rows < 2^32

// Sort source: the selected positions of the batch, key = row, value = position.
// With both phases in one call, key = row | (exclusive << kb): collision rows
// sort first, exclusive rows after them, each group in row order.
template <bool kRowBits>  // collision flags from the row bitmap (true) or the per-position mask
struct SrcRows {
  using Key = uint32_t;
  static constexpr bool kIndexValue = true;  // value = item index
  const int64_t* ids;
  const uint8_t* is_co;     // collision flag per position (kRowBits false)
  const uint32_t* co_rows;  // collision flag per row, bitmap (kRowBits true)
  int phase;
  int64_t R;
  int kb;  // bits of the largest row index
  static constexpr bool kFetch2 = kRowBits;
  struct Raw {
    int64_t id;
    uint32_t m;
  };
  // loads only: the ID and the mask byte independently; with the row bitmap,
  // fetch2 then reads the ID's row bit (L2-resident; an out-of-range ID reads
  // bit 0 and is rejected by make) after every ID of the tile is in flight
  template <bool>
  __device__ __forceinline__ Raw fetch(int64_t i) const {
    Raw r;
    r.id = __ldcs(ids + i);
    r.m = (!kRowBits && phase != FS_PHASE_ALL) ? uint32_t(__ldcs(is_co + i)) : 0u;
    return r;
  }
  template <bool>
  __device__ __forceinline__ void fetch2(Raw& r) const {
    if constexpr (kRowBits) {
      const uint64_t x = uint64_t(r.id) < uint64_t(R) ? uint64_t(r.id) : 0u;
      r.m = (__ldg(co_rows + (x >> 5)) >> (x & 31u)) & 1u;
    }
  }
  __device__ __forceinline__ bool make(const Raw& r, int64_t i, int, Key& key, uint32_t& val, int32_t* err) const {
    const int64_t id = r.id;
    uint32_t hi = 0;
    if (phase != FS_PHASE_ALL) {
      const uint32_t m = r.m;
      if (phase == FS_PHASE_COLLISION_THEN_EXCLUSIVE) {
        if (m > 1) return false;
        hi = uint32_t(1 - m) << kb;
      } else if ((phase == FS_PHASE_COLLISION) ? (m != 1) : (m != 0)) {
        return false;
      }
    }
    if (id < 0 || id >= R) {
      if (err) set_err(err, FS_ERR_ID_RANGE);
      return false;
    }
    key = static_cast<uint32_t>(id) | hi;
    val = static_cast<uint32_t>(i);
    return true;
  }
  __device__ __forceinline__ uint32_t digit(Key key, int shift, int bits, int) const {
    return (key >> shift) & ((1u << bits) - 1u);
  }
};

#ifndef FS_SHARD_SORT_MINB
#define FS_SHARD_SORT_MINB 4
#endif
#ifndef FS_SHARD_SORT2_MINB
#define FS_SHARD_SORT2_MINB 4
#endif

// Sources of the per-shard sort (fs_emb_sort_rows_sharded).  Pass 1 reads the
// shard-major IDs and their collision flags; the key is the same (phase bit |
// row) as SrcRows's and the value the entry's index, which the sink turns
// into its batch-major position (DstGatherPos) when it writes the entry, so
// no position waits in registers through the ranking (four blocks per SM fit
// where three did); the digit is the low `bits` bits of the row's offset
// inside its shard (the tile's segment).  An ID outside [0, R), outside the
// tile's shard, or with a flag above 1 is dropped (the first two set the
// error word).  The flag comes from a per-entry mask (kRowBits false) or from
// the row bitmap of the collision rows (kRowBits true: one bitmap word per
// entry, read after the IDs are in; in shard-major order a tile's words lie in
// its shard's stretch of the bitmap).  The digit does not depend on the flag;
// a bitmap flag is always 0 or 1, so the upsweep skips the bitmap (a mask byte
// above 1 drops the entry, so the upsweep reads the mask).
template <bool kRowBits>
struct SrcShardRows {
  using Key = uint32_t;
  static constexpr bool kIndexValue = true;  // value = entry index (DstGatherPos reads its position)
  static constexpr bool kFetch2 = kRowBits;
  static constexpr int kMinBlocks = FS_SHARD_SORT_MINB;
  const int64_t* sm_ids;
  const uint8_t* is_co;     // per shard-major entry (kRowBits false); null: one phase
  const uint32_t* co_rows;  // collision rows (kRowBits true)
  int64_t R;
  int64_t block;            // rows per shard
  int kb;                   // bits of the largest row index
  uint32_t row_mask;
  struct Raw {
    int64_t id;
    uint32_t m;
  };
  template <bool kVal>
  __device__ __forceinline__ Raw fetch(int64_t i) const {
    Raw r;
    r.id = __ldcs(sm_ids + i);
    // (the upsweep needs the mask too: a flag above 1 drops the entry there as well)
    r.m = (!kRowBits && is_co) ? uint32_t(__ldcs(is_co + i)) : 0u;
    return r;
  }
  template <bool kVal>
  __device__ __forceinline__ void fetch2(Raw& r) const {
    if constexpr (kRowBits) {
      if (kVal) {
        const uint64_t x = uint64_t(r.id) < uint64_t(R) ? uint64_t(r.id) : 0u;
        r.m = (__ldg(co_rows + (x >> 5)) >> (x & 31u)) & 1u;
      }
    }
  }
  __device__ __forceinline__ bool make(const Raw& r, int64_t i, int seg, Key& key, uint32_t& val, int32_t* err) const {
    if (r.m > 1) return false;
    if (r.id < 0 || r.id >= R) {
      if (err) set_err(err, FS_ERR_ID_RANGE);
      return false;
    }
    const int64_t local = r.id - int64_t(seg) * block;
    if (local < 0 || local >= block) {
      if (err) set_err(err, FS_ERR_BAD_OFFSETS);
      return false;
    }
    key = uint32_t(r.id) | ((kRowBits || is_co) ? (uint32_t(1 - r.m) << kb) : 0u);
    val = uint32_t(i);
    return true;
  }
  __device__ __forceinline__ uint32_t digit(Key key, int shift, int bits, int seg) const {
    const uint32_t local = (key & row_mask) - uint32_t(int64_t(seg) * block);
    return (local >> shift) & ((1u << bits) - 1u);
  }
};

// Sink of pass 1: the key, and the batch-major position of the entry whose
// index the downsweep hands over.
template <class PosT>
struct DstGatherPos {
  uint32_t* k;
  uint32_t* v;
  const PosT* pos;
  __device__ __forceinline__ void store(int64_t o, uint32_t key, uint32_t idx) const {
    k[o] = key;
    v[o] = uint32_t(__ldg(pos + idx));
  }
};

// Pass 2 of the per-shard sort: pass 1's (key, position) pairs; the digit is
// (phase bit, next `lbits` bits of the offset in the shard), the phase bit
// being the group (collision rows of every shard before exclusive ones).  As
// in pass 1 the value handed to the sink is the entry's index, and the sink
// (DstGatherPos over pass 1's positions) copies the position when it writes
// the entry.
struct SrcShardRows2 {
  using Key = uint32_t;
  static constexpr bool kIndexValue = true;
  static constexpr bool kFetch2 = false;
  static constexpr int kMinBlocks = FS_SHARD_SORT2_MINB;
  const uint32_t* k;
  int64_t block;
  int kb;
  uint32_t row_mask;
  int lbits;       // bits of the shard offset this pass sorts
  bool two_phase;  // the key's bit kb is the phase
  using Raw = uint32_t;
  template <bool>
  __device__ __forceinline__ Raw fetch(int64_t i) const { return __ldcs(k + i); }
  __device__ __forceinline__ bool make(Raw r, int64_t i, int, Key& key, uint32_t& val, int32_t*) const {
    key = r;
    val = uint32_t(i);
    return true;
  }
  __device__ __forceinline__ uint32_t digit(Key key, int shift, int, int seg) const {
    const uint32_t local = (key & row_mask) - uint32_t(int64_t(seg) * block);
    uint32_t d = (local >> shift) & ((1u << lbits) - 1u);
    if (two_phase) d |= ((key >> kb) & 1u) << lbits;
    return d;
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

// Optimizer step for one row (whole warp): w holds the lane's slice of the
// row's current weights, s_old its Adagrad state, g the reduced gradient.
template <bool BF16, int EPL>
__device__ __forceinline__ void apply_update(const UpdateArgs& u, uint32_t row, float (&w)[EPL], float s_old,
                                             const float (&g)[EPL], int lane) {
  constexpr int D = 32 * EPL;
  if (u.optim == FS_ROWWISE_ADAGRAD) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) ss = __fmaf_rn(g[i], g[i], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    // (the xor butterfly leaves the same bits in every lane: each level adds
    // the same two values, a + b == b + a)
    const float s = s_old + ss / float(D);
    const float step = __fdividef(u.lr, sqrtf(s) + u.eps);  // one division per row, within 2 ulp
    if (lane == 0) u.state[row] = s;
#pragma unroll
    for (int i = 0; i < EPL; ++i) w[i] = __fmaf_rn(-step, g[i], w[i]);
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) w[i] = __fmaf_rn(-u.lr, g[i], w[i]);
  }
  store_slice<BF16, EPL>(u.table, row, lane, w);
}

// Load, update and store one row (whole warp).
template <bool BF16, int EPL>
__device__ __forceinline__ void update_row(const UpdateArgs& u, uint32_t row, const float (&g)[EPL], int lane) {
  float w[EPL];
  load_slice<BF16, EPL, false>(u.table, row, lane, w);
  const float s_old = u.optim == FS_ROWWISE_ADAGRAD ? u.state[row] : 0.f;
  apply_update<BF16, EPL>(u, row, w, s_old, g, lane);
}

// a0 += b0, a1 += b1 in one paired fp32 add (sm_100+ add.f32x2: two
// independent round-to-nearest adds, the same bits as two scalar adds).
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  asm("{\n .reg .b64 a, b, r;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n add.rn.f32x2 r, a, b;\n"
      " mov.b64 {%0, %1}, r;\n}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// acc += row r of a shared-memory stage, lane's slice (elements
// [lane*EPL, lane*EPL + EPL)); bf16 pairs unpacked with one shift or mask each.
template <bool BF16, int EPL>
__device__ __forceinline__ void acc_slice(const unsigned char* stage, int r, int lane, float (&acc)[EPL]) {
  constexpr int ESZ = BF16 ? 2 : 4;
  const unsigned char* p = stage + (size_t(r) * 32 * EPL + size_t(lane) * EPL) * ESZ;
  if constexpr (EPL == 1) {
    acc[0] += BF16 ? __uint_as_float(uint32_t(*reinterpret_cast<const unsigned short*>(p)) << 16)
                   : *reinterpret_cast<const float*>(p);
  } else if constexpr (BF16) {
    constexpr int NW = EPL / 2;  // 32-bit words of the slice
    uint32_t w[NW];
    if constexpr (NW == 1) {
      w[0] = *reinterpret_cast<const uint32_t*>(p);
    } else if constexpr (NW == 2) {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      w[0] = v.x;
      w[1] = v.y;
    } else {
      const uint4 v = *reinterpret_cast<const uint4*>(p);
      w[0] = v.x;
      w[1] = v.y;
      w[2] = v.z;
      w[3] = v.w;
    }
#pragma unroll
    for (int j = 0; j < NW; ++j)
      add2(acc[2 * j], acc[2 * j + 1], __uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u));
  } else {
    float x[EPL];
    if constexpr (EPL == 2) {
      const float2 v = *reinterpret_cast<const float2*>(p);
      x[0] = v.x;
      x[1] = v.y;
    } else {
#pragma unroll
      for (int j = 0; j < EPL; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(p + j * 4);
        x[j] = v.x;
        x[j + 1] = v.y;
        x[j + 2] = v.z;
        x[j + 3] = v.w;
      }
    }
#pragma unroll
    for (int j = 0; j < EPL; j += 2) add2(acc[j], acc[j + 1], x[j], x[j + 1]);
  }
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Sorted entries [*begin_dev, *end_dev) (begin 0 when begin_dev is null);
// row = key & row_mask.  One warp per tile of `chunk` sorted entries; the
// gradient rows of a tile are summed in entry order, GROWS rows in flight.
// For each batch of 32 entries one ballot marks the entries that end a row
// (the next key differs), so the per-entry work is a load and an add.  A row
// that starts and ends in this tile is updated here; a row that crosses a
// tile edge leaves partial sums for fixup_kernel.
template <bool BF16, int EPL, int GROWS, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) reduce_kernel(const uint32_t* __restrict__ keys,
                                                             const uint32_t* __restrict__ vals,
                                                             const int64_t* begin_dev, const int64_t* end_dev,
                                                             uint32_t row_mask, const void* __restrict__ grads,
                                                             UpdateArgs u, float* carry_head, float* carry_tail,
                                                             uint8_t* head_cont, uint8_t* tail_flag, int64_t target) {
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int D = 32 * EPL;
  constexpr int RB = D * ESZ;
  constexpr int G = GROWS;  // gradient rows in flight per warp
  const int64_t b0 = begin_dev ? *begin_dev : 0;
  keys += b0;
  vals += b0;
  const int64_t n = *end_dev - b0;
  const int64_t chunk = tile_entries(n, target);
  const int64_t ntiles = (n + chunk - 1) / chunk;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < ntiles; t += nwarps) {
    const int64_t s0 = t * chunk;
    const int64_t s1 = (s0 + chunk < n) ? s0 + chunk : n;
    const uint32_t prev_key = s0 > 0 ? keys[s0 - 1] : kNoKey;
    const uint32_t next_key = s1 < n ? keys[s1] : kNoKey;
    bool from_prev = (keys[s0] == prev_key);  // the tile's first row began in an earlier tile
    if (lane == 0 && !from_prev) head_cont[t] = 0;  // every tile's flag is defined
    bool open = false;                        // acc holds entries of a row not yet finished
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
      const bool ends = lane < cnt && nk != my_k;
      const uint32_t end_mask = __ballot_sync(0xffffffffu, ends);
      if (ends) {  // bring the finished row's table row and state to L2
        const char* rp = static_cast<const char*>(u.table) + int64_t(my_k & row_mask) * RB;
#pragma unroll
        for (int b = 0; b < RB; b += 128) prefetch_l2(rp + b);
        if (u.state) prefetch_l2(u.state + (my_k & row_mask));
      }
      for (int e0 = 0; e0 < cnt; e0 += G) {
        float g[G][EPL];
#pragma unroll
        for (int q = 0; q < G; ++q) {
          const int e = e0 + q;
          const uint32_t p = __shfl_sync(0xffffffffu, my_p, e & 31);
          if (e < cnt) load_slice<BF16, EPL, true>(grads, p, lane, g[q]);
        }
        const uint32_t m = end_mask >> e0;
#pragma unroll
        for (int q = 0; q < G; ++q) {
          if (e0 + q < cnt) {
#pragma unroll
            for (int i = 0; i < EPL; ++i) acc[i] += g[q][i];
            open = true;
            if ((m >> q) & 1u) {  // entry e0 + q is its row's last
              if (from_prev) {    // the row began in an earlier tile and ends here
#pragma unroll
                for (int i = 0; i < EPL; ++i) carry_head[t * D + lane * EPL + i] = acc[i];
                if (lane == 0) head_cont[t] = 0;
                from_prev = false;
              } else {
                const uint32_t row = __shfl_sync(0xffffffffu, my_k, (e0 + q) & 31) & row_mask;
                update_row<BF16, EPL>(u, row, acc, lane);
              }
              open = false;
#pragma unroll
              for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
            }
          }
        }
      }
    }
    // a row still open continues into the next tile
    if (open) {
      if (from_prev) {  // spans the whole tile
#pragma unroll
        for (int i = 0; i < EPL; ++i) carry_head[t * D + lane * EPL + i] = acc[i];
        if (lane == 0) {
          head_cont[t] = 1;
          tail_flag[t] = 0;
        }
      } else {  // starts here
#pragma unroll
        for (int i = 0; i < EPL; ++i) carry_tail[t * D + lane * EPL + i] = acc[i];
        if (lane == 0) tail_flag[t] = 1;
      }
    } else if (lane == 0) {
      tail_flag[t] = 0;
    }
  }
}

// Shared-memory ring of the bulk-copy reduce: per warp kRingStages stages of
// BR gradient rows each (BR * RB <= 2 KB), the mbarriers in front.
constexpr int kRingStages = 4;
// Most gradient rows per ring stage (stages of 4 rows, four blocks per SM:
// no faster on the bf16 table, 0.5% slower on the f32 one).
constexpr int kRingRows = 8;
template <int RB>
struct Ring {
  static constexpr int BR = (2048 / RB) < kRingRows ? (2048 / RB) : kRingRows;  // rows per stage
  static constexpr int SPC = 32 / BR;                            // stages per 32-entry batch of keys
  static constexpr int kStageBytes = BR * RB;
  static constexpr int kWarpBytes = 128 + kRingStages * kStageBytes;
  static constexpr int kBlockBytes = (kThreads / 32) * kWarpBytes;
  static constexpr int kFit = (227 * 1024) / (kBlockBytes + 1024);
  static constexpr int kMinBlocks = kFit > 4 ? 4 : kFit;
  static_assert(SPC >= kRingStages - 1, "a copy issued ahead must fall in the current or the next key batch");
  static_assert(kMinBlocks >= 1, "ring too large");
};

// Reduce with the gradient rows brought in by bulk copies.  Same tiles,
// entry order, row ends and carries as reduce_kernel; what differs is how
// the rows arrive: each warp keeps kRingStages - 1 stages of BR rows in
// flight (one bulk copy per row into shared memory, completion counted in
// bytes on the stage's mbarrier) while it sums the stage that has landed,
// so no registers are tied up waiting for gradient rows and several KB per
// warp stay in flight.  Keys and positions are read two batches of 32
// ahead; table rows that a batch of 32 finishes are prefetched to L2 one
// batch ahead, and the table slices and Adagrad states of the rows a stage
// finishes are loaded before waiting for that stage.  A wait that exceeds
// wait_ns nanoseconds sets FS_ERR_TIMEOUT, waits (bounded) for the warp's copies
// still in flight and ends the warp.  Warps take tiles from the counter
// *tile_next (zero at launch).  skip_tile >= 0 is a test hook: the
// first stage of that tile is never copied, so its wait runs out.
template <bool BF16, int EPL, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) reduce_ring_kernel(
    const uint32_t* __restrict__ keys, const uint32_t* __restrict__ vals, const int64_t* begin_dev,
    const int64_t* end_dev, uint32_t row_mask, const void* __restrict__ grads, UpdateArgs u, float* carry_head,
    float* carry_tail, uint8_t* head_cont, uint8_t* tail_flag, int32_t* err, uint64_t wait_ns, int64_t skip_tile,
    int64_t target, uint32_t* tile_next) {
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int D = 32 * EPL;
  constexpr int RB = D * ESZ;
  using RG = Ring<RB>;
  constexpr int BR = RG::BR, SPC = RG::SPC, NS = kRingStages;
  static_assert((NS & (NS - 1)) == 0 && (SPC & (SPC - 1)) == 0, "powers of two");
  extern __shared__ __align__(128) unsigned char ring_smem[];
  const int lane = threadIdx.x & 31;
  unsigned char* wbase = ring_smem + (threadIdx.x >> 5) * RG::kWarpBytes;
  const uint32_t bar0 = bulk::smem_addr(wbase);
  const uint32_t data0 = bar0 + 128;
  const unsigned char* data = wbase + 128;
  if (lane == 0)
    for (int s = 0; s < NS; ++s) bulk::mbar_init(bar0 + 8 * s, 1);
  bulk::fence_init();
  __syncwarp();
  const uint64_t pol = bulk::evict_first_policy();
  const char* gbytes = static_cast<const char*>(grads);
  const bool adagrad = u.optim == FS_ROWWISE_ADAGRAD;

  const int64_t b0 = begin_dev ? *begin_dev : 0;
  keys += b0;
  vals += b0;
  const int64_t n = *end_dev - b0;
  const int64_t chunk = tile_entries(n, target);
  const int64_t ntiles = (n + chunk - 1) / chunk;
  uint32_t gb = 0;  // stages this warp has consumed (all tiles): stage gb % NS, phase gb / NS
  bool failed = false;
  // tiles are taken in order from a counter (zero before the launch): a warp
  // that drew cheap tiles takes more, so the slowest warp does not set the pace
  auto next_tile = [&]() -> int64_t {
    uint32_t v = 0;
    if (lane == 0) v = atomicAdd(tile_next, 1u);
    return int64_t(__shfl_sync(0xffffffffu, v, 0));
  };

  for (int64_t t = next_tile(); t < ntiles && !failed; t = next_tile()) {
    const int64_t s0 = t * chunk;
    const int m = int((s0 + chunk < n) ? chunk : n - s0);  // entries in this tile
    const uint32_t* tk = keys + s0;
    const uint32_t* tv = vals + s0;
    const uint32_t prev_key = s0 > 0 ? keys[s0 - 1] : kNoKey;
    const uint32_t next_key = s0 + m < n ? keys[s0 + m] : kNoKey;
    const uint32_t last_key = tk[m - 1];
    const uint32_t nb = uint32_t((m + BR - 1) / BR);  // stages in this tile
    const uint32_t gb_tile = gb;
    auto ld_k = [&](int c) { const int i = c * 32 + lane; return i < m ? __ldcs(tk + i) : kNoKey; };
    auto ld_p = [&](int c) { const int i = c * 32 + lane; return i < m ? __ldcs(tv + i) : 0u; };
    // bits of the entries of batch c (keys kc) that end a row; kn0 = first key of batch c + 1
    auto end_bits = [&](int c, uint32_t kc, uint32_t kn0) {
      const int cnt = m - c * 32;  // may be <= 0 or > 32
      uint32_t nk = __shfl_down_sync(0xffffffffu, kc, 1);
      if (lane == 31) nk = kn0;
      if (lane == cnt - 1) nk = next_key;  // the tile's last entry
      const bool e = lane < cnt && nk != kc;
      if (e) {  // bring the finished row's table row and state to L2
        const char* rp = static_cast<const char*>(u.table) + int64_t(kc & row_mask) * RB;
#pragma unroll
        for (int b = 0; b < RB; b += 128) prefetch_l2(rp + b);
        if (adagrad) prefetch_l2(u.state + (kc & row_mask));
      }
      return __ballot_sync(0xffffffffu, e);
    };
    uint32_t kc = ld_k(0), pc = ld_p(0), kn = ld_k(1), pn = ld_p(1), kn2 = ld_k(2), pn2 = ld_p(2);
    // copy stage tb of this tile (its rows belong to batch tb / SPC, which is c or c + 1)
    auto issue = [&](uint32_t tb, int c) {
      if (tb >= nb || (t == skip_tile && tb == 0)) return;  // (test hook: a stage that never arrives)
      const uint32_t p = (int(tb / SPC) == c) ? pc : pn;
      const int first = int(tb % SPC) * BR;
      const int left = m - int(tb) * BR;
      const int rows = left < BR ? left : BR;
      const uint32_t st = (gb_tile + tb) & (NS - 1);
      const uint32_t bar = bar0 + 8 * st;
      if (lane == first) bulk::arrive_expect_tx(bar, uint32_t(rows * RB));
      __syncwarp();
      const uint32_t r = uint32_t(lane - first);
      if (r < uint32_t(rows)) bulk::copy_g2s(data0 + st * RG::kStageBytes + r * RB, gbytes + uint64_t(p) * RB, RB, bar, pol);
    };
    for (int k = 0; k < NS - 1; ++k) issue(uint32_t(k), 0);

    bool from_prev = (__shfl_sync(0xffffffffu, kc, 0) == prev_key);
    if (lane == 0 && !from_prev) head_cont[t] = 0;  // every tile's flag is defined
    float acc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
    uint32_t em = end_bits(0, kc, __shfl_sync(0xffffffffu, kn, 0));

    // the entries of stage st (eb = its first entry in batch c); FULL: all BR present
    // (inlined at two call sites with a constant `full`: the bounds test folds away)
    auto consume = [&](bool full, int eb, int cnt, uint32_t st, uint32_t bm, float (&w)[BR][EPL], float my_s) {
      const unsigned char* sp = data + st * RG::kStageBytes;
#pragma unroll
      for (int r = 0; r < BR; ++r) {
        if (full || eb + r < cnt) {
          acc_slice<BF16, EPL>(sp, r, lane, acc);
          if ((bm >> r) & 1u) {  // entry eb + r is its row's last
            if (from_prev) {     // the row began in an earlier tile and ends here
#pragma unroll
              for (int q = 0; q < EPL; ++q) carry_head[t * D + lane * EPL + q] = acc[q];
              if (lane == 0) head_cont[t] = 0;
              from_prev = false;
            } else {
              const uint32_t row = __shfl_sync(0xffffffffu, kc, eb + r) & row_mask;
              const float s_old = __shfl_sync(0xffffffffu, my_s, eb + r);
              apply_update<BF16, EPL>(u, row, w[r], s_old, acc, lane);
            }
#pragma unroll
            for (int q = 0; q < EPL; ++q) acc[q] = 0.f;
          }
        }
      }
    };

    for (int c = 0; c * 32 < m; ++c) {
      const int cnt = (m - c * 32 < 32) ? m - c * 32 : 32;
      const uint32_t em_next = end_bits(c + 1, kn, __shfl_sync(0xffffffffu, kn2, 0));
      for (int i = 0; i < SPC; ++i) {
        const int eb = i * BR;
        if (eb >= cnt) break;
        const uint32_t tb = uint32_t(c * SPC + i);
        issue(tb + NS - 1, c);
        // table slices and states of the rows this stage finishes
        const uint32_t bm = (em >> eb) & ((BR == 32) ? 0xffffffffu : ((1u << BR) - 1u));
        float w[BR][EPL];
        float my_s = 0.f;
        if (bm) {
#pragma unroll
          for (int r = 0; r < BR; ++r) {
            if ((bm >> r) & 1u) {
              const uint32_t row = __shfl_sync(0xffffffffu, kc, eb + r) & row_mask;
              load_slice<BF16, EPL, false>(u.table, row, lane, w[r]);
            }
          }
          if (adagrad && ((em >> lane) & 1u) && uint32_t(lane - eb) < uint32_t(BR)) my_s = u.state[kc & row_mask];
        }
        const uint32_t st = (gb_tile + tb) & (NS - 1);
        const uint32_t par = ((gb_tile + tb) / NS) & 1u;
        if (!bulk::warp_wait(bar0 + 8 * st, par, wait_ns)) {
          // give up: record it, let this warp's other copies land, stop
          if (lane == 0) set_err(err, FS_ERR_TIMEOUT);
          for (uint32_t k = 1; k < NS; ++k) {
            const uint32_t g2 = gb_tile + tb + k;
            if (tb + k < nb) bulk::warp_wait(bar0 + 8 * (g2 & (NS - 1)), (g2 / NS) & 1u, wait_ns);
          }
          failed = true;
          break;
        }
        if (eb + BR <= cnt) consume(true, eb, cnt, st, bm, w, my_s);
        else consume(false, eb, cnt, st, bm, w, my_s);
        __syncwarp();  // every lane is done with the stage before it is refilled
      }
      if (failed) break;
      kc = kn;
      pc = pn;
      kn = kn2;
      pn = pn2;
      kn2 = ld_k(c + 3);
      pn2 = ld_p(c + 3);
      em = em_next;
    }
    if (failed) break;
    gb = gb_tile + nb;
    // a row still open continues into the next tile
    if (last_key == next_key) {
      if (from_prev) {  // spans the whole tile
#pragma unroll
        for (int q = 0; q < EPL; ++q) carry_head[t * D + lane * EPL + q] = acc[q];
        if (lane == 0) {
          head_cont[t] = 1;
          tail_flag[t] = 0;
        }
      } else {  // starts here
#pragma unroll
        for (int q = 0; q < EPL; ++q) carry_tail[t * D + lane * EPL + q] = acc[q];
        if (lane == 0) tail_flag[t] = 1;
      }
    } else if (lane == 0) {
      tail_flag[t] = 0;
    }
  }
  __syncwarp();
  if (lane == 0)
    for (int s = 0; s < NS; ++s) bulk::mbar_inval(bar0 + 8 * s);
}

// Carry chains of rows that cross tile boundaries.  A chain is the tail
// carry of its starting tile, then the head carries of the following tiles
// up to the first whose head does not continue.  A Zipf-hot row crosses
// thousands of tiles, so whole aligned blocks of kCarryBlock continuing
// tiles are summed first (block_sum_kernel, one warp per block), and the
// chain's owner adds block sums where it can and single tiles elsewhere.
// Sums are in fp64: the error stays at the level of one tile's fp32 sum.
// The order is fixed, so the result is identical run to run.
constexpr int kCarryBlock = 32;

template <int EPL>
__global__ void __launch_bounds__(kThreads) block_sum_kernel(const int64_t* begin_dev, const int64_t* end_dev,
                                                             const float* carry_head, const uint8_t* head_cont,
                                                             double* block_sum, uint8_t* block_full, int64_t target) {
  constexpr int D = 32 * EPL;
  const int64_t b0 = begin_dev ? *begin_dev : 0;
  const int64_t n = *end_dev - b0;
  const int64_t chunk = tile_entries(n, target);
  const int64_t ntiles = (n + chunk - 1) / chunk;
  const int64_t nblocks = ntiles / kCarryBlock;  // whole blocks only
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t bk = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; bk < nblocks; bk += nwarps) {
    const int64_t v0 = bk * kCarryBlock;
    const bool full = __all_sync(0xffffffffu, head_cont[v0 + lane] == 1);
    if (lane == 0) block_full[bk] = full ? 1 : 0;
    if (!full) continue;
    double acc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] = 0.0;
    for (int j = 0; j < kCarryBlock; j += 8) {
      float c[8][EPL];
#pragma unroll
      for (int q = 0; q < 8; ++q)
#pragma unroll
        for (int i = 0; i < EPL; ++i) c[q][i] = carry_head[(v0 + j + q) * D + lane * EPL + i];
#pragma unroll
      for (int q = 0; q < 8; ++q)
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc[i] += double(c[q][i]);
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) block_sum[bk * D + lane * EPL + i] = acc[i];
  }
}

template <bool BF16, int EPL>
__global__ void __launch_bounds__(kThreads) fixup_kernel(const uint32_t* __restrict__ keys, const int64_t* begin_dev,
                                                         const int64_t* end_dev, uint32_t row_mask, UpdateArgs u,
                                                         const float* carry_head, const float* carry_tail,
                                                         const uint8_t* head_cont, const uint8_t* tail_flag,
                                                         const double* block_sum, const uint8_t* block_full,
                                                         int64_t target) {
  constexpr int D = 32 * EPL;
  const int64_t b0 = begin_dev ? *begin_dev : 0;
  keys += b0;
  const int64_t n = *end_dev - b0;
  const int64_t chunk = tile_entries(n, target);
  const int64_t ntiles = (n + chunk - 1) / chunk;
  const int64_t nblocks = ntiles / kCarryBlock;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < ntiles; t += nwarps) {
    if (!tail_flag[t]) continue;
    const uint32_t row = keys[(t + 1) * chunk - 1] & row_mask;
    double acc64[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc64[i] = double(carry_tail[t * D + lane * EPL + i]);
    int64_t v = t + 1;
    while (v < ntiles) {
      if (v % kCarryBlock == 0 && v / kCarryBlock < nblocks) {
        // the run of full blocks starting here (one flag per lane, up to 32 blocks at a time),
        // their sums added in block order with Q loads in flight (a Zipf-hot row's chain
        // crosses hundreds of blocks: one dependent load per block would set the pace)
        const int64_t b0 = v / kCarryBlock;
        const bool f = b0 + lane < nblocks && block_full[b0 + lane];
        const unsigned fm = __ballot_sync(0xffffffffu, f);
        const int run = (fm == 0xffffffffu) ? 32 : (__ffs(~fm) - 1);
        if (run > 0) {
          constexpr int Q = EPL >= 8 ? 2 : (EPL >= 4 ? 4 : 8);
          int q = 0;
          for (; q + Q <= run; q += Q) {
            double c[Q][EPL];
#pragma unroll
            for (int qq = 0; qq < Q; ++qq)
#pragma unroll
              for (int i = 0; i < EPL; ++i) c[qq][i] = block_sum[(b0 + q + qq) * D + lane * EPL + i];
#pragma unroll
            for (int qq = 0; qq < Q; ++qq)
#pragma unroll
              for (int i = 0; i < EPL; ++i) acc64[i] += c[qq][i];
          }
          for (; q < run; ++q)
#pragma unroll
            for (int i = 0; i < EPL; ++i) acc64[i] += block_sum[(b0 + q) * D + lane * EPL + i];
          v += int64_t(run) * kCarryBlock;
          continue;
        }
      }
      // single tiles up to the end of v's block: stop at the first head
      // that does not continue
      const int64_t vend = (v / kCarryBlock + 1) * kCarryBlock < ntiles ? (v / kCarryBlock + 1) * kCarryBlock : ntiles;
      const int cntw = int(vend - v);
      const uint8_t hc = lane < cntw ? head_cont[v + lane] : uint8_t(1);
      const unsigned stop = __ballot_sync(0xffffffffu, lane < cntw && hc == 0);
      const int last = stop ? (__ffs(stop) - 1) : (cntw - 1);
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
      v = vend;
    }
    float acc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] = float(acc64[i]);
    update_row<BF16, EPL>(u, row, acc, lane);
  }
}

template <bool BF16, int EPL>
void launch_reduce(const uint32_t* k, const uint32_t* v, const int64_t* begin_dev, const int64_t* end_dev,
                   uint32_t row_mask, const void* grads, UpdateArgs u, float* ch, float* ct, uint8_t* hc,
                   uint8_t* tf, double* bsum, uint8_t* bfull, uint32_t* tile_next, int32_t* err, cudaStream_t st) {
  const unsigned sms = unsigned(sm_count());
  int64_t target = 0;  // tiles the range is cut into, per reducing warp: six (dynamic) or three (static)
  if (aligned(grads, 16)) {
    // gradient rows by bulk copy (needs 16-byte aligned rows)
    constexpr int RB = 32 * EPL * (BF16 ? 2 : 4);
    using RG = Ring<RB>;
    auto kern = reduce_ring_kernel<BF16, EPL, RG::kMinBlocks>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, RG::kBlockBytes);
    const unsigned grid = sms * RG::kMinBlocks;
    target = 6 * int64_t(grid) * (kThreads / 32);
    cudaMemsetAsync(tile_next, 0, sizeof(uint32_t), st);
    kern<<<grid, kThreads, RG::kBlockBytes, st>>>(k, v, begin_dev, end_dev, row_mask, grads, u, ch, ct, hc, tf, err,
                                                  uint64_t(spin_limit()) * 256u, debug_skip_tile(), target, tile_next);
  } else {
    // 8 gradient rows in flight per warp (fewer for wide rows) and 4 blocks
    // per SM fit the 64-register budget without spills
    constexpr int G = (16 / EPL) > 8 ? 8 : (16 / EPL);
    const unsigned grid = sms * 4;
    target = 3 * int64_t(grid) * (kThreads / 32);
    reduce_kernel<BF16, EPL, G, 4><<<grid, kThreads, 0, st>>>(k, v, begin_dev, end_dev, row_mask, grads, u, ch, ct,
                                                             hc, tf, target);
  }
  block_sum_kernel<EPL><<<sms * (2048 / kThreads), kThreads, 0, st>>>(begin_dev, end_dev, ch, hc, bsum, bfull, target);
  fixup_kernel<BF16, EPL><<<sms * (2048 / kThreads), kThreads, 0, st>>>(k, begin_dev, end_dev, row_mask, u, ch, ct,
                                                                         hc, tf, bsum, bfull, target);
}

// Number of sorted keys below `bound` (one thread; keys ascending).
__global__ void count_below_kernel(const uint32_t* keys, const int64_t* n_dev, uint32_t bound, int64_t* out) {
  int64_t lo = 0, hi = *n_dev;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (keys[mid] < bound) lo = mid + 1; else hi = mid;
  }
  *out = lo;
}

struct BwdLayout {
  radix::SortPlan plan;
  int64_t max_tiles = 0, max_blocks = 0;
  size_t carry_bytes = 0, flag_bytes = 0, block_bytes = 0, block_flag_bytes = 0;
};

BwdLayout bwd_layout(int64_t T, int64_t R, int32_t dim) {
  BwdLayout L;
  L.plan = radix::SortPlan(T, radix::bits_for(uint64_t(R > 0 ? R - 1 : 0)));
  L.max_tiles = (T + kMinChunk - 1) / kMinChunk;
  L.carry_bytes = align_up(size_t(L.max_tiles) * size_t(dim) * sizeof(float));
  L.flag_bytes = align_up(size_t(L.max_tiles));
  L.max_blocks = L.max_tiles / kCarryBlock + 1;
  L.block_bytes = align_up(size_t(L.max_blocks) * size_t(dim) * sizeof(double));
  L.block_flag_bytes = align_up(size_t(L.max_blocks));
  return L;
}

int epl_for(int32_t dim, fs_dtype dtype) {
  if (dim % 32 != 0) return 0;
  int e = dim / 32;
  if (e == 1 || e == 2 || e == 4) return e;
  if (e == 8 && dtype == FS_BF16) return e;
  return 0;
}

// Pointers into the backward workspace.  They follow from (T, R, dim, phase)
// alone, so the sort, the row-sorted gather and the update of one batch find
// the sorted entries where the sort left them.
struct BwdWs {
  BwdLayout L;
  radix::SortWs W;
  int kb = 0;                     // bits of the largest row index
  uint32_t row_mask = 0xFFFFFFFFu;
  uint32_t *sk = nullptr, *sv = nullptr;  // sorted (phase bit | row) keys, positions
  float *carry_head = nullptr, *carry_tail = nullptr;
  uint8_t *head_cont = nullptr, *tail_flag = nullptr;
  double* block_sum = nullptr;
  uint8_t* block_full = nullptr;
  int64_t* n_first = nullptr;     // sorted entries of collision rows (two-phase mode)
  uint32_t* tile_next = nullptr;
};

bool carve_bwd(int64_t T, int64_t R, int32_t dim, fs_phase phase, void* ws, size_t ws_bytes, BwdWs& B) {
  B.kb = radix::bits_for(uint64_t(R - 1));
  B.L = bwd_layout(T, R, dim);
  if (phase == FS_PHASE_COLLISION_THEN_EXCLUSIVE) {
    B.L.plan = radix::SortPlan(T, B.kb + 1);
    B.row_mask = (1u << B.kb) - 1u;
  }
  WsCursor cur(ws, ws_bytes);
  if (!radix::carve_sort_ws(B.L.plan, cur, B.W)) return false;
  B.sk = radix::sorted_keys(B.L.plan, B.W);
  B.sv = radix::sorted_values(B.L.plan, B.W);
  B.carry_head = cur.take<float>(size_t(B.L.max_tiles) * dim);
  B.carry_tail = cur.take<float>(size_t(B.L.max_tiles) * dim);
  B.head_cont = cur.take<uint8_t>(size_t(B.L.max_tiles));
  B.tail_flag = cur.take<uint8_t>(size_t(B.L.max_tiles));
  B.block_sum = cur.take<double>(size_t(B.L.max_blocks) * dim);
  B.block_full = cur.take<uint8_t>(size_t(B.L.max_blocks));
  B.n_first = cur.take<int64_t>(1);
  B.tile_next = cur.take<uint32_t>(1);
  return cur.ok;
}

// Row-sorted gather: out[pos] = table[key & row_mask] over the sorted entries
// [0, *n_dev).  Equal rows are adjacent, so a row leaves DRAM once and its
// further reads hit L1/L2; the writes land at the entries' batch-major
// positions (whole rows, scattered).  Rows of 16 * VPR bytes, VPR in
// {4, 8, 16, 32}: a warp instruction moves RPI = 32 / VPR rows, each lane keeps
// U independent 16-byte loads in flight; one coalesced load per warp
// iteration brings the keys and positions of RPI * U entries.  An entry whose
// row or position is out of range (the workspace does not hold this batch's
// sort) sets FS_ERR_BAD_OFFSETS and is skipped.
constexpr int kGatherThreads = 256;

// (three blocks per SM: 85 registers hold the U row loads and the next
// iteration's entries; at four blocks the spills cost more than the extra warps)
template <int VPR>
__global__ void __launch_bounds__(kGatherThreads, 3) gather_sorted_kernel(const int4* __restrict__ table, int64_t R,
                                                                       const uint32_t* __restrict__ keys,
                                                                       const uint32_t* __restrict__ pos,
                                                                       const int64_t* __restrict__ n_dev, int64_t T,
                                                                       uint32_t row_mask, int4* __restrict__ out,
                                                                       int32_t* err) {
  constexpr int RPI = 32 / VPR;
  constexpr int U = (32 / RPI) < 8 ? (32 / RPI) : 8;
  constexpr int RPW = RPI * U;
  static_assert(RPW <= 32, "one lane per entry");
  int64_t n = *n_dev;
  n = n < 0 ? 0 : (n > T ? T : n);
  const int lane = threadIdx.x & 31;
  const int sub = lane / VPR, c = lane % VPR;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t stride = nwarps * RPW;
  // the keys and positions of the warp's next iteration are loaded before the
  // current iteration's rows, so the entry stream's latency overlaps them
  uint32_t nk = 0, np = 0xFFFFFFFFu;
  auto load_entries = [&](int64_t e) {
    nk = 0;
    np = 0xFFFFFFFFu;  // position all ones: no entry
    if (lane < RPW && e + lane < n) {
      nk = __ldcs(keys + e + lane);
      np = __ldcs(pos + e + lane);
    }
  };
  int64_t e0 = ((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * RPW;
  load_entries(e0);
  for (; e0 < n; e0 += stride) {
    uint32_t my_row = nk & row_mask, my_pos = np;
    const bool live = lane < RPW && e0 + lane < n;
    load_entries(e0 + stride);
    if (live && (int64_t(my_row) >= R || int64_t(my_pos) >= T)) {
      set_err(err, FS_ERR_BAD_OFFSETS);
      my_pos = 0xFFFFFFFFu;
    }
    int4 v[U];
    uint32_t p[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t row = __shfl_sync(0xffffffffu, my_row, u * RPI + sub);
      p[u] = __shfl_sync(0xffffffffu, my_pos, u * RPI + sub);
      if (p[u] != 0xFFFFFFFFu) v[u] = __ldg(table + int64_t(row) * VPR + c);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (p[u] != 0xFFFFFFFFu) __stcs(out + int64_t(p[u]) * VPR + c, v[u]);
  }
}

}  // namespace
}  // namespace fs

using namespace fs;

extern "C" size_t fs_emb_backward_adagrad_workspace_size(int64_t T, int64_t num_rows, int32_t dim, fs_dtype dtype) {
  (void)dtype;
  if (T < 0 || num_rows < 1 || dim < 1) return 0;
  BwdLayout L = bwd_layout(T, num_rows, dim);
  // the single-call two-phase mode sorts one more key bit (the phase)
  const size_t sort_bytes = std::max(L.plan.bytes(), radix::SortPlan(T, L.plan.key_bits + 1).bytes());
  return sort_bytes + 2 * L.carry_bytes + 2 * L.flag_bytes + L.block_bytes + L.block_flag_bytes +
         align_up(sizeof(int64_t)) + align_up(sizeof(uint32_t)) + 256;
}

namespace fs {
namespace {

// Host checks shared by the one-call update and the row-sorted calls.
fs_status check_bwd(int64_t T, int64_t num_rows, int32_t dim, fs_dtype dtype, fs_phase phase, int32_t* err) {
  if (T < 0 || T > INT32_MAX || num_rows < 1 || num_rows >= (int64_t(1) << 32) || !err) return FS_ERR_INVALID_ARG;
  if (dtype != FS_F32 && dtype != FS_BF16) return FS_ERR_INVALID_ARG;
  if (phase != FS_PHASE_ALL && phase != FS_PHASE_COLLISION && phase != FS_PHASE_EXCLUSIVE &&
      phase != FS_PHASE_COLLISION_THEN_EXCLUSIVE)
    return FS_ERR_INVALID_ARG;
  if (epl_for(dim, dtype) == 0) return FS_ERR_INVALID_ARG;
  return FS_OK;
}

// The update's sort: (phase bit | row, position) pairs of the entries the
// phase keeps, ascending; in the two-phase mode also the number of collision
// entries (they sort first).
fs_status sort_rows(const BwdWs& B, const int64_t* ids, int64_t num_rows, const uint8_t* is_co,
                    const uint32_t* co_rows, fs_phase phase, int32_t* err, cudaStream_t st, int* launches) {
  uint32_t *sk = nullptr, *sv = nullptr;
  fs_status s = (phase != FS_PHASE_ALL && co_rows)
                    ? radix::run_sort(SrcRows<true>{ids, is_co, co_rows, int(phase), num_rows, B.kb}, B.L.plan,
                                      B.W, err, st, &sk, &sv, launches)
                    : radix::run_sort(SrcRows<false>{ids, is_co, co_rows, int(phase), num_rows, B.kb}, B.L.plan,
                                      B.W, err, st, &sk, &sv, launches);
  if (s != FS_OK) return s;
  if (phase == FS_PHASE_COLLISION_THEN_EXCLUSIVE) {
    count_below_kernel<<<1, 1, 0, st>>>(B.sk, B.W.pass.n_valid, 1u << B.kb, B.n_first);
    ++*launches;
  }
  return FS_OK;
}

// Segment-reduce + row update of the sorted entries: one range, or in the
// two-phase mode the collision rows in a first launch and the exclusive rows
// in a second, in stream order.
void update_rows(const BwdWs& B, void* table, float* state, int32_t dim, fs_dtype dtype, fs_optim optim,
                 const void* grads, fs_phase phase, float lr, float eps, int32_t* err, cudaStream_t st,
                 int* launches) {
  const int epl = epl_for(dim, dtype);
  UpdateArgs u{table, optim == FS_ROWWISE_ADAGRAD ? state : nullptr, int(optim), lr, eps};
  const bool bf = dtype == FS_BF16;
  auto reduce_range = [&](const int64_t* begin_dev, const int64_t* end_dev, uint32_t row_mask) {
#define FS_REDUCE(BF, E) \
  launch_reduce<BF, E>(B.sk, B.sv, begin_dev, end_dev, row_mask, grads, u, B.carry_head, B.carry_tail, B.head_cont, \
                       B.tail_flag, B.block_sum, B.block_full, B.tile_next, err, st)
    switch (epl) {
      case 1: if (bf) FS_REDUCE(true, 1); else FS_REDUCE(false, 1); break;
      case 2: if (bf) FS_REDUCE(true, 2); else FS_REDUCE(false, 2); break;
      case 4: if (bf) FS_REDUCE(true, 4); else FS_REDUCE(false, 4); break;
      default: FS_REDUCE(true, 8); break;
    }
#undef FS_REDUCE
    *launches += 3;
  };
  if (phase == FS_PHASE_COLLISION_THEN_EXCLUSIVE) {
    reduce_range(nullptr, B.n_first, B.row_mask);
    reduce_range(B.n_first, B.W.pass.n_valid, B.row_mask);
  } else {
    reduce_range(nullptr, B.W.pass.n_valid, 0xFFFFFFFFu);
  }
}

fs_status check_update_args(void* table, float* state, int32_t dim, fs_dtype dtype, fs_optim optim,
                            const void* grads) {
  if (optim != FS_SGD && optim != FS_ROWWISE_ADAGRAD) return FS_ERR_INVALID_ARG;
  if (optim == FS_ROWWISE_ADAGRAD && !state) return FS_ERR_INVALID_ARG;
  if (!table || !grads) return FS_ERR_INVALID_ARG;
  const size_t vec = size_t(epl_for(dim, dtype)) * (dtype == FS_F32 ? 4 : 2);
  if (!aligned(table, vec) || !aligned(grads, vec) || (state && !aligned(state, 4))) return FS_ERR_ALIGNMENT;
  return FS_OK;
}

}  // namespace
}  // namespace fs

extern "C" fs_status fs_emb_backward_adagrad(void* table, float* state, int64_t num_rows, int32_t dim, fs_dtype dtype,
                                             fs_optim optim, const int64_t* ids, const void* grads, int64_t T,
                                             const uint8_t* is_co, const uint32_t* co_rows, fs_phase phase,
                                             float lr, float eps, int32_t* err, void* ws, size_t ws_bytes,
                                             fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  fs_status s = check_bwd(T, num_rows, dim, dtype, phase, err);
  if (s != FS_OK) return s;
  if (optim != FS_SGD && optim != FS_ROWWISE_ADAGRAD) return FS_ERR_INVALID_ARG;
  if (optim == FS_ROWWISE_ADAGRAD && !state) return FS_ERR_INVALID_ARG;
  if (T == 0) return FS_OK;
  if (!ids) return FS_ERR_INVALID_ARG;
  if ((s = check_update_args(table, state, dim, dtype, optim, grads)) != FS_OK) return s;
  if (phase != FS_PHASE_ALL && (is_co == nullptr) == (co_rows == nullptr)) return FS_ERR_INVALID_ARG;
  if (co_rows && !aligned(co_rows, 4)) return FS_ERR_ALIGNMENT;
  if (!aligned(ids, 8)) return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_emb_backward_adagrad_workspace_size(T, num_rows, dim, dtype) || !ws) return FS_ERR_WORKSPACE;

  if (phase == FS_PHASE_COLLISION_THEN_EXCLUSIVE && radix::bits_for(uint64_t(num_rows - 1)) > 30) {
    // the phase bit does not fit beside the row bits: two calls, same result
    s = fs_emb_backward_adagrad(table, state, num_rows, dim, dtype, optim, ids, grads, T, is_co, co_rows,
                                FS_PHASE_COLLISION, lr, eps, err, ws, ws_bytes, stream);
    if (s != FS_OK) return s;
    return fs_emb_backward_adagrad(table, state, num_rows, dim, dtype, optim, ids, grads, T, is_co, co_rows,
                                   FS_PHASE_EXCLUSIVE, lr, eps, err, ws, ws_bytes, stream);
  }
  BwdWs B;
  if (!carve_bwd(T, num_rows, dim, phase, ws, ws_bytes, B)) return FS_ERR_WORKSPACE;
  int launches = 0;
  if ((s = sort_rows(B, ids, num_rows, is_co, co_rows, phase, err, st, &launches)) != FS_OK) return s;
  update_rows(B, table, state, dim, dtype, optim, grads, phase, lr, eps, err, st, &launches);
  count_launch(launches);
  return launch_status();
}

// ------------------------------------------------------------ row-sorted path

namespace fs {
namespace {

// The three row-sorted calls accept the phases whose sort keeps every entry
// with a valid ID (all of them, or collision and exclusive ones both), and the
// two-phase mode only while the phase bit fits beside the row bits.
fs_status check_sorted(int64_t T, int64_t num_rows, int32_t dim, fs_dtype dtype, fs_phase phase, int32_t* err,
                       const void* ws, size_t ws_bytes) {
  fs_status s = check_bwd(T, num_rows, dim, dtype, phase, err);
  if (s != FS_OK) return s;
  if (phase != FS_PHASE_ALL && phase != FS_PHASE_COLLISION_THEN_EXCLUSIVE) return FS_ERR_INVALID_ARG;
  if (phase == FS_PHASE_COLLISION_THEN_EXCLUSIVE && radix::bits_for(uint64_t(num_rows - 1)) > 30)
    return FS_ERR_INVALID_ARG;
  if (T > 0 && (ws_bytes < fs_emb_backward_adagrad_workspace_size(T, num_rows, dim, dtype) || !ws))
    return FS_ERR_WORKSPACE;
  return FS_OK;
}

}  // namespace
}  // namespace fs

extern "C" fs_status fs_emb_sort_rows(int64_t num_rows, int32_t dim, fs_dtype dtype, const int64_t* ids, int64_t T,
                                      const uint8_t* is_co, const uint32_t* co_rows, fs_phase phase, int32_t* err,
                                      void* ws, size_t ws_bytes, fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  fs_status s = check_sorted(T, num_rows, dim, dtype, phase, err, ws, ws_bytes);
  if (s != FS_OK) return s;
  if (T == 0) return FS_OK;
  if (!ids) return FS_ERR_INVALID_ARG;
  if (phase != FS_PHASE_ALL && (is_co == nullptr) == (co_rows == nullptr)) return FS_ERR_INVALID_ARG;
  if (co_rows && !aligned(co_rows, 4)) return FS_ERR_ALIGNMENT;
  if (!aligned(ids, 8)) return FS_ERR_ALIGNMENT;
  BwdWs B;
  if (!carve_bwd(T, num_rows, dim, phase, ws, ws_bytes, B)) return FS_ERR_WORKSPACE;
  int launches = 0;
  if ((s = sort_rows(B, ids, num_rows, is_co, co_rows, phase, err, st, &launches)) != FS_OK) return s;
  count_launch(launches);
  return launch_status();
}

// ------------------------------------------------------------ per-shard sort

namespace fs {
namespace {

// Bit split of the per-shard sort: a row's offset inside its shard has lb
// bits (shards of block = ceil(R / n) rows); pass 1 sorts the low b1 of them,
// pass 2 the other lb2 with the phase bit (two-phase mode) above them.
struct ShardSortPlan {
  int64_t block = 1;
  int lb = 1, ph = 0, b1 = 1, lb2 = 0;
  bool ok = false;
};

ShardSortPlan shard_sort_plan(int64_t R, int32_t n, fs_phase phase) {
  ShardSortPlan P;
  P.block = (R + n - 1) / n;
  P.lb = radix::bits_for(uint64_t(P.block - 1));
  P.ph = phase == FS_PHASE_COLLISION_THEN_EXCLUSIVE ? 1 : 0;
  P.b1 = (P.lb + P.ph) / 2;
  if (P.b1 < 1) P.b1 = 1;
  if (P.b1 > P.lb) P.b1 = P.lb;
  P.lb2 = P.lb - P.b1;
  P.ok = P.b1 <= 10 && P.lb2 + P.ph <= 10;
  return P;
}

size_t sharded_extra_bytes(int64_t T, int32_t n) {
  WsCounter c;
  radix::take_seg_ws(T, n, c, nullptr);
  return c.used;
}

}  // namespace
}  // namespace fs

extern "C" size_t fs_emb_sort_rows_sharded_workspace_size(int64_t T, int64_t num_rows, int32_t dim, fs_dtype dtype,
                                                          int32_t n) {
  if (T < 0 || num_rows < 1 || dim < 1 || n < 1 || n > radix::kSegThreads) return 0;
  return fs_emb_backward_adagrad_workspace_size(T, num_rows, dim, dtype) + sharded_extra_bytes(T, n) + 256;
}

extern "C" fs_status fs_emb_sort_rows_sharded(int64_t num_rows, int32_t dim, fs_dtype dtype, const int64_t* sm_ids,
                                              const int32_t* pos, int64_t T, const int64_t* shard_offsets, int32_t n,
                                              const uint8_t* is_co, const uint32_t* co_rows, fs_phase phase,
                                              int32_t* err, void* ws, size_t ws_bytes, fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  fs_status s = check_sorted(T, num_rows, dim, dtype, phase, err, ws, ws_bytes);
  if (s != FS_OK) return s;
  if (n < 1 || n > radix::kSegThreads || !shard_offsets) return FS_ERR_INVALID_ARG;
  const ShardSortPlan P = shard_sort_plan(num_rows, n, phase);
  if (!P.ok) return FS_ERR_INVALID_ARG;
  if (T == 0) return FS_OK;
  const bool two = phase == FS_PHASE_COLLISION_THEN_EXCLUSIVE;
  if (!sm_ids || !pos || (two && (is_co == nullptr) == (co_rows == nullptr))) return FS_ERR_INVALID_ARG;
  if (!aligned(sm_ids, 8) || !aligned(pos, 4) || !aligned(shard_offsets, 8) || (co_rows && !aligned(co_rows, 4)))
    return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_emb_sort_rows_sharded_workspace_size(T, num_rows, dim, dtype, n)) return FS_ERR_WORKSPACE;
  BwdWs B;
  if (!carve_bwd(T, num_rows, dim, phase, ws, ws_bytes, B)) return FS_ERR_WORKSPACE;
  // the passes' own scratch lies behind the layout the gather and the update read
  const size_t base = fs_emb_backward_adagrad_workspace_size(T, num_rows, dim, dtype);
  WsCursor cur(static_cast<char*>(ws) + base, ws_bytes - base);
  radix::SegWs W;
  radix::take_seg_ws(T, n, cur, &W);
  if (!cur.ok) return FS_ERR_WORKSPACE;
  // pass 2 writes where fs_emb_gather_sorted / fs_emb_update_sorted look; pass 1 into the other buffers
  uint32_t* k1 = (B.sk == B.W.k[0]) ? B.W.k[1] : B.W.k[0];
  uint32_t* v1 = (B.sv == B.W.v[0]) ? B.W.v[1] : B.W.v[0];
  int launches = 1;
  radix::seg_tiles_kernel<<<1, radix::kSegThreads, 0, st>>>(shard_offsets, n, T, W.seg_off[0], W.tile_base[0], err);
  if (two && co_rows) {
    const SrcShardRows<true> s1{sm_ids, nullptr, co_rows, num_rows, P.block, B.kb, B.row_mask};
    radix::run_seg_pass(s1, DstGatherPos<int32_t>{k1, v1, pos}, 0, P.b1, P.b1, W, 0, B.W.pass.n_valid, nullptr, err, st,
                        &launches);
  } else {
    const SrcShardRows<false> s1{sm_ids, two ? is_co : nullptr, nullptr, num_rows, P.block, B.kb, B.row_mask};
    radix::run_seg_pass(s1, DstGatherPos<int32_t>{k1, v1, pos}, 0, P.b1, P.b1, W, 0, B.W.pass.n_valid, nullptr, err, st,
                        &launches);
  }
  const SrcShardRows2 s2{k1, P.block, B.kb, B.row_mask, P.lb2, two};
  radix::run_seg_pass(s2, DstGatherPos<uint32_t>{B.sk, B.sv, v1}, P.b1, P.lb2 + P.ph, P.lb2, W, 1, B.W.pass.n_valid,
                      two ? B.n_first : nullptr, nullptr, st, &launches);
  count_launch(launches);
  return launch_status();
}

extern "C" fs_status fs_emb_gather_sorted(const void* table, int64_t num_rows, int32_t dim, fs_dtype dtype, int64_t T,
                                          fs_phase phase, void* out, int32_t* err, void* ws, size_t ws_bytes,
                                          fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  fs_status s = check_sorted(T, num_rows, dim, dtype, phase, err, ws, ws_bytes);
  if (s != FS_OK) return s;
  if (T == 0) return FS_OK;
  if (!table || !out) return FS_ERR_INVALID_ARG;
  if (!aligned(table, 16) || !aligned(out, 16)) return FS_ERR_ALIGNMENT;
  BwdWs B;
  if (!carve_bwd(T, num_rows, dim, phase, ws, ws_bytes, B)) return FS_ERR_WORKSPACE;
  const int vpr = int(int64_t(dim) * (dtype == FS_F32 ? 4 : 2) / 16);
  const unsigned grid = unsigned(sm_count()) * (2048 / kGatherThreads);
  const int4* tb = static_cast<const int4*>(table);
  int4* ob = static_cast<int4*>(out);
  const int64_t* n = B.W.pass.n_valid;
#define FS_GATHER_SORTED(V) \
  gather_sorted_kernel<V><<<grid, kGatherThreads, 0, st>>>(tb, num_rows, B.sk, B.sv, n, T, B.row_mask, ob, err)
  switch (vpr) {
    case 4: FS_GATHER_SORTED(4); break;
    case 8: FS_GATHER_SORTED(8); break;
    case 16: FS_GATHER_SORTED(16); break;
    case 32: FS_GATHER_SORTED(32); break;
    default: return FS_ERR_INVALID_ARG;
  }
#undef FS_GATHER_SORTED
  count_launch(1);
  return launch_status();
}

extern "C" fs_status fs_emb_update_sorted(void* table, float* state, int64_t num_rows, int32_t dim, fs_dtype dtype,
                                          fs_optim optim, const void* grads, int64_t T, fs_phase phase, float lr,
                                          float eps, int32_t* err, void* ws, size_t ws_bytes, fs_stream_t stream) {
  FS_NVTX_RANGE();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  fs_status s = check_sorted(T, num_rows, dim, dtype, phase, err, ws, ws_bytes);
  if (s != FS_OK) return s;
  if (optim != FS_SGD && optim != FS_ROWWISE_ADAGRAD) return FS_ERR_INVALID_ARG;
  if (optim == FS_ROWWISE_ADAGRAD && !state) return FS_ERR_INVALID_ARG;
  if (T == 0) return FS_OK;
  if ((s = check_update_args(table, state, dim, dtype, optim, grads)) != FS_OK) return s;
  BwdWs B;
  if (!carve_bwd(T, num_rows, dim, phase, ws, ws_bytes, B)) return FS_ERR_WORKSPACE;
  int launches = 0;
  update_rows(B, table, state, dim, dtype, optim, grads, phase, lr, eps, err, st, &launches);
  count_launch(launches);
  return launch_status();
}
