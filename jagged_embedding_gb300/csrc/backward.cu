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

#include <algorithm>

#include "radix.cuh"

namespace fs {
namespace {

using radix::kThreads;
constexpr int kChunk = 2048;                 // sorted entries per reduce tile
constexpr uint32_t kNoKey = 0xFFFFFFFFu;     // rows are < num_rows < 2^32

// Sort source: the selected positions of the batch, key = row, value = position.
// With both phases in one call, key = row | (exclusive << kb): collision rows
// sort first, exclusive rows after them, each group in row order.
struct SrcRows {
  using Key = uint32_t;
  static constexpr bool kIndexValue = true;  // value = item index
  const int64_t* ids;
  const uint8_t* is_co;
  int phase;
  int64_t R;
  int kb;  // bits of the largest row index
  __device__ __forceinline__ bool load(int64_t i, Key& key, uint32_t& val, int32_t* err) const {
    // the ID and the mask byte are loaded independently (no load-to-load dependency)
    const int64_t id = __ldcs(ids + i);
    uint32_t hi = 0;
    if (phase != FS_PHASE_ALL) {
      const uint8_t m = __ldcs(is_co + i);
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
    ss = __shfl_sync(0xffffffffu, ss, 0);  // one value for the whole row
    const float s = s_old + ss / float(D);
    const float step = u.lr / (sqrtf(s) + u.eps);  // one division per row
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

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Sorted entries [*begin_dev, *end_dev) (begin 0 when begin_dev is null);
// row = key & row_mask.  One warp per tile of kChunk sorted entries; the
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
                                                             uint8_t* head_cont, uint8_t* tail_flag) {
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int D = 32 * EPL;
  constexpr int RB = D * ESZ;
  constexpr int G = GROWS;  // gradient rows in flight per warp
  const int64_t b0 = begin_dev ? *begin_dev : 0;
  keys += b0;
  vals += b0;
  const int64_t n = *end_dev - b0;
  const int64_t ntiles = (n + kChunk - 1) / kChunk;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < ntiles; t += nwarps) {
    const int64_t s0 = t * kChunk;
    const int64_t s1 = (s0 + kChunk < n) ? s0 + kChunk : n;
    const uint32_t prev_key = s0 > 0 ? keys[s0 - 1] : kNoKey;
    const uint32_t next_key = s1 < n ? keys[s1] : kNoKey;
    bool from_prev = (keys[s0] == prev_key);  // the tile's first row began in an earlier tile
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

// Rows that cross tile boundaries: carry of the starting tile, then the head
// carries of the following tiles in order.
template <bool BF16, int EPL>
__global__ void __launch_bounds__(kThreads) fixup_kernel(const uint32_t* __restrict__ keys, const int64_t* begin_dev,
                                                         const int64_t* end_dev, uint32_t row_mask, UpdateArgs u,
                                                         const float* carry_head, const float* carry_tail,
                                                         const uint8_t* head_cont, const uint8_t* tail_flag) {
  constexpr int D = 32 * EPL;
  const int64_t b0 = begin_dev ? *begin_dev : 0;
  keys += b0;
  const int64_t n = *end_dev - b0;
  const int64_t ntiles = (n + kChunk - 1) / kChunk;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < ntiles; t += nwarps) {
    if (!tail_flag[t]) continue;
    const uint32_t row = keys[(t + 1) * kChunk - 1] & row_mask;
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

template <bool BF16, int EPL>
void launch_reduce(const uint32_t* k, const uint32_t* v, const int64_t* begin_dev, const int64_t* end_dev,
                   uint32_t row_mask, const void* grads, UpdateArgs u, float* ch, float* ct, uint8_t* hc,
                   uint8_t* tf, cudaStream_t st) {
  // 8 gradient rows in flight per warp (fewer for wide rows) and 4 blocks per
  // SM fit the 64-register budget without spills; measured best among the
  // launch shapes and staging schemes tried (see the design notes)
  constexpr int G = (16 / EPL) > 8 ? 8 : (16 / EPL);
  const unsigned sms = unsigned(sm_count());
  reduce_kernel<BF16, EPL, G, 4><<<sms * 4, kThreads, 0, st>>>(k, v, begin_dev, end_dev, row_mask, grads, u, ch, ct,
                                                              hc, tf);
  fixup_kernel<BF16, EPL><<<sms * (2048 / kThreads), kThreads, 0, st>>>(k, begin_dev, end_dev, row_mask, u, ch, ct,
                                                                         hc, tf);
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

extern "C" size_t fs_emb_backward_adagrad_workspace_size(int64_t T, int64_t num_rows, int32_t dim, fs_dtype dtype) {
  (void)dtype;
  if (T < 0 || num_rows < 1 || dim < 1) return 0;
  BwdLayout L = bwd_layout(T, num_rows, dim);
  // the single-call two-phase mode sorts one more key bit (the phase)
  const size_t sort_bytes = std::max(L.plan.bytes(), radix::SortPlan(T, L.plan.key_bits + 1).bytes());
  return sort_bytes + 2 * L.carry_bytes + 2 * L.flag_bytes + align_up(sizeof(int64_t)) + 256;
}

extern "C" fs_status fs_emb_backward_adagrad(void* table, float* state, int64_t num_rows, int32_t dim, fs_dtype dtype,
                                             fs_optim optim, const int64_t* ids, const void* grads, int64_t T,
                                             const uint8_t* is_co, fs_phase phase, float lr, float eps, int32_t* err,
                                             void* ws, size_t ws_bytes, fs_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T < 0 || T > INT32_MAX || num_rows < 1 || num_rows >= (int64_t(1) << 32) || !err) return FS_ERR_INVALID_ARG;
  if ((dtype != FS_F32 && dtype != FS_BF16) || (optim != FS_SGD && optim != FS_ROWWISE_ADAGRAD)) return FS_ERR_INVALID_ARG;
  if (phase != FS_PHASE_ALL && phase != FS_PHASE_COLLISION && phase != FS_PHASE_EXCLUSIVE &&
      phase != FS_PHASE_COLLISION_THEN_EXCLUSIVE)
    return FS_ERR_INVALID_ARG;
  const int epl = epl_for(dim, dtype);
  if (epl == 0) return FS_ERR_INVALID_ARG;
  if (optim == FS_ROWWISE_ADAGRAD && !state) return FS_ERR_INVALID_ARG;
  if (T == 0) return FS_OK;
  if (!table || !ids || !grads || (phase != FS_PHASE_ALL && !is_co)) return FS_ERR_INVALID_ARG;
  const size_t vec = size_t(epl) * (dtype == FS_F32 ? 4 : 2);
  if (!aligned(table, vec) || !aligned(grads, vec) || !aligned(ids, 8) || (state && !aligned(state, 4)))
    return FS_ERR_ALIGNMENT;
  if (ws_bytes < fs_emb_backward_adagrad_workspace_size(T, num_rows, dim, dtype) || !ws) return FS_ERR_WORKSPACE;

  const int kb = radix::bits_for(uint64_t(num_rows - 1));
  if (phase == FS_PHASE_COLLISION_THEN_EXCLUSIVE && kb > 30) {
    // the phase bit does not fit beside the row bits: two calls, same result
    fs_status s = fs_emb_backward_adagrad(table, state, num_rows, dim, dtype, optim, ids, grads, T, is_co,
                                          FS_PHASE_COLLISION, lr, eps, err, ws, ws_bytes, stream);
    if (s != FS_OK) return s;
    return fs_emb_backward_adagrad(table, state, num_rows, dim, dtype, optim, ids, grads, T, is_co,
                                   FS_PHASE_EXCLUSIVE, lr, eps, err, ws, ws_bytes, stream);
  }
  BwdLayout L = bwd_layout(T, num_rows, dim);
  if (phase == FS_PHASE_COLLISION_THEN_EXCLUSIVE) L.plan = radix::SortPlan(T, kb + 1);
  WsCursor cur(ws, ws_bytes);
  radix::SortWs W;
  if (!radix::carve_sort_ws(L.plan, cur, W)) return FS_ERR_WORKSPACE;
  float* carry_head = cur.take<float>(size_t(L.max_tiles) * dim);
  float* carry_tail = cur.take<float>(size_t(L.max_tiles) * dim);
  uint8_t* head_cont = cur.take<uint8_t>(size_t(L.max_tiles));
  uint8_t* tail_flag = cur.take<uint8_t>(size_t(L.max_tiles));
  int64_t* n_first = cur.take<int64_t>(1);
  if (!cur.ok) return FS_ERR_WORKSPACE;

  int launches = 0;
  uint32_t *sk = nullptr, *sv = nullptr;
  SrcRows src{ids, is_co, int(phase), num_rows, kb};
  fs_status s = radix::run_sort(src, L.plan, W, err, st, &sk, &sv, &launches);
  if (s != FS_OK) return s;
  UpdateArgs u{table, optim == FS_ROWWISE_ADAGRAD ? state : nullptr, int(optim), lr, eps};
  const bool bf = dtype == FS_BF16;
  const int64_t* n_valid = W.pass.n_valid;
  // one update launch over a range of the sorted entries
  auto reduce_range = [&](const int64_t* begin_dev, const int64_t* end_dev, uint32_t row_mask) {
#define FS_REDUCE(BF, E) \
  launch_reduce<BF, E>(sk, sv, begin_dev, end_dev, row_mask, grads, u, carry_head, carry_tail, head_cont, tail_flag, st)
    switch (epl) {
      case 1: if (bf) FS_REDUCE(true, 1); else FS_REDUCE(false, 1); break;
      case 2: if (bf) FS_REDUCE(true, 2); else FS_REDUCE(false, 2); break;
      case 4: if (bf) FS_REDUCE(true, 4); else FS_REDUCE(false, 4); break;
      default: FS_REDUCE(true, 8); break;
    }
#undef FS_REDUCE
    launches += 2;
  };
  if (phase == FS_PHASE_COLLISION_THEN_EXCLUSIVE) {
    // collision rows sort first: update them in a first launch, the exclusive
    // rows (phase bit set) in a second, in stream order
    const uint32_t row_mask = (1u << kb) - 1u;
    count_below_kernel<<<1, 1, 0, st>>>(sk, n_valid, 1u << kb, n_first);
    ++launches;
    reduce_range(nullptr, n_first, row_mask);
    reduce_range(n_first, n_valid, row_mask);
  } else {
    reduce_range(nullptr, n_valid, 0xFFFFFFFFu);
  }
  count_launch(launches);
  return launch_status();
}
