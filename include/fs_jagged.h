/*
 * fs_jagged.h -- C ABI of the GB300 (sm_103a) jagged index + embedding library.
 *
 * The library runs the data-parallel hot path of one FreeScale training
 * iteration ("FreeScale: Distributed Training for Sequence Recommendation
 * Models with Minimal Scaling Cost", arXiv 2604.24073) over n logical ranks
 * held in one GPU's memory:
 *
 *   balance (FBS, or VBS with optional AutoTune, §4.1)  ->  jagged sample
 *   permutation (Algorithm 1, Stage III; §4.2 indexed permute)  ->  row-wise
 *   bucketize into shard-major form (§3.2, Algorithm 2 line 8; §4.2 ranged
 *   dispatch)  ->  collision /
 *   exclusive split between iterations t and t+1 (Algorithm 2 line 10)  ->
 *   embedding gather into batch-major jagged output (Algorithm 2 lines 12
 *   and 15; ranged combine)  ->  gradient segment-reduce + row update
 *   (Algorithm 2 lines 7, 18 and 20).
 *
 * Conventions shared by every call:
 *  - Pointers are DEVICE pointers owned by the caller unless stated otherwise.
 *    Nothing is allocated, freed or synchronised inside a call; every call is
 *    asynchronous on `stream` (NULL = the legacy default stream).
 *  - Argument errors (bad sizes, NULL pointers, misalignment, workspace too
 *    small) are found on the host and returned at once; nothing is launched.
 *  - Data errors (an ID outside [0, num_rows), malformed offsets or
 *    permutation, an output capacity that is too small, a bounded wait that
 *    gave up) are written by the kernels into the caller's device word
 *    `*err` (int32, first error wins; the caller zeroes it).  fs_check() reads
 *    it.  After a data error the outputs of that call are unspecified, but
 *    every write stays inside the buffers described here.
 *  - Scratch memory comes from the caller: `ws` / `ws_bytes`, at least the
 *    size the matching *_workspace_size() query returns, 256-byte aligned.
 *  - Sizes of data-dependent outputs (list lengths, selected counts) stay on
 *    the device; the host never needs them to launch the next call.
 *  - Positions are int32: T (IDs per batch) must be < 2^31.
 */
#ifndef FS_JAGGED_H
#define FS_JAGGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fs_stream_t; /* same handle as cudaStream_t */

typedef enum {
  FS_OK = 0,
  FS_ERR_INVALID_ARG = 1, /* host: bad size, NULL pointer, unsupported dim/dtype; device: bad length */
  FS_ERR_ID_RANGE = 2,    /* device: an ID < 0 or >= num_rows */
  FS_ERR_BAD_OFFSETS = 3, /* device: offsets not monotone / permutation entry out of range */
  FS_ERR_CAPACITY = 4,    /* device: an output would exceed the capacity passed in */
  FS_ERR_WORKSPACE = 5,   /* host: ws_bytes smaller than the workspace query */
  FS_ERR_TIMEOUT = 6,     /* device: a bounded inter-block wait gave up (no hang) */
  FS_ERR_CUDA = 7,        /* host: a CUDA runtime call or launch failed */
  FS_ERR_ALIGNMENT = 8    /* host: a pointer is not aligned as documented */
} fs_status;

typedef enum { FS_F32 = 0, FS_BF16 = 1 } fs_dtype;
typedef enum { FS_SGD = 0, FS_ROWWISE_ADAGRAD = 1 } fs_optim;
typedef enum {
  FS_PHASE_ALL = 0,
  FS_PHASE_COLLISION = 1,
  FS_PHASE_EXCLUSIVE = 2,
  FS_PHASE_COLLISION_THEN_EXCLUSIVE = 3
} fs_phase;

/* ------------------------------------------------------------------------
 * FBS partition -- FreeScale §4.1 (Partitioning Algorithms), FBS paragraph.
 * Sorts the S samples by UIH length (ascending, ties by global index g, so the
 * partition is deterministic as Algorithm 1 requires) and deals the sorted
 * positions to the n ranks in snake order: sorted position p is in round
 * rho = p / n at place k = p % n and goes to rank k (rho even) or n-1-k (rho
 * odd); a rank lists its samples by round.  (The printed index list
 * [i, 2n-i, 2n+i, 4n-i, ...] is this rule with an off-by-one.)  Every rank
 * gets floor(S/n) or ceil(S/n) samples (exactly S/n when n divides S).
 *   uih_len      [S]   int32, >= 0 (negative -> FS_ERR_INVALID_ARG in *err)
 *   perm         [S]   int32 out: perm[new position] = g
 *   rank_offsets [n+1] int64 out: rank r owns new positions [ro[r], ro[r+1])
 * S in [0, 2^31), n >= 1.  Up to 16384 samples are sorted and dealt by one
 * block in shared memory (the workspace is not touched then); larger batches
 * use device-wide radix passes in the workspace.
 * ---------------------------------------------------------------------- */
size_t fs_balance_fbs_workspace_size(int64_t S, int32_t n);
fs_status fs_balance_fbs(const int32_t* uih_len, int64_t S, int32_t n, int32_t* perm, int64_t* rank_offsets,
                         int32_t* err, void* ws, size_t ws_bytes, fs_stream_t stream);

/* ------------------------------------------------------------------------
 * FBS partition without caller workspace (no counterpart on the pages: the
 * method itself says nothing about memory ownership).
 * For callers that cannot allocate device memory when they partition a batch
 * -- code running while a memory pool is frozen or torn down, a plugin inside
 * another framework's process whose allocator it does not own, a step with a
 * fixed memory plan.  Same result as fs_balance_fbs; the sort's scratch is a
 * fixed array inside the library (about 4.3 MB of device memory, held on every
 * device that loads the library until the process exits), so this call
 * allocates nothing.
 *   S must be <= 262144 (FS_ERR_INVALID_ARG otherwise).
 *   The first call on a device looks the array's device address up
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   Every call shares the one array: calls that overlap on the GPU (two
 *   streams, two host threads) race and must be serialised by the caller.
 *   The call clears the counters it needs itself; leftovers of earlier calls
 *   do not matter.
 * ---------------------------------------------------------------------- */
fs_status fs_balance_fbs_noalloc(const int32_t* uih_len, int64_t S, int32_t n, int32_t* perm, int64_t* rank_offsets,
                                 int32_t* err, fs_stream_t stream);

/* ------------------------------------------------------------------------
 * VBS partition -- FreeScale §4.1, VBS paragraph.  Sample weight L^alpha,
 * kept in fixed point w = round_half_even(256 * L^alpha) (uint64; L^alpha is
 * L*sqrt(L) for alpha = 1.5 and the matching exact products for alpha in
 * {0.5, 1, 2, 2.5, 3}, pow() otherwise).  The order is the (L, g)-sorted order
 * when sort_by_len != 0 ("partitions globally sorted samples"), else the
 * original rank-major order.  With P_j the exclusive prefix of the weights
 * along that order and W their total, sample j goes to rank
 * min(n-1, floor(n * P_j / W)); segments are contiguous and may be empty, and
 * the heaviest weighs at most W/n + max w.  If W = 0 the rank is
 * min(n-1, floor(n * j / S)).
 *   perm       [S]   int32 out: the order; rank r owns [ro[r], ro[r+1])
 *   seg_weight [n]   uint64 out: sum of w over rank r
 * S * max(w) must stay below 2^62 (else FS_ERR_INVALID_ARG in *err).
 * ---------------------------------------------------------------------- */
size_t fs_balance_vbs_workspace_size(int64_t S, int32_t n);
fs_status fs_balance_vbs(const int32_t* uih_len, int64_t S, int32_t n, double alpha, int32_t sort_by_len,
                         int32_t* perm, int64_t* rank_offsets, uint64_t* seg_weight, int32_t* err, void* ws,
                         size_t ws_bytes, fs_stream_t stream);

/* ------------------------------------------------------------------------
 * VBS AutoTune -- FreeScale §4.1, VBS paragraph, and the AutoTune module of
 * Figure 4: since L^alpha need not match the model's execution time, each
 * rank's local batch size is raised or lowered by how its local execution
 * time compares with the global average.
 *
 * fs_vbs_autotune: one update of the per-rank batch corrections.
 *   times       [n] int64 in: the ranks' local execution times of the last
 *                   iteration, integer units (e.g. ns), 0 <= t < 2^53
 *   batch_delta [n] int64 in/out: the corrections (samples), 0 at the start
 *   step        samples one adjustment moves, 0 <= step <= 2^31 - 1
 *   tol_ppm     dead band in parts per million of the average, [0, 10^6]
 * Rank r is slow when n * 10^6 * t_r > (10^6 + tol_ppm) * sum(t) and fast when
 * n * 10^6 * t_r < (10^6 - tol_ppm) * sum(t) (exact integers).  The global
 * batch is fixed, so with k = min(#slow, #fast) the k slowest ranks (time
 * descending, lower rank first on ties) lose `step` and the k fastest (time
 * ascending, lower rank first) gain `step`: sum(batch_delta) is unchanged.
 * 1 <= n <= 65536 (O(n^2) comparisons spread over the GPU).  A time outside
 * [0, 2^53) sets FS_ERR_INVALID_ARG in *err and leaves batch_delta as it was.
 *
 * fs_balance_vbs_tuned: fs_balance_vbs with a correction applied.  The cut's
 * segment ends e_r = rank_offsets[r+1] move by D_r = batch_delta[0] + ... +
 * batch_delta[r], are clamped to [0, S] and then made non-decreasing (each
 * end becomes the largest end up to it); perm is the cut's, seg_weight that of
 * the moved segments.  Where no clamp acts, rank r holds its cut count plus
 * batch_delta[r] samples.  batch_delta [n] (device) must sum to 0 with
 * |batch_delta[r]| <= S, else FS_ERR_INVALID_ARG in *err and the cut is left
 * unmoved.  Workspace: fs_balance_vbs_workspace_size(S, n).
 * ---------------------------------------------------------------------- */
fs_status fs_vbs_autotune(const int64_t* times, int32_t n, int64_t step, int32_t tol_ppm, int64_t* batch_delta,
                          int32_t* err, fs_stream_t stream);
fs_status fs_balance_vbs_tuned(const int32_t* uih_len, int64_t S, int32_t n, double alpha, int32_t sort_by_len,
                               const int64_t* batch_delta, int32_t* perm, int64_t* rank_offsets,
                               uint64_t* seg_weight, int32_t* err, void* ws, size_t ws_bytes, fs_stream_t stream);

/* ------------------------------------------------------------------------
 * Jagged sample permutation ("indexed permute") -- FreeScale Algorithm 1
 * Stage III (shuffle samples to match the partition) and §4.2.  Output sample
 * k is input sample perm[k] with all its IDs ([UIH | candidates]):
 *   out_offsets[k+1] - out_offsets[k] = offsets[perm[k]+1] - offsets[perm[k]]
 *   out_values[out_offsets[k] + i]    = values[offsets[perm[k]] + i]
 *   offsets     [S+1] int64, offsets[0] = 0, non-decreasing
 *   values      [offsets[S]] int64
 *   perm        [S]   int32 in [0, S)
 *   out_offsets [S+1] int64 out
 *   out_values  [capacity] int64 out; offsets[S] > capacity -> FS_ERR_CAPACITY
 * Optional (rank_offsets != NULL): rank_id_offsets[r] = out_offsets[rank_offsets[r]]
 * for r = 0..n, the ID range of each destination rank (input of the bucketize).
 * ---------------------------------------------------------------------- */
size_t fs_permute_jagged_workspace_size(int64_t S);
fs_status fs_permute_jagged(const int64_t* offsets, const int64_t* values, int64_t S, const int32_t* perm,
                            int64_t* out_offsets, int64_t* out_values, int64_t capacity,
                            const int64_t* rank_offsets, int32_t n, int64_t* rank_id_offsets, int32_t* err,
                            void* ws, size_t ws_bytes, fs_stream_t stream);

/* ------------------------------------------------------------------------
 * Keyed transpose -- FreeScale §4.2 (the jagged kernels convert jagged tensors
 * from the feature-major form to the batch-major form).  F features, B
 * samples; the input is feature-major (segment f*B + b holds feature f's IDs
 * of sample b), the output batch-major (segment b*F + f):
 *   out segment b*F + f = in segment f*B + b, element by element,
 *   plus row_base[f] on every ID when row_base != NULL (features with their
 *   own tables stacked in one: the IDs become rows of the stacked table).
 *   offsets     [F*B+1] int64, offsets[0] = 0, non-decreasing
 *   values      [offsets[F*B]] int64
 *   row_base    [F] int64 or NULL
 *   out_offsets [F*B+1] int64 out
 *   out_values  [capacity] int64 out; offsets[F*B] > capacity -> FS_ERR_CAPACITY
 * Bad offsets -> FS_ERR_BAD_OFFSETS (error word).  F >= 1, F*B < 2^31.
 * ---------------------------------------------------------------------- */
size_t fs_keyed_transpose_workspace_size(int64_t F, int64_t B);
fs_status fs_keyed_transpose(const int64_t* offsets, const int64_t* values, int64_t F, int64_t B,
                             const int64_t* row_base, int64_t* out_offsets, int64_t* out_values, int64_t capacity,
                             int32_t* err, void* ws, size_t ws_bytes, fs_stream_t stream);

/* ------------------------------------------------------------------------
 * Row-wise bucketize ("ranged dispatch") -- FreeScale §3.2 (batch-major and
 * shard-major forms), Algorithm 2 line 8, §4.2.  The table of num_rows rows is
 * row-wise sharded into n ranges of block = ceil(num_rows / n) rows; ID x
 * belongs to shard x / block.  Shard-major order is the stable sort of the
 * batch-major positions by shard (inside a shard: source rank, then position).
 *   ids             [T]   int64 batch-major, in [0, num_rows)
 *   rank_id_offsets [n+1] int64: source rank r owns positions [rio[r], rio[r+1]),
 *                         rio[0] = 0, rio[n] = T
 *   sm_ids          [T]   int64 out: shard-major IDs
 *   pos             [T]   int32 out: batch-major position of shard-major entry j
 *   splits          [n*n] int64 out: splits[r*n + s] = IDs of source rank r in shard s
 *                         (the AllToAll send splits)
 *   shard_offsets   [n+1] int64 out
 * n in [1, 1024].  An ID outside [0, num_rows) sets FS_ERR_ID_RANGE; its
 * entry still takes a place (shard 0 below the range, shard n-1 above it), but
 * its shard-major copy may be the clamped value (0, or num_rows) rather than
 * the ID itself.
 * ---------------------------------------------------------------------- */
size_t fs_bucketize_rowwise_workspace_size(int64_t T, int32_t n);
fs_status fs_bucketize_rowwise(const int64_t* ids, int64_t T, const int64_t* rank_id_offsets, int32_t n,
                               int64_t num_rows, int64_t* sm_ids, int32_t* pos, int64_t* splits,
                               int64_t* shard_offsets, int32_t* err, void* ws, size_t ws_bytes,
                               fs_stream_t stream);

/* ------------------------------------------------------------------------
 * Fused jagged permute + row-wise bucketize -- FreeScale Algorithm 1 Stage III
 * and §4.2 (the indexed permute and the ranged dispatch that prepare the IDs
 * AllToAll), Algorithm 2 line 8.  One call with the results of
 *   fs_permute_jagged(offsets, values, S, perm, out_offsets, out_values,
 *                     capacity, rank_offsets, n, rank_id_offsets, ...)
 * followed by
 *   fs_bucketize_rowwise(out_values, T, rank_id_offsets, n, num_rows, sm_ids,
 *                        pos, splits, shard_offsets, ...),   T = out_offsets[S],
 * bit for bit, but the source IDs are read once: each 4096-ID output tile is
 * counted per shard as it is written, so the bucketize needs no counting pass
 * of its own; T stays on the device.
 *   rank_offsets [n+1] required (n in [1, 1024]: ranks = shards)
 *   out_values, sm_ids [capacity] int64, pos [capacity] int32; offsets[S] >
 *   capacity -> FS_ERR_CAPACITY (the first `capacity` IDs are still written
 *   and bucketized)
 * Errors as the two calls (FS_ERR_BAD_OFFSETS, FS_ERR_ID_RANGE,
 * FS_ERR_CAPACITY in *err).
 * ---------------------------------------------------------------------- */
size_t fs_permute_bucketize_workspace_size(int64_t S, int64_t capacity, int32_t n);
fs_status fs_permute_bucketize(const int64_t* offsets, const int64_t* values, int64_t S, const int32_t* perm,
                               const int64_t* rank_offsets, int32_t n, int64_t num_rows, int64_t* out_offsets,
                               int64_t* out_values, int64_t capacity, int64_t* rank_id_offsets, int64_t* sm_ids,
                               int32_t* pos, int64_t* splits, int64_t* shard_offsets, int32_t* err, void* ws,
                               size_t ws_bytes, fs_stream_t stream);

/* ------------------------------------------------------------------------
 * Collision / exclusive split -- FreeScale Algorithm 2 line 10
 * (compute_collision) and the notation paragraph after Algorithm 2: a
 * collision row is used by both iteration t and t+1, an exclusive row by one
 * of them.  Sets are of rows, so the result does not depend on whether the
 * inputs are given batch-major or shard-major.
 *   co      = uniq(ids_t) & uniq(ids_next)    ascending int64
 *   ex_t    = uniq(ids_t) - uniq(ids_next)    ascending int64
 *   ex_next = uniq(ids_next) - uniq(ids_t)    ascending int64
 *   counts  [3] int64 out: |co|, |ex_t|, |ex_next|; a list longer than cap_rows
 *           sets FS_ERR_CAPACITY and is truncated
 *   *_shard_off [n+1] int64 out: list entries below k * ceil(num_rows/n)
 *   is_co_t [T_t], is_co_next [T_next] uint8 out, aligned with the inputs:
 *           1 when that entry's row is a collision row, else 0.  Either may be
 *           NULL when the caller does not need it (the synchronous order
 *           needs only is_co_t); its pass over the IDs is then skipped.
 * num_rows < 2^32.
 * ---------------------------------------------------------------------- */
size_t fs_collision_split_workspace_size(int64_t T_t, int64_t T_next, int64_t num_rows, int32_t n);
fs_status fs_collision_split(const int64_t* ids_t, int64_t T_t, const int64_t* ids_next, int64_t T_next,
                             int64_t num_rows, int32_t n, int64_t* co, int64_t* ex_t, int64_t* ex_next,
                             int64_t cap_rows, int64_t* counts, int64_t* co_shard_off, int64_t* ex_t_shard_off,
                             int64_t* ex_next_shard_off, uint8_t* is_co_t, uint8_t* is_co_next, int32_t* err,
                             void* ws, size_t ws_bytes, fs_stream_t stream);

/* ------------------------------------------------------------------------
 * The same split in two steps, so that a batch's row set is built once and
 * used by both pairs it belongs to ((t-1, t) and (t, t+1)).
 * fs_row_bitmap: presence bitmap of the rows of one batch,
 *   fs_row_bitmap_words(num_rows) uint32 words, bit (r % 32) of word r / 32;
 *   cleared and filled by the call (an ID outside [0, num_rows) sets
 *   FS_ERR_ID_RANGE).
 * fs_collision_split_bitmaps: the outputs of fs_collision_split from the two
 *   bitmaps; ids_t / ids_next are only read for the masks that are asked for.
 * ---------------------------------------------------------------------- */
size_t fs_row_bitmap_words(int64_t num_rows);
fs_status fs_row_bitmap(const int64_t* ids, int64_t T, int64_t num_rows, uint32_t* bitmap, int32_t* err,
                        fs_stream_t stream);
size_t fs_collision_split_bitmaps_workspace_size(int64_t num_rows);
fs_status fs_collision_split_bitmaps(const int64_t* ids_t, int64_t T_t, const uint32_t* bm_t, const int64_t* ids_next,
                                     int64_t T_next, const uint32_t* bm_next, int64_t num_rows, int32_t n,
                                     int64_t* co, int64_t* ex_t, int64_t* ex_next, int64_t cap_rows, int64_t* counts,
                                     int64_t* co_shard_off, int64_t* ex_t_shard_off, int64_t* ex_next_shard_off,
                                     uint8_t* is_co_t, uint8_t* is_co_next, int32_t* err, void* ws, size_t ws_bytes,
                                     fs_stream_t stream);

/* ------------------------------------------------------------------------
 * Embedding gather -- FreeScale Algorithm 2 line 12 (Lookup, then back to
 * batch-major: the ranged combine is fused, rows land directly at their
 * batch-major position) and line 15 (merge of the prefetched exclusive rows
 * and the collision rows into one batch); §2.1 (an ID list becomes a
 * sequence of embeddings, no pooling).
 *   out[p, :] = table[ids[p], :]  (a byte copy of one row)
 * With mask != NULL only positions p with mask[p] == sel are written; the
 * other rows of out are left untouched.
 *   table [num_rows, dim] of dtype, row-major;  out [T, dim] of dtype.
 * Row bytes must be a multiple of 4.  Unmasked calls with 16-byte aligned
 * table and out and rows of 16 B to 2 KB (a multiple of 16) move rows through
 * the copy engine (bulk copies into shared memory, one bulk store per stage);
 * other multiples of 16 take 16-byte vector loads, the rest 4-byte words.
 * ---------------------------------------------------------------------- */
fs_status fs_emb_gather(const void* table, int64_t num_rows, int32_t dim, fs_dtype dtype, const int64_t* ids,
                        int64_t T, const uint8_t* mask, uint8_t sel, void* out, int32_t* err,
                        fs_stream_t stream);

/* ------------------------------------------------------------------------
 * Embedding gather in shard-major order -- FreeScale Algorithm 2 line 12 as
 * the shards make it: each shard looks up the rows of its shard-major IDs,
 * and the ranged combine puts every row back at its batch-major position:
 *   out[pos[j], :] = table[sm_ids[j], :]   for j in [0, T)
 * With (sm_ids, pos) from fs_bucketize_rowwise (or fs_permute_bucketize) of
 * ids, pos is a permutation of [0, T) and the result is fs_emb_gather's
 * unmasked result, bit for bit.  A shard's entries come together, so a
 * shard's repeated rows are read from L2 rather than again from DRAM while it
 * is gathered (shards of up to tens of MB of rows).
 *   sm_ids [T] int64, pos [T] int32 (in [0, T); FS_ERR_BAD_OFFSETS and the
 *   entry skipped otherwise; an ID outside [0, num_rows) FS_ERR_ID_RANGE)
 *   table [num_rows, dim] of dtype, out [T, dim] of dtype.
 * Row bytes must be a multiple of 4; rows of 64, 128, 256 or 512 bytes with
 * 16-byte aligned table and out move as 16-byte vectors.
 * ---------------------------------------------------------------------- */
fs_status fs_emb_gather_shard_major(const void* table, int64_t num_rows, int32_t dim, fs_dtype dtype,
                                    const int64_t* sm_ids, const int32_t* pos, int64_t T, void* out, int32_t* err,
                                    fs_stream_t stream);

/* ------------------------------------------------------------------------
 * Embedding backward: gradient segment-reduce per row + row update --
 * FreeScale Algorithm 2 lines 7 and 20 (update_embedding on the exclusive and
 * the collision rows) and line 18 (split of the gradients).  The pages name
 * no optimizer; this implements
 *   g_r = sum of grads[p] over positions p with ids[p] = r selected by phase
 *         (fp32 accumulation in a fixed order: the result is identical run to run)
 *   FS_SGD:             W_r -= lr * g_r
 *   FS_ROWWISE_ADAGRAD: s_r += mean_d(g_{r,d}^2);  W_r -= lr * g_r / (sqrt(s_r) + eps)
 * bf16 tables read bf16 grads, accumulate in fp32 and store round-to-nearest-
 * even.  phase selects positions: ALL every position, COLLISION those of
 * collision rows, EXCLUSIVE those of the other rows.  The collision flag is
 * given either per position (is_co[p] in {0, 1}) or per row (co_rows: bit
 * r & 31 of word r >> 5 set iff row r is a collision row; for Algorithm 2 this
 * is the presence bitmap of batch t+1's rows, which fs_row_bitmap writes) --
 * exactly one of the two unless phase is ALL.  The bitmap form reads one
 * bitmap word per position in each pass of the sort, so when the mask exists
 * it is the faster input.
 * Collision is a property of the row, so COLLISION then EXCLUSIVE updates
 * every row of the batch once, collision rows first.  COLLISION_THEN_EXCLUSIVE
 * does exactly that in one call: one sort of all positions (the phase is the
 * key's top bit), then the collision rows' updates, then the exclusive rows'
 * updates, in stream order.
 *   table [num_rows, dim] in place;  state [num_rows] fp32 in place (NULL for SGD)
 *   ids [T] int64;  grads [T, dim] of dtype (batch-major)
 *   is_co [T] uint8 or NULL;  co_rows [fs_row_bitmap_words(num_rows)] or NULL
 * Supported: dim in {32, 64, 128} (fp32) or {32, 64, 128, 256} (bf16);
 * num_rows < 2^32.
 * ---------------------------------------------------------------------- */
size_t fs_emb_backward_adagrad_workspace_size(int64_t T, int64_t num_rows, int32_t dim, fs_dtype dtype);
fs_status fs_emb_backward_adagrad(void* table, float* state, int64_t num_rows, int32_t dim, fs_dtype dtype,
                                  fs_optim optim, const int64_t* ids, const void* grads, int64_t T,
                                  const uint8_t* is_co, const uint32_t* co_rows, fs_phase phase, float lr,
                                  float eps, int32_t* err, void* ws, size_t ws_bytes, fs_stream_t stream);

/* ------------------------------------------------------------------------
 * Row-sorted path: the update's sort, run before the lookup of the same batch,
 * also serves the lookup (Algorithm 2 line 12 and lines 18-20 on one batch).
 * fs_emb_backward_adagrad split in two around a gather that reads each
 * distinct table row once:
 *
 *   fs_emb_sort_rows      sorts the batch's entries by (phase bit, row);
 *   fs_emb_gather_sorted  out[p] = table[ids[p]] for every sorted entry p --
 *                         the same result as fs_emb_gather, bit for bit, but
 *                         equal rows are adjacent, so a row is read from DRAM
 *                         once and written to each of its positions;
 *   fs_emb_update_sorted  the segment-reduce + row update of those entries --
 *                         the same result as fs_emb_backward_adagrad with the
 *                         same arguments, bit for bit.
 *
 * The sorted entries stay in `ws` between the calls: pass the same ws (of
 * fs_emb_backward_adagrad_workspace_size(T, num_rows, dim, dtype) bytes) and
 * the same T, num_rows, dim, dtype and phase to the three calls, in stream
 * order, and use ws for nothing else in between (the gather and the update
 * read the sort's output and may run any number of times).
 *   phase: FS_PHASE_ALL, or FS_PHASE_COLLISION_THEN_EXCLUSIVE with is_co or
 *          co_rows as in fs_emb_backward_adagrad (num_rows <= 2^30 there, so
 *          that the phase bit fits beside the row bits); other phases keep
 *          only some entries and are refused (FS_ERR_INVALID_ARG).
 *   gather: table and out 16-byte aligned (FS_ERR_ALIGNMENT); row bytes
 *          64 to 512 as the update allows.  Positions whose ID is out of range
 *          (FS_ERR_ID_RANGE from the sort) or whose is_co byte is above 1 are
 *          not sorted, and their output rows are left untouched.  A sorted
 *          entry out of range (ws not holding this batch's sort) sets
 *          FS_ERR_BAD_OFFSETS and is skipped.
 *   update: reads the sorted entries without checks: calling it on a ws that
 *          fs_emb_sort_rows did not fill for the same batch is undefined.
 * ---------------------------------------------------------------------- */
fs_status fs_emb_sort_rows(int64_t num_rows, int32_t dim, fs_dtype dtype, const int64_t* ids, int64_t T,
                           const uint8_t* is_co, const uint32_t* co_rows, fs_phase phase, int32_t* err, void* ws,
                           size_t ws_bytes, fs_stream_t stream);
fs_status fs_emb_gather_sorted(const void* table, int64_t num_rows, int32_t dim, fs_dtype dtype, int64_t T,
                               fs_phase phase, void* out, int32_t* err, void* ws, size_t ws_bytes,
                               fs_stream_t stream);
fs_status fs_emb_update_sorted(void* table, float* state, int64_t num_rows, int32_t dim, fs_dtype dtype,
                               fs_optim optim, const void* grads, int64_t T, fs_phase phase, float lr, float eps,
                               int32_t* err, void* ws, size_t ws_bytes, fs_stream_t stream);

/* ------------------------------------------------------------------------
 * The update's sort, per shard -- FreeScale §3.2 and Algorithm 2 line 8: after
 * the IDs AllToAll each shard's rows arrive shard-major, so the shard that
 * updates them (lines 18-20) groups its own entries by row.  Same sorted
 * entries as fs_emb_sort_rows, bit for bit (ordered by phase bit, row,
 * position), written to the same place in ws, so fs_emb_gather_sorted and
 * fs_emb_update_sorted follow it unchanged; but the input is the bucketize
 * output, whose entries are already grouped by shard, so the sort only orders
 * each shard's entries by the row's offset inside the shard (two counting
 * passes where the row index would need three for 100M rows).
 *   sm_ids, pos, shard_offsets: the outputs of fs_bucketize_rowwise for the
 *          batch (n shards of block = ceil(num_rows / n) rows; n <= 1024)
 *   is_co  [T] uint8 per SHARD-MAJOR entry (e.g. the mask fs_collision_split
 *          writes when given sm_ids as its IDs): 1 for a collision row, 0 for
 *          an exclusive one; or
 *   co_rows the collision rows as a row bitmap (bit r & 31 of word r >> 5; for
 *          Algorithm 2 the presence bitmap of batch t+1, which fs_row_bitmap
 *          writes): the sort looks each entry's row up, so no mask pass is
 *          needed; entries come shard-major, so a tile's lookups stay in its
 *          shard's stretch of the bitmap.
 *          Exactly one of the two for FS_PHASE_COLLISION_THEN_EXCLUSIVE;
 *          both ignored for FS_PHASE_ALL.
 *   phase  FS_PHASE_ALL or FS_PHASE_COLLISION_THEN_EXCLUSIVE
 *   ws     fs_emb_sort_rows_sharded_workspace_size(T, num_rows, dim, dtype, n)
 *          bytes; its first fs_emb_backward_adagrad_workspace_size(...) bytes
 *          hold what the gather and the update read.
 * ceil(num_rows / n) must stay below 2^20 (2^19 with two phases) so that the
 * offset inside a shard (and the phase bit) fit two passes of at most 10 bits
 * (FS_ERR_INVALID_ARG otherwise; fs_emb_sort_rows has no such limit).  An ID
 * outside [0, num_rows) sets FS_ERR_ID_RANGE, an ID outside the shard that
 * shard_offsets gives it, or shard_offsets that are not non-decreasing from 0
 * to T, set FS_ERR_BAD_OFFSETS; such entries (and flags above 1) are not
 * sorted, as in fs_emb_sort_rows.
 * ---------------------------------------------------------------------- */
size_t fs_emb_sort_rows_sharded_workspace_size(int64_t T, int64_t num_rows, int32_t dim, fs_dtype dtype, int32_t n);
fs_status fs_emb_sort_rows_sharded(int64_t num_rows, int32_t dim, fs_dtype dtype, const int64_t* sm_ids,
                                   const int32_t* pos, int64_t T, const int64_t* shard_offsets, int32_t n,
                                   const uint8_t* is_co, const uint32_t* co_rows, fs_phase phase, int32_t* err,
                                   void* ws, size_t ws_bytes, fs_stream_t stream);

/* ------------------------------------------------------------------------
 * Utilities.
 * fs_check: waits for `stream`, then returns the code in *err (FS_OK if 0),
 *   or FS_ERR_CUDA if the stream reports an error.  Host-synchronous: meant for
 *   tests and benchmarks, not for the hot loop.
 * fs_set_spin_limit: polls before a bounded inter-block wait gives up with
 *   FS_ERR_TIMEOUT (default 1<<22, roughly a second); a wait for a bulk copy
 *   of gradient rows gives up after polls * 256 ns.  Applies to later calls.
 *   The Python binding applies the environment variable FS_SPIN_LIMIT (a
 *   positive integer) when it loads the library.
 * fs_get_spin_limit: the limit in force.
 * fs_launch_count: kernels this library has launched in this process.
 * fs_debug_skip_publish: test hook for the bounded waits.  Tile `tile` of the
 *   single-pass scans (VBS weights, permute offsets, collision compaction)
 *   skips publishing its look-back status, so every later tile's wait runs out
 *   and the call reports FS_ERR_TIMEOUT instead of hanging; in the embedding
 *   update, the first bulk copy of gradient rows for sorted tile `tile` is
 *   never issued, so the wait for it runs out the same way.  -1 (the default)
 *   turns it off.  Never used outside tests.
 * ---------------------------------------------------------------------- */
fs_status fs_check(const int32_t* err, fs_stream_t stream);
const char* fs_status_string(fs_status s);
void fs_set_spin_limit(int64_t polls);
int64_t fs_get_spin_limit(void);
void fs_debug_skip_publish(int64_t tile);
int64_t fs_launch_count(void);
const char* fs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FS_JAGGED_H */
