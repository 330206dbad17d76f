/*
 * zoomr.h -- C ABI of the GB300 (sm_103a) ZoomR decode step over a paged KV cache.
 *
 * One call computes, for every sequence b and every KV head g of a GQA layer
 * (a "unit"), the four stages of ZoomR's decode-time retrieval:
 *
 *   1. score    ZoomR page, 3.3 "Per-Head Importance Scoring and Voting", the
 *               equation alpha_i = q_t^T kbar_i: every segment's summary key is
 *               scored against the query. Per KV head the score is the maximum
 *               over the group's query heads. The ranking key is the exact
 *               real value of that dot product on the stored bf16/fp32 inputs
 *               (no rounding enters the decision); the 1/sqrt(d) scale does not
 *               change the ranking and is not applied to it.
 *   2. select   ZoomR 3.3, the equation I_top-k = argtop-k(alpha): the k_b
 *               segments with the largest keys; ties go to the lower segment
 *               index; k_b >= n_b selects every segment, k_b = 0 none.
 *   3. gather   ZoomR 3.3, "Constructing the Final Multi-Granularity Context",
 *               the equation for I_f: the token set is the union of the recent
 *               window [max(0, L_b - w), L_b) and the token ranges of the selected
 *               segments (deduplicated); every segment that is not selected
 *               contributes its one summary key/value row. Token t of sequence b
 *               is read through the block table as on the "KV-cache management"
 *               page, "Paged KV cache (PagedAttention)": physical block
 *               block_tables[b][t / 16], slot t % 16.
 *   4. attend   ZoomR 2 "Background", A = softmax(q K^T / sqrt(d)) V over exactly
 *               that set, for every query head of the group (GQA as on the
 *               "KV-cache management" page, "Fewer key/value heads per token"):
 *               query head h reads KV head h / (Hq / Hkv).
 *
 * Conventions
 *   - Every function returns a zr_status; nothing is thrown, nothing exits.
 *   - ZR_EINVAL from zr_plan means nothing was allocated or launched.
 *   - zr_decode_attend is asynchronous on the caller's stream and allocates
 *     nothing. Indices that are found bad on the device (a physical block id
 *     outside [0, num_blocks)) set a sticky error word in the workspace; the
 *     offending row is skipped (no trap, no fault). A non-finite query or
 *     summary-key value (unsupported) is ranked as zero and sets bit 3 (value 4)
 *     of the same word. zr_get_device_error reads and clears it.
 *   - The plan is immutable after creation and may be reused for any number of
 *     layers and calls. Calls that may overlap on the GPU need separate
 *     workspaces.
 *   - The library never allocates the big tensors: q, the K/V pools, the block
 *     tables, the summaries, the output and the workspace belong to the caller.
 */
#ifndef ZOOMR_H
#define ZOOMR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ZR_API __attribute__((visibility("default")))
#else
#define ZR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ZR_OK = 0,
  ZR_EINVAL = 1,        /* bad argument: a null pointer, a shape or a metadata array out of its contract */
  ZR_ENOMEM = 2,        /* a host or device allocation of the plan failed */
  ZR_ECUDA = 3,         /* a CUDA runtime call failed (no device, bad stream, launch failure) */
  ZR_EUNSUPPORTED = 4,  /* valid but outside the library's supported limits (head_dim, group size, segment count) */
  ZR_EDEVICE = 5        /* the device reported a bad index (see zr_get_device_error) */
} zr_status;

typedef enum { ZR_F32 = 0, ZR_BF16 = 1 } zr_dtype;

typedef struct zr_plan* zr_plan_t; /* opaque */

typedef struct {
  int32_t batch;              /* B >= 1 sequences */
  int32_t num_q_heads;        /* Hq >= 1 */
  int32_t num_kv_heads;       /* Hkv >= 1, Hq % Hkv == 0, group G = Hq / Hkv <= 16 */
  int32_t head_dim;           /* d, 64 or 128 */
  int32_t block_size;         /* tokens per KV block: must be 16 */
  int32_t num_blocks;         /* physical blocks in each K (and V) pool */
  int32_t max_blocks_per_seq; /* columns of block_tables */
  int32_t window;             /* w >= 0 recent tokens always attended */
  int32_t dtype;              /* zr_dtype of q, the K/V pools and the summaries */
} zr_config;

/*
 * zr_plan -- validate the host metadata and build an immutable plan.
 *
 * Host metadata (copied; the caller keeps ownership):
 *   seq_lens   [B]      L_b >= 1 cached tokens, L_b <= 16 * max_blocks_per_seq.
 *   seg_ptr    [B+1]    CSR over segments: sequence b owns segments
 *                       seg_ptr[b] .. seg_ptr[b+1]-1; n_b = seg_ptr[b+1]-seg_ptr[b],
 *                       1 <= n_b <= 4096; seg_ptr[0] = 0.
 *   seg_bounds [seg_ptr[B] + B]  sequence b's n_b + 1 strictly ascending token
 *                       bounds start at index seg_ptr[b] + b; the first is 0 and
 *                       the last is L_b (segments partition the cached tokens).
 *   topk       [B]      k_b >= 0; values above n_b are clipped to n_b.
 * Outputs: *out_plan, and *workspace_bytes = the device workspace one call needs.
 * zr_plan copies a few small device arrays (the metadata) with cudaMalloc on
 * the current device; that device must be current for every later call.
 * Errors: ZR_EINVAL (nothing allocated), ZR_EUNSUPPORTED, ZR_ENOMEM, ZR_ECUDA.
 */
ZR_API zr_status zr_plan(const zr_config* cfg, const int32_t* seq_lens, const int32_t* seg_ptr,
                  const int32_t* seg_bounds, const int32_t* topk, zr_plan_t* out_plan,
                  size_t* workspace_bytes);

/*
 * zr_plan_sink -- zr_plan with the prompt kept as an attention sink (ZoomR page,
 * 3.3 "Constructing the Final Multi-Granularity Context": the prompt tokens I_p
 * are in every final set; 3.4 "Prefill Stage": their cache is kept in full).
 *   sink_lens  [B]  N_s >= 0 prompt tokens of sequence b, always attended; the
 *                   segments then partition [N_s, L_b): the first bound of each
 *                   sequence is N_s instead of 0 (N_s < L_b).
 * Every unit's token set gains [0, N_s). The plan reserves one more range slot
 * per unit: zr_plan_dims reports k_max one larger than zr_plan would (the
 * selection output keeps its -1 padding). Everything else is as zr_plan.
 */
ZR_API zr_status zr_plan_sink(const zr_config* cfg, const int32_t* seq_lens, const int32_t* sink_lens,
                              const int32_t* seg_ptr, const int32_t* seg_bounds, const int32_t* topk,
                              zr_plan_t* out_plan, size_t* workspace_bytes);

/*
 * zr_plan_dims -- sizes of the optional debug outputs of a plan.
 *   *k_max = max_b min(topk[b], n_b) (at least 1), *n_max = max_b n_b.
 */
ZR_API zr_status zr_plan_dims(zr_plan_t plan, int32_t* k_max, int32_t* n_max);

/*
 * zr_decode_attend -- one decode step of one layer, every unit.
 *
 * All pointers are DEVICE pointers owned by the caller; the call is async on
 * `stream` (a cudaStream_t; NULL is the legacy default stream).
 *   workspace     >= workspace_bytes, 256-byte aligned; zero it once before its
 *                 first use (it holds the sticky error word). Scratch between
 *                 calls: one workspace per stream of concurrent calls.
 *   q             [B, Hq, d]                       dtype
 *   k_pool/v_pool [num_blocks, Hkv, 16, d]         dtype
 *   block_tables  [B, max_blocks_per_seq]          int32 (entries past a sequence's last block are not read)
 *   sum_k/sum_v   [seg_ptr[B], Hkv, d]             dtype, segment rows in CSR order
 *   out           [B, Hq, d]                       float32 (written)
 * Optional debug outputs (may be NULL), all int32:
 *   sel_out       [B, Hkv, k_max]    selected segment indices, ascending, -1 padded
 *   ranges_out    [B, Hkv, k_max+1, 2]  gathered token ranges [start, end), maximal
 *                 runs in ascending order (unused entries are left unwritten)
 *   nranges_out   [B, Hkv]           number of ranges
 * Errors: ZR_EINVAL for a null plan or required pointer, a workspace that is not
 * 256-byte aligned, or q/pool/summary pointers that are not 16-byte aligned;
 * ZR_ECUDA if a launch fails.
 */
ZR_API zr_status zr_decode_attend(zr_plan_t plan, void* workspace, const void* q, const void* k_pool,
                           const void* v_pool, const int32_t* block_tables, const void* sum_k,
                           const void* sum_v, float* out, int32_t* sel_out, int32_t* ranges_out,
                           int32_t* nranges_out, void* stream);

/*
 * zr_decode_attend_timed -- zr_decode_attend without debug outputs that also
 * records caller-owned CUDA events (cudaEvent_t, created with timing enabled)
 * on `stream`: ev_start right before the gather-attention kernel and ev_stop
 * right after it, so the caller can time that kernel alone. Either may be NULL
 * (not recorded), not both: with only one, the caller's own event before the
 * call times the select kernel (ev_start) or the select and gather-attention
 * kernels with their launch overlap intact (ev_stop). The events are recorded
 * with the "external" flag, so inside a stream capture they become event-record
 * nodes of the graph.
 */
ZR_API zr_status zr_decode_attend_timed(zr_plan_t plan, void* workspace, const void* q, const void* k_pool,
                                 const void* v_pool, const int32_t* block_tables, const void* sum_k,
                                 const void* sum_v, float* out, void* ev_start, void* ev_stop,
                                 void* stream);

/*
 * zr_decode_attend_static -- zr_decode_attend for callers that cannot allocate
 * device memory. (The pages have no counterpart: this is a deployment variant.)
 *
 * Some callers are only handed their input and output buffers: a plugin inside
 * a host engine that owns every device allocation and offers no scratch, or a
 * loop that must never call cudaMalloc because it can synchronize the device.
 * This entry point takes the same tensors as zr_decode_attend but no workspace
 * and allocates nothing: its scratch is a 16 MiB static device array that every
 * GPU loading this library holds until the process exits.
 *   - The plan still comes from zr_plan (create it once, at start-up).
 *   - The first call on a device looks up that array's device address with the
 *     device current; make that first call before any stream capture.
 *   - A plan whose workspace_bytes exceeds 16 MiB is rejected with
 *     ZR_EUNSUPPORTED before anything is launched.
 *   - All calls share the one array: calls that may overlap on the GPU (other
 *     streams, other threads) race and corrupt each other's results; serialize
 *     them on one stream.
 *   - Out-of-pool block ids are masked as in zr_decode_attend, but not
 *     reported: the error word is cleared at the start of every call.
 *   - The plan's device must be the current device (ZR_EINVAL otherwise).
 *   - The device address of the array is kept for the life of the process:
 *     do not use this entry point across a cudaDeviceReset.
 * Errors (all returned before anything is enqueued on the stream): ZR_EINVAL
 * (null plan or required pointer, misaligned pointer, another device current),
 * ZR_EUNSUPPORTED (workspace over 16 MiB), ZR_ECUDA.
 */
ZR_API zr_status zr_decode_attend_static(zr_plan_t plan, const void* q, const void* k_pool, const void* v_pool,
                                         const int32_t* block_tables, const void* sum_k, const void* sum_v,
                                         float* out, void* stream);

/*
 * zr_get_device_error -- synchronize `stream`, then read and clear the sticky
 * device error word of `workspace` into *err_code (0 = none; bit 1 (value 1) = a
 * physical block id outside the pool; bit 3 (value 4) = a non-finite query or
 * summary-key value, ranked as zero; bit 4 (value 8) = more blocks to stage than
 * zr_offload_map's capacity). Returns ZR_EDEVICE if the word was non-zero, ZR_OK
 * otherwise.
 */
ZR_API zr_status zr_get_device_error(zr_plan_t plan, void* workspace, void* stream, int32_t* err_code);

/*
 * ---------------------------------------------------------------- append path
 * Three plan-free calls that keep the cache a decode step reads up to date.
 * They take a zr_config for the shapes (batch, num_kv_heads, head_dim,
 * block_size = 16, num_blocks, max_blocks_per_seq and dtype are used; the other
 * fields are ignored), are asynchronous on `stream` and allocate nothing. `err`
 * is an optional device int32 word (NULL: none) into which device-detected bad
 * indices are OR-ed: bit 1 a physical block id outside [0, num_blocks), bit 2 a
 * token position, segment or row index out of range; the offending row, pair
 * or segment is skipped (no trap). Host errors: ZR_EINVAL for a bad config, a
 * null required pointer, a negative count or a pool/row pointer that is not
 * 16-byte aligned; ZR_EUNSUPPORTED for a head_dim other than 64 or 128 (in
 * both cases nothing is launched); ZR_ECUDA if a launch fails.
 */

/*
 * zr_append_kv -- write one new token's K and V rows per sequence into the
 * paged pools ("KV-cache management" page, "Paged KV cache (PagedAttention)":
 * token t of sequence b lives in physical block block_tables[b][t / 16], slot
 * t % 16, for every KV head).
 *   positions      [B] int32: the token index t_b sequence b writes; negative:
 *                  sequence b writes nothing; t_b >= 16 * max_blocks_per_seq: bit 2
 *   k_new, v_new   [B, Hkv, d] dtype
 *   block_tables   [B, max_blocks_per_seq] int32; the block of t_b must already
 *                  be in the table and private to sequence b (the caller adds a
 *                  block when the last one is full and copies a shared last
 *                  block first, with zr_copy_blocks)
 *   k_pool, v_pool [num_blocks, Hkv, 16, d] dtype (written)
 */
ZR_API zr_status zr_append_kv(const zr_config* cfg, const int32_t* positions, const void* k_new, const void* v_new,
                              const int32_t* block_tables, void* k_pool, void* v_pool, int32_t* err, void* stream);

/*
 * zr_copy_blocks -- the copy-on-write step of the "KV-cache management" page,
 * "Block sharing with reference counts and copy-on-write", batched into one
 * launch: every (src, dst) pair copies the whole physical block src (all KV
 * heads, 16 rows) onto block dst, in both pools.
 *   pairs          [n][2] int32 (src, dst); n >= 0. The dst blocks must be
 *                  distinct and none may be a src of the same call (the copies
 *                  run concurrently).
 */
ZR_API zr_status zr_copy_blocks(const zr_config* cfg, const int32_t* pairs, int32_t n, void* k_pool, void* v_pool,
                                int32_t* err, void* stream);

/*
 * zr_segment_summaries -- the summary rows of completed segments (ZoomR page,
 * 3.3 "Representing Context with Mean Summary Keys": the mean summary key is
 * the average of the key vectors of the segment's tokens, per KV head; the
 * summary value row is the same average of the V rows).
 *   segs           [n][4] int32 (sequence b, first token s, end token e > s,
 *                  output row r), 16-byte aligned; n >= 0
 *   block_tables, k_pool, v_pool as in zr_append_kv (read)
 *   sum_k, sum_v   [num_rows, Hkv, d] dtype; row r is written for every KV
 *                  head: the rows are added in fp64 in ascending token order,
 *                  the sum is divided by e - s, and the mean is rounded to fp32
 *                  and then to dtype, each to nearest even. A segment with an
 *                  out-of-range index, or a block id outside the pool, is not
 *                  written.
 */
ZR_API zr_status zr_segment_summaries(const zr_config* cfg, const int32_t* segs, int32_t n, const int32_t* block_tables,
                                      const void* k_pool, const void* v_pool, void* sum_k, void* sum_v,
                                      int32_t num_rows, int32_t* err, void* stream);

/*
 * ----------------------------------------------------------- consensus path
 * ZoomR's own selection (ZoomR page, 3.3 "Global Aggregation and Consensus" and
 * "Constructing the Final Multi-Granularity Context"): every query head of every
 * layer votes for its top-k summaries, the c summaries with the most votes are
 * zoomed into their full regular segments, the other voted-for summaries keep
 * their summary segments, the rest are dropped, and every layer and head of a
 * sequence then attends over the one final token set
 *   I_f = prompt [0, N_p) + window [max(0, L - w), L) + R_i (i in I_c) + S_i (i in I_s).
 *
 * Layout of sequence b: the prompt [0, N_p), then n_b pairs of a regular segment
 * R_i and its summary segment S_i laid end to end, then possibly a tail with no
 * summary yet (only the window reaches it). The 2 n_b + 1 strictly ascending pair
 * bounds bd start at index 2 seg_ptr[b] + b of pair_bounds, with bd[0] = N_p and
 * bd[2 n_b] <= L_b: R_i = [bd[2i], bd[2i+1]), S_i = [bd[2i+1], bd[2i+2]).
 *
 * A step: zr_consensus_vote once per layer (votes accumulate in the workspace),
 * zr_consensus_select once (consumes and clears the votes, writes I_f), then
 * zr_consensus_attend once per layer; I_f stays in the workspace until the next
 * zr_consensus_select, so attend calls may repeat between selections. Plans of
 * this kind are rejected by the decode entry points and vice versa; the
 * workspace rules, zr_get_device_error and zr_free are shared.
 */

/*
 * zr_consensus_plan -- validate the consensus problem and build a plan.
 *   cfg            as for zr_plan (window = w; dtype of q, mean keys and pools)
 *   seq_lens       [B]  1 <= L_b <= 16 * max_blocks_per_seq
 *   prompt_lens    [B]  0 <= N_p <= L_b
 *   seg_ptr        [B+1] CSR over the pairs, 1 <= n_b <= 4096, seg_ptr[0] = 0
 *   pair_bounds    [2 seg_ptr[B] + B]  as described above
 *   topk           [B]  k_b >= 0 per query head (clipped to n_b)
 *   consensus      [B]  c_b >= 0 (clipped to n_b, then to |I_all|)
 * A sequence with N_p = 0, w = 0 and k_b = 0 could attend nothing: ZR_EINVAL.
 * Ties: equal scores and equal vote counts go to the lower summary index.
 * Errors as for zr_plan.
 */
ZR_API zr_status zr_consensus_plan(const zr_config* cfg, const int32_t* seq_lens, const int32_t* prompt_lens,
                                   const int32_t* seg_ptr, const int32_t* pair_bounds, const int32_t* topk,
                                   const int32_t* consensus, zr_plan_t* out_plan, size_t* workspace_bytes);

/* zr_consensus_dims -- *c_max = max_b min(c_b, n_b) (at least 1), *n_max = max_b n_b. */
ZR_API zr_status zr_consensus_dims(zr_plan_t plan, int32_t* c_max, int32_t* n_max);

/*
 * zr_consensus_vote -- one layer's votes (ZoomR 3.3 "Per-Head Importance Scoring
 * and Voting"): for every query head h, alpha_i = q_h . kbar_i over the
 * sequence's n_b summaries, with kbar the mean summary key of S_i for the KV
 * head h / G; the top-k indices each get one vote. alpha is the exact dot
 * product of the stored values (no scale), as in zr_decode_attend.
 *   q          [B, Hq, d] dtype (device)
 *   mean_keys  [seg_ptr[B], Hkv, d] dtype (device), pair rows in CSR order
 *              (zr_segment_summaries over the S_i spans computes them)
 */
ZR_API zr_status zr_consensus_vote(zr_plan_t plan, void* workspace, const void* q, const void* mean_keys,
                                   void* stream);

/*
 * zr_consensus_select -- the consensus over the accumulated votes and the final
 * token set of every sequence; clears the votes. Optional debug outputs (NULL:
 * not written), all int32 device arrays:
 *   votes_out      [B, n_max]    v_i (0 past n_b)
 *   consensus_out  [B, c_max]    I_c ascending, -1 padded
 *   ranges_out     [B, n_max + 2, 2]  I_f as maximal ranges [start, end), ascending
 *   nranges_out    [B]           number of ranges
 */
ZR_API zr_status zr_consensus_select(zr_plan_t plan, void* workspace, int32_t* votes_out, int32_t* consensus_out,
                                     int32_t* ranges_out, int32_t* nranges_out, void* stream);

/*
 * zr_consensus_attend -- one layer's attention over the current I_f (ZoomR 2
 * "Background": softmax(q K^T / sqrt(d)) V for every query head over the K/V rows
 * of I_f of its KV head, read through the block table).
 *   q [B, Hq, d] dtype; k_pool/v_pool [num_blocks, Hkv, 16, d] dtype;
 *   block_tables [B, max_blocks_per_seq] int32; out [B, Hq, d] float32 (written)
 * Call zr_consensus_select at least once before the first attend on a workspace.
 */
ZR_API zr_status zr_consensus_attend(zr_plan_t plan, void* workspace, const void* q, const void* k_pool,
                                     const void* v_pool, const int32_t* block_tables, float* out, void* stream);

/*
 * zr_consensus_attend_timed -- zr_consensus_attend with two CUDA events
 * (cudaEvent_t, either may be NULL but not both) recorded on `stream` just
 * before and just after the gather-attention kernel, so that the kernel alone can
 * be timed; the merge follows the second event. In a stream capture the events
 * become event-record nodes. Errors: as zr_consensus_attend; ZR_EINVAL if both
 * events are NULL.
 */
ZR_API zr_status zr_consensus_attend_timed(zr_plan_t plan, void* workspace, const void* q, const void* k_pool,
                                           const void* v_pool, const int32_t* block_tables, float* out,
                                           void* ev_start, void* ev_stop, void* stream);

/*
 * ------------------------------------------- steps between selections (amortisation)
 * ZoomR page, 3.4 "Decoding Stage" and appendix A.3 "Semantic Boundaries": the
 * selection is recomputed only at semantic boundaries (about every 35 tokens)
 * and reused for the steps in between. Between two selections the selected parts
 * stay fixed and the recent window follows the newest token: with L' cached
 * tokens it is [max(0, L' - w), L'). Tokens appended since the selection belong to
 * no segment and are reached only through the window.
 *
 * seq_lens is a DEVICE int32 array [B] of the new lengths L'_b. Each must lie in
 * [L_b of the plan, 16 * max_blocks_per_seq]; otherwise bit 2 of the workspace
 * error word is set and that sequence keeps its previous token ranges. The calls
 * are asynchronous on `stream` and allocate nothing.
 */

/*
 * zr_decode_advance -- rebuild every unit's token ranges from the selection the
 * last zr_decode_attend stored in the workspace (its selected segments) and the
 * window of the new lengths; the summary rows stay those of that selection.
 */
ZR_API zr_status zr_decode_advance(zr_plan_t plan, void* workspace, const int32_t* seq_lens, void* stream);

/*
 * zr_decode_attend_reuse -- the gather-attention and merge of zr_decode_attend
 * over the token ranges and summary rows currently in the workspace (from the
 * last zr_decode_attend or zr_decode_advance); no scoring or selection. Same
 * arguments as zr_decode_attend without the debug outputs.
 */
ZR_API zr_status zr_decode_attend_reuse(zr_plan_t plan, void* workspace, const void* q, const void* k_pool,
                                        const void* v_pool, const int32_t* block_tables, const void* sum_k,
                                        const void* sum_v, float* out, void* stream);

/*
 * zr_consensus_advance -- the consensus path's final sets for the new lengths:
 * the prompt, zoomed regular segments and candidate summary segments of the last
 * zr_consensus_select, with the window of the new lengths. zr_consensus_attend
 * then attends over them.
 */
ZR_API zr_status zr_consensus_advance(zr_plan_t plan, void* workspace, const int32_t* seq_lens, void* stream);

/*
 * The offloaded cache: ZoomR page, 3.4 "System Implementation and Inference",
 * "Decoding Stage" (the full KV cache stays in host memory; for every layer only
 * the final context I_f is brought to the GPU, the next layer's while the current
 * one attends). The pools of every layer live in host memory the device can read
 * (pinned or registered); the caller owns two staging pools in HBM of `capacity`
 * blocks each, [capacity, Hkv, 16, d] dtype, and alternates them over the layers.
 *
 * zr_offload_map -- after a selection or an advance (zr_decode_attend,
 * zr_consensus_select, zr_decode_advance, zr_consensus_advance on this
 * workspace): give a staging slot to every physical block that the workspace's
 * current token ranges touch (the union over every KV head of a sequence, each
 * shared block once, slots in ascending physical order), and keep in the
 * workspace, per (block, KV head), the mask of the rows those ranges cover.
 *   block_tables  [B, max_blocks_per_seq] int32 (device): the host pools' tables
 *   capacity      slots per staging pool (>= 1)
 *   stage_ids     [capacity] int32 (device, out): physical block of each used slot
 *   remap_tables  [B, max_blocks_per_seq] int32 (device, out): the slot of every
 *                 logical block a range touches, -1 elsewhere; pass it as the
 *                 block tables of the attention over the staging pools
 *   n_staged      [1] int32 (device, out): slots used, min(blocks touched, capacity)
 * Asynchronous on `stream`. More blocks than `capacity` set bit 4 (value 8) of the
 * workspace error word; the blocks past capacity map to -1 and their rows are
 * masked. Errors: ZR_EINVAL (null pointer, capacity < 1), ZR_ECUDA.
 */
ZR_API zr_status zr_offload_map(zr_plan_t plan, void* workspace, const int32_t* block_tables, int32_t capacity,
                                int32_t* stage_ids, int32_t* remap_tables, int32_t* n_staged, void* stream);

/*
 * zr_offload_stage -- one layer's staging copy: slot i of stage_k / stage_v
 * receives the rows of block stage_ids[i] of host_k_pool / host_v_pool that the
 * workspace's ranges cover (row r of KV head h when some range of head h holds
 * that token: exactly the rows of I_f), for i < *n_staged (all from
 * zr_offload_map on this workspace, whose row masks it reads). The other rows of
 * a slot keep whatever they held; the attention never reads them. Pools
 * [num_blocks, Hkv, 16, d] in host memory the device can read; staging pools
 * [capacity, Hkv, 16, d] in device memory; all 16-byte aligned. Asynchronous on
 * `stream` (a copy stream, so the next layer's copy overlaps the current layer's
 * attention). Errors: ZR_EINVAL (null or misaligned pointer, capacity < 1),
 * ZR_EUNSUPPORTED (more than 256 KV heads), ZR_ECUDA.
 */
ZR_API zr_status zr_offload_stage(zr_plan_t plan, const void* workspace, const void* host_k_pool,
                                  const void* host_v_pool, const int32_t* stage_ids, const int32_t* n_staged,
                                  int32_t capacity, void* stage_k, void* stage_v, void* stream);

/*
 * zr_plan_set_deterministic -- choose how the gather-attention kernel of the
 * attend-only calls (zr_consensus_attend, zr_decode_attend_reuse and their timed
 * forms) splits a call's rows among its warps. The pages leave the schedule open;
 * this is a deployment choice, not part of the method.
 *   deterministic = 0 (the default of every plan): each unit's rows are handed out
 *     in 32-row batches from a per-unit counter in the workspace, so the warps of
 *     a unit keep streaming until its rows run out however fast their SMs run or
 *     however late their CTAs start. Which warp takes which batch changes from
 *     call to call, and with it the rounding of the output (within the documented
 *     tolerance of the exact result; selections, ranges and every integer output
 *     are unaffected). Plans whose units hold more than 94 ranges (k_max + 1 > 95)
 *     always take the even split.
 *   deterministic = 1: a fixed even split of the rows; the output bits of a plan
 *     are identical across calls, streams and the entry points that share a kernel.
 * zr_decode_attend (the decode step, select and attend) always takes the even
 * split: its attend CTAs are resident while the select kernel runs.
 * The counters return to zero by the end of every call, so a workspace zeroed once
 * before its first use stays valid in both modes. Takes effect at the next call.
 * Errors: ZR_EINVAL (null plan, or a value other than 0 or 1).
 */
ZR_API zr_status zr_plan_set_deterministic(zr_plan_t plan, int32_t deterministic);

/* zr_free -- release the plan and its small device metadata (NULL is a no-op). */
ZR_API void zr_free(zr_plan_t plan);

/* zr_status_string -- static, human-readable name of a status. */
ZR_API const char* zr_status_string(zr_status s);

#ifdef __cplusplus
}
#endif

#endif /* ZOOMR_H */
