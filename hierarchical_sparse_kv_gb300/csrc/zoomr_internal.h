// Internal declarations shared by the plan (host) and kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include "zoomr.h"

namespace zr {

constexpr int kBlockTokens = 16;      // tokens per paged KV block
constexpr int kSelPrefetchBlocks = 128;  // blocks before each unit's window the select kernel lists for prefetch
constexpr int kMaxSegments = 4096;    // n_b limit of the select kernel's shared memory
constexpr int kMaxGroup = 16;         // query heads per KV head
constexpr int kMmaMaxGroup = 8;       // the tensor-core attend kernel packs the group into 8 MMA columns
constexpr int kChunkRows = 256;       // rows of one attend warp's row table (a range is walked in such pieces)
constexpr int kBatchRows = 32;        // dynamic split: rows a warp claims at a time
constexpr int kRangeCache = 95;       // dynamic split: ranges per unit a warp keeps in its row table's space
constexpr int kCtrStride = 32;        // dynamic split: one counter per 128-byte line (claims of different units
                                      // meet in different L2 slices)
#ifndef ZR_ATTEND_WARPS
#define ZR_ATTEND_WARPS 4
#endif
constexpr int kAttendWarps = ZR_ATTEND_WARPS;  // warps per attend CTA
constexpr int kSelectThreads = 512;   // threads per select CTA
// Virtual rows in front of each unit in the attend kernels' split of a decode plan (measured best
// on the 16K-token workload in a sweep of 0 to 128; consensus plans use 0).
#ifndef ZR_UNIT_START_ROWS
#define ZR_UNIT_START_ROWS 48
#endif
constexpr int kUnitStartRows = ZR_UNIT_START_ROWS;
constexpr uint32_t kSummaryFlag = 0x80000000u;  // row id refers to the summary tensors
constexpr uint32_t kInvalidRow = 0xFFFFFFFFu;   // masked row (past the chunk end, or a bad block id)

enum : int32_t { kErrBadBlock = 1, kErrBadIndex = 2, kErrNonFinite = 4, kErrStage = 8 };

// Small device metadata copied from the host at plan time (one allocation).
struct DeviceMeta {
  int32_t* seq_lens;     // [B]
  int32_t* seg_ptr;      // [B+1]
  int32_t* seg_bounds;   // decode: [total_segments + B] segment bounds; consensus: [2 total_segments + B] pair bounds
  int32_t* topk;         // [B], already clipped to n_b
  int32_t* prompt_lens;  // consensus only: [B] N_p
  int32_t* consensus;    // consensus only: [B] c, already clipped to n_b
};

// Byte offsets into the caller's workspace.
struct WsLayout {
  size_t err;         // int32 sticky error word
  size_t unit_info;   // int32 [U][4]: n_ranges, n_tok, n_sum, 0
  size_t unit_rows;   // int32 [U]: n_tok + n_sum, the rows the unit gathers
  size_t ranges;      // int32 [U][k_max+1][2]
  size_t cum;         // int32 [U][k_max+2] prefix sums of range lengths
  size_t sumlist;     // int32 [U][n_max] non-selected segments, ascending
  size_t sel;         // int32 [U][k_max] selected segments, ascending
  size_t part_o;      // float [U + attend_warps][G][d] unnormalised split outputs
  size_t part_ml;     // float [U + attend_warps][G][2] split (max, sum) in log2 units
  size_t bigkeys;     // uint32 [U][n_max][20] exact keys of units that take the general (640-bit) path
  size_t stage_marks; // int32 [num_blocks] offload map: staging slot + 1 of every physical block (0: not staged)
  size_t stage_rows;  // uint32 [num_blocks][Hkv] offload map: rows of the block that a range of the head covers
  size_t pf_list;     // int32 [U][kSelPrefetchBlocks] selected blocks before each unit's window (-1: none)
  size_t tile_ctr;    // int32 [U][kCtrStride] dynamic split: the next 32-row batch of unit u at [u][0] (0 between launches)
  size_t votes;       // consensus only: int32 [B][n_max] vote counts, zero between selections
  size_t cruns;       // consensus only: int32 [B][n_max + 1][2] the last selection's runs before the window
  size_t cnruns;      // consensus only: int32 [B] their count
  size_t total;
};

enum PlanMode : int { kDecodePlan = 0, kConsensusPlan = 1 };

struct Plan {
  int mode;  // PlanMode
  zr_config cfg;
  int B, Hq, Hkv, G, d, window, num_blocks, max_blocks;
  int k_max, n_max, total_segments;  // consensus: k_max = n_max + 1 (range capacity n_max + 2 per unit)
  int c_max;                          // consensus: max clipped c (at least 1)
  int attend_ctas;   // persistent attend grid (one resident wave)
  int attend_warps;  // attend_ctas * kAttendWarps
  int fixed_rows;    // max over sequences of the tokens gathered whatever the selection: sink / prompt + window
  int pf_blocks;     // decode step: blocks before each unit's window scanned for the selected-tile prefetch
  int prompt_rows;   // max over sequences of the sink / prompt length
  int device;
  void* d_meta_base;
  DeviceMeta meta;
  WsLayout ws;
  int merge_parts;     // merge layout: 1 lanes over partials, 0 lanes over components
  int deterministic;   // 1: the attend kernels' static split (outputs bit-identical across calls)
  size_t select_smem;  // dynamic shared memory of the select kernel
  size_t attend_smem;  // dynamic shared memory of the attend kernel
};

// Everything one launch needs, passed by value.
struct StepArgs {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_tables;
  const void* sum_k;
  const void* sum_v;
  float* out;
  int32_t* sel_out;
  int32_t* ranges_out;
  int32_t* nranges_out;
  DeviceMeta meta;
  int32_t* err;
  int4* unit_info;
  int32_t* unit_rows;
  int32_t* ranges;
  int32_t* cum;
  int32_t* sumlist;
  int32_t* sel;
  float* part_o;
  float2* part_ml;
  uint32_t* bigkeys;
  int32_t* pf_list;  // decode step: blocks the attend kernel prefetches after its wait
  int32_t* tile_ctr;  // dynamic split: per-unit batch counters
  int32_t* cruns;   // consensus only
  int32_t* cnruns;  // consensus only
  int B, Hq, Hkv, G, window, num_blocks, max_blocks, k_max, n_max, attend_warps;
  int unit_cost;  // virtual rows in front of every unit in the attend kernels' even split (see kernels)
  int dynamic;    // 1: the tensor-core attend kernel hands out each unit's rows in 32-row batches (see kernels)
  int fixed_rows;  // rows per sequence prefetched before the attend kernel's wait (0: none)
  int fixed_window;  // 1: the window rows too (the decode step, whose lengths are the plan's); 0: the prompt only
  int pf_blocks;  // decode step: blocks before each window the select kernel scans and lists for the attend
                  // kernel's prefetch (entries up to kSelPrefetchBlocks, the rest -1); 0: no list, no prefetch
  float scale_log2;  // log2(e) / sqrt(d)
};

// Implemented in zoomr_plan.cpp: the launch arguments that point into `workspace` (plus the plan's sizes).
StepArgs step_args(const Plan& p, void* workspace);

// Implemented in zoomr_plan.cpp: the checks of a decode call's tensor arguments (null, alignment, plan
// kind); ZR_OK or ZR_EINVAL, nothing launched.
zr_status check_decode_args(zr_plan_t plan, const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* block_tables, const void* sum_k, const void* sum_v, const float* out);

// Implemented in zoomr_plan.cpp: argument checks, then one decode step on `workspace`.
zr_status decode_into(zr_plan_t plan, void* workspace, const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* block_tables, const void* sum_k, const void* sum_v, float* out,
                      int32_t* sel_out, int32_t* ranges_out, int32_t* nranges_out, void* stream, void* ev_start,
                      void* ev_stop);

// Implemented in zoomr_kernels.cu.
// Sets kernel attributes and sizes the persistent attend grid (p.attend_ctas, p.attend_warps)
// for at most `useful_warps` warps.
zr_status configure_kernels(Plan& p, int64_t useful_warps);
zr_status launch_step(const Plan& p, const StepArgs& a, void* stream, void* ev_start, void* ev_stop);
// Gather-attention and merge only, over the unit metadata already in the workspace; optional events
// (null: none) recorded just before and just after the gather-attention kernel.
zr_status launch_attend_only(const Plan& p, const StepArgs& a, void* stream, void* ev_start = nullptr,
                             void* ev_stop = nullptr);

// Implemented in zoomr_consensus.cu.
size_t vote_smem_bytes(int G, int d, int n_max);
size_t consensus_smem_bytes(int n_max);
zr_status launch_vote(const Plan& p, const StepArgs& a, const void* mean_keys, int32_t* votes, void* stream);
zr_status launch_consensus(const Plan& p, const StepArgs& a, int32_t* votes, int32_t* votes_out, int32_t* ic_out,
                           void* stream);
// Between selections: rebuild every unit's token ranges for new sequence lengths (device int32 [B]).
zr_status launch_decode_advance(const Plan& p, const StepArgs& a, const int32_t* seq_lens, void* stream);
zr_status launch_consensus_advance(const Plan& p, const StepArgs& a, const int32_t* seq_lens, void* stream);

}  // namespace zr

struct zr_plan {
  zr::Plan p;
};
