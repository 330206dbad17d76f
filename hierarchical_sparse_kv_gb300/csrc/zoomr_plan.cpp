// Host side of the C ABI: validation of the problem statement, the plan, the
// workspace layout, device-error readback.
//
// The plan turns the caller's host metadata (sequence lengths, segment bounds,
// per-sequence top-k) into a few small device arrays and sizes the persistent
// attend grid. The bound on a unit's gathered rows is exact arithmetic on the
// metadata: at most min(L, min(w, L) + sum of the k largest segment lengths)
// tokens (the window and the selected segments' ranges, ZoomR page 3.3
// "Constructing the Final Multi-Granularity Context") plus exactly n - k
// summary rows.

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <new>
#include <vector>

#include "zoomr_internal.h"

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

zr_status validate_shape(const zr_config* c);

zr_status validate(const zr_config* c, const int32_t* seq_lens, const int32_t* seg_ptr, const int32_t* seg_bounds,
                   const int32_t* topk, const int32_t* sink_lens) {
  if (!c || !seq_lens || !seg_ptr || !seg_bounds || !topk) return ZR_EINVAL;
  const zr_status st = validate_shape(c);
  if (st != ZR_OK) return st;
  if (seg_ptr[0] != 0) return ZR_EINVAL;
  for (int b = 0; b < c->batch; ++b) {
    const int32_t L = seq_lens[b];
    if (L < 1 || static_cast<int64_t>(L) > static_cast<int64_t>(c->max_blocks_per_seq) * zr::kBlockTokens)
      return ZR_EINVAL;
    const int64_t n = static_cast<int64_t>(seg_ptr[b + 1]) - seg_ptr[b];
    if (n < 1) return ZR_EINVAL;
    if (n > zr::kMaxSegments) return ZR_EUNSUPPORTED;
    if (topk[b] < 0) return ZR_EINVAL;
  }
  const int64_t total = seg_ptr[c->batch];
  if (total * c->num_kv_heads >= (int64_t(1) << 31)) return ZR_EUNSUPPORTED;
  for (int b = 0; b < c->batch; ++b) {
    const int32_t* bd = seg_bounds + seg_ptr[b] + b;
    const int n = seg_ptr[b + 1] - seg_ptr[b];
    const int32_t sink = sink_lens ? sink_lens[b] : 0;
    if (sink < 0 || bd[0] != sink || bd[n] != seq_lens[b]) return ZR_EINVAL;
    for (int i = 0; i < n; ++i)
      if (bd[i + 1] <= bd[i]) return ZR_EINVAL;
  }
  return ZR_OK;
}

// The shape checks shared by both plan kinds. Row ids of the pool are (block * Hkv + head) * 16 + slot
// and must stay below 2^31.
zr_status validate_shape(const zr_config* c) {
  if (c->batch < 1 || c->num_q_heads < 1 || c->num_kv_heads < 1) return ZR_EINVAL;
  if (c->num_q_heads % c->num_kv_heads != 0) return ZR_EINVAL;
  if (c->block_size != zr::kBlockTokens) return ZR_EINVAL;
  if (c->num_blocks < 1 || c->max_blocks_per_seq < 1 || c->window < 0) return ZR_EINVAL;
  if (c->dtype != ZR_F32 && c->dtype != ZR_BF16) return ZR_EINVAL;
  if (c->head_dim != 64 && c->head_dim != 128) return c->head_dim < 1 ? ZR_EINVAL : ZR_EUNSUPPORTED;
  if (c->num_q_heads / c->num_kv_heads > zr::kMaxGroup) return ZR_EUNSUPPORTED;
  if (static_cast<int64_t>(c->num_blocks) * c->num_kv_heads * zr::kBlockTokens >= (int64_t(1) << 31))
    return ZR_EUNSUPPORTED;
  return ZR_OK;
}

zr_status validate_consensus(const zr_config* c, const int32_t* seq_lens, const int32_t* prompt_lens,
                             const int32_t* seg_ptr, const int32_t* pair_bounds, const int32_t* topk,
                             const int32_t* consensus) {
  if (!c || !seq_lens || !prompt_lens || !seg_ptr || !pair_bounds || !topk || !consensus) return ZR_EINVAL;
  const zr_status st = validate_shape(c);
  if (st != ZR_OK) return st;
  if (seg_ptr[0] != 0) return ZR_EINVAL;
  for (int b = 0; b < c->batch; ++b) {
    const int32_t L = seq_lens[b];
    if (L < 1 || static_cast<int64_t>(L) > static_cast<int64_t>(c->max_blocks_per_seq) * zr::kBlockTokens)
      return ZR_EINVAL;
    const int64_t n = static_cast<int64_t>(seg_ptr[b + 1]) - seg_ptr[b];
    if (n < 1) return ZR_EINVAL;
    if (n > zr::kMaxSegments) return ZR_EUNSUPPORTED;
    if (topk[b] < 0 || consensus[b] < 0 || prompt_lens[b] < 0 || prompt_lens[b] > L) return ZR_EINVAL;
    // I_f must never be empty: a prompt, a window or at least one vote
    if (prompt_lens[b] == 0 && c->window == 0 && topk[b] == 0) return ZR_EINVAL;
  }
  const int64_t total = seg_ptr[c->batch];
  if (2 * total * c->num_kv_heads >= (int64_t(1) << 31)) return ZR_EUNSUPPORTED;
  for (int b = 0; b < c->batch; ++b) {
    const int32_t* bd = pair_bounds + 2 * static_cast<int64_t>(seg_ptr[b]) + b;
    const int n = seg_ptr[b + 1] - seg_ptr[b];
    if (bd[0] != prompt_lens[b] || bd[2 * n] > seq_lens[b]) return ZR_EINVAL;
    for (int i = 0; i < 2 * n; ++i)
      if (bd[i + 1] <= bd[i]) return ZR_EINVAL;
  }
  return ZR_OK;
}

// Workspace layout shared by both plan kinds (each region 256-byte aligned).
void layout_workspace(zr::Plan& p) {
  const size_t U = static_cast<size_t>(p.B) * p.Hkv;
  const size_t slots = U + static_cast<size_t>(p.attend_warps);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  p.ws.err = take(sizeof(int32_t));
  p.ws.unit_info = take(U * 4 * sizeof(int32_t));
  p.ws.unit_rows = take(U * sizeof(int32_t));
  p.ws.ranges = take(U * (p.k_max + 1) * 2 * sizeof(int32_t));
  p.ws.cum = take(U * (p.k_max + 2) * sizeof(int32_t));
  p.ws.sumlist = take(U * p.n_max * sizeof(int32_t));
  p.ws.sel = take(U * p.k_max * sizeof(int32_t));
  p.ws.part_o = take(slots * p.G * p.d * sizeof(float));
  p.ws.part_ml = take(slots * p.G * 2 * sizeof(float));
  p.ws.bigkeys = take(U * p.n_max * 20 * sizeof(uint32_t));
  p.ws.stage_marks = take(static_cast<size_t>(p.num_blocks) * sizeof(int32_t));
  p.ws.stage_rows = take(static_cast<size_t>(p.num_blocks) * p.Hkv * sizeof(uint32_t));
  p.ws.pf_list = take(U * zr::kSelPrefetchBlocks * sizeof(int32_t));
  p.ws.tile_ctr = take(U * zr::kCtrStride * sizeof(int32_t));
  const bool cons = p.mode == zr::kConsensusPlan;
  p.ws.votes = cons ? take(static_cast<size_t>(p.B) * p.n_max * sizeof(int32_t)) : 0;
  p.ws.cruns = cons ? take(static_cast<size_t>(p.B) * (p.n_max + 1) * 2 * sizeof(int32_t)) : 0;
  p.ws.cnruns = cons ? take(static_cast<size_t>(p.B) * sizeof(int32_t)) : 0;
  p.ws.total = off;
}

zr_status make_decode_plan(const zr_config* cfg, const int32_t* seq_lens, const int32_t* seg_ptr,
                           const int32_t* seg_bounds, const int32_t* topk, const int32_t* sink_lens,
                           zr_plan_t* out_plan, size_t* workspace_bytes);

}  // namespace

extern "C" {

zr_status zr_plan(const zr_config* cfg, const int32_t* seq_lens, const int32_t* seg_ptr, const int32_t* seg_bounds,
                  const int32_t* topk, zr_plan_t* out_plan, size_t* workspace_bytes) {
  return make_decode_plan(cfg, seq_lens, seg_ptr, seg_bounds, topk, nullptr, out_plan, workspace_bytes);
}

zr_status zr_plan_sink(const zr_config* cfg, const int32_t* seq_lens, const int32_t* sink_lens,
                       const int32_t* seg_ptr, const int32_t* seg_bounds, const int32_t* topk, zr_plan_t* out_plan,
                       size_t* workspace_bytes) {
  if (!sink_lens) return ZR_EINVAL;
  return make_decode_plan(cfg, seq_lens, seg_ptr, seg_bounds, topk, sink_lens, out_plan, workspace_bytes);
}

}  // extern "C"

namespace {

zr_status make_decode_plan(const zr_config* cfg, const int32_t* seq_lens, const int32_t* seg_ptr,
                           const int32_t* seg_bounds, const int32_t* topk, const int32_t* sink_lens,
                           zr_plan_t* out_plan, size_t* workspace_bytes) {
  if (!out_plan || !workspace_bytes) return ZR_EINVAL;
  *out_plan = nullptr;
  *workspace_bytes = 0;
  zr_status st = validate(cfg, seq_lens, seg_ptr, seg_bounds, topk, sink_lens);
  if (st != ZR_OK) return st;

  struct zr_plan* P = new (std::nothrow) struct zr_plan();
  if (!P) return ZR_ENOMEM;
  zr::Plan& p = P->p;
  p.mode = zr::kDecodePlan;
  p.cfg = *cfg;
  p.B = cfg->batch;
  p.Hq = cfg->num_q_heads;
  p.Hkv = cfg->num_kv_heads;
  p.G = p.Hq / p.Hkv;
  p.d = cfg->head_dim;
  p.window = cfg->window;
  p.num_blocks = cfg->num_blocks;
  p.max_blocks = cfg->max_blocks_per_seq;
  p.total_segments = seg_ptr[p.B];

  // Upper bound on the rows all units gather (window + the k longest segments, plus n - k summary
  // rows per unit): the attend grid never needs more than one warp per 16 of them.
  std::vector<int32_t> kclip(p.B);
  p.k_max = 1;
  p.n_max = 1;
  int64_t rows_bound = 0;
  bool any_sink = false;
  for (int b = 0; b < p.B; ++b) {
    const int n = seg_ptr[b + 1] - seg_ptr[b];
    const int32_t* bd = seg_bounds + seg_ptr[b] + b;
    const int L = seq_lens[b];
    kclip[b] = std::min(topk[b], n);
    p.k_max = std::max(p.k_max, kclip[b]);
    p.n_max = std::max(p.n_max, n);
    std::vector<int32_t> lens(n);
    for (int i = 0; i < n; ++i) lens[i] = bd[i + 1] - bd[i];
    std::sort(lens.begin(), lens.end(), std::greater<int32_t>());
    int64_t top = 0;
    for (int i = 0; i < kclip[b]; ++i) top += lens[i];
    const int32_t sink = sink_lens ? sink_lens[b] : 0;
    const int64_t tok_bound = std::min<int64_t>(L, sink + std::min<int64_t>(p.window, L) + top);
    p.fixed_rows =
        static_cast<int>(std::max<int64_t>(p.fixed_rows, std::min<int64_t>(L, sink + std::min(p.window, L))));
    p.prompt_rows = std::max(p.prompt_rows, static_cast<int>(sink));
    rows_bound += (tok_bound + (n - kclip[b])) * p.Hkv;
    any_sink = any_sink || sink > 0;
  }
  if (any_sink) ++p.k_max;  // one more range slot per unit for the sink's range
  // The selected-tile prefetch scans up to kSelPrefetchBlocks blocks per unit and about 8192 over all
  // units (about a quarter of them selected: some 16 MB of K and V, what the attend start-up leaves
  // idle); more units scan fewer blocks each (8 x 16K: 128; 32 ragged sequences: 32).
  p.pf_blocks = static_cast<int>(std::min<int64_t>(zr::kSelPrefetchBlocks,
                                                   std::max<int64_t>(8, 8192 / (static_cast<int64_t>(p.B) * p.Hkv))));
  if (cudaGetDevice(&p.device) != cudaSuccess) {
    cudaGetLastError();
    delete P;
    return ZR_ECUDA;
  }
  st = zr::configure_kernels(p, (rows_bound + 15) / 16);
  if (st != ZR_OK) {
    delete P;
    return st;
  }

  layout_workspace(p);

  // Device metadata: one allocation, synchronous copies.
  const size_t nb = static_cast<size_t>(p.B);
  const size_t n_bounds = static_cast<size_t>(p.total_segments) + nb;
  size_t moff = 0;
  auto mtake = [&](size_t count) {
    size_t at = moff;
    moff = align_up(moff + count * sizeof(int32_t), 256);
    return at;
  };
  const size_t o_len = mtake(nb), o_ptr = mtake(nb + 1), o_bnd = mtake(n_bounds), o_topk = mtake(nb),
               o_sink = mtake(nb);
  void* base = nullptr;
  cudaError_t ce = cudaMalloc(&base, moff);
  if (ce != cudaSuccess) {
    cudaGetLastError();
    delete P;
    return ce == cudaErrorMemoryAllocation ? ZR_ENOMEM : ZR_ECUDA;
  }
  p.d_meta_base = base;
  char* cb = static_cast<char*>(base);
  p.meta.seq_lens = reinterpret_cast<int32_t*>(cb + o_len);
  p.meta.seg_ptr = reinterpret_cast<int32_t*>(cb + o_ptr);
  p.meta.seg_bounds = reinterpret_cast<int32_t*>(cb + o_bnd);
  p.meta.topk = reinterpret_cast<int32_t*>(cb + o_topk);
  p.meta.prompt_lens = reinterpret_cast<int32_t*>(cb + o_sink);  // the sink lengths (0 without a sink)
  std::vector<int32_t> sinks(p.B, 0);
  if (sink_lens) std::copy(sink_lens, sink_lens + p.B, sinks.begin());
  bool ok = cudaMemcpy(p.meta.seq_lens, seq_lens, nb * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(p.meta.seg_ptr, seg_ptr, (nb + 1) * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(p.meta.seg_bounds, seg_bounds, n_bounds * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(p.meta.topk, kclip.data(), nb * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(p.meta.prompt_lens, sinks.data(), nb * 4, cudaMemcpyHostToDevice) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    cudaFree(base);
    delete P;
    return ZR_ECUDA;
  }
  *out_plan = P;
  *workspace_bytes = p.ws.total;
  return ZR_OK;
}

}  // namespace

extern "C" {

zr_status zr_plan_dims(zr_plan_t plan, int32_t* k_max, int32_t* n_max) {
  if (!plan || !k_max || !n_max || plan->p.mode != zr::kDecodePlan) return ZR_EINVAL;
  *k_max = plan->p.k_max;
  *n_max = plan->p.n_max;
  return ZR_OK;
}

}  // extern "C"

namespace zr {

zr_status check_decode_args(zr_plan_t plan, const void* q, const void* k_pool, const void* v_pool,
                             const int32_t* block_tables, const void* sum_k, const void* sum_v, const float* out) {
  if (!plan || !q || !k_pool || !v_pool || !block_tables || !sum_k || !sum_v || !out) return ZR_EINVAL;
  if (plan->p.mode != kDecodePlan) return ZR_EINVAL;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(sum_k, 16) ||
      !aligned(sum_v, 16) || !aligned(out, 16) || !aligned(block_tables, 4))
    return ZR_EINVAL;
  return ZR_OK;
}

zr_status decode_into(zr_plan_t plan, void* workspace, const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_tables, const void* sum_k, const void* sum_v, float* out,
                               int32_t* sel_out, int32_t* ranges_out, int32_t* nranges_out, void* stream,
                               void* ev_start, void* ev_stop) {
  const zr_status st = check_decode_args(plan, q, k_pool, v_pool, block_tables, sum_k, sum_v, out);
  if (st != ZR_OK) return st;
  if (!workspace || !aligned(workspace, 256)) return ZR_EINVAL;
  zr::StepArgs a = step_args(plan->p, workspace);
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.block_tables = block_tables;
  a.sum_k = sum_k;
  a.sum_v = sum_v;
  a.out = out;
  a.sel_out = sel_out;
  a.ranges_out = ranges_out;
  a.nranges_out = nranges_out;
  // The pools of a decode step are the plan's full pools, so the attend kernel may prefetch the rows every
  // unit gathers (sink and window) through the block tables before its wait. The attend-only entry points
  // can be given staging pools with fewer blocks (the offloaded cache) and do not prefetch.
  a.fixed_rows = plan->p.fixed_rows;
  a.fixed_window = 1;
  a.pf_blocks = plan->p.pf_blocks;
  // The decode step keeps the even split: its attend CTAs are resident and waiting while the select kernel
  // runs, and measured on the 8 x 16K-token workload the dynamic split's batch claims cost more there
  // (878 against 887 steps/s) than they save at the tail.
  a.dynamic = 0;
  return zr::launch_step(plan->p, a, stream, ev_start, ev_stop);
}

StepArgs step_args(const Plan& p, void* workspace) {
  char* ws = static_cast<char*>(workspace);
  StepArgs a{};
  a.meta = p.meta;
  a.err = reinterpret_cast<int32_t*>(ws + p.ws.err);
  a.unit_info = reinterpret_cast<int4*>(ws + p.ws.unit_info);
  a.unit_rows = reinterpret_cast<int32_t*>(ws + p.ws.unit_rows);
  a.ranges = reinterpret_cast<int32_t*>(ws + p.ws.ranges);
  a.cum = reinterpret_cast<int32_t*>(ws + p.ws.cum);
  a.sumlist = reinterpret_cast<int32_t*>(ws + p.ws.sumlist);
  a.sel = reinterpret_cast<int32_t*>(ws + p.ws.sel);
  a.part_o = reinterpret_cast<float*>(ws + p.ws.part_o);
  a.part_ml = reinterpret_cast<float2*>(ws + p.ws.part_ml);
  a.bigkeys = reinterpret_cast<uint32_t*>(ws + p.ws.bigkeys);
  a.pf_list = reinterpret_cast<int32_t*>(ws + p.ws.pf_list);
  a.tile_ctr = reinterpret_cast<int32_t*>(ws + p.ws.tile_ctr);
  a.cruns = p.mode == kConsensusPlan ? reinterpret_cast<int32_t*>(ws + p.ws.cruns) : nullptr;
  a.cnruns = p.mode == kConsensusPlan ? reinterpret_cast<int32_t*>(ws + p.ws.cnruns) : nullptr;
  a.B = p.B;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.G = p.G;
  a.window = p.window;
  a.num_blocks = p.num_blocks;
  a.max_blocks = p.max_blocks;
  a.k_max = p.k_max;
  a.n_max = p.n_max;
  a.attend_warps = p.attend_warps;
  // A second unit in a warp's share costs a second start. Decode units of one sequence gather
  // different tokens (each KV head selects its own segments); consensus units share one token set,
  // whose block-table entries the next unit finds cached, and a start there costs little.
  a.unit_cost = p.mode == kConsensusPlan ? 0 : kUnitStartRows;
  // Attend-only calls (consensus attention, steps between selections, the offloaded cache) take the dynamic
  // split unless the plan is deterministic. It keeps a unit's ranges in shared memory, so plans with more
  // range slots take the even split.
  a.dynamic = !p.deterministic && p.k_max + 1 <= kRangeCache ? 1 : 0;
  a.fixed_rows = 0;  // set by the decode step and the attend-only calls (see decode_into)
  a.fixed_window = 0;
  a.pf_blocks = 0;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(p.d)));
  return a;
}

}  // namespace zr

extern "C" {

zr_status zr_decode_attend(zr_plan_t plan, void* workspace, const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* block_tables, const void* sum_k, const void* sum_v, float* out,
                           int32_t* sel_out, int32_t* ranges_out, int32_t* nranges_out, void* stream) {
  return zr::decode_into(plan, workspace, q, k_pool, v_pool, block_tables, sum_k, sum_v, out, sel_out, ranges_out,
                       nranges_out, stream, nullptr, nullptr);
}

zr_status zr_decode_attend_timed(zr_plan_t plan, void* workspace, const void* q, const void* k_pool,
                                 const void* v_pool, const int32_t* block_tables, const void* sum_k,
                                 const void* sum_v, float* out, void* ev_start, void* ev_stop, void* stream) {
  if (!ev_start && !ev_stop) return ZR_EINVAL;
  return zr::decode_into(plan, workspace, q, k_pool, v_pool, block_tables, sum_k, sum_v, out, nullptr, nullptr,
                       nullptr, stream, ev_start, ev_stop);
}

zr_status zr_get_device_error(zr_plan_t plan, void* workspace, void* stream, int32_t* err_code) {
  if (!plan || !workspace || !err_code) return ZR_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* dev = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + plan->p.ws.err);
  int32_t v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess || cudaMemcpy(&v, dev, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return ZR_ECUDA;
  }
  *err_code = v;
  if (v != 0) {
    if (cudaMemset(dev, 0, sizeof(v)) != cudaSuccess) {
      cudaGetLastError();
      return ZR_ECUDA;
    }
    return ZR_EDEVICE;
  }
  return ZR_OK;
}

void zr_free(zr_plan_t plan) {
  if (!plan) return;
  if (plan->p.d_meta_base) cudaFree(plan->p.d_meta_base);
  delete plan;
}

zr_status zr_plan_set_deterministic(zr_plan_t plan, int32_t deterministic) {
  if (!plan || (deterministic != 0 && deterministic != 1)) return ZR_EINVAL;
  plan->p.deterministic = deterministic;
  return ZR_OK;
}

const char* zr_status_string(zr_status s) {
  switch (s) {
    case ZR_OK: return "ZR_OK";
    case ZR_EINVAL: return "ZR_EINVAL: invalid argument";
    case ZR_ENOMEM: return "ZR_ENOMEM: allocation failed";
    case ZR_ECUDA: return "ZR_ECUDA: CUDA runtime error";
    case ZR_EUNSUPPORTED: return "ZR_EUNSUPPORTED: outside the library's supported limits";
    case ZR_EDEVICE: return "ZR_EDEVICE: the device reported a bad index";
  }
  return "unknown zr_status";
}

}  // extern "C"

extern "C" {

zr_status zr_consensus_plan(const zr_config* cfg, const int32_t* seq_lens, const int32_t* prompt_lens,
                            const int32_t* seg_ptr, const int32_t* pair_bounds, const int32_t* topk,
                            const int32_t* consensus, zr_plan_t* out_plan, size_t* workspace_bytes) {
  if (!out_plan || !workspace_bytes) return ZR_EINVAL;
  *out_plan = nullptr;
  *workspace_bytes = 0;
  zr_status st = validate_consensus(cfg, seq_lens, prompt_lens, seg_ptr, pair_bounds, topk, consensus);
  if (st != ZR_OK) return st;
  struct zr_plan* P = new (std::nothrow) struct zr_plan();
  if (!P) return ZR_ENOMEM;
  zr::Plan& p = P->p;
  p.mode = zr::kConsensusPlan;
  p.cfg = *cfg;
  p.B = cfg->batch;
  p.Hq = cfg->num_q_heads;
  p.Hkv = cfg->num_kv_heads;
  p.G = p.Hq / p.Hkv;
  p.d = cfg->head_dim;
  p.window = cfg->window;
  p.num_blocks = cfg->num_blocks;
  p.max_blocks = cfg->max_blocks_per_seq;
  p.total_segments = seg_ptr[p.B];

  // Rows bound per unit: at most min(L, N_p + min(w, L) + the c longest regular segments + every
  // summary segment) tokens (I_c contributes regular segments, I_s summary segments).
  std::vector<int32_t> kclip(p.B), cclip(p.B);
  p.n_max = 1;
  p.c_max = 1;
  int64_t rows_bound = 0;
  for (int b = 0; b < p.B; ++b) {
    const int n = seg_ptr[b + 1] - seg_ptr[b];
    const int32_t* bd = pair_bounds + 2 * static_cast<int64_t>(seg_ptr[b]) + b;
    const int L = seq_lens[b];
    kclip[b] = std::min(topk[b], n);
    cclip[b] = std::min(consensus[b], n);
    p.n_max = std::max(p.n_max, n);
    p.c_max = std::max(p.c_max, cclip[b]);
    std::vector<int32_t> reg(n);
    int64_t sum_s = 0;
    for (int i = 0; i < n; ++i) {
      reg[i] = bd[2 * i + 1] - bd[2 * i];
      sum_s += bd[2 * i + 2] - bd[2 * i + 1];
    }
    std::sort(reg.begin(), reg.end(), std::greater<int32_t>());
    int64_t top = 0;
    for (int i = 0; i < cclip[b]; ++i) top += reg[i];
    const int64_t tok = std::min<int64_t>(L, prompt_lens[b] + std::min<int64_t>(p.window, L) + top + sum_s);
    rows_bound += tok * p.Hkv;
    p.fixed_rows = static_cast<int>(
        std::max<int64_t>(p.fixed_rows, std::min<int64_t>(L, prompt_lens[b] + std::min(p.window, L))));
    p.prompt_rows = std::max(p.prompt_rows, static_cast<int>(prompt_lens[b]));
  }
  p.k_max = p.n_max + 1;  // range capacity per unit: prompt, one piece per pair, window
  if (cudaGetDevice(&p.device) != cudaSuccess) {
    cudaGetLastError();
    delete P;
    return ZR_ECUDA;
  }
  st = zr::configure_kernels(p, (rows_bound + 15) / 16);
  if (st != ZR_OK) {
    delete P;
    return st;
  }
  layout_workspace(p);

  const size_t nb = static_cast<size_t>(p.B);
  const size_t n_bounds = 2 * static_cast<size_t>(p.total_segments) + nb;
  size_t moff = 0;
  auto mtake = [&](size_t count) {
    size_t at = moff;
    moff = align_up(moff + count * sizeof(int32_t), 256);
    return at;
  };
  const size_t o_len = mtake(nb), o_ptr = mtake(nb + 1), o_bnd = mtake(n_bounds), o_topk = mtake(nb),
               o_np = mtake(nb), o_c = mtake(nb);
  void* base = nullptr;
  cudaError_t ce = cudaMalloc(&base, moff);
  if (ce != cudaSuccess) {
    cudaGetLastError();
    delete P;
    return ce == cudaErrorMemoryAllocation ? ZR_ENOMEM : ZR_ECUDA;
  }
  p.d_meta_base = base;
  char* cb = static_cast<char*>(base);
  p.meta.seq_lens = reinterpret_cast<int32_t*>(cb + o_len);
  p.meta.seg_ptr = reinterpret_cast<int32_t*>(cb + o_ptr);
  p.meta.seg_bounds = reinterpret_cast<int32_t*>(cb + o_bnd);
  p.meta.topk = reinterpret_cast<int32_t*>(cb + o_topk);
  p.meta.prompt_lens = reinterpret_cast<int32_t*>(cb + o_np);
  p.meta.consensus = reinterpret_cast<int32_t*>(cb + o_c);
  bool ok = cudaMemcpy(p.meta.seq_lens, seq_lens, nb * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(p.meta.seg_ptr, seg_ptr, (nb + 1) * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(p.meta.seg_bounds, pair_bounds, n_bounds * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(p.meta.topk, kclip.data(), nb * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(p.meta.prompt_lens, prompt_lens, nb * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(p.meta.consensus, cclip.data(), nb * 4, cudaMemcpyHostToDevice) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    cudaFree(base);
    delete P;
    return ZR_ECUDA;
  }
  *out_plan = P;
  *workspace_bytes = p.ws.total;
  return ZR_OK;
}

zr_status zr_consensus_dims(zr_plan_t plan, int32_t* c_max, int32_t* n_max) {
  if (!plan || !c_max || !n_max || plan->p.mode != zr::kConsensusPlan) return ZR_EINVAL;
  *c_max = plan->p.c_max;
  *n_max = plan->p.n_max;
  return ZR_OK;
}

zr_status zr_consensus_vote(zr_plan_t plan, void* workspace, const void* q, const void* mean_keys, void* stream) {
  if (!plan || !workspace || !q || !mean_keys || plan->p.mode != zr::kConsensusPlan) return ZR_EINVAL;
  if (!aligned(workspace, 256) || !aligned(q, 16) || !aligned(mean_keys, 16)) return ZR_EINVAL;
  zr::StepArgs a = zr::step_args(plan->p, workspace);
  a.q = q;
  return zr::launch_vote(plan->p, a, mean_keys,
                         reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + plan->p.ws.votes), stream);
}

zr_status zr_consensus_select(zr_plan_t plan, void* workspace, int32_t* votes_out, int32_t* consensus_out,
                              int32_t* ranges_out, int32_t* nranges_out, void* stream) {
  if (!plan || !workspace || plan->p.mode != zr::kConsensusPlan) return ZR_EINVAL;
  if (!aligned(workspace, 256)) return ZR_EINVAL;
  zr::StepArgs a = zr::step_args(plan->p, workspace);
  a.ranges_out = ranges_out;
  a.nranges_out = nranges_out;
  return zr::launch_consensus(plan->p, a,
                              reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + plan->p.ws.votes),
                              votes_out, consensus_out, stream);
}

namespace {
// True when the device allocation holding p extends at least `bytes` past it (the driver's address-range
// query; false for host memory or when the query is unavailable).
bool spans_bytes(const void* p, size_t bytes) {
  using Fn = int (*)(unsigned long long*, size_t*, unsigned long long);
  static const Fn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return static_cast<Fn>(nullptr);
    }
    return reinterpret_cast<Fn>(f);
  }();
  if (!fn) return false;
  unsigned long long base = 0;
  size_t size = 0;
  const unsigned long long at = reinterpret_cast<unsigned long long>(p);
  if (fn(&base, &size, at) != 0) return false;
  return at >= base && at + bytes <= base + size;
}

// The attend-only calls prefetch the sink or prompt rows before their wait (as the decode step does) only
// when both pools lie in allocations that hold the plan's num_blocks blocks: then even a block table still
// being written by an earlier kernel can only send a prefetch elsewhere inside them. Staging pools of the
// offloaded cache, or pools in host memory, get no prefetch. The window is left out: between selections
// the sequences grow past the plan's lengths (the advance calls), and the prompt does not move.
int prompt_rows_if_full_pools(const zr::Plan& p, const void* k_pool, const void* v_pool) {
  const size_t eb = p.cfg.dtype == ZR_BF16 ? 2 : 4;
  const size_t bytes = static_cast<size_t>(p.num_blocks) * p.Hkv * zr::kBlockTokens * p.d * eb;
  return spans_bytes(k_pool, bytes) && spans_bytes(v_pool, bytes) ? p.prompt_rows : 0;
}

zr_status consensus_attend_into(zr_plan_t plan, void* workspace, const void* q, const void* k_pool,
                                const void* v_pool, const int32_t* block_tables, float* out, void* stream,
                                void* ev_start, void* ev_stop) {
  if (!plan || !workspace || !q || !k_pool || !v_pool || !block_tables || !out) return ZR_EINVAL;
  if (plan->p.mode != zr::kConsensusPlan) return ZR_EINVAL;
  if (!aligned(workspace, 256) || !aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
      !aligned(out, 16) || !aligned(block_tables, 4))
    return ZR_EINVAL;
  zr::StepArgs a = zr::step_args(plan->p, workspace);
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.block_tables = block_tables;
  a.sum_k = k_pool;  // no summary rows are gathered: every unit's summary count is 0
  a.sum_v = v_pool;
  a.out = out;
  a.fixed_rows = prompt_rows_if_full_pools(plan->p, k_pool, v_pool);
  a.fixed_window = 0;
  return zr::launch_attend_only(plan->p, a, stream, ev_start, ev_stop);
}
}  // namespace

zr_status zr_consensus_attend(zr_plan_t plan, void* workspace, const void* q, const void* k_pool,
                              const void* v_pool, const int32_t* block_tables, float* out, void* stream) {
  return consensus_attend_into(plan, workspace, q, k_pool, v_pool, block_tables, out, stream, nullptr, nullptr);
}

zr_status zr_consensus_attend_timed(zr_plan_t plan, void* workspace, const void* q, const void* k_pool,
                                    const void* v_pool, const int32_t* block_tables, float* out, void* ev_start,
                                    void* ev_stop, void* stream) {
  if (!ev_start && !ev_stop) return ZR_EINVAL;
  return consensus_attend_into(plan, workspace, q, k_pool, v_pool, block_tables, out, stream, ev_start, ev_stop);
}

}  // extern "C"

extern "C" {

zr_status zr_decode_advance(zr_plan_t plan, void* workspace, const int32_t* seq_lens, void* stream) {
  if (!plan || !workspace || !seq_lens || plan->p.mode != zr::kDecodePlan) return ZR_EINVAL;
  if (!aligned(workspace, 256) || !aligned(seq_lens, 4)) return ZR_EINVAL;
  return zr::launch_decode_advance(plan->p, zr::step_args(plan->p, workspace), seq_lens, stream);
}

zr_status zr_decode_attend_reuse(zr_plan_t plan, void* workspace, const void* q, const void* k_pool,
                                 const void* v_pool, const int32_t* block_tables, const void* sum_k,
                                 const void* sum_v, float* out, void* stream) {
  if (!plan || !workspace || !q || !k_pool || !v_pool || !block_tables || !sum_k || !sum_v || !out) return ZR_EINVAL;
  if (plan->p.mode != zr::kDecodePlan) return ZR_EINVAL;
  if (!aligned(workspace, 256) || !aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
      !aligned(sum_k, 16) || !aligned(sum_v, 16) || !aligned(out, 16) || !aligned(block_tables, 4))
    return ZR_EINVAL;
  zr::StepArgs a = zr::step_args(plan->p, workspace);
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.block_tables = block_tables;
  a.sum_k = sum_k;
  a.sum_v = sum_v;
  a.out = out;
  a.fixed_rows = prompt_rows_if_full_pools(plan->p, k_pool, v_pool);
  a.fixed_window = 0;
  return zr::launch_attend_only(plan->p, a, stream);
}

zr_status zr_consensus_advance(zr_plan_t plan, void* workspace, const int32_t* seq_lens, void* stream) {
  if (!plan || !workspace || !seq_lens || plan->p.mode != zr::kConsensusPlan) return ZR_EINVAL;
  if (!aligned(workspace, 256) || !aligned(seq_lens, 4)) return ZR_EINVAL;
  return zr::launch_consensus_advance(plan->p, zr::step_args(plan->p, workspace), seq_lens, stream);
}

}  // extern "C"
