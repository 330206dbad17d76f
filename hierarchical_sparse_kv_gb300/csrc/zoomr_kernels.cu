// sm_103a kernels of the ZoomR decode step and their launch sequence.
//
//   select  one CTA per (sequence b, KV head g) unit: scores every segment's
//           summary key (ZoomR page, 3.3 "Per-Head Importance Scoring and
//           Voting"), picks the top-k by rank counting (ties to the lower
//           index), and writes the unit's gathered token ranges (the window
//           merged with the selected segments, 3.3 "Constructing the Final
//           Multi-Granularity Context") and its summary list.
//   attend  one warp per split slot: walks up to kChunkRows gathered rows
//           (tokens through the block table, then summary rows), computes the
//           group's logits and an online softmax, and writes one unnormalised
//           partial (m, l, o) per query head (ZoomR 2 "Background", the
//           softmax(q K^T / sqrt d) V equation; rows fetched as on the
//           "KV-cache management" page, "Paged KV cache (PagedAttention)").
//           bf16: tensor cores (mma.sync m16n8k16) with K/V rows loaded straight
//           from HBM into fragment registers; f32: CUDA-core FMA.
//   merge   one warp per (sequence, query head): log-sum-exp combination of the
//           unit's partials into the fp32 output.
//
// Launches are chained with programmatic dependent launch: every kernel waits
// (griddepcontrol.wait) for its predecessor before it reads what that one writes.
// The attend kernel releases its dependents only after its own wait, so the merge
// kernel may read the select kernel's unit sizes before it waits on the attend.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "zoomr_exact_key.cuh"
#include "zoomr_internal.h"

namespace zr {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kWarpRangesMax = 256;  // segments up to which one warp builds a unit's lists and ranges

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// An L2 prefetch: a hint only (a later load still reads the current value), so kernels issue it for
// their inputs before waiting on the previous kernel, which cannot make it read anything stale.
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }
// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned address) into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Prefetch `bytes` at `base` into L2, one 128-byte line per thread of the grid slice [t0, t0 + nt).
__device__ __forceinline__ void prefetch_span(const void* base, size_t bytes, size_t t, size_t nt) {
  const char* c = static_cast<const char*>(base);
  for (size_t off = t * 128; off < bytes; off += nt * 128) prefetch_l2(c + off);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Load E (= 2 or 4) consecutive elements as floats.
template <typename T, int E>
__device__ __forceinline__ void load_e(const T* p, float (&v)[E]) {
  if constexpr (sizeof(T) == 4) {
    if constexpr (E == 4) {
      const float4 a = *reinterpret_cast<const float4*>(p);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else {
      const float2 a = *reinterpret_cast<const float2*>(p);
      v[0] = a.x; v[1] = a.y;
    }
  } else {
    if constexpr (E == 4) {
      const uint2 a = *reinterpret_cast<const uint2*>(p);
      v[0] = bf16_lo(a.x); v[1] = bf16_hi(a.x); v[2] = bf16_lo(a.y); v[3] = bf16_hi(a.y);
    } else {
      const uint32_t a = *reinterpret_cast<const uint32_t*>(p);
      v[0] = bf16_lo(a); v[1] = bf16_hi(a);
    }
  }
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ int warp_incl_scan(int x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive prefix sum of one int per thread over the CTA; *total receives the sum.
__device__ int block_exclusive_scan(int v, int* total) {
  __shared__ int wsum[32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = lane < nw ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, t, o);
      if (lane >= o) t += y;
    }
    wsum[lane] = t;
  }
  __syncthreads();
  const int base = w > 0 ? wsum[w - 1] : 0;
  *total = wsum[nw - 1];
  __syncthreads();
  return base + x - v;
}

// ------------------------------------------------------------------ select
// One warp: unit u's ranges [0, nr) and prefix sums (global, written by this CTA) gain the sink
// [0, Ns), which lies before every segment: it merges into range 0 if that starts at or before
// Ns, else every range moves up one slot (the plan reserves it) and the sink becomes range 0.
__device__ void add_sink_range(const StepArgs& a, int u, int Ns, int32_t* rg, int32_t* cum, int32_t* rout, int lane) {
  int4 info = a.unit_info[u];
  const int nr = info.x;
  int added;
  if (nr > 0 && rg[0] <= Ns) {
    added = rg[0];
    __syncwarp();
    if (lane == 0) rg[0] = 0;
    for (int r = 1 + lane; r <= nr; r += 32) cum[r] += added;
  } else {
    added = Ns;
    // move ranges and prefix sums up one slot, highest chunk first
    for (int base = (nr / 32) * 32; base >= 0; base -= 32) {
      const int r = base + lane;
      int s_ = 0, e_ = 0, c_ = 0;
      if (r < nr) {
        s_ = rg[2 * r];
        e_ = rg[2 * r + 1];
      }
      if (r <= nr) c_ = cum[r];
      __syncwarp();
      if (r < nr) {
        rg[2 * (r + 1)] = s_;
        rg[2 * (r + 1) + 1] = e_;
      }
      if (r <= nr) cum[r + 1] = c_ + Ns;
      __syncwarp();
    }
    if (lane == 0) {
      rg[0] = 0;
      rg[1] = Ns;
      cum[0] = 0;
    }
    info.x = nr + 1;
  }
  __syncwarp();
  const int nr2 = info.x;
  if (rout)
    for (int r = lane; r < nr2; r += 32) {
      rout[2 * r] = rg[2 * r];
      rout[2 * r + 1] = rg[2 * r + 1];
    }
  if (lane == 0) {
    info.y += added;
    a.unit_info[u] = info;
    a.unit_rows[u] += added;
    if (a.nranges_out) a.nranges_out[u] = nr2;
  }
}

// Once a unit's selection is final, the select CTA's idle warps list for the attend kernel the selected
// segments' blocks among the a.pf_blocks (at most kSelPrefetchBlocks) blocks just before the window
// (entry q of the unit's list: the physical block, or -1). The attend kernel prefetches their K and V tiles into L2 right after its
// wait, while its first row tables are built: it gathers these blocks last, so they have the longest
// time to arrive. (Prefetched by the select kernel itself, they would hold up its completion.)
__device__ void list_selected_tail(const StepArgs& a, int u, int b, int n, int W0, const int* flag, const int* bnd,
                                   int t, int nt) {
  int32_t* list = a.pf_list + static_cast<size_t>(u) * kSelPrefetchBlocks;
  for (int q = t; q < kSelPrefetchBlocks; q += nt) {
    const int j = W0 / kBlockTokens - 1 - q;  // a block wholly before the window, walking back
    int out = -1;
    if (j < 0 || q >= a.pf_blocks) {
      list[q] = out;
      continue;
    }
    const int t0 = j * kBlockTokens, t1 = t0 + kBlockTokens;
    // the segments overlapping [t0, t1): from the last bound <= t0 (bnd ascending, bnd[0] = 0)
    int lo = 0, hi = n;  // invariant: bnd[lo] <= t0 < bnd[hi] (or hi = n)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (bnd[mid] <= t0) lo = mid; else hi = mid;
    }
    bool any = false;
    for (int i = lo; i < n && bnd[i] < t1; ++i) any |= flag[i] != 0;
    if (any) {
      const int phys = a.block_tables[static_cast<size_t>(b) * a.max_blocks + j];
      if (static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks)) out = phys;
    }
    list[q] = out;
  }
}

// Shared memory: the exact-key scorer's query limb tables | the query table [G * D] | key high words
//   [n_max + 4] u64 | key low words [n_max + 4] u64 | flag [n_max + 2] | bounds [n_max + 1] | list [n_max] |
//   runs_s [n_max] | runs_e [n_max] | fp32 enclosures lo, hi [n_max] each
template <typename T, int D>
struct SelectLayout {
  using SC = xk::Scorer<T, D, kSelectThreads>;
  __host__ __device__ static constexpr size_t limb_bytes(int G) { return (SC::smem_bytes(G) + 15) / 16 * 16; }
  __host__ __device__ static constexpr size_t q_bytes(int G) {
    return limb_bytes(G) + sizeof(T) * static_cast<size_t>(G) * D;
  }
  __host__ __device__ static constexpr size_t bytes(int G, int n_max) {
    return q_bytes(G) + 2 * sizeof(uint64_t) * (static_cast<size_t>(n_max) + 4) +
           sizeof(int) * (5 * static_cast<size_t>(n_max) + 3) + 2 * sizeof(float) * static_cast<size_t>(n_max);
  }
};

// 80 registers per thread (no spills): a select CTA then leaves room on its SM for an attend CTA of
// the same layer, which launches early and waits (programmatic dependent launch).
template <typename T, int D>
__global__ void __maxnreg__(80) zr_select_kernel(StepArgs a) {
  using LY = SelectLayout<T, D>;
  using SC = typename LY::SC;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int g = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int u = b * a.Hkv + g;
  const int G = a.G, nmax = a.n_max;
  int* qh = reinterpret_cast<int*>(smem_raw);
  int* ql = qh + G * SC::kQRow;
  int* qtail = ql + G * SC::kQRow;
  uint4* qtab = reinterpret_cast<uint4*>(smem_raw + LY::limb_bytes(G));
  uint64_t* kh = reinterpret_cast<uint64_t*>(smem_raw + LY::q_bytes(G));
  uint64_t* kl = kh + nmax + 4;
  int* flag = reinterpret_cast<int*>(kl + nmax + 4);
  int* bnd = flag + nmax + 2;
  int* list = bnd + nmax + 1;
  int* runs_s = list + nmax;
  int* runs_e = runs_s + nmax;
  float* elo = reinterpret_cast<float*>(runs_e + nmax);
  float* ehi = elo + nmax;
  __shared__ int s_rstar;
  __shared__ int s_flags;
  __shared__ uint32_t s_red[4 * kSelectThreads / 32];
  __shared__ uint32_t s_cert[3 * kSelectThreads / 32];

  pdl_trigger();
  // Plan metadata is never written by a kernel: read it before waiting on the previous kernel.
  const int s0 = a.meta.seg_ptr[b];
  const int n = a.meta.seg_ptr[b + 1] - s0;
  const int L = a.meta.seq_lens[b];
  const int k = a.meta.topk[b];
  const int Ns = a.meta.prompt_lens[b];
  for (int i = tid; i <= n; i += blockDim.x) bnd[i] = a.meta.seg_bounds[s0 + b + i];
  const T* qg = static_cast<const T*>(a.q) + (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G) * D;
  const T* rows = static_cast<const T*>(a.sum_k) + (static_cast<size_t>(s0) * a.Hkv + g) * D;
  const size_t stride = static_cast<size_t>(a.Hkv) * D;
  {
    // the group's queries and the unit's summary-key rows, into L2 before the wait
    constexpr size_t RB = D * sizeof(T);
    if (tid < kSelectThreads / 2) {
      prefetch_span(qg, G * RB, tid, kSelectThreads / 2);
    } else {
      const int rows_pf = min(n, kSelectThreads);
      for (int i = tid - kSelectThreads / 2; i < rows_pf; i += kSelectThreads / 2)
        prefetch_span(rows + i * stride, RB, 0, 1);
    }
  }
  pdl_wait();

  // 1. ranking key: max over the group of the exact dot q_h . s_i. First an fp32 estimate of every key
  //    with an enclosure of the exact value (lane-parallel fused multiply-adds).
  {
    auto emit = [&](int r, int, float mid, float lo, float hi) {
      kh[r] = 0;
      kl[r] = xk::order_bits(mid);
      elo[r] = lo;
      ehi[r] = hi;
    };
    // 16 elements a lane (64 rows a pass), or 32 (128 rows a pass) when that saves a pass
    if (D == 128 && n > xk::EstShape<T, D, kSelectThreads, 16>::kRPP)
      xk::estimate_rows<T, D, kSelectThreads, true, D == 128 ? 32 : 16>(qg, G, qtab, 0, G, rows, stride, n, emit);
    else
      xk::estimate_rows<T, D, kSelectThreads, true, 16>(qg, G, qtab, 0, G, rows, stride, n, emit);
  }
  __syncthreads();

  // 2. top-k: segment i is selected iff fewer than k segments beat it (a greater exact key, or an equal
  //    key and a lower index). The top-k of the estimates is the exact one when its certificate holds
  //    (the enclosures separate at the k boundary); otherwise the uncertain segments' keys are computed
  //    exactly. (certify_top_k and resolve_top_k end with a barrier after the flags are written.)
  float cert_lo, cert_hi;
  if (!xk::certify_top_k<kSelectThreads>(elo, ehi, n, k, kh, kl, flag, s_cert, cert_lo, cert_hi)) {
    const int uflags = xk::resolve_top_k<T, D, kSelectThreads, true>(
        qg, G, 0, G, rows, stride, n, k, elo, ehi, cert_lo, cert_hi, flag, reinterpret_cast<int*>(elo),
        reinterpret_cast<int*>(ehi), kh, kl, qh, ql, qtail, s_red, &s_flags,
        a.bigkeys + static_cast<size_t>(u) * nmax * xk::kBigDigits);
    if ((uflags & xk::kFlagNonFinite) && tid == 0) atomicOr(a.err, kErrNonFinite);
  }

  // 3. the selected list (ascending), the summary list (the rest, ascending), the maximal runs of
  //    selected segments (consecutive segments touch), and the token ranges: the runs merged with
  //    the window [W0, L) -- the first run reaching W0 absorbs it, later runs lie inside it.
  int* sel_ws = a.sel + static_cast<size_t>(u) * a.k_max;
  int* sum_ws = a.sumlist + static_cast<size_t>(u) * a.n_max;
  int* rg = a.ranges + static_cast<size_t>(u) * (a.k_max + 1) * 2;
  int* cum = a.cum + static_cast<size_t>(u) * (a.k_max + 2);
  int* rout = a.ranges_out ? a.ranges_out + static_cast<size_t>(u) * (a.k_max + 1) * 2 : nullptr;
  const int W0 = max(0, L - a.window);
  if (n <= kWarpRangesMax) {
    // Warp 0 alone, 32 segments per pass: compaction and run numbering from ballots, with carries
    // between passes; then the ranges. No CTA barrier: the other warps prefetch and are done.
    if (tid >= 32 && a.pf_blocks > 0) list_selected_tail(a, u, b, n, W0, flag, bnd, tid - 32, blockDim.x - 32);
    if (tid < 32) {
      const int lane = tid;
      const unsigned lt = (1u << lane) - 1u;
      int c_sel = 0, c_run = 0, rstar = 0;
      for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        const bool in = i < n;
        const bool sel = in && flag[i];
        const bool rstart = sel && !(i > 0 && flag[i - 1]);
        const bool rend = sel && !(i + 1 < n && flag[i + 1]);
        const int e_i = in ? bnd[i + 1] : 0;
        const unsigned bs = __ballot_sync(kFull, sel), bst = __ballot_sync(kFull, rstart);
        const unsigned bbe = __ballot_sync(kFull, rend && e_i < W0);
        const int pos = c_sel + __popc(bs & lt);
        if (in) {
          if (sel) {
            list[pos] = i;
            sel_ws[pos] = i;
          } else {
            sum_ws[i - pos] = i;
          }
        }
        if (rstart) runs_s[c_run + __popc(bst & lt)] = bnd[i];
        if (rend) runs_e[c_run + __popc(bst & (lt | (1u << lane))) - 1] = e_i;
        c_sel += __popc(bs);
        c_run += __popc(bst);
        rstar += __popc(bbe);
      }
      __syncwarp();  // runs_s / runs_e are complete
      const int m = c_run;  // runs; rstar of them end before W0
      const int nr = rstar < m ? rstar + 1 : m + (W0 < L ? 1 : 0);
      int carry = 0;
      for (int r0 = 0; r0 < nr; r0 += 32) {
        const int r = r0 + lane;
        int s_ = 0, e_ = 0;
        if (r < nr) {
          if (r < rstar) {
            s_ = runs_s[r];
            e_ = runs_e[r];
          } else {
            s_ = rstar < m ? min(W0, runs_s[rstar]) : W0;
            e_ = L;
          }
        }
        const int len = e_ - s_;
        const int incl = warp_incl_scan(len, lane);
        if (r < nr) {
          rg[2 * r] = s_;
          rg[2 * r + 1] = e_;
          cum[r] = carry + incl - len;
          if (rout) {
            rout[2 * r] = s_;
            rout[2 * r + 1] = e_;
          }
        }
        carry += __shfl_sync(kFull, incl, 31);
      }
      if (lane == 0) {
        cum[nr] = carry;
        a.unit_info[u] = make_int4(nr, carry, n - k, 0);
        a.unit_rows[u] = carry + n - k;
        if (a.nranges_out) a.nranges_out[u] = nr;
      }
    }
  } else if (n <= kSelectThreads) {
    // One thread per segment: compaction and run numbering from warp ballots.
    __shared__ int s_cnt[3][kSelectThreads / 32];
    const int lane = tid & 31, wi = tid >> 5, nwarps = blockDim.x >> 5;
    const bool in = tid < n;
    const bool sel = in && flag[tid];
    const bool rstart = sel && !(tid > 0 && flag[tid - 1]);
    const bool rend = sel && !(tid + 1 < n && flag[tid + 1]);
    const int e_i = in ? bnd[tid + 1] : 0;
    const unsigned bs = __ballot_sync(kFull, sel), bst = __ballot_sync(kFull, rstart);
    const unsigned bbe = __ballot_sync(kFull, rend && e_i < W0);
    if (lane == 0) {
      s_cnt[0][wi] = __popc(bs);
      s_cnt[1][wi] = __popc(bst);
      s_cnt[2][wi] = __popc(bbe);
    }
    __syncthreads();
    // every warp scans the per-warp counts itself: lane w holds warp w's (nwarps <= 32)
    const int c0w = lane < nwarps ? s_cnt[0][lane] : 0, c1w = lane < nwarps ? s_cnt[1][lane] : 0;
    const int c2w = lane < nwarps ? s_cnt[2][lane] : 0;
    const int i0 = warp_incl_scan(c0w, lane), i1 = warp_incl_scan(c1w, lane), i2 = warp_incl_scan(c2w, lane);
    const int off_s = wi > 0 ? __shfl_sync(kFull, i0, wi - 1) : 0;
    const int off_r = wi > 0 ? __shfl_sync(kFull, i1, wi - 1) : 0;
    const int m = __shfl_sync(kFull, i1, 31), rstar = __shfl_sync(kFull, i2, 31);  // rstar: runs ending before W0
    const unsigned lt = (1u << lane) - 1u;
    const int pos = off_s + __popc(bs & lt);
    if (in) {
      if (sel) {
        list[pos] = tid;
        sel_ws[pos] = tid;
      } else {
        sum_ws[tid - pos] = tid;
      }
    }
    if (rstart) runs_s[off_r + __popc(bst & lt)] = bnd[tid];
    if (rend) runs_e[off_r + __popc(bst & (lt | (1u << lane))) - 1] = e_i;
    __syncthreads();
    const int nr = rstar < m ? rstar + 1 : m + (W0 < L ? 1 : 0);
    if (wi == 0) {
      int carry = 0;
      for (int r0 = 0; r0 < nr; r0 += 32) {
        const int r = r0 + lane;
        int s_ = 0, e_ = 0;
        if (r < nr) {
          if (r < rstar) {
            s_ = runs_s[r];
            e_ = runs_e[r];
          } else {
            s_ = rstar < m ? min(W0, runs_s[rstar]) : W0;
            e_ = L;
          }
        }
        const int len = e_ - s_;
        const int incl = warp_incl_scan(len, lane);
        if (r < nr) {
          rg[2 * r] = s_;
          rg[2 * r + 1] = e_;
          cum[r] = carry + incl - len;
          if (rout) {
            rout[2 * r] = s_;
            rout[2 * r + 1] = e_;
          }
        }
        carry += __shfl_sync(kFull, incl, 31);
      }
      if (lane == 0) {
        cum[nr] = carry;
        a.unit_info[u] = make_int4(nr, carry, n - k, 0);
        a.unit_rows[u] = carry + n - k;
        if (a.nranges_out) a.nranges_out[u] = nr;
      }
    }
  } else {
    // Any n: block-wide scans over contiguous per-thread slices. (No prefetch list here: the flags are
    // reused as scratch below.)
    if (a.pf_blocks > 0)
      for (int q = tid; q < kSelPrefetchBlocks; q += blockDim.x)
        a.pf_list[static_cast<size_t>(u) * kSelPrefetchBlocks + q] = -1;
    {
      const int per = (n + blockDim.x - 1) / blockDim.x;
      const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
      int local = 0;
      for (int i = i0; i < i1; ++i) local += flag[i];
      int total;
      int pos = block_exclusive_scan(local, &total);
      for (int i = i0; i < i1; ++i) {
        if (flag[i]) {
          list[pos] = i;
          sel_ws[pos] = i;
          ++pos;
        } else {
          sum_ws[i - pos] = i;
        }
      }
    }
    __syncthreads();
    int m;
    {
      const int per = (k + blockDim.x - 1) / blockDim.x;
      const int j0 = min(k, tid * per), j1 = min(k, j0 + per);
      int starts = 0;
      for (int j = j0; j < j1; ++j) starts += (j == 0) || (bnd[list[j - 1] + 1] != bnd[list[j]]);
      int ridx = block_exclusive_scan(starts, &m) - 1;
      for (int j = j0; j < j1; ++j) {
        const int seg = list[j];
        if ((j == 0) || (bnd[list[j - 1] + 1] != bnd[seg])) runs_s[++ridx] = bnd[seg];
        if ((j == k - 1) || (bnd[list[j + 1]] != bnd[seg + 1])) runs_e[ridx] = bnd[seg + 1];
      }
    }
    if (tid == 0) s_rstar = m;
    __syncthreads();
    for (int r = tid; r < m; r += blockDim.x)
      if (runs_e[r] >= W0 && (r == 0 || runs_e[r - 1] < W0)) s_rstar = r;
    __syncthreads();
    const int rstar = s_rstar;
    const int nr = rstar < m ? rstar + 1 : m + (W0 < L ? 1 : 0);
    int* lens = flag;  // flags are no longer needed
    for (int r = tid; r < nr; r += blockDim.x) {
      int s_, e_;
      if (r < rstar) {
        s_ = runs_s[r];
        e_ = runs_e[r];
      } else if (rstar < m) {
        s_ = min(W0, runs_s[rstar]);
        e_ = L;
      } else {
        s_ = W0;
        e_ = L;
      }
      rg[2 * r] = s_;
      rg[2 * r + 1] = e_;
      lens[r] = e_ - s_;
      if (rout) {
        rout[2 * r] = s_;
        rout[2 * r + 1] = e_;
      }
    }
    __syncthreads();
    int n_tok;
    {
      const int per = (nr + blockDim.x - 1) / blockDim.x;
      const int r0 = min(nr, tid * per), r1 = min(nr, r0 + per);
      int local = 0;
      for (int r = r0; r < r1; ++r) local += lens[r];
      int run = block_exclusive_scan(local, &n_tok);
      for (int r = r0; r < r1; ++r) {
        cum[r] = run;
        run += lens[r];
      }
    }
    if (tid == 0) {
      cum[nr] = n_tok;
      a.unit_info[u] = make_int4(nr, n_tok, n - k, 0);
      a.unit_rows[u] = n_tok + n - k;
      if (a.nranges_out) a.nranges_out[u] = nr;
    }
  }
  // 4. the prompt kept as an attention sink (sequences planned with one): [0, Ns) joins the token
  //    ranges -- merged into the first range when that one starts at or before Ns (the first
  //    segment, which begins at Ns, is selected, or the window reaches the prompt), else prepended.
  if (Ns > 0) {
    __syncthreads();  // this CTA's ranges, prefix sums and unit sizes are written
    if (tid < 32) add_sink_range(a, u, Ns, rg, cum, rout, tid);
  }
  if (a.sel_out) {
    __syncthreads();  // list is complete (on the one-warp path warp 0 alone wrote it)
    int* so = a.sel_out + static_cast<size_t>(u) * a.k_max;
    for (int j = tid; j < a.k_max; j += blockDim.x) so[j] = j < k ? list[j] : -1;
  }
}

// ------------------------------------------------------------------ attend: shared pieces
// The rows every unit gathers (its tokens through the block table, then its summary rows) are
// laid end to end in unit order, each unit preceded by a fixed start cost (below), C in all, and
// the attend grid's warps split that evenly: warp w takes [w*C/N, (w+1)*C/N) with N = min(warps,
// C), so every warp streams about the same number of bytes whatever the units' sizes. A warp
// writes one partial per unit whose rows its share touches, into slot u + w: the (unit, warp)
// pairs that intersect form a monotone staircase, so u + w is unique and the slots never exceed
// U + N.

__device__ __forceinline__ int unit_rows(const StepArgs& a, int u) { return a.unit_rows[u]; }

// Every attend warp needs the unit sizes to find its rows. Up to kStagedUnits of them are read
// once per CTA into shared memory (all threads, one round trip) rather than once per warp: the
// grid's warps would otherwise all hit the same few L2 lines at the same moment.
constexpr int kStagedUnits = 256;
struct UnitRows {
  const int32_t* p;  // shared copy, or the workspace array
  __device__ __forceinline__ int operator()(int u) const { return p[u]; }
};
__device__ __forceinline__ UnitRows stage_unit_rows(const StepArgs& a, int32_t* s_rows) {
  const int U = a.B * a.Hkv;
  if (U > kStagedUnits) return UnitRows{a.unit_rows};
  for (int i = threadIdx.x; i < U; i += blockDim.x) s_rows[i] = a.unit_rows[i];
  __syncthreads();
  return UnitRows{s_rows};
}

// The split runs over a cost coordinate: unit u costs a.unit_cost + its rows, the start cost first
// (a virtual stretch that holds no row). A warp whose share reaches into a second unit pays a
// second start (query fragments, two table round trips, a pipeline refill), measured at about 3 us
// on GB300 for decode units: such warps were the last to finish. The virtual stretch takes rows off
// their shares.

struct WarpRange {
  long long s, e;  // this warp's share [s, e) of the cost coordinate
  long long R;     // cost of all units
  long long N;     // warps that get a share
  int u;           // unit whose cost stretch contains s
  long long P;     // cost position where unit u starts (its rows start at P + a.unit_cost)
  int Ru;          // rows of unit u
};

// This warp's share of the cost coordinate and the unit where it starts; false when it gets none.
__device__ bool locate_range(const StepArgs& a, const UnitRows& rows, int w, int nwarps, int lane, WarpRange& wr) {
  const int U = a.B * a.Hkv;
  constexpr int K = 8;  // units kept in registers per lane: one memory round trip when U <= 256
  const bool fast = U <= 32 * K;
  int v[K];
  long long tot = 0;
  if (fast) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int u = 32 * k + lane;
      v[k] = u < U ? rows(u) : 0;
      tot += u < U ? v[k] + a.unit_cost : 0;
    }
  } else {
    for (int u = lane; u < U; u += 32) tot += rows(u) + a.unit_cost;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(kFull, tot, o);
  wr.R = tot;
  wr.N = min(static_cast<long long>(nwarps), tot);
  if (w >= wr.N) return false;
  wr.s = static_cast<long long>(w) * tot / wr.N;
  wr.e = static_cast<long long>(w + 1) * tot / wr.N;
  long long carry = 0;
  auto found = [&](int base, int r, int incl) {
    const unsigned m = __ballot_sync(kFull, carry + incl > wr.s);
    const int l = __ffs(m) - 1;
    wr.u = base + l;
    wr.Ru = __shfl_sync(kFull, r, l);
    wr.P = carry + __shfl_sync(kFull, incl, l) - (wr.Ru + a.unit_cost);
  };
  if (fast) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (32 * k < U) {
        const int c = 32 * k + lane < U ? v[k] + a.unit_cost : 0;
        const int incl = warp_incl_scan(c, lane);
        const int ctot = __shfl_sync(kFull, incl, 31);
        if (carry + ctot > wr.s) {
          found(32 * k, v[k], incl);
          return true;
        }
        carry += ctot;
      }
    }
  } else {
    for (int base = 0; base < U; base += 32) {
      const int r = base + lane < U ? rows(base + lane) : 0;
      const int incl = warp_incl_scan(base + lane < U ? r + a.unit_cost : 0, lane);
      const int ctot = __shfl_sync(kFull, incl, 31);
      if (carry + ctot > wr.s) {
        found(base, r, incl);
        return true;
      }
      carry += ctot;
    }
  }
  return false;  // not reached: position s < R lies in some unit
}

// Fill tab[0, kChunkRows) for the unit-local rows [r0, r0 + n) of unit u: the pool row id
// ((block * Hkv + g) * 16 + slot) of each gathered token, then (summary row id | flag) for the
// summary rows, kInvalidRow past n or for a block id outside the pool. Lane l owns entries
// l, l + 32, ...; the token ranges are walked 32 at a time, each lane holding one.
__device__ void build_row_table(const StepArgs& a, int b, int g, int u, int4 info, int r0, int n, uint32_t* tab,
                                int lane) {
  const int nr = info.x, n_tok = info.y;
  const int32_t* rg = a.ranges + static_cast<size_t>(u) * (a.k_max + 1) * 2;
  const int32_t* cum = a.cum + static_cast<size_t>(u) * (a.k_max + 2);
  const int32_t* sl = a.sumlist + static_cast<size_t>(u) * a.n_max;
  const int32_t* bt = a.block_tables + static_cast<size_t>(b) * a.max_blocks;
  const int seg0 = a.meta.seg_ptr[b];
  // The first 32 ranges' bounds are read before anything uses `info` (whatever nr is, they lie
  // within the unit's arrays; masked below), so this load overlaps the caller's load of `info`.
  const bool in0 = lane <= a.k_max;
  const int cs0 = in0 ? cum[lane] : 0, ce0 = in0 ? cum[lane + 1] : 0, st0 = in0 ? rg[2 * lane] : 0;
  __syncwarp();  // the previous table's readers are done
  for (int e = lane; e < kChunkRows; e += 32) tab[e] = kInvalidRow;
  const int tok_end = min(r0 + n, n_tok);
  for (int base = 0; base < nr && r0 < tok_end; base += 32) {
    const int i = base + lane;
    int cs_raw = cs0, ce_raw = ce0, st_raw = st0;
    if (base > 0) {
      const bool in_region = i <= a.k_max;
      cs_raw = in_region ? cum[i] : 0;
      ce_raw = in_region ? cum[i + 1] : 0;
      st_raw = in_region ? rg[2 * i] : 0;
    }
    const int cs = i < nr ? cs_raw : 0x7fffffff;
    const int ce = i < nr ? ce_raw : 0x7fffffff;
    const int st = i < nr ? st_raw : 0;
    unsigned m = __ballot_sync(kFull, i < nr && ce > r0 && cs < tok_end);
    while (m) {
      const int l = __ffs(m) - 1;
      m &= m - 1;
      const int rcs = __shfl_sync(kFull, cs, l), rce = __shfl_sync(kFull, ce, l), rst = __shfl_sync(kFull, st, l);
      const int e0 = max(rcs, r0) - r0, e1 = min(rce, tok_end) - r0;
      for (int e = e0 + ((lane - e0) & 31); e < e1; e += 32) {
        const int t = rst + (r0 + e - rcs);
        const int phys = bt[t >> 4];
        if (static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks)) {
          tab[e] = ((static_cast<uint32_t>(phys) * a.Hkv + g) << 4) | static_cast<uint32_t>(t & 15);
        } else {
          atomicOr(a.err, kErrBadBlock);
        }
      }
    }
    if (__shfl_sync(kFull, ce, 31) >= tok_end) break;  // the last range of this window reaches the end
  }
  for (int e = max(n_tok - r0, 0) + ((lane - max(n_tok - r0, 0)) & 31); e < n; e += 32) {
    const int seg = sl[r0 + e - n_tok];
    tab[e] = (static_cast<uint32_t>(seg0 + seg) * a.Hkv + g) | kSummaryFlag;
  }
  __syncwarp();
}

// Before its wait on the select kernel an attend CTA prefetches its slice of the block tables and
// of the queries (inputs, not written by the select kernel) into L2.
__device__ __forceinline__ void prefetch_attend_inputs(const StepArgs& a, size_t q_row_bytes) {
  const size_t t = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t nt = static_cast<size_t>(gridDim.x) * blockDim.x;
  prefetch_span(a.block_tables, static_cast<size_t>(a.B) * a.max_blocks * sizeof(int32_t), t, nt);
  prefetch_span(a.q, static_cast<size_t>(a.B) * a.Hq * q_row_bytes, t, nt);
}

// Before its wait an attend CTA also prefetches into L2 its slice of the K and V rows that every unit
// gathers whatever the selection decides: the sink or prompt [0, Ns) and the window [L - w, L) of each
// sequence, every KV head (one bulk prefetch per row). The memory system is otherwise idle while the
// select kernel runs, and these rows then come from L2 in the streaming phase. A prefetch moves no data
// the kernel uses: a block table still being written by an earlier kernel can only misdirect it (block
// ids are range-checked, so every address lies inside the pools).
__device__ void prefetch_fixed_rows(const StepArgs& a, uint32_t row_bytes) {
  const int F = a.fixed_rows, H = a.Hkv;
  const long long total = static_cast<long long>(a.B) * F * H;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(i / (static_cast<long long>(F) * H));
    const int r = static_cast<int>(i % (static_cast<long long>(F) * H));
    const int j = r / H, g = r - (r / H) * H;  // the j-th fixed token of b, KV head g
    const int L = a.meta.seq_lens[b], Ns = a.meta.prompt_lens[b];
    const int Wb = min(a.window, L);
    int t;
    if (j < Ns) {
      t = j;
    } else {
      if (!a.fixed_window) continue;
      t = L - Wb + (j - Ns);
      if (t >= L || t < Ns) continue;  // past the window, or a window token inside the prompt
    }
    const int phys = a.block_tables[static_cast<size_t>(b) * a.max_blocks + (t >> 4)];
    if (static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks)) continue;
    const size_t off = ((static_cast<size_t>(phys) * H + g) * kBlockTokens + (t & 15)) * row_bytes;
    prefetch_l2_bulk(static_cast<const char*>(a.k_pool) + off, row_bytes);
    prefetch_l2_bulk(static_cast<const char*>(a.v_pool) + off, row_bytes);
  }
}

// Right after its wait an attend CTA prefetches into L2 its slice of the select kernel's lists (the
// selected blocks just before each unit's window; see list_selected_tail): one bulk prefetch per K and V
// tile of a listed block, overlapping the round trips of the first row tables.
__device__ void prefetch_selected_lists(const StepArgs& a, uint32_t tile_bytes) {
  const int total = a.B * a.Hkv * kSelPrefetchBlocks;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int phys = a.pf_list[i];
    if (static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks)) continue;
    const int g = (i / kSelPrefetchBlocks) % a.Hkv;  // unit u = b * Hkv + g
    const size_t off = (static_cast<size_t>(phys) * a.Hkv + g) * tile_bytes;
    prefetch_l2_bulk(static_cast<const char*>(a.k_pool) + off, tile_bytes);
    prefetch_l2_bulk(static_cast<const char*>(a.v_pool) + off, tile_bytes);
  }
}

// One warp's walk over its rows: for every unit its range touches, begin_unit, run over row
// tables of up to kChunkRows rows, and end_unit into slot u + w.
template <class Worker>
__device__ void attend_balanced(const StepArgs& a, const UnitRows& rows, Worker& wk, uint32_t* tab, int warp,
                                int lane) {
  const int w = blockIdx.x * kAttendWarps + warp;
  WarpRange wr;
  if (!locate_range(a, rows, w, a.attend_warps, lane, wr)) return;
  int u = wr.u;
  long long P = wr.P;
  int Ru = wr.Ru;
  while (true) {
    // unit u's rows occupy [P + a.unit_cost, P + a.unit_cost + Ru) of the cost coordinate
    const long long first = P + a.unit_cost;
    const int lo = static_cast<int>(min(max(wr.s - first, 0LL), static_cast<long long>(Ru)));
    const int hi = static_cast<int>(min(max(wr.e - first, 0LL), static_cast<long long>(Ru)));
    if (lo < hi) {
      const int b = u / a.Hkv, g = u - b * a.Hkv;
      const int4 info = a.unit_info[u];
      wk.begin_unit(a, b, g, lane);
      for (int r0 = lo; r0 < hi; r0 += kChunkRows) {
        const int nrow = min(kChunkRows, hi - r0);
        build_row_table(a, b, g, u, info, r0, nrow, tab, lane);
        wk.run(a, tab, nrow, lane);
      }
      wk.end_unit(a, u + w, lane);
    }
    if (first + Ru >= wr.e) break;
    P = first + Ru;
    ++u;
    Ru = rows(u);
  }
}

template <typename T, int D>
__device__ __forceinline__ const T* row_ptr(uint32_t id, const T* pool, const T* sum) {
  return (id & kSummaryFlag) ? sum + static_cast<size_t>(id & ~kSummaryFlag) * D : pool + static_cast<size_t>(id) * D;
}

// ------------------------------------------------------------------ attend: tensor cores (bf16, G <= 8)
//
// A warp owns one split (up to kChunkRows gathered rows of one unit) and walks it in 16-row
// tiles through a ring of kStages shared-memory stages filled by cp.async:
//   staging   each warp-wide cp.async moves whole rows (D/8 consecutive lanes per row), so
//             every request reads full 128-byte lines; rows sit row-major with a 16-byte pad,
//             which makes every ldmatrix below conflict-free. Masked rows use the zero-fill
//             form (source size 0) and read nothing.
//   S = Q K^T  mma.sync m16n8k16 bf16 with M = query heads (G valid of 16), N = 8 tokens
//             (two n-tiles), K = d; K^T's B fragments come from ldmatrix.x4.
//   P         thread (r = lane/4, c = lane%4) holds S[head r][tokens 2c, 2c+1, 2c+8, 2c+9],
//             which is exactly the B fragment of P^T for the next product. P is split into
//             bf16 hi + lo parts (two MMAs) so it keeps ~16 bits.
//   O^T += V^T P^T  with M = d (D/16 m-tiles), N = heads, K = 16 tokens; V^T's A fragments
//             come from ldmatrix.x4.trans of the V rows.
// The online softmax runs in log2 units (scale log2(e)/sqrt(d)); O is rescaled only when some
// head's running maximum moved in this tile.
#ifndef ZR_ATTEND_STAGES
#define ZR_ATTEND_STAGES 2
#endif
constexpr int kStages = ZR_ATTEND_STAGES;  // 2: one tile in flight while one is computed, 3 CTAs / SM

template <int D>
__host__ __device__ constexpr int ring_row_bytes() {
  return D * 2 + 16;
}
template <int D>
constexpr size_t attend_ring_bytes() {
  return static_cast<size_t>(kAttendWarps) * kStages * 32 * ring_row_bytes<D>();
}

__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gsrc, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_dst), "l"(gsrc), "r"(src_bytes) : "memory");
}
// The same copy with an L2 eviction policy (createpolicy): the streamed K/V rows are read once per
// layer, so they are marked to leave L2 first, and the kernels' code, the metadata and the partials
// of the step stay resident.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void cp_async16_stream(uint32_t smem_dst, const void* gsrc, uint32_t src_bytes,
                                                  uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(smem_dst), "l"(gsrc),
               "r"(src_bytes), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// Per-lane source bases: the K/V pools and summary tensors, offset by this lane's 16-byte chunk.
struct LoadBases {
  const char* kp;
  const char* vp;
  const char* sk;
  const char* sv;
  uint64_t pol;  // L2 policy of the pool rows (evict first)
};

// Stage the 16 K rows and 16 V rows of tile t0. Every cp.async instruction moves whole rows
// (D/8 consecutive lanes per row, 16 bytes each), so each warp-wide copy reads full 128-byte
// lines: one row id serves both the K and the V copy of a row.
template <int D>
__device__ __forceinline__ void mma_issue_tile(uint32_t stage, const uint32_t* tab, int t0, int lane,
                                               const LoadBases& lb) {
  constexpr int RB = ring_row_bytes<D>();
  constexpr int CPR = D / 8;     // 16-byte chunks per row
  constexpr int RPI = 32 / CPR;  // rows per warp instruction
  const int sub = lane / CPR, ch = lane % CPR;
#pragma unroll
  for (int j = 0; j < 16 / RPI; ++j) {
    const int row = RPI * j + sub;
    const uint32_t id = tab[t0 + row];
    const bool ok = id != kInvalidRow;
    const bool is_sum = (id & kSummaryFlag) != 0;
    const size_t off = static_cast<size_t>(ok ? (id & ~kSummaryFlag) : 0u) * (D * 2);
    const uint32_t bytes = ok ? 16u : 0u;
    const uint32_t dst = stage + row * RB + ch * 16;
    cp_async16_stream(dst, (is_sum ? lb.sk : lb.kp) + off, bytes, lb.pol);
    cp_async16_stream(dst + 16 * RB, (is_sum ? lb.sv : lb.vp) + off, bytes, lb.pol);
  }
}

// The same copies with the pool and summary bases read from the kernel parameters at every issue
// (constant-bank operands) instead of registers: the dynamic split keeps more state live.
template <int D>
__device__ __forceinline__ void mma_issue_tile_p(uint32_t stage, const uint32_t* tab, int t0, int lane,
                                                 const StepArgs& a) {
  constexpr int RB = ring_row_bytes<D>();
  constexpr int CPR = D / 8;
  constexpr int RPI = 32 / CPR;
  const int sub = lane / CPR, ch = lane % CPR;
  const uint64_t pol = l2_evict_first_policy();
#pragma unroll
  for (int j = 0; j < 16 / RPI; ++j) {
    const int row = RPI * j + sub;
    const uint32_t id = tab[t0 + row];
    const bool ok = id != kInvalidRow;
    const bool is_sum = (id & kSummaryFlag) != 0;
    const size_t off = static_cast<size_t>(ok ? (id & ~kSummaryFlag) : 0u) * (D * 2) + ch * 16;
    const uint32_t bytes = ok ? 16u : 0u;
    const uint32_t dst = stage + row * RB + ch * 16;
    cp_async16_stream(dst, static_cast<const char*>(is_sum ? a.sum_k : a.k_pool) + off, bytes, pol);
    cp_async16_stream(dst + 16 * RB, static_cast<const char*>(is_sum ? a.sum_v : a.v_pool) + off, bytes, pol);
  }
}

template <int D>
struct MmaState {
  uint32_t qa0[D / 16], qa2[D / 16];  // Q A-fragments (rows r < G); rows r+8 are zero
  float o[D / 16][4];                  // O^T accumulators
  float m;                             // running max (log2 units) of head r
  float l;                             // this thread's part of head r's running sum
};

template <int D>
__device__ __forceinline__ void mma_compute_tile(MmaState<D>& st, uint32_t stage, uint32_t vmask16, float scale_log2,
                                                 int lane) {
  constexpr int RB = ring_row_bytes<D>();
  const int c = lane & 3;
  const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: this lane addresses row mr of matrix mi
  const uint32_t krow = stage + (8 * (mi >> 1) + mr) * RB + 16 * (mi & 1);
  const uint32_t vrow = krow + 16 * RB;
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    uint32_t b00, b01, b10, b11;
    ldsm_x4(krow + 32 * s, b00, b01, b10, b11);
    mma_bf16(s0, st.qa0[s], 0u, st.qa2[s], 0u, b00, b01);
    mma_bf16(s1, st.qa0[s], 0u, st.qa2[s], 0u, b10, b11);
  }
  const float ninf = -INFINITY;
  const float x0 = (vmask16 >> (2 * c)) & 1u ? s0[0] * scale_log2 : ninf;
  const float x1 = (vmask16 >> (2 * c + 1)) & 1u ? s0[1] * scale_log2 : ninf;
  const float x2 = (vmask16 >> (2 * c + 8)) & 1u ? s1[0] * scale_log2 : ninf;
  const float x3 = (vmask16 >> (2 * c + 9)) & 1u ? s1[1] * scale_log2 : ninf;
  float mt = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
  mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 1));
  mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 2));
  const float m_new = fmaxf(st.m, mt);
  const bool moved = m_new != st.m;
  const float alpha = fast_exp2(st.m - m_new);
  const float p0 = fast_exp2(x0 - m_new), p1 = fast_exp2(x1 - m_new);
  const float p2 = fast_exp2(x2 - m_new), p3 = fast_exp2(x3 - m_new);
  st.l = st.l * alpha + ((p0 + p1) + (p2 + p3));
  st.m = m_new;
  const uint32_t bh0 = pack_bf16(p0, p1), bh1 = pack_bf16(p2, p3);
  const uint32_t bl0 = pack_bf16(p0 - bf16_lo(bh0), p1 - bf16_hi(bh0));
  const uint32_t bl1 = pack_bf16(p2 - bf16_lo(bh1), p3 - bf16_hi(bh1));
  if (__any_sync(kFull, moved)) {
    // O^T columns of this thread are heads 2c and 2c+1, whose alphas live in lanes 8c and 8c+4.
    const float a_e = __shfl_sync(kFull, alpha, 8 * c);
    const float a_o = __shfl_sync(kFull, alpha, 8 * c + 4);
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      st.o[i][0] *= a_e;
      st.o[i][1] *= a_o;
      st.o[i][2] *= a_e;
      st.o[i][3] *= a_o;
    }
  }
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4_trans(vrow + 32 * i, a0, a1, a2, a3);
    mma_bf16(st.o[i], a0, a1, a2, a3, bh0, bh1);
    mma_bf16(st.o[i], a0, a1, a2, a3, bl0, bl1);
  }
}

template <int D>
struct MmaWorker {
  static constexpr uint32_t kStageBytes = 32 * ring_row_bytes<D>();
  MmaState<D> st;
  uint32_t ring;  // this warp's ring (shared-space address)
  LoadBases lb;

  __device__ void begin_unit(const StepArgs& a, int b, int g, int lane) {
    const int r = lane >> 2, c = lane & 3, G = a.G;
    const __nv_bfloat16* qg =
        static_cast<const __nv_bfloat16*>(a.q) + (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G) * D;
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      if (r < G) {
        st.qa0[k] = *reinterpret_cast<const uint32_t*>(qg + r * D + 16 * k + 2 * c);
        st.qa2[k] = *reinterpret_cast<const uint32_t*>(qg + r * D + 16 * k + 2 * c + 8);
      } else {
        st.qa0[k] = 0u;
        st.qa2[k] = 0u;
      }
    }
#pragma unroll
    for (int i = 0; i < D / 16; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.f;
    st.m = -1e30f;
    st.l = 0.f;
  }

  __device__ void run(const StepArgs& a, const uint32_t* tab, int nrows, int lane) {
    const int ntiles = (nrows + 15) >> 4;
    __syncwarp();  // no lane still reads a stage that the prologue refills
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) {
      if (i < ntiles) mma_issue_tile<D>(ring + i * kStageBytes, tab, 16 * i, lane, lb);
      cp_async_commit();
    }
    for (int i = 0; i < ntiles; ++i) {
      const int nx = i + kStages - 1;
      __syncwarp();  // every lane is done reading the stage that is refilled next
      if (nx < ntiles) mma_issue_tile<D>(ring + (nx % kStages) * kStageBytes, tab, 16 * nx, lane, lb);
      cp_async_commit();
      cp_async_wait<kStages - 1>();
      __syncwarp();  // tile i's rows, staged by all lanes, are visible to every lane
      const uint32_t vmask16 = __ballot_sync(kFull, lane < 16 && tab[16 * i + lane] != kInvalidRow) & 0xFFFFu;
      mma_compute_tile<D>(st, ring + (i % kStages) * kStageBytes, vmask16, a.scale_log2, lane);
    }
  }

  __device__ void end_unit(const StepArgs& a, int slot, int lane) {
    const int r = lane >> 2, c = lane & 3, G = a.G;
    // head r's sum: add the parts of the four lanes that share r.
    float l = st.l;
    l += __shfl_xor_sync(kFull, l, 1);
    l += __shfl_xor_sync(kFull, l, 2);
    if (c == 0 && r < G) a.part_ml[static_cast<size_t>(slot) * G + r] = make_float2(st.m, l);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = 2 * c + e;
      if (h < G) {
        float* dst = a.part_o + (static_cast<size_t>(slot) * G + h) * D + r;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
          dst[16 * i] = st.o[i][e];
          dst[16 * i + 8] = st.o[i][e + 2];
        }
      }
    }
  }
};

// ------------------------------------------------------------------ attend: dynamic split
//
// With a fixed even split every warp streams the same number of rows, and the grid ends with its
// slowest warp: SMs that stream more slowly, CTAs that start late behind the previous kernel and rows
// that miss L2 all lengthen one warp's share, and the last warps finish several microseconds after
// the median one. The dynamic split keeps which warps serve which unit (the home warps of a unit are
// the warps whose share of the cost coordinate meets its rows, so partial slot u + p and the merge are
// unchanged) but hands the unit's rows out in batches of 32 from a counter per unit, so all home
// warps of a unit keep streaming until its rows run out. Warp positions along the cost coordinate are
// taken warp-major over the grid (p = warp * ctas + cta), which spreads a unit's home warps over
// many SMs. The attend-only calls use it: there the previous layer's merge and attend kernels still
// hold SMs when the CTAs launch, and measured CTA entry times spread over up to 15 us. (The decode
// step, whose CTAs are all resident while the select kernel runs, keeps the even split.)
//
// Batches are handed out in row order: the attend-only calls prefetch the prompt, the first rows of
// every unit, into L2 before their wait, and the first claims find those rows there.
//
// Per warp the batches flow through three stages, each one batch ahead of the next: the claim of a
// batch (an atomic add), the loads that resolve its 32 row ids (one row per lane: a block-table entry
// or a summary index), and the cp.async copies of its tiles into the 2-stage ring. A batch has two
// 16-row tiles (one for a unit's final batch of at most 16 rows). On the last tile of batch n the warp
// writes batch n+1's table from the ids loaded a batch earlier and issues its first tile, then
// resolves the claim of batch n+2 (issued a batch earlier), starts loading its ids and claims again:
// the round trips of the claims and the id loads overlap a whole batch of copies, and the ring never
// drains between batches.
//
// Every home warp claims until its first failing claim (a value >= the unit's batch count T), so a
// unit's counter ends at T + H (H home warps); the warp whose failing claim returns T + H - 1 makes
// the last increment of the call and stores 0, which leaves the counter ready for the next call.
static_assert(kRangeCache == (kChunkRows - 2 * kBatchRows - 1) / 2, "two batch tables and the range cache share a row table");

// One lane's part in resolving a batch: its row's kind (-1 masked, 0..15 the token's slot in its block,
// 16 a summary row) and the value it loads (the token's block-table entry or the summary's segment).
struct RowPrep {
  int kind;
  int val;
};

struct UnitView {
  const int32_t* cache;  // shared memory: the range prefix sums [nr + 1], then the range starts [nr]
  int u, b, g, nr, n_tok, R, seg0;
};

__device__ __forceinline__ RowPrep prep_row(const StepArgs& a, const UnitView& v, int r) {
  RowPrep o{-1, 0};
  if (r >= v.R) return o;
  if (r >= v.n_tok) {
    o.kind = 16;
    o.val = a.sumlist[static_cast<size_t>(v.u) * a.n_max + (r - v.n_tok)];
    return o;
  }
  const int32_t* cum = v.cache;
  int lo = 0, hi = v.nr - 1;  // the last range whose first row is <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cum[mid] <= r) lo = mid; else hi = mid - 1;
  }
  const int t = cum[v.nr + 1 + lo] + (r - cum[lo]);
  o.kind = t & 15;
  o.val = a.block_tables[static_cast<size_t>(v.b) * a.max_blocks + (t >> 4)];
  return o;
}

__device__ __forceinline__ uint32_t finish_row(const StepArgs& a, const UnitView& v, RowPrep rp) {
  if (rp.kind < 0) return kInvalidRow;
  if (rp.kind == 16) return (static_cast<uint32_t>(v.seg0 + rp.val) * a.Hkv + v.g) | kSummaryFlag;
  if (static_cast<unsigned>(rp.val) < static_cast<unsigned>(a.num_blocks))
    return ((static_cast<uint32_t>(rp.val) * a.Hkv + v.g) << 4) | static_cast<uint32_t>(rp.kind);
  atomicOr(a.err, kErrBadBlock);
  return kInvalidRow;
}

// All rows of unit u that this warp claims, then its partial into `slot`. H: the unit's home warps.
template <int D>
__device__ void visit_unit_dynamic(const StepArgs& a, MmaWorker<D>& wk, uint32_t* tab, int u, int p, int H,
                                   int lane) {
  constexpr uint32_t SB = MmaWorker<D>::kStageBytes;
  const int b = u / a.Hkv, g = u - b * a.Hkv;
  const int32_t* rg = a.ranges + static_cast<size_t>(u) * (a.k_max + 1) * 2;
  const int32_t* cum = a.cum + static_cast<size_t>(u) * (a.k_max + 2);
  // One round trip: the first claim, the unit's sizes, the first 32 range bounds and the queries.
  int claim = 0;
  if (lane == 0) claim = atomicAdd(a.tile_ctr + static_cast<size_t>(u) * kCtrStride, 1);
  const int c_l = lane <= a.k_max + 1 ? cum[lane] : 0;
  const int s_l = lane <= a.k_max ? rg[2 * lane] : 0;
  const int4 info = a.unit_info[u];
  UnitView v;
  v.seg0 = a.meta.seg_ptr[b];
  wk.begin_unit(a, b, g, lane);
  v.u = u;
  v.b = b;
  v.g = g;
  v.nr = info.x;
  v.n_tok = info.y;
  v.R = info.y + info.z;
  const int T = (v.R + kBatchRows - 1) / kBatchRows;
  int32_t* cache = reinterpret_cast<int32_t*>(tab) + 2 * kBatchRows;
  __syncwarp();  // the previous unit's readers of the table and the cache are done
  // The plan enables the dynamic split only when k_max + 1 <= kRangeCache, so every unit's ranges fit.
  if (lane <= v.nr) cache[lane] = c_l;
  if (lane < v.nr) cache[v.nr + 1 + lane] = s_l;
  for (int i = 32 + lane; i <= v.nr; i += 32) cache[i] = cum[i];
  for (int i = 32 + lane; i < v.nr; i += 32) cache[v.nr + 1 + i] = rg[2 * i];
  v.cache = cache;
  __syncwarp();
  auto failed = [&](int c) {  // c: this warp's failing claim (>= T), the same in every lane
    if (lane == 0 && c + 1 == T + H) a.tile_ctr[static_cast<size_t>(u) * kCtrStride] = 0;
  };
  claim = __shfl_sync(kFull, claim, 0);
  if (claim >= T) {
    failed(claim);
    wk.end_unit(a, u + p, lane);
    return;
  }
  uint32_t* tb = tab;  // two 32-entry tables: batch parity s in tb + 32 s
  const size_t ci = static_cast<size_t>(u) * kCtrStride;
  int cur = claim, s = 0, stage = 0;
  RowPrep rp = prep_row(a, v, kBatchRows * cur + lane);
  int pend = 0;
  if (lane == 0) pend = atomicAdd(a.tile_ctr + ci, 1);
  tb[lane] = finish_row(a, v, rp);
  __syncwarp();
  mma_issue_tile_p<D>(wk.ring, tb, 0, lane, a);
  cp_async_commit();
  // The batch after cur: its row ids are loaded into rp a whole batch before its first tile is issued.
  int nxt = -1;
  // The outstanding claim: load its row ids and claim the batch after it. A claim is outstanding
  // exactly while the last one resolved succeeded, i.e. while nxt >= 0.
  auto resolve = [&]() {
    const int c = __shfl_sync(kFull, pend, 0);
    if (c < T) {
      rp = prep_row(a, v, kBatchRows * c + lane);
      if (lane == 0) pend = atomicAdd(a.tile_ctr + ci, 1);
      return c;
    }
    failed(c);
    return -1;
  };
  nxt = resolve();
  while (true) {
    const int nt = min(2, (v.R - kBatchRows * cur + 15) >> 4);  // tiles of batch cur (1: a final batch of <= 16 rows)
    int after = -1;
    for (int h = 0; h < nt; ++h) {
      __syncwarp();  // every lane is done reading the stage (and the table) that is refilled next
      if (h + 1 < nt) {
        mma_issue_tile_p<D>(wk.ring + (stage ^ 1) * SB, tb + kBatchRows * s, 16, lane, a);
      } else if (nxt >= 0) {  // cur's last tile: start the next batch, then prepare the one after it
        tb[kBatchRows * (s ^ 1) + lane] = finish_row(a, v, rp);
        __syncwarp();
        mma_issue_tile_p<D>(wk.ring + (stage ^ 1) * SB, tb + kBatchRows * (s ^ 1), 0, lane, a);
        after = resolve();
      }
      cp_async_commit();
      cp_async_wait<1>();
      __syncwarp();  // the tile's rows, staged by all lanes, are visible to every lane
      const uint32_t vmask16 =
          __ballot_sync(kFull, lane < 16 && tb[kBatchRows * s + 16 * h + lane] != kInvalidRow) & 0xFFFFu;
      mma_compute_tile<D>(wk.st, wk.ring + stage * SB, vmask16, a.scale_log2, lane);
      stage ^= 1;
    }
    if (nxt < 0) break;
    cur = nxt;
    nxt = after;
    s ^= 1;
  }
  wk.end_unit(a, u + p, lane);
}

// Home warps of the unit whose rows occupy [c0, c0 + Ru) of a cost coordinate of length C split
// evenly among N warps (the warp whose share holds position c is ceil((c + 1) N / C) - 1).
__device__ __forceinline__ int home_warps(long long c0, int Ru, long long C, long long N) {
  const long long wf = ((c0 + 1) * N + C - 1) / C - 1;
  const long long wl = ((c0 + Ru) * N + C - 1) / C - 1;
  return static_cast<int>(wl - wf + 1);
}

// One warp at position p: every unit whose rows its share meets, each visited until the unit's rows
// run out.
template <int D>
__device__ void attend_dynamic(const StepArgs& a, const UnitRows& rows, MmaWorker<D>& wk, uint32_t* tab, int p,
                               int lane) {
  WarpRange wr;
  if (!locate_range(a, rows, p, a.attend_warps, lane, wr)) return;
  int u = wr.u;
  long long P = wr.P;
  int Ru = wr.Ru;
  while (true) {
    const long long first = P + a.unit_cost;
    if (Ru > 0 && wr.s < first + Ru && wr.e > first)
      visit_unit_dynamic<D>(a, wk, tab, u, p, home_warps(first, Ru, wr.R, wr.N), lane);
    if (first + Ru >= wr.e) break;
    P = first + Ru;
    ++u;
    Ru = rows(u);
  }
}

template <int D>
__global__ void __launch_bounds__(kAttendWarps * 32, 3) zr_attend_mma_kernel(StepArgs a) {
  extern __shared__ __align__(16) unsigned char attend_smem[];
  __shared__ uint32_t rowtab[kAttendWarps][kChunkRows];
  __shared__ int32_t s_rows[kStagedUnits];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  prefetch_attend_inputs(a, sizeof(__nv_bfloat16) * D);
  prefetch_fixed_rows(a, sizeof(__nv_bfloat16) * D);
  pdl_wait();
  pdl_trigger();  // after the wait: the merge kernel may read the select kernel's unit sizes at once
  if (a.pf_blocks > 0) prefetch_selected_lists(a, kBlockTokens * D * sizeof(__nv_bfloat16));
  MmaWorker<D> wk;
  wk.ring = static_cast<uint32_t>(__cvta_generic_to_shared(attend_smem)) + warp * kStages * MmaWorker<D>::kStageBytes;
  const int chunk_off = (lane % (D / 8)) * 16;
  wk.lb = LoadBases{static_cast<const char*>(a.k_pool) + chunk_off, static_cast<const char*>(a.v_pool) + chunk_off,
                    static_cast<const char*>(a.sum_k) + chunk_off, static_cast<const char*>(a.sum_v) + chunk_off,
                    l2_evict_first_policy()};
  const UnitRows rows = stage_unit_rows(a, s_rows);
  if (a.dynamic)
    attend_dynamic<D>(a, rows, wk, rowtab[warp], warp * static_cast<int>(gridDim.x) + blockIdx.x, lane);
  else
    attend_balanced(a, rows, wk, rowtab[warp], warp, lane);
}

// ------------------------------------------------------------------ attend: CUDA cores (f32, or any G)
// Lanes split d (D/32 components each); rows are taken one at a time, logits reduced across the
// warp, and each query head keeps its own online-softmax state.
template <typename T, int D>
struct FmaWorker {
  static constexpr int E = D / 32;
  float qv[kMaxGroup][E], o[kMaxGroup][E], m[kMaxGroup], l[kMaxGroup];

  __device__ void begin_unit(const StepArgs& a, int b, int g, int lane) {
    const int G = a.G;
    const T* qg = static_cast<const T*>(a.q) + (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G) * D;
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      m[h] = -1e30f;
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) o[h][e] = 0.f;
      if (h < G) {
        load_e<T, E>(qg + h * D + lane * E, qv[h]);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) qv[h][e] = 0.f;
      }
    }
  }

  __device__ void run(const StepArgs& a, const uint32_t* tab, int nrows, int lane) {
    const int G = a.G;
    const T* kp = static_cast<const T*>(a.k_pool);
    const T* vp = static_cast<const T*>(a.v_pool);
    const T* skp = static_cast<const T*>(a.sum_k);
    const T* svp = static_cast<const T*>(a.sum_v);
    for (int j = 0; j < nrows; ++j) {
      const uint32_t id = tab[j];
      if (id == kInvalidRow) continue;
      float kv[E], vv[E];
      load_e<T, E>(row_ptr<T, D>(id, kp, skp) + lane * E, kv);
      load_e<T, E>(row_ptr<T, D>(id, vp, svp) + lane * E, vv);
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h) {
        if (h < G) {
          float dot = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) dot = fmaf(qv[h][e], kv[e], dot);
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) dot += __shfl_xor_sync(kFull, dot, o2);
          const float x = dot * a.scale_log2;
          const float mn = fmaxf(m[h], x);
          const float alpha = fast_exp2(m[h] - mn);
          const float p = fast_exp2(x - mn);
          l[h] = l[h] * alpha + p;
#pragma unroll
          for (int e = 0; e < E; ++e) o[h][e] = fmaf(p, vv[e], o[h][e] * alpha);
          m[h] = mn;
        }
      }
    }
  }

  __device__ void end_unit(const StepArgs& a, int slot, int lane) {
    const int G = a.G;
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      if (h < G) {
        float* dst = a.part_o + (static_cast<size_t>(slot) * G + h) * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) dst[e] = o[h][e];
        if (lane == 0) a.part_ml[static_cast<size_t>(slot) * G + h] = make_float2(m[h], l[h]);
      }
    }
  }
};

template <typename T, int D>
__global__ void __launch_bounds__(kAttendWarps * 32) zr_attend_fma_kernel(StepArgs a) {
  __shared__ uint32_t rowtab[kAttendWarps][kChunkRows];
  __shared__ int32_t s_rows[kStagedUnits];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  prefetch_attend_inputs(a, sizeof(T) * D);
  prefetch_fixed_rows(a, sizeof(T) * D);
  pdl_wait();
  pdl_trigger();  // after the wait: the merge kernel may read the select kernel's unit sizes at once
  if (a.pf_blocks > 0) prefetch_selected_lists(a, kBlockTokens * D * sizeof(T));
  FmaWorker<T, D> wk;
  attend_balanced(a, stage_unit_rows(a, s_rows), wk, rowtab[warp], warp, lane);
}

// ------------------------------------------------------------------ merge
// Two layouts of the same log-sum-exp combination; zr_plan picks one (configure_for).
//
// zr_merge_comp_kernel: one warp per (sequence, query head, 32-wide slice of d); lane j owns
// component j of the slice.
// The unit's partials are taken 32 at a time: lane k loads partial k's (m, l) while every lane
// loads its component of all 32 partial rows (all independent loads, one round trip); then each
// partial's weight 2^(m_k - M) is broadcast from lane k and accumulated. A running maximum keeps
// the weights bounded when a unit has more than 32 partials.
template <int D>
__global__ void __launch_bounds__(kAttendWarps * 32) zr_merge_comp_kernel(StepArgs a) {
  constexpr int NDC = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * kAttendWarps + warp;
  pdl_trigger();
  if (w >= a.B * a.Hq * NDC) return;
  const int dc = w % NDC, bh = w / NDC;
  const int b = bh / a.Hq, h = bh - b * a.Hq;
  const int G = a.G, g = h / G, hh = h - g * G;
  const int u = b * a.Hkv + g;
  // The warps holding unit u follow from the select kernel's unit sizes alone. This kernel is
  // launched only after every attend CTA has passed its own wait on the select kernel, so those
  // sizes are complete here, before the wait on the attend kernel.
  const int U = a.B * a.Hkv;
  long long R = 0, Pu = 0;
  int Ru = 0;
  for (int base = 0; base < U; base += 32) {
    const int uu = base + lane;
    const int r = uu < U ? unit_rows(a, uu) : 0;
    R += r;
    if (uu < u) Pu += r;
    if (uu == u) Ru = r;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    R += __shfl_xor_sync(kFull, R, o);
    Pu += __shfl_xor_sync(kFull, Pu, o);
    Ru += __shfl_xor_sync(kFull, Ru, o);
  }
  // the split's cost coordinate: unit u's rows at [Pu + (u + 1) X, Pu + (u + 1) X + Ru), C = R + U X
  const long long X = a.unit_cost, C = R + static_cast<long long>(U) * X;
  const long long N = min(static_cast<long long>(a.attend_warps), C);
  const long long c0 = Pu + (u + 1) * X, c1 = c0 + Ru - 1;  // the unit's first and last row
  // warp whose share holds cost position c: ceil((c + 1) N / C) - 1
  const long long wf = ((c0 + 1) * N + C - 1) / C - 1, wl = ((c1 + 1) * N + C - 1) / C - 1;
  const size_t first = static_cast<size_t>(u) + wf;
  const int cnt = static_cast<int>(wl - wf + 1);
  pdl_wait();
  float M = -INFINITY, Ls = 0.f, acc = 0.f;
  for (int c0 = 0; c0 < cnt; c0 += 32) {
    const int n = min(32, cnt - c0);
    float2 ml = make_float2(-INFINITY, 0.f);
    if (lane < n) ml = a.part_ml[(first + c0 + lane) * G + hh];
    float v[32];
    const float* src = a.part_o + ((first + c0) * G + hh) * D + 32 * dc + lane;
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = k < n ? src[static_cast<size_t>(k) * G * D] : 0.f;
    float mc = ml.x;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) mc = fmaxf(mc, __shfl_xor_sync(kFull, mc, o2));
    const float Mn = fmaxf(M, mc);
    const float rescale = fast_exp2(M - Mn);  // 0 on the first batch (M = -inf)
    acc *= rescale;
    Ls *= rescale;
    M = Mn;
    const float wk = lane < n ? fast_exp2(ml.x - M) : 0.f;
    float lsum = ml.y * wk;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) lsum += __shfl_xor_sync(kFull, lsum, o2);
    Ls += lsum;
#pragma unroll
    for (int k = 0; k < 32; ++k) acc = fmaf(__shfl_sync(kFull, wk, k), v[k], acc);
  }
  a.out[(static_cast<size_t>(b) * a.Hq + h) * D + 32 * dc + lane] = acc / Ls;
}

// zr_merge_part_kernel: one warp per (sequence, query head, kMergeComp-wide slice of d), four
// slices of one head per CTA. Lane j takes the unit's partials
// j, j + 32, ... (kMergeBatch per lane per memory round trip, so up to 32 * kMergeBatch partials
// arrive in one trip) and folds them into its own running (m, l, o) with log-sum-exp weights; the
// 32 lane states are then combined by a butterfly (max, rescale, sum). Each partial row slice is
// 32 contiguous bytes, a whole sector. The CTA's first warp finds which attend warps hold the unit.
constexpr int kMergeComp = 8;
constexpr int kMergeBatch = 4;
#ifndef ZR_MERGE_WARPS
#define ZR_MERGE_WARPS 4
#endif
// Warps per merge CTA: the slices of one query head, at most ZR_MERGE_WARPS of them.
template <int D>
__host__ __device__ constexpr int merge_warps() {
  return ZR_MERGE_WARPS < D / kMergeComp ? ZR_MERGE_WARPS : D / kMergeComp;
}

template <int D>
__global__ void __launch_bounds__(merge_warps<D>() * 32, 32 / merge_warps<D>()) zr_merge_part_kernel(StepArgs a) {
  constexpr int NC = D / kMergeComp;
  constexpr int kMergeWarps = merge_warps<D>();
  static_assert(NC % kMergeWarps == 0, "a CTA's slices belong to one query head");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * kMergeWarps + warp;
  const int cs = w % NC, bh = w / NC;
  const int b = bh / a.Hq, h = bh - b * a.Hq;
  const int G = a.G, g = h / G, hh = h - g * G;
  const int u = b * a.Hkv + g;
  __shared__ long long s_first;
  __shared__ int s_cnt;
  pdl_trigger();
  // The warps holding unit u follow from the select kernel's unit sizes alone. This kernel is
  // launched only after every attend CTA has passed its own wait on the select kernel, so those
  // sizes are complete here, before the wait on the attend kernel.
  if (warp == 0) {
    const int U = a.B * a.Hkv;
    long long R = 0, Pu = 0;
    int Ru = 0;
    for (int base = 0; base < U; base += 32) {
      const int uu = base + lane;
      const int r = uu < U ? unit_rows(a, uu) : 0;
      R += r;
      if (uu < u) Pu += r;
      if (uu == u) Ru = r;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      R += __shfl_xor_sync(kFull, R, o);
      Pu += __shfl_xor_sync(kFull, Pu, o);
      Ru += __shfl_xor_sync(kFull, Ru, o);
    }
    // the split's cost coordinate: unit u's rows at [Pu + (u + 1) X, Pu + (u + 1) X + Ru), C = R + U X
    const long long X = a.unit_cost, C = R + static_cast<long long>(U) * X;
    const long long N = min(static_cast<long long>(a.attend_warps), C);
    const long long c0 = Pu + (u + 1) * X, c1 = c0 + Ru - 1;  // the unit's first and last row
    // warp whose share holds cost position c: ceil((c + 1) N / C) - 1
    const long long wf = ((c0 + 1) * N + C - 1) / C - 1, wl = ((c1 + 1) * N + C - 1) / C - 1;
    if (lane == 0) {
      s_first = u + wf;
      s_cnt = static_cast<int>(wl - wf + 1);
    }
  }
  __syncthreads();
  const size_t first = static_cast<size_t>(s_first);
  const int cnt = s_cnt;
  pdl_wait();
  float m = -INFINITY, l = 0.f, acc[kMergeComp];
#pragma unroll
  for (int c = 0; c < kMergeComp; ++c) acc[c] = 0.f;
  for (int p0 = 0; p0 < cnt; p0 += 32 * kMergeBatch) {
    float2 ml[kMergeBatch];
    float4 o0[kMergeBatch], o1[kMergeBatch];
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      const int p = p0 + 32 * j + lane;
      if (p < cnt) {
        const size_t row = (first + p) * G + hh;
        ml[j] = a.part_ml[row];
        const float4* src = reinterpret_cast<const float4*>(a.part_o + row * D + kMergeComp * cs);
        o0[j] = src[0];
        o1[j] = src[1];
      }
    }
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      if (p0 + 32 * j + lane < cnt) {
        const float mn = fmaxf(m, ml[j].x);
        const float sc = fast_exp2(m - mn), wt = fast_exp2(ml[j].x - mn);  // sc = 0 while m = -inf
        l = fmaf(l, sc, ml[j].y * wt);
        const float v[kMergeComp] = {o0[j].x, o0[j].y, o0[j].z, o0[j].w, o1[j].x, o1[j].y, o1[j].z, o1[j].w};
#pragma unroll
        for (int c = 0; c < kMergeComp; ++c) acc[c] = fmaf(acc[c], sc, wt * v[c]);
        m = mn;
      }
    }
  }
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  const float s = fast_exp2(m - M);  // 0 for lanes that took no partial
  l *= s;
#pragma unroll
  for (int c = 0; c < kMergeComp; ++c) acc[c] *= s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    l += __shfl_xor_sync(kFull, l, o);
#pragma unroll
    for (int c = 0; c < kMergeComp; ++c) acc[c] += __shfl_xor_sync(kFull, acc[c], o);
  }
  if (lane == 0) {
    const float inv = 1.f / l;
    float4* dst = reinterpret_cast<float4*>(a.out + (static_cast<size_t>(b) * a.Hq + h) * D + kMergeComp * cs);
    dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
  }
}

// ------------------------------------------------------------------ launch
template <typename Kern>
cudaError_t launch_pdl(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const StepArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <typename T, int D>
size_t select_smem_bytes(int G, int n_max) {
  return SelectLayout<T, D>::bytes(G, n_max);
}

template <typename T, int D>
bool uses_mma(const Plan& p) {
  if constexpr (sizeof(T) == 2) return p.G <= kMmaMaxGroup;
  return false;
}

template <typename T, int D>
zr_status configure_for(Plan& p, int64_t useful_warps) {
  int sms = 0, occ = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p.device) != cudaSuccess) {
    cudaGetLastError();
    return ZR_ECUDA;
  }
  cudaError_t e = cudaSuccess;
  if (uses_mma<T, D>(p)) {
    p.attend_smem = attend_ring_bytes<D>();
    if constexpr (sizeof(T) == 2) {
      e = cudaFuncSetAttribute(zr_attend_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(p.attend_smem));
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, zr_attend_mma_kernel<D>, kAttendWarps * 32,
                                                          p.attend_smem);
    }
  } else {
    p.attend_smem = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, zr_attend_fma_kernel<T, D>, kAttendWarps * 32, 0);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ZR_ECUDA;
  }
#ifndef ZR_ATTEND_WAVES
#define ZR_ATTEND_WAVES 1
#endif
  int64_t ctas = static_cast<int64_t>(sms) * (occ > 0 ? occ : 1) * ZR_ATTEND_WAVES;
  ctas = std::min<int64_t>(ctas, (useful_warps + kAttendWarps - 1) / kAttendWarps);
  p.attend_ctas = static_cast<int>(std::max<int64_t>(ctas, 1));
  p.attend_warps = p.attend_ctas * kAttendWarps;
  // Merge layout (both measured on GB300): lanes over partials when a unit has few partials on
  // average (at most 64) and its warps fit one resident wave (64 registers: 32 warps per SM);
  // otherwise lanes over components, which is faster with many partials per unit or many heads.
  const int64_t units = static_cast<int64_t>(p.B) * p.Hkv;
  const int64_t part_warps = static_cast<int64_t>(p.B) * p.Hq * (D / kMergeComp);
  p.merge_parts = p.attend_warps <= 64 * units && part_warps <= static_cast<int64_t>(sms) * 32;
  if (const char* m = std::getenv("ZOOMR_MERGE")) {  // pin the layout (used by the tests to cover both)
    if (std::strcmp(m, "parts") == 0) p.merge_parts = 1;
    if (std::strcmp(m, "comp") == 0) p.merge_parts = 0;
  }
  // One shared-memory carveout for all three kernels: a kernel whose preferred L1/shared split
  // differs from the previous one's makes the SM drain and reconfigure between them.
  const int carve = cudaSharedmemCarveoutMaxShared;
  cudaFuncSetAttribute(zr_select_kernel<T, D>, cudaFuncAttributePreferredSharedMemoryCarveout, carve);
  cudaFuncSetAttribute(zr_merge_comp_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout, carve);
  cudaFuncSetAttribute(zr_merge_part_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout, carve);
  cudaFuncSetAttribute(zr_attend_fma_kernel<T, D>, cudaFuncAttributePreferredSharedMemoryCarveout, carve);
  if constexpr (sizeof(T) == 2)
    cudaFuncSetAttribute(zr_attend_mma_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout, carve);
  cudaGetLastError();
  // Set for every plan: the kernel's static shared memory counts against the 48 KB default too.
  p.select_smem = select_smem_bytes<T, D>(p.G, p.n_max);
  if (cudaFuncSetAttribute(zr_select_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(p.select_smem)) != cudaSuccess) {
    cudaGetLastError();
    return ZR_ECUDA;
  }
  return ZR_OK;
}

// Inside a stream capture an event record must be "external" to become an event-record node
// of the graph; outside a capture it is a plain record.
cudaError_t record_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, s);
}

void report(const char* what, cudaError_t e) {
  if (std::getenv("ZOOMR_VERBOSE")) std::fprintf(stderr, "zoomr: %s: %s\n", what, cudaGetErrorString(e));
}

template <typename T, int D>
cudaError_t launch_for(const Plan& p, const StepArgs& a, cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1) {
  cudaError_t e = launch_pdl(zr_select_kernel<T, D>, dim3(p.Hkv, p.B), dim3(kSelectThreads), p.select_smem, s, a);
  if (e != cudaSuccess) return report("select launch", e), e;
  if (ev0 && (e = record_event(ev0, s)) != cudaSuccess) return report("start event record", e), e;
  const dim3 grid_attend(p.attend_ctas), block(kAttendWarps * 32);
  if (uses_mma<T, D>(p)) {
    if constexpr (sizeof(T) == 2) e = launch_pdl(zr_attend_mma_kernel<D>, grid_attend, block, p.attend_smem, s, a);
  } else {
    e = launch_pdl(zr_attend_fma_kernel<T, D>, grid_attend, block, 0, s, a);
  }
  if (e != cudaSuccess) return report("attend launch", e), e;
  if (ev1 && (e = record_event(ev1, s)) != cudaSuccess) return report("stop event record", e), e;
  if (p.merge_parts) {
    e = launch_pdl(zr_merge_part_kernel<D>, dim3(p.B * p.Hq * (D / kMergeComp) / merge_warps<D>()),
                   dim3(merge_warps<D>() * 32), 0, s, a);
  } else {
    const dim3 grid_merge((p.B * p.Hq * (D / 32) + kAttendWarps - 1) / kAttendWarps);
    e = launch_pdl(zr_merge_comp_kernel<D>, grid_merge, block, 0, s, a);
  }
  if (e != cudaSuccess) report("merge launch", e);
  return e;
}

template <typename T, int D>
cudaError_t launch_attend_for(const Plan& p, const StepArgs& a, cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1) {
  const dim3 grid_attend(p.attend_ctas), block(kAttendWarps * 32);
  cudaError_t e = cudaSuccess;
  if (ev0 && (e = record_event(ev0, s)) != cudaSuccess) return report("start event record", e), e;
  if (uses_mma<T, D>(p)) {
    if constexpr (sizeof(T) == 2) e = launch_pdl(zr_attend_mma_kernel<D>, grid_attend, block, p.attend_smem, s, a);
  } else {
    e = launch_pdl(zr_attend_fma_kernel<T, D>, grid_attend, block, 0, s, a);
  }
  if (e != cudaSuccess) return report("attend launch", e), e;
  if (ev1 && (e = record_event(ev1, s)) != cudaSuccess) return report("stop event record", e), e;
  if (p.merge_parts) {
    e = launch_pdl(zr_merge_part_kernel<D>, dim3(p.B * p.Hq * (D / kMergeComp) / merge_warps<D>()),
                   dim3(merge_warps<D>() * 32), 0, s, a);
  } else {
    const dim3 grid_merge((p.B * p.Hq * (D / 32) + kAttendWarps - 1) / kAttendWarps);
    e = launch_pdl(zr_merge_comp_kernel<D>, grid_merge, block, 0, s, a);
  }
  if (e != cudaSuccess) report("merge launch", e);
  return e;
}

}  // namespace

zr_status configure_kernels(Plan& p, int64_t useful_warps) {
  if (p.cfg.dtype == ZR_BF16)
    return p.d == 64 ? configure_for<__nv_bfloat16, 64>(p, useful_warps)
                     : configure_for<__nv_bfloat16, 128>(p, useful_warps);
  return p.d == 64 ? configure_for<float, 64>(p, useful_warps) : configure_for<float, 128>(p, useful_warps);
}

zr_status launch_attend_only(const Plan& p, const StepArgs& a, void* stream, void* ev_start, void* ev_stop) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaEvent_t e0 = static_cast<cudaEvent_t>(ev_start), e1 = static_cast<cudaEvent_t>(ev_stop);
  cudaError_t e;
  if (p.cfg.dtype == ZR_BF16)
    e = p.d == 64 ? launch_attend_for<__nv_bfloat16, 64>(p, a, s, e0, e1)
                  : launch_attend_for<__nv_bfloat16, 128>(p, a, s, e0, e1);
  else
    e = p.d == 64 ? launch_attend_for<float, 64>(p, a, s, e0, e1) : launch_attend_for<float, 128>(p, a, s, e0, e1);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ZR_ECUDA;
  }
  return ZR_OK;
}

zr_status launch_step(const Plan& p, const StepArgs& a, void* stream, void* ev_start, void* ev_stop) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaEvent_t e0 = static_cast<cudaEvent_t>(ev_start), e1 = static_cast<cudaEvent_t>(ev_stop);
  cudaError_t e;
  if (p.cfg.dtype == ZR_BF16)
    e = p.d == 64 ? launch_for<__nv_bfloat16, 64>(p, a, s, e0, e1) : launch_for<__nv_bfloat16, 128>(p, a, s, e0, e1);
  else
    e = p.d == 64 ? launch_for<float, 64>(p, a, s, e0, e1) : launch_for<float, 128>(p, a, s, e0, e1);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ZR_ECUDA;
  }
  return ZR_OK;
}

}  // namespace zr
