// Consensus selection of the ZoomR page, section 3.3, on the device.
//
//   vote       one CTA per (sequence b, KV head g) and layer: for every query head
//              of the group, the top-k of the summaries by the exact score
//              alpha_i = q^T kbar_i of the stored values (3.3 "Per-Head Importance
//              Scoring and Voting"; ties to the lower index), and one vote per
//              selected summary added to the sequence's vote counts.
//   consensus  one CTA per sequence, once per selection: I_all (summaries with a
//              vote), I_c (the c with the most votes, ties to the lower index),
//              I_s = I_all minus I_c (3.3 "Global Aggregation and Consensus"); the
//              final token set I_f = prompt + window + R_i (i in I_c) + S_i (i in
//              I_s) as maximal ascending ranges (3.3 "Constructing the Final
//              Multi-Granularity Context"), written as the attend metadata of
//              every KV head of the sequence; the vote counts are cleared.
//
// Layout of a sequence: prompt [0, N_p), then pairs R_i = [bd[2i], bd[2i+1]),
// S_i = [bd[2i+1], bd[2i+2]) with bd[0] = N_p; S_{i-1} ends where R_i starts,
// and the prompt ends where R_0 starts: those are the only touching pieces.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "zoomr_exact_key.cuh"
#include "zoomr_internal.h"

namespace zr {
namespace {

constexpr unsigned kFullMask = 0xFFFFFFFFu;
constexpr int kVoteThreads = 256;
constexpr int kConsensusThreads = 256;

// Shared memory: the exact-key scorer's query limb tables | the query table [G * D] | key high words
// [n_max + 4] u64 | key low words [n_max + 4] u64 | flag [n_max + 2] | fp32 enclosures lo, hi [n_max] each.
template <typename T, int D>
struct VoteLayout {
  using SC = xk::Scorer<T, D, kVoteThreads>;
  __host__ __device__ static constexpr size_t limb_bytes(int G) { return (SC::smem_bytes(G) + 15) / 16 * 16; }
  __host__ __device__ static constexpr size_t q_bytes(int G) {
    return limb_bytes(G) + sizeof(T) * static_cast<size_t>(G) * D;
  }
  __host__ __device__ static constexpr size_t bytes(int G, int n_max) {
    return q_bytes(G) + 2 * sizeof(uint64_t) * (static_cast<size_t>(n_max) + 4) +
           sizeof(int) * (static_cast<size_t>(n_max) + 2) + 2 * sizeof(float) * static_cast<size_t>(n_max);
  }
};

// For every query head of the group, one at a time: the top-k of the summaries by the exact key
// alpha_i = q_h . kbar_i on the stored values (ties to the lower index) and one vote per selected summary.
// The fp32 estimates decide where their enclosures separate at the k boundary; otherwise the uncertain
// summaries' keys are computed exactly (the integer limbs, or the general 640-bit path).
template <typename T, int D>
__global__ void __maxnreg__(96) zr_vote_kernel(StepArgs a, const T* __restrict__ mean_keys,
                                               int32_t* __restrict__ votes) {
  using LY = VoteLayout<T, D>;
  using SC = typename LY::SC;
  extern __shared__ __align__(16) unsigned char vsmem[];
  const int G = a.G, nmax = a.n_max;
  int* qh = reinterpret_cast<int*>(vsmem);
  int* ql = qh + G * SC::kQRow;
  int* qtail = ql + G * SC::kQRow;
  uint4* qtab = reinterpret_cast<uint4*>(vsmem + LY::limb_bytes(G));
  uint64_t* kh = reinterpret_cast<uint64_t*>(vsmem + LY::q_bytes(G));
  uint64_t* kl = kh + nmax + 4;
  int* flag = reinterpret_cast<int*>(kl + nmax + 4);
  float* elo = reinterpret_cast<float*>(flag + nmax + 2);
  float* ehi = elo + nmax;
  __shared__ int s_flags;
  __shared__ uint32_t s_red[4 * kVoteThreads / 32];
  __shared__ uint32_t s_cert[3 * kVoteThreads / 32];
  const int g = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int u = b * a.Hkv + g;
  const int s0 = a.meta.seg_ptr[b];
  const int n = a.meta.seg_ptr[b + 1] - s0;
  const int k = a.meta.topk[b];  // clipped to n at plan time
  const T* qg = static_cast<const T*>(a.q) + (static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * G) * D;
  const T* rows = mean_keys + (static_cast<size_t>(s0) * a.Hkv + g) * D;
  const size_t stride = static_cast<size_t>(a.Hkv) * D;
  int32_t* vb = votes + static_cast<size_t>(b) * nmax;
  for (int h = 0; h < G; ++h) {
    // the first head builds the query table
    xk::estimate_rows<T, D, kVoteThreads, false, 16>(h == 0 ? qg : nullptr, G, qtab, h, 1, rows, stride, n,
                                                  [&](int r, int, float mid, float lo, float hi) {
                                                    kh[r] = 0;
                                                    kl[r] = xk::order_bits(mid);
                                                    elo[r] = lo;
                                                    ehi[r] = hi;
                                                  });
    __syncthreads();
    float cert_lo, cert_hi;
    if (!xk::certify_top_k<kVoteThreads>(elo, ehi, n, k, kh, kl, flag, s_cert, cert_lo, cert_hi)) {
      const int uflags = xk::resolve_top_k<T, D, kVoteThreads, false>(
          qg, G, h, 1, rows, stride, n, k, elo, ehi, cert_lo, cert_hi, flag, reinterpret_cast<int*>(elo),
          reinterpret_cast<int*>(ehi), kh, kl, qh, ql, qtail, s_red, &s_flags,
          a.bigkeys + static_cast<size_t>(u) * nmax * xk::kBigDigits);
      if ((uflags & xk::kFlagNonFinite) && tid == 0) atomicOr(a.err, kErrNonFinite);
    }
    // (certify_top_k and resolve_top_k end with a barrier after the flags are written)
    for (int i = tid; i < n; i += kVoteThreads)
      if (flag[i]) atomicAdd(vb + i, 1);
    __syncthreads();  // flag, the estimates and the keys are reused by the next head
  }
}

__device__ __forceinline__ int warp_inclusive_sum(int x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFullMask, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// The calling warp merges the runs [0, m) (ascending, disjoint, touching runs already joined; run r is
// [rs[r * stride], re[r * stride])) with the window [W0, L) -- the first run that reaches W0 absorbs it
// and every later run -- and writes the ranges and their prefix sums as the attend metadata of units
// u0 .. u0 + nu - 1, each with n_sum summary rows; rout / nrout (optional) receive the ranges too.
__device__ void emit_ranges(const StepArgs& a, const int* rs, const int* re, int stride, int m, int W0, int L,
                            size_t u0, int nu, int n_sum, int32_t* rout, int32_t* nrout, int lane) {
  int rstar = m;
  for (int base = 0; base < m; base += 32) {
    const int r = base + lane;
    const unsigned hit = __ballot_sync(kFullMask, r < m && re[r * stride] >= W0);
    if (hit) {
      rstar = base + __ffs(hit) - 1;
      break;
    }
  }
  const int nr = rstar < m ? rstar + 1 : m + (W0 < L ? 1 : 0);
  int carry = 0;
  for (int base = 0; base < nr; base += 32) {
    const int r = base + lane;
    int s_ = 0, e_ = 0;
    if (r < nr) {
      if (r < rstar) {
        s_ = rs[r * stride];
        e_ = re[r * stride];
      } else {
        s_ = rstar < m ? min(W0, rs[rstar * stride]) : W0;
        e_ = L;
      }
    }
    const int len = e_ - s_;
    const int incl = warp_inclusive_sum(len, lane);
    if (r < nr) {
      for (int j = 0; j < nu; ++j) {
        const size_t u = u0 + j;
        a.ranges[(u * (a.k_max + 1) + r) * 2] = s_;
        a.ranges[(u * (a.k_max + 1) + r) * 2 + 1] = e_;
        a.cum[u * (a.k_max + 2) + r] = carry + incl - len;
      }
      if (rout) {
        rout[2 * r] = s_;
        rout[2 * r + 1] = e_;
      }
    }
    carry += __shfl_sync(kFullMask, incl, 31);
  }
  for (int j = lane; j < nu; j += 32) {
    const size_t u = u0 + j;
    a.cum[u * (a.k_max + 2) + nr] = carry;
    a.unit_info[u] = make_int4(nr, carry, n_sum, 0);
    a.unit_rows[u] = carry + n_sum;
  }
  if (lane == 0 && nrout) *nrout = nr;
}

// Shared memory: votes [n_max] | flag [n_max + 1] | bd [2 n_max + 1] | runs_s, runs_e [n_max + 2] each.
__global__ void __launch_bounds__(kConsensusThreads) zr_consensus_kernel(StepArgs a, int32_t* __restrict__ votes,
                                                                         int32_t* votes_out, int32_t* ic_out,
                                                                         int c_max) {
  extern __shared__ __align__(16) int csmem[];
  const int nmax = a.n_max;
  int* v = csmem;
  int* flag = v + nmax;
  int* bd = flag + nmax + 1;
  int* runs_s = bd + 2 * nmax + 1;
  int* runs_e = runs_s + nmax + 2;
  __shared__ int s_cand;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s0 = a.meta.seg_ptr[b];
  const int n = a.meta.seg_ptr[b + 1] - s0;
  const int L = a.meta.seq_lens[b];
  const int Np = a.meta.prompt_lens[b];
  const int32_t* pb = a.meta.seg_bounds + 2 * static_cast<size_t>(s0) + b;
  int32_t* vb = votes + static_cast<size_t>(b) * nmax;
  if (tid == 0) s_cand = 0;
  __syncthreads();
  int local = 0;
  for (int i = tid; i < n; i += kConsensusThreads) {
    v[i] = vb[i];
    vb[i] = 0;  // consumed: the next selection starts from zero
    local += v[i] > 0;
  }
  for (int i = tid; i <= 2 * n; i += kConsensusThreads) bd[i] = pb[i];
  if (local) atomicAdd(&s_cand, local);
  __syncthreads();
  const int c = min(a.meta.consensus[b], s_cand);
  // I_c: candidates that fewer than c candidates beat (more votes, or as many and a lower index)
  for (int i = tid; i < n; i += kConsensusThreads) {
    const int vi = v[i];
    int f = 0;
    if (vi > 0) {
      int beat = 0;
      for (int j = 0; j < n; ++j) beat += (v[j] > vi) | ((v[j] == vi) & (j < i));
      f = beat < c ? 1 : 2;  // 1: zoom in (R_i), 2: keep the summary (S_i)
    }
    flag[i] = f;
  }
  if (tid == 0) flag[n] = 0;
  __syncthreads();
  if (votes_out)
    for (int i = tid; i < nmax; i += kConsensusThreads) votes_out[static_cast<size_t>(b) * nmax + i] = i < n ? v[i] : 0;
  if (ic_out && warp == 1) {
    int carry = 0;
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      const bool in = i < n && flag[i] == 1;
      const unsigned m = __ballot_sync(kFullMask, in);
      if (in) ic_out[static_cast<size_t>(b) * c_max + carry + __popc(m & ((1u << lane) - 1u))] = i;
      carry += __popc(m);
    }
    for (int j = carry + lane; j < c_max; j += 32) ic_out[static_cast<size_t>(b) * c_max + j] = -1;
  }
  // Runs of touching pieces, in ascending order; the prompt (if any) is run 0.
  const int prompt_runs = Np > 0 ? 1 : 0;
  if (warp == 0) {
    if (lane == 0 && prompt_runs) {
      runs_s[0] = 0;
      runs_e[0] = Np;  // replaced below if R_0 extends the prompt's run
    }
    int carry = 0;
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      const int f = i < n ? flag[i] : 0;
      const bool touch_prev = f == 1 && (i == 0 ? Np > 0 : flag[i - 1] == 2);
      const bool start = f != 0 && !touch_prev;
      const bool last = f != 0 && !(f == 2 && flag[i + 1] == 1);
      const unsigned m = __ballot_sync(kFullMask, start);
      const int rid = prompt_runs + carry + __popc(m & ((2u << lane) - 1u)) - 1;
      if (start) runs_s[rid] = f == 1 ? bd[2 * i] : bd[2 * i + 1];
      if (last) runs_e[rid] = f == 1 ? bd[2 * i + 1] : bd[2 * i + 2];
      carry += __popc(m);
    }
    __syncwarp();  // every lane's runs are written
    const int m = prompt_runs + carry;
    // keep the runs for the steps until the next selection, whose windows move on
    int32_t* cr = a.cruns + static_cast<size_t>(b) * (nmax + 1) * 2;
    for (int r = lane; r < m; r += 32) {
      cr[2 * r] = runs_s[r];
      cr[2 * r + 1] = runs_e[r];
    }
    if (lane == 0) a.cnruns[b] = m;
    __syncwarp();
    emit_ranges(a, runs_s, runs_e, 1, m, max(0, L - a.window), L, static_cast<size_t>(b) * a.Hkv, a.Hkv, 0,
                a.ranges_out ? a.ranges_out + static_cast<size_t>(b) * (a.k_max + 1) * 2 : nullptr,
                a.nranges_out ? a.nranges_out + b : nullptr, lane);
  }
}

// Between selections (consensus plan): the stored runs of sequence b merged with the window of its new
// length. One warp per sequence; a length below the selection's or past the block table sets the
// error word and leaves the sequence unchanged.
__global__ void __launch_bounds__(32) zr_consensus_advance_kernel(StepArgs a, const int32_t* __restrict__ seq_lens) {
  const int b = blockIdx.x, lane = threadIdx.x;
  const int L = seq_lens[b];
  if (L < a.meta.seq_lens[b] || L > a.max_blocks * kBlockTokens) {
    if (lane == 0) atomicOr(a.err, kErrBadIndex);
    return;
  }
  const int32_t* cr = a.cruns + static_cast<size_t>(b) * (a.n_max + 1) * 2;
  emit_ranges(a, cr, cr + 1, 2, a.cnruns[b], max(0, L - a.window), L, static_cast<size_t>(b) * a.Hkv, a.Hkv, 0,
              nullptr, nullptr, lane);
}

// Between selections (decode plan): unit (b, g)'s runs of touching selected segments, rebuilt from the
// selection the last decode step stored (with the sink's run first, for plans with a sink), merged with
// the window of the new length. One warp per unit; the summary rows stay those of the selection step.
__global__ void __launch_bounds__(32) zr_decode_advance_kernel(StepArgs a, const int32_t* __restrict__ seq_lens) {
  extern __shared__ int asmem[];  // runs_s [k_max + 1] | runs_e [k_max + 1]
  int* runs_s = asmem;
  int* runs_e = asmem + a.k_max + 1;
  const int g = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
  const size_t u = static_cast<size_t>(b) * a.Hkv + g;
  const int L = seq_lens[b];
  if (L < a.meta.seq_lens[b] || L > a.max_blocks * kBlockTokens) {
    if (lane == 0 && g == 0) atomicOr(a.err, kErrBadIndex);
    return;
  }
  const int s0 = a.meta.seg_ptr[b];
  const int n = a.meta.seg_ptr[b + 1] - s0;
  const int k = a.meta.topk[b];
  const int32_t* bnd = a.meta.seg_bounds + s0 + b;
  const int32_t* sel = a.sel + u * a.k_max;
  int carry = 0;
  for (int base = 0; base < k; base += 32) {
    const int j = base + lane;
    const int seg = j < k ? sel[j] : -1;
    const bool start = j < k && (j == 0 || sel[j - 1] != seg - 1);
    const bool last = j < k && (j == k - 1 || sel[j + 1] != seg + 1);
    const unsigned ms = __ballot_sync(kFullMask, start);
    const int rid = carry + __popc(ms & ((2u << lane) - 1u)) - 1;
    if (start) runs_s[rid] = bnd[seg];
    if (last) runs_e[rid] = bnd[seg + 1];
    carry += __popc(ms);
  }
  __syncwarp();
  int m = carry;
  const int Ns = a.meta.prompt_lens[b];  // the sink of a plan with one, else 0
  if (Ns > 0) {
    if (m > 0 && runs_s[0] <= Ns) {
      if (lane == 0) runs_s[0] = 0;  // the first segment (it begins at Ns) is selected: one run
    } else {
      for (int base = (m / 32) * 32; base >= 0; base -= 32) {
        const int r = base + lane;
        int s_ = 0, e_ = 0;
        if (r < m) {
          s_ = runs_s[r];
          e_ = runs_e[r];
        }
        __syncwarp();
        if (r < m) {
          runs_s[r + 1] = s_;
          runs_e[r + 1] = e_;
        }
        __syncwarp();
      }
      if (lane == 0) {
        runs_s[0] = 0;
        runs_e[0] = Ns;
      }
      ++m;
    }
    __syncwarp();
  }
  emit_ranges(a, runs_s, runs_e, 1, m, max(0, L - a.window), L, u, 1, n - k, nullptr, nullptr, lane);
}

}  // namespace

size_t vote_smem_bytes(int G, int d, int n_max) {
  return d == 64 ? VoteLayout<float, 64>::bytes(G, n_max) : VoteLayout<float, 128>::bytes(G, n_max);
}
size_t consensus_smem_bytes(int n_max) {
  return (static_cast<size_t>(n_max) + (n_max + 1) + (2 * n_max + 1) + 2 * (n_max + 2)) * sizeof(int);
}

zr_status launch_vote(const Plan& p, const StepArgs& a, const void* mean_keys, int32_t* votes, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 grid(p.Hkv, p.B), block(kVoteThreads);
  const size_t smem = vote_smem_bytes(p.G, p.d, p.n_max);
  cudaError_t e = cudaSuccess;
  if (p.cfg.dtype == ZR_BF16) {
    auto* mk = static_cast<const __nv_bfloat16*>(mean_keys);
    if (p.d == 64) {
      cudaFuncSetAttribute(zr_vote_kernel<__nv_bfloat16, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
      zr_vote_kernel<__nv_bfloat16, 64><<<grid, block, smem, s>>>(a, mk, votes);
    } else {
      cudaFuncSetAttribute(zr_vote_kernel<__nv_bfloat16, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
      zr_vote_kernel<__nv_bfloat16, 128><<<grid, block, smem, s>>>(a, mk, votes);
    }
  } else {
    auto* mk = static_cast<const float*>(mean_keys);
    if (p.d == 64) {
      cudaFuncSetAttribute(zr_vote_kernel<float, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
      zr_vote_kernel<float, 64><<<grid, block, smem, s>>>(a, mk, votes);
    } else {
      cudaFuncSetAttribute(zr_vote_kernel<float, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
      zr_vote_kernel<float, 128><<<grid, block, smem, s>>>(a, mk, votes);
    }
  }
  e = cudaGetLastError();
  return e == cudaSuccess ? ZR_OK : ZR_ECUDA;
}

zr_status launch_consensus(const Plan& p, const StepArgs& a, int32_t* votes, int32_t* votes_out, int32_t* ic_out,
                           void* stream) {
  const size_t smem = consensus_smem_bytes(p.n_max);
  cudaFuncSetAttribute(zr_consensus_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  zr_consensus_kernel<<<p.B, kConsensusThreads, smem, static_cast<cudaStream_t>(stream)>>>(a, votes, votes_out,
                                                                                           ic_out, p.c_max);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ECUDA;
}

zr_status launch_decode_advance(const Plan& p, const StepArgs& a, const int32_t* seq_lens, void* stream) {
  const size_t smem = 2 * static_cast<size_t>(p.k_max + 1) * sizeof(int);
  cudaFuncSetAttribute(zr_decode_advance_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  zr_decode_advance_kernel<<<dim3(p.Hkv, p.B), 32, smem, static_cast<cudaStream_t>(stream)>>>(a, seq_lens);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ECUDA;
}

zr_status launch_consensus_advance(const Plan& p, const StepArgs& a, const int32_t* seq_lens, void* stream) {
  zr_consensus_advance_kernel<<<p.B, 32, 0, static_cast<cudaStream_t>(stream)>>>(a, seq_lens);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ECUDA;
}

}  // namespace zr
