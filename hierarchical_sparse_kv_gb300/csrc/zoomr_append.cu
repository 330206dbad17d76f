// Append path of the paged KV cache: token-row writes, batched block copies
// and the mean summary rows of completed segments.
//
//   zr_append_kv          "KV-cache management", "Paged KV cache (PagedAttention)":
//                         token t of sequence b is stored in physical block
//                         block_tables[b][t / 16], slot t % 16, every KV head.
//   zr_copy_blocks        "KV-cache management", "Block sharing with reference
//                         counts and copy-on-write": a shared last block is
//                         copied whole before the sequence writes into it.
//   zr_segment_summaries  ZoomR page, 3.3 "Representing Context with Mean Summary
//                         Keys": a segment's summary key is the mean of its
//                         tokens' key rows (per KV head); the summary value row
//                         is the same mean over the V rows.
//
// All three are bandwidth- or latency-bound copies and reductions: no tensor
// cores. Each checks every index it reads against the config and skips (and
// reports in the optional error word) what falls outside; none traps.
//
// Summary precision: each component is accumulated in fp64 in ascending token
// order starting from +0.0, divided by the token count in fp64 (IEEE, round to
// nearest), then rounded to fp32 and then to the storage dtype, each to nearest
// even. bf16 and fp32 rows convert to fp64 exactly, so the result is a pure
// function of the stored rows and the segment bounds. fp32 rows are summed that
// way; bf16 rows are summed exactly in int64 fixed point, which gives the same
// bits whenever the values fit a window where the fp64 sum is exact too, and
// fall back to the fp64 loop otherwise (see the exact kernel below).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "zoomr_internal.h"

namespace zr {
namespace {

constexpr int kAppendThreads = 128;
constexpr int kCopyThreads = 256;
constexpr int kSumWarps = 4;       // (segment, head) items per summary CTA, one warp each
constexpr int kSumInFlight = 8;    // token rows loaded ahead of the in-order fp64 adds

__device__ __forceinline__ void report(int32_t* err, int32_t bit) {
  if (err) atomicOr(err, bit);
}

// One 16-byte vector per thread-iteration; the new rows of sequence b are
// Hkv * d elements of K then the same of V.
__global__ void __launch_bounds__(kAppendThreads) zr_append_kernel(
    const int32_t* __restrict__ positions, const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int32_t* __restrict__ block_tables, uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
    int32_t* err, int Hkv, int row_vecs, int num_blocks, int max_blocks) {
  const int b = blockIdx.x;
  const int t = positions[b];
  if (t < 0) return;
  if (t >= max_blocks * kBlockTokens) {
    if (threadIdx.x == 0) report(err, kErrBadIndex);
    return;
  }
  const int blk = block_tables[static_cast<size_t>(b) * max_blocks + t / kBlockTokens];
  if (blk < 0 || blk >= num_blocks) {
    if (threadIdx.x == 0) report(err, kErrBadBlock);
    return;
  }
  const int slot = t % kBlockTokens;
  const int per_pool = Hkv * row_vecs;
  for (int i = threadIdx.x; i < 2 * per_pool; i += kAppendThreads) {
    const bool is_v = i >= per_pool;
    const int j = is_v ? i - per_pool : i;
    const int g = j / row_vecs;
    const int c = j - g * row_vecs;
    const size_t src = (static_cast<size_t>(b) * Hkv + g) * row_vecs + c;
    const size_t dst = ((static_cast<size_t>(blk) * Hkv + g) * kBlockTokens + slot) * row_vecs + c;
    if (is_v)
      v_pool[dst] = v_new[src];
    else
      k_pool[dst] = k_new[src];
  }
}

// blockIdx.x = pair, blockIdx.y = 0 (K) or 1 (V); block_vecs 16-byte vectors per block.
__global__ void __launch_bounds__(kCopyThreads) zr_copy_blocks_kernel(
    const int32_t* __restrict__ pairs, uint4* k_pool, uint4* v_pool, int32_t* err, int block_vecs,
    int num_blocks) {
  const int src = pairs[2 * static_cast<size_t>(blockIdx.x)];
  const int dst = pairs[2 * static_cast<size_t>(blockIdx.x) + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) report(err, kErrBadBlock);
    return;
  }
  uint4* pool = blockIdx.y ? v_pool : k_pool;
  const uint4* s = pool + static_cast<size_t>(src) * block_vecs;
  uint4* d = pool + static_cast<size_t>(dst) * block_vecs;
  for (int i = threadIdx.x; i < block_vecs; i += kCopyThreads) d[i] = s[i];
}

// Per-lane slice of a row: D / 32 consecutive components, W 32-bit words.
template <typename T, int D>
struct Slice {
  static constexpr int kComp = D / 32;
  static constexpr int kWords = kComp * static_cast<int>(sizeof(T)) / 4;
  uint32_t w[kWords];
};

template <typename T, int D>
__device__ __forceinline__ Slice<T, D> load_slice(const T* row, int lane) {
  Slice<T, D> s;
  const char* p = reinterpret_cast<const char*>(row) + static_cast<size_t>(lane) * sizeof(s.w);
  if constexpr (Slice<T, D>::kWords == 1) {
    s.w[0] = __ldg(reinterpret_cast<const unsigned int*>(p));
  } else if constexpr (Slice<T, D>::kWords == 2) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    s.w[0] = v.x; s.w[1] = v.y;
  } else {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    s.w[0] = v.x; s.w[1] = v.y; s.w[2] = v.z; s.w[3] = v.w;
  }
  return s;
}

template <typename T, int D>
__device__ __forceinline__ void store_slice(T* row, int lane, const Slice<T, D>& s) {
  char* p = reinterpret_cast<char*>(row) + static_cast<size_t>(lane) * sizeof(s.w);
  if constexpr (Slice<T, D>::kWords == 1) {
    *reinterpret_cast<unsigned int*>(p) = s.w[0];
  } else if constexpr (Slice<T, D>::kWords == 2) {
    *reinterpret_cast<uint2*>(p) = make_uint2(s.w[0], s.w[1]);
  } else {
    *reinterpret_cast<uint4*>(p) = make_uint4(s.w[0], s.w[1], s.w[2], s.w[3]);
  }
}

// Component i of a slice as an exact fp64 value.
template <typename T, int D>
__device__ __forceinline__ double comp(const Slice<T, D>& s, int i) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t word = s.w[i >> 1];
    const uint32_t bits = (i & 1) ? (word & 0xFFFF0000u) : (word << 16);
    return static_cast<double>(__uint_as_float(bits));
  } else {
    return static_cast<double>(__uint_as_float(s.w[i]));
  }
}

// Rounds fp64 means to fp32, then to T, into a slice.
template <typename T, int D>
__device__ __forceinline__ Slice<T, D> pack_means(const double (&m)[D / 32]) {
  Slice<T, D> s;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    const float f = __double2float_rn(m[i]);
    if constexpr (sizeof(T) == 2) {
      const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(f));
      if (i & 1)
        s.w[i >> 1] |= h << 16;
      else
        s.w[i >> 1] = h;
    } else {
      s.w[i] = __float_as_uint(f);
    }
  }
  return s;
}

// One (segment, head) item of a summary launch, validated: tokens [s, e) of
// sequence b, output row r. Returns false (and reports) for a bad index.
struct SegItem {
  int b, s, e, r;
};

__device__ __forceinline__ bool check_item(const int4 sg, int B, int max_blocks, int num_rows, int32_t* err,
                                           bool reporter) {
  if (sg.x < 0 || sg.x >= B || sg.y < 0 || sg.z <= sg.y || sg.z > max_blocks * kBlockTokens || sg.w < 0 ||
      sg.w >= num_rows) {
    if (reporter) report(err, kErrBadIndex);
    return false;
  }
  return true;
}

// The definition, literally: one warp adds the lane's components of tokens
// s, s+1, ..., e-1 in fp64, in that order, starting from +0.0. Rows are loaded
// kSumInFlight tokens ahead. Returns false if a block id is outside the pool.
template <typename T, int D>
__device__ bool seq_sums(const SegItem& it, int g, int lane, const int32_t* bt, const T* __restrict__ k_pool,
                         const T* __restrict__ v_pool, int Hkv, int num_blocks, double (&ak)[D / 32],
                         double (&av)[D / 32]) {
  constexpr int C = D / 32;
#pragma unroll
  for (int i = 0; i < C; ++i) ak[i] = av[i] = 0.0;
  for (int t0 = it.s; t0 < it.e; t0 += kSumInFlight) {
    Slice<T, D> kr[kSumInFlight], vr[kSumInFlight];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kSumInFlight; ++j) {
      const int t = t0 + j;
      if (t < it.e) {
        const int blk = bt[t / kBlockTokens];
        if (blk < 0 || blk >= num_blocks) {
          bad = true;
        } else {
          const size_t row = ((static_cast<size_t>(blk) * Hkv + g) * kBlockTokens + t % kBlockTokens) * D;
          kr[j] = load_slice<T, D>(k_pool + row, lane);
          vr[j] = load_slice<T, D>(v_pool + row, lane);
        }
      }
    }
    if (bad) return false;
#pragma unroll
    for (int j = 0; j < kSumInFlight; ++j) {
      if (t0 + j < it.e) {
#pragma unroll
        for (int i = 0; i < C; ++i) {
          ak[i] = __dadd_rn(ak[i], comp<T, D>(kr[j], i));
          av[i] = __dadd_rn(av[i], comp<T, D>(vr[j], i));
        }
      }
    }
  }
  return true;
}

// Divides the fp64 sums by the token count (IEEE, nearest) and stores the
// rounded means of the lane's components into row r of both summary tensors.
template <typename T, int D>
__device__ __forceinline__ void store_means(const SegItem& it, int g, int lane, int Hkv, double (&ak)[D / 32],
                                            double (&av)[D / 32], T* __restrict__ sum_k, T* __restrict__ sum_v) {
  const double cnt = static_cast<double>(it.e - it.s);
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    ak[i] = __ddiv_rn(ak[i], cnt);
    av[i] = __ddiv_rn(av[i], cnt);
  }
  const size_t out = (static_cast<size_t>(it.r) * Hkv + g) * D;
  store_slice<T, D>(sum_k + out, lane, pack_means<T, D>(ak));
  store_slice<T, D>(sum_v + out, lane, pack_means<T, D>(av));
}

// fp32 rows: one warp per (segment, head) item, the definition as written.
template <typename T, int D>
__global__ void __launch_bounds__(kSumWarps * 32) zr_summaries_seq_kernel(
    const int4* __restrict__ segs, int n, const int32_t* __restrict__ block_tables, const T* __restrict__ k_pool,
    const T* __restrict__ v_pool, T* __restrict__ sum_k, T* __restrict__ sum_v, int num_rows, int32_t* err, int B,
    int Hkv, int num_blocks, int max_blocks) {
  const int lane = threadIdx.x & 31;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kSumWarps + (threadIdx.x >> 5);
  if (item >= static_cast<int64_t>(n) * Hkv) return;
  const int si = static_cast<int>(item / Hkv);
  const int g = static_cast<int>(item - static_cast<int64_t>(si) * Hkv);
  const int4 sg = segs[si];
  if (!check_item(sg, B, max_blocks, num_rows, err, lane == 0 && g == 0)) return;
  const SegItem it{sg.x, sg.y, sg.z, sg.w};
  double ak[D / 32], av[D / 32];
  if (!seq_sums<T, D>(it, g, lane, block_tables + static_cast<size_t>(it.b) * max_blocks, k_pool, v_pool, Hkv,
                      num_blocks, ak, av)) {
    if (lane == 0) report(err, kErrBadBlock);
    return;
  }
  store_means<T, D>(it, g, lane, Hkv, ak, av, sum_k, sum_v);
}

// ---- bf16 rows: exact fixed-point sums, any order
//
// For a segment of n tokens let lg = ceil(log2 n) and F = 33 for lg <= 10,
// F = 43 - lg above. Every bf16 value x with 2^(7-F) <= |x| < 2^10 has all its
// bits at or above 2^-F, so y = x * 2^F is an integer with |y| < 2^Y,
// Y = min(43, 53 - lg). Every partial sum of such values, in any order, is then
// an integer multiple of 2^-F below 2^53 of those units: it is exact in an
// int64 and, equally, each fp64 addition of the definition's in-order loop is
// exact, so both give the same sum.
//
// Per value, fp32 magic-constant steps split y into hi (a multiple of 2^22,
// |hi| <= 2^43) and lo = y - hi (|lo| <= 2^21) and leave hi / 2^22 and lo as
// the low bits of two floats with fixed exponents:
//   t  = x * 2^F + M_hi               = M_hi + hi
//   t2 = x * 2^F + ((M_hi + M_lo) - t) = M_lo + lo
// (M_hi + M_lo is exact in fp32, and so is the subtraction). Adding those
// floats' bit patterns in int32 sums hi / 2^22 and lo plus a known multiple of
// the constants' own bits, removed when the int32 sums are folded into int64
// totals (every 256 values, far below int32 overflow). The window is checked
// once per chain from the running smallest nonzero |x| and the largest |x|
// (NaN-propagating); zeros are exact and pass. A segment with any value outside
// it (tiny, subnormal, large, not finite) falls back to the fp64 in-order loop,
// so the result is the definition's in every case.
constexpr float kMagicHi = 0x1.8p45f;     // 1.5 * 2^45: ulp 2^22 in [2^45, 2^46)
constexpr float kMagicLo = 0x1.8p23f;     // 1.5 * 2^23: ulp 1 in [2^23, 2^24)
constexpr float kMagicSum = 0x1.800006p45f;  // kMagicHi + kMagicLo, exact
constexpr float kExactMax = 1024.0f;      // |x| < 2^10

__device__ __forceinline__ int exact_shift(int n) {
  const int lg = n > 1 ? 32 - __clz(n - 1) : 0;  // ceil(log2 n)
  return lg <= 10 ? 33 : 43 - lg;
}

struct ExactChain {
  uint32_t hi = 0u, lo = 0u;  // int32 sums of the split floats' bit patterns
  long long total = 0;        // folded sum of y
};

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// mnk tracks the smallest nonzero |x| as the key bits(x) * 2 - 2 (unsigned): the
// sign bit drops out, +-0 maps to the largest key, and the order of nonzero
// magnitudes is kept.
__device__ __forceinline__ void exact_add(float x, float scale, ExactChain& c, uint32_t& mnk, float& mx) {
  const float t = fmaf(x, scale, kMagicHi);
  const float t2 = fmaf(x, scale, __fsub_rn(kMagicSum, t));
  mnk = min(mnk, __float_as_uint(x) * 2u - 2u);
  mx = max_nan(mx, fabsf(x));
  c.hi += __float_as_uint(t);
  c.lo += __float_as_uint(t2);
}

// Adds the int32 sums of k values into the total and restarts them.
__device__ __forceinline__ void exact_fold(ExactChain& c, uint32_t k) {
  const int h = static_cast<int>(c.hi - k * __float_as_uint(kMagicHi));
  const int l = static_cast<int>(c.lo - k * __float_as_uint(kMagicLo));
  c.total += static_cast<long long>(h) * (1ll << 22) + l;
  c.hi = c.lo = 0u;
}

// True when every value seen lies in the exact window of shift F.
__device__ __forceinline__ bool exact_window_ok(uint32_t mnk, float mx, int F) {
  const uint32_t lo = static_cast<uint32_t>(127 + 7 - F) << 23;  // bits of 2^(7-F)
  return mnk >= lo * 2u - 2u && mx < kExactMax;  // false for NaN
}

// Rounds one fp64 sum / count to T and stores it.
template <typename T>
__device__ __forceinline__ void store_mean(T* dst, double sum, int count) {
  const float f = __double2float_rn(__ddiv_rn(sum, static_cast<double>(count)));
  if constexpr (sizeof(T) == 2)
    *dst = __float2bfloat16_rn(f);
  else
    *dst = f;
}

// 16-byte cp.async into shared memory; src_bytes 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

constexpr int kExactStages = 8;         // cp.async ring depth, in paged blocks
constexpr int kExactTableSlots = 1024;  // block-table entries staged in shared memory (16K tokens)

// One CTA of 4 D threads per (segment, KV head). A paged block holds the
// head's 16 rows as one contiguous 16 x D chunk per pool; thread i works on
// pool i / (2 D) (K, then V) and owns 16-byte vector i % (2 D) of that chunk
// (row (i % 2D) / (D/8), components 8 (i % (D/8)) .. + 7). It streams that
// vector of every block the segment touches through its own slots of a
// kExactStages-deep cp.async ring (rows outside the segment are zero-filled,
// not read), adds it, and keeps its folded int64 sums in its own shared-memory
// slots; the 16 row groups are reduced there at the end. Each thread reads
// back only what it copied itself, so the ring needs no CTA barrier.
template <int D>
__global__ void __launch_bounds__(4 * D, 2) zr_summaries_exact_kernel(
    const int4* __restrict__ segs, int n, const int32_t* __restrict__ block_tables,
    const __nv_bfloat16* __restrict__ k_pool, const __nv_bfloat16* __restrict__ v_pool,
    __nv_bfloat16* __restrict__ sum_k, __nv_bfloat16* __restrict__ sum_v, int num_rows, int32_t* err, int B,
    int Hkv, int num_blocks, int max_blocks) {
  using T = __nv_bfloat16;
  constexpr int NT = 4 * D;   // threads
  constexpr int VPR = D / 8;  // 16-byte vectors per row
  extern __shared__ uint4 ring[];  // [kExactStages][NT]
  __shared__ long long red[kBlockTokens][2 * D];
  __shared__ int32_t sbt[kExactTableSlots];  // the segment's block-table entries, from its first block on
  __shared__ uint32_t flags;  // bit 0 outside the exact window, bit 1 bad block
  const int tid = threadIdx.x;
  const int is_v = tid >= 2 * D;
  const int q = tid - is_v * 2 * D;
  const int row = q / VPR, vec = q % VPR;
  long long* slot = &red[row][is_v * D + 8 * vec];
  const int si = static_cast<int>(blockIdx.x / Hkv);
  const int g = static_cast<int>(blockIdx.x - static_cast<unsigned>(si) * Hkv);
  const int4 sg = segs[si];
  if (!check_item(sg, B, max_blocks, num_rows, err, tid == 0 && g == 0)) return;
  const SegItem it{sg.x, sg.y, sg.z, sg.w};
  if (tid == 0) flags = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) slot[i] = 0;
  const int32_t* bt = block_tables + static_cast<size_t>(it.b) * max_blocks;
  const uint4* pool = reinterpret_cast<const uint4*>(is_v ? v_pool : k_pool);
  const int j0 = it.s / kBlockTokens, j1 = (it.e - 1) / kBlockTokens;
  for (int j = j0 + tid; j <= j1 && j - j0 < kExactTableSlots; j += NT) sbt[j - j0] = bt[j];
  __syncthreads();
  uint32_t bad = 0u;
  // stage paged block j (a block index of the sequence) into ring slot st
  auto issue = [&](int j, int st) {
    const int t = j * kBlockTokens + row;
    const uint4* src = pool;
    int bytes = 0;
    if (j <= j1 && t >= it.s && t < it.e) {
      const int blk = j - j0 < kExactTableSlots ? sbt[j - j0] : bt[j];
      if (blk < 0 || blk >= num_blocks) {
        bad = 1u;
      } else {
        src = pool + ((static_cast<size_t>(blk) * Hkv + g) * kBlockTokens + row) * VPR + vec;
        bytes = 16;
      }
    }
    cp_async16(&ring[st * NT + tid], src, bytes);
    cp_async_commit();
  };
#pragma unroll
  for (int p = 0; p < kExactStages - 1; ++p) issue(j0 + p, p);
  const int F = exact_shift(it.e - it.s);
  const float scale = __int_as_float((127 + F) << 23);  // 2^F
  ExactChain ch[8];
  uint32_t mnk = 0xFFFFFFFFu;
  float mx = 0.0f;
  int since_fold = 0;
  for (int k = 0; j0 + k <= j1; ++k) {
    cp_async_wait<kExactStages - 2>();
    const uint4 xv = ring[(k % kExactStages) * NT + tid];
    issue(j0 + k + kExactStages - 1, (k + kExactStages - 1) % kExactStages);
    const int t = (j0 + k) * kBlockTokens + row;
    if (t < it.s || t >= it.e) continue;  // this thread's row is not in the segment for this block
    const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      exact_add(__uint_as_float(w[x] << 16), scale, ch[2 * x], mnk, mx);
      exact_add(__uint_as_float(w[x] & 0xFFFF0000u), scale, ch[2 * x + 1], mnk, mx);
    }
    if (++since_fold == 256) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        exact_fold(ch[i], 256u);
        slot[i] += ch[i].total;
        ch[i].total = 0;
      }
      since_fold = 0;
    }
  }
  cp_async_wait<0>();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    exact_fold(ch[i], static_cast<uint32_t>(since_fold));
    slot[i] += ch[i].total;
  }
  const uint32_t out = exact_window_ok(mnk, mx, F) ? 0u : 1u;
  if (out | bad) atomicOr(&flags, out | (bad << 1));
  __syncthreads();
  const uint32_t f = flags;
  if (f & 2u) {
    if (tid == 0) report(err, kErrBadBlock);
    return;
  }
  if (f & 1u) {
    // some value lies outside the exact window: the definition's own loop, in token order
    if (tid >= 32) return;
    double mk[D / 32], mv[D / 32];
    seq_sums<T, D>(it, g, tid, bt, k_pool, v_pool, Hkv, num_blocks, mk, mv);
    store_means<T, D>(it, g, tid, Hkv, mk, mv, sum_k, sum_v);
    return;
  }
  if (tid >= 2 * D) return;
  long long sum = 0;
#pragma unroll
  for (int r = 0; r < kBlockTokens; ++r) sum += red[r][tid];
  const double unit = __longlong_as_double(static_cast<long long>(1023 - F) << 52);  // 2^-F
  const int c = tid < D ? tid : tid - D;
  T* dst = (tid < D ? sum_k : sum_v) + (static_cast<size_t>(it.r) * Hkv + g) * D + c;
  store_mean<T>(dst, static_cast<double>(sum) * unit, it.e - it.s);  // |sum| < 2^53: exact
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_bytes(const zr_config& c) { return c.dtype == ZR_BF16 ? 2 : 4; }

zr_status check_cache_config(const zr_config* c) {
  if (!c) return ZR_EINVAL;
  if (c->batch < 1 || c->num_kv_heads < 1 || c->block_size != kBlockTokens) return ZR_EINVAL;
  if (c->num_blocks < 1 || c->max_blocks_per_seq < 1) return ZR_EINVAL;
  if (c->dtype != ZR_F32 && c->dtype != ZR_BF16) return ZR_EINVAL;
  if (c->head_dim != 64 && c->head_dim != 128) return c->head_dim < 1 ? ZR_EINVAL : ZR_EUNSUPPORTED;
  if (static_cast<int64_t>(c->num_blocks) * c->num_kv_heads * kBlockTokens >= (int64_t(1) << 31))
    return ZR_EUNSUPPORTED;
  if (static_cast<int64_t>(c->max_blocks_per_seq) * kBlockTokens >= (int64_t(1) << 31)) return ZR_EUNSUPPORTED;
  return ZR_OK;
}

zr_status launched() {
  if (cudaGetLastError() != cudaSuccess) return ZR_ECUDA;
  return ZR_OK;
}

template <typename T, int D>
void launch_summaries(const zr_config& c, const int32_t* segs, int32_t n, const int32_t* block_tables,
                      const void* k_pool, const void* v_pool, void* sum_k, void* sum_v, int32_t num_rows,
                      int32_t* err, cudaStream_t s) {
  const int4* sg = reinterpret_cast<const int4*>(segs);
  if constexpr (sizeof(T) == 2) {
    const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(n) * c.num_kv_heads);
    const size_t ring = static_cast<size_t>(kExactStages) * 4 * D * sizeof(uint4);
    cudaFuncSetAttribute(zr_summaries_exact_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(ring));
    zr_summaries_exact_kernel<D><<<grid, 4 * D, ring, s>>>(
        sg, n, block_tables, static_cast<const T*>(k_pool), static_cast<const T*>(v_pool), static_cast<T*>(sum_k),
        static_cast<T*>(sum_v), num_rows, err, c.batch, c.num_kv_heads, c.num_blocks, c.max_blocks_per_seq);
  } else {
    const int64_t items = static_cast<int64_t>(n) * c.num_kv_heads;
    const unsigned grid = static_cast<unsigned>((items + kSumWarps - 1) / kSumWarps);
    zr_summaries_seq_kernel<T, D><<<grid, kSumWarps * 32, 0, s>>>(
        sg, n, block_tables, static_cast<const T*>(k_pool), static_cast<const T*>(v_pool), static_cast<T*>(sum_k),
        static_cast<T*>(sum_v), num_rows, err, c.batch, c.num_kv_heads, c.num_blocks, c.max_blocks_per_seq);
  }
}

}  // namespace
}  // namespace zr

extern "C" {

zr_status zr_append_kv(const zr_config* cfg, const int32_t* positions, const void* k_new, const void* v_new,
                       const int32_t* block_tables, void* k_pool, void* v_pool, int32_t* err, void* stream) {
  const zr_status st = zr::check_cache_config(cfg);
  if (st != ZR_OK) return st;
  if (!positions || !k_new || !v_new || !block_tables || !k_pool || !v_pool) return ZR_EINVAL;
  if (!zr::aligned16(k_new) || !zr::aligned16(v_new) || !zr::aligned16(k_pool) || !zr::aligned16(v_pool))
    return ZR_EINVAL;
  const int row_vecs = static_cast<int>(cfg->head_dim * zr::elem_bytes(*cfg) / 16);
  zr::zr_append_kernel<<<cfg->batch, zr::kAppendThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      positions, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), block_tables,
      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), err, cfg->num_kv_heads, row_vecs, cfg->num_blocks,
      cfg->max_blocks_per_seq);
  return zr::launched();
}

zr_status zr_copy_blocks(const zr_config* cfg, const int32_t* pairs, int32_t n, void* k_pool, void* v_pool,
                         int32_t* err, void* stream) {
  const zr_status st = zr::check_cache_config(cfg);
  if (st != ZR_OK) return st;
  if (n < 0 || !k_pool || !v_pool || (n > 0 && !pairs)) return ZR_EINVAL;
  if (!zr::aligned16(k_pool) || !zr::aligned16(v_pool)) return ZR_EINVAL;
  if (n == 0) return ZR_OK;
  const int block_vecs =
      static_cast<int>(static_cast<size_t>(cfg->num_kv_heads) * zr::kBlockTokens * cfg->head_dim * zr::elem_bytes(*cfg) / 16);
  zr::zr_copy_blocks_kernel<<<dim3(static_cast<unsigned>(n), 2), zr::kCopyThreads, 0,
                              static_cast<cudaStream_t>(stream)>>>(pairs, static_cast<uint4*>(k_pool),
                                                                   static_cast<uint4*>(v_pool), err, block_vecs,
                                                                   cfg->num_blocks);
  return zr::launched();
}

zr_status zr_segment_summaries(const zr_config* cfg, const int32_t* segs, int32_t n, const int32_t* block_tables,
                               const void* k_pool, const void* v_pool, void* sum_k, void* sum_v, int32_t num_rows,
                               int32_t* err, void* stream) {
  const zr_status st = zr::check_cache_config(cfg);
  if (st != ZR_OK) return st;
  if (n < 0 || num_rows < 0 || !block_tables || !k_pool || !v_pool || !sum_k || !sum_v || (n > 0 && !segs))
    return ZR_EINVAL;
  if (!zr::aligned16(segs) || !zr::aligned16(k_pool) || !zr::aligned16(v_pool) || !zr::aligned16(sum_k) ||
      !zr::aligned16(sum_v))
    return ZR_EINVAL;
  if (n == 0) return ZR_OK;
  if (static_cast<int64_t>(n) * cfg->num_kv_heads > 0x7FFFFFFF) return ZR_EUNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf16 = cfg->dtype == ZR_BF16;
  if (cfg->head_dim == 128) {
    if (bf16)
      zr::launch_summaries<__nv_bfloat16, 128>(*cfg, segs, n, block_tables, k_pool, v_pool, sum_k, sum_v, num_rows,
                                               err, s);
    else
      zr::launch_summaries<float, 128>(*cfg, segs, n, block_tables, k_pool, v_pool, sum_k, sum_v, num_rows, err, s);
  } else {
    if (bf16)
      zr::launch_summaries<__nv_bfloat16, 64>(*cfg, segs, n, block_tables, k_pool, v_pool, sum_k, sum_v, num_rows,
                                              err, s);
    else
      zr::launch_summaries<float, 64>(*cfg, segs, n, block_tables, k_pool, v_pool, sum_k, sum_v, num_rows, err, s);
  }
  return zr::launched();
}

}  // extern "C"
