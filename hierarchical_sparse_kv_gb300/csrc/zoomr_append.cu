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
// function of the stored rows and the segment bounds.

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

// One warp per (segment, KV head): K and V means of tokens [s, e). Rows are
// loaded kSumInFlight tokens ahead and added strictly in token order.
template <typename T, int D>
__global__ void __launch_bounds__(kSumWarps * 32) zr_segment_summaries_kernel(
    const int4* __restrict__ segs, int n, const int32_t* __restrict__ block_tables, const T* __restrict__ k_pool,
    const T* __restrict__ v_pool, T* __restrict__ sum_k, T* __restrict__ sum_v, int num_rows, int32_t* err, int B,
    int Hkv, int num_blocks, int max_blocks) {
  constexpr int C = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kSumWarps + (threadIdx.x >> 5);
  if (item >= static_cast<int64_t>(n) * Hkv) return;
  const int si = static_cast<int>(item / Hkv);
  const int g = static_cast<int>(item - static_cast<int64_t>(si) * Hkv);
  const int4 sg = segs[si];
  const int b = sg.x, s = sg.y, e = sg.z, r = sg.w;
  if (b < 0 || b >= B || s < 0 || e <= s || e > max_blocks * kBlockTokens || r < 0 || r >= num_rows) {
    if (lane == 0 && g == 0) report(err, kErrBadIndex);
    return;
  }
  const int32_t* bt = block_tables + static_cast<size_t>(b) * max_blocks;
  double ak[C], av[C];
#pragma unroll
  for (int i = 0; i < C; ++i) ak[i] = av[i] = 0.0;
  bool bad = false;
  for (int t0 = s; t0 < e; t0 += kSumInFlight) {
    Slice<T, D> kr[kSumInFlight], vr[kSumInFlight];
#pragma unroll
    for (int j = 0; j < kSumInFlight; ++j) {
      const int t = t0 + j;
      if (t < e) {
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
    if (bad) break;
#pragma unroll
    for (int j = 0; j < kSumInFlight; ++j) {
      if (t0 + j < e) {
#pragma unroll
        for (int i = 0; i < C; ++i) {
          ak[i] = __dadd_rn(ak[i], comp<T, D>(kr[j], i));
          av[i] = __dadd_rn(av[i], comp<T, D>(vr[j], i));
        }
      }
    }
  }
  if (bad) {
    if (lane == 0) report(err, kErrBadBlock);
    return;
  }
  const double cnt = static_cast<double>(e - s);
#pragma unroll
  for (int i = 0; i < C; ++i) {
    ak[i] = __ddiv_rn(ak[i], cnt);
    av[i] = __ddiv_rn(av[i], cnt);
  }
  const size_t out = (static_cast<size_t>(r) * Hkv + g) * D;
  store_slice<T, D>(sum_k + out, lane, pack_means<T, D>(ak));
  store_slice<T, D>(sum_v + out, lane, pack_means<T, D>(av));
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
  const int64_t items = static_cast<int64_t>(n) * c.num_kv_heads;
  const unsigned grid = static_cast<unsigned>((items + kSumWarps - 1) / kSumWarps);
  zr_segment_summaries_kernel<T, D><<<grid, kSumWarps * 32, 0, s>>>(
      reinterpret_cast<const int4*>(segs), n, block_tables, static_cast<const T*>(k_pool),
      static_cast<const T*>(v_pool), static_cast<T*>(sum_k), static_cast<T*>(sum_v), num_rows, err, c.batch,
      c.num_kv_heads, c.num_blocks, c.max_blocks_per_seq);
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
  const int64_t grid = (static_cast<int64_t>(n) * cfg->num_kv_heads + zr::kSumWarps - 1) / zr::kSumWarps;
  if (grid > 0x7FFFFFFF) return ZR_EUNSUPPORTED;
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
