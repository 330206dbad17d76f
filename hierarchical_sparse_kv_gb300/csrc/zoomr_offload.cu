// The offloaded cache of the ZoomR page, 3.4 "System Implementation and Inference", "Decoding Stage":
// the full KV cache stays in host memory, and for every layer only the final context I_f is brought to
// the GPU, the next layer's blocks while the current one attends.
//
//   map    after a selection (or a window advance): every physical block that the workspace's current
//          token ranges touch, over all units of a sequence and each shared block once, gets a slot of
//          a staging pool in HBM (ascending physical order), and every (block, KV head) a mask of the
//          16 token rows that some range of that head covers. Writes the slot list, the sequences' block
//          tables remapped to slots (-1 for blocks no range touches) and the slot count; the row masks
//          stay in the workspace. Kernels: clear the per-block marks and masks, mark (one CTA per unit),
//          assign (one CTA, a scan over the pool), remap (one thread per table entry).
//   stage  one layer: the masked rows of every staged block (exactly the rows of I_f, per KV head)
//          copied from the pools in host memory into its slot, one CTA per (slot, pool), 16-byte
//          vectors, eight in flight per thread. Rows outside every range are not copied: the attention
//          never reads them.
//
// The attention then runs unchanged over the staging pools and the remapped tables.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "zoomr_internal.h"

namespace zr {
namespace {

constexpr int kMarkThreads = 256;
constexpr int kAssignThreads = 1024;
constexpr int kStageThreads = 256;
constexpr int kStageVecs = 8;  // 16-byte vectors in flight per thread
constexpr int kMaxStageHeads = 256;  // KV heads a staging copy takes (the plan's limit is lower)

__global__ void __launch_bounds__(256) zr_stage_clear_kernel(int32_t* __restrict__ marks, int n,
                                                              uint32_t* __restrict__ rows, int nrows) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) marks[i] = 0;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nrows; i += gridDim.x * blockDim.x) rows[i] = 0u;
}

// Unit (b, g): mark the physical block of every logical block its ranges touch, and OR into the block's
// row mask for KV head g the rows of each range piece inside it.
__global__ void __launch_bounds__(kMarkThreads) zr_stage_mark_kernel(StepArgs a, const int32_t* __restrict__ bt,
                                                                     int32_t* __restrict__ marks,
                                                                     uint32_t* __restrict__ rows) {
  const int g = blockIdx.x, b = blockIdx.y;
  const int u = b * a.Hkv + g;
  const int nr = a.unit_info[u].x;
  const int32_t* rg = a.ranges + static_cast<size_t>(u) * (a.k_max + 1) * 2;
  const int32_t* row = bt + static_cast<size_t>(b) * a.max_blocks;
  for (int r = 0; r < nr; ++r) {
    const int s = rg[2 * r], e = rg[2 * r + 1];
    if (e <= s) continue;
    const int b0 = s / kBlockTokens, b1 = min((e - 1) / kBlockTokens, a.max_blocks - 1);
    for (int j = b0 + threadIdx.x; j <= b1; j += kMarkThreads) {
      const int phys = row[j];
      if (static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks)) {
        marks[phys] = 1;
        const int lo = max(s - j * kBlockTokens, 0), hi = min(e - j * kBlockTokens, kBlockTokens);  // rows [lo, hi)
        atomicOr(&rows[static_cast<size_t>(phys) * a.Hkv + g], ((1u << hi) - 1u) & ~((1u << lo) - 1u));
      } else {
        atomicOr(a.err, kErrBadBlock);
      }
    }
  }
}

// One CTA: slots in ascending physical order. marks[p] becomes slot + 1 (or 0: not staged); stage_ids[slot]
// = p for slots below capacity; more marked blocks than capacity set kErrStage and leave the rest unstaged.
__global__ void __launch_bounds__(kAssignThreads) zr_stage_assign_kernel(StepArgs a, int32_t* __restrict__ marks,
                                                                         int32_t* __restrict__ stage_ids,
                                                                         int32_t* __restrict__ n_staged,
                                                                         int capacity) {
  __shared__ int wsum[kAssignThreads / 32];
  __shared__ int s_carry;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int nb = a.num_blocks;
  if (tid == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < nb; base += kAssignThreads) {
    const int p = base + tid;
    const int m = p < nb && marks[p] ? 1 : 0;
    int x = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[w] = x;
    __syncthreads();
    int before = s_carry, total = 0;
    for (int i = 0; i < kAssignThreads / 32; ++i) {
      before += i < w ? wsum[i] : 0;
      total += wsum[i];
    }
    const int slot = before + x - m;
    if (p < nb) {
      if (m && slot < capacity) {
        stage_ids[slot] = p;
        marks[p] = slot + 1;
      } else {
        marks[p] = 0;
      }
    }
    __syncthreads();  // every thread has read wsum and s_carry
    if (tid == 0) s_carry += total;
    __syncthreads();
  }
  if (tid == 0) {
    const int total = s_carry;
    *n_staged = total < capacity ? total : capacity;
    if (total > capacity) atomicOr(a.err, kErrStage);
  }
}

__global__ void __launch_bounds__(256) zr_stage_remap_kernel(StepArgs a, const int32_t* __restrict__ bt,
                                                             const int32_t* __restrict__ marks,
                                                             int32_t* __restrict__ remap) {
  const int n = a.B * a.max_blocks;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int phys = bt[i];
    remap[i] = static_cast<unsigned>(phys) < static_cast<unsigned>(a.num_blocks) ? marks[phys] - 1 : -1;
  }
}

// One CTA per (slot, pool): the masked rows of block stage_ids[slot] (row r of KV head h when bit r of
// rows[block * Hkv + h] is set; row_vecs 16-byte vectors a row) copied from the host pool into the slot,
// kStageVecs vectors in flight per thread. CTAs past *n_staged exit at once. Short-lived CTAs (no
// grid-stride loop) free their SM as soon as their block is done, so a layer's attention launched
// meanwhile on a higher-priority stream is not held back by the copy.
__global__ void __launch_bounds__(kStageThreads) zr_stage_copy_kernel(const uint4* __restrict__ hk,
                                                                      const uint4* __restrict__ hv,
                                                                      uint4* __restrict__ sk, uint4* __restrict__ sv,
                                                                      const int32_t* __restrict__ stage_ids,
                                                                      const int32_t* __restrict__ n_staged,
                                                                      const uint32_t* __restrict__ rows, int Hkv,
                                                                      int row_vecs) {
  __shared__ uint32_t s_rows[kMaxStageHeads];
  const int slot = blockIdx.x >> 1;
  if (slot >= *n_staged) return;
  const bool isv = blockIdx.x & 1;
  const int phys = stage_ids[slot];
  for (int h = threadIdx.x; h < Hkv; h += kStageThreads) s_rows[h] = rows[static_cast<size_t>(phys) * Hkv + h];
  __syncthreads();
  const int block_vecs = Hkv * kBlockTokens * row_vecs;
  const uint4* src = (isv ? hv : hk) + static_cast<long long>(phys) * block_vecs;
  uint4* dst = (isv ? sv : sk) + static_cast<long long>(slot) * block_vecs;
  for (int base = threadIdx.x; base < block_vecs; base += kStageThreads * kStageVecs) {
    uint4 v[kStageVecs];
    bool take[kStageVecs];
#pragma unroll
    for (int k = 0; k < kStageVecs; ++k) {
      const int i = base + k * kStageThreads;
      const int r = i / row_vecs;  // token row (head-major): head r / 16, slot r % 16
      take[k] = i < block_vecs && ((s_rows[r / kBlockTokens] >> (r % kBlockTokens)) & 1u);
      if (take[k]) v[k] = src[i];
    }
#pragma unroll
    for (int k = 0; k < kStageVecs; ++k) {
      const int i = base + k * kStageThreads;
      if (take[k]) dst[i] = v[k];
    }
  }
}

}  // namespace
}  // namespace zr

extern "C" {

zr_status zr_offload_map(zr_plan_t plan, void* workspace, const int32_t* block_tables, int32_t capacity,
                         int32_t* stage_ids, int32_t* remap_tables, int32_t* n_staged, void* stream) {
  if (!plan || !workspace || !block_tables || !stage_ids || !remap_tables || !n_staged || capacity < 1)
    return ZR_EINVAL;
  const zr::Plan& p = plan->p;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  zr::StepArgs a = zr::step_args(p, workspace);
  int32_t* marks = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + p.ws.stage_marks);
  uint32_t* rows = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + p.ws.stage_rows);
  const int nrows = p.num_blocks * p.Hkv;
  zr::zr_stage_clear_kernel<<<(nrows + 255) / 256 < 1024 ? (nrows + 255) / 256 : 1024, 256, 0, s>>>(
      marks, p.num_blocks, rows, nrows);
  zr::zr_stage_mark_kernel<<<dim3(p.Hkv, p.B), zr::kMarkThreads, 0, s>>>(a, block_tables, marks, rows);
  zr::zr_stage_assign_kernel<<<1, zr::kAssignThreads, 0, s>>>(a, marks, stage_ids, n_staged, capacity);
  const int entries = p.B * p.max_blocks;
  zr::zr_stage_remap_kernel<<<(entries + 255) / 256 < 1024 ? (entries + 255) / 256 : 1024, 256, 0, s>>>(
      a, block_tables, marks, remap_tables);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ECUDA;
}

zr_status zr_offload_stage(zr_plan_t plan, const void* workspace, const void* host_k_pool, const void* host_v_pool,
                           const int32_t* stage_ids, const int32_t* n_staged, int32_t capacity, void* stage_k,
                           void* stage_v, void* stream) {
  if (!plan || !workspace || !host_k_pool || !host_v_pool || !stage_ids || !n_staged || !stage_k || !stage_v ||
      capacity < 1)
    return ZR_EINVAL;
  const zr::Plan& p = plan->p;
  if (p.Hkv > zr::kMaxStageHeads) return ZR_EUNSUPPORTED;
  const size_t eb = p.cfg.dtype == ZR_BF16 ? 2 : 4;
  const size_t row_bytes = static_cast<size_t>(p.d) * eb;
  for (const void* q : {host_k_pool, host_v_pool, static_cast<const void*>(stage_k), static_cast<const void*>(stage_v)})
    if (reinterpret_cast<uintptr_t>(q) % 16 != 0) return ZR_EINVAL;
  if (row_bytes % 16 != 0) return ZR_EINVAL;
  const uint32_t* rows =
      reinterpret_cast<const uint32_t*>(static_cast<const char*>(workspace) + p.ws.stage_rows);
  // Two CTAs per slot (K and V); slots past *n_staged return at once.
  zr::zr_stage_copy_kernel<<<2 * capacity, zr::kStageThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(host_k_pool), static_cast<const uint4*>(host_v_pool), static_cast<uint4*>(stage_k),
      static_cast<uint4*>(stage_v), stage_ids, n_staged, rows, p.Hkv, static_cast<int>(row_bytes / 16));
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ECUDA;
}

}  // extern "C"
