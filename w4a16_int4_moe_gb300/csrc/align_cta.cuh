// align_cta.cuh -- moe_align_block_size by one CTA of kAlignThreads threads,
// shared by the plain align launch (align.cu) and the fused routing front end
// (topk.cu).
//
// Rows of one expert are placed in ascending flattened order, so the result
// is unique: the CTA counts rows per expert, pads each expert to block_m, and
// then walks the rows in chunks of kAlignThreads, ranking each row among the
// earlier rows of the same expert (warp match + per-warp counts).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace w4a16 {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;

// The placement of one CTA of kAlignThreads threads (num_experts <=
// kAlignThreads) over the global `ids`
// (read through L2, so ids that other CTAs of the same launch wrote before a
// fence are seen); `smem` holds (3 + kAlignWarps) * num_experts + 1 ints.
__device__ __forceinline__ void align_cta(const int32_t* ids, int numel, int num_experts, int block_m,
                          int capacity, int32_t* __restrict__ sorted_ids,
                          int32_t* __restrict__ expert_ids, int32_t* __restrict__ num_tokens_padded,
                          int* smem) {
  int* counts = smem;                      // [E]
  int* offsets = counts + num_experts;     // [E + 1]
  int* cursor = offsets + num_experts + 1; // [E]
  int* wcount = cursor + num_experts;      // [warps][E]
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  for (int e = tid; e < num_experts; e += kAlignThreads) counts[e] = 0;
  __syncthreads();
  for (int i = tid; i < numel; i += kAlignThreads) {
    const int e = __ldcg(ids + i);
    if (e >= 0 && e < num_experts) atomicAdd(&counts[e], 1);
  }
  __syncthreads();
  // offsets = exclusive scan of the padded counts, one expert per thread
  // (num_experts <= kAlignThreads): warp scans, then a scan of the warp sums
  {
    int* wsum = wcount;  // kAlignWarps ints, free until the placement
    const int v = tid < num_experts ? (counts[tid] + block_m - 1) / block_m * block_m : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      const int w = wsum[lane];
      int z = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, z, o);
        if (lane >= o) z += y;
      }
      wsum[lane] = z - w;  // exclusive: the warps before this one
    }
    __syncthreads();
    const int excl = wsum[warp] + x - v;
    if (tid < num_experts) offsets[tid] = excl;
    if (tid == num_experts - 1) {
      offsets[num_experts] = excl + v;
      *num_tokens_padded = excl + v;
    }
  }
  __syncthreads();
  for (int i = tid; i < capacity; i += kAlignThreads) sorted_ids[i] = numel;
  const int nblk = capacity / block_m;
  for (int b = tid; b < nblk; b += kAlignThreads) expert_ids[b] = -1;
  for (int e = tid; e < num_experts; e += kAlignThreads) cursor[e] = offsets[e];
  __syncthreads();
  for (int e = tid; e < num_experts; e += kAlignThreads) {
    for (int b = offsets[e] / block_m; b < offsets[e + 1] / block_m; ++b) expert_ids[b] = e;
  }

  // stable placement, chunk by chunk
  for (int base = 0; base < numel; base += kAlignThreads) {
    for (int x = tid; x < kAlignWarps * num_experts; x += kAlignThreads) wcount[x] = 0;
    __syncthreads();
    const int i = base + tid;
    int e = (i < numel) ? __ldcg(ids + i) : -1;
    const bool local = e >= 0 && e < num_experts;
    if (!local) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const unsigned lower = peers & ((1u << lane) - 1u);
    const int rank = __popc(lower);
    if (local && lower == 0) wcount[warp * num_experts + e] = __popc(peers);
    __syncthreads();
    if (local) {
      int pos = cursor[e] + rank;
      for (int w = 0; w < warp; ++w) pos += wcount[w * num_experts + e];
      sorted_ids[pos] = i;
    }
    __syncthreads();
    for (int x = tid; x < num_experts; x += kAlignThreads) {
      int add = 0;
      for (int w = 0; w < kAlignWarps; ++w) add += wcount[w * num_experts + x];
      cursor[x] += add;
    }
    __syncthreads();
  }
}

}  // namespace w4a16
