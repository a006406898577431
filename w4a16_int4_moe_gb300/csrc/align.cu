// align.cu -- moe_align_block_size on the GPU, bit-exact and deterministic.
//
// The indexed kernel consumes vLLM's sorted_ids / expert_ids /
// num_tokens_padded (page "vLLM 宣布 Humming 后端可运行 … Chord 内核 …",
// section "调度由每个专家收到的 token 数决定") on over-allocated buffers (page
// "vLLM と Novita AI が Chord をリリース …", section "ランタイムの考慮事項").
// Rows of one expert are placed in ascending flattened order, so the result
// is unique: one CTA walks the rows in chunks of 1024 and ranks each row
// among the earlier rows of the same expert (warp match + per-warp counts).

#include <cuda_runtime.h>

#include "internal.h"

namespace w4a16 {

namespace {
constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
}  // namespace

__global__ void __launch_bounds__(kAlignThreads) w4a16_align_kernel(
    const int32_t* __restrict__ topk_ids, int numel, int num_experts, int block_m, int capacity,
    int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
    int32_t* __restrict__ num_tokens_padded) {
  extern __shared__ int smem[];
  int* counts = smem;                      // [E]
  int* offsets = counts + num_experts;     // [E + 1]
  int* cursor = offsets + num_experts + 1; // [E]
  int* wcount = cursor + num_experts;      // [warps][E]
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  for (int e = tid; e < num_experts; e += kAlignThreads) counts[e] = 0;
  __syncthreads();
  for (int i = tid; i < numel; i += kAlignThreads) {
    const int e = topk_ids[i];
    if (e >= 0 && e < num_experts) atomicAdd(&counts[e], 1);
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int e = 0; e < num_experts; ++e) {
      offsets[e] = acc;
      acc += (counts[e] + block_m - 1) / block_m * block_m;
    }
    offsets[num_experts] = acc;
    *num_tokens_padded = acc;
  }
  __syncthreads();
  const int total = offsets[num_experts];
  for (int i = tid; i < capacity; i += kAlignThreads) sorted_ids[i] = numel;
  const int nblk = capacity / block_m;
  for (int b = tid; b < nblk; b += kAlignThreads) expert_ids[b] = -1;
  for (int e = tid; e < num_experts; e += kAlignThreads) cursor[e] = offsets[e];
  __syncthreads();
  for (int e = tid; e < num_experts; e += kAlignThreads) {
    for (int b = offsets[e] / block_m; b < offsets[e + 1] / block_m; ++b) expert_ids[b] = e;
  }
  (void)total;

  // stable placement, chunk by chunk
  for (int base = 0; base < numel; base += kAlignThreads) {
    for (int x = tid; x < kAlignWarps * num_experts; x += kAlignThreads) wcount[x] = 0;
    __syncthreads();
    const int i = base + tid;
    int e = (i < numel) ? topk_ids[i] : -1;
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

size_t align_smem_bytes(int num_experts) {
  return sizeof(int) * (static_cast<size_t>(num_experts) * (3 + kAlignWarps) + 1);
}

cudaError_t launch_align(const int32_t* topk_ids, int numel, int num_experts, int block_m,
                         int capacity, int32_t* sorted_ids, int32_t* expert_ids,
                         int32_t* num_tokens_padded, cudaStream_t stream) {
  const size_t smem = align_smem_bytes(num_experts);
  cudaError_t err = cudaFuncSetAttribute(w4a16_align_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  w4a16_align_kernel<<<1, kAlignThreads, smem, stream>>>(topk_ids, numel, num_experts, block_m,
                                                         capacity, sorted_ids, expert_ids,
                                                         num_tokens_padded);
  return cudaGetLastError();
}

}  // namespace w4a16
