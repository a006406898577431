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

#include "align_cta.cuh"
#include "internal.h"

namespace w4a16 {

__global__ void __launch_bounds__(kAlignThreads) w4a16_align_kernel(
    const int32_t* __restrict__ topk_ids, int numel, int num_experts, int block_m, int capacity,
    int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
    int32_t* __restrict__ num_tokens_padded) {
  extern __shared__ int smem[];
  align_cta(topk_ids, numel, num_experts, block_m, capacity, sorted_ids, expert_ids,
            num_tokens_padded, smem);
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
