// topk.cu -- the routing front end: router logits -> top-k local expert ids
// and weights, the inputs of moe_align_block_size.
//
// The pages route every token to the top 8 of 384 experts and hand the
// operator vLLM's routing tensors (page "vLLM 宣布 Humming 后端可运行 … Chord
// 内核 …", section "调度由每个专家收到的 token 数决定"); the router itself is
// the serving stack's. Reading taken here: softmax over all experts, the k
// largest logits (ties to the lower expert id), the chosen probabilities
// optionally renormalised to sum to 1, and global ids mapped to this GPU's
// local experts (-1 for another GPU's). Experts with a -inf logit are masked:
// never chosen; slots that find no expert hold id -1 and weight 0.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>

#include "align_cta.cuh"
#include "internal.h"

namespace w4a16 {

namespace {
constexpr int kTopkWarps = 8;       // warps per block, one token per warp
constexpr int kMaxPerLane = 32;     // experts per lane: up to 1024 experts
}  // namespace

// Top-k of token t by one warp (all 32 lanes take part); kPer logits per
// lane, so num_experts <= 32 * kPer.
template <int kPer>
__device__ __forceinline__ void route_token(const void* __restrict__ logits, int bf16_logits, int t,
                                            int num_experts, int topk, int renormalize,
                                            int expert_offset, int num_local,
                                            int32_t* __restrict__ topk_ids,
                                            float* __restrict__ topk_weights) {
  const int lane = threadIdx.x & 31;
  // this lane's logits: experts lane, lane + 32, ...
  float v[kPer];
  float mx = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    v[i] = -FLT_MAX;
    if (e < num_experts) {
      const long long at = static_cast<long long>(t) * num_experts + e;
      v[i] = bf16_logits ? __bfloat162float(static_cast<const __nv_bfloat16*>(logits)[at])
                         : static_cast<const float*>(logits)[at];
      mx = fmaxf(mx, v[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if (lane + 32 * i < num_experts) sum += expf(v[i] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);

  // k rounds of arg-max (largest logit, then lowest id); lane s keeps round s
  uint32_t taken = 0;
  float my_p = 0.f, sel_sum = 0.f;
  int my_id = -1;
  for (int s = 0; s < topk; ++s) {
    float bv = -FLT_MAX;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane + 32 * i;
      if (e < num_experts && !(taken & (1u << i)) && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    // no expert left to choose (the rest are masked with -inf logits): the
    // slot holds id -1 and weight 0
    const bool found = be < num_experts;
    if (found && (be & 31) == lane) taken |= 1u << (be >> 5);
    const float p = found ? expf(bv - mx) / sum : 0.f;
    sel_sum += p;
    if (lane == s) {
      my_p = p;
      my_id = found ? be : -1;
    }
  }
  if (lane < topk) {
    const int loc = my_id - expert_offset;
    const long long at = static_cast<long long>(t) * topk + lane;
    topk_ids[at] = (my_id >= 0 && loc >= 0 && loc < num_local) ? loc : -1;
    topk_weights[at] = renormalize ? (sel_sum > 0.f ? my_p / sel_sum : 0.f) : my_p;
  }
}

template <int kPer>
__global__ void __launch_bounds__(kTopkWarps * 32)
    w4a16_topk_softmax_kernel(const void* __restrict__ logits, int bf16_logits, int tokens,
                              int num_experts, int topk, int renormalize, int expert_offset,
                              int num_local, int32_t* __restrict__ topk_ids,
                              float* __restrict__ topk_weights) {
  const int warps = gridDim.x * kTopkWarps;
  for (int t = blockIdx.x * kTopkWarps + (threadIdx.x >> 5); t < tokens; t += warps)
    route_token<kPer>(logits, bf16_logits, t, num_experts, topk, renormalize, expert_offset,
                      num_local, topk_ids, topk_weights);
}

// Top-k over all CTAs, then moe_align_block_size by the CTA that finishes
// last (it counts the arrivals; no CTA waits on another). `arrivals` is zero
// on entry and reset to zero by that CTA.
template <int kPer>
__global__ void __launch_bounds__(kAlignThreads)
    w4a16_route_align_kernel(const void* __restrict__ logits, int bf16_logits, int tokens,
                             int num_experts, int topk, int renormalize, int expert_offset,
                             int num_local, int block_m, int capacity,
                             int32_t* __restrict__ topk_ids, float* __restrict__ topk_weights,
                             int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                             int32_t* __restrict__ num_tokens_padded,
                             unsigned int* __restrict__ arrivals) {
  extern __shared__ int smem[];
  __shared__ int is_last;
  // token t goes to CTA t % grid, so that few tokens share an SM
  for (int t = (threadIdx.x >> 5) * gridDim.x + blockIdx.x; t < tokens;
       t += kAlignWarps * gridDim.x)
    route_token<kPer>(logits, bf16_logits, t, num_experts, topk, renormalize, expert_offset,
                      num_local, topk_ids, topk_weights);
  __threadfence();  // this CTA's ids are visible before its arrival counts
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(arrivals, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  align_cta(topk_ids, tokens * topk, num_local, block_m, capacity, sorted_ids, expert_ids,
            num_tokens_padded, smem);
  if (threadIdx.x == 0) *arrivals = 0u;
}

cudaError_t launch_topk_softmax(const void* logits, int bf16_logits, int tokens, int num_experts,
                                int topk, int renormalize, int expert_offset, int num_local,
                                int32_t* topk_ids, float* topk_weights, int sms,
                                cudaStream_t stream) {
  if (tokens == 0) return cudaSuccess;
  const int want = (tokens + kTopkWarps - 1) / kTopkWarps;
  const int cap = (sms > 0 ? sms : 1) * 8;
  auto kernel =
      num_experts <= 512 ? w4a16_topk_softmax_kernel<16> : w4a16_topk_softmax_kernel<kMaxPerLane>;
  kernel<<<want < cap ? want : cap, kTopkWarps * 32, 0, stream>>>(
      logits, bf16_logits, tokens, num_experts, topk, renormalize, expert_offset, num_local,
      topk_ids, topk_weights);
  return cudaGetLastError();
}

cudaError_t launch_route_align(const void* logits, int bf16_logits, int tokens, int num_experts,
                               int topk, int renormalize, int expert_offset, int num_local,
                               int block_m, int capacity, int32_t* topk_ids, float* topk_weights,
                               int32_t* sorted_ids, int32_t* expert_ids,
                               int32_t* num_tokens_padded, unsigned int* arrivals, int sms,
                               cudaStream_t stream) {
  // 16 logits per lane cover 512 experts without spilling under the 64
  // registers a 1024-thread CTA leaves each thread
  auto kernel = num_experts <= 512 ? w4a16_route_align_kernel<16> : w4a16_route_align_kernel<32>;
  const size_t smem = align_smem_bytes(num_local);
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  // about kTopkWarps tokens per CTA (as the plain top-k launch), up to one
  // CTA per SM
  const int want = (tokens + kTopkWarps - 1) / kTopkWarps;
  const int cap = sms > 0 ? sms : 1;
  const int grid = want < 1 ? 1 : (want < cap ? want : cap);
  kernel<<<grid, kAlignThreads, smem, stream>>>(
      logits, bf16_logits, tokens, num_experts, topk, renormalize, expert_offset, num_local,
      block_m, capacity, topk_ids, topk_weights, sorted_ids, expert_ids, num_tokens_padded,
      arrivals);
  return cudaGetLastError();
}

}  // namespace w4a16
