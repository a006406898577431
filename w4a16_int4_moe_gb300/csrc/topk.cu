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

#include "internal.h"

namespace w4a16 {

namespace {
constexpr int kTopkWarps = 8;       // warps per block, one token per warp
constexpr int kMaxPerLane = 32;     // experts per lane: up to 1024 experts
}  // namespace

__global__ void __launch_bounds__(kTopkWarps * 32)
    w4a16_topk_softmax_kernel(const void* __restrict__ logits, int bf16_logits, int tokens,
                              int num_experts, int topk, int renormalize, int expert_offset,
                              int num_local, int32_t* __restrict__ topk_ids,
                              float* __restrict__ topk_weights) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * kTopkWarps;
  for (int t = blockIdx.x * kTopkWarps + (threadIdx.x >> 5); t < tokens; t += warps) {
    // this lane's logits: experts lane, lane + 32, ...
    float v[kMaxPerLane];
    float mx = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      v[i] = -FLT_MAX;
      if (e < num_experts) {
        const long long at = static_cast<long long>(t) * num_experts + e;
        v[i] = bf16_logits
                   ? __bfloat162float(static_cast<const __nv_bfloat16*>(logits)[at])
                   : static_cast<const float*>(logits)[at];
        mx = fmaxf(mx, v[i]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
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
      for (int i = 0; i < kMaxPerLane; ++i) {
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
      // no expert left to choose (the rest are masked with -inf logits):
      // the slot holds id -1 and weight 0
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
}

cudaError_t launch_topk_softmax(const void* logits, int bf16_logits, int tokens, int num_experts,
                                int topk, int renormalize, int expert_offset, int num_local,
                                int32_t* topk_ids, float* topk_weights, int sms,
                                cudaStream_t stream) {
  if (tokens == 0) return cudaSuccess;
  const int want = (tokens + kTopkWarps - 1) / kTopkWarps;
  const int cap = (sms > 0 ? sms : 1) * 8;
  w4a16_topk_softmax_kernel<<<want < cap ? want : cap, kTopkWarps * 32, 0, stream>>>(
      logits, bf16_logits, tokens, num_experts, topk, renormalize, expert_offset, num_local,
      topk_ids, topk_weights);
  return cudaGetLastError();
}

}  // namespace w4a16
