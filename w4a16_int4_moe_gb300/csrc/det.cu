// det.cu -- the deterministic down pass (W4A16_FLAG_DETERMINISTIC).
//
// The down pass adds each routed row's top-k weighted product into its
// token's output row (page "vLLM 宣布 Humming 后端可运行 … Chord 内核 …",
// section "六个场景的逐层测量与限定条件": gate_up, then down with the top-k
// weights). With atomic adds the FP32 summation order over a token's top-k
// rows follows the schedule. In the deterministic pass the GEMM instead
// stores every weighted row at its routing position, and the kernels here
// add each token's rows in ascending top-k slot order:
//   out[t, :] (+)= sum over k = 0..topk-1 of rows[pos(t*topk + k), :]
// where pos is the routing position of flattened row t*topk + k (rows not
// routed to a local expert are skipped). The GEMM's row values do not depend
// on the grid, the block size or the ring depths, so neither does the result.

#include <cuda_runtime.h>

#include "internal.h"

namespace w4a16 {

// inv[id] = routing position of flattened row id (inv starts at -1).
__global__ void w4a16_det_inverse_kernel(const int32_t* __restrict__ sorted_ids,
                                         const int32_t* __restrict__ num_tokens_padded,
                                         int capacity, int numel, int32_t* __restrict__ inv) {
  int rows = __ldg(num_tokens_padded);
  rows = min(max(rows, 0), capacity);
  const int stride = gridDim.x * blockDim.x;
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < rows; j += stride) {
    const int id = __ldg(sorted_ids + j);
    if (id >= 0 && id < numel) inv[id] = j;
  }
}

// One thread per 4 output columns of a token (n % 4 == 0), else per column.
__global__ void w4a16_det_reduce_kernel(const float* __restrict__ rows,
                                        const int32_t* __restrict__ inv, int tokens, int topk,
                                        int n, int accumulate, float* __restrict__ out) {
  const bool vec4 = (n & 3) == 0;
  const int per_token = vec4 ? n / 4 : n;
  const long long total = static_cast<long long>(tokens) * per_token;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const int t = static_cast<int>(idx / per_token);
    const int c = static_cast<int>(idx - static_cast<long long>(t) * per_token);
    float* o = out + static_cast<long long>(t) * n;
    if (vec4) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = 0; k < topk; ++k) {
        const int pos = __ldg(inv + static_cast<long long>(t) * topk + k);
        if (pos < 0) continue;
        const float4 r =
            __ldg(reinterpret_cast<const float4*>(rows + static_cast<long long>(pos) * n) + c);
        acc.x += r.x;
        acc.y += r.y;
        acc.z += r.z;
        acc.w += r.w;
      }
      float4* dst = reinterpret_cast<float4*>(o) + c;
      if (accumulate) {
        const float4 prev = *dst;
        acc = make_float4(prev.x + acc.x, prev.y + acc.y, prev.z + acc.z, prev.w + acc.w);
      }
      *dst = acc;
    } else {
      float acc = 0.f;
      for (int k = 0; k < topk; ++k) {
        const int pos = __ldg(inv + static_cast<long long>(t) * topk + k);
        if (pos >= 0) acc += __ldg(rows + static_cast<long long>(pos) * n + c);
      }
      o[c] = accumulate ? o[c] + acc : acc;
    }
  }
}

cudaError_t launch_det_inverse(const int32_t* sorted_ids, const int32_t* num_tokens_padded,
                               int capacity, int numel, int32_t* inv, int sms,
                               cudaStream_t stream) {
  if (numel <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(inv, 0xff, static_cast<size_t>(numel) * sizeof(int32_t), stream);
  if (e != cudaSuccess || capacity <= 0) return e;
  const int threads = 256;
  const int want = (capacity + threads - 1) / threads;
  const int cap = (sms > 0 ? sms : 1) * 4;
  w4a16_det_inverse_kernel<<<want < cap ? want : cap, threads, 0, stream>>>(
      sorted_ids, num_tokens_padded, capacity, numel, inv);
  return cudaGetLastError();
}

cudaError_t launch_det_reduce(const float* rows, const int32_t* inv, int tokens, int topk, int n,
                              bool accumulate, float* out, int sms, cudaStream_t stream) {
  const long long per_token = (n % 4 == 0) ? n / 4 : n;
  const long long total = static_cast<long long>(tokens) * per_token;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const long long want = (total + threads - 1) / threads;
  const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * 8;
  w4a16_det_reduce_kernel<<<static_cast<int>(want < cap ? want : cap), threads, 0, stream>>>(
      rows, inv, tokens, topk, n, accumulate ? 1 : 0, out);
  return cudaGetLastError();
}

}  // namespace w4a16
