// permute.cu -- routed activation rows, copied once into sorted order.
//
// The indexed GEMM reads its token operand in routing order: block b of the
// aligned routing (page "vLLM 宣布 Humming 后端可运行 … Chord 内核 …",
// section "调度由每个专家收到的 token 数决定": sorted_ids / expert_ids /
// num_tokens_padded) holds rows sorted_ids[b*block_m ...]. Copying those rows
// once into a dense [capacity, k_pad] buffer lets the GEMM fetch a block's
// rows for two k steps with a single TMA tensor copy instead of one gather
// per four rows per k step. Row j of the buffer is activation row
// sorted_ids[j] / a_div; columns k..k_pad-1 are zero (k_pad = k rounded up to
// 64, so the 64-column chunks of the tensor copy never reach into the next
// row); rows of sentinel entries are not written (the GEMM never uses their
// values: an MMA column depends only on its own row).

#include <cuda_runtime.h>

#include "internal.h"

namespace w4a16 {

// One thread per 16-byte chunk of a destination row.
__global__ void w4a16_permute_rows_kernel(const uint16_t* __restrict__ a, int k, int k_pad,
                                          int a_div, int numel, const int32_t* __restrict__ sorted_ids,
                                          const int32_t* __restrict__ num_tokens_padded,
                                          int capacity, uint16_t* __restrict__ dst) {
  int rows = __ldg(num_tokens_padded);
  rows = min(max(rows, 0), capacity);
  const int chunks = k_pad / 8;
  const long long total = static_cast<long long>(rows) * chunks;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const int j = static_cast<int>(idx / chunks);
    const int c = static_cast<int>(idx - static_cast<long long>(j) * chunks);
    const int id = __ldg(sorted_ids + j);
    if (id < 0 || id >= numel) continue;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (c * 8 < k)
      v = __ldg(reinterpret_cast<const uint4*>(a + static_cast<long long>(id / a_div) * k + c * 8));
    *reinterpret_cast<uint4*>(dst + static_cast<long long>(j) * k_pad + c * 8) = v;
  }
}

cudaError_t launch_permute_rows(const uint16_t* a, int k, int a_div, int numel,
                                const int32_t* sorted_ids, const int32_t* num_tokens_padded,
                                int capacity, uint16_t* dst, int sms, cudaStream_t stream) {
  const int k_pad = permuted_row_elems(k);
  const long long total = static_cast<long long>(capacity) * (k_pad / 8);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const long long want = (total + threads - 1) / threads;
  const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * 8;
  const int blocks = static_cast<int>(want < cap ? want : cap);
  w4a16_permute_rows_kernel<<<blocks, threads, 0, stream>>>(a, k, k_pad, a_div, numel, sorted_ids,
                                                            num_tokens_padded, capacity, dst);
  return cudaGetLastError();
}

}  // namespace w4a16
