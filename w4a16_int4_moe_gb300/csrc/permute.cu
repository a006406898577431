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

// One thread per 16-byte chunk of a destination row; the same grid also
// zeroes `zero` (zero_vec16 chunks of 16 bytes, the down pass's FP32 output)
// when it is given. The GEMM that consumes these rows is launched as a
// programmatic dependent of this grid: it may start (and stream weights)
// while this grid still runs, and waits for its completion before it reads
// the rows or adds into the output.
__global__ void w4a16_permute_rows_kernel(const uint16_t* __restrict__ a, int k, int k_pad,
                                          int a_div, int numel, const int32_t* __restrict__ sorted_ids,
                                          const int32_t* __restrict__ num_tokens_padded,
                                          int capacity, uint16_t* __restrict__ dst,
                                          uint4* __restrict__ zero, long long zero_vec16) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
         i < zero_vec16; i += stride)
      zero[i] = make_uint4(0u, 0u, 0u, 0u);
  }
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
                                int capacity, uint16_t* dst, void* zero, size_t zero_bytes,
                                int sms, cudaStream_t stream) {
  const int k_pad = permuted_row_elems(k);
  const long long total = static_cast<long long>(capacity) * (k_pad / 8);
  const long long zvec = static_cast<long long>(zero_bytes / 16);
  const long long work = total > zvec ? total : zvec;
  if (work == 0) return cudaSuccess;
  const int threads = 256;
  const long long want = (work + threads - 1) / threads;
  const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * 8;
  const int blocks = static_cast<int>(want < cap ? want : cap);
  w4a16_permute_rows_kernel<<<blocks, threads, 0, stream>>>(
      a, k, k_pad, a_div, numel, sorted_ids, num_tokens_padded, capacity, dst,
      static_cast<uint4*>(zero), zvec);
  return cudaGetLastError();
}

}  // namespace w4a16
