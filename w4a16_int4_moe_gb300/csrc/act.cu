// act.cu -- the activation between gate_up and down: silu(gate) * up.
//
// The pages leave the activation out of the timed gate_up + down pair (page
// "vLLM 宣布 Humming 后端可运行 … Chord 内核 …", section
// "六个场景的逐层测量与限定条件"); its form here is a reading: the gate_up
// output row is [gate | up], each half `inter` wide.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace w4a16 {

// One thread per 8 output elements (16-byte loads and stores).
// silu(g) * u = g / (1 + e^-g) * u in FP32 with the fast exponential and
// division intrinsics (a few FP32 ulps, far below the BF16 rounding of the
// result); the fused gate_up epilogue evaluates the same expression, so the
// two paths give the same bits.
__global__ void w4a16_silu_and_mul_kernel(const uint16_t* __restrict__ in, int rows, int inter,
                                          uint16_t* __restrict__ out) {
  const int vec_per_row = inter / 8;
  const long long total = static_cast<long long>(rows) * vec_per_row;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const long long r = idx / vec_per_row;
    const int c = static_cast<int>(idx % vec_per_row) * 8;
    const uint4 gv = *reinterpret_cast<const uint4*>(in + r * 2 * inter + c);
    const uint4 uv = *reinterpret_cast<const uint4*>(in + r * 2 * inter + inter + c);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
    const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&uv);
    uint4 ov;
    __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&ov);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 g = __bfloat1622float2(g2[i]);
      const float2 u = __bfloat1622float2(u2[i]);
      const float a0 = __fdividef(g.x, 1.0f + __expf(-g.x)) * u.x;
      const float a1 = __fdividef(g.y, 1.0f + __expf(-g.y)) * u.y;
      o2[i] = __floats2bfloat162_rn(a0, a1);
    }
    *reinterpret_cast<uint4*>(out + r * inter + c) = ov;
  }
}

cudaError_t launch_silu_and_mul(const uint16_t* in, int rows, int inter, uint16_t* out,
                                cudaStream_t stream) {
  const long long total = static_cast<long long>(rows) * (inter / 8);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const long long want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 16384 ? want : 16384);
  w4a16_silu_and_mul_kernel<<<blocks, threads, 0, stream>>>(in, rows, inter, out);
  return cudaGetLastError();
}

}  // namespace w4a16
