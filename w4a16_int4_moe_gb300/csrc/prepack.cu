// prepack.cu -- checkpoint uint4 group-32 weights -> the kernel's tiled layout.
//
// Input schema (page "vLLM 宣布 Humming 后端可运行 … Chord 内核 …", section
// "接入方式：用 Chord 替代公共 Humming 包"): uint4 codes, group 32 along K,
// BF16 scales; two codes per byte, even k in the low nibble; w = (q - 8) * s.
// The layout is fixed at load (same page, section
// "调度由每个专家收到的 token 数决定").
//
// Output: for each expert, 128-row tiles (rows in order, or, with
// W4A16_LAYOUT_KTILE64_GLU16, gate and up rows interleaved by 16: see
// packed_source_row); inside a tile, 64-k steps back to
// back; one step = q [2 groups][128 rows][16 B] then scales [2][128] BF16.
// Inside every 32-bit word (8 consecutive k) the nibbles are reordered so
// that (word >> 4i) & 0x000F000F holds k = 2i in the low half and k = 2i + 1
// in the high half, which is what the dequantiser extracts. Rows past n and k
// past k get code 8 with scale 0 (weight exactly 0).

#include <cuda_runtime.h>

#include "internal.h"

namespace w4a16 {

namespace {

// source word: nibble j at bits 4j (k = j)  ->  packed word: k = 2i at bits 4i,
// k = 2i + 1 at bits 16 + 4i.
__device__ __forceinline__ uint32_t shuffle_word(uint32_t v) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    r |= ((v >> (8 * i)) & 0xFu) << (4 * i);
    r |= ((v >> (8 * i + 4)) & 0xFu) << (16 + 4 * i);
  }
  return r;
}

__device__ __forceinline__ uint32_t unshuffle_word(uint32_t r) {
  uint32_t v = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v |= ((r >> (4 * i)) & 0xFu) << (8 * i);
    v |= ((r >> (16 + 4 * i)) & 0xFu) << (8 * i + 4);
  }
  return v;
}

}  // namespace

// One thread per (expert, tile, k step, group, row): 16 bytes of codes and
// one scale.
__global__ void w4a16_prepack_kernel(const uint8_t* __restrict__ q,
                                     const uint16_t* __restrict__ scales, int num_experts, int n,
                                     int k, int n_tiles, int k_steps, int layout,
                                     uint8_t* __restrict__ packed) {
  const long long total = static_cast<long long>(num_experts) * n_tiles * k_steps * 2 * kTileRows;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const int row = static_cast<int>(idx % kTileRows);
    long long rest = idx / kTileRows;
    const int g = static_cast<int>(rest % 2);
    rest /= 2;
    const int ks = static_cast<int>(rest % k_steps);
    rest /= k_steps;
    const int tile = static_cast<int>(rest % n_tiles);
    const int e = static_cast<int>(rest / n_tiles);
    const int nn = packed_source_row(n, layout, tile, row);
    const int k0 = ks * kKStep + g * kGroup;
    uint4 out = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
    uint16_t sc = 0;
    if (nn < n && k0 < k) {
      const long long src_row = static_cast<long long>(e) * n + nn;
      const uint4 in = *reinterpret_cast<const uint4*>(q + src_row * (k / 2) + k0 / 2);
      out = make_uint4(shuffle_word(in.x), shuffle_word(in.y), shuffle_word(in.z),
                       shuffle_word(in.w));
      sc = scales[src_row * (k / kGroup) + k0 / kGroup];
    }
    uint8_t* step = packed + ((static_cast<long long>(e) * n_tiles + tile) * k_steps + ks) *
                                 static_cast<long long>(kStepBytes);
    *reinterpret_cast<uint4*>(step + g * (kTileRows * 16) + row * 16) = out;
    *reinterpret_cast<uint16_t*>(step + kStepQBytes + g * (kTileRows * 2) + row * 2) = sc;
  }
}

__global__ void w4a16_unpack_kernel(const uint8_t* __restrict__ packed, int num_experts, int n,
                                    int k, int n_tiles, int k_steps, int layout,
                                    uint8_t* __restrict__ q, uint16_t* __restrict__ scales) {
  const long long total = static_cast<long long>(num_experts) * n * (k / kGroup);
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const int grp = static_cast<int>(idx % (k / kGroup));
    const long long src_row = idx / (k / kGroup);
    const int nn = static_cast<int>(src_row % n);
    const int e = static_cast<int>(src_row / n);
    int tile = nn / kTileRows, row = nn % kTileRows;
    if (layout == W4A16_LAYOUT_KTILE64_GLU16) {
      // inverse of packed_source_row: gate column c or up column c (n/2 + c)
      const bool up = nn >= n / 2;
      const int c = up ? nn - n / 2 : nn;
      tile = c / 64;
      row = ((c % 64) / 16) * 32 + (up ? 16 : 0) + c % 16;
    }
    const int ks = grp / 2, g = grp % 2;
    const uint8_t* step = packed + ((static_cast<long long>(e) * n_tiles + tile) * k_steps + ks) *
                                       static_cast<long long>(kStepBytes);
    const uint4 in = *reinterpret_cast<const uint4*>(step + g * (kTileRows * 16) + row * 16);
    *reinterpret_cast<uint4*>(q + src_row * (k / 2) + grp * 16) =
        make_uint4(unshuffle_word(in.x), unshuffle_word(in.y), unshuffle_word(in.z),
                   unshuffle_word(in.w));
    scales[src_row * (k / kGroup) + grp] =
        *reinterpret_cast<const uint16_t*>(step + kStepQBytes + g * (kTileRows * 2) + row * 2);
  }
}

cudaError_t launch_prepack(const uint8_t* q, const uint16_t* scales, int num_experts, int n,
                           int k, int layout, uint8_t* packed, cudaStream_t stream) {
  const long long total =
      static_cast<long long>(num_experts) * packed_tiles(n) * packed_ksteps(k) * 2 * kTileRows;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const long long want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 65536 ? want : 65536);
  w4a16_prepack_kernel<<<blocks, threads, 0, stream>>>(q, scales, num_experts, n, k,
                                                       packed_tiles(n), packed_ksteps(k), layout,
                                                       packed);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* packed, int num_experts, int n, int k, int layout,
                          uint8_t* q, uint16_t* scales, cudaStream_t stream) {
  const long long total = static_cast<long long>(num_experts) * n * (k / kGroup);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const long long want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 65536 ? want : 65536);
  w4a16_unpack_kernel<<<blocks, threads, 0, stream>>>(packed, num_experts, n, k, packed_tiles(n),
                                                      packed_ksteps(k), layout, q, scales);
  return cudaGetLastError();
}

}  // namespace w4a16
