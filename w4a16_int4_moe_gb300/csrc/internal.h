// internal.h -- host-side declarations shared by the library's translation
// units (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/w4a16moe.h"

namespace w4a16 {

// Packed weight layout (W4A16_LAYOUT_KTILE64): for every expert, 128-row
// tiles; inside a tile, 64-k steps back to back; one step holds
//   q      [2 groups][128 rows][16 bytes]  (32 codes of one group per row)
//   scales [2 groups][128 rows] BF16
// so a whole tile's k range is one contiguous run of bytes.
constexpr int kTileRows = 128;
constexpr int kKStep = 64;
constexpr int kGroup = 32;
constexpr int kStepQBytes = 2 * kTileRows * 16;        // 4096
constexpr int kStepBytes = kStepQBytes + 2 * kTileRows * 2;  // 4608
constexpr int kStatusBytes = 256;

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline long long ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

// Permuted activation rows of the indexed GEMM (in the workspace, after the
// status block): [capacity][k rounded up to 64] BF16.
inline int permuted_row_elems(int k) { return ceil_div(k, kKStep) * kKStep; }
inline size_t permuted_bytes(long long rows, int k) {
  return static_cast<size_t>(rows) * permuted_row_elems(k) * 2;
}

// Weighted FP32 rows of the deterministic down pass, [capacity][n], rounded
// up to 256 bytes (in the workspace after the routed rows).
inline size_t det_rows_bytes(int capacity, int n) {
  return (static_cast<size_t>(capacity) * n * 4 + 255) / 256 * 256;
}

inline int packed_tiles(int n) { return ceil_div(n, kTileRows); }
inline int packed_ksteps(int k) { return ceil_div(k, kKStep); }
inline size_t packed_expert_bytes(int n, int k) {
  return static_cast<size_t>(packed_tiles(n)) * packed_ksteps(k) * kStepBytes;
}

enum Family { kIndexed = 0, kContiguous = 1, kMasked = 2 };
// kOutF32Rows (the deterministic down pass): top-k weighted FP32 rows, each
// at its routing position, for a separate ordered sum per token.
enum OutMode { kOutBf16 = 0, kOutF32WeightedAdd = 1, kOutGluBf16 = 2, kOutF32Rows = 3 };

// Source row (of the [n, k] weight matrix) of row `row` of packed tile `tile`.
// W4A16_LAYOUT_KTILE64_GLU16 interleaves gate rows [0, n/2) and up rows
// [n/2, n) by 16 inside each 32-row quarter of a tile.
__host__ __device__ inline int packed_source_row(int n, int layout, int tile, int row) {
  if (layout != W4A16_LAYOUT_KTILE64_GLU16) return tile * kTileRows + row;
  const int q = row >> 5, i = row & 31;
  const int col = tile * 64 + q * 16 + (i & 15);
  return i < 16 ? col : n / 2 + col;
}

struct GemmArgs {
  // Activation tensor map: the permuted rows of the indexed family, or the
  // rows of a grouped family when k % 64 == 0, as a 3-D array (two k steps
  // per box); else the rows of a grouped family (2-D, one k step per box);
  // box rows = block_m, 128-byte swizzle.
  CUtensorMap tmap;
  int act_rows;
  int gather_rows;  // 1: the 3-D map (two k steps per copy), 0: the 2-D map
  const uint8_t* wpack;
  long long expert_bytes;
  int num_experts, n, k, n_tiles, k_steps;
  const uint16_t* act;  // BF16 rows of length k
  int family;
  int out_mode;
  // indexed routing
  const int32_t* sorted_ids;
  const int32_t* expert_ids;
  const int32_t* num_tokens_padded;
  int capacity;
  int numel;     // tokens * topk (sentinel)
  int a_div;     // activation row = id / a_div
  int o_div;     // output row = id / o_div
  const float* topk_weights;
  // grouped layouts
  const int32_t* layout;  // m_expert [m] or masked_m [E]
  int m;                  // rows (contiguous) or per-expert budget (masked)
  // common
  int block_m;
  void* out;
  int* status;
  // pipeline configuration (derived from the plan): weight ring stages (a
  // multiple of 4), activation ring stages (even), partial accumulators (MMA
  // issuers), accumulator slots and the TMEM columns of one accumulator
  int w_stages, b_stages, n_parts, d_slots, d_cols;
  int raster_rows;  // 1: grouped item order (see decode_item), 0: tile-major
  // 1: CTA pairs (clusters of 2) issue M = 256 MMAs over two weight tiles;
  // needs an even tile count and block_m a multiple of 32; grid even
  int pair;
  // the single-launch layer (w4a16_moe_layer): after the gate_up items (out =
  // the activation rows at their routing positions) come the down items of
  // the same routing blocks, with their own packed weights, reduction length
  // (k_steps2), width n2, activation map (tmap2) and FP32 output (out2); a
  // block's down items wait until block_done[block] reaches 4 * n_tiles
  const uint8_t* wpack2;
  long long expert_bytes2;
  int n2, n_tiles2, k_steps2;
  CUtensorMap tmap2;
  float* out2;
  int* block_done;
  int layer;
  long long timeout_cycles;
};

int device_sm_count(int device);

// w4a16_moe_indexed_gemm. With noalloc the workspace is the library's own
// scratch array of ws_bytes (noalloc.cu; `workspace` is ignored): its device
// address is looked up and its status words are zeroed on `stream` only once
// every host-side check has passed (a refused call makes no CUDA call).
w4a16_status indexed_gemm(int mode, const void* packed, int num_experts, int n, int k,
                          const uint16_t* a, int tokens, int topk, const int32_t* sorted_ids,
                          const int32_t* expert_ids, const int32_t* num_tokens_padded,
                          int capacity, const float* topk_weights, void* out, int flags,
                          const w4a16_plan_t* plan, void* workspace, size_t ws_bytes,
                          void* stream, bool noalloc);
// Device address of the no-allocation scratch array on the current device
// (nullptr on a CUDA error).
void* noalloc_scratch_address();
// Shared memory of a launch: b_stages activation slots (two k steps each, or
// one for blocks above 128 rows) and w_stages weight stages.
size_t gemm_smem_bytes(int block_m, int w_stages, int b_stages, bool pair = false);
// Blocks above 128 rows: the activation ring holds single k steps. An item
// whose MMA N exceeds 128 is filled by one copy of the whole block (map tmap);
// a smaller one by copies of kActivationBoxRowsSmall rows up to its N (map
// tmap2), so that a mostly empty block does not read the rows it lacks.
constexpr bool activation_slot_is_step(int block_m) { return block_m > 128; }
constexpr int kActivationBoxRowsSmall = 64;
// Token rows of one activation tensor copy of the main map (tmap).
constexpr int activation_box_rows(int block_m, bool pair) {
  return pair ? block_m / 2 : block_m;
}
// CTA pairs of the GEMM kernel for `args` that can be resident at once (0 on
// error).
int max_pair_clusters(const GemmArgs& args);
// TMEM split for a block of block_m rows and a reduction of k_steps 64-k
// steps: columns of one accumulator, the number of partial accumulators (MMA
// issuers) and of accumulator slots.
// False when even one accumulator does not fit.
bool tmem_accumulators(int block_m, int k_steps, int* d_cols, int* parts, int* d_slots);
// The epilogue frees the accumulator slot before its global stores.
bool early_epilogue(int block_m, int out_mode, bool pair);
// 2-D map of BF16 [rows, k] (box 64 x box_rows, 128-byte swizzle).
bool encode_act_tmap(CUtensorMap* map, const void* act, long long rows, int k, int box_rows);
// 3-D map of the permuted rows [rows, k_pad]: dims (64 columns, rows, k_pad /
// 64 chunks), box 64 x box_rows x box_steps (1 or 2 k steps), 128-byte swizzle.
bool encode_permuted_tmap(CUtensorMap* map, const void* act, long long rows, int k_pad,
                          int box_rows, int box_steps);
// dependent = true: launched as a programmatic dependent of the previous
// kernel on `stream` (the row permute), see w4a16_permute_rows_kernel.
cudaError_t launch_moe_gemm(const GemmArgs& args, int grid, bool dependent, cudaStream_t stream);

// Top-k routing and moe_align_block_size in one launch (topk.cu).
cudaError_t launch_route_align(const void* logits, int bf16_logits, int tokens, int num_experts,
                               int topk, int renormalize, int expert_offset, int num_local,
                               int block_m, int capacity, int32_t* topk_ids, float* topk_weights,
                               int32_t* sorted_ids, int32_t* expert_ids,
                               int32_t* num_tokens_padded, unsigned int* arrivals, int sms,
                               cudaStream_t stream);

cudaError_t launch_align(const int32_t* topk_ids, int numel, int num_experts, int block_m,
                         int capacity, int32_t* sorted_ids, int32_t* expert_ids,
                         int32_t* num_tokens_padded, cudaStream_t stream);
size_t align_smem_bytes(int num_experts);

cudaError_t launch_prepack(const uint8_t* q, const uint16_t* scales, int num_experts, int n,
                           int k, int layout, uint8_t* packed, cudaStream_t stream);
cudaError_t launch_unpack(const uint8_t* packed, int num_experts, int n, int k, int layout,
                          uint8_t* q, uint16_t* scales, cudaStream_t stream);

// Routed rows into routing order; also zeroes zero_bytes (a multiple of 16)
// at `zero` when given. Triggers the programmatic launch of the next kernel.
cudaError_t launch_permute_rows(const uint16_t* a, int k, int a_div, int numel,
                                const int32_t* sorted_ids, const int32_t* num_tokens_padded,
                                int capacity, uint16_t* dst, void* zero, size_t zero_bytes,
                                int sms, cudaStream_t stream);

// Deterministic down pass: inv[id] = routing position of flattened row id
// (-1 when not routed here), then out[t] (+)= the top-k weighted rows of
// token t added in ascending top-k slot order.
cudaError_t launch_det_inverse(const int32_t* sorted_ids, const int32_t* num_tokens_padded,
                               int capacity, int numel, int32_t* inv, int sms,
                               cudaStream_t stream);
cudaError_t launch_det_reduce(const float* rows, const int32_t* inv, int tokens, int topk, int n,
                              bool accumulate, float* out, int sms, cudaStream_t stream);

cudaError_t launch_topk_softmax(const void* logits, int bf16_logits, int tokens, int num_experts,
                                int topk, int renormalize, int expert_offset, int num_local,
                                int32_t* topk_ids, float* topk_weights, int sms,
                                cudaStream_t stream);

cudaError_t launch_silu_and_mul(const uint16_t* in, int rows, int inter, uint16_t* out,
                                cudaStream_t stream);

}  // namespace w4a16
