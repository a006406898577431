// api.cu -- the extern "C" entry points declared in include/w4a16moe.h:
// host-side argument checks, the tok_e scheduler, and the launches.

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "internal.h"

using namespace w4a16;

namespace {

constexpr int kMaxDynSmem = 232448;  // 227 KB per CTA on sm_103a
constexpr long long kDefaultTimeoutCycles = 2000000000LL;  // about a second

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

w4a16_status cuda_status(cudaError_t e) { return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA; }

long long wait_timeout_cycles() {
  const char* s = std::getenv("W4A16_WAIT_TIMEOUT_CYCLES");
  if (s != nullptr) {
    const long long v = std::atoll(s);
    if (v > 0) return v;
  }
  return kDefaultTimeoutCycles;
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

struct Pipeline {
  int w_stages, b_stages, d_cols, parts, d_slots;
  size_t smem;
};

// Validate a plan and derive the pipeline. TMEM holds four A slots of two k
// steps (64 columns each) and, in the other 256 columns, the partial
// accumulators of one or two items. plan.stages is the weight ring depth in
// stages of two k steps (rounded down to a multiple of 4: each of the four
// dequant warpgroups owns every fourth stage); plan.b_stages is the
// activation ring depth in k steps: a multiple of 4 (an even number of
// two-step slots up to 128 rows; above, single-step slots, a multiple of 4 so
// that each slot has one MMA issuer within an item).
bool plan_pipeline(const w4a16_plan_t& p, int k, Pipeline* out) {
  if (p.block_m < 16 || p.block_m > 256 || p.block_m % 16 != 0) return false;
  if (p.bn != kTileRows || p.bk != kKStep || p.split_k != 1) return false;
  if (p.layout != W4A16_LAYOUT_KTILE64 && p.layout != W4A16_LAYOUT_KTILE64_GLU16) return false;
  const bool step_slots = activation_slot_is_step(p.block_m);
  if (p.stages < 4 || p.stages > 16 || p.b_stages > 32) return false;
  if (p.b_stages < (step_slots ? 4 : 8) || p.b_stages % 4 != 0) return false;
  Pipeline pl;
  if (!tmem_accumulators(p.block_m, packed_ksteps(k), &pl.d_cols, &pl.parts, &pl.d_slots))
    return false;
  // single-step activation slots are read by one MMA issuer
  if (step_slots && pl.parts != 1) return false;
  pl.w_stages = p.stages / 4 * 4;
  pl.b_stages = step_slots ? p.b_stages : p.b_stages / 2;
  if (p.cta_pair != 0 && p.cta_pair != 1) return false;
  if (p.cta_pair && (p.block_m % 32 != 0 || step_slots)) return false;
  pl.smem = gemm_smem_bytes(p.block_m, pl.w_stages, pl.b_stages, p.cta_pair != 0);
  if (pl.smem > static_cast<size_t>(kMaxDynSmem)) return false;
  *out = pl;
  return true;
}

void fill_pipeline(const Pipeline& pl, GemmArgs* g) {
  g->w_stages = pl.w_stages;
  g->b_stages = pl.b_stages;
  g->n_parts = pl.parts;
  g->d_cols = pl.d_cols;
  g->d_slots = pl.d_slots;
}

// Ring depths of a plan: the deepest (activation, weight) pair that fits in
// shared memory next to block_m-row activation stages, an activation ring of
// at least six stages first (at EP8 prefill, 6 activation and 8 weight stages
// measured 10% faster than 4 and 12).
void set_ring_depths(w4a16_plan_t* p) {
  static const int kDepths[][2] = {{8, 16}, {6, 16}, {8, 12}, {6, 12}, {8, 8},
                                   {6, 8},  {4, 16}, {4, 12}, {4, 8},  {4, 4}};
  p->b_stages = 8;
  p->stages = 4;
  if (activation_slot_is_step(p->block_m)) {
    // single-step activation slots (a 256-row k step is 32 KB), a multiple
    // of 4, then the deepest weight ring beside them
    static const int kStepDepths[][2] = {{8, 8}, {8, 4}, {4, 8}, {4, 4}};
    for (const auto& dw : kStepDepths) {
      if (gemm_smem_bytes(p->block_m, dw[1], dw[0]) <= static_cast<size_t>(kMaxDynSmem)) {
        p->b_stages = dw[0];
        p->stages = dw[1];
        return;
      }
    }
    p->b_stages = 4;
    return;
  }
  for (const auto& dw : kDepths) {
    if (gemm_smem_bytes(p->block_m, dw[1], dw[0]) <= static_cast<size_t>(kMaxDynSmem)) {
      p->b_stages = 2 * dw[0];
      p->stages = dw[1];
      return;
    }
  }
}

// Trusted-routing validation off keeps a call capturable; on, the routing is
// copied back (after a stream synchronisation) and checked here.
w4a16_status validate_routing(const int32_t* sorted_ids, const int32_t* expert_ids,
                              const int32_t* num_tokens_padded, int capacity, int bm,
                              long long numel, int num_experts, cudaStream_t s) {
  if (cudaStreamSynchronize(s) != cudaSuccess) return W4A16_ERR_CUDA;
  int ntp = 0;
  if (cudaMemcpy(&ntp, num_tokens_padded, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return W4A16_ERR_CUDA;
  if (ntp < 0 || ntp > capacity || ntp % bm != 0) return W4A16_ERR_ROUTING;
  std::vector<int32_t> eid(ntp / bm), sid(ntp);
  if (ntp > 0) {
    if (cudaMemcpy(eid.data(), expert_ids, eid.size() * 4, cudaMemcpyDeviceToHost) !=
            cudaSuccess ||
        cudaMemcpy(sid.data(), sorted_ids, sid.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
      return W4A16_ERR_CUDA;
  }
  for (size_t b = 0; b < eid.size(); ++b) {
    if (eid[b] < -1 || eid[b] >= num_experts) return W4A16_ERR_ROUTING;
    for (int j = 0; j < bm; ++j) {
      const int id = sid[b * bm + j];
      if (id < 0 || id > numel) return W4A16_ERR_ROUTING;
    }
  }
  return W4A16_OK;
}

int current_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  return device_sm_count(dev);
}

}  // namespace

extern "C" {

const char* w4a16_status_string(int status) {
  switch (status) {
    case W4A16_OK: return "ok";
    case W4A16_ERR_INVALID_ARG: return "invalid argument";
    case W4A16_ERR_UNSUPPORTED: return "unsupported quantisation scheme or shape";
    case W4A16_ERR_ROUTING: return "routing tensors failed validation";
    case W4A16_ERR_WORKSPACE: return "workspace missing or too small";
    case W4A16_ERR_CUDA: return "CUDA error";
    case W4A16_ERR_TIMEOUT: return "a device-side wait gave up";
    default: return "unknown status";
  }
}

int w4a16_version(void) { return 122; }

w4a16_status w4a16_plan(int tokens, int topk, int num_experts, int n, int k, float tok_e_hint,
                        w4a16_plan_t* out) {
  if (out == nullptr || tokens < 0 || topk <= 0 || num_experts <= 0 || n <= 0 || k <= 0)
    return W4A16_ERR_INVALID_ARG;
  double tok_e = tok_e_hint > 0.f ? static_cast<double>(tok_e_hint)
                                  : static_cast<double>(tokens) * topk / num_experts;
  // tok_e decides the schedule (page "vLLM 宣布 Humming 后端可运行 … Chord 内核 …",
  // section "调度由每个专家收到的 token 数决定"; switch near 80 rows/expert).
  // Below the switch the block holds the expected rows of an expert with
  // headroom for the spread, so each weight tile streams once per expert;
  // above it the block is sized by padded expert rows. The MMA N of a block
  // is its real row count rounded to 16, so padding costs no tensor time.
  // Above the switch (GB300 measurements, 48 local experts): 64-row blocks
  // up to tok_e 120 (the skewed EP8 prefill shard, tok_e 81: layer 624 us at
  // 64, 697 at 128; uniform tok_e 128: 686 at 64, 576 at 128), then 128-row
  // blocks, whose BF16-staged
  // epilogue frees the accumulator before the stores and whose long
  // reductions take the grouped item order. They also beat 256-row blocks
  // (one 256-column accumulator slot, single-k-step activation slots) at
  // every heavier shape measured: gate_up at uniform tok_e 256 657 vs 708
  // us, at four times the EP8 prefill rows 967 vs 1132, at uniform tok_e 512
  // 1269 vs 1334. 256-row blocks stay available to an explicit plan.
  int block_m;
  if (tok_e <= 80.0) {
    block_m = round_up(std::max(16, static_cast<int>(std::ceil(1.5 * tok_e))), 16);
    block_m = std::min(block_m, 64);
  } else if (tok_e < 120.0) {
    block_m = 64;
  } else {
    block_m = 128;
  }
  w4a16_plan_t p;
  std::memset(&p, 0, sizeof(p));
  p.block_m = block_m;
  p.bn = kTileRows;
  p.bk = kKStep;
  set_ring_depths(&p);
  p.split_k = 1;
  p.ctas_per_sm = 1;
  p.swap_ab = 1;
  p.layout = W4A16_LAYOUT_KTILE64;
  p.grid = 0;
  *out = p;
  return W4A16_OK;
}

size_t w4a16_align_capacity(int numel, int num_experts, int block_m) {
  if (numel < 0 || num_experts <= 0 || block_m <= 0) return 0;
  const long long pad = static_cast<long long>(std::min(num_experts, numel)) * (block_m - 1);
  const long long cap = (static_cast<long long>(numel) + pad + block_m - 1) / block_m * block_m;
  return static_cast<size_t>(cap);
}

w4a16_status w4a16_moe_align_block_size(const int32_t* topk_ids, int tokens, int topk,
                                        int num_experts, int block_m, int capacity,
                                        int32_t* sorted_ids, int32_t* expert_ids,
                                        int32_t* num_tokens_padded, void* stream) {
  if (tokens < 0 || topk <= 0 || num_experts <= 0 || block_m <= 0 || capacity < 0)
    return W4A16_ERR_INVALID_ARG;
  // arrays of zero elements may be NULL (num_tokens_padded always has one)
  if (num_tokens_padded == nullptr ||
      (capacity > 0 && (sorted_ids == nullptr || expert_ids == nullptr)))
    return W4A16_ERR_INVALID_ARG;
  const long long numel = static_cast<long long>(tokens) * topk;
  if (numel > 0 && topk_ids == nullptr) return W4A16_ERR_INVALID_ARG;
  if (numel >= (1LL << 30)) return W4A16_ERR_UNSUPPORTED;
  if (num_experts > 1024 || block_m > 1024) return W4A16_ERR_UNSUPPORTED;
  if (capacity % block_m != 0) return W4A16_ERR_INVALID_ARG;
  if (static_cast<size_t>(capacity) <
      w4a16_align_capacity(static_cast<int>(numel), num_experts, block_m))
    return W4A16_ERR_INVALID_ARG;
  return cuda_status(launch_align(topk_ids, static_cast<int>(numel), num_experts, block_m,
                                  capacity, sorted_ids, expert_ids, num_tokens_padded,
                                  static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_prepack_size(int num_experts, int n, int k, int group, int layout,
                                size_t* bytes) {
  if (bytes == nullptr || num_experts <= 0 || n <= 0 || k <= 0) return W4A16_ERR_INVALID_ARG;
  if (group != kGroup || k % kGroup != 0) return W4A16_ERR_UNSUPPORTED;
  if (layout != W4A16_LAYOUT_KTILE64 && layout != W4A16_LAYOUT_KTILE64_GLU16)
    return W4A16_ERR_UNSUPPORTED;
  // the interleaved gate/up layout pairs 64-row halves of the two projections
  if (layout == W4A16_LAYOUT_KTILE64_GLU16 && n % kTileRows != 0) return W4A16_ERR_UNSUPPORTED;
  *bytes = static_cast<size_t>(num_experts) * packed_expert_bytes(n, k);
  return W4A16_OK;
}

w4a16_status w4a16_prepack(const uint8_t* q, const uint16_t* scales, int num_experts, int n,
                           int k, int group, int layout, void* packed, size_t packed_bytes,
                           void* stream) {
  size_t need = 0;
  const w4a16_status st = w4a16_prepack_size(num_experts, n, k, group, layout, &need);
  if (st != W4A16_OK) return st;
  if (q == nullptr || scales == nullptr || packed == nullptr) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(packed) || (reinterpret_cast<uintptr_t>(scales) & 1u))
    return W4A16_ERR_INVALID_ARG;
  if (packed_bytes < need) return W4A16_ERR_INVALID_ARG;
  return cuda_status(launch_prepack(q, scales, num_experts, n, k, layout,
                                    static_cast<uint8_t*>(packed),
                                    static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_unpack(const void* packed, int num_experts, int n, int k, int layout,
                          uint8_t* q, uint16_t* scales, void* stream) {
  if (packed == nullptr || q == nullptr || scales == nullptr || num_experts <= 0 || n <= 0 ||
      k <= 0)
    return W4A16_ERR_INVALID_ARG;
  size_t bytes = 0;
  const w4a16_status st = w4a16_prepack_size(num_experts, n, k, kGroup, layout, &bytes);
  if (st != W4A16_OK) return st;
  if (!aligned16(q) || !aligned16(packed) || (reinterpret_cast<uintptr_t>(scales) & 1u))
    return W4A16_ERR_INVALID_ARG;
  return cuda_status(launch_unpack(static_cast<const uint8_t*>(packed), num_experts, n, k, layout,
                                   q, scales, static_cast<cudaStream_t>(stream)));
}

size_t w4a16_deterministic_bytes(int capacity, int n, int numel) {
  if (capacity < 0 || n <= 0 || numel < 0) return 0;
  return det_rows_bytes(capacity, n) + (static_cast<size_t>(numel) * 4 + 255) / 256 * 256;
}

w4a16_status w4a16_grouped_plan(int kind, int m, int expected_m, int n, int k,
                                w4a16_plan_t* out) {
  if (out == nullptr || m < 0 || n <= 0 || k <= 0) return W4A16_ERR_INVALID_ARG;
  if (kind != W4A16_GROUPED_CONTIGUOUS && kind != W4A16_GROUPED_MASKED)
    return W4A16_ERR_INVALID_ARG;
  // every expert's rows form whole blocks: tok_e is the expected rows of one
  // expert (its row budget), else all rows
  const int rows = expected_m > 0 ? expected_m : std::max(1, m);
  const w4a16_status st = w4a16_plan(rows, 1, 1, n, k, static_cast<float>(rows), out);
  if (st != W4A16_OK) return st;
  if (rows > 80) {
    // long experts: the widest block (MMA N 128), measured faster than 64 on
    // the contiguous layouts whose experts hold 128..1024 rows
    out->block_m = 128;
    set_ring_depths(out);
  }
  return W4A16_OK;
}

w4a16_status w4a16_plan_info(const w4a16_plan_t* plan, int k, w4a16_plan_info_t* out) {
  if (plan == nullptr || out == nullptr || k <= 0) return W4A16_ERR_INVALID_ARG;
  Pipeline pl;
  if (!plan_pipeline(*plan, k, &pl)) return W4A16_ERR_INVALID_ARG;
  // blocks above 128 rows: four issuer threads, of which an item uses 1, 2
  // or 4 by its MMA N
  out->mma_issuers = activation_slot_is_step(plan->block_m) ? 4 : pl.parts;
  out->acc_slots = pl.d_slots;
  out->acc_cols = pl.d_cols;
  // (blocks of 65..128 rows free it early for a BF16 output only)
  out->early_epilogue = early_epilogue(plan->block_m, kOutBf16, plan->cta_pair != 0) ? 1 : 0;
  out->w_stages = pl.w_stages;
  out->b_stages = pl.b_stages;
  out->smem_bytes = pl.smem;
  return W4A16_OK;
}

size_t w4a16_workspace_size(const w4a16_plan_t* plan, int rows, int k) {
  (void)plan;
  if (rows <= 0 || k <= 0) return kStatusBytes;
  return kStatusBytes + (permuted_bytes(rows, k) + 255) / 256 * 256;
}

w4a16_status w4a16_moe_indexed_gemm(int mode, const void* packed, int num_experts, int n, int k,
                                    const uint16_t* a, int tokens, int topk,
                                    const int32_t* sorted_ids, const int32_t* expert_ids,
                                    const int32_t* num_tokens_padded, int capacity,
                                    const float* topk_weights, void* out, int flags,
                                    const w4a16_plan_t* plan, void* workspace, size_t ws_bytes,
                                    void* stream) {
  return w4a16::indexed_gemm(mode, packed, num_experts, n, k, a, tokens, topk, sorted_ids,
                             expert_ids, num_tokens_padded, capacity, topk_weights, out, flags,
                             plan, workspace, ws_bytes, stream, false);
}

}  // extern "C"

namespace w4a16 {

w4a16_status indexed_gemm(int mode, const void* packed, int num_experts, int n, int k,
                          const uint16_t* a, int tokens, int topk, const int32_t* sorted_ids,
                          const int32_t* expert_ids, const int32_t* num_tokens_padded,
                          int capacity, const float* topk_weights, void* out, int flags,
                          const w4a16_plan_t* plan, void* workspace, size_t ws_bytes,
                          void* stream, bool noalloc) {
  if (mode != W4A16_GATE_UP && mode != W4A16_DOWN && mode != W4A16_GATE_UP_SILU)
    return W4A16_ERR_INVALID_ARG;
  if (num_experts <= 0 || n <= 0 || k <= 0 || tokens < 0 || topk <= 0 || capacity < 0)
    return W4A16_ERR_INVALID_ARG;
  if (k % kGroup != 0) return W4A16_ERR_UNSUPPORTED;
  // arrays of zero elements may be NULL: the output and the activation when
  // there are no tokens, the routing arrays when the capacity is 0
  if (plan == nullptr || packed == nullptr || num_tokens_padded == nullptr)
    return W4A16_ERR_INVALID_ARG;
  if (tokens > 0 && (a == nullptr || out == nullptr)) return W4A16_ERR_INVALID_ARG;
  if (capacity > 0 && (sorted_ids == nullptr || expert_ids == nullptr))
    return W4A16_ERR_INVALID_ARG;
  if (mode == W4A16_DOWN && tokens > 0 && topk_weights == nullptr) return W4A16_ERR_INVALID_ARG;
  if ((flags & ~(W4A16_FLAG_VALIDATE_ROUTING | W4A16_FLAG_ACCUMULATE |
                 W4A16_FLAG_DETERMINISTIC)) != 0)
    return W4A16_ERR_INVALID_ARG;
  const bool det = (flags & W4A16_FLAG_DETERMINISTIC) != 0;
  if (det && mode != W4A16_DOWN) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(packed) || !aligned16(out) || (a != nullptr && !aligned16(a)))
    return W4A16_ERR_INVALID_ARG;
  const size_t ws_base = w4a16_workspace_size(plan, capacity, k);
  const long long numel_all = static_cast<long long>(tokens) * topk;
  if (numel_all >= (1LL << 30)) return W4A16_ERR_UNSUPPORTED;
  const size_t ws_det =
      det ? w4a16_deterministic_bytes(capacity, n, static_cast<int>(numel_all)) : 0;
  if ((!noalloc && workspace == nullptr) || ws_bytes < ws_base + ws_det)
    return W4A16_ERR_WORKSPACE;
  Pipeline pl;
  if (!plan_pipeline(*plan, k, &pl)) return W4A16_ERR_INVALID_ARG;
  // the fused activation needs the interleaved gate/up packing, and only it
  const bool glu = mode == W4A16_GATE_UP_SILU;
  if (glu != (plan->layout == W4A16_LAYOUT_KTILE64_GLU16)) return W4A16_ERR_INVALID_ARG;
  if (glu && n % kTileRows != 0) return W4A16_ERR_UNSUPPORTED;
  const int bm = plan->block_m;
  if (capacity % bm != 0) return W4A16_ERR_INVALID_ARG;
  const long long numel = numel_all;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (flags & W4A16_FLAG_VALIDATE_ROUTING) {
    const w4a16_status vs = validate_routing(sorted_ids, expert_ids, num_tokens_padded, capacity,
                                             bm, numel, num_experts, s);
    if (vs != W4A16_OK) return vs;
  }
  // every check passed: only now may anything be enqueued. The library's
  // own scratch array keeps what the previous call left: its status word is
  // cleared first.
  if (noalloc) {
    workspace = noalloc_scratch_address();
    if (workspace == nullptr) return W4A16_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, kStatusBytes, s) != cudaSuccess) return W4A16_ERR_CUDA;
  }

  // the down pass adds into `out`: zeroed first unless ACCUMULATE (by the
  // row-permute kernel below, or here when there is nothing to multiply)
  const size_t zero_bytes = (mode == W4A16_DOWN && !(flags & W4A16_FLAG_ACCUMULATE))
                                ? static_cast<size_t>(tokens) * n * sizeof(float)
                                : 0;
  if (numel == 0 || capacity == 0) {
    if (zero_bytes > 0 && cudaMemsetAsync(out, 0, zero_bytes, s) != cudaSuccess)
      return W4A16_ERR_CUDA;
    return W4A16_OK;
  }
  // deterministic down pass: the GEMM stores the weighted rows in the
  // workspace (after the routed rows) and a per-token ordered sum writes
  // every element of `out`, so nothing is zeroed first
  float* det_rows = nullptr;
  int32_t* det_inv = nullptr;
  if (det) {
    det_rows = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ws_base);
    det_inv = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(det_rows) +
                                         det_rows_bytes(capacity, n));
  }
  const size_t zero_now = det ? 0 : zero_bytes;

  GemmArgs g;
  std::memset(&g, 0, sizeof(g));
  g.wpack = static_cast<const uint8_t*>(packed);
  g.expert_bytes = static_cast<long long>(packed_expert_bytes(n, k));
  g.num_experts = num_experts;
  g.n = n;
  g.k = k;
  g.n_tiles = packed_tiles(n);
  g.k_steps = packed_ksteps(k);
  // routed rows into routing order (after the status block of the workspace)
  const int sms = current_sm_count();
  if (sms <= 0) return W4A16_ERR_CUDA;
  uint16_t* permuted =
      reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + kStatusBytes);
  const int a_div = mode == W4A16_DOWN ? 1 : topk;
  // CTA pairs: each CTA of a pair loads half of a block's rows
  const bool pair = plan->cta_pair != 0 && packed_tiles(n) % 2 == 0;
  const bool step_slots = !pair && activation_slot_is_step(bm);
  if (!encode_permuted_tmap(&g.tmap, permuted, capacity, permuted_row_elems(k),
                            activation_box_rows(bm, pair), step_slots ? 1 : 2) ||
      (step_slots && !encode_permuted_tmap(&g.tmap2, permuted, capacity, permuted_row_elems(k),
                                           kActivationBoxRowsSmall, 1)))
    return W4A16_ERR_CUDA;
  // (n * 4 bytes per row is a multiple of 16 when n % 4 == 0; otherwise the
  // tail is cleared separately)
  const size_t zero_vec_bytes = zero_now / 16 * 16;
  if (zero_now != zero_vec_bytes &&
      cudaMemsetAsync(static_cast<uint8_t*>(out) + zero_vec_bytes, 0, zero_now - zero_vec_bytes,
                      s) != cudaSuccess)
    return W4A16_ERR_CUDA;
  if (det && launch_det_inverse(sorted_ids, num_tokens_padded, capacity, static_cast<int>(numel),
                                det_inv, sms, s) != cudaSuccess)
    return W4A16_ERR_CUDA;
  if (launch_permute_rows(a, k, a_div, static_cast<int>(numel), sorted_ids, num_tokens_padded,
                          capacity, permuted, out, zero_vec_bytes, sms, s) != cudaSuccess)
    return W4A16_ERR_CUDA;
  g.act = permuted;
  g.gather_rows = 1;
  g.act_rows = capacity;
  g.family = kIndexed;
  g.out_mode = det                  ? kOutF32Rows
               : mode == W4A16_DOWN ? kOutF32WeightedAdd
               : (glu ? kOutGluBf16 : kOutBf16);
  g.sorted_ids = sorted_ids;
  g.expert_ids = expert_ids;
  g.num_tokens_padded = num_tokens_padded;
  g.capacity = capacity;
  g.numel = static_cast<int>(numel);
  g.a_div = a_div;
  g.o_div = mode == W4A16_DOWN ? topk : 1;
  g.topk_weights = topk_weights;
  g.block_m = bm;
  g.out = det ? static_cast<void*>(det_rows) : out;
  g.status = static_cast<int*>(workspace);
  fill_pipeline(pl, &g);
  // 256-row blocks come with tok_e >= 200 and long reductions: the routed
  // rows (hundreds of MB) exceed L2, and in tile-major order every weight
  // tile pass would read them from DRAM again (EP8 prefill at four times the
  // rows: 5.7 GB of DRAM reads per gate_up launch); grouped in blocks of 8,
  // a group's rows stay in L2 across its tiles
  // ... and blocks of 48..128 rows over a long reduction: the routed rows
  // of a prefill gate_up (EP8 prefill: 78 MB) are re-read per tile pass in
  // tile-major order (EP8 prefill gate_up 379 -> 368.5 us; 128-row blocks at
  // tok_e 163: 652 -> 557 us)
  g.raster_rows = (step_slots || (!pair && bm > 32 && k > 2048)) ? 1 : 0;
  g.timeout_cycles = wait_timeout_cycles();
  g.pair = pair ? 1 : 0;
  long long grid = plan->grid > 0 ? plan->grid : static_cast<long long>(sms) * plan->ctas_per_sm;
  const long long max_items = static_cast<long long>(capacity / bm) * g.n_tiles;
  grid = std::max<long long>(1, std::min(grid, max_items));
  if (pair) {
    const int clusters = max_pair_clusters(g);
    if (clusters <= 0) return W4A16_ERR_CUDA;
    grid = 2 * std::max<long long>(1, std::min<long long>(grid / 2, clusters));
  }
  if (launch_moe_gemm(g, static_cast<int>(grid), true, s) != cudaSuccess) return W4A16_ERR_CUDA;
  if (det && launch_det_reduce(det_rows, det_inv, tokens, topk, n,
                               (flags & W4A16_FLAG_ACCUMULATE) != 0, static_cast<float*>(out), sms,
                               s) != cudaSuccess)
    return W4A16_ERR_CUDA;
  return W4A16_OK;
}

}  // namespace w4a16

extern "C" {

w4a16_status w4a16_moe_grouped_gemm(int kind, const void* packed, int num_experts, int n, int k,
                                    const uint16_t* a, int m, const int32_t* layout,
                                    int expected_m, uint16_t* out, int flags,
                                    const w4a16_plan_t* plan, void* workspace, size_t ws_bytes,
                                    void* stream) {
  if (kind != W4A16_GROUPED_CONTIGUOUS && kind != W4A16_GROUPED_MASKED)
    return W4A16_ERR_INVALID_ARG;
  if (num_experts <= 0 || n <= 0 || k <= 0 || m < 0) return W4A16_ERR_INVALID_ARG;
  if (k % kGroup != 0) return W4A16_ERR_UNSUPPORTED;
  // arrays of zero elements may be NULL: a, out and the contiguous layout
  // when m is 0 (the masked layout always has num_experts entries)
  if (packed == nullptr) return W4A16_ERR_INVALID_ARG;
  if (m > 0 && (a == nullptr || out == nullptr || layout == nullptr)) return W4A16_ERR_INVALID_ARG;
  if (kind == W4A16_GROUPED_MASKED && layout == nullptr) return W4A16_ERR_INVALID_ARG;
  if ((flags & ~W4A16_FLAG_VALIDATE_ROUTING) != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(packed) || !aligned16(out) || (a != nullptr && !aligned16(a)))
    return W4A16_ERR_INVALID_ARG;
  w4a16_plan_t local;
  if (plan == nullptr) {
    const w4a16_status ps = w4a16_grouped_plan(kind, m, expected_m, n, k, &local);
    if (ps != W4A16_OK) return ps;
    plan = &local;
  }
  if (workspace == nullptr || ws_bytes < kStatusBytes) return W4A16_ERR_WORKSPACE;
  Pipeline pl;
  if (!plan_pipeline(*plan, k, &pl) || plan->layout != W4A16_LAYOUT_KTILE64)
    return W4A16_ERR_INVALID_ARG;
  const int bm = plan->block_m;
  const long long rows_total =
      kind == W4A16_GROUPED_MASKED ? static_cast<long long>(num_experts) * m : m;
  if (rows_total >= (1LL << 30)) return W4A16_ERR_UNSUPPORTED;
  if (kind == W4A16_GROUPED_CONTIGUOUS && (128 % bm != 0 || m % bm != 0))
    return W4A16_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (flags & W4A16_FLAG_VALIDATE_ROUTING) {
    if (cudaStreamSynchronize(s) != cudaSuccess) return W4A16_ERR_CUDA;
    const int cnt = kind == W4A16_GROUPED_CONTIGUOUS ? m : num_experts;
    std::vector<int32_t> lay(cnt);
    if (cnt > 0 &&
        cudaMemcpy(lay.data(), layout, cnt * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
      return W4A16_ERR_CUDA;
    if (kind == W4A16_GROUPED_CONTIGUOUS) {
      for (int b0 = 0; b0 < m; b0 += 128) {
        const int head = lay[b0];
        for (int r = b0; r < std::min(m, b0 + 128); ++r) {
          if (lay[r] < -1 || lay[r] >= num_experts) return W4A16_ERR_ROUTING;
          if (lay[r] >= 0 && lay[r] != head) return W4A16_ERR_ROUTING;
        }
      }
    } else {
      for (int e = 0; e < num_experts; ++e)
        if (lay[e] < 0 || lay[e] > m) return W4A16_ERR_ROUTING;
    }
  }
  if (rows_total == 0) return W4A16_OK;

  GemmArgs g;
  std::memset(&g, 0, sizeof(g));
  g.wpack = static_cast<const uint8_t*>(packed);
  g.expert_bytes = static_cast<long long>(packed_expert_bytes(n, k));
  g.num_experts = num_experts;
  g.n = n;
  g.k = k;
  g.n_tiles = packed_tiles(n);
  g.k_steps = packed_ksteps(k);
  g.act = a;
  g.act_rows = static_cast<int>(rows_total);
  const bool pair = plan->cta_pair != 0 && g.n_tiles % 2 == 0;
  const bool step_slots = !pair && activation_slot_is_step(bm);
  // k a multiple of 64 (two-step slots): the rows seen as the 3-D array
  // (64 columns, rows, k / 64), so that one tensor copy brings both k steps
  // of a stage, as for the indexed family's permuted rows (grouped masked,
  // budget 32: gate_up 236 -> 208 us, down 126 -> 113 us); else one 2-D copy
  // per k step
  const bool two_step_copies = !step_slots && k % kKStep == 0;
  g.gather_rows = two_step_copies ? 1 : 0;
  if (two_step_copies) {
    if (!encode_permuted_tmap(&g.tmap, a, rows_total, k, activation_box_rows(bm, pair), 2))
      return W4A16_ERR_CUDA;
  } else if (!encode_act_tmap(&g.tmap, a, rows_total, k, activation_box_rows(bm, pair)) ||
             (step_slots &&
              !encode_act_tmap(&g.tmap2, a, rows_total, k, kActivationBoxRowsSmall))) {
    return W4A16_ERR_CUDA;
  }
  g.family = kind == W4A16_GROUPED_CONTIGUOUS ? kContiguous : kMasked;
  g.out_mode = kOutBf16;
  g.layout = layout;
  g.m = m;
  g.block_m = bm;
  g.out = out;
  g.status = static_cast<int*>(workspace);
  fill_pipeline(pl, &g);
  // group the item order once all token rows are a good part of L2 (129 MB)
  g.raster_rows = static_cast<double>(rows_total) * k * 2.0 > 64.0 * (1 << 20) ? 1 : 0;
  g.timeout_cycles = wait_timeout_cycles();
  const int sms = current_sm_count();
  if (sms <= 0) return W4A16_ERR_CUDA;
  const long long blocks = kind == W4A16_GROUPED_CONTIGUOUS
                               ? m / bm
                               : static_cast<long long>(num_experts) * ((m + bm - 1) / bm);
  g.pair = pair ? 1 : 0;
  long long grid = plan->grid > 0 ? plan->grid : static_cast<long long>(sms) * plan->ctas_per_sm;
  grid = std::max<long long>(1, std::min(grid, blocks * g.n_tiles));
  if (pair) {
    const int clusters = max_pair_clusters(g);
    if (clusters <= 0) return W4A16_ERR_CUDA;
    grid = 2 * std::max<long long>(1, std::min<long long>(grid / 2, clusters));
  }
  return cuda_status(launch_moe_gemm(g, static_cast<int>(grid), false, s));
}

w4a16_status w4a16_topk_softmax(const void* logits, int logits_dtype, int tokens,
                                int num_experts, int topk, int renormalize, int expert_offset,
                                int num_local_experts, int32_t* topk_ids, float* topk_weights,
                                void* stream) {
  if (tokens < 0 || num_experts <= 0 || topk <= 0 || num_local_experts < 0)
    return W4A16_ERR_INVALID_ARG;
  if (logits_dtype != W4A16_DTYPE_F32 && logits_dtype != W4A16_DTYPE_BF16)
    return W4A16_ERR_INVALID_ARG;
  if (num_experts > 1024 || topk > 32 || topk > num_experts) return W4A16_ERR_UNSUPPORTED;
  if (tokens > 0 && (logits == nullptr || topk_ids == nullptr || topk_weights == nullptr))
    return W4A16_ERR_INVALID_ARG;
  const int sms = current_sm_count();
  if (sms <= 0) return W4A16_ERR_CUDA;
  return cuda_status(launch_topk_softmax(logits, logits_dtype == W4A16_DTYPE_BF16, tokens,
                                         num_experts, topk, renormalize != 0, expert_offset,
                                         num_local_experts, topk_ids, topk_weights, sms,
                                         static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_moe_route_align(const void* logits, int logits_dtype, int tokens,
                                   int num_experts, int topk, int renormalize, int expert_offset,
                                   int num_local_experts, int block_m, int capacity,
                                   int32_t* topk_ids, float* topk_weights, int32_t* sorted_ids,
                                   int32_t* expert_ids, int32_t* num_tokens_padded,
                                   uint32_t* arrivals, void* stream) {
  if (tokens < 0 || num_experts <= 0 || topk <= 0 || num_local_experts <= 0 || block_m <= 0 ||
      capacity < 0)
    return W4A16_ERR_INVALID_ARG;
  if (logits_dtype != W4A16_DTYPE_F32 && logits_dtype != W4A16_DTYPE_BF16)
    return W4A16_ERR_INVALID_ARG;
  if (num_experts > 1024 || topk > 32 || topk > num_experts) return W4A16_ERR_UNSUPPORTED;
  if (num_local_experts > 1024 || block_m > 1024) return W4A16_ERR_UNSUPPORTED;
  const long long numel = static_cast<long long>(tokens) * topk;
  if (numel >= (1LL << 30)) return W4A16_ERR_UNSUPPORTED;
  // arrays of zero elements may be NULL (the routing arrays at capacity 0)
  if (num_tokens_padded == nullptr || arrivals == nullptr ||
      (capacity > 0 && (sorted_ids == nullptr || expert_ids == nullptr)))
    return W4A16_ERR_INVALID_ARG;
  if (tokens > 0 && (logits == nullptr || topk_ids == nullptr || topk_weights == nullptr))
    return W4A16_ERR_INVALID_ARG;
  if (capacity % block_m != 0) return W4A16_ERR_INVALID_ARG;
  if (static_cast<size_t>(capacity) <
      w4a16_align_capacity(static_cast<int>(numel), num_local_experts, block_m))
    return W4A16_ERR_INVALID_ARG;
  const int sms = current_sm_count();
  if (sms <= 0) return W4A16_ERR_CUDA;
  return cuda_status(launch_route_align(
      logits, logits_dtype == W4A16_DTYPE_BF16, tokens, num_experts, topk, renormalize != 0,
      expert_offset, num_local_experts, block_m, capacity, topk_ids, topk_weights, sorted_ids,
      expert_ids, num_tokens_padded, arrivals, sms, static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_silu_and_mul(const uint16_t* in, int rows, int inter, uint16_t* out,
                                void* stream) {
  if (rows < 0 || inter <= 0 || inter % 8 != 0) return W4A16_ERR_INVALID_ARG;
  if (rows > 0 && (in == nullptr || out == nullptr)) return W4A16_ERR_INVALID_ARG;
  if (rows > 0 && (!aligned16(in) || !aligned16(out))) return W4A16_ERR_INVALID_ARG;
  return cuda_status(launch_silu_and_mul(in, rows, inter, out, static_cast<cudaStream_t>(stream)));
}

size_t w4a16_layer_workspace_size(const w4a16_plan_t* plan, int rows, int hidden, int inter) {
  if (plan == nullptr || plan->block_m <= 0 || rows <= 0 || hidden <= 0 || inter <= 0)
    return kStatusBytes;
  const size_t flags_bytes = (static_cast<size_t>(rows / plan->block_m + 1) * 4 + 255) / 256 * 256;
  return kStatusBytes + (permuted_bytes(rows, hidden) + 255) / 256 * 256 +
         (permuted_bytes(rows, inter) + 255) / 256 * 256 + flags_bytes;
}

w4a16_status w4a16_moe_layer(const void* packed_gate_up, const void* packed_down, int num_experts,
                             int hidden, int inter, const uint16_t* x, int tokens, int topk,
                             const int32_t* sorted_ids, const int32_t* expert_ids,
                             const int32_t* num_tokens_padded, int capacity,
                             const float* topk_weights, float* out, int flags,
                             const w4a16_plan_t* plan, void* workspace, size_t ws_bytes,
                             void* stream) {
  if (num_experts <= 0 || hidden <= 0 || inter <= 0 || tokens < 0 || topk <= 0 || capacity < 0)
    return W4A16_ERR_INVALID_ARG;
  if (hidden % kGroup != 0 || inter % 64 != 0 || hidden % 4 != 0) return W4A16_ERR_UNSUPPORTED;
  // arrays of zero elements may be NULL: x, the weights and the output when
  // there are no tokens, the routing arrays when the capacity is 0
  if (plan == nullptr || packed_gate_up == nullptr || packed_down == nullptr ||
      num_tokens_padded == nullptr)
    return W4A16_ERR_INVALID_ARG;
  if (tokens > 0 && (x == nullptr || topk_weights == nullptr || out == nullptr))
    return W4A16_ERR_INVALID_ARG;
  if (capacity > 0 && (sorted_ids == nullptr || expert_ids == nullptr))
    return W4A16_ERR_INVALID_ARG;
  if ((flags & ~(W4A16_FLAG_VALIDATE_ROUTING | W4A16_FLAG_ACCUMULATE)) != 0)
    return W4A16_ERR_INVALID_ARG;
  if (!aligned16(packed_gate_up) || !aligned16(packed_down) || !aligned16(out) ||
      (x != nullptr && !aligned16(x)))
    return W4A16_ERR_INVALID_ARG;
  // the gate_up weights carry the interleaved gate/up packing of the fused
  // activation; the layer runs unpaired, on blocks of at most 128 rows
  if (plan->layout != W4A16_LAYOUT_KTILE64_GLU16 || plan->cta_pair != 0 ||
      activation_slot_is_step(plan->block_m))
    return W4A16_ERR_INVALID_ARG;
  Pipeline pl;
  if (!plan_pipeline(*plan, std::max(hidden, inter), &pl)) return W4A16_ERR_INVALID_ARG;
  const int bm = plan->block_m;
  if (capacity % bm != 0) return W4A16_ERR_INVALID_ARG;
  const long long numel = static_cast<long long>(tokens) * topk;
  if (numel >= (1LL << 30)) return W4A16_ERR_UNSUPPORTED;
  if (workspace == nullptr || ws_bytes < w4a16_layer_workspace_size(plan, capacity, hidden, inter))
    return W4A16_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (flags & W4A16_FLAG_VALIDATE_ROUTING) {
    const w4a16_status vs = validate_routing(sorted_ids, expert_ids, num_tokens_padded, capacity,
                                             bm, numel, num_experts, s);
    if (vs != W4A16_OK) return vs;
  }
  const size_t zero_bytes = (flags & W4A16_FLAG_ACCUMULATE)
                                ? 0
                                : static_cast<size_t>(tokens) * hidden * sizeof(float);
  if (numel == 0 || capacity == 0) {
    if (zero_bytes > 0 && cudaMemsetAsync(out, 0, zero_bytes, s) != cudaSuccess)
      return W4A16_ERR_CUDA;
    return W4A16_OK;
  }
  const int sms = current_sm_count();
  if (sms <= 0) return W4A16_ERR_CUDA;
  // workspace: status words, x rows in routing order, activation rows in
  // routing order, one completion counter per routing block
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* x_sorted = reinterpret_cast<uint16_t*>(ws + kStatusBytes);
  uint16_t* act_sorted = reinterpret_cast<uint16_t*>(
      ws + kStatusBytes + (permuted_bytes(capacity, hidden) + 255) / 256 * 256);
  int* block_done = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(act_sorted) +
                                           (permuted_bytes(capacity, inter) + 255) / 256 * 256);
  const int blocks = capacity / bm;
  GemmArgs g;
  std::memset(&g, 0, sizeof(g));
  g.wpack = static_cast<const uint8_t*>(packed_gate_up);
  g.expert_bytes = static_cast<long long>(packed_expert_bytes(2 * inter, hidden));
  g.num_experts = num_experts;
  g.n = 2 * inter;
  g.k = hidden;
  g.n_tiles = packed_tiles(2 * inter);
  g.k_steps = packed_ksteps(hidden);
  g.wpack2 = static_cast<const uint8_t*>(packed_down);
  g.expert_bytes2 = static_cast<long long>(packed_expert_bytes(hidden, inter));
  g.n2 = hidden;
  g.n_tiles2 = packed_tiles(hidden);
  g.k_steps2 = packed_ksteps(inter);
  if (!encode_permuted_tmap(&g.tmap, x_sorted, capacity, permuted_row_elems(hidden), bm, 2) ||
      !encode_permuted_tmap(&g.tmap2, act_sorted, capacity, inter, bm, 2))
    return W4A16_ERR_CUDA;
  if (cudaMemsetAsync(block_done, 0, static_cast<size_t>(blocks) * 4, s) != cudaSuccess)
    return W4A16_ERR_CUDA;
  const size_t zero_vec_bytes = zero_bytes / 16 * 16;
  if (zero_bytes != zero_vec_bytes &&
      cudaMemsetAsync(reinterpret_cast<uint8_t*>(out) + zero_vec_bytes, 0,
                      zero_bytes - zero_vec_bytes, s) != cudaSuccess)
    return W4A16_ERR_CUDA;
  if (launch_permute_rows(x, hidden, topk, static_cast<int>(numel), sorted_ids, num_tokens_padded,
                          capacity, x_sorted, out, zero_vec_bytes, sms, s) != cudaSuccess)
    return W4A16_ERR_CUDA;
  g.act = x_sorted;
  g.gather_rows = 1;
  g.act_rows = capacity;
  g.family = kIndexed;
  g.out_mode = kOutGluBf16;
  g.sorted_ids = sorted_ids;
  g.expert_ids = expert_ids;
  g.num_tokens_padded = num_tokens_padded;
  g.capacity = capacity;
  g.numel = static_cast<int>(numel);
  g.a_div = topk;
  g.o_div = topk;
  g.topk_weights = topk_weights;
  g.block_m = bm;
  g.out = act_sorted;
  g.out2 = out;
  g.block_done = block_done;
  g.layer = 1;
  g.status = static_cast<int*>(workspace);
  fill_pipeline(pl, &g);
  g.timeout_cycles = wait_timeout_cycles();
  long long grid = plan->grid > 0 ? plan->grid : static_cast<long long>(sms) * plan->ctas_per_sm;
  // every CTA must be resident at once (down items wait on other CTAs'
  // gate_up items): at most one CTA per SM
  grid = std::max<long long>(1, std::min<long long>(grid, sms));
  grid = std::min<long long>(grid, static_cast<long long>(blocks) * (g.n_tiles + g.n_tiles2));
  if (launch_moe_gemm(g, static_cast<int>(grid), true, s) != cudaSuccess) return W4A16_ERR_CUDA;
  return W4A16_OK;
}

w4a16_status w4a16_read_device_status(void* workspace, int* detail, void* stream) {
  if (workspace == nullptr) return W4A16_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return W4A16_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return W4A16_ERR_CUDA;
  if (detail != nullptr) *detail = word;
  if (word == 0) return W4A16_OK;
  if (cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return W4A16_ERR_CUDA;
  return W4A16_ERR_TIMEOUT;
}

}  // extern "C"
