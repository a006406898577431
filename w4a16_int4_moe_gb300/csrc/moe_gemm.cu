// moe_gemm.cu -- the W4A16 MoE expert GEMM on sm_103a tensor cores.
//
// One kernel serves gate_up, down and both grouped layouts of the
// Chord/Humming operator (page "vLLM 宣布 Humming 后端可运行 … Chord 内核 …",
// sections "调度由每个专家收到的 token 数决定" and "六个场景的逐层测量与限定条件";
// page "vLLM と Novita AI が Chord をリリース …", section
// "カーネルレベルの最適化"). The pages' decode kernel swaps the MMA operands so
// that the dequantised weight takes the MMA M side; this kernel does the same
// for every shape and builds it on tcgen05:
//
//   weights (packed uint4 + BF16 scales) --bulk copy--> shared-memory ring
//     --dequant warpgroups: (q - 8) * s in registers, tcgen05.st--> TMEM (A)
//   tokens --TMA tensor copies, 128-byte swizzle--> shared-memory ring (B):
//     the indexed family's routed rows, copied once into routing order
//     (permute.cu), arrive two k steps per copy; the grouped families' rows
//     one k step per copy
//   tcgen05.mma kind::f16, M = 128 weight rows, N = the block's tokens
//     (rounded to 16, chosen per block at run time), K = 16 per instruction,
//     FP32 accumulators in TMEM (D)
//   epilogue warps: tcgen05.ld --> BF16 row stores, the top-k weighted FP32
//     scatter-add of the down pass, or (deterministic down pass) the
//     weighted FP32 rows at their routing positions.
//
// Writing the dequantised weights to TMEM instead of shared memory keeps the
// shared-memory port free for the token operand: at decode (N = 16) a
// shared-memory A operand would cost more shared bandwidth than the HBM
// stream delivers weights.
//
// The pipeline moves in stages of two 64-k steps (9216 bytes of packed
// weights): every handshake is paid once per stage, four dequant warpgroups
// work on four consecutive stages, and up to four MMA issuers split the k
// steps (one thread issues a tcgen05.mma only every 100-125 cycles whatever N
// is, measured on GB300, so at small N the issue rate, not the tensor core,
// sets the pace). Each issuer
// owns a partial FP32 accumulator; the epilogue adds them in a fixed order,
// so results do not depend on the schedule.
//
// Work item = (routing block, 128-row weight tile), full K. Persistent grid;
// CTA c takes items c, c + grid, ... Every device-side wait is bounded: a wait
// that runs out sets the workspace status word, all roles leave their loops,
// and the CTA frees its TMEM and exits.

#include <cuda_bf16.h>

#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

// Role timing for development builds (-DW4A16_ROLE_PROFILE): each warp adds
// the SM cycles between consecutive marks into per-category counters, stored
// per CTA and warp when it finishes. Compiled out otherwise.
#ifdef W4A16_ROLE_PROFILE
__device__ long long g_w4a16_role_prof[256][32][8];
#define W4A16_PROF_DECL                 \
  long long prof_acc_[8] = {0};         \
  long long prof_t_ = clock64();
#define W4A16_PROF_MARK(i)              \
  do {                                  \
    const long long t_ = clock64();     \
    prof_acc_[i] += t_ - prof_t_;       \
    prof_t_ = t_;                       \
  } while (0)
#define W4A16_PROF_STORE()                                                        \
  do {                                                                            \
    if ((threadIdx.x & 31) == 0 && blockIdx.x < 256)                              \
      for (int i_ = 0; i_ < 8; ++i_)                                              \
        g_w4a16_role_prof[blockIdx.x][threadIdx.x >> 5][i_] = prof_acc_[i_];      \
  } while (0)
extern "C" int w4a16_debug_role_profile(long long* out, int bytes) {
  const int n = bytes < static_cast<int>(sizeof(g_w4a16_role_prof))
                    ? bytes : static_cast<int>(sizeof(g_w4a16_role_prof));
  return cudaMemcpyFromSymbol(out, g_w4a16_role_prof, n) == cudaSuccess ? 0 : 1;
}
#else
#define W4A16_PROF_DECL
#define W4A16_PROF_MARK(i)
#define W4A16_PROF_STORE()
#endif

namespace w4a16 {

namespace {

constexpr int kThreads = 864;
constexpr int kWStageBytes = 2 * kStepBytes;  // one stage = 2 k steps of packed weights
constexpr int kASlots = 4;                    // A slots in TMEM = dequant warpgroups
constexpr int kAColsPerSlot = 64;             // 2 k steps x 64 BF16 of K per TMEM lane
constexpr int kAColsPerStep = 32;
constexpr int kItemSlots = 8;                 // routing-info ring depth (items)
constexpr int kMaxDSlots = 4;                 // accumulator slots (items in flight in TMEM)
constexpr int kMaxIssuers = 4;
constexpr int kTmemCols = 512;
// Epilogue staging rows per warp: the whole block for blocks of 48 or 64 rows
// (so that the accumulator slot is freed before the stores), else 16 rows: a
// block of up to 32 rows mostly holds at most 16 (decode), and the shared
// memory of blocks above 64 rows goes to the activation ring.
__host__ __device__ constexpr int epi_stage_rows(int block_m) {
  return (block_m > 32 && block_m <= 64) ? (block_m + 15) / 16 * 16 : 16;
}
__host__ __device__ constexpr int epi_tile_bytes(int block_m) {
  return 4 * epi_stage_rows(block_m) * 32 * 4;  // 4 epilogue warps x rows x 32 FP32
}
// Blocks of 65..128 rows with a BF16 output stage the whole block as BF16
// (32 KB at 128 rows, a region of its own after the rest of the carve-up), so
// that their accumulator slot, the only one, is freed before the stores too.
__host__ __device__ constexpr bool epi_half_stage(int block_m) {
  return block_m > 64 && block_m <= 128;
}
__host__ __device__ constexpr int epi_half_bytes(int block_m) {
  return epi_half_stage(block_m) ? 4 * block_m * 32 * 2 : 0;  // 4 warps x rows x 32 BF16
}
// Blocks above 128 rows: one 64-k step of token rows is up to 32 KB, so the
// activation ring holds single k steps (two stage-sized slots would leave
// room for too few in flight), and the one MMA issuer waits on each k step.
__host__ __device__ constexpr bool b_per_step(int block_m) {
  return activation_slot_is_step(block_m);
}
// Blocks above 128 rows: the 256 accumulator columns hold P partial
// accumulators of 256 / P columns, P chosen per item from its MMA N: four
// issuers up to 64 token rows, two up to 128, one above (one thread issues a
// tcgen05.mma only every hundred-odd cycles, so small N needs several).
constexpr int kBigAccCols = 256;
constexpr int kSmallBoxRows = kActivationBoxRowsSmall;  // token rows per copy of tmap2
__device__ __forceinline__ int big_block_parts(int n16) {
  return n16 <= 64 ? 4 : (n16 <= 128 ? 2 : 1);
}

// Warp roles. The dequant and epilogue warpgroups start at multiples of 4
// warps, so that warp % 4 selects the TMEM lane quarter each warp may access.
constexpr int kWarpProducer = 0;    // weight bulk copies
constexpr int kWarpMma0 = 1;        // MMA issuers 0..2 in warps 1..3 (warp 1 allocates TMEM)
constexpr int kWarpDequant0 = 4;    // 16 warps: 4 warpgroups, one per A slot
constexpr int kWarpEpilogue0 = 20;  // 4 warps
constexpr int kWarpMma3 = 24;       // MMA issuer 3
constexpr int kWarpGather = 25;     // activation rows
constexpr int kWarpRouter = 26;     // per-item routing info, items ahead of the MMA

// where codes recorded in the status word when a wait gives up
enum Where {
  kWhereProducer = 1, kWhereDequantW = 2, kWhereDequantA = 3, kWhereGatherItem = 4,
  kWhereGatherB = 5, kWhereMmaItem = 6, kWhereMmaAcc = 7, kWhereMmaA = 8, kWhereMmaB = 9,
  kWhereEpiAcc = 10, kWhereEpiItem = 11, kWhereDrain = 12, kWhereRouter = 13, kWhereRelay = 14,
  kWhereBlockDone = 15
};

struct Smem {
  uint8_t* b_ring;      // [BS slots][2 k steps, or 1 (b_per_step)][block_m rows][128 B], 128-byte swizzle
  uint8_t* w_ring;      // [WS stages][2 k steps][kStepBytes]
  int* info_dst;        // [kItemSlots][block_m]: output row, -1 = not a real row
  float* info_wt;       // [kItemSlots][block_m]: top-k weight (down pass)
  int* info_n16;        // [kItemSlots]: MMA N of the item
  int* info_rows;       // [kItemSlots]: real rows (last real row + 1)
  float* epi_tile;      // [4 epilogue warps][stage rows][32 weight rows]
  uint64_t* bars;
  uint32_t* tmem_base;
  volatile int* abort_flag;
  __nv_bfloat16* epi_half;  // (kEarly) [4 warps][block_m token rows][32]: BF16 staging
};

// mbarrier addresses (shared-window offsets, 8 bytes each)
struct Bars {
  uint32_t w_full, w_empty, a_full, a_empty, b_full, b_empty, item_full, item_empty, acc_full,
      acc_empty, final_bar;
  __device__ uint32_t wf(int i) const { return w_full + 8u * i; }
  __device__ uint32_t we(int i) const { return w_empty + 8u * i; }
  __device__ uint32_t af(int i) const { return a_full + 8u * i; }
  __device__ uint32_t ae(int i) const { return a_empty + 8u * i; }
  __device__ uint32_t bf(int i) const { return b_full + 8u * i; }
  __device__ uint32_t be(int i) const { return b_empty + 8u * i; }
  __device__ uint32_t itf(int i) const { return item_full + 8u * i; }
  __device__ uint32_t ite(int i) const { return item_empty + 8u * i; }
  __device__ uint32_t accf(int i) const { return acc_full + 8u * i; }
  __device__ uint32_t acce(int i) const { return acc_empty + 8u * i; }
  __device__ uint32_t fin(int i) const { return final_bar + 8u * i; }
};
constexpr int kNumBarsFixed = 2 * kASlots + 2 * kItemSlots + 2 * kMaxDSlots + kMaxIssuers;

__device__ __forceinline__ size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bounded wait: true when the phase of parity `parity` has completed; false
// when the CTA is aborting or this wait ran out (then it starts the abort).
// kCluster: the phase may be completed by arrivals from the other CTA of a
// pair (remote arrives or multicast commits): acquire at cluster scope.
template <bool kCluster = false>
__device__ __forceinline__ bool try_wait_any(uint32_t bar, uint32_t parity, uint32_t suspend_ns) {
  if constexpr (kCluster) return mbar_try_wait_cluster(bar, parity, suspend_ns);
  return mbar_try_wait_sleep(bar, parity, suspend_ns);
}
template <bool kCluster = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                        int* status, int where, long long timeout) {
  constexpr uint32_t kSuspendNs = 1000000;  // the thread sleeps until completion or 1 ms
  if (try_wait_any<kCluster>(bar, parity, kSuspendNs)) return true;
  const long long t0 = clock64();
  while (true) {
    if (try_wait_any<kCluster>(bar, parity, kSuspendNs)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > timeout) {
      *abort_flag = 1;
      if (status != nullptr) atomicCAS(status, 0, 0x1000 | where);
      return false;
    }
  }
}

// Bounded wait until the counter at `flag` (global memory, raised by other
// CTAs) reaches `target`; acquires at GPU scope. False when the CTA is
// aborting or the wait ran out (then it starts the abort).
__device__ __forceinline__ bool wait_count(const int* flag, int target, volatile int* abort_flag,
                                           int* status, int where, long long timeout) {
  const long long t0 = clock64();
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v >= target) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > timeout) {
      *abort_flag = 1;
      if (status != nullptr) atomicCAS(status, 0, 0x1000 | where);
      return false;
    }
    __nanosleep(256);
  }
}

// Warp-uniform bounded wait: every lane observes the phase itself (so each
// lane's later reads are ordered after the completion it saw); the warp goes
// on only if all lanes saw it.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, int* status, int where,
                                             long long timeout) {
  return __all_sync(0xffffffffu,
                    wait_phase<kCluster>(bar, parity, abort_flag, status, where, timeout));
}

// Bounded wait of the dequant warpgroups: polls without a suspend hint and
// sleeps 128 ns between polls. These are the warps that issue almost every
// instruction of the SM; a waiting warpgroup that backs off leaves the issue
// slots to the three that work (measured 0.8% faster at EP8 decode than the
// suspending wait, which the other roles keep: for them it was slower).
template <bool kCluster = false>
__device__ __forceinline__ bool try_wait_now(uint32_t bar, uint32_t parity) {
  if constexpr (kCluster) return mbar_try_wait_cluster_now(bar, parity);
  return mbar_try_wait(bar, parity);
}
template <bool kCluster = false>
__device__ __forceinline__ bool wait_phase_backoff(uint32_t bar, uint32_t parity,
                                                   volatile int* abort_flag, int* status,
                                                   int where, long long timeout) {
  if (try_wait_now<kCluster>(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    __nanosleep(128);
    if (try_wait_now<kCluster>(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > timeout) {
      *abort_flag = 1;
      if (status != nullptr) atomicCAS(status, 0, 0x1000 | where);
      return false;
    }
  }
}
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait_phase_backoff(uint32_t bar, uint32_t parity,
                                                        volatile int* abort_flag, int* status,
                                                        int where, long long timeout) {
  return __all_sync(0xffffffffu, wait_phase_backoff<kCluster>(bar, parity, abort_flag, status,
                                                              where, timeout));
}

// Drain wait (abort path): wait for a phase that copies or MMAs already
// issued will complete. They finish within microseconds, so the bound is a
// fixed, generous one (about 2 s) and never the wait timeout, which a caller
// may set very short: a CTA must not exit while its copies still land.
constexpr long long kDrainCycles = 4000000000LL;
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity, long long timeout) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < timeout) {
  }
}

// Position in a ring of mbarrier-guarded slots: slot index and the parity of
// the slot's current phase (advanced without divisions).
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
  // advance by `step` slots, step <= n
  __device__ __forceinline__ void advance(int step, int n) {
    slot += step;
    if (slot >= n) {
      slot -= n;
      phase ^= 1u;
    }
  }
  // advance by any number of slots
  __device__ __forceinline__ void skip(int step, int n) {
    const int t = slot + step;
    const int wraps = t / n;
    slot = t - wraps * n;
    phase ^= static_cast<uint32_t>(wraps & 1);
  }
};

// How the k steps of an item are split among the MMA issuers: with P partial
// accumulators, issuer q takes the k steps ks with ks % P == q. Stage u
// (k steps 2u, 2u + 1) is then read by min(P, 2) issuers; for P == 4,
// issuer q sees only the stages of parity q >> 1.
struct IssuerPlan {
  int stride, first, j0, j1;  // stages u = first + stride * i; k steps j0..j1 of each
};
__device__ __forceinline__ IssuerPlan issuer_plan(int q, int parts) {
  IssuerPlan p;
  if (parts == 4) {
    p.stride = 2;
    p.first = q >> 1;
    p.j0 = p.j1 = q & 1;
  } else if (parts == 2) {
    p.stride = 1;
    p.first = 0;
    p.j0 = p.j1 = q;
  } else {
    p.stride = 1;
    p.first = 0;
    p.j0 = 0;
    p.j1 = 1;
  }
  return p;
}

struct ItemDesc {
  int blk, tile, e;
  int phase;  // the single-launch layer: 0 gate_up, 1 down (else 0)
};

// Which routing block and weight tile item `it` is, and its expert (-1: skip).
// Item order. Plain: tile-major (all blocks for tile 0, then tile 1, ...),
// so the CTAs working at one time stream different experts' weights and
// every block's token rows are read once per tile. Rastered (kRaster, for
// grouped GEMMs whose token rows are too many for L2): blocks in groups of
// kRasterBlocks consecutive blocks, tile-major inside a group, so a group's
// token rows stay in L2 across the tiles. The rastered order is a separate
// kernel instantiation: its integer divisions, even untaken, cost the plain
// kernel measurable time on short items (instruction footprint).
constexpr int kRasterBlocks = 8;

template <bool kRaster, bool kPair, bool kLayer>
__device__ __forceinline__ ItemDesc decode_item(const GemmArgs& a, int it, int num_blocks,
                                                int blocks_per_expert, uint32_t rank) {
  ItemDesc d;
  d.phase = 0;
  if constexpr (kLayer) {
    // the single-launch layer: every gate_up item, then every down item, each
    // list block-major, so that a block's activation rows are complete early
    // and the down items of early blocks can fill the gate_up tail
    const int items_gu = num_blocks * a.n_tiles;
    if (it < items_gu) {
      d.blk = it / a.n_tiles;
      d.tile = it - d.blk * a.n_tiles;
    } else {
      const int j = it - items_gu;
      d.phase = 1;
      d.blk = j / a.n_tiles2;
      d.tile = j - d.blk * a.n_tiles2;
    }
  } else if constexpr (kRaster) {
    const int per_group = kRasterBlocks * (kPair ? a.n_tiles >> 1 : a.n_tiles);
    const int group = it / per_group;
    const int rem = it - group * per_group;
    const int gsize = min(kRasterBlocks, num_blocks - group * kRasterBlocks);
    d.tile = rem / gsize;
    d.blk = group * kRasterBlocks + (rem - d.tile * gsize);
  } else {
    d.tile = it / num_blocks;
    d.blk = it - d.tile * num_blocks;
  }
  // a CTA pair takes a pair of weight tiles: the even-ranked CTA the first
  if constexpr (kPair) d.tile = d.tile * 2 + static_cast<int>(rank);
  int e = -1;
  if (a.family == kIndexed) {
    e = __ldg(a.expert_ids + d.blk);
  } else if (a.family == kContiguous) {
    e = __ldg(a.layout + static_cast<long long>(d.blk) * a.block_m);
  } else {
    e = d.blk / blocks_per_expert;
    const int j0 = (d.blk - e * blocks_per_expert) * a.block_m;
    int valid = __ldg(a.layout + e);
    valid = min(max(valid, 0), a.m);
    if (j0 >= valid) e = -1;
  }
  d.e = (e >= 0 && e < a.num_experts) ? e : -1;
  return d;
}

// Row j of block `blk`: output row (-1 = not a real row) and the top-k
// weight of the down pass.
// kRows (the deterministic down pass): the output row is the routing
// position itself.
template <bool kRows, bool kLayer>
__device__ __forceinline__ void row_info(const GemmArgs& a, const ItemDesc& d, int j, int& dst,
                                         float& wt) {
  dst = -1;
  wt = 0.f;
  if (a.family == kIndexed) {
    const long long pos = static_cast<long long>(d.blk) * a.block_m + j;
    const int id = __ldg(a.sorted_ids + pos);
    if (id >= 0 && id < a.numel) {
      if constexpr (kLayer) {
        // gate_up: activation rows at their routing positions; down: the
        // top-k weighted add into the token's row
        if (d.phase == 0) {
          dst = static_cast<int>(pos);
          wt = 1.f;
        } else {
          dst = id / a.o_div;
          wt = __ldg(a.topk_weights + id);
        }
      } else if constexpr (kRows) {
        dst = static_cast<int>(pos);
        wt = __ldg(a.topk_weights + id);
      } else {
        dst = id / a.o_div;
        wt = (a.out_mode == kOutF32WeightedAdd) ? __ldg(a.topk_weights + id) : 1.f;
      }
    }
  } else if (a.family == kContiguous) {
    const int r = d.blk * a.block_m + j;
    if (r < a.m && __ldg(a.layout + r) == d.e) {
      dst = r;
      wt = 1.f;
    }
  } else {
    const int bpe = (a.m + a.block_m - 1) / a.block_m;
    const int rl = (d.blk - d.e * bpe) * a.block_m + j;
    const int valid = min(max(__ldg(a.layout + d.e), 0), a.m);
    if (rl < valid) {
      dst = d.e * a.m + rl;
      wt = 1.f;
    }
  }
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t x, uint32_t mask, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(mask), "r"(magic));
  return r;
}

// 32 codes of one group (prepacked nibble order) -> 16 BF16x2 columns
// (column c holds k = 2c in its low half and k = 2c + 1 in its high half).
// OR-ing a code into the mantissa of BF16 128.0 gives 128 + q exactly;
// subtracting 136 gives q - 8 exactly; the scale product is rounded once.
__device__ __forceinline__ void dequant_group(const uint4 q, uint32_t scale_bits,
                                              uint32_t* out) {
  const uint32_t words[4] = {q.x, q.y, q.z, q.w};
  const uint32_t s2u = scale_bits | (scale_bits << 16);
  const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162*>(&s2u);
  const uint32_t off_u = 0x43084308u;  // BF16 136.0 in both halves
  const __nv_bfloat162 off = *reinterpret_cast<const __nv_bfloat162*>(&off_u);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t t = lop3_and_or(words[w] >> (4 * i), 0x000F000Fu, 0x43004300u);
      __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&t);
      v = __hmul2(__hsub2(v, off), s2);
      out[4 * w + i] = *reinterpret_cast<uint32_t*>(&v);
    }
  }
}

}  // namespace

// Stage bookkeeping shared by every role. An item's k range is split into
// stages of two 64-k steps; the stage count is padded to an even number (the
// pad stage moves no data), so that every item starts on an even global
// stage and the split of k steps among the MMA issuers is the same for every
// item. Global stage u -> A slot u % 4 (dequant warpgroup u % 4), B slot
// u % BS, weight slot u % WS (WS % 4 == 0, BS even).

// kGlu: the fused-activation epilogue (out_mode kOutGluBf16), kRaster: the
// grouped item order, and kEarly: the epilogue that frees the accumulator
// slot before its stores (blocks of 48 or 64 rows, whose accumulators fill
// TMEM's single slot), and kRows: the deterministic down pass (out_mode
// kOutF32Rows), kPair: the CTA-pair kernel, kLayer: the single-launch
// layer (gate_up items, then down items), kBig: blocks above 128 rows, and
// kHalf: the BF16 staging of 65..128-row blocks are compiled into their own
// instantiations so that they cannot change the
// register allocation or the instruction footprint of the plain kernel
// (compiled into it, the 256-row code made the TP8 down pass 18% slower).
template <bool kGlu, bool kRaster, bool kEarly, bool kRows, bool kPair, bool kLayer = false,
          bool kBig = false, bool kHalf = false>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_moe_gemm_kernel(const __grid_constant__ GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // A CTA pair (kPair, a cluster of 2) works on 256 weight rows at a time:
  // each CTA dequantises its own 128 rows into its own TMEM and loads half of
  // the block's token rows; the even-ranked CTA (the leader) issues M = 256
  // MMAs over both. Otherwise every CTA works alone.
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit0 = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  // ---- shared-memory carve-up (base aligned to 1024 for the swizzle) ----
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const int bm = args.block_m;
  const int WS = args.w_stages;
  const int BS = args.b_stages;
  const int parts = args.n_parts;
  const bool gather = args.gather_rows != 0;
  // token rows of a block held by this CTA (a pair splits them in halves)
  const int bm_local = kPair ? bm >> 1 : bm;
  const uint32_t b_step_bytes = static_cast<uint32_t>(bm_local) * 128u;
  const uint32_t b_stage_bytes = 2u * b_step_bytes;
  // kBig (blocks above 128 rows; never a pair or the single-launch layer,
  // which refuse such blocks): activation ring of single k steps, issuers
  // chosen per item
  constexpr bool b_steps = kBig && !kPair && !kLayer;
  const uint32_t b_slot_bytes = b_steps ? b_step_bytes : b_stage_bytes;
  Smem sm;
  size_t off = 0;
  sm.b_ring = base;
  off += static_cast<size_t>(BS) * b_slot_bytes;
  sm.w_ring = base + off;
  off += static_cast<size_t>(WS) * kWStageBytes;
  sm.info_dst = reinterpret_cast<int*>(base + off);
  off += kItemSlots * bm * sizeof(int);
  sm.info_wt = reinterpret_cast<float*>(base + off);
  off += kItemSlots * bm * sizeof(float);
  sm.info_n16 = reinterpret_cast<int*>(base + off);
  off += kItemSlots * sizeof(int);
  sm.info_rows = reinterpret_cast<int*>(base + off);
  off += kItemSlots * sizeof(int);
  off = align_up(off, 16);
  sm.epi_tile = reinterpret_cast<float*>(base + off);
  off += epi_tile_bytes(bm);
  off = align_up(off, 8);
  sm.bars = reinterpret_cast<uint64_t*>(base + off);
  off += (2 * WS + 2 * BS + kNumBarsFixed) * 8;
  sm.tmem_base = reinterpret_cast<uint32_t*>(base + off);
  off += 4;
  sm.abort_flag = reinterpret_cast<volatile int*>(base + off);
  if constexpr (kHalf) sm.epi_half = reinterpret_cast<__nv_bfloat16*>(base + align_up(off + 4, 16));

  Bars B;
  {
    uint32_t b0 = smem_u32(sm.bars);
    B.w_full = b0;
    b0 += 8 * WS;
    B.w_empty = b0;
    b0 += 8 * WS;
    B.b_full = b0;
    b0 += 8 * BS;
    B.b_empty = b0;
    b0 += 8 * BS;
    B.a_full = b0;
    b0 += 8 * kASlots;
    B.a_empty = b0;
    b0 += 8 * kASlots;
    B.item_full = b0;
    b0 += 8 * kItemSlots;
    B.item_empty = b0;
    b0 += 8 * kItemSlots;
    B.acc_full = b0;
    b0 += 8 * kMaxDSlots;
    B.acc_empty = b0;
    b0 += 8 * kMaxDSlots;
    B.final_bar = b0;
  }
  // issuers that read each stage (each commits once per stage); blocks above
  // 128 rows: one reader per activation slot, two commits per A slot
  const int readers = parts < 2 ? parts : 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < WS; ++i) {
      mbar_init(B.wf(i), 1);  // the producer's arrival (+ the copy's bytes)
      mbar_init(B.we(i), 4);  // the 4 warps of the warpgroup that read the stage
    }
    for (int i = 0; i < BS; ++i) {
      // the gather warp's arrival (+ tensor-copy bytes); the pair leader's
      // also counts the peer's relayed arrival for its half of the rows
      mbar_init(B.bf(i), (kPair && leader) ? 2 : 1);
      mbar_init(B.be(i), b_steps ? 2 : readers);  // tcgen05.commit of the slot's issuers
    }
    for (int i = 0; i < kASlots; ++i) {
      // the 4 warps of the slot's dequant warpgroup (of both CTAs of a pair)
      mbar_init(B.af(i), kPair ? 8 : 4);
      mbar_init(B.ae(i), b_steps ? 2 : readers);
    }
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(B.itf(i), 1);  // the router warp
      mbar_init(B.ite(i), 4);  // the 4 epilogue warps
    }
    for (int i = 0; i < kMaxDSlots; ++i) {
      // one tcgen05.commit per MMA issuer (blocks above 128 rows: all four,
      // the issuers without MMAs in the item by a plain arrive)
      mbar_init(B.accf(i), b_steps ? kMaxIssuers : parts);
      mbar_init(B.acce(i), kPair ? 8 : 4);  // the epilogue warps (of both CTAs of a pair)
    }
    for (int i = 0; i < kMaxIssuers; ++i) mbar_init(B.fin(i), 1);
    *sm.abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kWarpMma0) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_u32(sm.tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(sm.tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // a pair's barriers must be initialised in both CTAs before either arrives
  // on the other's
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_base;

  // ---- work decomposition ----
  int num_blocks = 0, bpe = 1;
  if (args.family == kIndexed) {
    int t = __ldg(args.num_tokens_padded);
    t = min(max(t, 0), args.capacity);
    num_blocks = t / bm;
  } else if (args.family == kContiguous) {
    num_blocks = args.m / bm;
  } else {
    bpe = (args.m + bm - 1) / bm;
    num_blocks = args.num_experts * bpe;
  }
  const int items = kLayer ? num_blocks * (args.n_tiles + args.n_tiles2)
                           : num_blocks * (kPair ? args.n_tiles >> 1 : args.n_tiles);
  // TMEM columns: the kASlots A slots (64 columns each), then per accumulator
  // slot the `parts` partial accumulators, d_cols each.
  const int d_col_base = kASlots * kAColsPerSlot;
  const int n_st = (args.k_steps + 1) / 2;  // stages holding data
  const int n_stp = n_st + (n_st & 1);      // stages per item (even)
  // the single-launch layer's down items: their own reduction length
  const int n_st2 = kLayer ? (args.k_steps2 + 1) / 2 : n_st;
  const int n_stp2 = kLayer ? n_st2 + (n_st2 & 1) : n_stp;
  // reduction steps and stages of an item (the layer's down items differ)
  auto ksteps_of = [&](const ItemDesc& d) { return (kLayer && d.phase) ? args.k_steps2 : args.k_steps; };
  auto nstp_of = [&](const ItemDesc& d) { return (kLayer && d.phase) ? n_stp2 : n_stp; };
  const long long tmo = args.timeout_cycles;
  volatile int* abort_flag = sm.abort_flag;
  int* status = args.status;
  const int mma_q = warp == kWarpMma3 ? 3 : warp - kWarpMma0;  // issuer index of MMA warps

  if (warp == kWarpProducer) {
    // ======================= weight producer (bulk copies) ==================
    if (lane == 0) {
      const uint64_t policy = policy_evict_first();
      uint32_t issued = 0;  // stages whose w_full phase this thread started
      RingPos wp;
      bool ok = true;
      for (int it = unit0; it < items && ok; it += units) {
        const ItemDesc d = decode_item<kRaster, kPair, kLayer>(args, it, num_blocks, bpe, rank);
        if (d.e < 0) continue;
        const int ks = ksteps_of(d);
        const uint8_t* wbase = (kLayer && d.phase) ? args.wpack2 : args.wpack;
        const long long ebytes = (kLayer && d.phase) ? args.expert_bytes2 : args.expert_bytes;
        const uint8_t* src = wbase + static_cast<long long>(d.e) * ebytes +
                             static_cast<long long>(d.tile) * ks * kStepBytes;
        const int nst_i = nstp_of(d);
        for (int st = 0; st < nst_i; ++st, wp.next(WS)) {
          if (!wait_phase(B.we(wp.slot), wp.phase ^ 1, abort_flag, status, kWhereProducer, tmo)) {
            ok = false;
            break;
          }
          const int nks = min(2, max(0, ks - 2 * st));
          if (nks > 0) {
            const uint32_t bytes = static_cast<uint32_t>(nks * kStepBytes);
            mbar_arrive_expect_tx(B.wf(wp.slot), bytes);
            bulk_g2s(smem_u32(sm.w_ring + static_cast<size_t>(wp.slot) * kWStageBytes),
                     src + static_cast<long long>(st) * kWStageBytes, bytes, B.wf(wp.slot),
                     policy);
          } else {
            mbar_arrive(B.wf(wp.slot));  // pad stage: no data
          }
          ++issued;
        }
      }
      if (!ok) {
        // Let every copy already issued land before the CTA can exit.
        const uint32_t first = issued > static_cast<uint32_t>(WS) ? issued - WS : 0;
        for (uint32_t u = first; u < issued; ++u)
          drain_phase(B.wf(u % WS), (u / WS) & 1, kDrainCycles);
      }
    }
  } else if ((warp >= kWarpMma0 && warp < kWarpDequant0) || warp == kWarpMma3) {
    // ======================= MMA issuers ====================================
    // Issuer q takes the k steps ks % parts == q of every item and
    // accumulates them into its own FP32 partial accumulator. In a CTA pair
    // the leader's issuers issue M = 256 MMAs over both CTAs' A slots and
    // token halves; the peer issues none, and its warp of issuer 0 relays the
    // completion of the peer's token-row copies to the leader instead.
    const int q = mma_q;
    if (kPair && !leader && q == 0 && lane == 0) {
      W4A16_PROF_DECL
      RingPos bp;
      const uint32_t leader_bf = map_to_cta(B.b_full, 0);
      bool ok = true;
      for (int it = unit0; it < items && ok; it += units) {
        const ItemDesc d = decode_item<kRaster, kPair, kLayer>(args, it, num_blocks, bpe, rank);
        if (d.e < 0) continue;
        const int nst_i = nstp_of(d);
        for (int st = 0; st < nst_i; ++st, bp.next(BS)) {
          W4A16_PROF_MARK(2);
          if (!wait_phase(B.bf(bp.slot), bp.phase, abort_flag, status, kWhereRelay, tmo)) {
            ok = false;
            break;
          }
          W4A16_PROF_MARK(0);
          mbar_arrive_remote_relaxed(leader_bf + 8u * bp.slot);
          W4A16_PROF_MARK(1);
        }
      }
      W4A16_PROF_MARK(2);
      W4A16_PROF_STORE();
    }
    W4A16_PROF_DECL
    if (b_steps) {
      // Blocks above 128 rows: an item of at most 128 rows is split along K,
      // P = big_block_parts(N) issuers, issuer q taking the k steps
      // ks % P == q into its own partial; an item above 128 rows along N, two
      // issuers each taking half of the token columns (0..127, 128..N) of the
      // one partial. Every issuer walks every item: it reads the item's N,
      // waits until the previous item's accumulator is released and adds one
      // arrival to the item's accumulator barrier (the issuers by
      // tcgen05.commit). Within an item each activation slot (BS % 4 == 0)
      // and each A slot has fixed readers, which alone free it, by two
      // arrivals: two readers' commits, or one reader's commit and a plain
      // arrive. The release wait at every item start keeps an issuer that
      // skipped slots from waiting on a phase two behind or ahead of the
      // barrier.
      if (lane == 0) {
        RingPos ip, ap, bp;
        uint32_t acc_phase = 0;  // one accumulator slot
        bool ok = true;
        const uint64_t b_desc0 = smem_desc_sw128_kmajor(smem_u32(sm.b_ring));
        for (int it = unit0; it < items && ok; it += units) {
          const ItemDesc d = decode_item<kRaster, kPair, kLayer>(args, it, num_blocks, bpe, rank);
          if (d.e < 0) continue;
          W4A16_PROF_MARK(5);
          if (!wait_phase(B.itf(ip.slot), ip.phase, abort_flag, status, kWhereMmaItem, tmo)) {
            ok = false;
            break;
          }
          W4A16_PROF_MARK(0);
          if (!wait_phase(B.acce(0), acc_phase ^ 1, abort_flag, status, kWhereMmaAcc, tmo)) {
            ok = false;
            break;
          }
          W4A16_PROF_MARK(1);
          const int n16 = sm.info_n16[ip.slot];
          const bool nsplit = n16 > 128;
          const int P = nsplit ? 1 : big_block_parts(n16);
          const int nst_i = nstp_of(d);
          if (q >= (nsplit ? 2 : P)) {
            // no MMAs in this item: pass its slots
            mbar_arrive(B.accf(0));
            ap.skip(nst_i, kASlots);
            bp.skip(2 * nst_i, BS);
          } else {
            tc_fence_after();
            // an N split: issuer q takes token columns 128 q.., its rows of the
            // activation slot start 128 q rows (16 KB) in
            const uint32_t n_q = nsplit ? (q == 0 ? 128u : static_cast<uint32_t>(n16 - 128))
                                        : static_cast<uint32_t>(n16);
            const uint32_t idesc = idesc_bf16_m128(n_q);
            const uint32_t d_tmem = tmem + d_col_base + (nsplit ? q * 128 : q * (kBigAccCols / P));
            const uint64_t b_row_off = nsplit ? static_cast<uint64_t>(q) * (128u * 128u >> 4) : 0u;
            const int ks = ksteps_of(d);
            uint32_t acc = 0;
            for (int st = 0; st < nst_i && ok; ++st) {
              const int r0 = nsplit ? q : (2 * st) & (P - 1);
              const int r1 = nsplit ? q : (2 * st + 1) & (P - 1);
              if (r0 != q && r1 != q) {
                ap.next(kASlots);
                bp.skip(2, BS);
                continue;
              }
              W4A16_PROF_MARK(5);
              if (!wait_phase(B.af(ap.slot), ap.phase, abort_flag, status, kWhereMmaA, tmo)) {
                ok = false;
                break;
              }
              W4A16_PROF_MARK(2);
              for (int j = 0; j < 2; ++j, bp.next(BS)) {
                if ((j ? r1 : r0) != q) continue;
                if (!wait_phase(B.bf(bp.slot), bp.phase, abort_flag, status, kWhereMmaB, tmo)) {
                  ok = false;
                  break;
                }
                W4A16_PROF_MARK(3);
                tc_fence_after();
                if (2 * st + j < ks) {
                  // slot offsets are multiples of 1024 bytes
                  const uint64_t b_desc =
                      b_desc0 + ((static_cast<uint32_t>(bp.slot) * b_step_bytes) >> 4) + b_row_off;
                  const uint32_t a_tmem = tmem + ap.slot * kAColsPerSlot + j * kAColsPerStep;
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk) {
                    mma_bf16_ts(d_tmem, a_tmem + kk * 8, b_desc + 2 * kk, idesc, acc);
                    acc = 1;
                  }
                }
                W4A16_PROF_MARK(4);
                // two arrivals per slot: a lone reader adds a plain one
                if (!nsplit) mbar_arrive(B.be(bp.slot));
                tc_commit(B.be(bp.slot));
                W4A16_PROF_MARK(6);
              }
              if (!ok) break;
              tc_commit(B.ae(ap.slot));
              W4A16_PROF_MARK(6);
              ap.next(kASlots);
            }
            if (!ok) break;
            tc_commit(B.accf(0));
          }
          acc_phase ^= 1u;
          ip.next(kItemSlots);
        }
        tc_commit(B.fin(q));
        drain_phase(B.fin(q), 0, kDrainCycles);
      }
    } else if ((!kPair || leader) && lane == 0 && q < parts) {
      const IssuerPlan pl = issuer_plan(q, parts);
      RingPos ip, dp, ap, bp;
      ap.slot = pl.first;
      bp.slot = pl.first;
      bool ok = true;
      const uint64_t b_desc0 = smem_desc_sw128_kmajor(smem_u32(sm.b_ring));
      for (int it = unit0; it < items && ok; it += units) {
        const ItemDesc d = decode_item<kRaster, kPair, kLayer>(args, it, num_blocks, bpe, rank);
        if (d.e < 0) continue;
        W4A16_PROF_MARK(5);
        if (!wait_phase(B.itf(ip.slot), ip.phase, abort_flag, status, kWhereMmaItem, tmo)) {
          ok = false;
          break;
        }
        W4A16_PROF_MARK(0);
        const int n16 = sm.info_n16[ip.slot];
        if (!wait_phase<kPair>(B.acce(dp.slot), dp.phase ^ 1, abort_flag, status, kWhereMmaAcc,
                               tmo)) {
          ok = false;
          break;
        }
        W4A16_PROF_MARK(1);
        tc_fence_after();
        // a pair's MMA takes N/2 token rows from each CTA: N is the whole block
        const uint32_t idesc = kPair ? idesc_bf16(256u, static_cast<uint32_t>(bm))
                                     : idesc_bf16_m128(static_cast<uint32_t>(n16));
        const uint32_t d_tmem = tmem + d_col_base + (dp.slot * parts + q) * args.d_cols;
        uint32_t acc = 0;
        const int ks = ksteps_of(d);
        const int nst_i = nstp_of(d);
        for (int st = pl.first; st < nst_i; st += pl.stride) {
          W4A16_PROF_MARK(5);
          if (!wait_phase<kPair>(B.af(ap.slot), ap.phase, abort_flag, status, kWhereMmaA, tmo)) {
            ok = false;
            break;
          }
          W4A16_PROF_MARK(2);
          if (!wait_phase<kPair>(B.bf(bp.slot), bp.phase, abort_flag, status, kWhereMmaB, tmo)) {
            ok = false;
            break;
          }
          W4A16_PROF_MARK(3);
          tc_fence_after();
          for (int j = pl.j0; j <= pl.j1; ++j) {
            if (2 * st + j >= ks) break;
            // slot and k-step offsets are multiples of 1024 bytes
            const uint64_t b_desc =
                b_desc0 + ((static_cast<uint32_t>(bp.slot) * b_stage_bytes + j * b_step_bytes) >> 4);
            const uint32_t a_tmem = tmem + ap.slot * kAColsPerSlot + j * kAColsPerStep;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              // +32 bytes of K per MMA inside the 128-byte swizzle row
              if constexpr (kPair) {
                mma_bf16_ts_pair(d_tmem, a_tmem + kk * 8, b_desc + 2 * kk, idesc, acc);
              } else {
                mma_bf16_ts(d_tmem, a_tmem + kk * 8, b_desc + 2 * kk, idesc, acc);
              }
              acc = 1;
            }
          }
          W4A16_PROF_MARK(4);
          if constexpr (kPair) {
            // the slots are freed in both CTAs of the pair
            tc_commit_pair_mc(B.ae(ap.slot), 0x3);
            tc_commit_pair_mc(B.be(bp.slot), 0x3);
          } else {
            tc_commit(B.ae(ap.slot));
            tc_commit(B.be(bp.slot));
          }
          ap.advance(pl.stride, kASlots);
          bp.advance(pl.stride, BS);
          W4A16_PROF_MARK(6);
        }
        if (!ok) break;
        if constexpr (kPair) {
          tc_commit_pair_mc(B.accf(dp.slot), 0x3);
        } else {
          tc_commit(B.accf(dp.slot));
        }
        ip.next(kItemSlots);
        dp.next(args.d_slots);
      }
      // every MMA issued by this thread has finished once its final barrier flips
      if constexpr (kPair) {
        tc_commit_pair_mc(B.fin(q), 0x1);
      } else {
        tc_commit(B.fin(q));
      }
      drain_phase(B.fin(q), 0, kDrainCycles);
    }
    W4A16_PROF_MARK(5);
    W4A16_PROF_STORE();
  } else if (warp == kWarpRouter) {
    // ======================= routing info, items ahead ======================
    // Resolves each item's rows (activation row, output row, top-k weight)
    // into the item ring up to kItemSlots items ahead, so that the global
    // loads of the routing tensors stay off the copy and MMA critical path.
    RingPos ip;
    for (int it = unit0; it < items; it += units) {
      const ItemDesc d = decode_item<kRaster, kPair, kLayer>(args, it, num_blocks, bpe, rank);
      if (d.e < 0) continue;
      if (!warp_wait_phase(B.ite(ip.slot), ip.phase ^ 1, abort_flag, status, kWhereRouter, tmo))
        break;
      int* idst = sm.info_dst + ip.slot * bm;
      float* iwt = sm.info_wt + ip.slot * bm;
      int maxj = -1;
      for (int j = lane; j < bm; j += 32) {
        int dd;
        float w;
        row_info<kRows, kLayer>(args, d, j, dd, w);
        idst[j] = dd;
        iwt[j] = w;
        if (dd >= 0) maxj = j;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) maxj = max(maxj, __shfl_xor_sync(0xffffffffu, maxj, o));
      const int rows = max(maxj + 1, 1);
      if (lane == 0) {
        sm.info_rows[ip.slot] = rows;
        sm.info_n16[ip.slot] = (rows + 15) & ~15;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(B.itf(ip.slot));
      ip.next(kItemSlots);
    }
  } else if (warp == kWarpGather) {
    // ======================= activation rows (TMA) ==========================
    // Fills the B slot of every stage with the block's rows in the
    // 128-byte-swizzled K-major layout of the MMA descriptor (8-row atoms of
    // 1024 bytes), counted in bytes on the slot's mbarrier:
    //  - indexed family: the routed rows were copied into sorted order
    //    beforehand, so block b's rows are rows b*block_m.. of that buffer and
    //    one 3-D box (64 columns x block_m rows x 2 k steps) fills a stage;
    //  - grouped families: one 2-D box (64 columns x block_m rows) per k step.
    // Rows past the tensor and k steps past k read zeros.
    // the token rows may come from the previous grid (the row permute)
    grid_dependency_wait();
    if (lane == 0) {
      RingPos bp, gip;
      uint32_t issued = 0;  // stages whose b_full phase this thread started
      bool ok = true;
      for (int it = unit0; it < items && ok; it += units) {
        const ItemDesc d = decode_item<kRaster, kPair, kLayer>(args, it, num_blocks, bpe, rank);
        if (d.e < 0) continue;
        // a pair's CTA loads its half of the block's rows
        const int box_row = ((args.family == kMasked) ? d.e * args.m + (d.blk - d.e * bpe) * bm
                                                      : d.blk * bm) +
                            static_cast<int>(rank) * bm_local;
        const CUtensorMap* tmap = &args.tmap;
        if (kLayer && d.phase) {
          // the layer's down item reads the block's activation rows, written
          // by the gate_up items of this launch (any CTA): wait until all of
          // them are out (4 epilogue warps per gate_up tile), then order the
          // tensor copies after what the wait observed
          if (!wait_count(args.block_done + d.blk, 4 * args.n_tiles, abort_flag, status,
                          kWhereBlockDone, tmo)) {
            ok = false;
            break;
          }
          asm volatile("fence.proxy.async.global;" ::: "memory");
          tmap = &args.tmap2;
        }
        const int ks = ksteps_of(d);
        const int nst_i = nstp_of(d);
        // blocks above 128 rows: an item with N > 128 takes the whole block in
        // one copy, a smaller one its rows up to N in copies of kSmallBoxRows
        // (N from the item ring)
        int chunks = 1;
        bool whole = true;
        if (b_steps) {
          if (!wait_phase(B.itf(gip.slot), gip.phase, abort_flag, status, kWhereGatherItem, tmo)) {
            ok = false;
            break;
          }
          const int n16 = sm.info_n16[gip.slot];
          whole = n16 > 128;
          chunks = whole ? 1 : (n16 + kSmallBoxRows - 1) / kSmallBoxRows;
          gip.next(kItemSlots);
        }
        for (int st = 0; st < nst_i; ++st, bp.next(BS)) {
          if (!wait_phase<kPair>(B.be(bp.slot), bp.phase ^ 1, abort_flag, status, kWhereGatherB,
                                 tmo)) {
            ok = false;
            break;
          }
          const int nks = min(2, max(0, ks - 2 * st));
          const uint32_t dst = smem_u32(sm.b_ring + static_cast<size_t>(bp.slot) * b_slot_bytes);
          if (b_steps) {
            // one k step per slot: this stage's second k step has the next slot
            for (int j = 0; j < 2 && ok; ++j) {
              if (j == 1) {
                ++issued;
                bp.next(BS);
                if (!wait_phase(B.be(bp.slot), bp.phase ^ 1, abort_flag, status, kWhereGatherB,
                                tmo)) {
                  ok = false;
                  break;
                }
              }
              const uint32_t dj = smem_u32(sm.b_ring + static_cast<size_t>(bp.slot) * b_step_bytes);
              if (j >= nks) {
                mbar_arrive(B.bf(bp.slot));  // pad k step: no data
              } else {
                const CUtensorMap* map = whole ? &args.tmap : &args.tmap2;
                mbar_arrive_expect_tx(B.bf(bp.slot),
                                      whole ? b_step_bytes
                                            : static_cast<uint32_t>(chunks * kSmallBoxRows * 128));
                for (int c = 0; c < chunks; ++c) {
                  const uint32_t dc = dj + static_cast<uint32_t>(c * kSmallBoxRows * 128);
                  const int row = box_row + c * kSmallBoxRows;
                  if (gather) {
                    tma_load_3d(dc, map, 0, row, 2 * st + j, B.bf(bp.slot));
                  } else {
                    tma_load_2d(dc, map, (2 * st + j) * kKStep, row, B.bf(bp.slot));
                  }
                }
              }
            }
            if (!ok) break;
          } else if (nks == 0) {
            mbar_arrive(B.bf(bp.slot));  // pad stage: no data
          } else if (gather) {
            mbar_arrive_expect_tx(B.bf(bp.slot), b_stage_bytes);
            tma_load_3d(dst, tmap, 0, box_row, 2 * st, B.bf(bp.slot));
          } else {
            mbar_arrive_expect_tx(B.bf(bp.slot), nks * b_step_bytes);
            for (int j = 0; j < nks; ++j)
              tma_load_2d(dst + j * b_step_bytes, &args.tmap, (2 * st + j) * kKStep, box_row,
                          B.bf(bp.slot));
          }
          ++issued;
        }
      }
      if (!ok) {
        // wait, bounded, for the last tensor copies issued
        const uint32_t first = issued > static_cast<uint32_t>(BS) ? issued - BS : 0;
        for (uint32_t x = first; x < issued; ++x)
          drain_phase(B.bf(x % BS), (x / BS) & 1, kDrainCycles);
      }
    }
  } else if (warp >= kWarpDequant0 && warp < kWarpEpilogue0) {
    // ======================= dequantisation into TMEM =======================
    // Warpgroup wg dequantises the stages with global index u % 4 == wg into
    // A slot wg; thread r of the warpgroup owns weight row r (TMEM lane r).
    const int wg = (warp - kWarpDequant0) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t a_cols = tmem + lane_base + wg * kAColsPerSlot;
    RingPos wp;            // weight slot of this warpgroup's next stage
    wp.advance(wg, WS);    // its first stage is global stage wg (WS % 4 == 0)
    uint32_t a_phase = 0;  // uses of A slot wg so far, mod 2
    int u = 0;             // global stage index of this CTA
    bool ok = true;
    W4A16_PROF_DECL
    for (int it = unit0; it < items && ok; it += units) {
      const ItemDesc d = decode_item<kRaster, kPair, kLayer>(args, it, num_blocks, bpe, rank);
      if (d.e < 0) continue;
      const int ks = ksteps_of(d);
      const int nst_i = nstp_of(d);
      // item-local stages of this warpgroup: st = wg - u (mod 4), step 4
      for (int st = (wg - u) & 3; st < nst_i; st += 4) {
        W4A16_PROF_MARK(4);
        ok = warp_wait_phase_backoff(B.wf(wp.slot), wp.phase, abort_flag, status, kWhereDequantW,
                                     tmo);
        if (!ok) break;
        W4A16_PROF_MARK(0);
        const int nks = min(2, max(0, ks - 2 * st));
        const uint8_t* stp = sm.w_ring + static_cast<size_t>(wp.slot) * kWStageBytes;
        uint4 qv[2][2];
        uint32_t sc[2][2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (j < nks) {
            const uint8_t* sj = stp + j * kStepBytes;
            qv[j][0] = *reinterpret_cast<const uint4*>(sj + r * 16);
            qv[j][1] = *reinterpret_cast<const uint4*>(sj + 2048 + r * 16);
            sc[j][0] = *reinterpret_cast<const uint16_t*>(sj + kStepQBytes + r * 2);
            sc[j][1] = *reinterpret_cast<const uint16_t*>(sj + kStepQBytes + 256 + r * 2);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(B.we(wp.slot));
        wp.advance(4, WS);
        // the MMAs of this slot's previous use must be done before overwriting
        W4A16_PROF_MARK(1);
        ok = warp_wait_phase_backoff<kPair>(B.ae(wg), a_phase ^ 1, abort_flag, status,
                                            kWhereDequantA, tmo);
        if (!ok) break;
        W4A16_PROF_MARK(2);
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (j < nks) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // one 32-k group: 16 BF16x2 columns
              uint32_t v[16];
              dequant_group(qv[j][h], sc[j][h], v);
              tmem_st_32x32b_x16(a_cols + j * kAColsPerStep + h * 16, v);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        W4A16_PROF_MARK(3);
        if (lane == 0) {
          // the pair's leader issues the MMAs: the peer's warps arrive there
          if (kPair && !leader) {
            mbar_arrive_remote_relaxed(map_to_cta(B.af(wg), 0));
          } else {
            mbar_arrive(B.af(wg));
          }
        }
        a_phase ^= 1u;
        W4A16_PROF_MARK(5);
      }
      u += nst_i;
    }
    W4A16_PROF_MARK(4);
    W4A16_PROF_STORE();
  } else if (warp >= kWarpEpilogue0 && warp < kWarpEpilogue0 + 4) {
    // ======================= epilogue =======================================
    // Warp q reads TMEM lanes 32q..32q+31 (weight rows of the tile = output
    // columns tile*128 + 32q + lane): per 16 token columns it adds the
    // partial accumulators in a fixed order, stages the values transposed in
    // shared memory, and then writes 4 consecutive output columns of one
    // token row per operation (an 8-byte BF16 store, or a float4 atomic add
    // of the top-k weighted values in the down pass).
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int live_parts = min(parts, args.k_steps);  // partial q holds k step q first
    // this warp's staging tile: [stage_rows token rows][32 weight rows]
    const int stage_rows = epi_stage_rows(bm);
    float* tile = sm.epi_tile + quarter * (stage_rows * 32);
    const int c4 = lane & 7;                            // 4-column group of this lane
    const int jr0 = lane >> 3;                          // first token row of this lane
    const bool vec4 = (args.n & 3) == 0;
    // the accumulator slot is freed on the barrier of the CTA that issues the
    // MMAs (the pair's leader)
    auto release_acc = [&](uint32_t bar) {
      if (kPair && !leader) {
        mbar_arrive_remote_relaxed(map_to_cta(bar, 0));
      } else {
        mbar_arrive(bar);
      }
    };
    grid_dependency_wait();  // the previous grid may zero the output this one adds into
    W4A16_PROF_DECL
    RingPos ip, dp;
    for (int it = unit0; it < items; it += units) {
      const ItemDesc d = decode_item<kRaster, kPair, kLayer>(args, it, num_blocks, bpe, rank);
      if (d.e < 0) continue;
      const int islot = ip.slot;
      const int dslot = dp.slot;
      W4A16_PROF_MARK(3);
      if (!warp_wait_phase<kPair>(B.accf(dslot), dp.phase, abort_flag, status, kWhereEpiAcc,
                                  tmo) ||
          !warp_wait_phase(B.itf(islot), ip.phase, abort_flag, status, kWhereEpiItem, tmo))
        break;
      W4A16_PROF_MARK(0);
      tc_fence_after();
      const int rows = sm.info_rows[islot];
      const int* idst = sm.info_dst + islot * bm;
      const float* iwt = sm.info_wt + islot * bm;
      // first output column of this lane's 4-column group
      const int ng = d.tile * kTileRows + quarter * 32 + 4 * c4;
      const uint32_t dcol0 = tmem + lane_base + d_col_base + dslot * parts * args.d_cols;
      if constexpr (kEarly) {
        // Token rows go through the warp's staging tile in passes. When the
        // whole block fits (stage_rows), one pass first moves every partial sum
        // out of TMEM and frees the accumulator slot, so that the next item's
        // MMAs overlap this item's stores; otherwise each 16-row pass is staged
        // and written, and the slot is freed at the end. A 65..128-row block
        // with a BF16 output (half_stage) is staged whole as BF16 in tile_h.
        constexpr bool half_stage = kHalf && !kGlu && !kRows;
        __nv_bfloat16* tile_h = half_stage ? sm.epi_half + quarter * (bm * 32) : nullptr;
        const int stage_rows_e = half_stage ? bm : stage_rows;
        const bool early = rows <= stage_rows_e;  // (kEarly launches only)
        const int pass_rows = early ? stage_rows_e : 16;
        for (int p0 = 0; p0 < rows; p0 += pass_rows) {
          const int p1 = min(rows, p0 + pass_rows);
          for (int j0 = p0; j0 < p1; j0 += 16) {
            float* slab = tile + (j0 - p0) * 32;  // 16 token rows x 32
            // the first two partial accumulators with one TMEM round trip, any
            // further ones one by one; summed in the fixed order
            // ((p0 + p1) + p2) + p3
            uint32_t v[16], w[16];
            tmem_ld_32x32b_x16(dcol0 + j0, v);
            if (live_parts > 1) tmem_ld_32x32b_x16(dcol0 + args.d_cols + j0, w);
            tmem_ld_wait();
            if (live_parts > 1) {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj)
                v[jj] = __float_as_uint(__uint_as_float(v[jj]) + __uint_as_float(w[jj]));
            }
            for (int p = 2; p < live_parts; ++p) {
              tmem_ld_32x32b_x16(dcol0 + p * args.d_cols + j0, w);
              tmem_ld_wait();
#pragma unroll
              for (int jj = 0; jj < 16; ++jj)
                v[jj] = __float_as_uint(__uint_as_float(v[jj]) + __uint_as_float(w[jj]));
            }
            if constexpr (kGlu) {
              // Fused activation: lanes 0..15 hold gate columns, lanes 16..31 the
              // matching up columns (W4A16_LAYOUT_KTILE64_GLU16). Per pair of
              // token columns, lane l < 16 computes column 2m and lane l + 16
              // column 2m + 1: one exchange gives each the other half of its
              // (gate, up) pair. Both are rounded to BF16 as the unfused gate_up
              // output would be, then combined as in w4a16_silu_and_mul; the
              // 16 x 16 results are staged transposed ([token row][16]).
              const bool hi_lane = lane >= 16;
#pragma unroll
              for (int m = 0; m < 8; ++m) {
                const float v0 = __uint_as_float(v[2 * m]);
                const float v1 = __uint_as_float(v[2 * m + 1]);
                const float recv = __shfl_xor_sync(0xffffffffu, hi_lane ? v0 : v1, 16);
                const float g = __bfloat162float(__float2bfloat16_rn(hi_lane ? recv : v0));
                const float u = __bfloat162float(__float2bfloat16_rn(hi_lane ? v1 : recv));
                slab[(2 * m + (hi_lane ? 1 : 0)) * 16 + (lane & 15)] =
                    __fdividef(g, 1.0f + __expf(-g)) * u;
              }
            } else if (half_stage) {
              // transposed and rounded to the BF16 the output holds
              __nv_bfloat16* slab_h = tile_h + (j0 - p0) * 32;
#pragma unroll
              for (int jj = 0; jj < 16; ++jj)
                slab_h[jj * 32 + lane] = __float2bfloat16_rn(__uint_as_float(v[jj]));
            } else {
              // transposed: slab[jj][lane] = value of token column j0 + jj for
              // weight row lane
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) slab[jj * 32 + lane] = __uint_as_float(v[jj]);
            }
          }
          __syncwarp();
          if (early) {
            tc_fence_before();
            if (lane == 0) release_acc(B.acce(dslot));
          }
          W4A16_PROF_MARK(1);
          for (int j0 = p0; j0 < p1; j0 += 16) {
            const float* slab = tile + (j0 - p0) * 32;
            if constexpr (kGlu) {
              const int inter = args.n >> 1;
              const int gcol = d.tile * 64 + quarter * 16 + 4 * (lane & 3);
              for (int jr = lane >> 2; jr < 16 && j0 + jr < rows; jr += 8) {
                const int dr = idst[j0 + jr];
                if (dr < 0) continue;
                const float4 x = *reinterpret_cast<const float4*>(slab + jr * 16 + 4 * (lane & 3));
                const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
                uint2 pk;
                pk.x = *reinterpret_cast<const uint32_t*>(&lo);
                pk.y = *reinterpret_cast<const uint32_t*>(&hi);
                *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(args.out) +
                                          static_cast<long long>(dr) * inter + gcol) = pk;
              }
            } else {
              // lane (jr, c4) writes token row j0 + jr, columns ng..ng+3
              for (int jr = jr0; jr < 16 && j0 + jr < rows; jr += 4) {
                const int j = j0 + jr;
                const int dr = idst[j];
                if (dr < 0 || ng >= args.n) continue;
                if (half_stage) {
                  const uint2 pk =
                      *reinterpret_cast<const uint2*>(tile_h + (j - p0) * 32 + 4 * c4);
                  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(args.out) +
                                     static_cast<long long>(dr) * args.n + ng;
                  if (vec4) {
                    *reinterpret_cast<uint2*>(o) = pk;
                  } else {
                    const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(&pk);
                    o[0] = hv[0];
                    if (ng + 1 < args.n) o[1] = hv[1];
                    if (ng + 2 < args.n) o[2] = hv[2];
                    if (ng + 3 < args.n) o[3] = hv[3];
                  }
                  continue;
                }
                const float4 x = *reinterpret_cast<const float4*>(slab + jr * 32 + 4 * c4);
                if constexpr (kRows) {
                  // deterministic down pass: the weighted row at its routing position
                  float* o =
                      static_cast<float*>(args.out) + static_cast<long long>(dr) * args.n + ng;
                  const float wt = iwt[j];
                  if (vec4) {
                    *reinterpret_cast<float4*>(o) =
                        make_float4(wt * x.x, wt * x.y, wt * x.z, wt * x.w);
                  } else {
                    o[0] = wt * x.x;
                    if (ng + 1 < args.n) o[1] = wt * x.y;
                    if (ng + 2 < args.n) o[2] = wt * x.z;
                    if (ng + 3 < args.n) o[3] = wt * x.w;
                  }
                } else if (args.out_mode == kOutF32WeightedAdd) {
                  float* o =
                      static_cast<float*>(args.out) + static_cast<long long>(dr) * args.n + ng;
                  const float wt = iwt[j];
                  if (vec4) {
                    atomicAdd(reinterpret_cast<float4*>(o),
                              make_float4(wt * x.x, wt * x.y, wt * x.z, wt * x.w));
                  } else {
                    atomicAdd(o, wt * x.x);
                    if (ng + 1 < args.n) atomicAdd(o + 1, wt * x.y);
                    if (ng + 2 < args.n) atomicAdd(o + 2, wt * x.z);
                    if (ng + 3 < args.n) atomicAdd(o + 3, wt * x.w);
                  }
                } else {
                  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(args.out) +
                                     static_cast<long long>(dr) * args.n + ng;
                  const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
                  const __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
                  if (vec4) {
                    uint2 pk;
                    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
                    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(o) = pk;
                  } else {
                    o[0] = lo.x;
                    if (ng + 1 < args.n) o[1] = lo.y;
                    if (ng + 2 < args.n) o[2] = hi.x;
                    if (ng + 3 < args.n) o[3] = hi.y;
                  }
                }
              }
            }
          }
          __syncwarp();  // the tile is rewritten by the next pass
        }
        if (!early) tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (!early) release_acc(B.acce(dslot));
          mbar_arrive(B.ite(islot));
        }
        W4A16_PROF_MARK(2);
      } else {
        // the item's partial accumulators and their column stride (blocks
        // above 128 rows choose them per item; the others read the launch's)
        int big_parts = 1;
        if constexpr (b_steps) big_parts = big_block_parts(sm.info_n16[islot]);
        auto pstride = [&]() -> int {
          if constexpr (b_steps) {
            return kBigAccCols / big_parts;
          } else {
            return args.d_cols;
          }
        };
        const int live = kLayer    ? min(parts, ksteps_of(d))
                         : b_steps ? min(big_parts, ksteps_of(d))
                                   : live_parts;
        for (int j0 = 0; j0 < rows; j0 += 16) {
          // the first two partial accumulators with one TMEM round trip, any
          // further ones one by one; summed in the fixed order
          // ((p0 + p1) + p2) + p3
          uint32_t v[16], w[16];
          if (live == 4 && rows - j0 <= 8) {
            // at most 8 token columns left (TP8 blocks): all four partials in
            // one TMEM round trip, added in the same fixed order (measured
            // 9-13% faster on TP8 down than three round trips)
            uint32_t a8[8], b8[8], c8[8], d8[8];
            tmem_ld_32x32b_x8(dcol0 + j0, a8);
            tmem_ld_32x32b_x8(dcol0 + pstride() + j0, b8);
            tmem_ld_32x32b_x8(dcol0 + 2 * pstride() + j0, c8);
            tmem_ld_32x32b_x8(dcol0 + 3 * pstride() + j0, d8);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
              v[jj] = __float_as_uint(((__uint_as_float(a8[jj]) + __uint_as_float(b8[jj])) +
                                       __uint_as_float(c8[jj])) +
                                      __uint_as_float(d8[jj]));
#pragma unroll
            for (int jj = 8; jj < 16; ++jj) v[jj] = 0u;
          } else {
            tmem_ld_32x32b_x16(dcol0 + j0, v);
            if (live > 1) tmem_ld_32x32b_x16(dcol0 + pstride() + j0, w);
            tmem_ld_wait();
            if (live > 1) {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj)
                v[jj] = __float_as_uint(__uint_as_float(v[jj]) + __uint_as_float(w[jj]));
            }
            for (int p = 2; p < live; ++p) {
              tmem_ld_32x32b_x16(dcol0 + p * pstride() + j0, w);
              tmem_ld_wait();
#pragma unroll
              for (int jj = 0; jj < 16; ++jj)
                v[jj] = __float_as_uint(__uint_as_float(v[jj]) + __uint_as_float(w[jj]));
            }
          }
          if (kGlu || (kLayer && d.phase == 0)) {
            // Fused activation: lanes 0..15 hold gate columns, lanes 16..31 the
            // matching up columns (W4A16_LAYOUT_KTILE64_GLU16). Per pair of
            // token columns, lane l < 16 computes column 2m and lane l + 16
            // column 2m + 1: one exchange gives each the other half of its
            // (gate, up) pair. Both are rounded to BF16 as the unfused gate_up
            // output would be, then combined as in w4a16_silu_and_mul; the
            // 16 x 16 results are staged transposed and written 4 columns of
            // one token row at a time.
            const bool hi_lane = lane >= 16;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const float v0 = __uint_as_float(v[2 * m]);
              const float v1 = __uint_as_float(v[2 * m + 1]);
              const float recv = __shfl_xor_sync(0xffffffffu, hi_lane ? v0 : v1, 16);
              const float g = __bfloat162float(__float2bfloat16_rn(hi_lane ? recv : v0));
              const float u = __bfloat162float(__float2bfloat16_rn(hi_lane ? v1 : recv));
              tile[(2 * m + (hi_lane ? 1 : 0)) * 16 + (lane & 15)] =
                  __fdividef(g, 1.0f + __expf(-g)) * u;
            }
            __syncwarp();
            const int inter = args.n >> 1;
            const int gcol = d.tile * 64 + quarter * 16 + 4 * (lane & 3);
            for (int jr = lane >> 2; jr < 16 && j0 + jr < rows; jr += 8) {
              const int dr = idst[j0 + jr];
              if (dr < 0) continue;
              const float4 x = *reinterpret_cast<const float4*>(tile + jr * 16 + 4 * (lane & 3));
              const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
              const __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
              uint2 pk;
              pk.x = *reinterpret_cast<const uint32_t*>(&lo);
              pk.y = *reinterpret_cast<const uint32_t*>(&hi);
              *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(args.out) +
                                        static_cast<long long>(dr) * inter + gcol) = pk;
            }
            __syncwarp();  // the tile is rewritten by the next 16 token columns
          } else {
            // the layer's down items add into the layer output (width n2)
            const int nn = kLayer ? args.n2 : args.n;
            void* out_ptr = kLayer ? args.out2 : args.out;
            const bool wadd = kLayer || args.out_mode == kOutF32WeightedAdd;
            // transpose through shared memory: tile[jj][lane] = value of token
            // column j0 + jj for weight row lane
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) tile[jj * 32 + lane] = __uint_as_float(v[jj]);
            __syncwarp();
            // lane (jr, c4) writes token row j0 + jr, columns ng..ng+3
            for (int jr = jr0; jr < 16 && j0 + jr < rows; jr += 4) {
              const int j = j0 + jr;
              const int dr = idst[j];
              if (dr < 0 || ng >= nn) continue;
              const float4 x = *reinterpret_cast<const float4*>(tile + jr * 32 + 4 * c4);
              if constexpr (kRows) {
                // deterministic down pass: the weighted row at its routing position
                float* o =
                    static_cast<float*>(out_ptr) + static_cast<long long>(dr) * nn + ng;
                const float wt = iwt[j];
                if (vec4) {
                  *reinterpret_cast<float4*>(o) =
                      make_float4(wt * x.x, wt * x.y, wt * x.z, wt * x.w);
                } else {
                  o[0] = wt * x.x;
                  if (ng + 1 < nn) o[1] = wt * x.y;
                  if (ng + 2 < nn) o[2] = wt * x.z;
                  if (ng + 3 < nn) o[3] = wt * x.w;
                }
              } else if (wadd) {
                float* o = static_cast<float*>(out_ptr) + static_cast<long long>(dr) * nn + ng;
                const float wt = iwt[j];
                if (vec4) {
                  atomicAdd(reinterpret_cast<float4*>(o),
                            make_float4(wt * x.x, wt * x.y, wt * x.z, wt * x.w));
                } else {
                  atomicAdd(o, wt * x.x);
                  if (ng + 1 < nn) atomicAdd(o + 1, wt * x.y);
                  if (ng + 2 < nn) atomicAdd(o + 2, wt * x.z);
                  if (ng + 3 < nn) atomicAdd(o + 3, wt * x.w);
                }
              } else {
                __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out_ptr) +
                                   static_cast<long long>(dr) * nn + ng;
                const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
                if (vec4) {
                  uint2 pk;
                  pk.x = *reinterpret_cast<const uint32_t*>(&lo);
                  pk.y = *reinterpret_cast<const uint32_t*>(&hi);
                  *reinterpret_cast<uint2*>(o) = pk;
                } else {
                  o[0] = lo.x;
                  if (ng + 1 < nn) o[1] = lo.y;
                  if (ng + 2 < nn) o[2] = hi.x;
                  if (ng + 3 < nn) o[3] = hi.y;
                }
              }
            }
            __syncwarp();  // the tile is rewritten by the next 16 token columns
          }
        }
        if (kLayer && d.phase == 0) {
          // this warp's activation rows of the block are out: count them for
          // the down items that wait on the block (any CTA)
          __threadfence();
          __syncwarp();
          if (lane == 0) atomicAdd(args.block_done + d.blk, 1);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          release_acc(B.acce(dslot));
          mbar_arrive(B.ite(islot));
        }
      }
      ip.next(kItemSlots);
      dp.next(args.d_slots);
    }
    W4A16_PROF_MARK(3);
    W4A16_PROF_STORE();
  }

  // ---- teardown ----
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // a pair's leader may still read the peer's TMEM and shared memory until
  // its issuers have drained: both CTAs leave together
  if constexpr (kPair) cluster_sync_all();
  if (warp == kWarpMma0) {
    tc_fence_after();
    if constexpr (kPair) {
      tmem_dealloc_pair(tmem, kTmemCols);
    } else {
      tmem_dealloc(tmem, kTmemCols);
    }
  }
}

size_t gemm_smem_bytes(int block_m, int w_stages, int b_stages, bool pair) {
  size_t off = 1024;  // alignment slack
  // a CTA of a pair holds half of the block's token rows; a slot holds two
  // k steps, or one above 128 rows
  const int steps_per_slot = (!pair && b_per_step(block_m)) ? 1 : 2;
  off += static_cast<size_t>(b_stages) * steps_per_slot * (pair ? block_m / 2 : block_m) * 128;
  off += static_cast<size_t>(w_stages) * kWStageBytes;
  off += static_cast<size_t>(kItemSlots) * block_m * (4 + 4) + 2 * kItemSlots * 4;
  off = (off + 15) / 16 * 16 + epi_tile_bytes(block_m);
  off = (off + 7) / 8 * 8;
  off += (2 * w_stages + 2 * b_stages + kNumBarsFixed) * 8;
  off += 8;
  // the BF16 staging of 65..128-row blocks (unpaired), 16-byte aligned
  if (!pair && epi_half_stage(block_m)) off = (off + 15) / 16 * 16 + epi_half_bytes(block_m);
  return off;
}

// The epilogue that frees the accumulator slot before its stores: exactly
// the launches whose staging tile holds a whole block (48..64 rows in FP32;
// 65..128 rows in BF16 when the output is BF16, unpaired).
bool early_epilogue(int block_m, int out_mode, bool pair) {
  return epi_stage_rows(block_m) > 16 || (epi_half_stage(block_m) && out_mode == kOutBf16 && !pair);
}

bool tmem_accumulators(int block_m, int k_steps, int* d_cols, int* parts, int* d_slots) {
  const int dcols = (block_m + 31) / 32 * 32;
  const int free_cols = kTmemCols - kASlots * kAColsPerSlot;
  // Four issuers while their accumulators fit: one thread issues a
  // tcgen05.mma only every hundred-odd cycles, so even short reductions
  // (TP8 down, k = 256) gain more from four parallel MMA chains (measured 3-7%)
  // than from holding more items in TMEM at once with two.
  int p = kMaxIssuers;
  while (p > 1 && p * dcols > free_cols) p >>= 1;
  if (p * dcols > free_cols) return false;
  // 128-row blocks over a short reduction (k <= 2048): one issuer and two
  // accumulator slots, so that an item's epilogue overlaps the next item's
  // MMAs (grouped contiguous down, k = 2048: 271 -> 220 us at 128 rows per
  // expert); over k = 7168 two issuers and one slot stay faster (377 vs 416).
  if (dcols == 128 && k_steps <= 32) p = 1;
  *d_cols = dcols;
  *parts = p;
  const int slots = free_cols / (p * dcols);
  *d_slots = slots < kMaxDSlots ? slots : kMaxDSlots;
  return true;
}

bool encode_act_tmap(CUtensorMap* map, const void* act, long long rows, int k, int box_rows) {
  using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;
  static EncodeFn encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<EncodeFn>(fn);
  });
  if (encode == nullptr || rows <= 0 || rows > (1LL << 31) || k <= 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(k) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kKStep), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(act), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool encode_permuted_tmap(CUtensorMap* map, const void* act, long long rows, int k_pad,
                          int box_rows, int box_steps) {
  using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;
  static EncodeFn encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<EncodeFn>(fn);
  });
  if (encode == nullptr || rows <= 0 || rows > (1LL << 31) || k_pad <= 0 || k_pad % kKStep != 0 ||
      box_steps < 1 || box_steps > 2)
    return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kKStep), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(k_pad / kKStep)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(k_pad) * 2, kKStep * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kKStep), static_cast<cuuint32_t>(box_rows),
                            static_cast<cuuint32_t>(box_steps)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(act), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

int device_sm_count(int device) {
  static std::mutex mu;
  static int cache[64] = {0};
  if (device < 0 || device >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[device] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    cache[device] = v;
  }
  return cache[device];
}

template <bool kPair>
void* pick_kernel(const GemmArgs& args) {
  const bool glu = args.out_mode == kOutGluBf16;
  const bool rows = args.out_mode == kOutF32Rows;
  const bool early = early_epilogue(args.block_m, args.out_mode, kPair);
  if (!kPair && early && epi_half_stage(args.block_m)) {
    // 65..128-row blocks with a BF16 output: the BF16 staging tile
    auto half = args.raster_rows
                    ? w4a16_moe_gemm_kernel<false, true, true, false, false, false, false, true>
                    : w4a16_moe_gemm_kernel<false, false, true, false, false, false, false, true>;
    return reinterpret_cast<void*>(half);
  }
  if (!kPair && b_per_step(args.block_m)) {
    // blocks above 128 rows: no early release; the grouped item order when
    // the call asks for it (every indexed call does; the fused activation
    // exists only there, and the deterministic rows pass keeps tile-major)
    const bool raster = args.raster_rows != 0;
    auto big = rows ? w4a16_moe_gemm_kernel<false, false, false, true, false, false, true>
               : glu ? w4a16_moe_gemm_kernel<true, true, false, false, false, false, true>
               : raster ? w4a16_moe_gemm_kernel<false, true, false, false, false, false, true>
                        : w4a16_moe_gemm_kernel<false, false, false, false, false, false, true>;
    return reinterpret_cast<void*>(big);
  }
  auto kernel =
      rows ? (early ? w4a16_moe_gemm_kernel<false, false, true, true, kPair>
                    : w4a16_moe_gemm_kernel<false, false, false, true, kPair>)
      : glu ? (early ? w4a16_moe_gemm_kernel<true, false, true, false, kPair>
                     : w4a16_moe_gemm_kernel<true, false, false, false, kPair>)
      : args.raster_rows ? (early ? w4a16_moe_gemm_kernel<false, true, true, false, kPair>
                                  : w4a16_moe_gemm_kernel<false, true, false, false, kPair>)
                         : (early ? w4a16_moe_gemm_kernel<false, false, true, false, kPair>
                                  : w4a16_moe_gemm_kernel<false, false, false, false, kPair>);
  return reinterpret_cast<void*>(kernel);
}

size_t launch_smem_bytes(const GemmArgs& args) {
  // At least 118 KB so that two CTAs never share an SM: each CTA allocates
  // all 512 TMEM columns.
  size_t smem = gemm_smem_bytes(args.block_m, args.w_stages, args.b_stages, args.pair != 0);
  return smem < 118 * 1024 ? 118 * 1024 : smem;
}

int max_pair_clusters(const GemmArgs& args) {
  // CTA pairs that can be resident at once (a pair needs two SMs of one GPC)
  static std::mutex mu;
  static int cache[8][2] = {};
  const bool early = early_epilogue(args.block_m, args.out_mode, true);
  const int key = (args.out_mode == kOutGluBf16 ? 4 : 0) + (args.raster_rows ? 2 : 0) + (early ? 1 : 0);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[key][0] != dev + 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = launch_smem_bytes(args);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    void* k = pick_kernel<true>(args);
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(cfg.dynamicSmemBytes)) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess)
      return 0;
    cache[key][0] = dev + 1;
    cache[key][1] = n;
  }
  return cache[key][1];
}

cudaError_t launch_moe_gemm(const GemmArgs& args, int grid, bool dependent, cudaStream_t stream) {
  const size_t smem = launch_smem_bytes(args);
  // the single-launch layer: the fused activation for its gate_up items and
  // the weighted add for its down items, chosen per item
  void* kernel = args.layer ? reinterpret_cast<void*>(
                                  w4a16_moe_gemm_kernel<false, false, false, false, false, true>)
                 : args.pair ? pick_kernel<true>(args)
                             : pick_kernel<false>(args);
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = dependent ? 1 : 0;
  int nattr = 1;
  if (args.pair) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    nattr = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  void* params[] = {const_cast<GemmArgs*>(&args)};
  return cudaLaunchKernelExC(&cfg, kernel, params);
}

}  // namespace w4a16
