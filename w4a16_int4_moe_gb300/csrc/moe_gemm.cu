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
//     --dequant warps: (q - 8) * s in registers, tcgen05.st--> TMEM (A)
//   tokens (BF16 rows gathered through the routing) --cp.async, 128-byte
//     swizzle--> shared-memory ring (B)
//   tcgen05.mma kind::f16, M = 128 weight rows, N = the block's tokens
//     (rounded to 16, chosen per block at run time), K = 16 per instruction,
//     FP32 accumulators in TMEM (D)
//   epilogue warps: tcgen05.ld --> BF16 row stores, or the top-k weighted
//     FP32 scatter-add of the down pass.
//
// Writing the dequantised weights to TMEM instead of shared memory keeps the
// shared-memory port free for the token operand: at decode (N = 16) a
// shared-memory A operand would cost more shared bandwidth than the HBM
// stream delivers weights.
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

namespace w4a16 {

namespace {

constexpr int kThreads = 576;
constexpr int kWStageBytes = 2 * kStepBytes;  // one weight stage = 2 k steps
constexpr int kAColsPerSlot = 32;             // 64 BF16 of K per TMEM lane
constexpr int kTmemCols = 512;

// warp roles (warp 3 idles; the warpgroups start at multiples of 4 warps so
// that warp % 4 selects the TMEM lane quarter each warp may access)
constexpr int kWarpProducer = 0;
constexpr int kWarpMma0 = 1;        // MMA issuer of the even k steps (+ TMEM allocation)
constexpr int kWarpMma1 = 2;        // MMA issuer of the odd k steps
constexpr int kWarpDequant0 = 4;    // 8 warps (2 warpgroups)
constexpr int kWarpEpilogue0 = 12;  // 4 warps
constexpr int kWarpGather0 = 16;    // 2 warps

// where codes recorded in the status word when a wait gives up
enum Where {
  kWhereProducer = 1, kWhereDequantW = 2, kWhereDequantA = 3, kWhereGatherItem = 4,
  kWhereGatherB = 5, kWhereMmaItem = 6, kWhereMmaAcc = 7, kWhereMmaA = 8, kWhereMmaB = 9,
  kWhereEpiAcc = 10, kWhereEpiItem = 11, kWhereDrain = 12
};

struct Smem {
  uint8_t* b_ring;      // [2 parities][S slots][block_m rows][128 B], 128-byte swizzle
  uint8_t* w_ring;      // [WS stages][2 k steps][kStepBytes]
  int* info_row;        // [2 gather warps][2 item slots][block_m]: activation row, -1 = none
  int* info_dst;        // [2][2][block_m]: output row, -1 = not a real row
  float* info_wt;       // [2][2][block_m]: top-k weight (down pass)
  int* info_n16;        // [2][2]: MMA N of the item
  uint64_t* bars;
  uint32_t* tmem_base;
  volatile int* abort_flag;
};

// mbarrier addresses (shared-window offsets, 8 bytes each)
struct Bars {
  uint32_t w_full, w_empty, a_full, b_full, ab_empty, item_full, item_empty, acc_full, acc_empty,
      final_bar;
  __device__ uint32_t wf(int i) const { return w_full + 8u * i; }
  __device__ uint32_t we(int i) const { return w_empty + 8u * i; }
  __device__ uint32_t af(int i) const { return a_full + 8u * i; }
  __device__ uint32_t bf(int i) const { return b_full + 8u * i; }
  __device__ uint32_t abe(int i) const { return ab_empty + 8u * i; }
  __device__ uint32_t itf(int i) const { return item_full + 8u * i; }
  __device__ uint32_t ite(int i) const { return item_empty + 8u * i; }
  __device__ uint32_t accf(int i) const { return acc_full + 8u * i; }
  __device__ uint32_t acce(int i) const { return acc_empty + 8u * i; }
  __device__ uint32_t fin(int i) const { return final_bar + 8u * i; }
};

__device__ __forceinline__ size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bounded wait: true when the phase of parity `parity` has completed; false
// when the CTA is aborting or this wait ran out (then it starts the abort).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                        int* status, int where, long long timeout) {
  constexpr uint32_t kSuspendNs = 1000000;  // the thread sleeps until completion or 1 ms
  if (mbar_try_wait_sleep(bar, parity, kSuspendNs)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kSuspendNs)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > timeout) {
      *abort_flag = 1;
      if (status != nullptr) atomicCAS(status, 0, 0x1000 | where);
      return false;
    }
  }
}

// Position in a ring of mbarrier-guarded slots: slot index and the parity of
// the slot's current phase (incremented without divisions).
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

struct ItemDesc {
  int blk, tile, e;
};

// Which routing block and weight tile item `it` is, and its expert (-1: skip).
__device__ __forceinline__ ItemDesc decode_item(const GemmArgs& a, int it, int num_blocks,
                                                int blocks_per_expert) {
  ItemDesc d;
  d.tile = it / num_blocks;
  d.blk = it - d.tile * num_blocks;
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

// Row j of block `blk`: activation row, output row (-1 = not a real row) and
// the top-k weight of the down pass.
__device__ __forceinline__ void row_info(const GemmArgs& a, const ItemDesc& d, int j, int& src,
                                         int& dst, float& wt) {
  src = -1;
  dst = -1;
  wt = 0.f;
  if (a.family == kIndexed) {
    const int id = __ldg(a.sorted_ids + static_cast<long long>(d.blk) * a.block_m + j);
    if (id >= 0 && id < a.numel) {
      src = id / a.a_div;
      dst = id / a.o_div;
      wt = (a.out_mode == kOutF32WeightedAdd) ? __ldg(a.topk_weights + id) : 1.f;
    }
  } else if (a.family == kContiguous) {
    const int r = d.blk * a.block_m + j;
    if (r < a.m && __ldg(a.layout + r) == d.e) {
      src = r;
      dst = r;
      wt = 1.f;
    }
  } else {
    const int bpe = (a.m + a.block_m - 1) / a.block_m;
    const int rl = (d.blk - d.e * bpe) * a.block_m + j;
    const int valid = min(max(__ldg(a.layout + d.e), 0), a.m);
    if (rl < valid) {
      src = d.e * a.m + rl;
      dst = src;
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

__global__ void __launch_bounds__(kThreads, 1)
    w4a16_moe_gemm_kernel(const __grid_constant__ GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- shared-memory carve-up (base aligned to 1024 for the swizzle) ----
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const int bm = args.block_m;
  const int S = args.a_slots;  // operand ring slots per k-step parity
  const int WS = args.w_stages;
  const bool gather = args.gather_rows != 0;
  const uint32_t b_slot_bytes = static_cast<uint32_t>(max_mma_n(bm, gather)) * 128u;
  Smem sm;
  size_t off = 0;
  sm.b_ring = base;
  off += static_cast<size_t>(2 * S) * b_slot_bytes;
  sm.w_ring = base + off;
  off += static_cast<size_t>(WS) * kWStageBytes;
  sm.info_row = reinterpret_cast<int*>(base + off);
  off += 4 * bm * sizeof(int);
  sm.info_dst = reinterpret_cast<int*>(base + off);
  off += 4 * bm * sizeof(int);
  sm.info_wt = reinterpret_cast<float*>(base + off);
  off += 4 * bm * sizeof(float);
  sm.info_n16 = reinterpret_cast<int*>(base + off);
  off += 4 * sizeof(int);
  off = align_up(off, 8);
  sm.bars = reinterpret_cast<uint64_t*>(base + off);
  off += (2 * WS + 6 * S + 10) * 8;
  sm.tmem_base = reinterpret_cast<uint32_t*>(base + off);
  off += 4;
  sm.abort_flag = reinterpret_cast<volatile int*>(base + off);

  Bars B;
  {
    uint32_t b0 = smem_u32(sm.bars);
    B.w_full = b0;
    b0 += 8 * WS;
    B.w_empty = b0;
    b0 += 8 * WS;
    B.a_full = b0;
    b0 += 8 * 2 * S;
    B.b_full = b0;
    b0 += 8 * 2 * S;
    B.ab_empty = b0;
    b0 += 8 * 2 * S;
    B.item_full = b0;
    b0 += 16;
    B.item_empty = b0;
    b0 += 16;
    B.acc_full = b0;
    b0 += 16;
    B.acc_empty = b0;
    b0 += 16;
    B.final_bar = b0;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < WS; ++i) {
      mbar_init(B.wf(i), 1);
      mbar_init(B.we(i), 8);  // every dequant warp releases every stage
    }
    for (int i = 0; i < 2 * S; ++i) {
      mbar_init(B.af(i), 4);   // the 4 warps of the dequant warpgroup
      mbar_init(B.bf(i), 1);   // the gather warp's expect_tx (plus the copies' bytes)
      mbar_init(B.abe(i), 1);  // one tcgen05.commit of the MMA issuer
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(B.itf(i), 2);   // lane 0 of each gather warp
      mbar_init(B.ite(i), 4);   // the 4 epilogue warps
      mbar_init(B.accf(i), 2);  // one tcgen05.commit per MMA issuer
      mbar_init(B.acce(i), 4);
      mbar_init(B.fin(i), 1);
    }
    *sm.abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kWarpMma0) {
    tmem_alloc(smem_u32(sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
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
  const int items = num_blocks * args.n_tiles;
  // TMEM columns: the 2*S A slots (32 columns each), then per accumulator
  // slot the two partial accumulators (even / odd k steps), d_cols each.
  const int d_col_base = 2 * S * kAColsPerSlot;
  const int n_wst = (args.k_steps + 1) / 2;
  const long long tmo = args.timeout_cycles;
  volatile int* abort_flag = sm.abort_flag;
  int* status = args.status;

  // The k steps of one parity g form one pipeline: dequant warpgroup g fills
  // the A slot (TMEM), gather warp g the B slot (shared memory) of ring slot
  // g*S + c % S, where c counts that parity's k steps over all items; MMA
  // issuer g consumes both and frees the slot with one tcgen05.commit.

  if (warp == kWarpProducer) {
    // ======================= weight producer (bulk copies) ==================
    if (lane == 0) {
      const uint64_t policy = policy_evict_first();
      uint32_t wcnt = 0;
      RingPos wp;
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        const ItemDesc d = decode_item(args, it, num_blocks, bpe);
        if (d.e < 0) continue;
        const uint8_t* src = args.wpack + static_cast<long long>(d.e) * args.expert_bytes +
                             static_cast<long long>(d.tile) * args.k_steps * kStepBytes;
        for (int st = 0; st < n_wst; ++st, ++wcnt, wp.next(WS)) {
          if (!wait_phase(B.we(wp.slot), wp.phase ^ 1, abort_flag, status, kWhereProducer, tmo)) {
            ok = false;
            break;
          }
          const int nks = min(2, args.k_steps - 2 * st);
          const uint32_t bytes = static_cast<uint32_t>(nks * kStepBytes);
          mbar_arrive_expect_tx(B.wf(wp.slot), bytes);
          bulk_g2s(smem_u32(sm.w_ring + static_cast<size_t>(wp.slot) * kWStageBytes),
                   src + static_cast<long long>(st) * kWStageBytes, bytes, B.wf(wp.slot), policy);
        }
      }
      if (!ok) {
        // Let every copy already issued land before the CTA can exit.
        const uint32_t first = wcnt > static_cast<uint32_t>(WS) ? wcnt - WS : 0;
        for (uint32_t u = first; u < wcnt; ++u) {
          const int slot = u % WS;
          const uint32_t ph = (u / WS) & 1;
          const long long t0 = clock64();
          while (!mbar_try_wait(B.wf(slot), ph) && clock64() - t0 < tmo) {
          }
        }
      }
    }
  } else if (warp == kWarpMma0 || warp == kWarpMma1) {
    // ======================= MMA issuers ====================================
    // Issuer g owns the k steps with ks % 2 == g and accumulates into its own
    // FP32 partial accumulator; the epilogue adds the two partials in a fixed
    // order. At small N one issuing thread, not the tensor core, sets the
    // pace (each tcgen05.mma blocks its issuer for tens of cycles), so two
    // independent issuers double the MMA rate.
    const int g = warp - kWarpMma0;
    if (lane == 0) {
      RingPos rp, ip, dp;
      bool ok = true;
      // descriptor of ring slot 0 of this parity; later slots add their offset
      const uint64_t b_desc0 =
          smem_desc_sw128_kmajor(smem_u32(sm.b_ring + static_cast<size_t>(g * S) * b_slot_bytes));
      const uint32_t b_slot_step = b_slot_bytes >> 4;  // in descriptor address units
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        const ItemDesc d = decode_item(args, it, num_blocks, bpe);
        if (d.e < 0) continue;
        if (!wait_phase(B.itf(ip.slot), ip.phase, abort_flag, status, kWhereMmaItem, tmo)) {
          ok = false;
          break;
        }
        const int n16 = sm.info_n16[ip.slot];  // gather warp 0's copy
        if (!wait_phase(B.acce(dp.slot), dp.phase ^ 1, abort_flag, status, kWhereMmaAcc, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_m128(static_cast<uint32_t>(n16));
        const uint32_t d_tmem = tmem + d_col_base + (dp.slot * 2 + g) * args.d_cols;
        uint32_t acc = 0;
        for (int ks = g; ks < args.k_steps; ks += 2, rp.next(S)) {
          const int slot = g * S + rp.slot;
          if (!wait_phase(B.af(slot), rp.phase, abort_flag, status, kWhereMmaA, tmo) ||
              !wait_phase(B.bf(slot), rp.phase, abort_flag, status, kWhereMmaB, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t b_desc = b_desc0 + static_cast<uint64_t>(rp.slot) * b_slot_step;
          const uint32_t a_tmem = tmem + slot * kAColsPerSlot;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // +32 bytes of K per MMA inside the 128-byte swizzle row
            mma_bf16_ts(d_tmem, a_tmem + kk * 8, b_desc + 2 * kk, idesc, acc);
            acc = 1;
          }
          tc_commit(B.abe(slot));
        }
        if (!ok) break;
        tc_commit(B.accf(dp.slot));
        ip.next(2);
        dp.next(args.d_slots);
      }
      // every MMA issued by this thread has finished once its final barrier flips
      tc_commit(B.fin(g));
      const long long t0 = clock64();
      while (!mbar_try_wait(B.fin(g), 0) && clock64() - t0 < tmo) {
      }
    }
  } else if (warp >= kWarpGather0) {
    // ======================= activation loads (TMA) =========================
    // Gather warp g fills the B slots of parity g with tensor copies that
    // write the 128-byte-swizzled K-major layout the MMA descriptor expects
    // and count their bytes on the slot's mbarrier.
    //  - gathered rows (indexed family): tile::gather4 puts 4 routed rows at
    //    the start of an 8-row swizzle atom (rows 4..7 of the atom are not
    //    used), so every copy starts 1024-byte aligned; the MMA N covers 8
    //    columns per 4 rows and the epilogue skips the unused columns;
    //  - consecutive rows (grouped families): one 64 x 8 box per atom.
    const int g = warp - kWarpGather0;
    const void* map = &args.tmap;
    RingPos rp, ip;
    bool ok = true;
    for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
      const ItemDesc d = decode_item(args, it, num_blocks, bpe);
      if (d.e < 0) continue;
      const int islot = ip.slot;
      ok = __all_sync(0xffffffffu, wait_phase(B.ite(islot), ip.phase ^ 1, abort_flag, status,
                                               kWhereGatherItem, tmo));
      if (!ok) break;
      const int copy = g * 2 + islot;
      int* irow = sm.info_row + copy * bm;
      int* idst = sm.info_dst + copy * bm;
      float* iwt = sm.info_wt + copy * bm;
      int maxj = -1;
      for (int j = lane; j < bm; j += 32) {
        int s, dd;
        float w;
        row_info(args, d, j, s, dd, w);
        irow[j] = s;
        idst[j] = dd;
        iwt[j] = w;
        if (dd >= 0) maxj = j;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) maxj = max(maxj, __shfl_xor_sync(0xffffffffu, maxj, o));
      // atoms to load and the MMA N (a multiple of 16 columns)
      const int rows_needed = max(maxj + 1, 1);
      const int n_copies = gather ? (rows_needed + 3) / 4 : (rows_needed + 7) / 8;
      const int n_mma = ((n_copies * 8) + 15) & ~15;
      if (lane == 0) sm.info_n16[copy] = n_mma;
      __syncwarp();
      if (lane == 0) mbar_arrive(B.itf(islot));
      // per-lane copy coordinates, fixed for the item
      int r0 = args.act_rows, r1 = args.act_rows, r2 = args.act_rows, r3 = args.act_rows;
      if (lane < n_copies) {
        if (gather) {
          const int j = 4 * lane;
          r0 = irow[j] >= 0 ? irow[j] : args.act_rows;
          r1 = (j + 1 < bm && irow[j + 1] >= 0) ? irow[j + 1] : args.act_rows;
          r2 = (j + 2 < bm && irow[j + 2] >= 0) ? irow[j + 2] : args.act_rows;
          r3 = (j + 3 < bm && irow[j + 3] >= 0) ? irow[j + 3] : args.act_rows;
        } else {
          // first row of this atom in the activation tensor (consecutive rows)
          r0 = (args.family == kContiguous) ? d.blk * bm + 8 * lane
                                            : d.e * args.m + (d.blk - d.e * bpe) * bm + 8 * lane;
        }
      }
      const uint32_t copy_bytes = gather ? 512u : 1024u;
      for (int ks = g; ks < args.k_steps; ks += 2, rp.next(S)) {
        const int slot = g * S + rp.slot;
        ok = __all_sync(0xffffffffu, wait_phase(B.abe(slot), rp.phase ^ 1, abort_flag, status,
                                                 kWhereGatherB, tmo));
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(B.bf(slot), n_copies * copy_bytes);
        __syncwarp();
        if (lane < n_copies) {
          const uint32_t dst =
              smem_u32(sm.b_ring + static_cast<size_t>(slot) * b_slot_bytes) + lane * 1024u;
          if (gather) {
            tma_gather4(dst, map, ks * kKStep, r0, r1, r2, r3, B.bf(slot));
          } else {
            tma_load_2d(dst, map, ks * kKStep, r0, B.bf(slot));
          }
        }
      }
      if (!ok) break;
      ip.next(2);
    }
  } else if (warp >= kWarpDequant0 && warp < kWarpEpilogue0) {
    // ======================= dequantisation into TMEM =======================
    // Warpgroup g dequantises the k steps with ks % 2 == g; thread r of the
    // warpgroup owns weight row r of the tile, i.e. TMEM lane r.
    const int g = (warp - kWarpDequant0) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    RingPos wp, rp;
    bool ok = true;
    for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
      const ItemDesc d = decode_item(args, it, num_blocks, bpe);
      if (d.e < 0) continue;
      for (int st = 0; st < n_wst; ++st, wp.next(WS)) {
        const int wslot = wp.slot;
        ok = __all_sync(0xffffffffu, wait_phase(B.wf(wslot), wp.phase, abort_flag, status,
                                                 kWhereDequantW, tmo));
        if (!ok) break;
        const int ks = 2 * st + g;
        if (ks >= args.k_steps) {
          __syncwarp();
          if (lane == 0) mbar_arrive(B.we(wslot));
          continue;
        }
        const uint8_t* stp = sm.w_ring + static_cast<size_t>(wslot) * kWStageBytes + g * kStepBytes;
        const uint4 q0 = *reinterpret_cast<const uint4*>(stp + r * 16);
        const uint4 q1 = *reinterpret_cast<const uint4*>(stp + 2048 + r * 16);
        const uint32_t s0 = *reinterpret_cast<const uint16_t*>(stp + kStepQBytes + r * 2);
        const uint32_t s1 = *reinterpret_cast<const uint16_t*>(stp + kStepQBytes + 256 + r * 2);
        __syncwarp();
        if (lane == 0) mbar_arrive(B.we(wslot));
        uint32_t v[32];
        dequant_group(q0, s0, v);
        dequant_group(q1, s1, v + 16);
        const int slot = g * S + rp.slot;
        ok = __all_sync(0xffffffffu, wait_phase(B.abe(slot), rp.phase ^ 1, abort_flag, status,
                                                 kWhereDequantA, tmo));
        if (!ok) break;
        tc_fence_after();
        tmem_st_32x32b_x32(tmem + lane_base + slot * kAColsPerSlot, v);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B.af(slot));
        rp.next(S);
      }
    }
  } else if (warp >= kWarpEpilogue0) {
    // ======================= epilogue =======================================
    // Thread r owns weight row r of the tile (TMEM lane r): it reads the
    // block's token columns of both partial accumulators and writes output
    // column tile*128 + r.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    RingPos ip, dp;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
      const ItemDesc d = decode_item(args, it, num_blocks, bpe);
      if (d.e < 0) continue;
      const int islot = ip.slot;
      const int dslot = dp.slot;
      bool ok = wait_phase(B.accf(dslot), dp.phase, abort_flag, status, kWhereEpiAcc, tmo) &&
                wait_phase(B.itf(islot), ip.phase, abort_flag, status, kWhereEpiItem, tmo);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int n16 = sm.info_n16[islot];  // gather warp 0's copy
      const int* idst = sm.info_dst + islot * bm;
      const float* iwt = sm.info_wt + islot * bm;
      const int ng = d.tile * kTileRows + r;
      const bool row_ok = ng < args.n;
      const uint32_t dcol0 = tmem + lane_base + d_col_base + (dslot * 2) * args.d_cols;
      const uint32_t dcol1 = dcol0 + args.d_cols;
      const bool odd_steps = args.k_steps > 1;  // the odd-k accumulator holds data
      for (int j0 = 0; j0 < n16; j0 += 16) {
        uint32_t v[16], w[16];
        tmem_ld_32x32b_x16(dcol0 + j0, v);
        if (odd_steps) tmem_ld_32x32b_x16(dcol1 + j0, w);
        tmem_ld_wait();
        if (!row_ok) continue;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          // MMA column -> block row (gathered rows use 4 of every 8 columns)
          const int c = j0 + jj;
          int j = c;
          if (gather) {
            if ((c & 7) >= 4) continue;
            j = (c >> 3) * 4 + (c & 3);
          }
          if (j >= bm) continue;
          const int dr = idst[j];
          if (dr < 0) continue;
          const float x = odd_steps ? __uint_as_float(v[jj]) + __uint_as_float(w[jj])
                                    : __uint_as_float(v[jj]);
          if (args.out_mode == kOutF32WeightedAdd) {
            float* o = static_cast<float*>(args.out) + static_cast<long long>(dr) * args.n + ng;
            atomicAdd(o, iwt[j] * x);
          } else {
            __nv_bfloat16* o =
                static_cast<__nv_bfloat16*>(args.out) + static_cast<long long>(dr) * args.n + ng;
            *o = __float2bfloat16_rn(x);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(B.acce(dslot));
        mbar_arrive(B.ite(islot));
      }
      ip.next(2);
      dp.next(args.d_slots);
    }
  }

  // ---- teardown ----
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

size_t gemm_smem_bytes(int block_m, bool gather, int w_stages, int ring_slots) {
  size_t off = 1024;  // alignment slack
  off += static_cast<size_t>(2 * ring_slots) * max_mma_n(block_m, gather) * 128;
  off += static_cast<size_t>(w_stages) * kWStageBytes;
  off += 4 * static_cast<size_t>(block_m) * (4 + 4 + 4) + 4 * 4;
  off = (off + 7) / 8 * 8;
  off += (2 * w_stages + 6 * ring_slots + 10) * 8;
  off += 8;
  return off;
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

cudaError_t launch_moe_gemm(const GemmArgs& args, int grid, cudaStream_t stream) {
  // At least 118 KB so that two CTAs never share an SM: each CTA allocates
  // all 512 TMEM columns.
  size_t smem = gemm_smem_bytes(args.block_m, args.gather_rows != 0, args.w_stages, args.a_slots);
  if (smem < 118 * 1024) smem = 118 * 1024;
  cudaError_t err = cudaFuncSetAttribute(w4a16_moe_gemm_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  w4a16_moe_gemm_kernel<<<grid, kThreads, smem, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace w4a16
