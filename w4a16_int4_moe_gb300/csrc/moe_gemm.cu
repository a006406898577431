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

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace w4a16 {

namespace {

constexpr int kThreads = 576;
constexpr int kWStageBytes = 2 * kStepBytes;  // one weight stage = 2 k steps
constexpr int kMaxASlots = 16;                // A slots over both dequant warpgroups
constexpr int kAColsPerSlot = 32;             // 64 BF16 of K per TMEM lane
constexpr int kTmemCols = 512;
constexpr int kGatherLag = 2;

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
  uint8_t* b_ring;
  uint8_t* w_ring;
  int* info_src;   // [2 gather warps][2 item slots][block_m]
  int* info_dst;   // [2][2][block_m]
  float* info_wt;  // [2][2][block_m]
  int* info_n16;   // [2][2]
  uint64_t* bars;
  uint32_t* tmem_base;
  volatile int* abort_flag;
};

struct Bars {
  uint32_t w_full, w_empty, a_full, a_empty, b_full, b_empty, item_full, item_empty, acc_full,
      acc_empty, final_bar;
  int ws, bs;
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
};

__device__ __forceinline__ size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bounded wait: true when the phase of parity `parity` has completed; false
// when the CTA is aborting or this wait ran out (then it starts the abort).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                        int* status, int where, long long timeout) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > timeout) {
      *abort_flag = 1;
      if (status != nullptr) atomicCAS(status, 0, 0x1000 | where);
      return false;
    }
  }
}

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

__global__ void __launch_bounds__(kThreads, 1) w4a16_moe_gemm_kernel(const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- shared-memory carve-up (base aligned to 1024 for the swizzle) ----
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  Smem sm;
  size_t off = 0;
  const int bm = args.block_m;
  sm.b_ring = base + off;
  off += static_cast<size_t>(args.b_stages) * bm * 128;
  sm.w_ring = base + off;
  off += static_cast<size_t>(args.w_stages) * kWStageBytes;
  sm.info_src = reinterpret_cast<int*>(base + off);
  off += 4 * bm * sizeof(int);
  sm.info_dst = reinterpret_cast<int*>(base + off);
  off += 4 * bm * sizeof(int);
  sm.info_wt = reinterpret_cast<float*>(base + off);
  off += 4 * bm * sizeof(float);
  sm.info_n16 = reinterpret_cast<int*>(base + off);
  off += 4 * sizeof(int);
  off = align_up(off, 8);
  sm.bars = reinterpret_cast<uint64_t*>(base + off);
  const int WS = args.w_stages, BS = args.b_stages;
  const int SA = args.a_slots;  // A slots per dequant warpgroup
  const int n_bars = 2 * WS + 4 * SA + 2 * BS + 2 + 2 + 2 + 2 + 2;
  off += n_bars * 8;
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
    b0 += 8 * 2 * SA;
    B.a_empty = b0;
    b0 += 8 * 2 * SA;
    B.b_full = b0;
    b0 += 8 * BS;
    B.b_empty = b0;
    b0 += 8 * BS;
    B.item_full = b0;
    b0 += 16;
    B.item_empty = b0;
    b0 += 16;
    B.acc_full = b0;
    b0 += 16;
    B.acc_empty = b0;
    b0 += 16;
    B.final_bar = b0;
    B.ws = WS;
    B.bs = BS;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < WS; ++i) {
      mbar_init(B.wf(i), 1);
      mbar_init(B.we(i), 8);  // every dequant warp releases every stage
    }
    for (int i = 0; i < 2 * SA; ++i) {
      mbar_init(B.af(i), 4);  // the 4 warps of the owning warpgroup
      mbar_init(B.ae(i), 1);  // tcgen05.commit
    }
    for (int i = 0; i < BS; ++i) {
      mbar_init(B.bf(i), 32);  // every lane of the owning gather warp
      mbar_init(B.be(i), 1);   // tcgen05.commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(B.itf(i), 2);  // lane 0 of each gather warp
      mbar_init(B.ite(i), 4);
      mbar_init(B.accf(i), 2);  // one tcgen05.commit per MMA issuer
      mbar_init(B.acce(i), 4);
    }
    mbar_init(B.final_bar, 1);
    mbar_init(B.final_bar + 8, 1);
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
  // TMEM columns: A slots first, then per accumulator slot the two partial
  // accumulators (even / odd k steps) of d_cols columns each.
  const int d_col_base = 2 * SA * kAColsPerSlot;
  const int n_wst = (args.k_steps + 1) / 2;
  const long long tmo = args.timeout_cycles;
  volatile int* abort_flag = sm.abort_flag;
  int* status = args.status;

  if (warp == kWarpProducer) {
    // ======================= weight producer (bulk copies) ==================
    if (lane == 0) {
      const uint64_t policy = policy_evict_first();
      uint32_t wcnt = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        const ItemDesc d = decode_item(args, it, num_blocks, bpe);
        if (d.e < 0) continue;
        const uint8_t* src = args.wpack + static_cast<long long>(d.e) * args.expert_bytes +
                             static_cast<long long>(d.tile) * args.k_steps * kStepBytes;
        for (int st = 0; st < n_wst; ++st, ++wcnt) {
          const int slot = wcnt % WS;
          const uint32_t ph = (wcnt / WS) & 1;
          if (!wait_phase(B.we(slot), ph ^ 1, abort_flag, status, kWhereProducer, tmo)) {
            ok = false;
            break;
          }
          const int nks = min(2, args.k_steps - 2 * st);
          const uint32_t bytes = static_cast<uint32_t>(nks * kStepBytes);
          mbar_arrive_expect_tx(B.wf(slot), bytes);
          bulk_g2s(smem_u32(sm.w_ring + static_cast<size_t>(slot) * kWStageBytes),
                   src + static_cast<long long>(st) * kWStageBytes, bytes, B.wf(slot), policy);
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
    // Issuer g owns the k steps with ks % 2 == g: it consumes dequant
    // warpgroup g's A slots and gather warp g's B stages, and accumulates into
    // its own FP32 partial accumulator; the epilogue adds the two partials in
    // a fixed order. At small N one issuing thread, not the tensor core, sets
    // the pace (each tcgen05.mma blocks its issuer for tens of cycles), so two
    // independent issuers double the MMA rate.
    const int g = warp - kWarpMma0;
    if (lane == 0) {
      uint32_t acnt = 0, bcnt = 0, icnt = 0, dcnt = 0;
      const int bhalf = BS / 2;
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        const ItemDesc d = decode_item(args, it, num_blocks, bpe);
        if (d.e < 0) continue;
        const int islot = icnt & 1;
        if (!wait_phase(B.itf(islot), (icnt >> 1) & 1, abort_flag, status, kWhereMmaItem, tmo)) {
          ok = false;
          break;
        }
        const int n16 = sm.info_n16[islot];  // gather warp 0's copy
        const int dslot = dcnt % args.d_slots;
        if (!wait_phase(B.acce(dslot), ((dcnt / args.d_slots) & 1) ^ 1, abort_flag, status,
                        kWhereMmaAcc, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_m128(static_cast<uint32_t>(n16));
        const uint32_t d_tmem = tmem + d_col_base + (dslot * 2 + g) * args.d_cols;
        for (int ks = g; ks < args.k_steps; ks += 2) {
          const int aslot = g * SA + static_cast<int>(acnt % SA);
          const int bslot = 2 * static_cast<int>(bcnt % bhalf) + g;
          if (!wait_phase(B.af(aslot), (acnt / SA) & 1, abort_flag, status, kWhereMmaA, tmo) ||
              !wait_phase(B.bf(bslot), (bcnt / bhalf) & 1, abort_flag, status, kWhereMmaB, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t b_addr = smem_u32(sm.b_ring + static_cast<size_t>(bslot) * bm * 128);
          const uint32_t a_tmem = tmem + aslot * kAColsPerSlot;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            mma_bf16_ts(d_tmem, a_tmem + kk * 8, smem_desc_sw128_kmajor(b_addr + kk * 32), idesc,
                        (ks != g || kk != 0) ? 1u : 0u);
          }
          tc_commit(B.ae(aslot));
          tc_commit(B.be(bslot));
          ++acnt;
          ++bcnt;
        }
        if (!ok) break;
        tc_commit(B.accf(dslot));
        ++icnt;
        ++dcnt;
      }
      // every MMA issued by this thread has finished once its final barrier flips
      tc_commit(B.final_bar + 8 * g);
      const long long t0 = clock64();
      while (!mbar_try_wait(B.final_bar + 8 * g, 0) && clock64() - t0 < tmo) {
      }
    }
  } else if (warp >= kWarpGather0) {
    // ======================= token gather (cp.async) ========================
    // Gather warp gw fills the B stages of the k steps with ks % 2 == gw into
    // its own half of the ring, and keeps its own copy of the block's row
    // information, so the two warps never wait on each other.
    const int gw = warp - kWarpGather0;
    const int half = BS / 2;
    const int lag = half > 2 ? kGatherLag : 1;
    uint32_t bcnt = 0, icnt = 0;
    int npend = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
      const ItemDesc d = decode_item(args, it, num_blocks, bpe);
      if (d.e < 0) continue;
      const int islot = icnt & 1;
      ok = __all_sync(0xffffffffu, wait_phase(B.ite(islot), ((icnt >> 1) & 1) ^ 1, abort_flag,
                                               status, kWhereGatherItem, tmo));
      if (!ok) break;
      const int copy = gw * 2 + islot;
      int* isrc = sm.info_src + copy * bm;
      int* idst = sm.info_dst + copy * bm;
      float* iwt = sm.info_wt + copy * bm;
      int maxj = -1;
      for (int j = lane; j < bm; j += 32) {
        int s, dd;
        float w;
        row_info(args, d, j, s, dd, w);
        isrc[j] = s;
        idst[j] = dd;
        iwt[j] = w;
        if (dd >= 0) maxj = j;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) maxj = max(maxj, __shfl_xor_sync(0xffffffffu, maxj, o));
      int n16 = (maxj + 1 + 15) & ~15;
      if (n16 == 0) n16 = 16;  // a block with no real row still runs a valid MMA
      if (lane == 0) sm.info_n16[copy] = n16;
      __syncwarp();
      if (lane == 0) mbar_arrive(B.itf(islot));
      const int chunks = n16 * 8;
      for (int ks = gw; ks < args.k_steps; ks += 2, ++bcnt) {
        const int bslot = 2 * (bcnt % half) + gw;
        ok = __all_sync(0xffffffffu, wait_phase(B.be(bslot), ((bcnt / half) & 1) ^ 1, abort_flag,
                                                 status, kWhereGatherB, tmo));
        if (!ok) break;
        const uint32_t stage = smem_u32(sm.b_ring + static_cast<size_t>(bslot) * bm * 128);
        for (int idx = lane; idx < chunks; idx += 32) {
          const int j = idx >> 3, c = idx & 7;
          const int srow = isrc[j];
          const int kidx = ks * kKStep + c * 8;
          const uint32_t dst = stage + (j >> 3) * 1024 + (j & 7) * 128 + ((c ^ (j & 7)) << 4);
          if (srow >= 0 && kidx < args.k) {
            cp_async_16(dst, args.act + static_cast<long long>(srow) * args.k + kidx, 16);
          } else {
            cp_async_16(dst, args.act, 0);
          }
        }
        cp_async_commit();
        ++npend;
        if (npend > lag) {
          if (lag == 2) cp_async_wait<2>(); else cp_async_wait<1>();
          fence_proxy_async_smem();
          const uint32_t u = bcnt - lag;
          mbar_arrive(B.bf(2 * (u % half) + gw));
          --npend;
        }
      }
      // Flush at the end of every item: the next item's stages may wait on
      // this item's epilogue, which waits on these stages.
      cp_async_wait<0>();
      fence_proxy_async_smem();
      for (; npend > 0; --npend) {
        const uint32_t u = bcnt - npend;
        mbar_arrive(B.bf(2 * (u % half) + gw));
      }
      if (!ok) break;
      ++icnt;
    }
    cp_async_wait<0>();
  } else if (warp >= kWarpDequant0 && warp < kWarpEpilogue0) {
    // ======================= dequantisation into TMEM =======================
    // Warpgroup g dequantises the k steps with ks % 2 == g; thread r of the
    // warpgroup owns weight row r of the tile, i.e. TMEM lane r.
    const int g = (warp - kWarpDequant0) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t wcnt = 0, acnt = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
      const ItemDesc d = decode_item(args, it, num_blocks, bpe);
      if (d.e < 0) continue;
      for (int st = 0; st < n_wst; ++st, ++wcnt) {
        const int slot = wcnt % WS;
        ok = __all_sync(0xffffffffu, wait_phase(B.wf(slot), (wcnt / WS) & 1, abort_flag, status,
                                                 kWhereDequantW, tmo));
        if (!ok) break;
        const int ks = 2 * st + g;
        if (ks >= args.k_steps) {
          __syncwarp();
          if (lane == 0) mbar_arrive(B.we(slot));
          continue;
        }
        const uint8_t* stp = sm.w_ring + static_cast<size_t>(slot) * kWStageBytes + g * kStepBytes;
        const uint4 q0 = *reinterpret_cast<const uint4*>(stp + r * 16);
        const uint4 q1 = *reinterpret_cast<const uint4*>(stp + 2048 + r * 16);
        const uint32_t s0 = *reinterpret_cast<const uint16_t*>(stp + kStepQBytes + r * 2);
        const uint32_t s1 = *reinterpret_cast<const uint16_t*>(stp + kStepQBytes + 256 + r * 2);
        __syncwarp();
        if (lane == 0) mbar_arrive(B.we(slot));
        uint32_t v[32];
        dequant_group(q0, s0, v);
        dequant_group(q1, s1, v + 16);
        const int aslot = g * SA + static_cast<int>(acnt % SA);
        ok = __all_sync(0xffffffffu, wait_phase(B.ae(aslot), ((acnt / SA) & 1) ^ 1, abort_flag,
                                                 status, kWhereDequantA, tmo));
        if (!ok) break;
        tc_fence_after();
        tmem_st_32x32b_x32(tmem + lane_base + aslot * kAColsPerSlot, v);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B.af(aslot));
        ++acnt;
      }
    }
  } else if (warp >= kWarpEpilogue0) {
    // ======================= epilogue =======================================
    // Thread r owns weight row r of the tile (TMEM lane r): it reads the
    // block's token columns and writes output column tile*128 + r.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t icnt = 0, dcnt = 0;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
      const ItemDesc d = decode_item(args, it, num_blocks, bpe);
      if (d.e < 0) continue;
      const int islot = icnt & 1;
      const int dslot = dcnt % args.d_slots;
      bool ok = wait_phase(B.accf(dslot), (dcnt / args.d_slots) & 1, abort_flag, status,
                           kWhereEpiAcc, tmo) &&
                wait_phase(B.itf(islot), (icnt >> 1) & 1, abort_flag, status, kWhereEpiItem, tmo);
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
          const int dr = idst[j0 + jj];
          if (dr < 0) continue;
          const float x = odd_steps ? __uint_as_float(v[jj]) + __uint_as_float(w[jj])
                                    : __uint_as_float(v[jj]);
          if (args.out_mode == kOutF32WeightedAdd) {
            float* o = static_cast<float*>(args.out) + static_cast<long long>(dr) * args.n + ng;
            atomicAdd(o, iwt[j0 + jj] * x);
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
      ++icnt;
      ++dcnt;
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

size_t gemm_smem_bytes(int block_m, int w_stages, int b_stages) {
  size_t off = 1024;  // alignment slack
  off += static_cast<size_t>(b_stages) * block_m * 128;
  off += static_cast<size_t>(w_stages) * kWStageBytes;
  off += 3 * 4 * static_cast<size_t>(block_m) * 4 + 4 * 4;
  off = (off + 7) / 8 * 8;
  off += (2 * w_stages + 2 * kMaxASlots + 2 * b_stages + 10) * 8;
  off += 8;
  return off;
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
  size_t smem = gemm_smem_bytes(args.block_m, args.w_stages, args.b_stages);
  if (smem < 118 * 1024) smem = 118 * 1024;
  cudaError_t err = cudaFuncSetAttribute(w4a16_moe_gemm_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  w4a16_moe_gemm_kernel<<<grid, kThreads, smem, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace w4a16
