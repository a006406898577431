/*
 * w4a16moe.h -- C ABI of the GB300 (sm_103a) W4A16 INT4 MoE expert GEMM pair.
 *
 * The operator is the Chord/Humming W4A16 MoE expert pair: gate_up, then
 * down, over INT4 group-32 weights with BF16 scales and BF16 activations.
 * Sources (page titles abbreviated):
 *   [P-arex]   "vLLM 宣布 Humming 后端可运行 Novita 开源的 Chord 内核，称 H200 TP8
 *              提速 1.33x、B300 EP8 decode 提速 2.15x" (arex-research)
 *   [P-lens]   "vLLM と Novita AI が Chord をリリース：Kimi K2.x 用の高速 INT4 MoE
 *              カーネル" (agentlenshq)
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer named *_d / a / out / packed / workspace is DEVICE memory
 *   of the current CUDA device, allocated and owned by the caller. The
 *   library allocates no memory and keeps no per-call state.
 * - BF16 tensors are passed as uint16_t bit patterns.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream). Work is enqueued asynchronously; a call returns once it is
 *   enqueued. Unless a flag says otherwise no call synchronises, so calls can
 *   be captured in a CUDA graph (the over-allocated routing buffers make the
 *   grid independent of the routing, [P-lens] "ランタイムの考慮事項").
 * - A pointer to an array of zero elements may be NULL: the activation,
 *   the output and the top-k weights when there are no tokens (m = 0 for
 *   the grouped calls), sorted_ids and expert_ids when the capacity is 0.
 *   num_tokens_padded, the packed weights and the plan are never NULL.
 *   An empty call enqueues nothing that touches them.
 * - Every call validates its arguments on the host before it enqueues
 *   anything and returns a w4a16_status; nothing is enqueued on error.
 *   A failed launch returns W4A16_ERR_CUDA.
 * - All entry points are thread-safe.
 */
#ifndef W4A16MOE_H
#define W4A16MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  W4A16_OK = 0,
  W4A16_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum     */
  W4A16_ERR_UNSUPPORTED = 2,  /* quantisation scheme or shape not handled:
                                 reported at load, never a silent fallback
                                 ([P-arex] "接入方式", [P-lens] "vLLM との統合") */
  W4A16_ERR_ROUTING = 3,      /* routing tensors failed validation         */
  W4A16_ERR_WORKSPACE = 4,    /* workspace missing or too small            */
  W4A16_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed      */
  W4A16_ERR_TIMEOUT = 6       /* a device-side wait gave up (see
                                 w4a16_read_device_status)                 */
} w4a16_status;

/* GEMM modes of the indexed family. */
enum {
  W4A16_GATE_UP = 0,      /* out BF16 [tokens*topk, n]: the gate_up projection   */
  W4A16_DOWN = 1,         /* out FP32 [tokens, n]: weighted scatter-add           */
  W4A16_GATE_UP_SILU = 2  /* gate_up with the activation fused into the epilogue:
                             out BF16 [tokens*topk, n/2] = bf16(silu(g) * u),
                             g, u the BF16-rounded gate and up outputs; weights
                             packed with W4A16_LAYOUT_KTILE64_GLU16 and the plan's
                             layout set to it                                  */
};
/* Grouped families. */
enum { W4A16_GROUPED_CONTIGUOUS = 0, W4A16_GROUPED_MASKED = 1 };
/* Call flags. */
enum {
  W4A16_FLAG_VALIDATE_ROUTING = 1, /* copy the routing tensors to the host and
                                      check them before the launch; this
                                      synchronises `stream` and is therefore
                                      not graph-capturable ([P-lens]
                                      "ランタイムの考慮事項": trusted routing
                                      validation off = capturable)          */
  W4A16_FLAG_ACCUMULATE = 2,       /* DOWN: add into `out` instead of first
                                      zeroing it                            */
  W4A16_FLAG_DETERMINISTIC = 8     /* DOWN: sum each token's top-k rows in a
                                      fixed order (see
                                      w4a16_moe_indexed_gemm)               */
};
/* Packed weight layouts (w4a16_prepack). One layout serves every family. */
enum {
  W4A16_LAYOUT_KTILE64 = 0,      /* 128 consecutive rows per tile                */
  W4A16_LAYOUT_KTILE64_GLU16 = 1 /* gate_up weights [2I, k] with gate rows [0, I)
                                    and up rows [I, 2I): tile t holds, for each
                                    of its four 32-row quarters q, gate rows
                                    64t+16q .. +15 then the matching up rows
                                    I+64t+16q .. +15 (I % 64 == 0), so that the
                                    epilogue pairs them inside one warp        */
};

/* Static description of a status code. Never NULL. */
const char* w4a16_status_string(int status);

/* ABI version of this header (major * 100 + minor). */
int w4a16_version(void);

/*
 * Schedule chosen from the shape and from tok_e, the routed rows per expert
 * ([P-arex] "调度由每个专家收到的 token 数决定": tok_e, not the total token
 * count, decides which schedule wins; [P-lens] "カーネルレベルの最適化").
 */
typedef struct {
  int block_m;     /* routing block rows: the align block size and the
                      largest MMA N of one work item (16..256, step 16)   */
  int bn;          /* weight rows per tile (MMA M) = 128                  */
  int bk;          /* K elements per pipeline step = 64                   */
  int stages;      /* weight ring depth, in stages of 2 K steps (4..16;
                      rounded down to a multiple of 4)                    */
  int b_stages;    /* activation ring depth in K steps, a multiple of 4:
                      8..32 for block_m <= 128 (slots of 2 K steps), 4..32
                      above (slots of 1 K step)                           */
  int split_k;     /* 1 (no split of K)                                   */
  int ctas_per_sm; /* 1 (persistent, one CTA per SM)                      */
  int swap_ab;     /* 1: weights are the MMA M operand, tokens the N one  */
  int layout;      /* W4A16_LAYOUT_KTILE64                                */
  int grid;        /* CTAs to launch; 0 = number of SMs x ctas_per_sm     */
  int cta_pair;    /* 1: pairs of CTAs (2-CTA clusters) each work on 256
                      weight rows, the pair's even CTA issuing M = 256
                      tensor-core MMAs over both CTAs' operands; needs
                      block_m % 32 == 0 and block_m <= 128 (else the plan
                      is refused); used
                      when the weight tile count (n / 128, rounded up) is
                      even, else the call runs unpaired. 0: unpaired      */
} w4a16_plan_t;

/*
 * Fill *out for a GEMM with output width n and reduction length k over
 * `tokens` tokens routed top-`topk` to `num_experts` local experts.
 * tok_e_hint > 0 overrides the expected rows per expert (default
 * tokens * topk / num_experts); it is known on the host without a sync.
 * block_m from tok_e: up to 80, roundup16(1.5 tok_e) within 16..64; then 64
 * below 120, else 128 (256-row blocks are accepted in a plan the caller
 * sets; each call takes routing aligned to its own plan's block_m). Host
 * only. Errors: INVALID_ARG on non-positive sizes or a NULL out.
 */
w4a16_status w4a16_plan(int tokens, int topk, int num_experts, int n, int k,
                        float tok_e_hint, w4a16_plan_t* out);

/*
 * The plan a grouped call (w4a16_moe_grouped_gemm with plan NULL) uses:
 * w4a16_plan with tok_e = expected_m (the masked layout's row budget), else
 * m, and block_m 128 when that tok_e exceeds 80 rows. Host only. Errors:
 * INVALID_ARG on a bad kind, negative m or non-positive n, k.
 */
w4a16_status w4a16_grouped_plan(int kind, int m, int expected_m, int n, int k,
                                w4a16_plan_t* out);

/* What a plan becomes on the device. */
typedef struct {
  int mma_issuers;    /* threads issuing tcgen05.mma, each into its own
                         partial FP32 accumulator (1, 2 or 4; block_m
                         above 128: 4, of which a work item uses 1, 2 or 4
                         by its MMA N, 256 / that many columns each)      */
  int acc_slots;      /* work items whose accumulators TMEM holds at once */
  int acc_cols;       /* TMEM columns of one partial accumulator          */
  int early_epilogue; /* 1: the accumulator slot is freed before the
                         epilogue's global stores                         */
  int w_stages;       /* weight ring, stages of 2 K steps                 */
  int b_stages;       /* activation ring slots: 2 K steps each, 1 K step
                         for block_m above 128                            */
  size_t smem_bytes;  /* dynamic shared memory of one CTA                 */
} w4a16_plan_info_t;

/*
 * Describe a plan for a GEMM of reduction length k (host only). Errors:
 * INVALID_ARG for a NULL pointer, k <= 0, or a plan the GEMM entry points
 * would refuse.
 */
w4a16_status w4a16_plan_info(const w4a16_plan_t* plan, int k, w4a16_plan_info_t* out);

/*
 * Rows to allocate for sorted_ids so that any routing of `numel` rows over
 * `num_experts` experts fits after padding every expert to block_m:
 * roundup(numel + min(num_experts, numel) * (block_m - 1), block_m).
 * expert_ids needs capacity / block_m entries. Host only; 0 on bad input.
 */
size_t w4a16_align_capacity(int numel, int num_experts, int block_m);

/*
 * moe_align_block_size ([P-arex] "调度由每个专家收到的 token 数决定": the
 * indexed kernel consumes sorted_ids / expert_ids / num_tokens_padded).
 *   topk_ids   int32 [tokens, topk] device: local expert id of each routed
 *              row, any value outside [0, num_experts) = not local (skipped).
 *   sorted_ids int32 [capacity] device out: for e ascending, the flattened
 *              rows i = t*topk + k with topk_ids.flat[i] == e in ascending i,
 *              padded with the sentinel tokens*topk to a multiple of block_m;
 *              entries past the padded total also hold the sentinel.
 *   expert_ids int32 [capacity/block_m] device out: expert of each block,
 *              -1 past the padded total.
 *   num_tokens_padded int32 [1] device out: the padded total.
 * capacity must be a multiple of block_m and at least
 * w4a16_align_capacity(tokens*topk, num_experts, block_m), so the output
 * always fits. block_m in [1, 1024]; num_experts in [1, 1024].
 * Deterministic: the result is unique and bit-exact.
 */
w4a16_status w4a16_moe_align_block_size(const int32_t* topk_ids, int tokens, int topk,
                                        int num_experts, int block_m, int capacity,
                                        int32_t* sorted_ids, int32_t* expert_ids,
                                        int32_t* num_tokens_padded, void* stream);

/*
 * Bytes of the packed weights of `num_experts` experts of shape [n, k].
 * Schema ([P-arex] "接入方式"): uint4, group 32, BF16 scales. group must be
 * 32 and k a positive multiple of 32, else W4A16_ERR_UNSUPPORTED; layout
 * must be W4A16_LAYOUT_KTILE64, or W4A16_LAYOUT_KTILE64_GLU16 with n a
 * multiple of 128 (else W4A16_ERR_UNSUPPORTED). Host only.
 */
w4a16_status w4a16_prepack_size(int num_experts, int n, int k, int group, int layout,
                                size_t* bytes);

/*
 * Repack checkpoint weights into the kernel layout (once, at load; the layout
 * is fixed at load, [P-arex] "调度由每个专家收到的 token 数决定").
 *   q       uint8 [num_experts, n, k/2] device: uint4 codes, even k in the
 *           low nibble; the weight is (q - 8) * scale.
 *   scales  BF16 [num_experts, n, k/32] device: one scale per 32 k.
 *   packed  device out, packed_bytes >= w4a16_prepack_size(...), 16-byte
 *           aligned. Opaque: 128-row tiles x 64-k steps, contiguous along k
 *           inside a tile; rows past n and k past k hold zero weights.
 */
w4a16_status w4a16_prepack(const uint8_t* q, const uint16_t* scales, int num_experts, int n,
                           int k, int group, int layout, void* packed, size_t packed_bytes,
                           void* stream);

/* Inverse of w4a16_prepack (for checking a packed blob byte for byte);
 * `layout` is the one the blob was packed with. */
w4a16_status w4a16_unpack(const void* packed, int num_experts, int n, int k, int layout, uint8_t* q,
                          uint16_t* scales, void* stream);

/*
 * Device workspace bytes for a GEMM call under `plan`.
 *   rows: the routing capacity (rows of sorted_ids) of an indexed GEMM, or 0
 *         for a grouped GEMM;
 *   k:    the GEMM's reduction length (columns of its activation rows).
 * Layout: 256 bytes of device status words, then (indexed GEMM) the routed
 * activation rows copied into routing order, rows x roundup(k, 64) BF16.
 * The caller zero-fills a new workspace once; the library keeps the status
 * words zero except when a device-side wait gives up. One workspace serves
 * calls that are ordered on one stream.
 */
size_t w4a16_workspace_size(const w4a16_plan_t* plan, int rows, int k);

/*
 * Extra workspace bytes of a DOWN call with W4A16_FLAG_DETERMINISTIC, placed
 * after the w4a16_workspace_size part: the weighted rows, capacity x n FP32,
 * then the routing position of each of the numel = tokens * topk flattened
 * rows (int32); each part rounded up to 256 bytes. 0 on bad sizes.
 */
size_t w4a16_deterministic_bytes(int capacity, int n, int numel);

/*
 * Indexed W4A16 MoE GEMM ([P-arex] "调度由每个专家收到的 token 数决定",
 * "六个场景的逐层测量与限定条件"; [P-lens] "コア貢献").
 * Weights: `packed` from w4a16_prepack with [num_experts, n, k].
 * For each block b < num_tokens_padded / plan->block_m with expert
 * e = expert_ids[b] in [0, num_experts) and each row i = sorted_ids[...] of
 * the block with i < tokens*topk:
 *   GATE_UP: a = x BF16 [tokens, k]; out BF16 [tokens*topk, n]:
 *            out[i, :] = bf16( x[i / topk, :] . W_e^T ), fp32 accumulation.
 *            Rows of out not routed to a local expert are left untouched.
 *   DOWN:    a = activation BF16 [tokens*topk, k] (rows by flattened id);
 *            topk_weights fp32 [tokens, topk]; out fp32 [tokens, n]:
 *            out[i / topk, :] += topk_weights.flat[i] * ( a[i, :] . W_e^T ).
 *            `out` is zeroed first unless W4A16_FLAG_ACCUMULATE. Summation
 *            order across the top-k rows of a token is not fixed, unless
 *            W4A16_FLAG_DETERMINISTIC: then the GEMM stores every weighted
 *            row (FP32) in the workspace and a second kernel sets
 *            out[t, :] (+)= the sum of token t's rows in ascending top-k
 *            slot order, so the result does not depend on the grid, the
 *            block size or the timing. That needs ws_bytes >=
 *            w4a16_workspace_size(plan, capacity, k) +
 *            w4a16_deterministic_bytes(capacity, n, tokens * topk).
 *   GATE_UP_SILU: as GATE_UP with n = 2*inter (gate rows, then up rows), but
 *            out BF16 [tokens*topk, n/2] receives
 *            bf16( silu(g) * u ), g = bf16(x . Wgate^T), u = bf16(x . Wup^T),
 *            silu(g) as in w4a16_silu_and_mul: the same values as GATE_UP
 *            followed by w4a16_silu_and_mul, in one pass (the activation is
 *            this library's reading, see w4a16_silu_and_mul). Requires
 *            packed with W4A16_LAYOUT_KTILE64_GLU16, plan->layout equal to
 *            it, and n % 128 == 0.
 * The routing buffers may be over-allocated (capacity rows); the grid does
 * not depend on their contents. Blocks with expert -1 and sentinel rows are
 * skipped; ids out of range are ignored, never dereferenced.
 * Requires: k % 32 == 0, n >= 1, plan from w4a16_plan (block_m equal to the
 * align block size, 16..256 step 16), ws_bytes >=
 * w4a16_workspace_size(plan, capacity, k), a, out 16-byte aligned.
 * The call first copies the routed rows of `a` into routing order in the
 * workspace (one extra kernel on `stream`), then runs the GEMM on them.
 */
w4a16_status w4a16_moe_indexed_gemm(int mode, const void* packed, int num_experts, int n, int k,
                                    const uint16_t* a, int tokens, int topk,
                                    const int32_t* sorted_ids, const int32_t* expert_ids,
                                    const int32_t* num_tokens_padded, int capacity,
                                    const float* topk_weights, void* out, int flags,
                                    const w4a16_plan_t* plan, void* workspace, size_t ws_bytes,
                                    void* stream);

/*
 * Grouped W4A16 MoE GEMM ([P-lens] "グループ化 SM90 カーネル技術").
 *   CONTIGUOUS: a BF16 [m, k] with each expert's rows padded to a multiple
 *     of 128 rows; layout = m_expert int32 [m], the expert of every row or
 *     -1 for padding; every aligned 128-row block holds rows of one expert.
 *     out BF16 [m, n]: out[r] = bf16(a[r] . W_{m_expert[r]}^T) for valid r.
 *     m must be a multiple of plan->block_m, which must divide 128.
 *   MASKED: a BF16 [num_experts, m, k] (m = the fixed row budget max_m);
 *     layout = masked_m int32 [num_experts]; out BF16 [num_experts, m, n]:
 *     rows r < masked_m[e] of expert e get bf16(a[e, r] . W_e^T).
 * Padding rows of out are left untouched. expected_m is the expected rows
 * per expert (schedule hint only).
 */
w4a16_status w4a16_moe_grouped_gemm(int kind, const void* packed, int num_experts, int n, int k,
                                    const uint16_t* a, int m, const int32_t* layout,
                                    int expected_m, uint16_t* out, int flags,
                                    const w4a16_plan_t* plan, void* workspace, size_t ws_bytes,
                                    void* stream);

/* Element types of w4a16_topk_softmax's logits. */
enum { W4A16_DTYPE_F32 = 0, W4A16_DTYPE_BF16 = 1 };

/*
 * Routing front end: router logits -> the top-k routing tensors the align
 * and the GEMMs consume. The pages route each token to the top 8 of 384
 * experts and hand the operator the serving stack's routing tensors
 * ([P-arex] "调度由每个专家收到的 token 数决定"); the router is this library's
 * reading:
 *   p = softmax(logits[t, :]) over all num_experts experts (FP32);
 *   the topk experts with the largest logits are chosen, larger first, ties
 *   to the lower expert id (the logit decides, exactly);
 *   topk_weights[t, s] = p of choice s, divided by the sum of the chosen p
 *   when `renormalize` != 0;
 *   topk_ids[t, s] = choice s - expert_offset when that lies in
 *   [0, num_local_experts) (an expert of this GPU), else -1.
 * logits: device [tokens, num_experts] of logits_dtype; topk_ids int32 and
 * topk_weights fp32 [tokens, topk], device. num_experts <= 1024, topk <= 32
 * (W4A16_ERR_UNSUPPORTED beyond). No host synchronisation: graph-capturable.
 */
w4a16_status w4a16_topk_softmax(const void* logits, int logits_dtype, int tokens,
                                int num_experts, int topk, int renormalize, int expert_offset,
                                int num_local_experts, int32_t* topk_ids, float* topk_weights,
                                void* stream);

/*
 * The routing front end in ONE launch: w4a16_topk_softmax followed by
 * w4a16_moe_align_block_size over its topk_ids (num_experts of the align =
 * num_local_experts). Every CTA routes a share of the tokens; the CTA that
 * finishes last (it counts arrivals in `arrivals`; no CTA waits on another)
 * then runs the alignment. Outputs are bit-identical to the two calls.
 *   arrivals  uint32 [1] device: zero before the first call (e.g. cudaMemset
 *             once at allocation); each call leaves it zero. Calls that may
 *             run at the same time need separate counters.
 * Other arguments as w4a16_topk_softmax and w4a16_moe_align_block_size
 * (sentinel tokens*topk; capacity a multiple of block_m and at least
 * w4a16_align_capacity(tokens*topk, num_local_experts, block_m)).
 * num_local_experts in [1, 1024], block_m in [1, 1024]. No host
 * synchronisation: graph-capturable.
 */
w4a16_status w4a16_moe_route_align(const void* logits, int logits_dtype, int tokens,
                                   int num_experts, int topk, int renormalize, int expert_offset,
                                   int num_local_experts, int block_m, int capacity,
                                   int32_t* topk_ids, float* topk_weights, int32_t* sorted_ids,
                                   int32_t* expert_ids, int32_t* num_tokens_padded,
                                   uint32_t* arrivals, void* stream);

/*
 * Activation between gate_up and down (the pages leave it out of the timed
 * pair, [P-arex] "六个场景的逐层测量与限定条件"; its form is this library's
 * reading): in BF16 [rows, 2*inter] = [gate | up]; out BF16 [rows, inter]
 * = bf16(silu(gate) * up) with silu(g) = g / (1 + e^-g), computed in fp32
 * with the fast exponential and division (a few fp32 ulps before the BF16
 * rounding). inter % 8 == 0.
 */
w4a16_status w4a16_silu_and_mul(const uint16_t* in, int rows, int inter, uint16_t* out,
                                void* stream);

/*
 * Synchronise `stream`, read the device status word of `workspace`, reset it
 * to zero, and return W4A16_OK or W4A16_ERR_TIMEOUT (a device-side wait of a
 * GEMM gave up after about a second; the kernel then ended early and its
 * output is incomplete). *detail (optional) receives the raw word:
 * 0x1000 | code of the wait that gave up.
 * The bound, in SM clock cycles, is read from the environment variable
 * W4A16_WAIT_TIMEOUT_CYCLES at each GEMM call (default 2e9); lowering it
 * makes the failure path testable without any GPU fault.
 */
w4a16_status w4a16_read_device_status(void* workspace, int* detail, void* stream);

/*
 * Device workspace bytes of w4a16_moe_layer: 256 bytes of status words, the
 * x rows in routing order (rows x roundup(hidden, 64) BF16), the activation
 * rows in routing order (rows x inter BF16), one int32 completion counter per
 * routing block; each part rounded up to 256 bytes. rows = the routing
 * capacity.
 */
size_t w4a16_layer_workspace_size(const w4a16_plan_t* plan, int rows, int hidden, int inter);

/*
 * The whole expert pair of one MoE layer in a single GEMM launch: gate_up
 * with the activation fused (W4A16_GATE_UP_SILU), then down with the top-k
 * weighted scatter-add (W4A16_DOWN), over the same routing blocks ([P-arex]
 * "调度由每个专家收到的 token 数决定": gate_up then down over sorted_ids /
 * expert_ids / num_tokens_padded; the activation between them is the glue the
 * pages leave out of the timed pair).
 *   packed_gate_up  [num_experts, 2*inter, hidden] packed with
 *                   W4A16_LAYOUT_KTILE64_GLU16 (plan->layout must say so);
 *   packed_down     [num_experts, hidden, inter] packed with
 *                   W4A16_LAYOUT_KTILE64;
 *   x               BF16 [tokens, hidden]; topk_weights fp32 [tokens, topk];
 *   out             FP32 [tokens, hidden]: zeroed first unless
 *                   W4A16_FLAG_ACCUMULATE, then every token's top-k weighted
 *                   down rows are added (in no fixed order).
 * One persistent launch runs every gate_up work item, then every down work
 * item; the down items of a routing block start once all gate_up items of the
 * block (on any CTA) have written its activation rows to the workspace (a
 * per-block counter in device memory, polled with a bounded wait). The
 * result equals w4a16_moe_indexed_gemm(W4A16_GATE_UP_SILU) followed by
 * w4a16_moe_indexed_gemm(W4A16_DOWN) up to the order of the FP32 additions.
 * Requirements: inter % 64 == 0, hidden % 32 == 0 and hidden % 4 == 0
 * (else W4A16_ERR_UNSUPPORTED); plan->cta_pair == 0 and plan->block_m <= 128
 * (else W4A16_ERR_INVALID_ARG); flags
 * VALIDATE_ROUTING and ACCUMULATE only (else W4A16_ERR_INVALID_ARG); ws_bytes
 * >= w4a16_layer_workspace_size(plan, capacity, hidden, inter) (else
 * W4A16_ERR_WORKSPACE). Every CTA of the launch must be resident at once (it
 * uses at most one CTA per SM); if the device is shared so that some cannot
 * start, the waits run out and w4a16_read_device_status reports
 * W4A16_ERR_TIMEOUT.
 */
w4a16_status w4a16_moe_layer(const void* packed_gate_up, const void* packed_down, int num_experts,
                             int hidden, int inter, const uint16_t* x, int tokens, int topk,
                             const int32_t* sorted_ids, const int32_t* expert_ids,
                             const int32_t* num_tokens_padded, int capacity,
                             const float* topk_weights, float* out, int flags,
                             const w4a16_plan_t* plan, void* workspace, size_t ws_bytes,
                             void* stream);

/*
 * No-allocation variant of w4a16_moe_indexed_gemm. The pages have no
 * counterpart of this call; it exists for callers that cannot allocate
 * device memory when they call the operator: a host whose caching allocator
 * owns all device memory and hands out no raw buffers, code that must not
 * allocate after start-up (cudaMalloc/cudaFree may synchronise the device
 * and take a global lock), or a plugin interface that passes only the
 * operation's tensors.
 * Same arguments and results as w4a16_moe_indexed_gemm, without the
 * workspace: the library uses a fixed 32 MiB array of device memory compiled
 * into it, which every GPU that loads the library holds until the process
 * exits. The call allocates nothing. The caller still provides every input
 * and output buffer.
 * - Returns W4A16_ERR_WORKSPACE if w4a16_workspace_size(plan, capacity, k)
 *   exceeds 32 MiB (for k = 7168 that is a routing capacity above 2340
 *   rows).
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current), and so does the first
 *   call after the device's context changed (cudaDeviceReset); make that
 *   first call before any stream capture begins.
 * - Every call on a device shares the array. Once every argument check has
 *   passed, the call clears the array's status word on `stream`, then
 *   launches; a refused call enqueues nothing. Calls that overlap on the GPU
 *   (different streams without ordering) race on the array: order them, or
 *   use w4a16_moe_indexed_gemm with one workspace per stream.
 * - flags: those of w4a16_moe_indexed_gemm except W4A16_FLAG_DETERMINISTIC
 *   (refused with W4A16_ERR_INVALID_ARG: its row buffer needs a workspace
 *   sized by the caller), plus W4A16_FLAG_SYNC_STATUS to synchronise
 *   `stream` after the launch and return W4A16_ERR_TIMEOUT if a device-side
 *   wait gave up (without it such a failure is not reported).
 */
enum { W4A16_FLAG_SYNC_STATUS = 4 };
w4a16_status w4a16_moe_indexed_gemm_noalloc(int mode, const void* packed, int num_experts, int n,
                                            int k, const uint16_t* a, int tokens, int topk,
                                            const int32_t* sorted_ids, const int32_t* expert_ids,
                                            const int32_t* num_tokens_padded, int capacity,
                                            const float* topk_weights, void* out, int flags,
                                            const w4a16_plan_t* plan, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16MOE_H */
