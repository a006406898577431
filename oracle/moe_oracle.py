"""Plain float64 CPU oracle of the W4A16 INT4 MoE expert GEMM pair.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product
path imports this module, and it imports nothing from the product package.

What the method computes, restated from the pages (titles abbreviated):

* Weight format -- page "vLLM 宣布 Humming 后端可运行 … Chord 内核 …"
  (arex-research), section "接入方式：用 Chord 替代公共 Humming 包": the schema
  is uint4 weights in groups of 32 along K with one BF16 scale per group, as in
  the compressed-tensors pack-quantized INT4 group-32 checkpoints. Reading
  taken here (the pages name no zero point and no nibble order): the uint4 code
  q carries the implicit zero point 8, so w = (q - 8) * s; two codes share a
  byte, the even k in the low nibble.
* Routing interface -- same page, section "调度由每个专家收到的 token 数决定":
  the indexed kernel consumes vLLM's ``sorted_ids / expert_ids /
  num_tokens_padded``; page "vLLM と Novita AI が Chord をリリース …"
  (agentlenshq), section "ランタイムの考慮事項": those buffers are
  over-allocated.
* The pair -- arex-research page, section "六个场景的逐层测量与限定条件": one
  layer is the gate_up GEMM followed by the down GEMM (routing, activation and
  communication sit outside the timed pair). The top-k weights are applied in
  the down pass, which sums each token's expert outputs.
* Grouped families -- agentlenshq page, section "グループ化 SM90 カーネル技術":
  contiguous prefill pads every expert to a 128-row boundary; masked decode
  gives every expert a fixed row budget of which the first ``masked_m[e]``
  rows are real.

Every floating-point step is evaluated in float64. Activations and scales are
BF16 inputs and are decoded exactly. A BF16 output of the method (the gate_up
result and the activation result) is rounded to BF16 with round-to-nearest-
even, because that is the type of the tensor that crosses the boundary.
"""

from __future__ import annotations

import numpy as np

GROUP_SIZE = 32   # K elements sharing one BF16 scale (uint4 group-32 schema)
ZERO_POINT = 8    # implicit zero point of the uint4 code (reading, see above)


# --------------------------------------------------------------------------
# BF16 <-> float64
# --------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode BF16 bit patterns (uint16) exactly: a BF16 is the top half of
    an IEEE binary32, so the bits shifted left by 16 are that float32."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest BF16 value, ties to even.

    BF16 keeps 8 significant bits. With x = m * 2**e (0.5 <= |m| < 1), the
    spacing of BF16 numbers around x is 2**(e - 8); below the smallest normal
    (2**-126, i.e. e = -125) the spacing stays 2**-133 (subnormals). Values
    past the largest finite BF16 after rounding become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    fin = np.isfinite(x)
    xf = x[fin]
    _, e = np.frexp(xf)
    e = np.maximum(e, -125)
    scale = np.ldexp(np.ones_like(xf), 8 - e)   # exact powers of two
    r = np.rint(xf * scale) / scale              # np.rint rounds half to even
    max_bf16 = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > max_bf16, np.copysign(np.inf, r), r)
    out[fin] = r
    return out


def f64_to_bf16_bits(x) -> np.ndarray:
    """float64 -> BF16 bit patterns (uint16), round-to-nearest-even; NaN maps
    to the canonical quiet NaN 0x7FC0."""
    r = round_to_bf16(x)
    bits = (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = np.where(np.isnan(r), np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


# --------------------------------------------------------------------------
# Weight format
# --------------------------------------------------------------------------

def unpack_codes(q_packed) -> np.ndarray:
    """uint8 [..., K/2] -> uint4 codes [..., K]; byte j holds k = 2j in its
    low nibble and k = 2j + 1 in its high nibble."""
    q = np.asarray(q_packed, dtype=np.uint8)
    codes = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.uint8)
    codes[..., 0::2] = q & np.uint8(0x0F)
    codes[..., 1::2] = q >> np.uint8(4)
    return codes


def dequant_weights(q_packed, scales_bits) -> np.ndarray:
    """W[..., n, k] = (q[..., n, k] - 8) * s[..., n, k // 32], in float64.

    The product of a 4-bit integer and a BF16 scale is exact in float64."""
    codes = unpack_codes(q_packed).astype(np.float64)
    s = bf16_bits_to_f64(scales_bits)
    k = codes.shape[-1]
    if s.shape[-1] * GROUP_SIZE != k:
        raise ValueError("scales must hold one entry per group of 32 along K")
    return (codes - ZERO_POINT) * np.repeat(s, GROUP_SIZE, axis=-1)


def _expert_weights(q_packed, scales_bits, e, cols):
    """Dequantised W_e restricted to the output rows ``cols`` (all if None)."""
    if cols is None:
        return dequant_weights(q_packed[e], scales_bits[e])
    cols = np.asarray(cols)
    return dequant_weights(q_packed[e][cols], scales_bits[e][cols])


# --------------------------------------------------------------------------
# Routing alignment (moe_align_block_size)
# --------------------------------------------------------------------------

def moe_align_block_size(topk_ids, num_experts: int, block_m: int, capacity: int):
    """Group the flattened routed rows i = t * topk + k by expert.

    For e = 0 .. E-1 in ascending order, the rows i with topk_ids.flat[i] == e
    are listed in ascending i, then padded with the sentinel T * topk up to a
    multiple of ``block_m``; every block of ``block_m`` entries gets its expert
    id. Ids outside [0, E) (non-local experts, -1) are skipped. Experts with no
    rows get no block. The buffers are over-allocated to ``capacity`` rows:
    unused tail entries hold the sentinel in ``sorted_ids`` and -1 in
    ``expert_ids``. ``num_tokens_padded`` is the padded total.

    Returns (sorted_ids int32 [capacity], expert_ids int32 [capacity/block_m],
    num_tokens_padded int32 [1]).
    """
    flat = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    numel = flat.size
    if block_m <= 0 or capacity % block_m != 0:
        raise ValueError("capacity must be a positive multiple of block_m")
    sentinel = numel
    sorted_parts, expert_parts = [], []
    for e in range(num_experts):
        rows = np.nonzero(flat == e)[0]
        if rows.size == 0:
            continue
        padded = -(-rows.size // block_m) * block_m
        sorted_parts.append(rows)
        sorted_parts.append(np.full(padded - rows.size, sentinel, dtype=np.int64))
        expert_parts.append(np.full(padded // block_m, e, dtype=np.int64))
    body = np.concatenate(sorted_parts) if sorted_parts else np.zeros(0, np.int64)
    blocks = np.concatenate(expert_parts) if expert_parts else np.zeros(0, np.int64)
    total = body.size
    if total > capacity:
        raise ValueError("capacity too small for the padded routing")
    sorted_ids = np.full(capacity, sentinel, dtype=np.int32)
    sorted_ids[:total] = body
    expert_ids = np.full(capacity // block_m, -1, dtype=np.int32)
    expert_ids[: blocks.size] = blocks
    return sorted_ids, expert_ids, np.array([total], dtype=np.int32)


# --------------------------------------------------------------------------
# The GEMM pair
# --------------------------------------------------------------------------

def indexed_gate_up(x_bits, topk_ids, q_packed, scales_bits, cols=None) -> np.ndarray:
    """gate_up over routed rows: G[i, n] = sum_k x[i // topk, k] * W_e[n, k]
    for every flattened row i routed to a local expert e = topk_ids.flat[i].

    x_bits: BF16 [T, K]; weights [E, N, K/2] + scales [E, N, K/32].
    Returns float64 [T * topk, len(cols) or N], unrounded; rows not routed to
    a local expert are NaN.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    topk = ids.shape[1]
    flat = ids.reshape(-1)
    num_experts = q_packed.shape[0]
    x = bf16_bits_to_f64(x_bits)
    ncols = q_packed.shape[1] if cols is None else len(cols)
    g = np.full((flat.size, ncols), np.nan)
    for e in range(num_experts):
        rows = np.nonzero(flat == e)[0]
        if rows.size == 0:
            continue
        w = _expert_weights(q_packed, scales_bits, e, cols)
        g[rows] = x[rows // topk] @ w.T
    return g


def silu_and_mul(g_bits) -> np.ndarray:
    """Activation between the two GEMMs (its form is a reading; the pages
    leave it out of the timed pair): with G = [gate | up] split in halves
    along the feature axis, A = bf16(silu(gate) * up), silu(g) = g / (1 + e^-g).
    Input and output are BF16 bit patterns."""
    g = bf16_bits_to_f64(g_bits)
    half = g.shape[-1] // 2
    gate, up = g[..., :half], g[..., half:]
    with np.errstate(over="ignore", invalid="ignore"):
        a = gate / (1.0 + np.exp(-gate)) * up
    return f64_to_bf16_bits(a)


def indexed_down(a_bits, topk_ids, topk_weights, q_packed, scales_bits, cols=None) -> np.ndarray:
    """down with the top-k weighted sum:
    Y[t, n] = sum over k with a local expert e = topk_ids[t, k] of
              topk_weights[t, k] * sum_j A[t * topk + k, j] * W_e[n, j].

    a_bits: BF16 [T * topk, I] indexed by flattened row. Returns float64
    [T, len(cols) or N]; tokens with no local expert get 0.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    tokens, topk = ids.shape
    flat = ids.reshape(-1)
    wts = np.asarray(topk_weights, dtype=np.float32).astype(np.float64).reshape(-1)
    num_experts = q_packed.shape[0]
    a = bf16_bits_to_f64(a_bits)
    ncols = q_packed.shape[1] if cols is None else len(cols)
    y = np.zeros((tokens, ncols))
    for e in range(num_experts):
        rows = np.nonzero(flat == e)[0]
        if rows.size == 0:
            continue
        w = _expert_weights(q_packed, scales_bits, e, cols)
        contrib = wts[rows, None] * (a[rows] @ w.T)
        np.add.at(y, rows // topk, contrib)
    return y


def grouped_contiguous(a_bits, m_expert, q_packed, scales_bits, cols=None) -> np.ndarray:
    """Contiguous grouped GEMM: C[r, n] = sum_k A[r, k] * W_{m_expert[r]}[n, k]
    for every row r with m_expert[r] in [0, E); padding rows (-1) are NaN."""
    m_expert = np.asarray(m_expert, dtype=np.int64)
    num_experts = q_packed.shape[0]
    a = bf16_bits_to_f64(a_bits)
    ncols = q_packed.shape[1] if cols is None else len(cols)
    c = np.full((a.shape[0], ncols), np.nan)
    for e in range(num_experts):
        rows = np.nonzero(m_expert == e)[0]
        if rows.size == 0:
            continue
        w = _expert_weights(q_packed, scales_bits, e, cols)
        c[rows] = a[rows] @ w.T
    return c


def grouped_masked(a_bits, masked_m, q_packed, scales_bits, cols=None) -> np.ndarray:
    """Masked grouped GEMM over a fixed per-expert row budget:
    C[e, r, n] = sum_k A[e, r, k] * W_e[n, k] for r < masked_m[e]; rows past
    masked_m[e] are NaN."""
    masked_m = np.asarray(masked_m, dtype=np.int64)
    a = bf16_bits_to_f64(a_bits)
    num_experts, max_m = a.shape[0], a.shape[1]
    ncols = q_packed.shape[1] if cols is None else len(cols)
    c = np.full((num_experts, max_m, ncols), np.nan)
    for e in range(num_experts):
        m = int(min(max(masked_m[e], 0), max_m))
        if m == 0:
            continue
        w = _expert_weights(q_packed, scales_bits, e, cols)
        c[e, :m] = a[e, :m] @ w.T
    return c


def moe_layer(x_bits, topk_ids, topk_weights, q_gu, s_gu, q_dn, s_dn):
    """The whole pair: gate_up -> BF16 -> silu_and_mul -> down with the top-k
    weighted sum. Returns (G float64, G BF16 bits, A BF16 bits, Y float64)."""
    g = indexed_gate_up(x_bits, topk_ids, q_gu, s_gu)
    g_bits = f64_to_bf16_bits(np.nan_to_num(g, nan=0.0))
    a_bits = silu_and_mul(g_bits)
    y = indexed_down(a_bits, topk_ids, topk_weights, q_dn, s_dn)
    return g, g_bits, a_bits, y


def topk_softmax(logits, topk: int, renormalize: bool = True, expert_offset: int = 0,
                 num_local_experts=None):
    """Routing front end: softmax over the global experts, top-k, local ids.

    Reading (the pages route top-8 of 384 experts but leave the router to
    the serving stack; the workloads draw softmax weights renormalised over
    the chosen k):
    * p = softmax(logits) over all experts, in float64;
    * the k experts with the largest logits are chosen, larger first, ties
      to the lower expert id. The logit decides, not p, so the choice is made
      on the input values themselves;
    * weights = p of the chosen experts, divided by their sum if `renormalize`;
    * ids become local: g - expert_offset when that lies in
      [0, num_local_experts), else -1 (an expert of another GPU);
    * an expert whose logit is -inf is masked: it is never chosen (its
      softmax probability is 0). When fewer than k experts can be chosen, the
      remaining slots hold id -1 and weight 0.

    logits float [T, E]. Returns (ids int32 [T, k], weights float64 [T, k])."""
    lg = np.asarray(logits, dtype=np.float64)
    t, e = lg.shape
    if num_local_experts is None:
        num_local_experts = e
    ids = np.full((t, topk), -1, dtype=np.int32)
    w = np.zeros((t, topk), dtype=np.float64)
    for i in range(t):
        row = lg[i]
        cand = np.flatnonzero(row > -np.inf)              # the experts that can be chosen
        if cand.size == 0:
            continue
        p = np.where(row > -np.inf, np.exp(row - row[cand].max()), 0.0)
        p /= p.sum()
        order = cand[np.lexsort((cand, -row[cand]))][:topk]   # by logit desc, then id asc
        sel = p[order]
        if renormalize:
            sel = sel / sel.sum()
        loc = order - expert_offset
        n = order.size
        ids[i, :n] = np.where((loc >= 0) & (loc < num_local_experts), loc, -1)
        w[i, :n] = sel
    return ids, w
