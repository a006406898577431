"""Seeded synthetic workloads for the W4A16 INT4 MoE expert GEMM pair.

This module only draws random inputs. It holds none of the method's
arithmetic (no dequantisation, no GEMM, no routing alignment), so both the
CUDA path and the CPU oracle can be fed from it. It imports neither.

Shapes follow the Kimi K2.x shard shapes that the Chord/Humming pages measure
(page "vLLM 宣布 Humming 后端可运行 … Chord 内核 …", sections
"六个场景的逐层测量与限定条件" and "调度由每个专家收到的 token 数决定"):
hidden 7168, moe_intermediate 2048, 384 global experts, top-8; EP8 keeps 48
experts per GPU, TP8 keeps all 384 with the intermediate split by 8.

Value recipe (shared by every workload):
* uint4 codes q ~ U{0..15}, packed two per byte (even k in the low nibble):
  a uniform random byte is two independent uniform codes;
* BF16 group-32 scales s = bf16(|N(0,1)| * 0.02);
* BF16 activations x ~ N(0,1);
* top-k weights: softmax of N(0,1) logits over the token's k slots.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

GROUP = 32


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> BF16 bit patterns (uint16), via torch's conversion."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def random_weights(rng: np.random.Generator, num_experts: int, n: int, k: int):
    """(q uint8 [E, n, k/2], scales BF16 bits uint16 [E, n, k/32])."""
    q = rng.integers(0, 256, size=(num_experts, n, k // 2), dtype=np.uint8)
    s = np.abs(rng.standard_normal((num_experts, n, k // GROUP), dtype=np.float32)) * np.float32(0.02)
    return q, to_bf16_bits(s)


def random_activations(rng: np.random.Generator, *shape: int) -> np.ndarray:
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def softmax_weights(rng: np.random.Generator, tokens: int, topk: int) -> np.ndarray:
    logits = rng.standard_normal((tokens, topk))
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    return (w / w.sum(axis=1, keepdims=True)).astype(np.float32)


@dataclass
class MoEProblem:
    """One layer of routed tokens: inputs of the gate_up / down pair."""
    name: str
    tokens: int
    hidden: int
    inter: int
    num_experts: int          # local experts held by this GPU
    topk: int
    x: np.ndarray             # BF16 bits [T, hidden]
    topk_ids: np.ndarray      # int32 [T, topk], local expert id or -1
    topk_weights: np.ndarray  # float32 [T, topk]
    q_gu: np.ndarray          # uint8 [E, 2*inter, hidden/2]
    s_gu: np.ndarray          # BF16 bits [E, 2*inter, hidden/32]
    q_dn: np.ndarray          # uint8 [E, hidden, inter/2]
    s_dn: np.ndarray          # BF16 bits [E, hidden, inter/32]
    meta: dict = field(default_factory=dict)

    @property
    def numel(self) -> int:
        return self.tokens * self.topk

    def routed_rows(self) -> int:
        ids = self.topk_ids
        return int(((ids >= 0) & (ids < self.num_experts)).sum())

    def tok_e_hint(self) -> float:
        """Expected routed rows per local expert, known without a device sync."""
        return self.routed_rows() / max(1, self.num_experts)


def _uniform_topk(rng, tokens, num_experts, topk):
    keys = rng.random((tokens, num_experts))
    return np.argsort(keys, axis=1)[:, :topk].astype(np.int32)


def _place_local_picks(rng, tokens, topk, per_expert_tokens):
    """Scatter each expert's token list into random free slots of the tokens'
    top-k rows; every other slot is a non-local expert (-1 in the local view)."""
    ids = np.full((tokens, topk), -1, dtype=np.int32)
    fill = np.zeros(tokens, dtype=np.int64)
    for e, toks in enumerate(per_expert_tokens):
        for t in toks:
            ids[t, fill[t]] = e
            fill[t] += 1
    for t in range(tokens):           # random slot order per token
        ids[t] = ids[t, rng.permutation(topk)]
    return ids


def _draw_expert_tokens(rng, tokens, topk, counts):
    """Each expert draws counts[e] distinct tokens; a token may hold at most
    topk local experts, otherwise the draw is repeated."""
    while True:
        lists = [rng.choice(tokens, size=int(c), replace=False) for c in counts]
        per_token = np.bincount(np.concatenate(lists), minlength=tokens) if lists else np.zeros(tokens)
        if per_token.max(initial=0) <= topk:
            return lists


def make_problem(name, rng, tokens, hidden, inter, num_experts, topk, topk_ids, meta=None,
                 weights=True):
    """weights=False leaves the four weight arrays None (routing and
    activations only, for callers that draw the weights elsewhere)."""
    q_gu = s_gu = q_dn = s_dn = None
    if weights:
        q_gu, s_gu = random_weights(rng, num_experts, 2 * inter, hidden)
        q_dn, s_dn = random_weights(rng, num_experts, hidden, inter)
    x = random_activations(rng, tokens, hidden)
    w = softmax_weights(rng, tokens, topk)
    return MoEProblem(name, tokens, hidden, inter, num_experts, topk, x,
                      np.ascontiguousarray(topk_ids, dtype=np.int32), w,
                      q_gu, s_gu, q_dn, s_dn, meta or {})


def uniform_problem(tokens, hidden, inter, num_experts, topk, seed=0, name=None, weights=True):
    """Top-k uniform-random routing over all (local) experts."""
    rng = np.random.default_rng(seed)
    ids = _uniform_topk(rng, tokens, num_experts, topk)
    return make_problem(name or f"uniform_T{tokens}_H{hidden}_I{inter}_E{num_experts}_k{topk}",
                        rng, tokens, hidden, inter, num_experts, topk, ids, weights=weights)


def tiny(seed=0):
    """Tiny: T=64, hidden 512, 8 experts, top-2, intermediate 512."""
    return uniform_problem(64, 512, 512, 8, 2, seed, name="tiny_T64_H512_I512_E8_top2")


def ep8_decode(seed=0, tokens=576, hidden=7168, inter=2048, local_experts=48, topk=8,
               weights=True):
    """EP8 decode shard: 48 local experts of 384, 576 routed local rows with
    tokens-per-expert U{9..15} (corrected to sum to 576)."""
    rng = np.random.default_rng(seed)
    counts = rng.integers(9, 16, size=local_experts)
    target = tokens
    while counts.sum() != target:
        e = rng.integers(local_experts)
        if counts.sum() < target and counts[e] < 15:
            counts[e] += 1
        elif counts.sum() > target and counts[e] > 9:
            counts[e] -= 1
    lists = _draw_expert_tokens(rng, tokens, topk, counts)
    ids = _place_local_picks(rng, tokens, topk, lists)
    return make_problem(f"ep8_decode_T{tokens}_H{hidden}_I{inter}_E{local_experts}_top{topk}",
                        rng, tokens, hidden, inter, local_experts, topk, ids,
                        {"tok_e": counts.tolist()}, weights=weights)


def tp8(tokens, seed=0, hidden=7168, inter_shard=256, experts=384, topk=8, weights=True):
    """TP8 single-instance shard: all 384 experts, intermediate 2048/8."""
    p = uniform_problem(tokens, hidden, inter_shard, experts, topk, seed,
                        name=f"tp8_T{tokens}_H{hidden}_I{inter_shard}_E{experts}_top{topk}",
                        weights=weights)
    return p


def ep8_prefill_counts(local_experts=48, seed=0, scale=1):
    """tok_e for the skewed prefill shard: scale * round(600 * (1 + 0.447 e)^-1.1),
    randomly permuted (600 .. 20 rows, 3904 in total, at scale 1)."""
    rng = np.random.default_rng(seed)
    e = np.arange(local_experts)
    counts = np.round(600.0 * (1.0 + 0.447 * e) ** -1.1).astype(np.int64) * scale
    return counts[rng.permutation(local_experts)]


def ep8_prefill(seed=0, tokens=8192, hidden=7168, inter=2048, local_experts=48, topk=8,
                weights=True, scale=1):
    """The skewed EP8 prefill shard; scale multiplies the tokens and every
    expert's rows (scale 4: T = 32768, tok_e 80 .. 2400, mean 325)."""
    rng = np.random.default_rng(seed)
    tokens = tokens * scale
    counts = ep8_prefill_counts(local_experts, seed, scale)
    lists = _draw_expert_tokens(rng, tokens, topk, counts)
    ids = _place_local_picks(rng, tokens, topk, lists)
    return make_problem(f"ep8_prefill_T{tokens}_H{hidden}_I{inter}_E{local_experts}_top{topk}",
                        rng, tokens, hidden, inter, local_experts, topk, ids,
                        {"tok_e": counts.tolist()}, weights=weights)


@dataclass
class GroupedProblem:
    """Inputs of one grouped GEMM (gate_up shapes: K = hidden, N = 2*inter)."""
    name: str
    kind: str                 # "contiguous" | "masked"
    num_experts: int
    n: int
    k: int
    a: np.ndarray             # BF16 bits: [M_pad, k] (contiguous) or [E, max_m, k] (masked)
    layout: np.ndarray        # int32: m_expert [M_pad] or masked_m [E]
    q: np.ndarray
    s: np.ndarray
    expected_m: int = 0

    def valid_rows(self) -> int:
        if self.kind == "contiguous":
            return int((self.layout >= 0).sum())
        return int(np.minimum(self.layout, self.a.shape[1]).clip(min=0).sum())


def grouped_contiguous_problem(rows_per_expert, num_experts=48, n=4096, k=7168, seed=0,
                               align=128, name=None):
    """Contiguous layout: each expert's rows, padded up to a multiple of
    ``align`` rows with m_expert = -1. ``rows_per_expert`` is an int (all
    experts equal) or a sequence."""
    rng = np.random.default_rng(seed)
    if np.isscalar(rows_per_expert):
        m_e = np.full(num_experts, int(rows_per_expert), dtype=np.int64)
    else:
        m_e = np.asarray(rows_per_expert, dtype=np.int64)
    padded = -(-m_e // align) * align
    m_expert = np.concatenate([
        np.concatenate([np.full(m, e), np.full(p - m, -1)]) for e, (m, p) in enumerate(zip(m_e, padded))
    ]).astype(np.int32)
    q, s = random_weights(rng, num_experts, n, k)
    a = random_activations(rng, int(padded.sum()), k)
    return GroupedProblem(name or f"grouped_contiguous_E{num_experts}_N{n}_K{k}", "contiguous",
                          num_experts, n, k, a, m_expert, q, s, int(m_e.mean()))


def contiguous_layout(rows_per_expert, num_experts=48, align=128):
    """m_expert [M_pad] int32 of the contiguous layout: each expert's rows,
    padded up to a multiple of ``align`` rows with -1."""
    if np.isscalar(rows_per_expert):
        m_e = np.full(num_experts, int(rows_per_expert), dtype=np.int64)
    else:
        m_e = np.asarray(rows_per_expert, dtype=np.int64)
    padded = -(-m_e // align) * align
    return np.concatenate([
        np.concatenate([np.full(m, e), np.full(p - m, -1)]) for e, (m, p) in enumerate(zip(m_e, padded))
    ]).astype(np.int32)


def masked_counts(num_experts=48, max_m=32, seed=0):
    """masked_m ~ U{1..max_m} per expert (the draw of grouped_masked_problem)."""
    rng = np.random.default_rng(seed)
    return rng.integers(1, max_m + 1, size=num_experts).astype(np.int32)


def grouped_masked_problem(num_experts=48, max_m=32, n=4096, k=7168, seed=0, name=None,
                           expected_m=16):
    """Masked layout: a budget of max_m rows per expert, masked_m ~ U{1..max_m}."""
    rng = np.random.default_rng(seed)
    masked_m = rng.integers(1, max_m + 1, size=num_experts).astype(np.int32)
    q, s = random_weights(rng, num_experts, n, k)
    a = random_activations(rng, num_experts, max_m, k)
    return GroupedProblem(name or f"grouped_masked_E{num_experts}_M{max_m}_N{n}_K{k}", "masked",
                          num_experts, n, k, a, masked_m, q, s, expected_m)
