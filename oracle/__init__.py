"""CPU oracle for the W4A16 INT4 MoE expert GEMM pair.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product path (``w4a16_int4_moe_gb300``) never imports it and has
no CPU fallback; the two share no code.

Every function is a plain, slow, obviously-correct restatement of what the
method computes, in float64, from the pages that describe the Chord/Humming
operator:

* "vLLM と Novita AI が Chord をリリース：Kimi K2.x 用の高速 INT4 MoE カーネル"
  (agentlenshq), sections "コア貢献", "vLLM との統合 / ランタイムの考慮事項",
  "カーネルレベルの最適化";
* "vLLM 宣布 Humming 后端可运行 Novita 开源的 Chord 内核，称 H200 TP8 提速 1.33x、
  B300 EP8 decode 提速 2.15x" (arex-research), sections
  "六个场景的逐层测量与限定条件", "调度由每个专家收到的 token 数决定",
  "接入方式：用 Chord 替代公共 Humming 包".

Pins (tests/test_oracle_pins.py) tie each function to something other than
itself: brute-force per-token loops, closed forms, invariants, special cases
that reduce to a library routine, and hand-derived fixtures under
tests/golden/.
"""

from .moe_oracle import (  # noqa: F401
    GROUP_SIZE,
    ZERO_POINT,
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    round_to_bf16,
    unpack_codes,
    dequant_weights,
    moe_align_block_size,
    indexed_gate_up,
    silu_and_mul,
    indexed_down,
    grouped_contiguous,
    grouped_masked,
    moe_layer,
    topk_softmax,
)
