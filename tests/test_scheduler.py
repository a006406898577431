"""The per-shape scheduler, host only: the plan each workload family gets,
and what that plan becomes on the device (MMA issuers, accumulator slots,
epilogue, rings). The pages make tok_e, the routed rows per expert, the
quantity that decides the schedule, with a switch near 80 rows (page
"vLLM 宣布 Humming 后端可运行 … Chord 内核 …", section
"调度由每个专家收到的 token 数决定"). Each pinned choice below was measured
against its alternatives on GB300; the numbers are in the design notes."""

import pytest

from w4a16_int4_moe_gb300 import ops
from w4a16_int4_moe_gb300 import workloads as wl

H, I = 7168, 2048          # hidden and expert intermediate size of the EP8 shard


def _plan(tokens, topk, experts, n, k, hint=0.0):
    return ops.w4a16_plan(tokens, topk, experts, n, k, hint)


def _with(plan, **fields):
    p = ops.Plan.from_buffer_copy(plan)
    for f, v in fields.items():
        setattr(p, f, v)
    return p


@pytest.mark.parametrize("tok_e,block_m", [
    (0.3, 16), (5.3, 16), (10.0, 16), (10.66, 16),  # 1.5 tok_e <= 16
    (10.7, 32),
    (11.0, 32), (12.0, 32), (21.0, 32),             # the EP8 decode shard: 12
    (22.0, 48), (32.0, 48),
    (33.0, 64), (80.0, 64),                         # capped at 64
    (80.1, 64), (119.0, 64),                        # above the switch (EP8 prefill: 81)
    (120.0, 128), (199.0, 128), (200.0, 128), (600.0, 128),
])
def test_block_m_follows_tok_e(tok_e, block_m):
    assert _plan(1, 1, 1, 4096, H, tok_e).block_m == block_m


@pytest.mark.parametrize("tok_e,block_m", [(100.0, 64), (150.0, 128), (200.0, 128),
                                           (600.0, 128)])
def test_both_projections_get_the_same_blocks(tok_e, block_m):
    # the down projection (k = 2048) follows the same rule
    assert _plan(1, 1, 1, H, I, tok_e).block_m == block_m


def test_plan_ignores_total_tokens_given_tok_e():
    # the same tok_e from very different token counts gives the same plan
    a = _plan(64, 8, 48, 4096, H).as_dict()      # tok_e = 64 * 8 / 48 = 10.7
    b = _plan(6400, 8, 4800, 4096, H).as_dict()
    assert a == b


# the five workload families, as the bench runs them
CASES = {
    # name: (plan, k, expected block_m, issuers, accumulator slots, early epilogue
    # (for 65..128-row blocks: with a BF16 output, so not the down pass itself))
    "tiny": (lambda: _plan(64, 2, 8, 1024, 512, 16.0), 512, 32, 4, 2, 0),
    "ep8_decode gate_up": (lambda: _plan(576, 8, 48, 2 * I, H, 12.0), H, 32, 4, 2, 0),
    "ep8_decode down": (lambda: _plan(576, 8, 48, H, I, 12.0), I, 32, 4, 2, 0),
    "tp8 T=16 gate_up": (lambda: _plan(16, 8, 384, 512, H), H, 16, 4, 2, 0),
    "tp8 T=64 down": (lambda: _plan(64, 8, 384, H, 256), 256, 16, 4, 2, 0),
    "tp8 T=256 gate_up": (lambda: _plan(256, 8, 384, 512, H), H, 16, 4, 2, 0),
    "ep8_prefill gate_up": (lambda: _plan(8192, 8, 48, 2 * I, H, 81.33), H, 64, 4, 1, 1),
    "ep8_prefill down": (lambda: _plan(8192, 8, 48, H, I, 81.33), I, 64, 4, 1, 1),
    # four times the EP8 prefill rows (tok_e 325): 128-row blocks for both
    "heavy prefill gate_up": (lambda: _plan(32768, 8, 48, 2 * I, H, 325.3), H, 128, 2, 1, 1),
    "heavy prefill down": (lambda: _plan(32768, 8, 48, H, I, 325.3), I, 128, 1, 2, 1),
    # a 256-row plan the caller sets: four issuer threads, of which an item
    # uses 1, 2 or 4, over one 256-column accumulator slot
    "256-row plan": (lambda: _with(_plan(32768, 8, 48, 2 * I, H, 325.3), block_m=256,
                                   b_stages=4, stages=8), H, 256, 4, 1, 0),
    "grouped contiguous 128": (
        lambda: ops.w4a16_grouped_plan(ops.W4A16_GROUPED_CONTIGUOUS, 48 * 128, 2 * I, H, 128),
        H, 128, 2, 1, 1),
    # 128-row blocks: two issuers over k = 7168, one issuer and two slots over
    # the down projection's k = 2048 (the epilogue overlaps the next item)
    "grouped contiguous 1024 gate_up": (
        lambda: ops.w4a16_grouped_plan(ops.W4A16_GROUPED_CONTIGUOUS, 48 * 1024, 2 * I, H, 1024),
        H, 128, 2, 1, 1),
    "grouped contiguous 1024 down": (
        lambda: ops.w4a16_grouped_plan(ops.W4A16_GROUPED_CONTIGUOUS, 48 * 1024, H, I, 1024),
        I, 128, 1, 2, 1),
    "grouped masked 32": (
        lambda: ops.w4a16_grouped_plan(ops.W4A16_GROUPED_MASKED, 32, 2 * I, H, 16),
        H, 32, 4, 2, 0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_choices_at_each_workload(name):
    make, k, block_m, issuers, slots, early = CASES[name]
    plan = make()
    info = ops.w4a16_plan_info(plan, k)
    got = (plan.block_m, info.mma_issuers, info.acc_slots, info.early_epilogue)
    assert got == (block_m, issuers, slots, early), (name, plan.as_dict(), info.as_dict())
    # fixed by design: 128 weight rows per tile, whole K per item, one
    # persistent CTA per SM, no CTA pairs (measured no faster)
    assert (plan.bn, plan.split_k, plan.ctas_per_sm, plan.grid, plan.cta_pair) == (128, 1, 1, 0, 0)
    # the TMEM split: A slots (256 columns) + issuers x slots x block columns;
    # above 128 rows one slot of 256 columns that an item splits among the
    # issuers it uses
    if block_m > 128:
        assert info.acc_cols == 256 and info.acc_slots == 1
    else:
        assert 256 + info.mma_issuers * info.acc_slots * info.acc_cols <= 512
        assert info.acc_cols == (block_m + 31) // 32 * 32
    # the rings fill the shared memory a CTA may take, activation ring first
    assert info.smem_bytes <= 227 * 1024
    assert info.b_stages >= 4 and info.w_stages >= 4 and info.w_stages % 4 == 0
    if block_m > 128:
        assert info.b_stages % 4 == 0   # single-step slots: one reader per slot


# (activation stages, weight stages) in order of preference: an activation
# ring of at least six stages first (at EP8 prefill 6 + 8 stages measured 10%
# faster than 4 + 12), then the deepest weight ring
RING_PREFERENCE = [(8, 16), (6, 16), (8, 12), (6, 12), (8, 8), (6, 8), (4, 16), (4, 12),
                   (4, 8), (4, 4)]


@pytest.mark.parametrize("tok_e", [5.0, 12.0, 30.0, 81.0])
def test_rings_are_the_first_preference_that_fits(tok_e):
    plan = _plan(1, 1, 1, 4096, H, tok_e)
    chosen = (plan.b_stages // 2, plan.stages)
    assert chosen in RING_PREFERENCE
    for b, w in RING_PREFERENCE[: RING_PREFERENCE.index(chosen)]:
        p = ops.Plan(**{f: getattr(plan, f) for f, _ in ops.Plan._fields_})
        p.b_stages, p.stages = 2 * b, w
        with pytest.raises(ops.W4A16Error):     # does not fit in shared memory
            ops.w4a16_plan_info(p, H)
    assert ops.w4a16_plan_info(plan, H).smem_bytes > 150 * 1024


def test_plan_info_refuses_what_the_gemm_refuses():
    plan = _plan(576, 8, 48, 2 * I, H, 12.0)
    for field, bad in (("block_m", 24), ("block_m", 272), ("split_k", 2), ("bn", 64),
                       ("stages", 2), ("b_stages", 6)):
        p = ops.Plan(**{f: getattr(plan, f) for f, _ in ops.Plan._fields_})
        setattr(p, field, bad)
        with pytest.raises(ops.W4A16Error) as ei:
            ops.w4a16_plan_info(p, H)
        assert ei.value.status == ops.W4A16_ERR_INVALID_ARG
    with pytest.raises(ops.W4A16Error):
        ops.w4a16_grouped_plan(7, 32, 4096, H)


def test_single_launch_layer_rule():
    # the layer runs gate_up + activation + down as one launch when the
    # gate_up weights carry the interleaved gate/up layout, the pass is not
    # deterministic, the down reduction is long (inter >= 1024) and the
    # routing blocks hold at most 32 rows
    from w4a16_int4_moe_gb300.moe import single_launch_default
    glu, plain = ops.W4A16_LAYOUT_KTILE64_GLU16, ops.W4A16_LAYOUT_KTILE64
    decode_bm = _plan(576, 8, 48, 2 * I, H, 12.0).block_m
    prefill_bm = _plan(8192, 8, 48, 2 * I, H, 81.33).block_m
    assert single_launch_default(glu, False, I, decode_bm)        # EP8 decode shard
    assert not single_launch_default(glu, False, I, prefill_bm)   # EP8 prefill shard
    assert not single_launch_default(glu, False, 256, 16)         # TP8 shard
    assert not single_launch_default(plain, False, I, decode_bm)
    assert not single_launch_default(glu, True, I, decode_bm)


def test_bench_workloads_hit_the_intended_branches():
    # the synthetic workloads' tok_e land where the pages put them
    assert wl.ep8_decode(weights=False).tok_e_hint() == pytest.approx(12.0)
    prefill = wl.ep8_prefill(weights=False)
    assert prefill.tok_e_hint() > 80.0
