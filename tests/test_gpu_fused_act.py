"""The gate_up GEMM with the activation fused into its epilogue
(W4A16_GATE_UP_SILU over W4A16_LAYOUT_KTILE64_GLU16 weights).

It must give exactly the bits of the unfused path (gate_up to BF16, then
w4a16_silu_and_mul), and match the oracle's silu(g) * up on the BF16 gate_up
outputs within the activation tolerance.
"""

import numpy as np
import pytest
import torch

import oracle
from w4a16_int4_moe_gb300 import moe as moe_mod
from w4a16_int4_moe_gb300 import ops
from w4a16_int4_moe_gb300 import workloads as wl
from helpers import assert_close, bf16_bits, bf16_tensor, dev

pytestmark = pytest.mark.gpu


def _fused_and_unfused(p, device, bm=None, cta_pair=0):
    q, s = dev(p.q_gu, device), dev(p.s_gu.view(np.int16), device)
    pk = ops.w4a16_prepack(q, s)
    pk_glu = ops.w4a16_prepack(q, s, layout=ops.W4A16_LAYOUT_KTILE64_GLU16)
    plan = ops.w4a16_plan(p.tokens, p.topk, p.num_experts, 2 * p.inter, p.hidden,
                          p.tok_e_hint())
    if bm:
        plan.block_m = bm
        # fit larger token stages (256 rows: four single-k-step slots)
        plan.stages, plan.b_stages = min(plan.stages, 8), (4 if bm > 128 else 8)
    plan.cta_pair = cta_pair
    sid, eid, ntp = ops.w4a16_moe_align_block_size(dev(p.topk_ids, device), p.num_experts,
                                                   plan.block_m)
    ws = ops.new_workspace(plan, device, sid.numel(), p.hidden)
    x = bf16_tensor(p.x, device)
    g = ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, pk, p.num_experts, 2 * p.inter, p.hidden,
                                   x, p.tokens, p.topk, sid, eid, ntp, plan, ws)
    act_ref = ops.w4a16_silu_and_mul(g)
    glu_plan = ops.Plan.from_buffer_copy(plan)
    glu_plan.layout = ops.W4A16_LAYOUT_KTILE64_GLU16
    act = torch.full((p.numel, p.inter), float("nan"), dtype=torch.bfloat16, device=device)
    ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP_SILU, pk_glu, p.num_experts, 2 * p.inter,
                               p.hidden, x, p.tokens, p.topk, sid, eid, ntp, glu_plan, ws,
                               out=act)
    st, word = ops.w4a16_read_device_status(ws)
    assert st == ops.W4A16_OK, hex(word)
    routed = ((p.topk_ids >= 0) & (p.topk_ids < p.num_experts)).reshape(-1)
    return bf16_bits(g), bf16_bits(act_ref), bf16_bits(act), routed


@pytest.mark.parametrize("bm", [16, 32, 64, 256])
def test_fused_activation_tiny(cuda_dev, bm):
    p = wl.tiny(seed=51)
    g_bits, ref_bits, act_bits, routed = _fused_and_unfused(p, cuda_dev, bm)
    np.testing.assert_array_equal(act_bits[routed], ref_bits[routed])
    a_ref = oracle.bf16_bits_to_f64(oracle.silu_and_mul(g_bits[routed]))
    assert_close(oracle.bf16_bits_to_f64(act_bits[routed]), a_ref, f"fused act bm={bm}",
                 rel_l2=4e-3, max_abs_frac=1e-2)
    # against the float64 chain from the inputs: gate_up, BF16, then silu * up
    g_ref = oracle.indexed_gate_up(p.x, p.topk_ids, p.q_gu, p.s_gu)
    a_chain = oracle.silu_and_mul(oracle.f64_to_bf16_bits(np.nan_to_num(g_ref[routed])))
    # the activation of the BF16 gate and up values: the GEMM tolerance holds
    # (measured rel-L2 3.8e-3 on GB300)
    e = assert_close(oracle.bf16_bits_to_f64(act_bits[routed]), oracle.bf16_bits_to_f64(a_chain),
                     f"fused act vs oracle chain bm={bm}")
    print(f"fused act vs oracle chain bm={bm}: rel-L2 {e[0]:.3e} max-abs {e[1]:.3e}")


@pytest.mark.parametrize("bm", [32, 64])
def test_fused_activation_pair(cuda_dev, bm):
    # CTA pairs: the fused epilogue of each CTA's tile gives the unfused bits
    p = wl.tiny(seed=53)
    g_bits, ref_bits, act_bits, routed = _fused_and_unfused(p, cuda_dev, bm, cta_pair=1)
    np.testing.assert_array_equal(act_bits[routed], ref_bits[routed])


def test_fused_activation_256_row_blocks(cuda_dev):
    # 256-row blocks with items of every kind: K split over 4 or 2 issuers
    # (at most 64 / 128 rows) and N split over 2 (above 128 rows)
    p = wl.uniform_problem(640, 1024, 256, 5, 2, seed=55)    # ~256 rows per expert
    p.topk_ids[290:][p.topk_ids[290:] == 4] = -1             # expert 4: 65..128 rows
    counts = np.bincount(p.topk_ids[p.topk_ids >= 0], minlength=5)
    assert counts.max() > 256 and (counts % 256 <= 64).any() and 64 < counts[4] <= 128
    g_bits, ref_bits, act_bits, routed = _fused_and_unfused(p, cuda_dev, 256)
    np.testing.assert_array_equal(act_bits[routed], ref_bits[routed])


def test_fused_activation_tp8_shape(cuda_dev):
    p = wl.uniform_problem(64, 1024, 256, 48, 8, seed=52)   # I = 256: 4 fused tiles
    g_bits, ref_bits, act_bits, routed = _fused_and_unfused(p, cuda_dev)
    np.testing.assert_array_equal(act_bits[routed], ref_bits[routed])


def test_fused_activation_ep8_decode_full_size(cuda_dev):
    p = wl.ep8_decode()
    g_bits, ref_bits, act_bits, routed = _fused_and_unfused(p, cuda_dev)
    np.testing.assert_array_equal(act_bits[routed], ref_bits[routed])
    # sampled act columns against the oracle on their gate and up columns
    cols = np.array([0, 1, 63, 64, 511, 1000, 1337, 2047])
    g_ref = oracle.indexed_gate_up(p.x, p.topk_ids, p.q_gu, p.s_gu,
                                   cols=np.concatenate([cols, p.inter + cols]))
    gb = oracle.f64_to_bf16_bits(np.nan_to_num(g_ref[routed]))
    g = oracle.bf16_bits_to_f64(gb[:, :len(cols)])
    u = oracle.bf16_bits_to_f64(gb[:, len(cols):])
    a_ref = g / (1.0 + np.exp(-g)) * u
    assert_close(oracle.bf16_bits_to_f64(act_bits[routed][:, cols]), a_ref,
                 "fused act EP8 sampled columns")


def test_layer_forward_with_fused_activation(cuda_dev):
    p = wl.tiny(seed=53)

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(cuda_dev)

    dn = moe_mod.PackedExperts.from_checkpoint(t(p.q_dn), t(p.s_dn.view(np.int16)))
    gu = moe_mod.PackedExperts.from_checkpoint(t(p.q_gu), t(p.s_gu.view(np.int16)))
    gu_glu = moe_mod.PackedExperts.from_checkpoint(
        t(p.q_gu), t(p.s_gu.view(np.int16)), layout=ops.W4A16_LAYOUT_KTILE64_GLU16)
    x, ids, w = bf16_tensor(p.x, cuda_dev), t(p.topk_ids), t(p.topk_weights)
    y_plain = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, device=cuda_dev).forward(x, ids, w)
    layer = moe_mod.W4A16MoE(gu_glu, dn, p.topk, p.tokens, device=cuda_dev)
    assert layer.fused_act
    y_fused = layer.forward(x, ids, w)
    torch.cuda.synchronize()
    # same activation bits, so the down pass sees the same input; only the
    # order of its atomic adds may differ
    assert_close(y_fused.cpu().numpy(), y_plain.cpu().numpy(), "layer fused vs plain",
                 rel_l2=1e-6, max_abs_frac=1e-6)


def test_gemm_from_pack_quantized_checkpoint(cuda_dev):
    # weights handed over as compressed-tensors int32 words give the same GEMM
    from w4a16_int4_moe_gb300 import checkpoint
    p = wl.tiny(seed=54)
    words = torch.from_numpy(np.ascontiguousarray(p.q_gu)).view(torch.int32).to(cuda_dev)
    scales = torch.from_numpy(p.s_gu.view(np.int16)).view(torch.bfloat16).to(cuda_dev)
    pe = checkpoint.packed_experts_from_pack_quantized(words, scales)
    ref = ops.w4a16_prepack(dev(p.q_gu, cuda_dev), dev(p.s_gu.view(np.int16), cuda_dev))
    assert torch.equal(pe.packed, ref)


# --------------------------------------------------- the single-launch layer --

def _layers(p, device, single_bm=None):
    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)
    gu = moe_mod.PackedExperts.from_checkpoint(t(p.q_gu), t(p.s_gu.view(np.int16)),
                                               layout=ops.W4A16_LAYOUT_KTILE64_GLU16)
    dn = moe_mod.PackedExperts.from_checkpoint(t(p.q_dn), t(p.s_dn.view(np.int16)))
    # two launches asked for explicitly: at the EP8 decode shard the default
    # is the single launch, which leaves the layer's act_buf unwritten
    two = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, tok_e_hint=p.tok_e_hint(), device=device,
                           single_launch=False)
    one = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, tok_e_hint=p.tok_e_hint(), device=device,
                           single_launch=True)
    return two, one, t


@pytest.mark.parametrize("maker", ["tiny", "ragged", "tp8_like"])
def test_single_launch_layer_matches_two_launches_and_oracle(cuda_dev, maker):
    # gate_up (fused activation) and down in one persistent launch: the same
    # result as the two launches up to the order of the FP32 additions, and
    # the oracle's layer on the same activation
    if maker == "tiny":
        p = wl.tiny(seed=81)
    elif maker == "ragged":
        p = wl.uniform_problem(77, 320, 192, 6, 3, seed=82)
        p.topk_ids[::5, 0] = -1
    else:
        p = wl.uniform_problem(16, 1024, 256, 96, 8, seed=83)    # ~1.3 rows per expert
    two, one, t = _layers(p, cuda_dev)
    x = bf16_tensor(p.x, cuda_dev)
    ids, w = t(p.topk_ids), t(p.topk_weights)
    y2 = two.forward(x, ids, w)
    y1 = one.forward(x, ids, w)
    torch.cuda.synchronize()
    for layer in (two, one):
        ws = layer.layer_workspace if layer.single_launch else layer.workspace
        st, word = ops.w4a16_read_device_status(ws)
        assert st == ops.W4A16_OK, hex(word)
    assert_close(y1.cpu().numpy(), y2.cpu().numpy(), f"{maker}: one launch vs two",
                 rel_l2=1e-6, max_abs_frac=1e-5)
    # the oracle's down pass on the activation both paths computed
    routed = ((p.topk_ids >= 0) & (p.topk_ids < p.num_experts)).reshape(-1)
    act_bits = bf16_bits(two.act_buf[: p.numel])
    a = np.where(routed[:, None], act_bits, 0).astype(np.uint16)
    y_ref = oracle.indexed_down(a, p.topk_ids, p.topk_weights, p.q_dn, p.s_dn)
    assert_close(y1.cpu().numpy(), y_ref, f"{maker}: one launch vs oracle down")


def _layer_call(one, x, p, t, out, flags=0):
    return ops.w4a16_moe_layer(
        one.gate_up.packed, one.down.packed, one.num_experts, one.hidden, one.inter, x,
        p.tokens, p.topk, one.sorted_ids, one.expert_ids, one.ntp, one.plan_gu,
        one.layer_workspace, t(p.topk_weights), out=out, flags=flags)


def test_single_launch_layer_flags_and_empty_routing(cuda_dev):
    # ACCUMULATE adds into the output; VALIDATE_ROUTING checks the routing on
    # the host first; a routing with no local rows launches no work item and
    # leaves a zeroed output (or the prior one, with ACCUMULATE)
    p = wl.tiny(seed=85)
    two, one, t = _layers(p, cuda_dev)
    x = bf16_tensor(p.x, cuda_dev)
    ids, w = t(p.topk_ids), t(p.topk_weights)
    y = one.forward(x, ids, w)
    torch.cuda.synchronize()
    prior = torch.full_like(y, 0.25)
    out = prior.clone()
    _layer_call(one, x, p, t, out, flags=ops.W4A16_FLAG_ACCUMULATE | ops.W4A16_FLAG_VALIDATE_ROUTING)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), (y + prior).cpu().numpy(), "layer ACCUMULATE",
                 rel_l2=1e-6, max_abs_frac=1e-5)
    # no local rows: every id belongs to another GPU
    none = np.full_like(p.topk_ids, -1)
    one.align(t(none))
    out = torch.full_like(y, float("nan"))
    _layer_call(one, x, p, t, out)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
    out = prior.clone()
    _layer_call(one, x, p, t, out, flags=ops.W4A16_FLAG_ACCUMULATE)
    torch.cuda.synchronize()
    assert torch.equal(out, prior)
    st, word = ops.w4a16_read_device_status(one.layer_workspace)
    assert st == ops.W4A16_OK, hex(word)


def test_single_launch_layer_refuses_corrupt_routing(cuda_dev):
    # with VALIDATE_ROUTING an expert id out of range is refused before launch
    p = wl.tiny(seed=86)
    two, one, t = _layers(p, cuda_dev)
    x = bf16_tensor(p.x, cuda_dev)
    one.align(t(p.topk_ids))
    one.expert_ids[0] = p.num_experts + 3
    out = torch.zeros((p.tokens, p.hidden), dtype=torch.float32, device=cuda_dev)
    with pytest.raises(ops.W4A16Error) as ei:
        _layer_call(one, x, p, t, out, flags=ops.W4A16_FLAG_VALIDATE_ROUTING)
    assert ei.value.status == ops.W4A16_ERR_ROUTING


@pytest.mark.slow
def test_single_launch_layer_ep8_decode_full_size(cuda_dev):
    # the layer's default at the EP8 decode shard: the single launch equals the
    # two launches (same activation bits, FP32 adds in another order) and the
    # oracle's down pass on sampled output columns
    p = wl.ep8_decode()
    two, one, t = _layers(p, cuda_dev)
    assert moe_mod.W4A16MoE(one.gate_up, one.down, p.topk, p.tokens,
                            tok_e_hint=p.tok_e_hint(), device=cuda_dev).single_launch
    x = bf16_tensor(p.x, cuda_dev)
    ids, w = t(p.topk_ids), t(p.topk_weights)
    y2 = two.forward(x, ids, w)
    y1 = one.forward(x, ids, w)
    torch.cuda.synchronize()
    st, word = ops.w4a16_read_device_status(one.layer_workspace)
    assert st == ops.W4A16_OK, hex(word)
    assert_close(y1.cpu().numpy(), y2.cpu().numpy(), "EP8 decode: one launch vs two",
                 rel_l2=1e-6, max_abs_frac=1e-5)
    routed = ((p.topk_ids >= 0) & (p.topk_ids < p.num_experts)).reshape(-1)
    act_bits = bf16_bits(two.act_buf[: p.numel])
    a = np.where(routed[:, None], act_bits, 0).astype(np.uint16)
    cols = np.array([0, 5, 127, 128, 2048, 4095, 5000, 7167])
    y_ref = oracle.indexed_down(a, p.topk_ids, p.topk_weights, p.q_dn, p.s_dn, cols=cols)
    assert_close(y1.cpu().numpy()[:, cols], y_ref, "EP8 decode: one launch vs oracle down")
