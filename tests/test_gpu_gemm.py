"""Parity of the tcgen05 W4A16 MoE GEMMs with the float64 oracle.

Every comparison goes through the C ABI (ctypes binding). Stages are compared
one at a time: the GPU's down pass is checked on the GPU's own BF16
activation fed to the oracle, so errors do not compound across stages.
Small shapes are compared element by element over every routed row; the
full-size shard shapes are compared on sampled output columns (the oracle
evaluates the plain definition only there) or sampled rows.
"""

import functools

import numpy as np
import pytest
import torch

import oracle
from w4a16_int4_moe_gb300 import moe as moe_mod
from w4a16_int4_moe_gb300 import ops
from w4a16_int4_moe_gb300 import workloads as wl
from helpers import assert_close, bf16_bits, bf16_tensor, dev

pytestmark = pytest.mark.gpu


def _pack(q, s, device):
    return ops.w4a16_prepack(dev(q, device), dev(s.view(np.int16), device))


def _routing(ids, experts, bm, device):
    t = dev(ids, device)
    cap = ops.w4a16_align_capacity(t.numel(), experts, bm)
    return ops.w4a16_moe_align_block_size(t, experts, bm, cap)


def _plan(bm, n, k, stages=None, b_stages=None, grid=0, pair=False):
    p = ops.w4a16_plan(64, 1, 1, n, k, float(bm))
    p.block_m = bm
    if bm > 128:
        # four activation slots of one k step (32 KB at 256 rows), eight weight stages
        p.b_stages = b_stages or 4
        p.stages = stages or 8
    else:
        p.b_stages = b_stages or 8
        p.stages = stages or min(p.stages, 8)
    p.grid = grid
    p.cta_pair = int(pair)
    return p


def _gate_up(p, packed, routing, plan, device):
    sid, eid, ntp = routing
    ws = ops.new_workspace(plan, device, sid.numel(), p.hidden)
    x = bf16_tensor(p.x, device)
    out = torch.full((p.numel, 2 * p.inter), float("nan"), dtype=torch.bfloat16, device=device)
    ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, packed, p.num_experts, 2 * p.inter, p.hidden,
                               x, p.tokens, p.topk, sid, eid, ntp, plan, ws, out=out)
    st, word = ops.w4a16_read_device_status(ws)
    assert st == ops.W4A16_OK, hex(word)
    return out


def _down(p, packed, routing, plan, act_bits, device):
    sid, eid, ntp = routing
    ws = ops.new_workspace(plan, device, sid.numel(), p.inter)
    a = bf16_tensor(act_bits, device)
    w = dev(p.topk_weights, device)
    out = torch.full((p.tokens, p.hidden), float("nan"), dtype=torch.float32, device=device)
    ops.w4a16_moe_indexed_gemm(ops.W4A16_DOWN, packed, p.num_experts, p.hidden, p.inter, a,
                               p.tokens, p.topk, sid, eid, ntp, plan, ws, topk_weights=w, out=out)
    st, word = ops.w4a16_read_device_status(ws)
    assert st == ops.W4A16_OK, hex(word)
    return out


def _routed(p):
    flat = p.topk_ids.reshape(-1)
    return (flat >= 0) & (flat < p.num_experts)


def _check_pair(p, device, bm, cols_gu=None, cols_dn=None, what="", cta_pair=False, bm_dn=None):
    """gate_up vs oracle, then down (on the GPU's activation) vs oracle; the
    down GEMM on its own routing blocks of bm_dn rows when given."""
    pk_gu = _pack(p.q_gu, p.s_gu, device)
    pk_dn = _pack(p.q_dn, p.s_dn, device)
    routing = _routing(p.topk_ids, p.num_experts, bm, device)
    g = _gate_up(p, pk_gu, routing, _plan(bm, 2 * p.inter, p.hidden, pair=cta_pair), device)
    g_bits = bf16_bits(g)
    routed = _routed(p)
    g_ref = oracle.indexed_gate_up(p.x, p.topk_ids, p.q_gu, p.s_gu, cols=cols_gu)
    g_got = oracle.bf16_bits_to_f64(g_bits)
    if cols_gu is not None:
        g_got = g_got[:, cols_gu]
    e1 = assert_close(g_got[routed], g_ref[routed], f"{what} gate_up")
    # activation (untimed glue) on the GPU's own gate_up output
    act = ops.w4a16_silu_and_mul(g)
    a_bits = bf16_bits(act)
    a_ref = oracle.bf16_bits_to_f64(oracle.silu_and_mul(g_bits[routed]))
    assert_close(oracle.bf16_bits_to_f64(a_bits[routed]), a_ref, f"{what} silu_and_mul",
                 rel_l2=4e-3, max_abs_frac=1e-2)
    a_bits_clean = a_bits.copy()
    a_bits_clean[~routed] = 0
    bm_dn = bm_dn or bm
    routing_dn = routing if bm_dn == bm else _routing(p.topk_ids, p.num_experts, bm_dn, device)
    y = _down(p, pk_dn, routing_dn, _plan(bm_dn, p.hidden, p.inter, pair=cta_pair), a_bits_clean,
              device)
    y_ref = oracle.indexed_down(a_bits_clean, p.topk_ids, p.topk_weights, p.q_dn, p.s_dn,
                                cols=cols_dn)
    y_got = y.cpu().numpy()
    if cols_dn is not None:
        y_got = y_got[:, cols_dn]
    e2 = assert_close(y_got, y_ref, f"{what} down")
    print(f"{what}: gate_up rel-L2 {e1[0]:.2e} max-abs {e1[1]:.2e}; "
          f"down rel-L2 {e2[0]:.2e} max-abs {e2[1]:.2e}")
    return g_bits


# ------------------------------------------------------------ small shapes --

@pytest.mark.parametrize("bm", [16, 32, 48, 64, 128, 256])
def test_tiny_all_block_sizes(cuda_dev, bm):
    _check_pair(wl.tiny(), cuda_dev, bm, what=f"tiny bm={bm}")


@pytest.mark.parametrize("bm", [64, 128, 256])
def test_blocks_of_mixed_fill(cuda_dev, bm):
    # 50..73 rows per expert: at block_m 64 an expert fills one block and
    # part of a second, at block_m 128 a block is between 39% and 57% full,
    # at 256 between 20% and 29%
    p = wl.uniform_problem(256, 1024, 512, 16, 4, seed=61)
    _check_pair(p, cuda_dev, bm, what=f"mixed fill bm={bm}")


@pytest.mark.parametrize("tokens,hidden,inter,experts,topk,bm", [
    (37, 96, 96, 5, 3, 16),      # k = 32 mod 64 on both GEMMs, ragged n (192 / 96 rows)
    (200, 320, 224, 6, 2, 64),   # ragged n tiles (448 / 320 rows), k = 32 mod 64 on down
    (5, 64, 32, 40, 4, 16),      # far more experts than rows: many empty experts
    (130, 256, 160, 3, 1, 64),   # top-1, several blocks per expert
    (37, 96, 96, 5, 3, 256),     # 256-row blocks: k = 32 mod 64, so pad k steps on both GEMMs
    (700, 320, 192, 2, 1, 256),  # 256-row blocks, two or more per expert, ragged last block
])
def test_ragged_shapes(cuda_dev, tokens, hidden, inter, experts, topk, bm):
    p = wl.uniform_problem(tokens, hidden, inter, experts, topk, seed=tokens)
    _check_pair(p, cuda_dev, bm, what=f"ragged {tokens}x{hidden}x{inter}")


def test_nonlocal_and_degenerate_routing(cuda_dev):
    p = wl.uniform_problem(48, 128, 64, 6, 2, seed=21)
    p.topk_ids[::3, 0] = -1          # non-local experts
    p.topk_ids[1::5, 1] = 9          # ids >= E are not local either
    _check_pair(p, cuda_dev, 16, what="non-local")


def test_all_zero_point_weights_give_zero(cuda_dev):
    p = wl.tiny(seed=4)
    p.q_gu[:] = 0x88
    pk = _pack(p.q_gu, p.s_gu, cuda_dev)
    routing = _routing(p.topk_ids, p.num_experts, 32, cuda_dev)
    g = _gate_up(p, pk, routing, _plan(32, 2 * p.inter, p.hidden), cuda_dev)
    routed = _routed(p)
    assert torch.all(g[torch.from_numpy(routed).to(cuda_dev)] == 0)


def test_no_routed_rows_leaves_output_untouched(cuda_dev):
    p = wl.tiny(seed=5)
    p.topk_ids[:] = -1
    pk = _pack(p.q_gu, p.s_gu, cuda_dev)
    routing = _routing(p.topk_ids, p.num_experts, 16, cuda_dev)
    g = _gate_up(p, pk, routing, _plan(16, 2 * p.inter, p.hidden), cuda_dev)
    assert torch.all(torch.isnan(g))


@pytest.mark.parametrize("single_launch", [False, True])
def test_empty_batch(cuda_dev, single_launch):
    # no tokens at all: align writes a padded total of 0 (its zero-element
    # arrays passed as NULL), and the layer returns an empty output, through
    # two launches or one
    p = wl.tiny(seed=12)
    ids = torch.empty((0, p.topk), dtype=torch.int32, device=cuda_dev)
    assert ops.w4a16_align_capacity(0, p.num_experts, 32) == 0
    ntp = torch.full((1,), -5, dtype=torch.int32, device=cuda_dev)
    empty = torch.empty(0, dtype=torch.int32, device=cuda_dev)
    ops.w4a16_moe_align_block_size(ids, p.num_experts, 32, 0, out=(empty, empty, ntp))
    assert int(ntp.item()) == 0
    layout = ops.W4A16_LAYOUT_KTILE64_GLU16 if single_launch else ops.W4A16_LAYOUT_KTILE64
    gu = moe_mod.PackedExperts.from_checkpoint(dev(p.q_gu, cuda_dev),
                                               dev(p.s_gu.view(np.int16), cuda_dev), layout=layout)
    dn = moe_mod.PackedExperts.from_checkpoint(dev(p.q_dn, cuda_dev),
                                               dev(p.s_dn.view(np.int16), cuda_dev))
    layer = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, device=cuda_dev,
                             single_launch=single_launch)
    x = torch.empty((0, p.hidden), dtype=torch.bfloat16, device=cuda_dev)
    w = torch.empty((0, p.topk), dtype=torch.float32, device=cuda_dev)
    y = layer.forward(x, ids, w)
    torch.cuda.synchronize()
    assert y.shape == (0, p.hidden)
    assert int(layer.ntp.item()) == 0
    ws = layer.layer_workspace if single_launch else layer.workspace
    assert ops.w4a16_read_device_status(ws)[0] == ops.W4A16_OK
    # the same layer on a real batch afterwards
    y = layer.forward(bf16_tensor(p.x, cuda_dev), dev(p.topk_ids, cuda_dev),
                      dev(p.topk_weights, cuda_dev))
    _, _, _, y_ref = oracle.moe_layer(p.x, p.topk_ids, p.topk_weights, p.q_gu, p.s_gu,
                                      p.q_dn, p.s_dn)
    assert_close(y.cpu().numpy(), y_ref, "layer after an empty batch")


def test_schedules_are_bitwise_identical(cuda_dev):
    # Pipelining and scheduling choices do not change any gate_up output bit
    # (every row's K reduction runs in the same order): block size, ring
    # depths and grid size.
    p = wl.uniform_problem(96, 512, 256, 8, 2, seed=8)
    pk = _pack(p.q_gu, p.s_gu, cuda_dev)
    ref = None
    for bm, st, bst, grid in [(16, 8, 8, 0), (32, 4, 16, 0), (64, 8, 8, 3), (64, 4, 12, 1),
                              (16, 12, 12, 5), (48, 7, 8, 7)]:
        routing = _routing(p.topk_ids, p.num_experts, bm, cuda_dev)
        g = _gate_up(p, pk, routing, _plan(bm, 2 * p.inter, p.hidden, st, bst, grid), cuda_dev)
        bits = bf16_bits(g)[_routed(p)]
        if ref is None:
            ref = bits
        else:
            np.testing.assert_array_equal(bits, ref, err_msg=f"bm={bm} stages={st}")


def test_over_allocated_routing_and_validation(cuda_dev):
    p = wl.tiny(seed=6)
    pk = _pack(p.q_gu, p.s_gu, cuda_dev)
    t = dev(p.topk_ids, cuda_dev)
    cap = ops.w4a16_align_capacity(t.numel(), 8, 32) + 32 * 8   # extra unused blocks
    sid, eid, ntp = ops.w4a16_moe_align_block_size(t, 8, 32, cap)
    plan = _plan(32, 2 * p.inter, p.hidden)
    ws = ops.new_workspace(plan, cuda_dev, cap, p.hidden)
    out = torch.empty((p.numel, 2 * p.inter), dtype=torch.bfloat16, device=cuda_dev)
    ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, pk, 8, 2 * p.inter, p.hidden,
                               bf16_tensor(p.x, cuda_dev), p.tokens, p.topk, sid, eid, ntp, plan,
                               ws, out=out, flags=ops.W4A16_FLAG_VALIDATE_ROUTING)
    g_ref = oracle.indexed_gate_up(p.x, p.topk_ids, p.q_gu, p.s_gu)
    assert_close(oracle.bf16_bits_to_f64(bf16_bits(out)), g_ref, "over-allocated")
    # corrupt routing is refused when validation is on
    eid[0] = 99
    with pytest.raises(ops.W4A16Error) as ei:
        ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, pk, 8, 2 * p.inter, p.hidden,
                                   bf16_tensor(p.x, cuda_dev), p.tokens, p.topk, sid, eid, ntp,
                                   plan, ws, out=out, flags=ops.W4A16_FLAG_VALIDATE_ROUTING)
    assert ei.value.status == ops.W4A16_ERR_ROUTING
    # ... and is ignored (never dereferenced) when validation is off
    ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, pk, 8, 2 * p.inter, p.hidden,
                               bf16_tensor(p.x, cuda_dev), p.tokens, p.topk, sid, eid, ntp, plan,
                               ws, out=out)
    assert ops.w4a16_read_device_status(ws)[0] == ops.W4A16_OK


def _down_det(p, packed, routing, plan, act_bits, device, out=None, accumulate=False):
    sid, eid, ntp = routing
    ws = ops.new_workspace(plan, device, sid.numel(), p.inter, det_n=p.hidden,
                           det_numel=p.numel)
    a = bf16_tensor(act_bits, device)
    w = dev(p.topk_weights, device)
    if out is None:
        out = torch.full((p.tokens, p.hidden), float("nan"), dtype=torch.float32, device=device)
    flags = ops.W4A16_FLAG_DETERMINISTIC | (ops.W4A16_FLAG_ACCUMULATE if accumulate else 0)
    ops.w4a16_moe_indexed_gemm(ops.W4A16_DOWN, packed, p.num_experts, p.hidden, p.inter, a,
                               p.tokens, p.topk, sid, eid, ntp, plan, ws, topk_weights=w,
                               out=out, flags=flags)
    st, word = ops.w4a16_read_device_status(ws)
    assert st == ops.W4A16_OK, hex(word)
    return out


def test_down_deterministic_256_row_blocks(cuda_dev):
    # the deterministic pass on 256-row blocks (items of 1-4 issuers): the
    # same bits for any grid, the oracle's values, 0 for a token without a
    # local expert
    p = wl.uniform_problem(512, 1024, 512, 6, 3, seed=66)   # ~256 rows per expert
    p.topk_ids[200:][p.topk_ids[200:] == 5] = -1             # expert 5: 65..128 rows
    p.topk_ids[7, :] = -1
    counts = np.bincount(p.topk_ids[p.topk_ids >= 0], minlength=6)
    assert counts.max() > 256 and 64 < counts[5] <= 128
    pk = _pack(p.q_dn, p.s_dn, cuda_dev)
    a_bits = wl.random_activations(np.random.default_rng(67), p.numel, p.inter)
    a_bits[~_routed(p)] = 0
    ref = oracle.indexed_down(a_bits, p.topk_ids, p.topk_weights, p.q_dn, p.s_dn)
    routing = _routing(p.topk_ids, p.num_experts, 256, cuda_dev)
    outs = [_down_det(p, pk, routing, _plan(256, p.hidden, p.inter, grid=g), a_bits,
                      cuda_dev).cpu().numpy() for g in (0, 5)]
    np.testing.assert_array_equal(outs[1].view(np.uint32), outs[0].view(np.uint32))
    assert np.all(outs[0][7] == 0.0)
    assert_close(outs[0], ref, "deterministic down, 256-row blocks")


def test_down_deterministic(cuda_dev):
    # W4A16_FLAG_DETERMINISTIC: each weighted row goes to the workspace and a
    # second kernel adds every token's rows in top-k slot order. The output
    # bits are then the same for every block size and grid, the values match
    # the oracle, tokens without a local expert get 0, and ACCUMULATE adds.
    p = wl.uniform_problem(256, 1024, 512, 16, 4, seed=63)
    p.topk_ids[::7, 1] = -1          # some rows routed elsewhere
    p.topk_ids[5, :] = -1            # a token with no local expert
    pk = _pack(p.q_dn, p.s_dn, cuda_dev)
    a_bits = wl.random_activations(np.random.default_rng(64), p.numel, p.inter)
    a_bits[~_routed(p)] = 0
    ref = oracle.indexed_down(a_bits, p.topk_ids, p.topk_weights, p.q_dn, p.s_dn)
    outs = []
    for bm, grid in ((16, 0), (32, 7), (48, 0), (64, 13)):
        routing = _routing(p.topk_ids, p.num_experts, bm, cuda_dev)
        y = _down_det(p, pk, routing, _plan(bm, p.hidden, p.inter, grid=grid), a_bits, cuda_dev)
        outs.append(y.cpu().numpy())
    for y in outs[1:]:
        np.testing.assert_array_equal(y.view(np.uint32), outs[0].view(np.uint32))
    assert np.all(outs[0][5] == 0.0)
    assert_close(outs[0], ref, "deterministic down")
    routing = _routing(p.topk_ids, p.num_experts, 32, cuda_dev)
    prior = torch.full((p.tokens, p.hidden), 0.5, dtype=torch.float32, device=cuda_dev)
    y2 = _down_det(p, pk, routing, _plan(32, p.hidden, p.inter), a_bits, cuda_dev, out=prior,
                   accumulate=True)
    np.testing.assert_array_equal(y2.cpu().numpy(), np.float32(0.5) + outs[1])


def test_layer_deterministic_matches_oracle(cuda_dev):
    p = wl.tiny(seed=65)

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(cuda_dev)

    gu = moe_mod.PackedExperts.from_checkpoint(t(p.q_gu), t(p.s_gu.view(np.int16)))
    dn = moe_mod.PackedExperts.from_checkpoint(t(p.q_dn), t(p.s_dn.view(np.int16)))
    layer = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, device=cuda_dev, deterministic=True)
    x, ids, w = bf16_tensor(p.x, cuda_dev), t(p.topk_ids), t(p.topk_weights)
    y1 = layer.forward(x, ids, w).cpu().numpy()
    y2 = layer.forward(x, ids, w).cpu().numpy()
    np.testing.assert_array_equal(y1.view(np.uint32), y2.view(np.uint32))
    _, _, _, y_ref = oracle.moe_layer(p.x, p.topk_ids, p.topk_weights, p.q_gu, p.s_gu,
                                      p.q_dn, p.s_dn)
    assert_close(y1, y_ref, "deterministic layer")


def test_down_accumulate_flag(cuda_dev):
    p = wl.tiny(seed=7)
    pk = _pack(p.q_dn, p.s_dn, cuda_dev)
    routing = _routing(p.topk_ids, 8, 32, cuda_dev)
    plan = _plan(32, p.hidden, p.inter)
    rng = np.random.default_rng(1)
    a_bits = wl.random_activations(rng, p.numel, p.inter)
    y = _down(p, pk, routing, plan, a_bits, cuda_dev)
    sid, eid, ntp = routing
    ws = ops.new_workspace(plan, cuda_dev, sid.numel(), p.inter)
    y2 = y.clone()
    ops.w4a16_moe_indexed_gemm(ops.W4A16_DOWN, pk, 8, p.hidden, p.inter,
                               bf16_tensor(a_bits, cuda_dev), p.tokens, p.topk, sid, eid, ntp,
                               plan, ws, topk_weights=dev(p.topk_weights, cuda_dev), out=y2,
                               flags=ops.W4A16_FLAG_ACCUMULATE)
    assert_close(y2.cpu().numpy(), 2.0 * y.cpu().numpy(), "accumulate", rel_l2=1e-6,
                 max_abs_frac=1e-6)


def test_layer_forward_and_graph_capture(cuda_dev):
    p = wl.tiny(seed=9)
    gu = moe_mod.PackedExperts.from_checkpoint(dev(p.q_gu, cuda_dev),
                                               dev(p.s_gu.view(np.int16), cuda_dev))
    dn = moe_mod.PackedExperts.from_checkpoint(dev(p.q_dn, cuda_dev),
                                               dev(p.s_dn.view(np.int16), cuda_dev))
    layer = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens)
    x = bf16_tensor(p.x, cuda_dev)
    ids = dev(p.topk_ids, cuda_dev)
    w = dev(p.topk_weights, cuda_dev)
    y = layer.forward(x, ids, w)
    torch.cuda.synchronize()
    g, g_bits, a_bits, y_ref = oracle.moe_layer(p.x, p.topk_ids, p.topk_weights, p.q_gu, p.s_gu,
                                                p.q_dn, p.s_dn)
    assert_close(y.cpu().numpy(), y_ref, "layer forward")
    # the whole pair captured in one CUDA graph (routing validation off)
    s = torch.cuda.Stream()
    out = torch.zeros_like(y)
    with torch.cuda.stream(s):
        layer.forward(x, ids, w, out=out)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        layer.forward(x, ids, w, out=out)
    graph.replay()
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), y_ref, "graph replay")


@pytest.mark.parametrize("from_logits", [False, True])
def test_layer_with_different_blocks_per_gemm(cuda_dev, from_logits, monkeypatch):
    # gate_up (k = 4096) on 256-row blocks, down (k = 256) on 128, each on its
    # own routing (the plan of the long reduction is set to 256 rows here);
    # experts of a little under or over 256 rows give items of 1 issuer and of
    # 4 (a short second block); the result is the oracle layer's
    rng = np.random.default_rng(23)
    tokens, hidden, inter, experts, topk = 512, 4096, 256, 8, 4
    logits = rng.standard_normal((tokens, experts)).astype(np.float32)
    ids, wts = oracle.topk_softmax(logits, topk, renormalize=True)
    ids = ids.astype(np.int32)
    wts = wts.astype(np.float32)
    p = wl.make_problem("blocks_per_gemm", rng, tokens, hidden, inter, experts, topk, ids)
    gu = moe_mod.PackedExperts.from_checkpoint(dev(p.q_gu, cuda_dev),
                                               dev(p.s_gu.view(np.int16), cuda_dev))
    dn = moe_mod.PackedExperts.from_checkpoint(dev(p.q_dn, cuda_dev),
                                               dev(p.s_dn.view(np.int16), cuda_dev))
    plan = ops.w4a16_plan

    def gate_up_on_256_rows(tokens_, topk_, experts_, n_, k_, hint_=0.0):
        p_ = plan(tokens_, topk_, experts_, n_, k_, hint_)
        if k_ == hidden:
            p_.block_m, p_.b_stages, p_.stages = 256, 4, 8
        return p_

    monkeypatch.setattr(ops, "w4a16_plan", gate_up_on_256_rows)
    layer = moe_mod.W4A16MoE(gu, dn, topk, tokens, tok_e_hint=256.0)
    assert (layer.block_m, layer.block_m_dn) == (256, 128)
    x = bf16_tensor(p.x, cuda_dev)
    if from_logits:
        y = layer.forward_from_logits(x, dev(logits, cuda_dev))
    else:
        y = layer.forward(x, dev(ids, cuda_dev), dev(wts, cuda_dev))
    torch.cuda.synchronize()
    _, _, _, y_ref = oracle.moe_layer(p.x, ids, wts, p.q_gu, p.s_gu, p.q_dn, p.s_dn)
    assert_close(y.cpu().numpy(), y_ref, f"layer, blocks 256 / 128, from_logits={from_logits}")


# ---------------------------------------------------------- grouped GEMMs --

def _grouped(gp, device, plan=None):
    pk = _pack(gp.q, gp.s, device)
    ws = ops.new_workspace(plan or ops.w4a16_plan(16, 1, 1, gp.n, gp.k, 16.0), device)
    a = bf16_tensor(gp.a, device)
    lay = dev(gp.layout, device)
    kind = ops.W4A16_GROUPED_CONTIGUOUS if gp.kind == "contiguous" else ops.W4A16_GROUPED_MASKED
    m = gp.a.shape[0] if gp.kind == "contiguous" else gp.a.shape[1]
    # rows the call leaves untouched (padding, past a masked count) read as zeros
    shape = (m, gp.n) if gp.kind == "contiguous" else (gp.num_experts, m, gp.n)
    out = torch.zeros(shape, dtype=torch.bfloat16, device=device)
    ops.w4a16_moe_grouped_gemm(kind, pk, gp.num_experts, gp.n, gp.k, a, m, lay, ws, plan=plan,
                               expected_m=gp.expected_m, out=out)
    st, word = ops.w4a16_read_device_status(ws)
    assert st == ops.W4A16_OK, hex(word)
    return oracle.bf16_bits_to_f64(bf16_bits(out))


@pytest.mark.parametrize("bm", [32, 64, 128])
def test_grouped_contiguous_small(cuda_dev, bm):
    gp = wl.grouped_contiguous_problem([5, 128, 0, 77], num_experts=4, n=200, k=96, seed=bm)
    got = _grouped(gp, cuda_dev, _plan(bm, gp.n, gp.k))
    ref = oracle.grouped_contiguous(gp.a, gp.layout, gp.q, gp.s)
    valid = gp.layout >= 0
    assert_close(got[valid], ref[valid], f"contiguous bm={bm}")


@pytest.mark.parametrize("bm,n", [(128, 198), (64, 198), (128, 130)])
def test_grouped_contiguous_width_not_multiple_of_4(cuda_dev, bm, n):
    # output rows whose width is not a multiple of 4 take the scalar stores
    # of the staged epilogue (128 rows: BF16 staging; 64 rows: FP32)
    gp = wl.grouped_contiguous_problem([5, 128, 0, 77], num_experts=4, n=n, k=96, seed=n + bm)
    got = _grouped(gp, cuda_dev, _plan(bm, gp.n, gp.k))
    ref = oracle.grouped_contiguous(gp.a, gp.layout, gp.q, gp.s)
    valid = gp.layout >= 0
    assert_close(got[valid], ref[valid], f"contiguous bm={bm} n={n}")


@pytest.mark.parametrize("bm", [16, 32])
def test_grouped_masked_small(cuda_dev, bm):
    gp = wl.grouped_masked_problem(num_experts=6, max_m=32, n=256, k=160, seed=bm)
    gp.layout[2] = 0      # an expert with no rows
    gp.layout[3] = 32     # a full budget
    got = _grouped(gp, cuda_dev, _plan(bm, gp.n, gp.k))
    ref = oracle.grouped_masked(gp.a, gp.layout, gp.q, gp.s)
    valid = ~np.isnan(ref[..., 0])
    assert_close(got[valid], ref[valid], f"masked bm={bm}")


@pytest.mark.parametrize("k", [160, 192])
def test_grouped_masked_256_row_blocks(cuda_dev, k):
    # a 300-row budget on 256-row blocks: two blocks per expert, items of
    # every issuer split (N <= 64, <= 128 and above), one k step per copy
    # (k = 32 mod 64 gives a pad k step)
    gp = wl.grouped_masked_problem(num_experts=5, max_m=300, n=256, k=k, seed=k)
    gp.layout[:] = [300, 40, 0, 100, 257]
    got = _grouped(gp, cuda_dev, _plan(256, gp.n, gp.k))
    ref = oracle.grouped_masked(gp.a, gp.layout, gp.q, gp.s)
    valid = ~np.isnan(ref[..., 0])
    assert_close(got[valid], ref[valid], f"masked bm=256 k={k}")


# ------------------------------------------------- full-size shard shapes --

@functools.lru_cache(maxsize=1)
def _ep8_decode():
    return wl.ep8_decode()


def _sample_cols(n, count, seed):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(n, size=min(n, count), replace=False))


@pytest.mark.slow
def test_ep8_decode_full_size(cuda_dev):
    p = _ep8_decode()
    plan_bm = ops.w4a16_plan(p.tokens, p.topk, p.num_experts, 2 * p.inter, p.hidden,
                             p.tok_e_hint()).block_m
    _check_pair(p, cuda_dev, plan_bm, cols_gu=_sample_cols(4096, 384, 1),
                cols_dn=_sample_cols(7168, 384, 2), what="EP8 decode")


@pytest.mark.slow
@pytest.mark.parametrize("tokens", [16, 64, 256])
def test_tp8_full_size(cuda_dev, tokens):
    p = wl.tp8(tokens)
    bm = ops.w4a16_plan(p.tokens, p.topk, p.num_experts, 2 * p.inter, p.hidden).block_m
    _check_pair(p, cuda_dev, bm, cols_gu=_sample_cols(512, 128, 3),
                cols_dn=_sample_cols(7168, 256, 4), what=f"TP8 T={tokens}")


@pytest.mark.slow
def test_ep8_prefill_full_size(cuda_dev):
    p = wl.ep8_prefill()
    bm = ops.w4a16_plan(p.tokens, p.topk, p.num_experts, 2 * p.inter, p.hidden,
                        p.tok_e_hint()).block_m
    _check_pair(p, cuda_dev, bm, cols_gu=_sample_cols(4096, 128, 5),
                cols_dn=_sample_cols(7168, 128, 6), what="EP8 prefill")


@pytest.mark.slow
@pytest.mark.parametrize("bm", [128, 256])
def test_ep8_prefill_heavy_full_size(cuda_dev, bm):
    # four times the prefill rows (tok_e 80 .. 2400): the scheduler's 128-row
    # blocks, and gate_up on 256-row blocks (items of 1, 2 or 4 issuers by
    # their rows; a plan the caller sets) with down on 128
    p = wl.ep8_prefill(scale=4)
    hint = p.tok_e_hint()
    assert ops.w4a16_plan(p.tokens, p.topk, p.num_experts, 2 * p.inter, p.hidden,
                          hint).block_m == 128
    assert ops.w4a16_plan(p.tokens, p.topk, p.num_experts, p.hidden, p.inter,
                          hint).block_m == 128
    _check_pair(p, cuda_dev, bm, cols_gu=_sample_cols(4096, 96, 7),
                cols_dn=_sample_cols(7168, 96, 8), what=f"EP8 prefill x4 bm={bm}", bm_dn=128)


@pytest.mark.slow
def test_grouped_masked_full_size(cuda_dev):
    gp = wl.grouped_masked_problem()
    got = _grouped(gp, cuda_dev)
    cols = _sample_cols(gp.n, 256, 7)
    ref = oracle.grouped_masked(gp.a, gp.layout, gp.q, gp.s, cols=cols)
    valid = ~np.isnan(ref[..., 0])
    assert_close(got[..., cols][valid], ref[valid], "masked full size")


@pytest.mark.slow
def test_grouped_contiguous_full_size_ragged(cuda_dev):
    rng = np.random.default_rng(11)
    gp = wl.grouped_contiguous_problem(rng.integers(128, 1025, size=48), seed=11)
    got = _grouped(gp, cuda_dev, _plan(128, gp.n, gp.k))
    rows = np.sort(rng.choice(gp.a.shape[0], size=384, replace=False))
    cols = _sample_cols(gp.n, 128, 12)
    ref = oracle.grouped_contiguous(gp.a[rows], gp.layout[rows], gp.q, gp.s, cols=cols)
    valid = gp.layout[rows] >= 0
    assert_close(got[rows][:, cols][valid], ref[valid], "contiguous full size")


@pytest.mark.slow
def test_grouped_masked_full_size_down_shape(cuda_dev):
    # the down projection's shape (n = hidden 7168, k = inter 2048), the
    # default plan the grouped call picks itself
    gp = wl.grouped_masked_problem(n=7168, k=2048, seed=13)
    got = _grouped(gp, cuda_dev)
    cols = _sample_cols(gp.n, 256, 14)
    ref = oracle.grouped_masked(gp.a, gp.layout, gp.q, gp.s, cols=cols)
    valid = ~np.isnan(ref[..., 0])
    assert_close(got[..., cols][valid], ref[valid], "masked full size, down shape")


@pytest.mark.slow
def test_grouped_contiguous_full_size_down_shape(cuda_dev):
    rng = np.random.default_rng(15)
    gp = wl.grouped_contiguous_problem(rng.integers(128, 1025, size=48), n=7168, k=2048,
                                       seed=15)
    plan = ops.w4a16_grouped_plan(ops.W4A16_GROUPED_CONTIGUOUS, gp.a.shape[0], gp.n, gp.k,
                                  expected_m=gp.expected_m)
    assert plan.block_m == 128
    got = _grouped(gp, cuda_dev, plan)
    rows = np.sort(rng.choice(gp.a.shape[0], size=384, replace=False))
    cols = _sample_cols(gp.n, 128, 16)
    ref = oracle.grouped_contiguous(gp.a[rows], gp.layout[rows], gp.q, gp.s, cols=cols)
    valid = gp.layout[rows] >= 0
    assert_close(got[rows][:, cols][valid], ref[valid], "contiguous full size, down shape")


# ------------------------------------------------------------- CTA pairs --
# Pairs of CTAs (2-CTA clusters) issue M = 256 MMAs over two weight tiles, each
# CTA holding one tile's dequantised rows and half of the block's token rows.

@pytest.mark.parametrize("bm", [32, 64, 128])
def test_pair_tiny_matches_oracle(cuda_dev, bm):
    _check_pair(wl.tiny(seed=71), cuda_dev, bm, what=f"pair tiny bm={bm}", cta_pair=True)


@pytest.mark.parametrize("tokens,hidden,inter,experts,topk,bm", [
    (200, 320, 224, 6, 2, 64),   # gate_up 4 tiles (last one ragged); down 3 tiles: unpaired
    (37, 96, 96, 5, 3, 32),      # k = 32 mod 64; 2 tiles / 1 tile (unpaired)
    (5, 64, 32, 40, 4, 32),      # many empty experts
])
def test_pair_ragged_shapes(cuda_dev, tokens, hidden, inter, experts, topk, bm):
    p = wl.uniform_problem(tokens, hidden, inter, experts, topk, seed=tokens + 1)
    _check_pair(p, cuda_dev, bm, what=f"pair ragged {tokens}x{hidden}x{inter}", cta_pair=True)


@pytest.mark.parametrize("bm", [32, 64])
def test_pair_is_bitwise_the_unpaired_result(cuda_dev, bm):
    # the pair MMA forms every output element from the same K slices in the
    # same order as the one-CTA MMA: the bits agree
    p = wl.uniform_problem(96, 512, 256, 8, 2, seed=72)
    pk = _pack(p.q_gu, p.s_gu, cuda_dev)
    routing = _routing(p.topk_ids, p.num_experts, bm, cuda_dev)
    g1 = _gate_up(p, pk, routing, _plan(bm, 2 * p.inter, p.hidden), cuda_dev)
    g2 = _gate_up(p, pk, routing, _plan(bm, 2 * p.inter, p.hidden, pair=True), cuda_dev)
    routed = _routed(p)
    np.testing.assert_array_equal(bf16_bits(g2)[routed], bf16_bits(g1)[routed])


def test_pair_refuses_block_not_multiple_of_32(cuda_dev):
    p = wl.tiny(seed=73)
    pk = _pack(p.q_gu, p.s_gu, cuda_dev)
    routing = _routing(p.topk_ids, p.num_experts, 16, cuda_dev)
    with pytest.raises(ops.W4A16Error) as ei:
        _gate_up(p, pk, routing, _plan(16, 2 * p.inter, p.hidden, pair=True), cuda_dev)
    assert ei.value.status == ops.W4A16_ERR_INVALID_ARG


@pytest.mark.parametrize("kind", ["contiguous", "masked"])
def test_pair_grouped_matches_oracle(cuda_dev, kind):
    if kind == "contiguous":
        gp = wl.grouped_contiguous_problem([5, 128, 0, 77], num_experts=4, n=256, k=96, seed=74)
        got = _grouped(gp, cuda_dev, _plan(32, gp.n, gp.k, pair=True))
        ref = oracle.grouped_contiguous(gp.a, gp.layout, gp.q, gp.s)
        valid = gp.layout >= 0
    else:
        gp = wl.grouped_masked_problem(num_experts=6, max_m=32, n=256, k=160, seed=75)
        gp.layout[2] = 0
        gp.layout[3] = 32
        got = _grouped(gp, cuda_dev, _plan(32, gp.n, gp.k, pair=True))
        ref = oracle.grouped_masked(gp.a, gp.layout, gp.q, gp.s)
        valid = ~np.isnan(ref[..., 0])
    assert_close(got[valid], ref[valid], f"pair grouped {kind}")
