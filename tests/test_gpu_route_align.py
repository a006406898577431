"""The fused routing front end (w4a16_moe_route_align: top-k and
moe_align_block_size in one launch) against the oracle's top-k and
alignment, and the whole layer from router logits captured in one CUDA
graph against the oracle's layer on the oracle's routing."""

import numpy as np
import pytest
import torch

import oracle
from w4a16_int4_moe_gb300 import moe as moe_mod
from w4a16_int4_moe_gb300 import ops
from w4a16_int4_moe_gb300 import workloads as wl
from helpers import assert_close, bf16_tensor, dev

pytestmark = pytest.mark.gpu


def _route_align(lg_t, lg_ref, topk, renorm, offset, local, block_m, device, capacity=None):
    """Two calls on one counter (it must come back to zero), both checked
    bit-exact against oracle.topk_softmax followed by oracle.moe_align_block_size."""
    tokens = lg_t.shape[0]
    if capacity is None:
        capacity = ops.w4a16_align_capacity(tokens * topk, local, block_m)
    arrivals = torch.zeros(1, dtype=torch.int32, device=device)
    rid, rw = oracle.topk_softmax(lg_ref, topk, renorm, offset, local)
    rs, re_, rn = oracle.moe_align_block_size(rid, local, block_m, capacity)
    for _ in range(2):
        ids, w, s, e, n = ops.w4a16_moe_route_align(lg_t, topk, block_m, arrivals, renorm,
                                                    offset, local, capacity)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ids.cpu().numpy(), rid)
        np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=1e-5, atol=1e-8)
        np.testing.assert_array_equal(s.cpu().numpy(), rs)
        np.testing.assert_array_equal(e.cpu().numpy(), re_)
        np.testing.assert_array_equal(n.cpu().numpy(), rn)
        assert int(arrivals.item()) == 0
    return ids, w


@pytest.mark.parametrize("tokens,experts,topk,offset,local,block_m", [
    (64, 16, 2, 0, 16, 16),           # tiny-sized layer, one CTA
    (576, 384, 8, 96, 48, 16),        # EP8 decode shard of a top-8-of-384 router
    (16, 384, 8, 0, 384, 16),         # TP8 single instance, T = 16 / 64 / 256
    (64, 384, 8, 0, 384, 16),
    (256, 384, 8, 0, 384, 16),
    (8192, 384, 8, 48, 48, 128),      # EP8 prefill: every SM routes, one CTA aligns
    (1000, 1024, 32, 100, 500, 64),   # the largest expert and top-k counts
    (33, 64, 4, 0, 64, 1),
    (0, 384, 8, 0, 384, 16),          # no tokens: empty routing, sentinel tail
])
def test_route_align_matches_oracle(cuda_dev, tokens, experts, topk, offset, local, block_m):
    rng = np.random.default_rng(tokens * 7 + experts)
    lg = rng.standard_normal((tokens, experts)).astype(np.float32)
    # two spare blocks: the tail past the padded total must hold the sentinel
    cap = ops.w4a16_align_capacity(tokens * topk, local, block_m) + 2 * block_m
    _route_align(dev(lg, cuda_dev), lg, topk, True, offset, local, block_m, cuda_dev, cap)


def test_route_align_bf16_ties_masked_and_unnormalised(cuda_dev):
    # coarse BF16 logits tie often (lower id wins); -inf logits mask experts,
    # leaving id -1 / weight 0 slots; over-allocated capacity keeps its tail
    rng = np.random.default_rng(11)
    lg = np.clip(np.round(rng.standard_normal((300, 96)) * 4) / 4, -2, 2).astype(np.float32)
    for t in range(0, 300, 7):
        lg[t, rng.choice(96, size=90, replace=False)] = -np.inf
    bits = wl.to_bf16_bits(lg)
    ref = oracle.bf16_bits_to_f64(bits)
    for renorm in (True, False):
        _route_align(bf16_tensor(bits, cuda_dev), ref, 8, renorm, 32, 32, 32, cuda_dev,
                     capacity=32 * 200)


def test_route_align_refuses_bad_arguments(cuda_dev):
    lg = torch.zeros((4, 64), device=cuda_dev)
    arrivals = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    with pytest.raises(ops.W4A16Error) as ei:      # capacity below the bound
        ops.w4a16_moe_route_align(lg, 8, 16, arrivals, capacity=16)
    assert ei.value.status == ops.W4A16_ERR_INVALID_ARG
    with pytest.raises(ops.W4A16Error) as ei:      # capacity not a multiple of block_m
        ops.w4a16_moe_route_align(lg, 8, 16, arrivals, capacity=16 * 40 + 8)
    assert ei.value.status == ops.W4A16_ERR_INVALID_ARG
    with pytest.raises(ops.W4A16Error) as ei:
        ops.w4a16_moe_route_align(torch.zeros((4, 1025), device=cuda_dev), 8, 16, arrivals)
    assert ei.value.status == ops.W4A16_ERR_UNSUPPORTED


def _layer_problem(maker):
    if maker == "tiny":
        p = wl.tiny(seed=91)
        glob, offset = 32, 8                 # this GPU holds global experts 8..15
    else:
        # long down reduction (inter 1024): the layer runs as one launch
        p = wl.uniform_problem(40, 512, 1024, 6, 4, seed=92)
        glob, offset = 24, 12
    rng = np.random.default_rng(93)
    logits = rng.standard_normal((p.tokens, glob)).astype(np.float32)
    return p, logits, offset


@pytest.mark.parametrize("maker,single", [("tiny", False), ("tiny", True), ("long", True)])
def test_layer_from_logits_in_one_graph(cuda_dev, maker, single):
    # route + align (one launch) -> gate_up (fused activation) -> down,
    # captured once and replayed, equals the oracle's layer on the oracle's
    # routing of the same logits
    p, logits, offset = _layer_problem(maker)
    gu = moe_mod.PackedExperts.from_checkpoint(dev(p.q_gu, cuda_dev),
                                               dev(p.s_gu.view(np.int16), cuda_dev),
                                               layout=ops.W4A16_LAYOUT_KTILE64_GLU16)
    dn = moe_mod.PackedExperts.from_checkpoint(dev(p.q_dn, cuda_dev),
                                               dev(p.s_dn.view(np.int16), cuda_dev))
    layer = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, device=cuda_dev, single_launch=single)
    x = bf16_tensor(p.x, cuda_dev)
    lg = dev(logits, cuda_dev)
    out = torch.empty((p.tokens, p.hidden), dtype=torch.float32, device=cuda_dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward_from_logits(x, lg, expert_offset=offset, out=out)   # warm-up
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.forward_from_logits(x, lg, expert_offset=offset, out=out)
    rid, rw = oracle.topk_softmax(logits, p.topk, True, offset, p.num_experts)
    _, _, _, y_ref = oracle.moe_layer(p.x, rid, rw, p.q_gu, p.s_gu, p.q_dn, p.s_dn)
    for _ in range(2):                       # replays reuse the arrival counter
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(layer._route_ids[: p.tokens].cpu().numpy(), rid)
        assert_close(out.cpu().numpy(), y_ref, f"{maker}: graph layer vs oracle")
