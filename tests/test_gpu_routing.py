"""The routing front end on the GPU (w4a16_topk_softmax) against the oracle:
the chosen experts (ids, local mapping, order) bit-exact, the weights within
FP32 rounding of the float64 softmax."""

import numpy as np
import pytest
import torch

import oracle
from w4a16_int4_moe_gb300 import moe as moe_mod
from w4a16_int4_moe_gb300 import ops
from w4a16_int4_moe_gb300 import workloads as wl
from helpers import assert_close, bf16_tensor

pytestmark = pytest.mark.gpu


def _check(logits_t, logits_f64, topk, renorm, offset, local):
    ids, w = ops.w4a16_topk_softmax(logits_t, topk, renorm, offset, local)
    rid, rw = oracle.topk_softmax(logits_f64, topk, renorm, offset, local)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=1e-5, atol=1e-8)


@pytest.mark.parametrize("tokens,experts,topk,renorm,offset,local", [
    (257, 384, 8, True, 48, 48),      # EP8 rank 1 of Kimi-like routing
    (64, 384, 8, True, 0, 384),       # TP8: every expert local
    (33, 256, 6, False, 0, 256),
    (5, 1024, 32, True, 100, 500),    # the largest supported sizes
    (9, 7, 7, False, 0, 7),           # k = all experts: plain softmax order
    (0, 384, 8, True, 0, 384),        # no tokens
])
def test_topk_softmax_fp32(cuda_dev, tokens, experts, topk, renorm, offset, local):
    rng = np.random.default_rng(tokens + experts)
    lg = rng.standard_normal((tokens, experts)).astype(np.float32)
    _check(torch.from_numpy(lg).to(cuda_dev), lg, topk, renorm, offset, local)


def test_topk_softmax_bf16_ties(cuda_dev):
    # coarse BF16 logits (quarters in [-2, 2]) tie often: lower id must win
    rng = np.random.default_rng(3)
    lg = np.round(rng.standard_normal((300, 384)) * 4) / 4
    lg = np.clip(lg, -2, 2).astype(np.float32)
    bits = wl.to_bf16_bits(lg)
    _check(bf16_tensor(bits, cuda_dev), oracle.bf16_bits_to_f64(bits), 8, True, 0, 384)


def test_topk_softmax_masked_experts(cuda_dev):
    # -inf logits mask experts; rows with fewer than k unmasked experts get
    # id -1 and weight 0 in the remaining slots, also when every expert is masked
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((40, 64)).astype(np.float32)
    for t in range(40):
        keep = rng.choice(64, size=t % 12, replace=False)   # 0..11 experts left
        row = np.full(64, -np.inf, dtype=np.float32)
        row[keep] = lg[t, keep]
        lg[t] = row
    for renorm in (True, False):
        _check(torch.from_numpy(lg).to(cuda_dev), lg, 8, renorm, 0, 64)


def test_unsupported_sizes_are_refused(cuda_dev):
    lg = torch.zeros((4, 1025), device=cuda_dev)
    with pytest.raises(ops.W4A16Error) as ei:
        ops.w4a16_topk_softmax(lg, 8)
    assert ei.value.status == ops.W4A16_ERR_UNSUPPORTED
    with pytest.raises(ops.W4A16Error):
        ops.w4a16_topk_softmax(torch.zeros((4, 64), device=cuda_dev), 33)


def test_layer_from_router_logits(cuda_dev):
    # route -> align -> gate_up -> act -> down on the device equals the layer
    # fed with the oracle's routing
    p = wl.tiny(seed=61)
    rng = np.random.default_rng(62)
    logits = rng.standard_normal((p.tokens, 32)).astype(np.float32)   # 32 global experts
    offset = 8                                                        # this GPU: 8..15

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(cuda_dev)

    gu = moe_mod.PackedExperts.from_checkpoint(t(p.q_gu), t(p.s_gu.view(np.int16)))
    dn = moe_mod.PackedExperts.from_checkpoint(t(p.q_dn), t(p.s_dn.view(np.int16)))
    layer = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, device=cuda_dev)
    x = bf16_tensor(p.x, cuda_dev)
    y = layer.forward_from_logits(x, t(logits), expert_offset=offset)
    rid, rw = oracle.topk_softmax(logits, p.topk, True, offset, p.num_experts)
    layer2 = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, device=cuda_dev)
    y2 = layer2.forward(x, t(rid), t(rw.astype(np.float32)))
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), y2.cpu().numpy(), "layer from logits", rel_l2=1e-5,
                 max_abs_frac=1e-5)
