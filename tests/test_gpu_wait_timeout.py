"""Failure detection without a GPU fault.

Every device-side wait of the GEMM kernel is bounded. With the bound lowered
far below the time its waits normally take (W4A16_WAIT_TIMEOUT_CYCLES), the
kernel gives up: it records which wait ran out in the workspace status word,
lets the copies and MMAs it already issued finish, frees its TMEM and exits.
The host reads W4A16_ERR_TIMEOUT, and the next call with the default bound
runs normally on the same context. Nothing here traps, faults or hangs: the
waits simply run out.
"""

import numpy as np
import pytest
import torch

import oracle
from w4a16_int4_moe_gb300 import ops
from w4a16_int4_moe_gb300 import workloads as wl
from helpers import assert_close, bf16_bits, bf16_tensor, dev

pytestmark = pytest.mark.gpu


def _run_gate_up(p, pk, routing, plan, ws, device):
    sid, eid, ntp = routing
    out = torch.zeros((p.numel, 2 * p.inter), dtype=torch.bfloat16, device=device)
    ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, pk, p.num_experts, 2 * p.inter, p.hidden,
                               bf16_tensor(p.x, device), p.tokens, p.topk, sid, eid, ntp, plan,
                               ws, out=out)
    return out


@pytest.mark.parametrize("cta_pair", [0, 1])
def test_expired_waits_are_reported_and_the_context_recovers(cuda_dev, monkeypatch, cta_pair):
    # cta_pair 1: CTA pairs, whose cross-CTA waits give up the same way
    p = wl.uniform_problem(256, 2048, 512, 8, 2, seed=41)
    pk = ops.w4a16_prepack(dev(p.q_gu, cuda_dev), dev(p.s_gu.view(np.int16), cuda_dev))
    plan = ops.w4a16_plan(p.tokens, p.topk, p.num_experts, 2 * p.inter, p.hidden)
    plan.block_m = 32
    plan.cta_pair = cta_pair
    t = dev(p.topk_ids, cuda_dev)
    routing = ops.w4a16_moe_align_block_size(t, p.num_experts, plan.block_m)
    ws = ops.new_workspace(plan, cuda_dev, routing[0].numel(), p.hidden)

    # a bound of 500 cycles runs out long before a whole item's accumulator
    # (or even the first weight copy from HBM) is ready
    monkeypatch.setenv("W4A16_WAIT_TIMEOUT_CYCLES", "500")
    _run_gate_up(p, pk, routing, plan, ws, cuda_dev)
    st, word = ops.w4a16_read_device_status(ws)
    assert st == ops.W4A16_ERR_TIMEOUT, (st, hex(word))
    assert word & 0x1000, hex(word)           # "a wait gave up", low bits: which wait
    assert 1 <= (word & 0xFF) <= 14, hex(word)

    # the status word was reset by the read; the default bound works again
    monkeypatch.delenv("W4A16_WAIT_TIMEOUT_CYCLES")
    out = _run_gate_up(p, pk, routing, plan, ws, cuda_dev)
    st, word = ops.w4a16_read_device_status(ws)
    assert st == ops.W4A16_OK, hex(word)
    routed = ((p.topk_ids >= 0) & (p.topk_ids < p.num_experts)).reshape(-1)
    ref = oracle.indexed_gate_up(p.x, p.topk_ids, p.q_gu, p.s_gu)
    got = oracle.bf16_bits_to_f64(bf16_bits(out))
    assert_close(got[routed], ref[routed], "gate_up after a timed-out call")


def test_single_launch_layer_wait_runs_out_and_recovers(cuda_dev, monkeypatch):
    # the down items of the single-launch layer wait on a per-block counter
    # raised by other CTAs: with the bound lowered, that wait (or another)
    # gives up, the call reports it, and the next call is correct
    from w4a16_int4_moe_gb300 import moe as moe_mod
    p = wl.uniform_problem(128, 1024, 256, 8, 2, seed=44)

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(cuda_dev)
    gu = moe_mod.PackedExperts.from_checkpoint(t(p.q_gu), t(p.s_gu.view(np.int16)),
                                               layout=ops.W4A16_LAYOUT_KTILE64_GLU16)
    dn = moe_mod.PackedExperts.from_checkpoint(t(p.q_dn), t(p.s_dn.view(np.int16)))
    layer = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, device=cuda_dev, single_launch=True)
    x, ids, w = bf16_tensor(p.x, cuda_dev), t(p.topk_ids), t(p.topk_weights)
    monkeypatch.setenv("W4A16_WAIT_TIMEOUT_CYCLES", "500")
    layer.forward(x, ids, w)
    st, word = ops.w4a16_read_device_status(layer.layer_workspace)
    assert st == ops.W4A16_ERR_TIMEOUT, (st, hex(word))
    assert word & 0x1000 and 1 <= (word & 0xFF) <= 15, hex(word)
    monkeypatch.delenv("W4A16_WAIT_TIMEOUT_CYCLES")
    y = layer.forward(x, ids, w)
    st, word = ops.w4a16_read_device_status(layer.layer_workspace)
    assert st == ops.W4A16_OK, hex(word)
    ref = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, device=cuda_dev).forward(x, ids, w)
    assert_close(y.cpu().numpy(), ref.cpu().numpy(), "layer after a timed-out call",
                 rel_l2=1e-6, max_abs_frac=1e-5)
