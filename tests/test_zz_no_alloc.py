"""The no-allocation GEMM entry point, for callers that cannot allocate
device memory at call time (an allocator that owns all device memory, code
that must not allocate after start-up, a plugin interface that passes only
the operation's tensors).

It must give the same results as the workspace entry point, on consecutive
calls that share its built-in device array. This file is collected last so a
failure here comes after every other test has run; it also passes on its own
in a fresh process (the first call on the device performs the set-up)."""

import numpy as np
import pytest
import torch

from w4a16_int4_moe_gb300 import ops
from w4a16_int4_moe_gb300 import workloads as wl
from helpers import assert_close, bf16_tensor, dev

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice(cuda_dev):
    p = wl.tiny(seed=31)
    q_gu, s_gu = dev(p.q_gu, cuda_dev), dev(p.s_gu.view(np.int16), cuda_dev)
    q_dn, s_dn = dev(p.q_dn, cuda_dev), dev(p.s_dn.view(np.int16), cuda_dev)
    pk_gu, pk_dn = ops.w4a16_prepack(q_gu, s_gu), ops.w4a16_prepack(q_dn, s_dn)
    plan = ops.w4a16_plan(p.tokens, p.topk, p.num_experts, 2 * p.inter, p.hidden)
    plan_dn = ops.w4a16_plan(p.tokens, p.topk, p.num_experts, p.hidden, p.inter)
    plan_dn.block_m = plan.block_m
    ids = dev(p.topk_ids, cuda_dev)
    sid, eid, ntp = ops.w4a16_moe_align_block_size(ids, p.num_experts, plan.block_m)
    x = bf16_tensor(p.x, cuda_dev)
    w = dev(p.topk_weights, cuda_dev)
    ws = ops.new_workspace(plan, cuda_dev, sid.numel(), max(p.hidden, p.inter))

    g_ref = ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, pk_gu, p.num_experts, 2 * p.inter,
                                       p.hidden, x, p.tokens, p.topk, sid, eid, ntp, plan, ws)
    act = ops.w4a16_silu_and_mul(g_ref)
    y_ref = ops.w4a16_moe_indexed_gemm(ops.W4A16_DOWN, pk_dn, p.num_experts, p.hidden, p.inter,
                                       act, p.tokens, p.topk, sid, eid, ntp, plan_dn, ws,
                                       topk_weights=w)
    torch.cuda.synchronize()
    routed = torch.from_numpy(((p.topk_ids >= 0) & (p.topk_ids < p.num_experts)).reshape(-1))

    for call in range(2):
        g = torch.zeros_like(g_ref)
        ops.w4a16_moe_indexed_gemm_noalloc(ops.W4A16_GATE_UP, pk_gu, p.num_experts, 2 * p.inter,
                                           p.hidden, x, p.tokens, p.topk, sid, eid, ntp, plan,
                                           out=g, flags=ops.W4A16_FLAG_SYNC_STATUS)
        y = torch.full_like(y_ref, float("nan"))
        ops.w4a16_moe_indexed_gemm_noalloc(ops.W4A16_DOWN, pk_dn, p.num_experts, p.hidden,
                                           p.inter, act, p.tokens, p.topk, sid, eid, ntp, plan_dn,
                                           topk_weights=w, out=y,
                                           flags=ops.W4A16_FLAG_SYNC_STATUS)
        torch.cuda.synchronize()
        assert_close(g.float().cpu().numpy()[routed.numpy()],
                     g_ref.float().cpu().numpy()[routed.numpy()], f"gate_up call {call}")
        assert_close(y.cpu().numpy(), y_ref.cpu().numpy(), f"down call {call}")


def test_noalloc_rejects_unknown_flags(cuda_dev, lib):
    import ctypes
    plan = ops.w4a16_plan(64, 2, 8, 1024, 512)
    fake = ctypes.c_void_p(1 << 20)
    # an unknown flag is refused before anything is enqueued
    assert lib.w4a16_moe_indexed_gemm_noalloc(0, fake, 8, 1024, 512, fake, 64, 2, fake, fake,
                                              fake, 256, None, fake, 64, ctypes.byref(plan),
                                              None) == ops.W4A16_ERR_INVALID_ARG
    # so is the deterministic down pass, whose row buffer needs a sized workspace
    assert lib.w4a16_moe_indexed_gemm_noalloc(ops.W4A16_DOWN, fake, 8, 1024, 512, fake, 64, 2,
                                              fake, fake, fake, 256, fake, fake,
                                              ops.W4A16_FLAG_DETERMINISTIC, ctypes.byref(plan),
                                              None) == ops.W4A16_ERR_INVALID_ARG
