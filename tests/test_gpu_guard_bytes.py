"""Guard bytes around every buffer a device call writes.

Each output and workspace is a view into the middle of a larger allocation
whose head and tail hold a fixed byte pattern. After the call, both ends must
be intact: a write past either end of an output, a workspace or a routing
array would land there. The guards are 4 KB on each side, a multiple of 256
bytes, so every view keeps the alignment the calls require (16 bytes for the
tensor-map bases and the vector stores). The results inside the views must
equal those of the same call on plain tensors: bit-exact where the call is
deterministic, and up to the order of the FP32 additions otherwise.

The shapes are small and ragged, so that every kernel meets its edges:
- a reduction of 96 (one full and one half 64-k step);
- output widths of 96, 192 and 200 (partial weight tiles);
- routing blocks of 16 to 256 rows;
- tokens routed to experts that are not local.
"""

import numpy as np
import pytest
import torch

from w4a16_int4_moe_gb300 import moe as moe_mod
from w4a16_int4_moe_gb300 import ops
from w4a16_int4_moe_gb300 import workloads as wl
from helpers import Guarded, bf16_tensor, dev

pytestmark = pytest.mark.gpu


def _ws(size, device):
    return Guarded(size, torch.uint8, device, fill=0)


def _problem(inter=96, seed=91):
    # 37 tokens top-3 over 5 local experts of 6, hidden 96; inter 96 (gate_up
    # width 192: a partial weight tile), or 128 for the fused activation,
    # whose weight layout needs whole 128-row tiles
    p = wl.uniform_problem(37, 96, inter, 6, 3, seed=seed)
    p.num_experts = 5
    p.topk_ids = np.where(p.topk_ids == 5, -1, p.topk_ids).astype(np.int32)
    p.q_gu, p.s_gu = p.q_gu[:5], p.s_gu[:5]
    p.q_dn, p.s_dn = p.q_dn[:5], p.s_dn[:5]
    return p


def _plan(bm, n, k):
    p = ops.w4a16_plan(64, 1, 1, n, k, float(bm))
    p.block_m = bm
    if bm > 128:
        p.b_stages, p.stages = 4, 8
    else:
        p.b_stages, p.stages = 8, min(p.stages, 8)
    return p


@pytest.mark.parametrize("bm", [16, 64])
def test_align_block_size_writes_only_its_arrays(cuda_dev, bm):
    p = _problem()
    ids = dev(p.topk_ids, cuda_dev)
    cap = ops.w4a16_align_capacity(p.numel, p.num_experts, bm)
    s = Guarded(cap, torch.int32, cuda_dev)
    e = Guarded(cap // bm, torch.int32, cuda_dev)
    n = Guarded(1, torch.int32, cuda_dev)
    ops.w4a16_moe_align_block_size(ids, p.num_experts, bm, cap, out=(s.t, e.t, n.t))
    for g, what in ((s, "sorted_ids"), (e, "expert_ids"), (n, "num_tokens_padded")):
        g.check(what)
    rs, re_, rn = ops.w4a16_moe_align_block_size(ids, p.num_experts, bm, cap)
    assert torch.equal(s.t, rs) and torch.equal(e.t, re_) and torch.equal(n.t, rn)


@pytest.mark.parametrize("layout", [ops.W4A16_LAYOUT_KTILE64, ops.W4A16_LAYOUT_KTILE64_GLU16])
def test_prepack_writes_only_its_blob(cuda_dev, layout):
    p = _problem(96 if layout == ops.W4A16_LAYOUT_KTILE64 else 128)
    q = dev(p.q_gu, cuda_dev)
    sc = dev(p.s_gu.view(np.int16), cuda_dev)
    size = ops.w4a16_prepack_size(p.num_experts, 2 * p.inter, p.hidden, layout=layout)
    out = Guarded(size, torch.uint8, cuda_dev)
    ops.w4a16_prepack(q, sc, layout=layout, out=out.t)
    out.check("packed weights")
    assert torch.equal(out.t, ops.w4a16_prepack(q, sc, layout=layout))


def _indexed_pair(p, plan_gu, plan_dn, device, what, deterministic=True):
    """gate_up, then down on silu_and_mul of it, into guarded outputs and
    workspaces; each against the same call on plain tensors."""
    pk_gu = ops.w4a16_prepack(dev(p.q_gu, device), dev(p.s_gu.view(np.int16), device))
    pk_dn = ops.w4a16_prepack(dev(p.q_dn, device), dev(p.s_dn.view(np.int16), device))
    ids = dev(p.topk_ids, device)
    x = bf16_tensor(p.x, device)
    w = dev(p.topk_weights, device)
    n_gu, k_gu, n_dn, k_dn = 2 * p.inter, p.hidden, p.hidden, p.inter

    # gate_up: BF16 rows at their routing positions
    cap = ops.w4a16_align_capacity(p.numel, p.num_experts, plan_gu.block_m)
    sid, eid, ntp = ops.w4a16_moe_align_block_size(ids, p.num_experts, plan_gu.block_m, cap)
    ws = _ws(ops.w4a16_workspace_size(plan_gu, cap, k_gu), device)
    out = Guarded((p.numel, n_gu), torch.bfloat16, device, fill=0.0)
    ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, pk_gu, p.num_experts, n_gu, k_gu, x,
                               p.tokens, p.topk, sid, eid, ntp, plan_gu, ws.t, out=out.t)
    out.check(f"{what}: gate_up output")
    ws.check(f"{what}: gate_up workspace")
    assert ops.w4a16_read_device_status(ws.t)[0] == ops.W4A16_OK
    ref = torch.zeros((p.numel, n_gu), dtype=torch.bfloat16, device=device)
    ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, pk_gu, p.num_experts, n_gu, k_gu, x,
                               p.tokens, p.topk, sid, eid, ntp, plan_gu,
                               ops.new_workspace(plan_gu, device, cap, k_gu), out=ref)
    assert torch.equal(out.t.view(torch.int16), ref.view(torch.int16))
    del out, ws

    # down: the top-k weighted FP32 adds into the token rows
    act = ops.w4a16_silu_and_mul(ref)
    del ref
    cap = ops.w4a16_align_capacity(p.numel, p.num_experts, plan_dn.block_m)
    sid, eid, ntp = ops.w4a16_moe_align_block_size(ids, p.num_experts, plan_dn.block_m, cap)
    ws = _ws(ops.w4a16_workspace_size(plan_dn, cap, k_dn), device)
    out = Guarded((p.tokens, n_dn), torch.float32, device, fill=float("nan"))
    ops.w4a16_moe_indexed_gemm(ops.W4A16_DOWN, pk_dn, p.num_experts, n_dn, k_dn, act,
                               p.tokens, p.topk, sid, eid, ntp, plan_dn, ws.t, topk_weights=w,
                               out=out.t)
    out.check(f"{what}: down output")
    ws.check(f"{what}: down workspace")
    assert ops.w4a16_read_device_status(ws.t)[0] == ops.W4A16_OK
    y = ops.w4a16_moe_indexed_gemm(ops.W4A16_DOWN, pk_dn, p.num_experts, n_dn, k_dn, act,
                                   p.tokens, p.topk, sid, eid, ntp, plan_dn,
                                   ops.new_workspace(plan_dn, device, cap, k_dn), topk_weights=w)
    torch.testing.assert_close(out.t, y, rtol=1e-5, atol=1e-5)
    if not deterministic:
        return

    # the deterministic down pass: rows parked in the workspace, then summed
    size = (ops.w4a16_workspace_size(plan_dn, cap, k_dn)
            + ops.w4a16_deterministic_bytes(cap, n_dn, p.numel))
    ws = _ws(size, device)
    out = Guarded((p.tokens, n_dn), torch.float32, device, fill=float("nan"))
    ops.w4a16_moe_indexed_gemm(ops.W4A16_DOWN, pk_dn, p.num_experts, n_dn, k_dn, act,
                               p.tokens, p.topk, sid, eid, ntp, plan_dn, ws.t, topk_weights=w,
                               out=out.t, flags=ops.W4A16_FLAG_DETERMINISTIC)
    out.check(f"{what}: deterministic down output")
    ws.check(f"{what}: deterministic down workspace")
    torch.testing.assert_close(out.t, y, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("bm", [16, 32, 64, 128, 256])
def test_indexed_gemms_write_only_their_outputs(cuda_dev, bm):
    p = _problem()
    _indexed_pair(p, _plan(bm, 2 * p.inter, p.hidden), _plan(bm, p.hidden, p.inter), cuda_dev,
                  f"bm={bm}")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["ep8_decode", "tp8_64", "ep8_prefill", "ep8_prefill_x4"])
def test_full_size_shards_write_only_their_outputs(cuda_dev, name):
    # the shard shapes in the plans the scheduler gives them (block_m 32, 16,
    # 64 and 128; the long gate_up reductions of the prefill shards take the
    # rastered item order, the four-times shard's gate_up the BF16 staging)
    if name == "ep8_decode":
        p = wl.ep8_decode()
    elif name == "tp8_64":
        p = wl.tp8(64)
    else:
        p = wl.ep8_prefill(scale=4 if name.endswith("x4") else 1)
    hint = p.tok_e_hint()
    plan_gu = ops.w4a16_plan(p.tokens, p.topk, p.num_experts, 2 * p.inter, p.hidden, hint)
    plan_dn = ops.w4a16_plan(p.tokens, p.topk, p.num_experts, p.hidden, p.inter, hint)
    _indexed_pair(p, plan_gu, plan_dn, cuda_dev, name, deterministic=False)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("bm", [32, 128])
def test_fused_activation_writes_only_its_output(cuda_dev, bm):
    p = _problem(128, seed=96)
    glu = ops.w4a16_prepack(dev(p.q_gu, cuda_dev), dev(p.s_gu.view(np.int16), cuda_dev),
                            layout=ops.W4A16_LAYOUT_KTILE64_GLU16)
    ids = dev(p.topk_ids, cuda_dev)
    cap = ops.w4a16_align_capacity(p.numel, p.num_experts, bm)
    sid, eid, ntp = ops.w4a16_moe_align_block_size(ids, p.num_experts, bm, cap)
    x = bf16_tensor(p.x, cuda_dev)
    plan = _plan(bm, 2 * p.inter, p.hidden)
    plan.layout = ops.W4A16_LAYOUT_KTILE64_GLU16
    ws = _ws(ops.w4a16_workspace_size(plan, cap, p.hidden), cuda_dev)
    out = Guarded((p.numel, p.inter), torch.bfloat16, cuda_dev, fill=0.0)
    ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP_SILU, glu, p.num_experts, 2 * p.inter,
                               p.hidden, x, p.tokens, p.topk, sid, eid, ntp, plan, ws.t,
                               out=out.t)
    out.check(f"fused activation output bm={bm}")
    ws.check(f"fused activation workspace bm={bm}")
    ref = torch.zeros((p.numel, p.inter), dtype=torch.bfloat16, device=cuda_dev)
    ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP_SILU, glu, p.num_experts, 2 * p.inter,
                               p.hidden, x, p.tokens, p.topk, sid, eid, ntp, plan,
                               ops.new_workspace(plan, cuda_dev, cap, p.hidden), out=ref)
    assert torch.equal(out.t.view(torch.int16), ref.view(torch.int16))


def test_silu_and_mul_writes_only_its_output(cuda_dev):
    rng = np.random.default_rng(92)
    x = bf16_tensor(wl.random_activations(rng, 37, 2 * 96), cuda_dev)
    out = Guarded((37, 96), torch.bfloat16, cuda_dev)
    ops.w4a16_silu_and_mul(x, out=out.t)
    out.check("silu_and_mul output")
    assert torch.equal(out.t.view(torch.int16), ops.w4a16_silu_and_mul(x).view(torch.int16))


@pytest.mark.parametrize("kind,bm", [("contiguous", 32), ("contiguous", 64),
                                     ("contiguous", 128), ("masked", 16), ("masked", 32)])
def test_grouped_gemms_write_only_their_outputs(cuda_dev, kind, bm):
    if kind == "contiguous":
        gp = wl.grouped_contiguous_problem([5, 128, 0, 77], num_experts=4, n=200, k=96,
                                           seed=93 + bm)
    else:
        gp = wl.grouped_masked_problem(num_experts=6, max_m=32, n=200, k=96, seed=94 + bm)
        gp.layout[2] = 0
        gp.layout[5] = 32     # the last expert's full budget ends at the buffer's end
    pk = ops.w4a16_prepack(dev(gp.q, cuda_dev), dev(gp.s.view(np.int16), cuda_dev))
    a = bf16_tensor(gp.a, cuda_dev)
    lay = dev(gp.layout, cuda_dev)
    contiguous = kind == "contiguous"
    code = ops.W4A16_GROUPED_CONTIGUOUS if contiguous else ops.W4A16_GROUPED_MASKED
    m = gp.a.shape[0] if contiguous else gp.a.shape[1]
    shape = (m, gp.n) if contiguous else (gp.num_experts, m, gp.n)
    plan = _plan(bm, gp.n, gp.k)
    ws = _ws(ops.w4a16_workspace_size(plan), cuda_dev)
    out = Guarded(shape, torch.bfloat16, cuda_dev, fill=0.0)
    ops.w4a16_moe_grouped_gemm(code, pk, gp.num_experts, gp.n, gp.k, a, m, lay, ws.t,
                               plan=plan, expected_m=gp.expected_m, out=out.t)
    out.check(f"{kind} output bm={bm}")
    ws.check(f"{kind} workspace bm={bm}")
    assert ops.w4a16_read_device_status(ws.t)[0] == ops.W4A16_OK
    ref = torch.zeros(shape, dtype=torch.bfloat16, device=cuda_dev)
    ops.w4a16_moe_grouped_gemm(code, pk, gp.num_experts, gp.n, gp.k, a, m, lay,
                               ops.new_workspace(plan, cuda_dev), plan=plan,
                               expected_m=gp.expected_m, out=ref)
    assert torch.equal(out.t.view(torch.int16), ref.view(torch.int16))


def test_single_launch_layer_writes_only_its_output(cuda_dev):
    p = wl.uniform_problem(77, 320, 192, 6, 3, seed=97)
    p.topk_ids[::5, 0] = -1

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(cuda_dev)

    gu = moe_mod.PackedExperts.from_checkpoint(t(p.q_gu), t(p.s_gu.view(np.int16)),
                                               layout=ops.W4A16_LAYOUT_KTILE64_GLU16)
    dn = moe_mod.PackedExperts.from_checkpoint(t(p.q_dn), t(p.s_dn.view(np.int16)))
    one = moe_mod.W4A16MoE(gu, dn, p.topk, p.tokens, device=cuda_dev, single_launch=True)
    x, ids, w = bf16_tensor(p.x, cuda_dev), t(p.topk_ids), t(p.topk_weights)
    y = one.forward(x, ids, w)
    torch.cuda.synchronize()
    ws = _ws(ops.w4a16_layer_workspace_size(one.plan_gu, one.capacity, one.hidden, one.inter),
             cuda_dev)
    out = Guarded((p.tokens, p.hidden), torch.float32, cuda_dev, fill=float("nan"))
    ops.w4a16_moe_layer(gu.packed, dn.packed, one.num_experts, one.hidden, one.inter, x,
                        p.tokens, p.topk, one.sorted_ids, one.expert_ids, one.ntp, one.plan_gu,
                        ws.t, w, out=out.t)
    out.check("layer output")
    ws.check("layer workspace")
    assert ops.w4a16_read_device_status(ws.t)[0] == ops.W4A16_OK
    torch.testing.assert_close(out.t, y, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("tokens,experts,topk,offset,local,block_m", [
    (37, 16, 3, 0, 16, 16),
    (37, 64, 8, 16, 24, 64),
])
def test_routing_front_end_writes_only_its_outputs(cuda_dev, tokens, experts, topk, offset,
                                                   local, block_m):
    rng = np.random.default_rng(95 + experts)
    lg = dev(rng.standard_normal((tokens, experts)).astype(np.float32), cuda_dev)
    ids = Guarded((tokens, topk), torch.int32, cuda_dev)
    wts = Guarded((tokens, topk), torch.float32, cuda_dev)
    ops.w4a16_topk_softmax(lg, topk, True, offset, local, out=(ids.t, wts.t))
    ids.check("top-k ids")
    wts.check("top-k weights")
    rid, rw = ops.w4a16_topk_softmax(lg, topk, True, offset, local)
    assert torch.equal(ids.t, rid) and torch.equal(wts.t, rw)

    cap = ops.w4a16_align_capacity(tokens * topk, local, block_m)
    outs = (Guarded((tokens, topk), torch.int32, cuda_dev),
            Guarded((tokens, topk), torch.float32, cuda_dev),
            Guarded(cap, torch.int32, cuda_dev),
            Guarded(cap // block_m, torch.int32, cuda_dev),
            Guarded(1, torch.int32, cuda_dev))
    arrivals = Guarded(1, torch.int32, cuda_dev, fill=0)
    ops.w4a16_moe_route_align(lg, topk, block_m, arrivals.t, True, offset, local, cap,
                              out=tuple(g.t for g in outs))
    names = ("ids", "weights", "sorted_ids", "expert_ids", "num_tokens_padded")
    for g, what in zip(outs, names):
        g.check(f"route_align {what}")
    arrivals.check("route_align arrival counter")
    assert int(arrivals.t.item()) == 0
    ref = ops.w4a16_moe_route_align(lg, topk, block_m,
                                    torch.zeros(1, dtype=torch.int32, device=cuda_dev), True,
                                    offset, local, cap)
    for g, r, what in zip(outs, ref, names):
        assert torch.equal(g.t, r), what


def test_noalloc_entry_writes_only_its_output(cuda_dev):
    p = _problem()
    pk = ops.w4a16_prepack(dev(p.q_gu, cuda_dev), dev(p.s_gu.view(np.int16), cuda_dev))
    ids = dev(p.topk_ids, cuda_dev)
    cap = ops.w4a16_align_capacity(p.numel, p.num_experts, 32)
    sid, eid, ntp = ops.w4a16_moe_align_block_size(ids, p.num_experts, 32, cap)
    x = bf16_tensor(p.x, cuda_dev)
    plan = _plan(32, 2 * p.inter, p.hidden)
    out = Guarded((p.numel, 2 * p.inter), torch.bfloat16, cuda_dev, fill=0.0)
    ops.w4a16_moe_indexed_gemm_noalloc(ops.W4A16_GATE_UP, pk, p.num_experts, 2 * p.inter,
                                       p.hidden, x, p.tokens, p.topk, sid, eid, ntp, plan,
                                       out=out.t)
    out.check("no-alloc gate_up output")
    ref = torch.zeros((p.numel, 2 * p.inter), dtype=torch.bfloat16, device=cuda_dev)
    ops.w4a16_moe_indexed_gemm(ops.W4A16_GATE_UP, pk, p.num_experts, 2 * p.inter, p.hidden, x,
                               p.tokens, p.topk, sid, eid, ntp, plan,
                               ops.new_workspace(plan, cuda_dev, cap, p.hidden), out=ref)
    assert torch.equal(out.t.view(torch.int16), ref.view(torch.int16))
