"""moe_align_block_size on the GPU against the oracle: bit-exact."""

import numpy as np
import pytest
import torch

import oracle
from w4a16_int4_moe_gb300 import ops
from w4a16_int4_moe_gb300 import workloads as wl
from helpers import dev

pytestmark = pytest.mark.gpu


def _check(ids, experts, bm, device, capacity=None):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    numel = ids.size
    cap = capacity or ops.w4a16_align_capacity(numel, experts, bm)
    s, e, n = ops.w4a16_moe_align_block_size(dev(ids, device), experts, bm, cap)
    torch.cuda.synchronize()
    rs, re_, rn = oracle.moe_align_block_size(ids, experts, bm, cap)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    np.testing.assert_array_equal(e.cpu().numpy(), re_)
    np.testing.assert_array_equal(n.cpu().numpy(), rn)


@pytest.mark.parametrize("bm", [16, 32, 64, 128, 256])
def test_align_tiny_and_decode(cuda_dev, bm):
    _check(wl.tiny().topk_ids, 8, bm, cuda_dev)
    _check(wl.ep8_decode().topk_ids, 48, bm, cuda_dev)


@pytest.mark.parametrize("tokens", [16, 64, 256])
def test_align_tp8(cuda_dev, tokens):
    rng = np.random.default_rng(tokens)
    ids = np.argsort(rng.random((tokens, 384)), axis=1)[:, :8]
    _check(ids, 384, 16, cuda_dev)


def test_align_prefill(cuda_dev):
    counts = wl.ep8_prefill_counts()
    rng = np.random.default_rng(0)
    lists = [rng.choice(8192, size=int(c), replace=False) for c in counts]
    ids = np.full((8192, 8), -1, np.int32)
    fill = np.zeros(8192, np.int64)
    for e, toks in enumerate(lists):
        for t in toks:
            ids[t, fill[t]] = e
            fill[t] += 1
    for bm in (64, 128, 256):
        _check(ids, 48, bm, cuda_dev)


def test_align_edge_cases(cuda_dev):
    rng = np.random.default_rng(3)
    # non-local ids (-1 and >= E), several chunks of 1024 rows
    ids = rng.integers(-3, 20, size=(700, 3))
    _check(ids, 16, 16, cuda_dev)
    # every row on one expert (longest run), and no local row at all
    _check(np.zeros((300, 4)), 8, 32, cuda_dev)
    _check(np.full((50, 2), -1), 8, 16, cuda_dev)
    # over-allocated capacity: the tail stays sentinel / -1
    _check(rng.integers(0, 8, size=(33, 2)), 8, 16, cuda_dev, capacity=16 * 64)
    # a single routed row
    _check(np.array([[5]]), 8, 16, cuda_dev)


def test_align_is_graph_capturable(cuda_dev):
    ids = dev(wl.ep8_decode().topk_ids, cuda_dev)
    cap = ops.w4a16_align_capacity(ids.numel(), 48, 32)
    bufs = (torch.empty(cap, dtype=torch.int32, device=cuda_dev),
            torch.empty(cap // 32, dtype=torch.int32, device=cuda_dev),
            torch.empty(1, dtype=torch.int32, device=cuda_dev))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ops.w4a16_moe_align_block_size(ids, 48, 32, cap, out=bufs)   # warm-up outside capture
    torch.cuda.synchronize()
    for b in bufs:
        b.fill_(-7)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ops.w4a16_moe_align_block_size(ids, 48, 32, cap, out=bufs)
    g.replay()
    torch.cuda.synchronize()
    rs, re_, rn = oracle.moe_align_block_size(ids.cpu().numpy(), 48, 32, cap)
    np.testing.assert_array_equal(bufs[0].cpu().numpy(), rs)
    np.testing.assert_array_equal(bufs[1].cpu().numpy(), re_)
    np.testing.assert_array_equal(bufs[2].cpu().numpy(), rn)
