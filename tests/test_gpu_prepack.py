"""Prepack round trip on the GPU: unpack(prepack(q, s)) reproduces the
checkpoint bytes exactly, including ragged n and k = 32 (mod 64)."""

import numpy as np
import pytest
import torch

from w4a16_int4_moe_gb300 import ops
from w4a16_int4_moe_gb300 import workloads as wl
from helpers import dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("e,n,k", [(1, 128, 64), (3, 130, 96), (2, 1024, 512), (4, 7, 32),
                                   (2, 4096, 7168)])
def test_prepack_round_trip(cuda_dev, e, n, k):
    rng = np.random.default_rng(e * 1000 + n + k)
    q, s = wl.random_weights(rng, e, n, k)
    packed = ops.w4a16_prepack(dev(q, cuda_dev), dev(s.view(np.int16), cuda_dev))
    assert packed.numel() == ops.w4a16_prepack_size(e, n, k)
    q2, s2 = ops.w4a16_unpack(packed, e, n, k)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q2.cpu().numpy(), q)
    np.testing.assert_array_equal(s2.cpu().numpy().view(np.uint16), s)


def test_prepack_padding_is_zero_weight(cuda_dev):
    # rows past n and k past k carry code 8 (0x88 bytes) and scale 0
    rng = np.random.default_rng(5)
    q, s = wl.random_weights(rng, 1, 130, 96)
    packed = ops.w4a16_prepack(dev(q, cuda_dev), dev(s.view(np.int16), cuda_dev)).cpu().numpy()
    step = 4608
    tiles, ksteps = 2, 2
    blob = packed.reshape(1, tiles, ksteps, step)
    # tile 1 holds rows 128..255: rows 2.. are padding
    qpart = blob[0, 1, 0, :4096].reshape(2, 128, 16)
    assert np.all(qpart[:, 2:, :] == 0x88)
    spart = blob[0, 1, 0, 4096:].view(np.uint16).reshape(2, 128)
    assert np.all(spart[:, 2:] == 0)
    # k step 1 covers k = 64..127; k = 96..127 (group 1) is padding
    q_step1 = blob[0, 0, 1, :4096].reshape(2, 128, 16)
    assert np.all(q_step1[1] == 0x88)
    assert np.all(blob[0, 0, 1, 4096:].view(np.uint16).reshape(2, 128)[1] == 0)


@pytest.mark.parametrize("e,n,k", [(2, 256, 96), (3, 1024, 512), (1, 512, 7168)])
def test_glu16_layout_round_trip_and_row_order(cuda_dev, e, n, k):
    # gate_up weights [n = 2I, k]: tile t of the interleaved layout holds, per
    # 32-row quarter q, gate rows 64t+16q..+15 then up rows I+64t+16q..+15
    rng = np.random.default_rng(n + k)
    q, s = wl.random_weights(rng, e, n, k)
    glu = ops.W4A16_LAYOUT_KTILE64_GLU16
    packed = ops.w4a16_prepack(dev(q, cuda_dev), dev(s.view(np.int16), cuda_dev), layout=glu)
    assert packed.numel() == ops.w4a16_prepack_size(e, n, k)
    q2, s2 = ops.w4a16_unpack(packed, e, n, k, layout=glu)
    np.testing.assert_array_equal(q2.cpu().numpy(), q)
    np.testing.assert_array_equal(s2.cpu().numpy().view(np.uint16), s)
    # read back as if it were the plain layout: row r of tile t is the source
    # row the interleaving names
    q3, _ = ops.w4a16_unpack(packed, e, n, k)
    half = n // 2
    t, r = np.divmod(np.arange(n), 128)
    quarter, i = np.divmod(r, 32)
    col = 64 * t + 16 * quarter + (i % 16)
    src = np.where(i < 16, col, half + col)
    np.testing.assert_array_equal(q3.cpu().numpy(), q[:, src, :])
