"""The compressed-tensors pack-quantized adapter (host side, no GPU).

The packed int32 words are built here from signed int4 weights by the
format's own rule (code = weight + 8, code i of a word in bits 4i..4i+3),
independently of the library's byte layout, and the adapter's view must be
the library's checkpoint bytes (even k in the low nibble) that encode the
same weights."""

import numpy as np
import pytest
import torch

from w4a16_int4_moe_gb300 import checkpoint, ops
from w4a16_int4_moe_gb300 import workloads as wl


def _pack_int32(wq):
    """Signed int4 weights [n, k] -> int32 words [n, k/8] (format rule)."""
    n, k = wq.shape
    codes = (wq + 8).astype(np.uint32)
    words = np.zeros((n, k // 8), dtype=np.uint32)
    for i in range(8):
        words |= codes[:, i::8] << np.uint32(4 * i)
    return words.view(np.int32)


def test_pack_quantized_view_equals_library_bytes():
    rng = np.random.default_rng(3)
    wq = rng.integers(-8, 8, size=(2, 5, 64))            # two experts, n = 5, k = 64
    words = np.stack([_pack_int32(w) for w in wq])
    scales = wl.to_bf16_bits(np.abs(rng.standard_normal((2, 5, 2), dtype=np.float32)))
    q, s = checkpoint.pack_quantized_to_codes(torch.from_numpy(words),
                                              torch.from_numpy(scales.view(np.int16)).view(
                                                  torch.bfloat16))
    q = q.numpy()
    assert q.shape == (2, 5, 32) and q.dtype == np.uint8
    # the library's rule: byte j holds k = 2j (low nibble) and 2j + 1 (high)
    lo, hi = (q & 0xF).astype(np.int64) - 8, (q >> 4).astype(np.int64) - 8
    np.testing.assert_array_equal(lo, wq[..., 0::2])
    np.testing.assert_array_equal(hi, wq[..., 1::2])
    np.testing.assert_array_equal(s.view(torch.int16).numpy().view(np.uint16), scales)


def test_view_shares_memory():
    words = torch.zeros((3, 128, 8), dtype=torch.int32)
    scales = torch.zeros((3, 128, 2), dtype=torch.bfloat16)
    q, _ = checkpoint.pack_quantized_to_codes(words, scales)
    words[1, 2, 3] = 0x7654_3210
    assert q[1, 2, 12:16].tolist() == [0x10, 0x32, 0x54, 0x76]


@pytest.mark.parametrize("kw,what", [
    (dict(num_bits=8), "8-bit"),
    (dict(group_size=128), "group 128"),
    (dict(strategy="channel"), "channel"),
    (dict(symmetric=False), "asymmetric"),
])
def test_unsupported_schemes_are_refused_at_load(kw, what):
    words = torch.zeros((128, 8), dtype=torch.int32)
    scales = torch.zeros((128, 2), dtype=torch.bfloat16)
    with pytest.raises(checkpoint.UnsupportedScheme) as ei:
        checkpoint.pack_quantized_to_codes(words, scales, **kw)
    assert ei.value.status == ops.W4A16_ERR_UNSUPPORTED, what


def test_fp16_scales_and_wrong_shapes_are_refused():
    words = torch.zeros((128, 8), dtype=torch.int32)
    with pytest.raises(checkpoint.UnsupportedScheme):
        checkpoint.pack_quantized_to_codes(words, torch.zeros((128, 2), dtype=torch.float16))
    with pytest.raises(checkpoint.UnsupportedScheme):
        checkpoint.pack_quantized_to_codes(words.to(torch.int64),
                                           torch.zeros((128, 2), dtype=torch.bfloat16))
    with pytest.raises(ops.W4A16Error) as ei:
        checkpoint.pack_quantized_to_codes(words, torch.zeros((128, 3), dtype=torch.bfloat16))
    assert ei.value.status == ops.W4A16_ERR_INVALID_ARG
