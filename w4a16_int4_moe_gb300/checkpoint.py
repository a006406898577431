"""Load-time adapter from compressed-tensors pack-quantized INT4 weights.

The pages name the checkpoint format the operator loads: compressed-tensors
pack-quantized INT4 with groups of 32 along K and BF16 scales (page
"vLLM 宣布 Humming 后端可运行 … Chord 内核 …", section
"接入方式：用 Chord 替代公共 Humming 包"), and unsupported schemes are refused
at load instead of falling back to another kernel (page "vLLM と Novita AI が
Chord をリリース …", section "vLLM との統合").

Format, as this adapter reads it. Per expert and projection:
* ``weight_packed``: int32 [n, k/8]. Word j of a row holds the codes of
  k = 8j .. 8j+7, code i in bits 4i .. 4i+3.
* A code is the offset-binary uint4 value q of the symmetric int4 weight
  q - 8 (zero point 8).
* ``weight_scale``: BF16 [n, k/32].

On a little-endian device, the bytes of those int32 words are exactly this
library's checkpoint bytes: uint8 [n, k/2], even k in the low nibble. So the
adapter is a checked, zero-copy reinterpretation that is handed to
``w4a16_prepack``.
"""

from __future__ import annotations

import sys

import torch

from . import ops


class UnsupportedScheme(ops.W4A16Error):
    """The checkpoint's quantisation scheme is not the one the kernels run."""

    def __init__(self, why: str):
        super().__init__("load", ops.W4A16_ERR_UNSUPPORTED, why)


def pack_quantized_to_codes(weight_packed: torch.Tensor, weight_scale: torch.Tensor,
                            num_bits: int = 4, group_size: int = 32, symmetric: bool = True,
                            strategy: str = "group"):
    """(weight_packed int32 [..., n, k/8], weight_scale BF16 [..., n, k/32])
    -> (q uint8 [..., n, k/2], scales BF16), views of the same memory.

    Raises UnsupportedScheme for anything but symmetric 4-bit group-32 with
    BF16 scales: the kernels run exactly that scheme, and converting another
    one (for example FP16 scales) would change the weights silently."""
    if num_bits != 4:
        raise UnsupportedScheme(f"{num_bits}-bit weights (only 4-bit)")
    if strategy != "group" or group_size != 32:
        raise UnsupportedScheme(f"strategy {strategy!r}, group {group_size} (only group 32)")
    if not symmetric:
        raise UnsupportedScheme("asymmetric zero points (only the implicit zero point 8)")
    if weight_packed.dtype != torch.int32:
        raise UnsupportedScheme(f"packed weights of dtype {weight_packed.dtype} (only int32)")
    if weight_scale.dtype != torch.bfloat16:
        raise UnsupportedScheme(f"scales of dtype {weight_scale.dtype} (only bfloat16)")
    if sys.byteorder != "little":
        raise UnsupportedScheme("big-endian host")
    *lead, n, k8 = weight_packed.shape
    k = 8 * k8
    if tuple(weight_scale.shape) != (*lead, n, k // 32):
        raise ops.W4A16Error("load", ops.W4A16_ERR_INVALID_ARG,
                             f"scales {tuple(weight_scale.shape)} do not match weights "
                             f"[{', '.join(map(str, lead + [n]))}, {k}]")
    q = weight_packed.contiguous().view(torch.uint8).reshape(*lead, n, k // 2)
    return q, weight_scale.contiguous()


def packed_experts_from_pack_quantized(weight_packed: torch.Tensor, weight_scale: torch.Tensor,
                                       layout: int = ops.W4A16_LAYOUT_KTILE64, **scheme):
    """Stacked experts [E, n, k/8] int32 + [E, n, k/32] BF16 (on the GPU) ->
    PackedExperts ready for W4A16MoE."""
    from .moe import PackedExperts
    q, s = pack_quantized_to_codes(weight_packed, weight_scale, **scheme)
    if q.dim() != 3:
        raise ops.W4A16Error("load", ops.W4A16_ERR_INVALID_ARG,
                             "expected stacked experts [E, n, k/8]")
    return PackedExperts.from_checkpoint(q, s.view(torch.int16), layout=layout)
