"""Thin ctypes binding of ``libw4a16moe.so`` (declared in include/w4a16moe.h).

Names follow the C entry points. Every function only marshals arguments:
tensors become ``data_ptr()`` values, the stream is torch's current CUDA
stream. All computation happens in the library's CUDA kernels; a missing or
unloadable library raises ``RuntimeError`` (there is no CPU fallback).
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

W4A16_OK = 0
W4A16_ERR_INVALID_ARG = 1
W4A16_ERR_UNSUPPORTED = 2
W4A16_ERR_ROUTING = 3
W4A16_ERR_WORKSPACE = 4
W4A16_ERR_CUDA = 5
W4A16_ERR_TIMEOUT = 6

W4A16_GATE_UP = 0
W4A16_DOWN = 1
W4A16_GATE_UP_SILU = 2
W4A16_GROUPED_CONTIGUOUS = 0
W4A16_GROUPED_MASKED = 1
W4A16_FLAG_VALIDATE_ROUTING = 1
W4A16_FLAG_ACCUMULATE = 2
W4A16_FLAG_DETERMINISTIC = 8
W4A16_LAYOUT_KTILE64 = 0
W4A16_LAYOUT_KTILE64_GLU16 = 1
W4A16_DTYPE_F32 = 0
W4A16_DTYPE_BF16 = 1
W4A16_FLAG_SYNC_STATUS = 4

# Every symbol include/w4a16moe.h declares.
EXPORTED = (
    "w4a16_status_string", "w4a16_version", "w4a16_plan", "w4a16_align_capacity",
    "w4a16_moe_align_block_size", "w4a16_prepack_size", "w4a16_prepack", "w4a16_unpack",
    "w4a16_workspace_size", "w4a16_moe_indexed_gemm", "w4a16_moe_grouped_gemm",
    "w4a16_silu_and_mul", "w4a16_read_device_status", "w4a16_moe_indexed_gemm_noalloc",
    "w4a16_topk_softmax", "w4a16_deterministic_bytes", "w4a16_layer_workspace_size",
    "w4a16_moe_layer", "w4a16_moe_route_align", "w4a16_grouped_plan", "w4a16_plan_info",
)


class Plan(ctypes.Structure):
    """Mirror of w4a16_plan_t."""
    _fields_ = [(name, ctypes.c_int) for name in (
        "block_m", "bn", "bk", "stages", "b_stages", "split_k", "ctas_per_sm", "swap_ab",
        "layout", "grid", "cta_pair")]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class PlanInfo(ctypes.Structure):
    """Mirror of w4a16_plan_info_t."""
    _fields_ = [(name, ctypes.c_int) for name in (
        "mma_issuers", "acc_slots", "acc_cols", "early_epilogue", "w_stages", "b_stages")] + [
        ("smem_bytes", ctypes.c_size_t)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class W4A16Error(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t


def load_library(path: Optional[str] = None):
    """Load the library (building it first when it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = _build.LIB
        if _build.is_stale():
            _build.build_library()
    if not os.path.exists(path):
        raise RuntimeError(f"W4A16 MoE CUDA library not found at {path}")
    lib = ctypes.CDLL(path)
    sig = {
        "w4a16_status_string": (ctypes.c_char_p, [_I]),
        "w4a16_version": (_I, []),
        "w4a16_plan": (_I, [_I, _I, _I, _I, _I, ctypes.c_float, ctypes.POINTER(Plan)]),
        "w4a16_align_capacity": (_Z, [_I, _I, _I]),
        "w4a16_grouped_plan": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(Plan)]),
        "w4a16_plan_info": (_I, [ctypes.POINTER(Plan), _I, ctypes.POINTER(PlanInfo)]),
        "w4a16_moe_align_block_size": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
        "w4a16_prepack_size": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_Z)]),
        "w4a16_prepack": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
        "w4a16_unpack": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
        "w4a16_workspace_size": (_Z, [ctypes.POINTER(Plan), _I, _I]),
        "w4a16_deterministic_bytes": (_Z, [_I, _I, _I]),
        "w4a16_moe_indexed_gemm": (_I, [_I, _P, _I, _I, _I, _P, _I, _I, _P, _P, _P, _I, _P, _P,
                                        _I, ctypes.POINTER(Plan), _P, _Z, _P]),
        "w4a16_moe_grouped_gemm": (_I, [_I, _P, _I, _I, _I, _P, _I, _P, _I, _P, _I,
                                        ctypes.POINTER(Plan), _P, _Z, _P]),
        "w4a16_silu_and_mul": (_I, [_P, _I, _I, _P, _P]),
        "w4a16_topk_softmax": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
        "w4a16_moe_route_align": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                       _P, _P, _P]),
        "w4a16_read_device_status": (_I, [_P, ctypes.POINTER(_I), _P]),
        "w4a16_layer_workspace_size": (_Z, [ctypes.POINTER(Plan), _I, _I, _I]),
        "w4a16_moe_layer": (_I, [_P, _P, _I, _I, _I, _P, _I, _I, _P, _P, _P, _I, _P, _P, _I,
                                 ctypes.POINTER(Plan), _P, _Z, _P]),
        "w4a16_moe_indexed_gemm_noalloc": (_I, [_I, _P, _I, _I, _I, _P, _I, _I, _P, _P, _P, _I,
                                                _P, _P, _I, ctypes.POINTER(Plan), _P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().w4a16_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != W4A16_OK:
        raise W4A16Error(fn, status, status_string(status))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ------------------------------------------------------------- host only --

def w4a16_version() -> int:
    return load_library().w4a16_version()


def w4a16_plan(tokens: int, topk: int, num_experts: int, n: int, k: int,
               tok_e_hint: float = 0.0) -> Plan:
    p = Plan()
    _check("w4a16_plan", load_library().w4a16_plan(tokens, topk, num_experts, n, k,
                                                    float(tok_e_hint), ctypes.byref(p)))
    return p


def w4a16_align_capacity(numel: int, num_experts: int, block_m: int) -> int:
    return int(load_library().w4a16_align_capacity(numel, num_experts, block_m))


def w4a16_prepack_size(num_experts: int, n: int, k: int, group: int = 32,
                       layout: int = W4A16_LAYOUT_KTILE64) -> int:
    out = _Z(0)
    _check("w4a16_prepack_size", load_library().w4a16_prepack_size(
        num_experts, n, k, group, layout, ctypes.byref(out)))
    return int(out.value)


def w4a16_grouped_plan(kind: int, m: int, n: int, k: int, expected_m: int = 0) -> Plan:
    """The plan w4a16_moe_grouped_gemm uses when given none."""
    p = Plan()
    _check("w4a16_grouped_plan", load_library().w4a16_grouped_plan(
        kind, m, expected_m, n, k, ctypes.byref(p)))
    return p


def w4a16_plan_info(plan: Plan, k: int) -> PlanInfo:
    """What a plan becomes on the device for reduction length k."""
    info = PlanInfo()
    _check("w4a16_plan_info", load_library().w4a16_plan_info(ctypes.byref(plan), k,
                                                             ctypes.byref(info)))
    return info


def w4a16_workspace_size(plan: Plan, rows: int = 0, k: int = 0) -> int:
    """rows: routing capacity of an indexed GEMM (0 for grouped); k: the
    GEMM's reduction length."""
    return int(load_library().w4a16_workspace_size(ctypes.byref(plan), rows, k))


# ---------------------------------------------------------------- device --

def w4a16_moe_align_block_size(topk_ids: torch.Tensor, num_experts: int, block_m: int,
                               capacity: Optional[int] = None, out=None, stream=None):
    """Returns (sorted_ids, expert_ids, num_tokens_padded) int32 device tensors."""
    tokens, topk = topk_ids.shape
    numel = tokens * topk
    if capacity is None:
        capacity = w4a16_align_capacity(numel, num_experts, block_m)
    dev = topk_ids.device
    if out is None:
        out = (torch.empty(capacity, dtype=torch.int32, device=dev),
               torch.empty(capacity // block_m, dtype=torch.int32, device=dev),
               torch.empty(1, dtype=torch.int32, device=dev))
    sorted_ids, expert_ids, ntp = out
    _check("w4a16_moe_align_block_size", load_library().w4a16_moe_align_block_size(
        _ptr(topk_ids), tokens, topk, num_experts, block_m, capacity,
        _ptr(sorted_ids), _ptr(expert_ids), _ptr(ntp), _stream(stream)))
    return sorted_ids, expert_ids, ntp


def w4a16_prepack(q: torch.Tensor, scales: torch.Tensor, group: int = 32,
                  layout: int = W4A16_LAYOUT_KTILE64, out: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """q uint8 [E, n, k/2], scales BF16 [E, n, k/32] -> packed uint8 blob."""
    e, n, kh = q.shape
    k = kh * 2
    size = w4a16_prepack_size(e, n, k, group, layout)
    if out is None:
        out = torch.empty(size, dtype=torch.uint8, device=q.device)
    _check("w4a16_prepack", load_library().w4a16_prepack(
        _ptr(q), _ptr(scales), e, n, k, group, layout, _ptr(out), out.numel(), _stream(stream)))
    return out


def w4a16_unpack(packed: torch.Tensor, num_experts: int, n: int, k: int,
                 layout: int = W4A16_LAYOUT_KTILE64, stream=None):
    q = torch.empty((num_experts, n, k // 2), dtype=torch.uint8, device=packed.device)
    s = torch.empty((num_experts, n, k // 32), dtype=torch.int16, device=packed.device)
    _check("w4a16_unpack", load_library().w4a16_unpack(
        _ptr(packed), num_experts, n, k, layout, _ptr(q), _ptr(s), _stream(stream)))
    return q, s


def w4a16_deterministic_bytes(capacity: int, n: int, numel: int) -> int:
    """Extra workspace of a W4A16_FLAG_DETERMINISTIC down call."""
    return int(load_library().w4a16_deterministic_bytes(capacity, n, numel))


def new_workspace(plan: Plan, device, rows: int = 0, k: int = 0, det_n: int = 0,
                  det_numel: int = 0) -> torch.Tensor:
    """det_n, det_numel: room for a deterministic down pass of width det_n
    over det_numel flattened rows (0: none)."""
    size = w4a16_workspace_size(plan, rows, k)
    if det_n > 0:
        size += w4a16_deterministic_bytes(rows, det_n, det_numel)
    return torch.zeros(size, dtype=torch.uint8, device=device)


def w4a16_moe_indexed_gemm(mode: int, packed: torch.Tensor, num_experts: int, n: int, k: int,
                           a: torch.Tensor, tokens: int, topk: int, sorted_ids: torch.Tensor,
                           expert_ids: torch.Tensor, num_tokens_padded: torch.Tensor,
                           plan: Plan, workspace: torch.Tensor,
                           topk_weights: Optional[torch.Tensor] = None,
                           out: Optional[torch.Tensor] = None, flags: int = 0, stream=None):
    """GATE_UP: out BF16 [tokens*topk, n]; GATE_UP_SILU: out BF16
    [tokens*topk, n/2]; DOWN: out FP32 [tokens, n]."""
    if out is None:
        if mode == W4A16_GATE_UP:
            out = torch.empty((tokens * topk, n), dtype=torch.bfloat16, device=a.device)
        elif mode == W4A16_GATE_UP_SILU:
            out = torch.empty((tokens * topk, n // 2), dtype=torch.bfloat16, device=a.device)
        else:
            out = torch.empty((tokens, n), dtype=torch.float32, device=a.device)
    _check("w4a16_moe_indexed_gemm", load_library().w4a16_moe_indexed_gemm(
        mode, _ptr(packed), num_experts, n, k, _ptr(a), tokens, topk, _ptr(sorted_ids),
        _ptr(expert_ids), _ptr(num_tokens_padded), sorted_ids.numel(), _ptr(topk_weights),
        _ptr(out), flags, ctypes.byref(plan), _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return out


def w4a16_moe_grouped_gemm(kind: int, packed: torch.Tensor, num_experts: int, n: int, k: int,
                           a: torch.Tensor, m: int, layout: torch.Tensor, workspace: torch.Tensor,
                           plan: Optional[Plan] = None, expected_m: int = 0,
                           out: Optional[torch.Tensor] = None, flags: int = 0, stream=None):
    """CONTIGUOUS: a [m, k] -> out [m, n]; MASKED: a [E, m, k] -> out [E, m, n] (BF16)."""
    if out is None:
        shape = (m, n) if kind == W4A16_GROUPED_CONTIGUOUS else (num_experts, m, n)
        out = torch.empty(shape, dtype=torch.bfloat16, device=a.device)
    _check("w4a16_moe_grouped_gemm", load_library().w4a16_moe_grouped_gemm(
        kind, _ptr(packed), num_experts, n, k, _ptr(a), m, _ptr(layout), expected_m, _ptr(out),
        flags, None if plan is None else ctypes.byref(plan), _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return out


def w4a16_layer_workspace_size(plan: Plan, rows: int, hidden: int, inter: int) -> int:
    return int(load_library().w4a16_layer_workspace_size(ctypes.byref(plan), rows, hidden, inter))


def w4a16_moe_layer(packed_gate_up: torch.Tensor, packed_down: torch.Tensor, num_experts: int,
                    hidden: int, inter: int, x: torch.Tensor, tokens: int, topk: int,
                    sorted_ids: torch.Tensor, expert_ids: torch.Tensor,
                    num_tokens_padded: torch.Tensor, plan: Plan, workspace: torch.Tensor,
                    topk_weights: torch.Tensor, out: Optional[torch.Tensor] = None,
                    flags: int = 0, stream=None):
    """The layer's gate_up (fused activation) and down in one launch:
    out FP32 [tokens, hidden]."""
    if out is None:
        out = torch.empty((tokens, hidden), dtype=torch.float32, device=x.device)
    _check("w4a16_moe_layer", load_library().w4a16_moe_layer(
        _ptr(packed_gate_up), _ptr(packed_down), num_experts, hidden, inter, _ptr(x), tokens,
        topk, _ptr(sorted_ids), _ptr(expert_ids), _ptr(num_tokens_padded), sorted_ids.numel(),
        _ptr(topk_weights), _ptr(out), flags, ctypes.byref(plan), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return out


def w4a16_topk_softmax(logits: torch.Tensor, topk: int, renormalize: bool = True,
                       expert_offset: int = 0, num_local_experts: Optional[int] = None,
                       out=None, stream=None):
    """logits fp32/BF16 [T, E] -> (topk_ids int32 [T, topk] local or -1,
    topk_weights fp32 [T, topk])."""
    tokens, e = logits.shape
    if num_local_experts is None:
        num_local_experts = e
    dtype = {torch.float32: W4A16_DTYPE_F32, torch.bfloat16: W4A16_DTYPE_BF16}.get(logits.dtype)
    if dtype is None:
        raise W4A16Error("w4a16_topk_softmax", W4A16_ERR_INVALID_ARG,
                         f"logits of dtype {logits.dtype}")
    if out is None:
        out = (torch.empty((tokens, topk), dtype=torch.int32, device=logits.device),
               torch.empty((tokens, topk), dtype=torch.float32, device=logits.device))
    ids, w = out
    _check("w4a16_topk_softmax", load_library().w4a16_topk_softmax(
        _ptr(logits.contiguous()), dtype, tokens, e, topk, int(bool(renormalize)), expert_offset,
        num_local_experts, _ptr(ids), _ptr(w), _stream(stream)))
    return ids, w


def w4a16_moe_route_align(logits: torch.Tensor, topk: int, block_m: int,
                          arrivals: torch.Tensor, renormalize: bool = True,
                          expert_offset: int = 0, num_local_experts: Optional[int] = None,
                          capacity: Optional[int] = None, out=None, stream=None):
    """Top-k routing and moe_align_block_size in one launch. arrivals: int32
    [1] device, zero before the first call (each call leaves it zero).
    Returns (topk_ids, topk_weights, sorted_ids, expert_ids, num_tokens_padded)."""
    tokens, e = logits.shape
    if num_local_experts is None:
        num_local_experts = e
    dtype = {torch.float32: W4A16_DTYPE_F32, torch.bfloat16: W4A16_DTYPE_BF16}.get(logits.dtype)
    if dtype is None:
        raise W4A16Error("w4a16_moe_route_align", W4A16_ERR_INVALID_ARG,
                         f"logits of dtype {logits.dtype}")
    if capacity is None:
        capacity = w4a16_align_capacity(tokens * topk, num_local_experts, block_m)
    dev = logits.device
    if out is None:
        out = (torch.empty((tokens, topk), dtype=torch.int32, device=dev),
               torch.empty((tokens, topk), dtype=torch.float32, device=dev),
               torch.empty(capacity, dtype=torch.int32, device=dev),
               torch.empty(capacity // block_m, dtype=torch.int32, device=dev),
               torch.empty(1, dtype=torch.int32, device=dev))
    ids, w, sorted_ids, expert_ids, ntp = out
    logits = logits.contiguous()
    _check("w4a16_moe_route_align", load_library().w4a16_moe_route_align(
        _ptr(logits), dtype, tokens, e, topk, int(bool(renormalize)), expert_offset,
        num_local_experts, block_m, sorted_ids.numel(), _ptr(ids), _ptr(w), _ptr(sorted_ids),
        _ptr(expert_ids), _ptr(ntp), _ptr(arrivals), _stream(stream)))
    return ids, w, sorted_ids, expert_ids, ntp


def w4a16_silu_and_mul(x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None):
    rows, two_i = x.shape
    inter = two_i // 2
    if out is None:
        out = torch.empty((rows, inter), dtype=torch.bfloat16, device=x.device)
    _check("w4a16_silu_and_mul", load_library().w4a16_silu_and_mul(
        _ptr(x), rows, inter, _ptr(out), _stream(stream)))
    return out


def w4a16_read_device_status(workspace: torch.Tensor, stream=None):
    """(status, raw word): W4A16_OK, or W4A16_ERR_TIMEOUT when a wait gave up."""
    detail = _I(0)
    st = load_library().w4a16_read_device_status(_ptr(workspace), ctypes.byref(detail),
                                                 _stream(stream))
    if st not in (W4A16_OK, W4A16_ERR_TIMEOUT):
        _check("w4a16_read_device_status", st)
    return st, int(detail.value)


def w4a16_moe_indexed_gemm_noalloc(mode: int, packed: torch.Tensor, num_experts: int, n: int,
                                   k: int, a: torch.Tensor, tokens: int, topk: int,
                                   sorted_ids: torch.Tensor, expert_ids: torch.Tensor,
                                   num_tokens_padded: torch.Tensor, plan: Plan,
                                   topk_weights: Optional[torch.Tensor] = None,
                                   out: Optional[torch.Tensor] = None, flags: int = 0,
                                   stream=None):
    """w4a16_moe_indexed_gemm for callers that cannot allocate device memory:
    no workspace argument; the library's built-in 32 MiB device array serves
    as the workspace. Only ``out`` is allocated here when the caller passes
    none (a caller that cannot allocate passes its own)."""
    if out is None:
        if mode == W4A16_GATE_UP:
            out = torch.empty((tokens * topk, n), dtype=torch.bfloat16, device=a.device)
        else:
            out = torch.empty((tokens, n), dtype=torch.float32, device=a.device)
    _check("w4a16_moe_indexed_gemm_noalloc", load_library().w4a16_moe_indexed_gemm_noalloc(
        mode, _ptr(packed), num_experts, n, k, _ptr(a), tokens, topk, _ptr(sorted_ids),
        _ptr(expert_ids), _ptr(num_tokens_padded), sorted_ids.numel(), _ptr(topk_weights),
        _ptr(out), flags, ctypes.byref(plan), _stream(stream)))
    return out
