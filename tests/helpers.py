"""Shared helpers of the test suite (no method arithmetic here)."""

import numpy as np
import torch

# Parity bar for floating-point GEMM outputs against the float64 oracle.
REL_L2_TOL = 5e-3
MAX_ABS_FRAC = 2e-2


def assert_close(got, ref, what="", rel_l2=REL_L2_TOL, max_abs_frac=MAX_ABS_FRAC):
    """relative L2 error <= rel_l2 and max |got - ref| <= max_abs_frac * max |ref|."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = got - ref
    denom = np.linalg.norm(ref)
    rel = np.linalg.norm(diff) / denom if denom > 0 else np.linalg.norm(diff)
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    mx = np.max(np.abs(diff)) if diff.size else 0.0
    assert rel <= rel_l2, f"{what}: relative L2 error {rel:.3e} > {rel_l2}"
    assert mx <= max_abs_frac * scale + 1e-30, f"{what}: max abs error {mx:.3e} > {max_abs_frac} * {scale:.3e}"
    return rel, mx


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """BF16 bit patterns (uint16) -> torch.bfloat16 device tensor (bit-exact)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


GUARD = 4096      # guard bytes on each side: a multiple of 256 keeps every view aligned
PATTERN = 0xA5


class Guarded:
    """A buffer of `shape` and `dtype` in the middle of a larger allocation
    whose first and last GUARD bytes hold PATTERN; ``t`` is the view a call
    writes into, ``check`` asserts that both guards are intact."""

    def __init__(self, shape, dtype, device, fill=None):
        shape = tuple(shape) if isinstance(shape, (tuple, list)) else (shape,)
        numel = int(np.prod(shape)) if shape else 1
        self.nbytes = numel * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + self.nbytes + GUARD,), PATTERN, dtype=torch.uint8,
                              device=device)
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def check(self, what):
        if self.raw.is_cuda:
            torch.cuda.synchronize()
        head = np.flatnonzero(self.raw[:GUARD].cpu().numpy() != PATTERN)
        tail = np.flatnonzero(self.raw[GUARD + self.nbytes:].cpu().numpy() != PATTERN)
        assert head.size == 0 and tail.size == 0, (
            f"{what}: guard bytes changed (head offsets {head[:8] - GUARD}, "
            f"tail offsets past the end {tail[:8]})")
