"""Helpers for the GPU parity tests: guard-banded device buffers and
host <-> device views of bf16 bit patterns."""
import numpy as np
import torch

GUARD = 4096            # bytes of 0xA5 on each side of every output buffer
FILL = 0xA5


class Guarded:
    """A device buffer with guard bands; `.t` is the aligned payload view."""

    def __init__(self, numel, dtype, device="cuda"):
        esize = torch.empty(0, dtype=dtype).element_size()
        nbytes = numel * esize
        self.raw = torch.full((GUARD * 2 + nbytes + 16,), FILL, dtype=torch.uint8, device=device)
        self.nbytes = nbytes
        self.t = self.raw[GUARD:GUARD + nbytes].view(dtype)

    def intact(self):
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == FILL).all()) and bool((tail == FILL).all())


def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> host uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def bf16_from_bits(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def assert_same_f32(a: np.ndarray, b: np.ndarray, what=""):
    """Bit equality of float32 arrays (NaNs must not appear)."""
    a = np.ascontiguousarray(a, np.float32).view(np.uint32)
    b = np.ascontiguousarray(b, np.float32).view(np.uint32)
    if not np.array_equal(a, b):
        bad = np.nonzero(a != b)[0]
        i = bad[0]
        raise AssertionError(f"{what}: {bad.size} mismatches, first at {i}: "
                             f"{a[i]:#010x} ({a.view(np.float32)[i]!r}) vs {b[i]:#010x} ({b.view(np.float32)[i]!r})")


def assert_same(a: np.ndarray, b: np.ndarray, what=""):
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    if not np.array_equal(a, b):
        bad = np.nonzero(a.ravel() != b.ravel())[0]
        i = bad[0]
        raise AssertionError(f"{what}: {bad.size} mismatches of {a.size}, first at {i}: "
                             f"{a.ravel()[i]!r} vs {b.ravel()[i]!r}")


def varied_bf16(n: int, seed: int) -> np.ndarray:
    """bf16 bit patterns whose 128-blocks span many binades, with zero
    blocks, signed zeros, subnormals, outliers and the largest bf16."""
    rng = np.random.default_rng(seed)
    nb = (n + 127) // 128
    mag = np.repeat(10.0 ** rng.uniform(-38, 38, nb), 128)[:n]
    x = (rng.standard_normal(n) * mag).astype(np.float32)
    if nb > 3:
        x[128:256] = 0.0
        x[128 + 5] = -0.0
        x[256:384] = (rng.standard_normal(128) * 1e-40).astype(np.float32)     # bf16 subnormals
    out = rng.random(n) < 0.002
    x[out] *= 1000.0
    x = np.nan_to_num(x, nan=0.0, posinf=3.0e38, neginf=-3.0e38)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    if n > 600:
        bits[511] = 0x7F7F        # largest finite bf16
        bits[512] = 0xFF7F
    bits[(bits & 0x7F80) == 0x7F80] = 0x3F80      # no inf / NaN
    return bits
