"""Helpers for the GPU parity tests: move seeded host arrays to the device
with guard zones, and read results back as numpy bit patterns."""
import numpy as np
import torch

GUARD = 256          # guard bytes before and after every destination buffer
CANARY = 0xAB

NP_TO_TORCH = {np.float32: torch.float32, np.uint16: torch.bfloat16, np.int32: torch.int32}
TORCH_TO_NP = {torch.float32: np.float32, torch.bfloat16: np.uint16, torch.int32: np.int32}
DT_CODE = {"f32": 0, "bf16": 1, "i32": 2}
NP_OF = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32}
TORCH_OF = {"f32": torch.float32, "bf16": torch.bfloat16, "i32": torch.int32}


def to_device(x: np.ndarray, dev="cuda") -> torch.Tensor:
    """Host array (bf16 as uint16 bits) -> device tensor of the matching dtype."""
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(x).to(dev)


def to_host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class Guarded:
    """A device buffer of `n` elements inside a byte allocation with canary
    guard zones; `offset_bytes` shifts the buffer start (misalignment tests)."""

    def __init__(self, n: int, dtype: str, offset_bytes: int = 0, dev="cuda"):
        es = np.dtype(NP_OF[dtype]).itemsize
        self.n, self.es, self.off = n, es, GUARD + offset_bytes
        self.raw = torch.full((GUARD * 2 + offset_bytes + n * es,), CANARY, dtype=torch.uint8,
                              device=dev)
        self.tensor = self.raw[self.off:self.off + n * es].view(TORCH_OF[dtype])

    def guards_intact(self) -> bool:
        head = self.raw[:self.off]
        tail = self.raw[self.off + self.n * self.es:]
        return bool((head == CANARY).all().item() and (tail == CANARY).all().item())

    def host(self) -> np.ndarray:
        return to_host(self.tensor)


def same_bits(a: np.ndarray, b: np.ndarray) -> bool:
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


def first_mismatch(a: np.ndarray, b: np.ndarray):
    """(index of the first differing element, number of differing elements) or None."""
    ua = a.view(np.uint8).reshape(a.size, -1)
    ub = b.view(np.uint8).reshape(b.size, -1)
    diff = np.nonzero(np.any(ua != ub, axis=1))[0]
    return None if diff.size == 0 else (int(diff[0]), int(diff.size))


def within_summation_bound(got, exp, xs):
    """Every element of an fp32 sum in another order within
    2 (P-1) 2^-24 sum_r |x_r| of the ascending fold (each side is within
    (P-1) 2^-24 sum_r |x_r| of the exact sum), or within 4 fp32 ulps of it.
    Returns (ok, elements that needed the summation bound)."""
    p = len(xs)
    abs_sum = np.zeros(exp.shape, dtype=np.float64)
    for x in xs:
        abs_sum += np.abs(x.astype(np.float64))
    d = np.abs(got.astype(np.float64) - exp.astype(np.float64))
    ulp = np.spacing(np.abs(exp).astype(np.float32)).astype(np.float64)
    by_ulp = d <= 4 * ulp
    by_bound = d <= 2 * (p - 1) * 2.0 ** -24 * abs_sum
    return bool(np.all(by_ulp | by_bound)), int(np.count_nonzero(~by_ulp & by_bound))
