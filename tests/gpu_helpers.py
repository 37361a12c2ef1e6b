"""Helpers shared by the -m gpu parity tests (test infrastructure)."""
import numpy as np
import torch

import __graft_entry__

GEMM_REL_FROB = 1e-3      # vs the BF16-rounded float64 oracle
GEMM_ELEM_REL = 4e-3      # |Y - Y64| <= 4e-3 * (|A| |W|^T) + 1e-6
GEMM_ELEM_ABS = 1e-6

_built = False


def device():
    global _built
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    if not _built:
        __graft_entry__.build()
        _built = True
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def np_f32_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


class Canary:
    """An output buffer with guard bytes on both sides; check() asserts the
    kernel wrote nothing outside the view it was given."""

    def __init__(self, numel: int, dtype, dev, pad: int = 4096, fill=0x5A):
        self.pad = pad
        itemsize = torch.empty((), dtype=dtype).element_size()
        total = (numel + 2 * pad) * itemsize
        self.raw = torch.full((total,), fill, dtype=torch.uint8, device=dev)
        self.fill = fill
        self.view = self.raw[pad * itemsize:pad * itemsize + numel * itemsize].view(dtype)
        self.itemsize = itemsize

    def check(self):
        raw = self.raw.cpu().numpy()
        p = self.pad * self.itemsize
        assert (raw[:p] == self.fill).all(), "write before the output buffer"
        assert (raw[-p:] == self.fill).all(), "write after the output buffer"


def check_gemm(y_gpu: torch.Tensor, y64: np.ndarray, absprod: np.ndarray, what=""):
    import oracle
    yg = y_gpu.float().cpu().numpy().astype(np.float64)
    ref16 = oracle.bf16_round(y64).astype(np.float64)
    num = np.linalg.norm(yg - ref16)
    den = np.linalg.norm(ref16)
    assert num <= GEMM_REL_FROB * den + 1e-30, "%s: rel Frobenius %.3g" % (what, num / max(den, 1e-300))
    bound = GEMM_ELEM_REL * absprod + GEMM_ELEM_ABS
    bad = np.abs(yg - y64) > bound
    assert not bad.any(), "%s: %d elements outside |d| <= 4e-3 |A||W| + 1e-6, worst %s" % (
        what, bad.sum(), np.max(np.abs(yg - y64) / bound))
